"""CPU checks of the C ABI: the library loads, exports every declared entry
point, and rejects invalid arguments on the host before touching the GPU.
The host-side COD count rule is compared with the oracle exactly."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "peagle.h")


@pytest.fixture(scope="module")
def pe():
    import __graft_entry__
    __graft_entry__.build()
    import eagle_speculative_drafting_gb300 as pe
    return pe


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(peagle_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for f in ("peagle_draft_step", "peagle_verify_accept", "peagle_cod_select",
              "peagle_parallel_forward"):
        assert f in names


def test_library_exports_every_declared_symbol(pe):
    lib = ctypes.CDLL(pe.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(pe):
    assert "sm_103a" in pe.peagle_version()
    assert pe._lib.peagle_status_string(pe.PEAGLE_ERR_WORKSPACE).decode().startswith("workspace")


@pytest.mark.parametrize("n,K,r,rmin", [(4096, 4, 0.7, 0.2), (32768, 8, 0.7, 0.2), (0, 3, 0.7, 0.2),
                                         (1, 1, 0.5, 0.5), (999, 16, 0.93, 0.01), (12345, 7, 1.0, 1.0),
                                         (100, 5, 0.5, 0.3)])
def test_cod_counts_match_oracle(pe, n, K, r, rmin):
    from oracle import peagle_oracle as O
    assert pe.peagle_cod_counts(n, K, r, rmin) == O.cod_counts(n, K, r, rmin)


@pytest.mark.parametrize("args", [(10, 0, 0.7, 0.2), (10, 17, 0.7, 0.2), (10, 4, 0.7, 0.8),
                                  (10, 4, 1.5, 0.2), (10, 4, 0.7, 0.0), (-1, 4, 0.7, 0.2)])
def test_cod_counts_rejects(pe, args):
    with pytest.raises(pe.PeagleError) as e:
        pe.peagle_cod_counts(*args)
    assert e.value.status == pe.PEAGLE_ERR_INVALID_ARG


def test_verify_rejects_bad_sizes_without_launch(pe):
    before = pe.peagle_kernel_launches()
    with pytest.raises(pe.PeagleError) as e:
        pe.peagle_verify_accept(4, 0, 1, 1, 1, 1, stream=0)
    assert e.value.status == pe.PEAGLE_ERR_INVALID_ARG
    with pytest.raises(pe.PeagleError):
        pe.peagle_verify_accept(4, 3, None, 1, 1, 1, stream=0)
    pe.peagle_verify_accept(0, 3, None, None, None, None, stream=0)   # empty batch: no-op
    assert pe.peagle_kernel_launches() == before


def _cfg(pe, **kw):
    base = dict(hidden=64, target_hidden=32, num_aux=3, num_layers=1, num_q_heads=4,
                num_kv_heads=2, head_dim=64, intermediate=128, target_vocab=100, draft_vocab=100,
                ptd_token_id=99, dtype="bf16")
    base.update(kw)
    return pe.make_config(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(ptd_token_id=100), 1), (dict(ptd_token_id=-1), 1), (dict(num_q_heads=3), 1),
    (dict(head_dim=96), 2), (dict(hidden=0), 1), (dict(dtype=7), 1), (dict(intermediate=100), 2),
    (dict(rms_eps=0.0), 1), (dict(norm_before_residual=2), 1), (dict(hidden=16384), 2)])
def test_model_create_validates_config_first(pe, kw, status):
    cfg = _cfg(pe, **kw)
    if "dtype" in kw and kw["dtype"] == 7:
        cfg.dtype = 7
    w = pe.peagle_weights()
    with pytest.raises(pe.PeagleError) as e:
        pe.peagle_model_create(cfg, w, stream=0)
    assert e.value.status == status


def test_model_create_requires_weights(pe):
    with pytest.raises(pe.PeagleError) as e:
        pe.peagle_model_create(_cfg(pe), pe.peagle_weights(), stream=0)
    assert e.value.status == pe.PEAGLE_ERR_INVALID_ARG
    assert "NULL" in pe.peagle_last_error()


def test_draft_step_rejects_null_model_and_bad_K(pe):
    for B, K in ((1, 4), (1, 0), (1, 17)):
        with pytest.raises(pe.PeagleError) as e:
            pe.peagle_draft_step(None, B, K, 0, 0, 0, [0], [0], 0, 0, 0, 0, 0, 0, None, 0, 0, stream=0)
        assert e.value.status == pe.PEAGLE_ERR_INVALID_ARG


def test_gemm_and_forward_validation(pe):
    with pytest.raises(pe.PeagleError):
        pe.peagle_gemm(pe.PEAGLE_BF16, 4, 4, 0, 1, 1, 1, None, 0, stream=0)
    with pytest.raises(pe.PeagleError):
        pe.peagle_gemm(9, 4, 4, 8, 1, 1, 1, None, 0, stream=0)
    assert pe.peagle_gemm_workspace_size(pe.PEAGLE_F32, 4, 4, 8) == 0
    with pytest.raises(pe.PeagleError):
        pe.peagle_parallel_forward(None, 4, 0, 0, 0, 0, 1, 0, None, 4, 0.7, 0.2, 0, 0.8,
                                   0, 0, 0, 0, None, None, None, 0, 0, stream=0)


def test_probe_api_validates(pe):
    with pytest.raises(pe.PeagleError):
        pe.peagle_probe_begin(99, 4)
    assert pe.peagle_op_name(4) == "gate_up"


def test_verify_sample_rejects_bad_sizes_without_launch(pe):
    before = pe.peagle_kernel_launches()
    for B, K, V in ((2, 0, 10), (2, 65, 10), (2, 4, 0), (2, 4, (1 << 23) + 1), (-1, 4, 10)):
        with pytest.raises(pe.PeagleError) as e:
            pe.peagle_verify_sample(B, K, V, 1, 1, 1, 1, 1, 1, 1, stream=0)
        assert e.value.status == pe.PEAGLE_ERR_INVALID_ARG
    with pytest.raises(pe.PeagleError):
        pe.peagle_verify_sample(2, 4, 10, None, 1, 1, 1, 1, 1, 1, stream=0)
    pe.peagle_verify_sample(0, 4, 10, None, None, None, None, None, None, None, stream=0)
    assert pe.peagle_kernel_launches() == before
