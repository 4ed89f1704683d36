"""Checkpoint I/O through the C ABI in host-memory mode (no GPU needed): the
files must be what vLLM's parallel-drafting loader reads -- a standard
EAGLE-3 draft checkpoint plus "mask_hidden" [1, num_aux * target_hidden] and
"parallel_drafting" / "ptd_token_id" in config.json ("feat(speculative) ...
#2376", Checkpoint contract) -- and must round-trip bit for bit. The files
are read back here with an independent safetensors reader."""
import json
import os
import struct

import numpy as np
import pytest

import synth


@pytest.fixture(scope="module")
def pe():
    import __graft_entry__
    __graft_entry__.build()
    import eagle_speculative_drafting_gb300 as m
    return m


def small(dtype="bf16", **kw):
    base = synth.WORKLOADS["tiny_f32_decode"].scaled(
        dtype=dtype, hidden=64, target_hidden=32, num_aux=3, num_layers=2, num_q_heads=4,
        num_kv_heads=2, head_dim=16, intermediate=96, vocab=300, seed=91)
    return base.scaled(**kw) if kw else base


def host_buffers(wl, W):
    """The weights as host arrays in the model dtype (bf16 as raw uint16)."""
    def conv(a):
        a = np.ascontiguousarray(a, dtype=np.float32)
        return (a.view(np.uint32) >> 16).astype(np.uint16) if wl.dtype == "bf16" else a
    out = {}
    for k, v in W.items():
        if k == "layers":
            out["layers"] = [{kk: (None if vv is None else conv(vv)) for kk, vv in L.items()} for L in v]
        elif k in ("d2t", "t2d"):
            out[k] = None if v is None else np.ascontiguousarray(v, dtype=np.int32)
        else:
            out[k] = conv(v)
    return out


def empty_like_buffers(buf):
    out = {}
    for k, v in buf.items():
        if k == "layers":
            out["layers"] = [{kk: (None if vv is None else np.full_like(vv, 7)) for kk, vv in L.items()} for L in v]
        else:
            out[k] = None if v is None else np.full_like(v, 7)
    return out


def read_safetensors(path):
    raw = open(path, "rb").read()
    n = struct.unpack("<Q", raw[:8])[0]
    header = json.loads(raw[8:8 + n])
    data = raw[8 + n:]
    np_dt = {"BF16": np.uint16, "F32": np.float32, "I64": np.int64, "BOOL": np.bool_}
    out = {}
    for name, e in header.items():
        if name == "__metadata__":
            continue
        b, end = e["data_offsets"]
        out[name] = (e["dtype"], np.frombuffer(data[b:end], dtype=np_dt[e["dtype"]]).reshape(e["shape"]))
    return out


def maps(V, Vd, seed):
    d2t = np.sort(np.random.default_rng(seed).choice(V, Vd, replace=False)).astype(np.int32)
    t2d = np.full(V, -1, dtype=np.int32)
    t2d[d2t] = np.arange(Vd)
    return d2t, t2d


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_checkpoint_round_trip_host(pe, tmp_path, dtype):
    from eagle_speculative_drafting_gb300.marshal import config_of
    from eagle_speculative_drafting_gb300.model import weights_struct
    wl = small(dtype)
    W = synth.make_weights(wl)
    Vd = 200
    d2t, t2d = maps(wl.vocab, Vd, 3)
    W = dict(W, lm_head_w=W["lm_head_w"][:Vd].copy(), d2t=d2t, t2d=t2d)
    cfg = config_of(wl, norm_before_residual=0, draft_vocab=Vd)
    buf = host_buffers(wl, W)
    w, keep = weights_struct(buf)
    pe.peagle_checkpoint_save(str(tmp_path), cfg, w, memory=pe.PEAGLE_MEM_HOST)

    # config.json: the P-EAGLE additions and the sizes
    cj = json.load(open(tmp_path / "config.json"))
    assert cj["parallel_drafting"] is True and cj["ptd_token_id"] == wl.ptd_token_id
    assert cj["hidden_size"] == wl.hidden and cj["num_hidden_layers"] == wl.num_layers
    assert cj["vocab_size"] == wl.vocab and cj["draft_vocab_size"] == Vd
    assert cj["num_key_value_heads"] == wl.num_kv_heads and cj["norm_before_residual"] is False
    # model.safetensors: names, shapes, dtypes, values
    st = read_safetensors(tmp_path / "model.safetensors")
    A, Ht, H = wl.num_aux, wl.target_hidden, wl.hidden
    sdt = "BF16" if dtype == "bf16" else "F32"
    assert st["mask_hidden"][0] == sdt and st["mask_hidden"][1].shape == (1, A * Ht)
    assert np.array_equal(st["mask_hidden"][1], buf["mask_hidden"])
    assert np.array_equal(st["fc.weight"][1], buf["fc_w"])
    assert np.array_equal(st["lm_head.weight"][1], buf["lm_head_w"])
    nq, nkv, hd, I = wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.intermediate
    for l, L in enumerate(buf["layers"]):
        p = f"layers.{l}."
        q = st[p + "self_attn.q_proj.weight"][1]
        k = st[p + "self_attn.k_proj.weight"][1]
        v = st[p + "self_attn.v_proj.weight"][1]
        assert np.array_equal(np.concatenate([q, k, v]), L["qkv_w"])
        assert q.shape == (nq * hd, 2 * H if l == 0 else H) and k.shape == v.shape == (nkv * hd, q.shape[1])
        assert np.array_equal(np.concatenate([st[p + "mlp.gate_proj.weight"][1], st[p + "mlp.up_proj.weight"][1]]),
                              L["gate_up_w"])
        assert st[p + "mlp.gate_proj.weight"][1].shape == (I, H)
        assert ((p + "hidden_norm.weight") in st) == (l == 0)
    assert st["d2t"][0] == "I64" and np.array_equal(st["d2t"][1], d2t - np.arange(Vd))
    assert st["t2d"][0] == "BOOL" and np.array_equal(st["t2d"][1], t2d >= 0)

    # read back: config, then every buffer bit for bit
    cfg2 = pe.peagle_checkpoint_load_config(str(tmp_path))
    for f, _ in cfg._fields_:
        assert getattr(cfg2, f) == getattr(cfg, f), f
    out = empty_like_buffers(buf)
    w2, keep2 = weights_struct(out)
    pe.peagle_checkpoint_load(str(tmp_path), cfg2, w2, memory=pe.PEAGLE_MEM_HOST)
    for k, v in buf.items():
        if k == "layers":
            for L, L2 in zip(v, out["layers"]):
                for kk in L:
                    if L[kk] is not None:
                        assert np.array_equal(L[kk], L2[kk]), kk
        else:
            assert np.array_equal(v, out[k]), k


def test_checkpoint_f32_file_into_bf16_model(pe, tmp_path):
    # an fp32 checkpoint of bf16-representable values loads exactly into a
    # bf16 model (round to nearest even on the host)
    from eagle_speculative_drafting_gb300.marshal import config_of
    from eagle_speculative_drafting_gb300.model import weights_struct
    wl32 = small("f32")
    W = synth.make_weights(wl32.scaled(dtype="bf16"))   # values already bf16-rounded
    buf32 = host_buffers(wl32, W)
    w, keep = weights_struct(buf32)
    pe.peagle_checkpoint_save(str(tmp_path), config_of(wl32), w, memory=pe.PEAGLE_MEM_HOST)
    wl16 = small("bf16")
    buf16 = host_buffers(wl16, W)
    out = empty_like_buffers(buf16)
    w2, keep2 = weights_struct(out)
    pe.peagle_checkpoint_load(str(tmp_path), config_of(wl16), w2, memory=pe.PEAGLE_MEM_HOST)
    assert np.array_equal(out["fc_w"], buf16["fc_w"])
    assert np.array_equal(out["layers"][1]["down_w"], buf16["layers"][1]["down_w"])


def test_checkpoint_rejects_non_peagle_and_incomplete(pe, tmp_path):
    from eagle_speculative_drafting_gb300.marshal import config_of
    from eagle_speculative_drafting_gb300.model import weights_struct
    wl = small("f32")
    W = synth.make_weights(wl)
    buf = host_buffers(wl, W)
    w, keep = weights_struct(buf)
    cfg = config_of(wl)
    pe.peagle_checkpoint_save(str(tmp_path), cfg, w, memory=pe.PEAGLE_MEM_HOST)
    cj = json.load(open(tmp_path / "config.json"))
    # no ptd_token_id: no silent default
    bad = dict(cj)
    del bad["ptd_token_id"]
    json.dump(bad, open(tmp_path / "config.json", "w"))
    with pytest.raises(pe.PeagleError) as e:
        pe.peagle_checkpoint_load_config(str(tmp_path))
    assert "ptd_token_id" in pe.peagle_last_error()
    bad = dict(cj, parallel_drafting=False)
    json.dump(bad, open(tmp_path / "config.json", "w"))
    with pytest.raises(pe.PeagleError):
        pe.peagle_checkpoint_load_config(str(tmp_path))
    # a model shape the file does not hold
    out = empty_like_buffers(buf)
    w2, keep2 = weights_struct(out)
    cfg_big = config_of(wl.scaled(intermediate=wl.intermediate + 8))
    with pytest.raises(pe.PeagleError) as e:
        pe.peagle_checkpoint_load(str(tmp_path), cfg_big, w2, memory=pe.PEAGLE_MEM_HOST)
    assert e.value.status == pe.PEAGLE_ERR_INVALID_ARG and "shape" in pe.peagle_last_error()
    # a missing directory
    with pytest.raises(pe.PeagleError):
        pe.peagle_checkpoint_load_config(str(tmp_path / "nowhere"))
