"""peagle_gemm_noalloc: the dense contraction for callers that cannot
allocate device memory (engines whose allocator owns the whole device heap,
plugins forbidden to allocate, latency-critical loops that cannot take
cudaMalloc's synchronisation). Its split-K scratch is a fixed array inside
the library. Its results must match peagle_gemm, the entry point that takes
a caller workspace, on two calls in a row (the array keeps the previous
call's contents). This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import eagle_speculative_drafting_gb300 as m
    return m


def _operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    X = synth.bf16_round(rng.standard_normal((M, K), dtype=np.float32))
    W = synth.bf16_round(rng.standard_normal((N, K), dtype=np.float32))
    return (torch.from_numpy(X).to(torch.bfloat16).cuda(),
            torch.from_numpy(W).to(torch.bfloat16).cuda())


def _with_workspace(pe, M, N, K, X, W):
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    nb = pe.peagle_gemm_workspace_size(pe.PEAGLE_BF16, M, N, K)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    pe.peagle_gemm(pe.PEAGLE_BF16, M, N, K, X, W, D, ws, ws.numel())
    return D


def _max_abs_rel(a, b):
    a = a.double().cpu()
    b = b.double().cpu()
    return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))


@pytest.mark.parametrize("shapes", [[(4, 4096, 4096), (16, 1000, 2048)],
                                    [(64, 4096, 1024), (4, 4096, 4096)],
                                    # more than 256 rows: wide tiles whose long K is cut into
                                    # four slices, summed through the fixed array
                                    [(300, 1024, 9000), (16, 1000, 2048)]])
def test_noalloc_matches_workspace_gemm_twice_in_a_row(pe, shapes):
    ops = [_operands(M, N, K, seed=M + N + K + i) for i, (M, N, K) in enumerate(shapes)]
    refs = [_with_workspace(pe, M, N, K, X, W) for (M, N, K), (X, W) in zip(shapes, ops)]
    outs = []
    for (M, N, K), (X, W) in zip(shapes, ops):      # two calls back to back
        D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        pe.peagle_gemm_noalloc(pe.PEAGLE_BF16, M, N, K, X, W, D)
        outs.append(D)
    torch.cuda.synchronize()
    for (M, N, K), D, ref in zip(shapes, outs, refs):
        assert _max_abs_rel(D, ref) <= 1e-5, (M, N, K)


def test_noalloc_rejects_sizes_beyond_its_array(pe):
    M, N, K = 512, 32000, 64
    X, W = _operands(M, N, K, seed=3)
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    with pytest.raises(pe.PeagleError) as e:
        pe.peagle_gemm_noalloc(pe.PEAGLE_BF16, M, N, K, X, W, D)
    assert e.value.status == pe.PEAGLE_ERR_UNSUPPORTED
    assert "partial floats" in pe.peagle_last_error()


def test_noalloc_f32_matches_workspace_gemm(pe):
    # the fp32 contraction runs on the CUDA cores straight into D
    rng = np.random.default_rng(5)
    M, N, K = 65, 130, 100
    X = torch.from_numpy(rng.standard_normal((M, K), dtype=np.float32)).cuda()
    W = torch.from_numpy(rng.standard_normal((N, K), dtype=np.float32)).cuda()
    ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
    pe.peagle_gemm(pe.PEAGLE_F32, M, N, K, X, W, ref, None, 0)
    for _ in range(2):
        D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        pe.peagle_gemm_noalloc(pe.PEAGLE_F32, M, N, K, X, W, D)
        torch.cuda.synchronize()
        assert _max_abs_rel(D, ref) <= 1e-6
