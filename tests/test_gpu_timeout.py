"""The timeout path of the tensor-core contraction, made to run out on
purpose and without any fault: the test hook sets the bound of every
in-kernel wait to a single try, so the first wait that finds its phase still
open gives up. The kernel must report PEAGLE_DEV_TIMEOUT in the library
status word, drain what it issued, and leave the device usable: after the
status is cleared and the bound restored, the same contraction is exact."""
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


def _case(M, N, K, seed):
    rng = np.random.default_rng(seed)
    X = synth.bf16_round(rng.standard_normal((M, K), dtype=np.float32))
    W = synth.bf16_round(rng.standard_normal((N, K), dtype=np.float32))
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    return (torch.from_numpy(X).to(torch.bfloat16).cuda(), torch.from_numpy(W).to(torch.bfloat16).cuda(),
            ref)


def _rel(D, ref):
    return float(np.max(np.abs(D.cpu().numpy() - ref)) / np.max(np.abs(ref)))


@pytest.mark.parametrize("noalloc", [False, True])
@pytest.mark.parametrize("M,N,K", [(4, 512, 256),
                                   # 512 rows in four K slices whose CTAs wait for one
                                   # another to share each tile's sum
                                   (512, 1024, 4096)])
def test_wait_that_runs_out_is_reported_and_the_device_recovers(pe, noalloc, M, N, K):
    X, W, ref = _case(M, N, K, seed=11)
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    nb = pe.peagle_gemm_workspace_size(pe.PEAGLE_BF16, M, N, K)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")

    def run():
        if noalloc:
            pe.peagle_gemm_noalloc(pe.PEAGLE_BF16, M, N, K, X, W, D)
        else:
            pe.peagle_gemm(pe.PEAGLE_BF16, M, N, K, X, W, D, ws, ws.numel())

    pe.peagle_clear_library_status()
    assert pe.peagle_get_library_status() == 0
    pe.peagle_set_wait_limit_ns(0)
    try:
        run()
        status = pe.peagle_get_library_status()
    finally:
        pe.peagle_set_wait_limit_ns(10 ** 9)
    assert status & pe.PEAGLE_DEV_TIMEOUT, status
    pe.peagle_clear_library_status()
    assert pe.peagle_get_library_status() == 0
    D.fill_(float("nan"))
    run()
    torch.cuda.synchronize()
    assert pe.peagle_get_library_status() == 0
    assert _rel(D, ref) < 1e-5
