"""GPU parity: the CUDA library through its C ABI against the CPU oracle on
the same seeded inputs.

Bars: integers bit-exact (COD indices, verify, argmax tokens given clear
margins); floats within max|gpu - ref| / max|ref| <= 1e-4 (fp32 models) or
2e-2 (bf16 models). A bf16 draft token may differ from the oracle's only at a
near-tie: where the oracle's own top-1 / top-2 margin is below 2e-2 of the
largest |logit|; and every GPU token must equal the argmax of the GPU's own
exported logits exactly.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import peagle_oracle as O

pytestmark = pytest.mark.gpu

F32_TOL = 1e-4
BF16_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def H():
    from tests import harness
    return harness


def pe():
    import eagle_speculative_drafting_gb300 as m
    return m


# ------------------------------------------------------------------ GEMM
GEMM_SHAPES = [(1, 128, 64), (4, 256, 128), (3, 200, 520), (16, 384, 1024), (17, 1000, 256),
               (64, 4096, 4096), (100, 1000, 2048), (256, 512, 256), (257, 640, 512),
               (512, 4096, 1024), (1000, 300, 200), (333, 32000, 128),
               # swapped with at least as many tiles as SMs: whole tiles per CTA
               # after the stream-K share of the leftover tiles
               (4, 32000, 256), (16, 20480, 512), (2, 39040, 1040),
               # wide tiles, ragged in every dimension, several rounds
               (300, 40000, 320), (512, 32000, 512),
               # few wide tiles with a long K: 256-wide tiles in four K slices
               (300, 1024, 9000),
               # a few hundred rows (a batched decode step): the O and down
               # projections in K slices whose CTAs share the sum, a ragged
               # width, 1024 rows in three K slices, a single K step, a ragged
               # width in K slices; 256-row items under (512, 32000, 512) above
               (512, 4096, 4096), (512, 4096, 14336), (768, 1300, 600), (1024, 640, 1000), (512, 200, 64),
               (512, 3000, 4096)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_bf16_tensor_core(M, N, K):
    rng = np.random.default_rng(M * 7 + N + K)
    X = synth.bf16_round(rng.standard_normal((M, K), dtype=np.float32))
    W = synth.bf16_round(rng.standard_normal((N, K), dtype=np.float32))
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    m = pe()
    Xd = torch.from_numpy(X).to(torch.bfloat16).cuda()
    Wd = torch.from_numpy(W).to(torch.bfloat16).cuda()
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    nb = m.peagle_gemm_workspace_size(m.PEAGLE_BF16, M, N, K)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    m.peagle_gemm(m.PEAGLE_BF16, M, N, K, Xd, Wd, D, ws, ws.numel())
    torch.cuda.synchronize()
    err = H().max_abs_rel(D.cpu().numpy(), ref)
    assert err < 1e-5, err


@pytest.mark.parametrize("M,N,K", [(1, 70, 33), (5, 64, 64), (65, 130, 100)])
def test_gemm_f32_cuda_core(M, N, K):
    rng = np.random.default_rng(M + N + K)
    X = rng.standard_normal((M, K), dtype=np.float32)
    W = rng.standard_normal((N, K), dtype=np.float32)
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    m = pe()
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    m.peagle_gemm(m.PEAGLE_F32, M, N, K, torch.from_numpy(X).cuda(), torch.from_numpy(W).cuda(), D,
                  None, 0)
    torch.cuda.synchronize()
    assert H().max_abs_rel(D.cpu().numpy(), ref) < 1e-6


# ---------------------------------------------------------------- verify
def test_verify_accept_exhaustive_and_random():
    import itertools
    V, K = 3, 3
    d, t = [], []
    for dd in itertools.product(range(V), repeat=K):
        for tt in itertools.product(range(V), repeat=K + 1):
            d.append(dd)
            t.append(tt)
    d = np.array(d, dtype=np.int32)
    t = np.array(t, dtype=np.int32)
    a, n = H().run_verify(d, t)
    ra, rn = O.verify_accept(d, t)
    assert np.array_equal(a, ra) and np.array_equal(n, rn)
    rng = np.random.default_rng(1)
    for B, K in ((1, 1), (64, 8), (1000, 16), (7, 64)):
        d = rng.integers(0, 4, (B, K)).astype(np.int32)
        t = rng.integers(0, 4, (B, K + 1)).astype(np.int32)
        match = rng.random((B, K)) < 0.6
        tk = t[:, :K]
        tk[match] = d[match]
        a, n = H().run_verify(d, t)
        ra, rn = O.verify_accept(d, t)
        assert np.array_equal(a, ra) and np.array_equal(n, rn)


# ------------------------------------------------------------------- COD
@pytest.mark.parametrize("n,K,r,rmin,seed", [(1, 3, 0.7, 0.2, 5), (7, 4, 0.7, 0.2, 1),
                                             (1000, 8, 0.7, 0.2, 42), (4096, 4, 0.7, 0.2, 7),
                                             (32768, 8, 0.7, 0.2, 0x5EED04D7), (5000, 16, 0.9, 0.05, 3),
                                             (2048, 3, 1.0, 1.0, 9), (100003, 5, 0.6, 0.3, 2**63 + 5)])
def test_cod_select_bit_exact(n, K, r, rmin, seed):
    m = pe()
    counts = m.peagle_cod_counts(n, K, r, rmin)
    R = sum(counts)
    idx = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    row_of = torch.full((K * n,), -7, dtype=torch.int32, device="cuda")
    got_counts = m.peagle_cod_select(n, K, r, rmin, seed, idx, row_of)
    torch.cuda.synchronize()
    rc, sets = O.cod_select(n, K, r, rmin, seed)
    assert got_counts == rc
    want = np.concatenate(sets).astype(np.int32)
    assert np.array_equal(idx.cpu().numpy(), want)
    ro = row_of.cpu().numpy().reshape(K, n)
    off = np.concatenate([[0], np.cumsum(rc)])
    for d in range(K):
        w = np.full(n, -1, dtype=np.int64)
        w[sets[d]] = off[d] + np.arange(len(sets[d]))
        assert np.array_equal(ro[d], w)


# ---------------------------------------------------------------- decode
def small_bf16_decode(**kw):
    wl = synth.WORKLOADS["decode_b64_ragged_k8"].scaled(
        hidden=256, target_hidden=128, num_aux=3, num_layers=2, num_q_heads=4, num_kv_heads=2,
        head_dim=64, intermediate=512, vocab=1000, K=4, batch=5, kv_len_range=(0, 300),
        max_position=2048, seed=501)
    return wl.scaled(**kw) if kw else wl


def check_decode(wl, got, ref, tol, d2t=None):
    err = H().max_abs_rel(got["logits"], ref["logits"])
    assert err <= tol, f"logits max-abs-rel {err:.3e} > {tol}"
    # every GPU token is (the target id of) the argmax of the GPU's own logits
    own = np.argmax(got["logits"], axis=-1)
    assert np.array_equal(got["draft_tokens"], own if d2t is None else np.asarray(d2t)[own])
    if tol <= F32_TOL:
        assert np.array_equal(got["draft_tokens"], ref["draft_tokens"])
    else:
        bad = H().token_mismatches_explained(got["draft_tokens"], ref["logits"], d2t=d2t)
        assert not bad, bad
    return err


def test_decode_tiny_f32():
    wl = synth.WORKLOADS["tiny_f32_decode"]
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl)
    model = H().make_model(wl, W)
    got = H().run_decode(wl, model, inp, want_logits=True)
    ref = H().oracle_decode(wl, W, inp)
    check_decode(wl, got, ref, F32_TOL)
    assert pe().peagle_get_device_status(model.handle) == 0


@pytest.mark.parametrize("kw", [dict(), dict(batch=80, K=3), dict(num_layers=1, K=1),
                                dict(kv_len_range=(0, 0)), dict(batch=1, K=16, kv_len_range=(700, 700)),
                                dict(intermediate=200),
                                # head tiles whole in one CTA (register argmax path), mixed with split ones
                                dict(vocab=24000, batch=2, K=8), dict(vocab=40000, hidden=512, batch=1),
                                # 320 rows: wide head tiles with the fused argmax
                                dict(vocab=40000, batch=40, K=8),
                                # head dim 128, chunks of 512-1024 keys (32 and 6 query rows per
                                # KV head, chunks past the context end, ragged last tiles)
                                dict(head_dim=128, num_q_heads=8, num_kv_heads=2, hidden=1024, batch=12, K=8,
                                     kv_len_range=(0, 4000), max_position=8192),
                                dict(head_dim=128, num_q_heads=4, num_kv_heads=2, hidden=512, batch=9, K=3,
                                     kv_len_range=(200, 2600), max_position=8192),
                                # 512 rows in 256-row items: fused SwiGLU (96 of 192 columns gate,
                                # the last tile ragged) and the argmax head over a ragged vocab
                                dict(batch=64, K=8, vocab=5000, intermediate=640),
                                # a wide gated SwiGLU over 512 rows (two rounds of 256-wide
                                # tiles) and the down projection in K slices sharing their sum
                                dict(batch=64, K=8, intermediate=6144)])
def test_decode_bf16_small(kw):
    wl = small_bf16_decode(**kw)
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl)
    model = H().make_model(wl, W)
    got = H().run_decode(wl, model, inp, want_logits=True)
    ref = H().oracle_decode(wl, W, inp)
    check_decode(wl, got, ref, BF16_TOL)
    assert pe().peagle_get_device_status(model.handle) == 0


def test_decode_f32_multilayer_gqa_append():
    wl = small_bf16_decode(dtype="f32", batch=3, kv_len_range=(1, 40))
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl)
    model = H().make_model(wl, W)
    got = H().run_decode(wl, model, inp, want_logits=True, append=True)
    ref = H().oracle_decode(wl, W, inp, append=True)
    check_decode(wl, got, ref, F32_TOL)
    d = got["dev"]
    for l in range(wl.num_layers):
        kc = d["k_cache"][l].cpu().numpy()
        vc = d["v_cache"][l].cpu().numpy()
        for b in range(wl.batch):
            row = int(inp["kv_offsets"][b] + inp["kv_lens"][b])
            rk, rv = ref["appended"][l][b]
            assert H().max_abs_rel(kc[row], rk) <= F32_TOL
            assert H().max_abs_rel(vc[row], rv) <= F32_TOL


@pytest.mark.parametrize("kw", [dict(batch=2, K=4), dict(batch=1, K=3, head_dim=128, hidden=512)])
def test_decode_bf16_few_rows_append(kw):
    # few bf16 decode rows over two layers: rotary q/k, the anchor rows'
    # k/v appended to their context slots, the layer-0 residual seed
    wl = small_bf16_decode(kv_len_range=(1, 40), **kw)
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl)
    model = H().make_model(wl, W)
    got = H().run_decode(wl, model, inp, want_logits=True, append=True)
    ref = H().oracle_decode(wl, W, inp, append=True)
    check_decode(wl, got, ref, BF16_TOL)
    d = got["dev"]
    for l in range(wl.num_layers):
        kc = d["k_cache"][l].float().cpu().numpy()
        vc = d["v_cache"][l].float().cpu().numpy()
        for b in range(wl.batch):
            row = int(inp["kv_offsets"][b] + inp["kv_lens"][b])
            rk, rv = ref["appended"][l][b]
            assert H().max_abs_rel(kc[row], rk) <= BF16_TOL
            assert H().max_abs_rel(vc[row], rv) <= BF16_TOL
    assert pe().peagle_get_device_status(model.handle) == 0


def draft_vocab_maps(V, Vd, seed):
    """A draft vocab of Vd target ids (sorted): d2t[j] = target id of draft
    id j; t2d[t] = j, or -1 for target ids outside the draft vocab."""
    d2t = np.sort(np.random.default_rng(seed).choice(V, Vd, replace=False)).astype(np.int32)
    t2d = np.full(V, -1, dtype=np.int32)
    t2d[d2t] = np.arange(Vd, dtype=np.int32)
    return d2t, t2d


@pytest.mark.parametrize("dtype,tol", [("f32", F32_TOL), ("bf16", BF16_TOL)])
def test_decode_draft_vocab_smaller_than_target_vocab(dtype, tol):
    # the head projects onto a 600-id draft vocab and every token comes back
    # as the target id d2t[argmax] ("feat(speculative) ... #2376", Changelog:
    # the draft-vocab projection)
    wl = small_bf16_decode(dtype=dtype, batch=7)
    W = synth.make_weights(wl)
    Vd = 600
    d2t, t2d = draft_vocab_maps(wl.vocab, Vd, 31)
    W = dict(W, lm_head_w=W["lm_head_w"][:Vd].copy(), d2t=d2t, t2d=t2d)
    inp = synth.make_decode_inputs(wl)
    model = H().make_model(wl, W)
    got = H().run_decode(wl, model, inp, want_logits=True)
    ref = H().oracle_decode(wl, W, inp)
    assert got["logits"].shape[-1] == Vd
    check_decode(wl, got, ref, tol, d2t=d2t)
    assert np.isin(got["draft_tokens"], d2t).all()
    assert pe().peagle_get_device_status(model.handle) == 0


@pytest.mark.parametrize("dtype,tol", [("f32", F32_TOL), ("bf16", BF16_TOL)])
def test_decode_without_norm_before_residual(dtype, tol):
    # --no-norm-before-residual ("P-EAGLE" user guide, Key Parameters): the
    # layer-0 residual is the fc-projected hidden state itself, for the anchor
    # rows and for the masked rows' shared constant alike
    wl = small_bf16_decode(dtype=dtype, batch=4)
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl)
    model = H().make_model(wl, W, norm_before_residual=0)
    got = H().run_decode(wl, model, inp, want_logits=True, append=True)
    ref = H().oracle_decode(wl, W, inp, append=True, norm_before_residual=False)
    err = check_decode(wl, got, ref, tol)
    # the flag is seen: the GPU sits far closer to the flag-off oracle than
    # the flag-on oracle does
    on = H().oracle_decode(wl, W, inp)
    assert err < 0.25 * H().max_abs_rel(on["logits"], ref["logits"])
    assert pe().peagle_get_device_status(model.handle) == 0


def test_decode_prefix_consistency_on_gpu():
    wl = small_bf16_decode(dtype="f32", batch=2)
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl)
    model = H().make_model(wl, W)
    full = H().run_decode(wl, model, inp, want_logits=True, K=4)
    part = H().run_decode(wl, model, inp, want_logits=True, K=2)
    assert H().max_abs_rel(part["logits"], full["logits"][:, :2]) < 1e-5


def test_decode_flags_out_of_range_token():
    wl = synth.WORKLOADS["tiny_f32_decode"]
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl)
    inp["anchor_tokens"] = np.array([wl.vocab + 5], dtype=np.int32)
    model = H().make_model(wl, W)
    H().run_decode(wl, model, inp)
    assert pe().peagle_get_device_status(model.handle) & pe().PEAGLE_DEV_BOUNDS
    pe().peagle_clear_device_status(model.handle)
    assert pe().peagle_get_device_status(model.handle) == 0


@pytest.mark.parametrize("kw", [dict(),
                                # tcgen05 contractions, 2-CTA multicast pairs, chunked attention
                                dict(head_dim=128, num_q_heads=8, num_kv_heads=2, hidden=1024, batch=40,
                                     K=8, vocab=40000, kv_len_range=(0, 4000), max_position=8192)])
def test_decode_step_replays_as_cuda_graph(kw):
    # the draft step + verify, captured once as a CUDA graph: replays give
    # the eager step's tokens and logits bit for bit, and read the inputs'
    # current contents (nothing host-side is frozen into the graph but
    # pointers and sizes)
    import torch
    wl = small_bf16_decode(**kw)
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl)
    model = H().make_model(wl, W)
    d = H().upload_decode(wl, inp)
    B, K, Vd = wl.batch, wl.K, model.cfg.draft_vocab
    max_kv = int(np.max(inp["kv_lens"]))
    cap = int(inp["kv_capacity"])
    rng = np.random.default_rng(77)
    targets = torch.from_numpy(rng.integers(0, wl.vocab, (B, K)).astype(np.int32)).cuda()
    dev = dict(device="cuda")

    def step(toks, logits, acc, nxt, stream=None):
        model.draft_step(K, d["aux"], d["anchor_tokens"], d["anchor_pos"], d["k_cache"], d["v_cache"],
                         d["kv_offsets"], d["kv_lens"], cap, max_kv, False, draft_tokens=toks,
                         logits=logits, stream=stream)
        pe().peagle_verify_accept(B, K, toks, targets, acc, nxt, stream=stream)

    def bufs():
        return (torch.empty((B, K), dtype=torch.int32, **dev), torch.empty((B, K, Vd), dtype=torch.float32, **dev),
                torch.empty(B, dtype=torch.int32, **dev), torch.empty(B, dtype=torch.int32, **dev))

    def host(b):
        return [x.cpu().numpy() for x in b]

    eager = bufs()
    step(*eager)
    torch.cuda.synchronize()
    want = host(eager)

    g = torch.cuda.CUDAGraph()
    gb = bufs()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(*gb, stream=torch.cuda.current_stream())
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for x in gb:
        x.fill_(-7)
    with torch.cuda.graph(g):
        step(*gb, stream=torch.cuda.current_stream())
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(host(gb), want):
        assert np.array_equal(a, b)

    # new anchors and aux rows in place: the replay follows them
    d["anchor_tokens"].copy_(torch.from_numpy(rng.integers(0, wl.vocab, B).astype(np.int32)))
    d["aux"].mul_(-0.5)
    g.replay()
    step(*eager)
    torch.cuda.synchronize()
    got, want2 = host(gb), host(eager)
    for a, b in zip(got, want2):
        assert np.array_equal(a, b)
    assert not np.array_equal(got[1], want[1])
    assert pe().peagle_get_device_status(model.handle) == 0


def test_closed_loop_with_stochastic_verification_matches_the_oracle():
    # three rounds of draft -> rejection-sampling verify -> next context: the
    # drafter is greedy, so its distribution q is one-hot at each draft; the
    # target's p is a random softmax; uniforms and draws are seeded. GPU and
    # oracle see the same inputs and must agree on every integer
    from eagle_speculative_drafting_gb300.loop import DraftLoop
    wl = small_bf16_decode(dtype="f32", batch=5, K=4, kv_len_range=(3, 40))
    W = synth.make_weights(wl)
    T = 3
    inp = synth.make_decode_inputs(wl, spare=T * (wl.K + 1))
    model = H().make_model(wl, W)
    om = H().oracle_model(wl, W)
    d = H().upload_decode(wl, inp)
    B, K, V = wl.batch, wl.K, wl.vocab
    loop = DraftLoop(model, K, d["k_cache"], d["v_cache"], d["kv_offsets"], d["kv_lens"], inp["kv_capacity"])
    loop.start(inp["anchor_tokens"], inp["kv_lens"].copy())
    kc = [k.copy() for k in inp["k_cache"]]
    vc = [v.copy() for v in inp["v_cache"]]
    lens = inp["kv_lens"].astype(np.int64).copy()
    rtok = [[int(t)] for t in inp["anchor_tokens"]]
    rpos = [[int(p)] for p in inp["kv_lens"]]
    rng = np.random.default_rng(2024)
    accepted = []
    for t in range(T):
        goff = loop.new_offsets.cpu().numpy()
        aux_rows = np.stack([_target_aux(wl, b, p) for b in range(B) for p in rpos[b]])
        drafts = loop.draft(H().dev(aux_rows)).cpu().numpy()
        ref = O.draft_step_ctx(om, [aux_rows[goff[b]:goff[b + 1]] for b in range(B)], rtok, rpos, kc, vc,
                               inp["kv_offsets"], lens, K)
        assert np.array_equal(drafts, ref["draft_tokens"]), t
        for b in range(B):
            o = int(inp["kv_offsets"][b] + lens[b])
            for l in range(wl.num_layers):
                k, v = ref["appended"][l][b]
                kc[l][o:o + len(k)] = k
                vc[l][o:o + len(v)] = v
        q = np.eye(V, dtype=np.float32)[drafts]
        p = _softmax32(rng.standard_normal((B, K + 1, V)) * 2.0)
        # make acceptance likely for some drafts: raise p at the draft token
        for b in range(B):
            for i in range(K):
                if (b + i + t) % 3:
                    p[b, i, drafts[b, i]] += 4.0
        p /= p.sum(-1, keepdims=True)
        u = rng.random((B, K)).astype(np.float32)
        draws = rng.integers(0, 2 ** 32, B, dtype=np.uint64)
        a, nx = run_verify_sample(drafts, q, p, u, draws)
        ra, rn = O.verify_sample(drafts, q, p, u, draws)
        assert np.array_equal(a, ra) and np.array_equal(nx, rn), t
        accepted.append(a.copy())
        loop.advance_after(torch.from_numpy(a).cuda(), torch.from_numpy(nx).cuda())
        anchor = [pp[-1] for pp in rpos]
        lens += np.array([len(pp) for pp in rpos])
        rtok, rpos = O.next_context(ref["draft_tokens"], ra, rn, anchor)
        assert np.array_equal(loop.kv_lens.cpu().numpy(), lens)
        gtok = loop.new_tokens.cpu().numpy()
        goff = loop.new_offsets.cpu().numpy()
        assert [list(gtok[goff[b]:goff[b + 1]]) for b in range(B)] == rtok
    assert np.concatenate(accepted).max() > 0   # some drafts were kept
    assert pe().peagle_get_device_status(model.handle) == 0


def test_empty_calls_succeed_and_launch_nothing():
    # no requests, no rows, no bytes: each call returns PEAGLE_OK without a
    # kernel launch (the library's launch counter does not move)
    import torch
    m = pe()
    wl = synth.WORKLOADS["tiny_f32_decode"]
    model = H().make_model(wl, synth.make_weights(wl))
    cache = [torch.zeros((1, wl.num_kv_heads, wl.head_dim), device="cuda") for _ in range(wl.num_layers)]
    torch.cuda.synchronize()
    n0 = m.peagle_kernel_launches()
    m.peagle_draft_step(model.handle, 0, wl.K, None, None, None, cache, cache, None, None, 1, 0, 0, None, None,
                        None, 0)
    m.peagle_verify_accept(0, wl.K, None, None, None, None)
    D = torch.empty((0, 16), device="cuda")
    m.peagle_gemm(m.PEAGLE_BF16, 0, 16, 64, D, D, D, None, 0)
    m.peagle_copy_to_device(D, D, 0)
    m.peagle_copy_to_host(D, D, 0)
    torch.cuda.synchronize()
    assert m.peagle_kernel_launches() == n0
    assert m.peagle_get_device_status(model.handle) == 0


def test_staging_copies_through_mapped_host_memory():
    # the copies in the launch chain: vector and byte paths, both directions,
    # offsets off the 16-byte grid; memory the device cannot reach as host
    # memory (pageable, or device memory) is refused before any launch
    import torch
    m = pe()
    g = torch.Generator().manual_seed(3)
    for nbytes, off in ((16, 0), (1576464, 0), (1000003, 0), (4104, 8), (77, 5)):
        src = torch.randint(0, 256, (nbytes + off,), dtype=torch.uint8, generator=g).pin_memory()
        dev = torch.zeros(nbytes + off, dtype=torch.uint8, device="cuda")
        back = torch.zeros(nbytes + off, dtype=torch.uint8).pin_memory()
        m.peagle_copy_to_device(dev.data_ptr() + off, src.data_ptr() + off, nbytes)
        m.peagle_copy_to_host(back.data_ptr() + off, dev.data_ptr() + off, nbytes)
        torch.cuda.synchronize()
        assert torch.equal(dev.cpu()[off:], src[off:]) and torch.equal(back[off:], src[off:])
        assert not dev.cpu()[:off].any() and not back[:off].any()
    m.peagle_copy_to_device(dev, src, 0)
    pageable = torch.zeros(64, dtype=torch.uint8)
    d64 = torch.zeros(64, dtype=torch.uint8, device="cuda")
    for bad in (pageable, torch.zeros(64, dtype=torch.uint8, device="cuda")):
        with pytest.raises(m.PeagleError):
            m.peagle_copy_to_device(d64, bad, 64)
        with pytest.raises(m.PeagleError):
            m.peagle_copy_to_host(bad, d64, 64)
    torch.cuda.synchronize()


def test_draft_step_with_staged_inputs_and_outputs():
    # inputs staged in from page-locked host memory, the step and greedy
    # verify, the results staged out: the plain step's tokens, bit for bit
    import torch
    wl = small_bf16_decode(batch=12, K=4)
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl)
    model = H().make_model(wl, W)
    d = H().upload_decode(wl, inp)
    B, K = wl.batch, wl.K
    cap, max_kv = int(inp["kv_capacity"]), int(np.max(inp["kv_lens"]))
    want = H().run_decode(wl, model, inp, d=d)["draft_tokens"]
    aux_h = d["aux"].cpu().pin_memory()
    tok_h = d["anchor_tokens"].cpu().pin_memory()
    aux_d, tok_d = torch.empty_like(d["aux"]), torch.empty_like(d["anchor_tokens"])
    toks = torch.empty((B, K), dtype=torch.int32, device="cuda")
    toks_h = torch.full((B, K), -1, dtype=torch.int32).pin_memory()
    m = pe()
    m.peagle_copy_to_device(aux_d, aux_h, aux_h.numel() * aux_h.element_size())
    m.peagle_copy_to_device(tok_d, tok_h, tok_h.numel() * 4)
    model.draft_step(K, aux_d, tok_d, d["anchor_pos"], d["k_cache"], d["v_cache"], d["kv_offsets"],
                     d["kv_lens"], cap, max_kv, False, draft_tokens=toks)
    m.peagle_copy_to_host(toks_h, toks, B * K * 4)
    torch.cuda.synchronize()
    assert np.array_equal(toks_h.numpy(), want)
    assert m.peagle_get_device_status(model.handle) == 0


# -------------------------------------------------------------- training
def small_train(dtype="f32", n=64, lens=(20, 1, 30, 13), K=4, **kw):
    wl = small_bf16_decode(dtype=dtype, kind="train", n_tokens=n, K=K, **kw)
    rng = np.random.default_rng(n + K)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    assert cu[-1] == n
    pos = np.concatenate([np.arange(l) for l in lens]).astype(np.int32)
    aux = rng.standard_normal((n, wl.num_aux * wl.target_hidden)).astype(np.float32)
    if dtype == "bf16":
        aux = synth.bf16_round(aux)
    inp = dict(aux=aux, input_ids=rng.integers(0, wl.vocab, n), position_ids=pos, cu_seqlens=cu,
               labels=rng.integers(0, wl.vocab, n), loss_mask=None)
    return wl, inp


def check_train(wl, inp, K, r, rmin, seed, tol, W=None, norm_before_residual=True):
    W = synth.make_weights(wl) if W is None else W
    model = H().make_model(wl, W, norm_before_residual=int(norm_before_residual))
    got = H().run_train(wl, model, inp, K, r, rmin, seed, want_logits=True)
    ref = O.parallel_forward(H().oracle_model(wl, W, norm_before_residual), **inp, K=K, r=r, r_min=rmin,
                             seed=seed)
    assert got["counts"] == ref["counts"]
    assert H().max_abs_rel(got["logits"], ref["logits"]) <= tol
    assert np.array_equal(got["per_depth_valid"], ref["per_depth_valid"])
    assert H().max_abs_rel(got["per_depth_loss"], ref["per_depth_loss"]) <= tol
    assert abs(float(got["loss"][0]) - ref["loss"]) <= tol * max(1.0, abs(ref["loss"]))
    lab = ref["row_label"] >= 0
    assert np.all(np.isnan(got["row_ce"][~lab]))
    assert H().max_abs_rel(got["row_ce"][lab], ref["row_ce"][lab]) <= tol
    assert np.array_equal(got["row_argmax"], np.argmax(got["logits"], -1))
    if tol <= F32_TOL:
        assert np.array_equal(got["row_argmax"], ref["row_argmax"])
        assert np.allclose(got["per_depth_acc"], ref["per_depth_acc"], atol=1e-6)
    else:
        assert not H().token_mismatches_explained(got["row_argmax"], ref["logits"])
    assert pe().peagle_get_device_status(model.handle) == 0
    return got, ref


def test_train_tiny_f32():
    wl, inp = small_train()
    check_train(wl, inp, 4, 0.7, 0.2, 11, F32_TOL)


def test_train_f32_all_rows_and_loss_mask():
    wl, inp = small_train(n=50, lens=(50,), K=3)
    inp["loss_mask"] = (np.arange(50) % 3 != 0).astype(np.uint8)
    check_train(wl, inp, 3, 1.0, 1.0, 2, F32_TOL)


def test_train_bf16_small():
    wl, inp = small_train(dtype="bf16", n=300, lens=(120, 7, 100, 73), K=5)
    check_train(wl, inp, 5, 0.7, 0.2, 99, BF16_TOL)


def test_train_bf16_swapped_rows():
    # at most 128 rows: every GEMM runs swapped, so the cross-entropy
    # statistics come from the swapped epilogue
    wl, inp = small_train(dtype="bf16", n=60, lens=(35, 25), K=2)
    check_train(wl, inp, 2, 0.7, 0.2, 8, BF16_TOL)


def test_train_bf16_rows_between_the_plans():
    # 170 rows: wide tiles of the few-hundred-row planner under the
    # cross-entropy head
    wl, inp = small_train(dtype="bf16", n=100, lens=(60, 40), K=2)
    check_train(wl, inp, 2, 0.7, 0.2, 8, BF16_TOL)


@pytest.mark.parametrize("n,lens,K", [(300, (120, 7, 100, 73), 5), (300, (70, 230), 3), (100, (60, 40), 2),
                                     (700, (300, 400), 2)])
def test_train_bf16_hd128_tensor_core_attention(n, lens, K):
    # head_dim 128 routes the training attention through the tcgen05 kernel:
    # several 128-key tiles, conversation starts off the 64-key grid, chain
    # keys up to depth 4, and one or several 128-row query tiles per depth
    wl, inp = small_train(dtype="bf16", n=n, lens=lens, K=K, head_dim=128)
    check_train(wl, inp, K, 0.7, 0.2, 13, BF16_TOL)


def test_train_bf16_unfused_swiglu_width():
    # 2I not a multiple of 256: the SwiGLU runs as its own kernel
    wl, inp = small_train(dtype="bf16", n=300, lens=(120, 180), K=3, intermediate=200)
    check_train(wl, inp, 3, 0.7, 0.2, 4, BF16_TOL)


@pytest.mark.parametrize("n,lens,kw", [(512, (200, 312), dict(vocab=32000)), (768, (500, 268), {}),
                                      (512, (300, 212), dict(head_dim=128)),
                                      (512, (200, 312), dict(hidden=2048, intermediate=512))])
def test_train_bf16_two_block_items(n, lens, kw):
    # depth 0 only: every contraction of the forward has 512 or 768 rows, the
    # plans of a batched decode step: 256-row items under the cross-entropy
    # head (32000 columns), and with a long K (hidden 2048) K slices whose
    # CTAs share the tile's sum before the cross-entropy / SwiGLU step
    wl, inp = small_train(dtype="bf16", n=n, lens=lens, K=1, **kw)
    check_train(wl, inp, 1, 0.7, 0.2, 17, BF16_TOL)


def test_backward_bf16_two_block_items():
    # 512 rows: the forward and backward contractions over them in 256-row items
    wl, inp = small_train(dtype="bf16", n=512, lens=(200, 312), K=1)
    check_backward(wl, inp, 1, 0.7, 0.2, 17, BF16_TOL)


def test_train_bf16_multi_chunk_rows():
    # more than 256 rows per GEMM so the wide (non-swapped) tensor-core tiles run
    wl, inp = small_train(dtype="bf16", n=700, lens=(300, 400), K=2)
    check_train(wl, inp, 2, 0.7, 0.2, 5, BF16_TOL)


@pytest.mark.parametrize("dtype,tol", [("f32", F32_TOL), ("bf16", BF16_TOL)])
def test_train_labels_outside_the_draft_vocab(dtype, tol):
    # labels are target ids; t2d maps them into the 600-id draft vocab, and a
    # label with t2d = -1 has no draft id, so its row carries no loss
    # ("feat(speculative) ... #2376", Pre checks: out-of-draft-vocab masking)
    wl, inp = small_train(dtype=dtype, n=300, lens=(120, 7, 100, 73), K=4)
    W = synth.make_weights(wl)
    Vd = 600
    d2t, t2d = draft_vocab_maps(wl.vocab, Vd, 32)
    W = dict(W, lm_head_w=W["lm_head_w"][:Vd].copy(), d2t=d2t, t2d=t2d)
    got, ref = check_train(wl, inp, 4, 0.7, 0.2, 21, tol, W=W)
    # about 40% of the uniform labels fall outside the draft vocab
    lab_all, _ = O.row_labels(wl.n_tokens, 4, 0.7, 0.2, 21, inp["cu_seqlens"], inp["labels"])
    assert got["per_depth_valid"].sum() < 0.8 * (lab_all >= 0).sum()
    assert np.array_equal(got["per_depth_valid"], ref["per_depth_valid"])


@pytest.mark.parametrize("dtype,tol", [("f32", F32_TOL), ("bf16", BF16_TOL)])
def test_train_without_norm_before_residual(dtype, tol):
    wl, inp = small_train(dtype=dtype, n=300, lens=(120, 7, 100, 73), K=4)
    check_train(wl, inp, 4, 0.7, 0.2, 17, tol, norm_before_residual=False)


# ------------------------------------------------------------- checkpoint
def test_checkpoint_round_trip_gives_the_same_draft_step(tmp_path):
    # save the device weights in vLLM's P-EAGLE layout, load them into fresh
    # device buffers, and draft again: identical logits and tokens
    from eagle_speculative_drafting_gb300.model import load_checkpoint
    wl = small_bf16_decode(batch=3)
    W = synth.make_weights(wl)
    d2t, t2d = draft_vocab_maps(wl.vocab, 700, 5)
    W = dict(W, lm_head_w=W["lm_head_w"][:700].copy(), d2t=d2t, t2d=t2d)
    inp = synth.make_decode_inputs(wl)
    model = H().make_model(wl, W)
    a = H().run_decode(wl, model, inp, want_logits=True)
    model.save_checkpoint(str(tmp_path))
    model2 = load_checkpoint(str(tmp_path))
    assert model2.cfg.draft_vocab == 700 and model2.cfg.ptd_token_id == wl.ptd_token_id
    b = H().run_decode(wl, model2, inp, want_logits=True)
    assert np.array_equal(a["logits"], b["logits"])
    assert np.array_equal(a["draft_tokens"], b["draft_tokens"])
    assert np.array_equal(model2._keep["t2d"].cpu().numpy(), t2d)


# --------------------------------------------------- stochastic verification
def _softmax32(x):
    x = x - x.max(-1, keepdims=True)
    e = np.exp(x)
    return (e / e.sum(-1, keepdims=True)).astype(np.float32)


def run_verify_sample(drafts, q, p, u, draws):
    m = pe()
    B, K = drafts.shape
    V = p.shape[-1]
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dt).cuda()
    a = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    m.peagle_verify_sample(B, K, V, dev(drafts, torch.int32), dev(q, torch.float32), dev(p, torch.float32),
                           dev(u, torch.float32), dev(np.asarray(draws, np.uint32).view(np.int32), torch.int32), a, n)
    torch.cuda.synchronize()
    return a.cpu().numpy(), n.cpu().numpy()


@pytest.mark.parametrize("B,K,V,temp", [(64, 8, 32000, 1.0), (64, 8, 32000, 0.3), (5, 1, 3, 1.0),
                                        (300, 4, 7, 2.0), (3, 16, 1000, 0.05), (40, 64, 129, 1.0)])
def test_verify_sample_bit_exact(B, K, V, temp):
    rng = np.random.default_rng(B * 31 + K + V)
    # draft and target distributions from nearby logits, drafts drawn from q
    base = rng.standard_normal((B, K + 1, V)) * 3.0
    p = _softmax32((base + 0.5 * rng.standard_normal(base.shape)) / temp)
    q = _softmax32(base[:, :K] / temp)
    cdf = np.cumsum(q.astype(np.float64), -1)
    drafts = np.minimum((cdf > rng.random((B, K, 1))).argmax(-1), V - 1).astype(np.int32)
    u = rng.random((B, K)).astype(np.float32)
    draws = rng.integers(0, 2 ** 32, B, dtype=np.uint64)
    a, n = run_verify_sample(drafts, q, p, u, draws)
    ra, rn = O.verify_sample(drafts, q, p, u, draws)
    assert np.array_equal(a, ra) and np.array_equal(n, rn)
    assert 0 < a.mean() < K or K == 1
    assert pe().peagle_get_library_status() == 0


def test_verify_sample_edge_cases():
    rng = np.random.default_rng(2)
    B, K, V = 6, 3, 50
    # one-hot distributions: greedy verify, on the GPU as in the oracle
    d = rng.integers(0, V, (B, K)).astype(np.int32)
    t = rng.integers(0, V, (B, K + 1)).astype(np.int32)
    t[:3, :K] = d[:3]
    q = np.eye(V, dtype=np.float32)[d]
    p = np.eye(V, dtype=np.float32)[t]
    u = rng.random((B, K)).astype(np.float32)
    draws = rng.integers(0, 2 ** 32, B, dtype=np.uint64)
    a, n = run_verify_sample(d, q, p, u, draws)
    ga, gn = O.verify_accept(d, t)
    assert np.array_equal(a, ga) and np.array_equal(n, gn)
    # p == q, drafts of zero probability: rejected, empty residual -> argmax
    pz = np.full((B, K + 1, V), 0.0, np.float32)
    pz[..., 7] = 0.5
    pz[..., 9] = 0.5
    a, n = run_verify_sample(np.zeros((B, K), np.int32), pz[:, :K], pz, u, draws)
    assert (a == 0).all() and (n == 7).all()
    # NaN and out-of-[0,1] weights count as 0 / 1 on both sides
    pn = _softmax32(rng.standard_normal((B, K + 1, V)))
    pn[:, :, 3] = np.nan
    pn[:, :, 4] = 5.0
    qn = _softmax32(rng.standard_normal((B, K, V)))
    a, n = run_verify_sample(d, qn, pn, u, draws)
    ra, rn = O.verify_sample(d, qn, pn, u, draws)
    assert np.array_equal(a, ra) and np.array_equal(n, rn)
    # a draft id outside the vocab is a rejection and a bounds fault
    pe().peagle_clear_library_status()
    bad = d.copy()
    bad[0, 0] = V + 3
    a, n = run_verify_sample(bad, q, p, u, draws)
    assert a[0] == 0
    assert pe().peagle_get_library_status() & pe().PEAGLE_DEV_BOUNDS
    pe().peagle_clear_library_status()


# ------------------------------------------------------ data-parallel training
def test_data_parallel_forward_sums_two_sequences_like_the_oracle():
    # one process: two packed sequences accumulate their depth sums in one
    # buffer; the combined loss is the oracle's batch loss. A single sequence
    # combined reproduces the forward's own outputs exactly.
    from eagle_speculative_drafting_gb300 import dp
    wl, inp = small_train(dtype="bf16", n=300, lens=(120, 7, 100, 73), K=4)
    _, inp2 = small_train(dtype="bf16", n=200, lens=(150, 50), K=4)
    W = synth.make_weights(wl)
    model = H().make_model(wl, W)
    seqs = [(0, H().upload_train(wl, inp)), (1, H().upload_train(wl, inp2))]
    fwd = dp.DataParallelForward(model, 4, 0.7, 0.2, base_seed=77)
    out = {k: v.cpu().numpy() for k, v in fwd.step(seqs).items()}
    om = H().oracle_model(wl, W)
    ref = O.loss_from_depth_sums(sum(
        O.depth_sums(O.parallel_forward(om, **x, K=4, r=0.7, r_min=0.2, seed=dp.sequence_seed(77, i)), 4)
        for i, x in ((0, inp), (1, inp2))))
    assert np.array_equal(out["per_depth_valid"], ref["per_depth_valid"])
    assert H().max_abs_rel(out["per_depth_loss"], ref["per_depth_loss"]) <= BF16_TOL
    assert abs(float(out["loss"][0]) - ref["loss"]) <= BF16_TOL * max(1.0, ref["loss"])
    one = {k: v.cpu().numpy() for k, v in dp.DataParallelForward(model, 4, 0.7, 0.2, 77).step(seqs[:1]).items()}
    direct = H().run_train(wl, model, inp, 4, 0.7, 0.2, dp.sequence_seed(77, 0))
    for k in ("per_depth_loss", "per_depth_acc", "per_depth_valid", "loss"):
        assert np.array_equal(one[k], direct[k]), k


# ------------------------------------------------- new context rows, closed loop
def _ctx_rows(wl, inp, counts, seed):
    rng = np.random.default_rng(seed)
    aux, tok, pos = [], [], []
    for b, n in enumerate(counts):
        a = rng.standard_normal((n, wl.num_aux * wl.target_hidden)).astype(np.float32)
        aux.append(synth.bf16_round(a) if wl.dtype == "bf16" else a)
        tok.append(rng.integers(0, wl.vocab, n).astype(np.int32))
        L = int(inp["kv_lens"][b])
        pos.append(np.arange(L, L + n, dtype=np.int32))
    return aux, tok, pos


@pytest.mark.parametrize("dtype,tol,kw", [("f32", F32_TOL, dict()), ("bf16", BF16_TOL, dict()),
                                          ("bf16", BF16_TOL, dict(head_dim=128, num_q_heads=8, num_kv_heads=2,
                                                                  hidden=1024, batch=6, K=8,
                                                                  kv_len_range=(0, 3000), max_position=8192)),
                                          # 8 query heads per KV head: up to 64 query rows per KV
                                          # head, two row groups sharing each key tile
                                          ("bf16", BF16_TOL, dict(head_dim=64, num_q_heads=16, num_kv_heads=2,
                                                                  hidden=1024, batch=6, K=4,
                                                                  kv_len_range=(0, 3000), max_position=8192))])
def test_draft_step_over_new_context_rows(dtype, tol, kw):
    # ragged new rows per request (1..9): causal among themselves over the
    # cached context, K/V appended, masked depths after the anchor
    wl = small_bf16_decode(dtype=dtype, **kw)
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl, spare=12)
    counts = [1 + (3 * b) % min(9, wl.K + 1) for b in range(wl.batch)]
    aux, tok, pos = _ctx_rows(wl, inp, counts, 4)
    model = H().make_model(wl, W)
    d = H().upload_decode(wl, inp)
    got = H().run_decode_ctx(wl, model, aux, tok, pos, d, inp["kv_lens"], inp["kv_capacity"],
                             int(np.max(inp["kv_lens"])), want_logits=True)
    ref = O.draft_step_ctx(H().oracle_model(wl, W), aux, tok, pos, inp["k_cache"], inp["v_cache"],
                           inp["kv_offsets"], inp["kv_lens"], wl.K)
    check_decode(wl, got, ref, tol)
    for l in range(wl.num_layers):
        kc = d["k_cache"][l].float().cpu().numpy()
        vc = d["v_cache"][l].float().cpu().numpy()
        for b in range(wl.batch):
            o = int(inp["kv_offsets"][b] + inp["kv_lens"][b])
            rk, rv = ref["appended"][l][b]
            assert H().max_abs_rel(kc[o:o + counts[b]], rk) <= tol
            assert H().max_abs_rel(vc[o:o + counts[b]], rv) <= tol
    assert pe().peagle_get_device_status(model.handle) == 0


def _target_aux(wl, b, p):
    # the synthetic target's aux hidden state of request b at position p
    a = np.random.default_rng([wl.seed, 77, b, int(p)]).standard_normal(wl.num_aux * wl.target_hidden)
    a = a.astype(np.float32)
    return synth.bf16_round(a) if wl.dtype == "bf16" else a


def test_closed_draft_verify_loop_matches_the_oracle():
    # four rounds of draft -> greedy verify -> next context on the GPU
    # (DraftLoop) and in the oracle: the same drafts, accept lengths, next
    # tokens and appended cache rows every round
    from eagle_speculative_drafting_gb300.loop import DraftLoop
    wl = small_bf16_decode(dtype="f32", batch=5, K=4, kv_len_range=(3, 40))
    W = synth.make_weights(wl)
    T = 4
    inp = synth.make_decode_inputs(wl, spare=T * (wl.K + 1))
    model = H().make_model(wl, W)
    om = H().oracle_model(wl, W)
    d = H().upload_decode(wl, inp)
    B, K = wl.batch, wl.K
    loop = DraftLoop(model, K, d["k_cache"], d["v_cache"], d["kv_offsets"], d["kv_lens"], inp["kv_capacity"])
    first_tok, first_pos = inp["anchor_tokens"], inp["kv_lens"].copy()
    loop.start(first_tok, first_pos)
    kc = [k.copy() for k in inp["k_cache"]]
    vc = [v.copy() for v in inp["v_cache"]]
    lens = inp["kv_lens"].astype(np.int64).copy()
    rtok = [[int(t)] for t in first_tok]
    rpos = [[int(p)] for p in first_pos]
    for t in range(T):
        # the target's aux states of this round's new rows, both sides
        gtok = loop.new_tokens.cpu().numpy()
        gpos = loop.new_pos.cpu().numpy()
        goff = loop.new_offsets.cpu().numpy()
        assert [list(gtok[goff[b]:goff[b + 1]]) for b in range(B)] == rtok
        assert [list(gpos[goff[b]:goff[b + 1]]) for b in range(B)] == rpos
        aux_rows = np.stack([_target_aux(wl, b, p) for b in range(B) for p in rpos[b]])
        drafts = loop.draft(H().dev(aux_rows)).cpu().numpy()
        ref = O.draft_step_ctx(om, [aux_rows[goff[b]:goff[b + 1]] for b in range(B)], rtok, rpos, kc, vc,
                               inp["kv_offsets"], lens, K)
        assert np.array_equal(drafts, ref["draft_tokens"]), t
        for b in range(B):   # the oracle's cache gains the new rows
            o = int(inp["kv_offsets"][b] + lens[b])
            for l in range(wl.num_layers):
                k, v = ref["appended"][l][b]
                kc[l][o:o + len(k)] = k
                vc[l][o:o + len(v)] = v
        acc_draw = synth.draw_accept_lengths(wl, B, K, salt=t)
        tgt = synth.make_targets_with_accept(wl, drafts, acc_draw, salt=t)
        a, nx = loop.verify_greedy(torch.from_numpy(tgt).cuda())
        ra, rn = O.verify_accept(ref["draft_tokens"], tgt)
        assert np.array_equal(a.cpu().numpy(), ra) and np.array_equal(nx.cpu().numpy(), rn)
        anchor = [p[-1] for p in rpos]
        lens += np.array([len(p) for p in rpos])
        rtok, rpos = O.next_context(ref["draft_tokens"], ra, rn, anchor)
        assert np.array_equal(loop.kv_lens.cpu().numpy(), lens)
    for l in range(wl.num_layers):
        g = d["k_cache"][l].cpu().numpy()
        for b in range(B):
            o = int(inp["kv_offsets"][b])
            assert H().max_abs_rel(g[o:o + lens[b]], kc[l][o:o + lens[b]]) <= F32_TOL
    assert pe().peagle_get_device_status(model.handle) == 0


# ------------------------------------------------------------------ backward
def _grad_pairs(got, ref):
    for k in O.GRAD_KEYS:
        yield k, got[k], ref[k]
    for l, (gl, rl) in enumerate(zip(got["layers"], ref["layers"])):
        for k, v in rl.items():
            yield f"layers.{l}.{k}", gl[k], v


def check_backward(wl, inp, K, r, rmin, seed, tol, W=None, nbr=True):
    W = synth.make_weights(wl) if W is None else W
    model = H().make_model(wl, W, norm_before_residual=int(nbr))
    d = H().upload_train(wl, inp)
    loss, g = model.parallel_backward(d["aux"], d["input_ids"], d["position_ids"], d["cu_seqlens"], d["labels"],
                                      K, r, rmin, seed, loss_mask=d["loss_mask"])
    torch.cuda.synchronize()
    got = {k: (v.cpu().numpy() if v is not None else None) for k, v in g.items() if k != "layers"}
    got["layers"] = [{k: (v.cpu().numpy() if v is not None else None) for k, v in L.items()} for L in g["layers"]]
    om = H().oracle_model(wl, W, nbr)
    ref_loss, ref = O.parallel_grads(om, **{k: inp[k] for k in ("aux", "input_ids", "position_ids", "cu_seqlens",
                                                                "labels", "loss_mask")}, K=K, r=r, r_min=rmin,
                                     seed=seed)
    assert abs(float(loss.item()) - ref_loss) <= tol * max(1.0, abs(ref_loss))
    worst = {}
    for name, a, b in _grad_pairs(got, ref):
        err = H().max_abs_rel(np.asarray(a).reshape(np.shape(b)), b)
        worst[name] = err
    assert max(worst.values()) <= tol, sorted(worst.items(), key=lambda kv: -kv[1])[:5]
    assert pe().peagle_get_device_status(model.handle) == 0
    return model, d, g, loss


@pytest.mark.parametrize("nbr", [True, False])
def test_backward_f32_matches_autograd(nbr):
    wl, inp = small_train()
    check_backward(wl, inp, 4, 0.7, 0.2, 11, F32_TOL, nbr=nbr)


def test_backward_bf16_matches_autograd():
    wl, inp = small_train(dtype="bf16", n=300, lens=(120, 7, 100, 73), K=4)
    check_backward(wl, inp, 4, 0.7, 0.2, 99, BF16_TOL)


def test_backward_bf16_hd128_gqa_long_conversations():
    # head dim 128, three query heads per KV head, K = 6: conversations span
    # several 64-key tiles of the tensor-core backward, with ragged tails
    wl, inp = small_train(dtype="bf16", n=700, lens=(300, 5, 129, 200, 66), K=6, hidden=384, num_q_heads=6,
                          num_kv_heads=2, head_dim=128)
    check_backward(wl, inp, 6, 0.7, 0.2, 21, BF16_TOL)


def test_backward_f32_draft_vocab_and_loss_mask():
    # a 600-id draft vocab (t2d = -1 labels carry no loss), a loss mask, and a
    # vocabulary width that is not a multiple of 8
    wl, inp = small_train(n=50, lens=(30, 20), K=3)
    W = synth.make_weights(wl)
    d2t, t2d = draft_vocab_maps(wl.vocab, 606, 8)
    W = dict(W, lm_head_w=W["lm_head_w"][:606].copy(), d2t=d2t, t2d=t2d)
    inp["loss_mask"] = (np.arange(50) % 4 != 1).astype(np.uint8)
    check_backward(wl, inp, 3, 0.7, 0.2, 5, F32_TOL, W=W)


def test_backward_step_lowers_the_loss():
    # one plain gradient step on the device weights lowers the forward loss
    wl, inp = small_train(dtype="bf16", n=300, lens=(120, 7, 100, 73), K=4)
    W = synth.make_weights(wl)
    model, d, g, loss0 = check_backward(wl, inp, 4, 0.7, 0.2, 3, BF16_TOL, W=W)
    lr = 0.5
    with torch.no_grad():
        for k in O.GRAD_KEYS:
            w = model._keep[k]
            w.copy_((w.float() - lr * g[k].reshape(w.shape)).to(w.dtype))
        for L, G in zip(model._keep["layers"], g["layers"]):
            for k, gv in G.items():
                if gv is not None and L.get(k) is not None:
                    L[k].copy_((L[k].float() - lr * gv).to(L[k].dtype))
    model2 = pe().Model(model.cfg, model._keep)   # the masked-row constants follow the new weights
    out = model2.parallel_forward(d["aux"], d["input_ids"], d["position_ids"], d["cu_seqlens"], d["labels"], 4, 0.7,
                                  0.2, 3)
    assert float(out["loss"].item()) < float(loss0.item()) - 1e-3
