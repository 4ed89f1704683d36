"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test ties one oracle function to something it cannot agree with by
construction: published test vectors, hand-worked values, closed forms,
brute-force enumerations, independent formulations (complex rotation for
RoPE, a plain EAGLE-3 step-0 forward, library cross-entropy) or invariants.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import synth
from oracle import peagle_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def tiny_workload(**kw):
    base = synth.WORKLOADS["tiny_f32_decode"].scaled(
        hidden=32, target_hidden=16, num_aux=3, num_layers=2, num_q_heads=4,
        num_kv_heads=2, head_dim=8, intermediate=48, vocab=64, K=4, batch=3,
        kv_len=0, kv_len_range=(3, 7), max_position=256, seed=77)
    return base.scaled(**kw) if kw else base


def tiny_model(wl, **cfg_over):
    W = synth.make_weights(wl)
    cfg = O.model_config(wl)
    cfg.update(cfg_over)
    return O.DraftModel(cfg, W), W


def tiny_train(n=23, S_lens=(9, 1, 13), K=4, seed=5, **kw):
    wl = tiny_workload(kind="train", n_tokens=n, K=K, **kw)
    model, W = tiny_model(wl)
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(S_lens)]).astype(np.int32)
    assert cu[-1] == n
    pos = np.concatenate([np.arange(l) for l in S_lens]).astype(np.int32)
    inp = dict(
        aux=rng.standard_normal((n, wl.num_aux * wl.target_hidden)),
        input_ids=rng.integers(0, wl.vocab, n), position_ids=pos, cu_seqlens=cu,
        labels=rng.integers(0, wl.vocab, n), loss_mask=None)
    return wl, model, W, inp


# ---------------------------------------------------------------- SplitMix64
def test_splitmix64_published_vectors():
    for line in open(os.path.join(GOLD, "splitmix64.txt")):
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        if f[0] == "first5":
            seed, want = int(f[1]), [int(x) for x in f[2:]]
            assert [int(x) for x in O.splitmix64(seed, len(want))] == want
        elif f[0] == "buckets":
            seed, cnt, want = int(f[1]), int(f[2]), [int(x) for x in f[3:]]
            z = O.splitmix64(seed, cnt)
            # floor(z * 5 / 2^64) exactly, in integers
            b = [(int(v) * 5) >> 64 for v in z]
            assert [b.count(i) for i in range(5)] == want


# ------------------------------------------------------------------------ COD
def test_cod_counts_hand_worked():
    seen = 0
    for line in open(os.path.join(GOLD, "cod_counts.txt")):
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        n, K, r, rmin = int(f[0]), int(f[1]), float(f[2]), float(f[3])
        assert O.cod_counts(n, K, r, rmin) == [int(x) for x in f[4:]]
        seen += 1
    assert seen == 4


@pytest.mark.parametrize("n,K,r,rmin,seed", [(4096, 4, 0.7, 0.2, 11), (1000, 8, 0.7, 0.2, 3),
                                             (17, 5, 0.9, 0.3, 0), (1, 3, 0.7, 0.2, 9),
                                             (0, 3, 0.7, 0.2, 9)])
def test_cod_sets_nested_sorted_sized(n, K, r, rmin, seed):
    counts, sets = O.cod_select(n, K, r, rmin, seed)
    assert len(sets) == K
    assert np.array_equal(sets[0], np.arange(n))
    for d in range(K):
        assert len(sets[d]) == counts[d]
        assert np.all(np.diff(sets[d]) > 0)
        if d:
            assert set(sets[d].tolist()) <= set(sets[d - 1].tolist())


def test_cod_sets_are_smallest_keys():
    # brute force: S_d is exactly the c_d positions of smallest key
    n, K = 50, 4
    counts, sets = O.cod_select(n, K, 0.7, 0.2, 1234)
    keys = [int(x) for x in O.splitmix64(1234, n)]
    for d in range(1, K):
        thr = sorted(keys)[counts[d] - 1]
        assert sets[d].tolist() == [i for i in range(n) if keys[i] <= thr]


def test_cod_inclusion_is_uniform():
    # over many seeds every position is kept at depth d with probability c_d/n
    n, K, trials = 40, 3, 2000
    hits = np.zeros((K, n))
    for s in range(trials):
        counts, sets = O.cod_select(n, K, 0.7, 0.2, 1000 + s)
        for d in range(K):
            hits[d, sets[d]] += 1
    for d in range(1, K):
        expect = trials * counts[d] / n
        chi2 = np.sum((hits[d] - expect) ** 2 / expect)
        # 39 degrees of freedom: P(chi2 > 80) < 1e-4 (hypergeometric cells
        # are slightly less spread than binomial, which only helps)
        assert chi2 < 80, chi2


# --------------------------------------------------------------------- verify
def test_verify_bruteforce_small_alphabet():
    # every draft/target pair over V=3, K=3 against os.path.commonprefix
    V, K = 3, 3
    import itertools
    drafts, targets = [], []
    for d in itertools.product(range(V), repeat=K):
        for t in itertools.product(range(V), repeat=K + 1):
            drafts.append(d)
            targets.append(t)
    drafts = np.array(drafts)
    targets = np.array(targets)
    acc, nxt = O.verify_accept(drafts, targets)
    for b in range(len(drafts)):
        a = len(os.path.commonprefix([list(drafts[b]), list(targets[b, :K])]))
        assert acc[b] == a and nxt[b] == targets[b, a]
    assert set(acc.tolist()) == set(range(K + 1))


# ------------------------------------------------------------ dense pieces
def test_rmsnorm_closed_form():
    g = np.array([1.0, 2.0, -0.5, 3.0])
    for c in (0.3, -2.0, 7.0):
        x = np.full(4, c)
        eps = 1e-5
        assert np.allclose(O.rms_norm(x, g, eps), g * c / math.sqrt(c * c + eps), rtol=0, atol=1e-15)
    x = np.array([3.0, 4.0])          # mean square 12.5
    assert np.allclose(O.rms_norm(x, np.ones(2), 0.0), x / math.sqrt(12.5), atol=1e-15)


def test_argmax_lowest_index_on_ties():
    rng = np.random.default_rng(0)
    for _ in range(200):
        x = rng.integers(-3, 3, size=rng.integers(1, 12)).astype(np.float64)
        m = max(x)
        first = next(i for i in range(len(x)) if x[i] == m)
        assert O.argmax_lowest(x[None])[0] == first
    assert O.argmax_lowest(np.array([[1.0, np.nan, 5.0, np.nan]]))[0] == 1


def test_logsumexp_and_silu():
    x = np.random.default_rng(1).standard_normal((5, 33)) * 30
    assert np.allclose(O.logsumexp(x), scipy.special.logsumexp(x, axis=-1), rtol=1e-13)
    z = np.linspace(-20, 20, 101)
    assert np.allclose(O.silu(z), z * scipy.special.expit(z), rtol=1e-13)


# ----------------------------------------------------------------------- RoPE
def _rope_complex(x, pos, theta):
    # independent formulation: pair (x_j, x_{j+hd/2}) as x_j + i x_{j+hd/2},
    # rotated by exp(i * pos * theta^(-2j/hd))
    hd = x.shape[-1]
    half = hd // 2
    z = x[..., :half] + 1j * x[..., half:]
    j = np.arange(half)
    w = np.exp(1j * np.outer(pos, [theta ** (-2.0 * t / hd) for t in j]))
    z = z * w[:, None, :]
    return np.concatenate([z.real, z.imag], axis=-1)


def test_rope_matches_complex_rotation_and_gathers_by_value():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((6, 3, 16))
    for pos in ([0, 1, 2, 3, 4, 5], [7, 3, 3, 100, 5000, 1], [40000, 0, 65535, 2, 9, 8]):
        pos = np.array(pos)
        assert np.allclose(O.apply_rope(x, pos, 5e5), _rope_complex(x, pos, 5e5), atol=1e-12)
    # position 0 is the identity
    assert np.allclose(O.apply_rope(x, np.zeros(6, int), 1e4), x, atol=0)


def test_rope_head_dim_two_is_plain_rotation():
    x = np.array([[[1.0, 0.0]], [[0.0, 1.0]], [[2.0, -1.0]]])
    pos = np.array([1, 2, 3])
    out = O.apply_rope(x, pos, 12345.0)
    for r in range(3):
        c, s = math.cos(pos[r]), math.sin(pos[r])
        a, b = x[r, 0]
        assert np.allclose(out[r, 0], [a * c - b * s, a * s + b * c], atol=1e-14)


def test_rope_gather_equals_contiguous_slice_and_shift():
    # arange positions = the leading slice of the table; offset positions
    # arange+d = the slice shifted by d; out-of-seq_len positions work
    S, hd, theta = 9, 8, 5e5
    cos_t, sin_t = O.rope_table(64, hd, theta)
    x = np.random.default_rng(3).standard_normal((S, 1, hd))
    half = hd // 2

    def by_slice(c, s):
        x1, x2 = x[..., :half], x[..., half:]
        return np.concatenate([x1 * c[:, None] - x2 * s[:, None], x2 * c[:, None] + x1 * s[:, None]], -1)

    assert np.allclose(O.apply_rope(x, np.arange(S), theta), by_slice(cos_t[:S], sin_t[:S]), atol=1e-14)
    for d in (1, 3, 40):
        assert np.allclose(O.apply_rope(x, np.arange(S) + d, theta),
                           by_slice(cos_t[d:S + d], sin_t[d:S + d]), atol=1e-14)


def test_rope_relative_position_invariance():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 1, 32))
    k = rng.standard_normal((1, 1, 32))
    base = None
    for p in (0, 5, 300, 9000):
        qa = O.apply_rope(q, np.array([p + 7]), 5e5)
        ka = O.apply_rope(k, np.array([p]), 5e5)
        dot = float(np.sum(qa * ka))
        base = dot if base is None else base
        assert abs(dot - base) < 1e-9


# ------------------------------------------------------------------ attention
def test_attention_one_hot_values_reveal_mask():
    # with q = 0 every allowed key has the same score, so v_j = one-hot(j)
    # returns 1/|allowed| exactly on the allowed keys
    rng = np.random.default_rng(5)
    Rq, Rk, nq, nkv = 7, 11, 4, 2
    allowed = rng.random((Rq, Rk)) < 0.5
    allowed[:, 0] = True
    q = np.zeros((Rq, nq, Rk))
    k = rng.standard_normal((Rk, nkv, Rk))
    v = np.tile(np.eye(Rk)[:, None, :], (1, nkv, 1))
    o = O.masked_attention(q, k, v, allowed)
    for h in range(nq):
        assert np.allclose(o[:, h, :], allowed / allowed.sum(1, keepdims=True), atol=1e-15)


def test_attention_gqa_equals_repeated_heads_and_softmax():
    rng = np.random.default_rng(6)
    Rq, Rk, nq, nkv, hd = 5, 9, 6, 2, 4
    q = rng.standard_normal((Rq, nq, hd))
    k = rng.standard_normal((Rk, nkv, hd))
    v = rng.standard_normal((Rk, nkv, hd))
    allowed = rng.random((Rq, Rk)) < 0.7
    allowed[:, -1] = True
    o = O.masked_attention(q, k, v, allowed)
    krep = np.repeat(k, nq // nkv, axis=1)
    vrep = np.repeat(v, nq // nkv, axis=1)
    assert np.allclose(o, O.masked_attention(q, krep, vrep, allowed), atol=1e-14)
    for r in range(Rq):
        for h in range(nq):
            s = np.array([q[r, h] @ k[j, h // 3] / 2.0 if allowed[r, j] else -np.inf for j in range(Rk)])
            p = scipy.special.softmax(s)
            assert np.allclose(o[r, h], p @ v[:, h // 3], atol=1e-13)


def test_decode_mask_hand_listed():
    # 2 context rows, K=3: depth d reads the context and chain rows 0..d
    m = O.decode_allowed(2, 3)
    want = [[1, 1, 1, 0, 0],
            [1, 1, 1, 1, 0],
            [1, 1, 1, 1, 1]]
    assert m.astype(int).tolist() == want


def test_train_mask_hand_listed():
    # conversation A = positions 0..2, conversation B = positions 3..4
    # rows: (0,0)(1,0)(2,0)(3,0)(4,0) | (1,1)(3,1) | (1,2)
    anchor = np.array([0, 1, 2, 3, 4, 1, 3, 1])
    depth = np.array([0, 0, 0, 0, 0, 1, 1, 2])
    start = np.array([0, 0, 0, 3, 3])
    m = O.train_allowed(anchor, depth, start).astype(int).tolist()
    want = [
        [1, 0, 0, 0, 0, 0, 0, 0],   # (0,0): itself
        [1, 1, 0, 0, 0, 0, 0, 0],   # (1,0): 0..1
        [1, 1, 1, 0, 0, 0, 0, 0],   # (2,0): 0..2
        [0, 0, 0, 1, 0, 0, 0, 0],   # (3,0): conversation B starts at 3
        [0, 0, 0, 1, 1, 0, 0, 0],   # (4,0)
        [1, 1, 0, 0, 0, 1, 0, 0],   # (1,1): context 0..1 + chain (1,1)
        [0, 0, 0, 1, 0, 0, 1, 0],   # (3,1): context 3 + chain (3,1)
        [1, 1, 0, 0, 0, 1, 0, 1],   # (1,2): context 0..1 + chain (1,1),(1,2)
    ]
    assert m == want


# ------------------------------------------------------------------ the model
def test_mask_hidden_shape():
    wl = synth.WORKLOADS["decode_b1_ctx2048_k4"].scaled(
        hidden=32, intermediate=64, vocab=128, num_q_heads=2, num_kv_heads=1, head_dim=16)
    W = synth.make_weights(wl)
    assert W["mask_hidden"].shape == (1, 3 * 4096) == (1, 12288)
    model = O.DraftModel(O.model_config(wl), W)
    assert model.mask_hidden.shape == (1, 12288)


def _decode_case(wl, model):
    inp = synth.make_decode_inputs(wl)
    return inp


def test_decode_structured_equals_dense_bruteforce():
    wl = tiny_workload()
    model, _ = tiny_model(wl)
    inp = synth.make_decode_inputs(wl)
    args = (inp["aux"], inp["anchor_tokens"], inp["anchor_pos"], inp["k_cache"], inp["v_cache"],
            inp["kv_offsets"], inp["kv_lens"], wl.K)
    a = O.draft_step(model, *args, append_anchor_kv=True)
    b = O.draft_step(model, *args, append_anchor_kv=True, dense_attention=True)
    assert np.allclose(a["logits"], b["logits"], atol=1e-12)
    assert np.array_equal(a["draft_tokens"], b["draft_tokens"])
    for l in range(wl.num_layers):
        for r in range(wl.batch):
            assert np.allclose(a["appended"][l][r][0], b["appended"][l][r][0], atol=1e-12)


def _eagle3_step0(W, cfg, aux, token, pos, k_ctx, v_ctx, norm_before_residual=True):
    """A plain EAGLE-3 first draft step for one request, written without any
    of the parallel-drafting machinery (no depths, no mask_hidden, no ptd).
    With norm_before_residual off, the layer-0 residual is the fc-projected
    hidden state itself rather than its hidden-norm output ("P-EAGLE" user
    guide, Key Parameters: --no-norm-before-residual)."""
    f64 = lambda a: np.asarray(a, dtype=np.float64)
    eps = cfg["rms_eps"]
    nq, nkv, hd = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]

    def norm(x, g):
        return x / math.sqrt(float(np.mean(x * x)) + eps) * f64(g)

    def rot(x):  # x [heads, hd] at position pos, complex form
        half = hd // 2
        out = np.empty_like(x)
        for j in range(half):
            ang = pos * cfg["rope_theta"] ** (-2.0 * j / hd)
            c, s = math.cos(ang), math.sin(ang)
            out[:, j] = x[:, j] * c - x[:, j + half] * s
            out[:, j + half] = x[:, j + half] * c + x[:, j] * s
        return out

    hid = norm(f64(W["fc_w"]) @ f64(aux), W["fc_norm_w"])
    h = None
    for l, L in enumerate(W["layers"]):
        if l == 0:
            hn = norm(hid, L["hidden_norm_w"])
            x = np.concatenate([norm(f64(W["embed"])[token], L["in_norm_w"]), hn])
            resid = hn if norm_before_residual else hid
        else:
            x = norm(h, L["in_norm_w"])
            resid = h
        qkv = f64(L["qkv_w"]) @ x
        q = rot(qkv[:nq * hd].reshape(nq, hd))
        k = rot(qkv[nq * hd:(nq + nkv) * hd].reshape(nkv, hd))
        v = qkv[(nq + nkv) * hd:].reshape(nkv, hd)
        keys = np.concatenate([f64(k_ctx[l]), k[None]], 0)
        vals = np.concatenate([f64(v_ctx[l]), v[None]], 0)
        o = np.zeros((nq, hd))
        for hh in range(nq):
            g = hh // (nq // nkv)
            p = scipy.special.softmax(keys[:, g] @ q[hh] / math.sqrt(hd))
            o[hh] = p @ vals[:, g]
        h1 = resid + f64(L["o_w"]) @ o.reshape(-1)
        y = norm(h1, L["post_norm_w"])
        I = cfg["intermediate"]
        gu = f64(L["gate_up_w"]) @ y
        h = h1 + f64(L["down_w"]) @ (gu[:I] * scipy.special.expit(gu[:I]) * gu[I:])
    return f64(W["lm_head_w"]) @ norm(h, W["final_norm_w"])


def test_k1_equals_eagle3_step0_and_ignores_masked_inputs():
    wl = tiny_workload(K=1)
    model, W = tiny_model(wl)
    inp = synth.make_decode_inputs(wl)
    args = (inp["aux"], inp["anchor_tokens"], inp["anchor_pos"], inp["k_cache"], inp["v_cache"],
            inp["kv_offsets"], inp["kv_lens"], 1)
    out = O.draft_step(model, *args)
    for b in range(wl.batch):
        o, L = int(inp["kv_offsets"][b]), int(inp["kv_lens"][b])
        ref = _eagle3_step0(W, model.cfg, inp["aux"][b], int(inp["anchor_tokens"][b]),
                            int(inp["anchor_pos"][b]),
                            [kc[o:o + L] for kc in inp["k_cache"]],
                            [vc[o:o + L] for vc in inp["v_cache"]])
        assert np.allclose(out["logits"][b, 0], ref, atol=1e-12)
    # poison mask_hidden and the ptd embedding row: K=1 must not read them
    W2 = dict(W)
    W2["mask_hidden"] = np.full_like(W["mask_hidden"], np.nan)
    emb = W["embed"].copy()
    emb[model.cfg["ptd_token_id"]] = np.nan
    W2["embed"] = emb
    if (inp["anchor_tokens"] == model.cfg["ptd_token_id"]).any():
        pytest.skip("anchor token hit the ptd id")
    out2 = O.draft_step(O.DraftModel(model.cfg, W2), *args)
    assert np.array_equal(out2["logits"], out["logits"])


def test_k1_without_norm_before_residual_equals_eagle3_step0():
    # the residual branch the flag switches: the fc-projected hidden state
    # (not its hidden-norm output) seeds the layer-0 residual stream
    wl = tiny_workload(K=1)
    model, W = tiny_model(wl, norm_before_residual=False)
    inp = synth.make_decode_inputs(wl)
    out = O.draft_step(model, inp["aux"], inp["anchor_tokens"], inp["anchor_pos"], inp["k_cache"],
                       inp["v_cache"], inp["kv_offsets"], inp["kv_lens"], 1)
    on, _ = tiny_model(wl)
    out_on = O.draft_step(on, inp["aux"], inp["anchor_tokens"], inp["anchor_pos"], inp["k_cache"],
                          inp["v_cache"], inp["kv_offsets"], inp["kv_lens"], 1)
    for b in range(wl.batch):
        o, L = int(inp["kv_offsets"][b]), int(inp["kv_lens"][b])
        ctx = ([kc[o:o + L] for kc in inp["k_cache"]], [vc[o:o + L] for vc in inp["v_cache"]])
        ref = _eagle3_step0(W, model.cfg, inp["aux"][b], int(inp["anchor_tokens"][b]),
                            int(inp["anchor_pos"][b]), *ctx, norm_before_residual=False)
        assert np.allclose(out["logits"][b, 0], ref, atol=1e-12)
        ref_on = _eagle3_step0(W, model.cfg, inp["aux"][b], int(inp["anchor_tokens"][b]),
                               int(inp["anchor_pos"][b]), *ctx, norm_before_residual=True)
        # the flag matters: the two readings give different logits
        assert not np.allclose(ref, ref_on, atol=1e-6)
        assert np.allclose(out_on["logits"][b, 0], ref_on, atol=1e-12)


def test_to_target_maps_the_argmax_id_through_d2t():
    # a hand-built draft-vocab logits row: the maximum 3.0 sits at draft ids
    # 1 and 2, so the lowest (1) wins and d2t turns it into a target id
    wl = tiny_workload()
    model, W = tiny_model(wl)
    perm = np.random.default_rng(4).permutation(wl.vocab)
    W2 = dict(W, d2t=perm)
    m2 = O.DraftModel(model.cfg, W2)
    row = np.full((1, wl.vocab), -2.0)
    row[0, 1] = row[0, 2] = 3.0
    row[0, 7] = 2.5
    assert int(m2.to_target(O.argmax_lowest(row))[0]) == int(perm[1])
    assert int(model.to_target(O.argmax_lowest(row))[0]) == 1
    # in a draft step the map acts on the argmax id only: the logits are
    # unchanged, and every token is perm[argmax of its own logits row]
    inp = synth.make_decode_inputs(wl)
    args = (inp["aux"], inp["anchor_tokens"], inp["anchor_pos"], inp["k_cache"], inp["v_cache"],
            inp["kv_offsets"], inp["kv_lens"], wl.K)
    a = O.draft_step(model, *args)
    b = O.draft_step(m2, *args)
    assert np.array_equal(a["logits"], b["logits"])
    assert np.array_equal(b["draft_tokens"], perm[np.argmax(a["logits"], axis=-1)])
    assert np.array_equal(a["draft_tokens"], np.argmax(a["logits"], axis=-1))
    # a draft vocab smaller than the target vocab: draft id j -> target id d2t[j]
    Vd = wl.vocab // 2
    d2t = np.sort(np.random.default_rng(5).choice(wl.vocab, Vd, replace=False))
    W3 = dict(W, lm_head_w=W["lm_head_w"][:Vd], d2t=d2t)
    cfg3 = dict(model.cfg, draft_vocab=Vd)
    c = O.draft_step(O.DraftModel(cfg3, W3), *args)
    assert c["logits"].shape[-1] == Vd
    assert np.array_equal(c["logits"], a["logits"][..., :Vd])
    assert np.array_equal(c["draft_tokens"], d2t[np.argmax(a["logits"][..., :Vd], axis=-1)])


def test_prefix_consistency_and_no_recurrence():
    wl = tiny_workload()
    model, W = tiny_model(wl)
    inp = synth.make_decode_inputs(wl)
    args = lambda K: (inp["aux"], inp["anchor_tokens"], inp["anchor_pos"], inp["k_cache"],
                      inp["v_cache"], inp["kv_offsets"], inp["kv_lens"], K)
    full = O.draft_step(model, *args(wl.K), keep_hidden=True)
    for Kp in range(1, wl.K):
        part = O.draft_step(model, *args(Kp))
        assert np.allclose(part["logits"], full["logits"][:, :Kp], atol=1e-12)
    # a different lm_head changes the drafts but no hidden state: depths do
    # not feed their outputs to one another
    W2 = dict(W)
    W2["lm_head_w"] = W["lm_head_w"][::-1].copy()
    other = O.draft_step(O.DraftModel(model.cfg, W2), *args(wl.K), keep_hidden=True)
    assert np.array_equal(other["hidden"], full["hidden"])
    assert not np.allclose(other["logits"], full["logits"])


def test_parallel_forward_matches_expanded_decode():
    # the training layout at (i, d) equals a decode step anchored at i whose
    # cache holds the depth-0 K/V of rows s(i)..i-1 of every layer
    wl, model, W, inp = tiny_train()
    res = O.parallel_forward(model, **inp, K=wl.K, r=1.0, r_min=1.0, seed=3, keep_kv=True)
    n = wl.n_tokens
    conv, start, end = O.conversation_bounds(inp["cu_seqlens"], n)
    for i in range(n):
        s = int(start[i])
        L = i - s
        kc = [res["kv"][l][0][s:i] for l in range(wl.num_layers)]
        vc = [res["kv"][l][1][s:i] for l in range(wl.num_layers)]
        out = O.draft_step(model, inp["aux"][i:i + 1], inp["input_ids"][i:i + 1],
                           inp["position_ids"][i:i + 1], kc, vc, np.array([0, L]),
                           np.array([L]), wl.K)
        for d in range(wl.K):
            row = d * n + i
            assert res["anchor"][row] == i and res["depth"][row] == d
            assert np.allclose(out["logits"][0, d], res["logits"][row], atol=1e-12, rtol=0)


def test_parallel_forward_dense_mask_bruteforce():
    wl, model, W, inp = tiny_train()
    res = O.parallel_forward(model, **inp, K=wl.K, r=0.7, r_min=0.2, seed=9)
    dense = O.parallel_forward(model, **inp, K=wl.K, r=0.7, r_min=0.2, seed=9, dense_rows=True)
    assert np.allclose(res["logits"], dense["logits"], atol=1e-12)


def test_labels_past_conversation_end_are_ignored():
    wl, model, W, inp = tiny_train()
    res = O.parallel_forward(model, **inp, K=wl.K, r=0.7, r_min=0.2, seed=9)
    cu = inp["cu_seqlens"]
    for d in range(wl.K):
        S = res["sets"][d]
        ends = [next(cu[c + 1] for c in range(len(cu) - 1) if cu[c] <= i < cu[c + 1]) for i in S]
        expect = sum(1 for i, e in zip(S, ends) if i + d < e)
        assert res["per_depth_valid"][d] == expect


def test_loss_matches_library_cross_entropy():
    wl, model, W, inp = tiny_train()
    res = O.parallel_forward(model, **inp, K=wl.K, r=0.7, r_min=0.2, seed=9)
    total = 0.0
    for d in range(wl.K):
        m = (res["depth"] == d) & (res["row_label"] >= 0)
        ce = torch.nn.functional.cross_entropy(torch.from_numpy(res["logits"][m]),
                                               torch.from_numpy(res["row_label"][m]))
        assert abs(float(ce) - res["per_depth_loss"][d]) < 1e-12
        acc = float(np.mean(np.argmax(res["logits"][m], -1) == res["row_label"][m]))
        assert abs(acc - res["per_depth_acc"][d]) < 1e-15
        total += 0.8 ** d * float(ce)
    assert abs(total - res["loss"]) < 1e-12


def test_out_of_draft_vocab_labels_equal_loss_mask():
    # a label outside the draft vocab (t2d = -1) drops its rows exactly like
    # masking its position out of the loss
    wl, model, W, inp = tiny_train()
    bad = {int(inp["labels"][3]), int(inp["labels"][10])}
    t2d = np.arange(wl.vocab)
    for t in bad:
        t2d[t] = -1
    W2 = dict(W)
    W2["t2d"] = t2d
    m2 = O.DraftModel(model.cfg, W2)
    a = O.parallel_forward(m2, **inp, K=wl.K, r=0.7, r_min=0.2, seed=9)
    mask = np.array([int(x) not in bad for x in inp["labels"]])
    inp_m = dict(inp, loss_mask=mask)
    b = O.parallel_forward(model, **inp_m, K=wl.K, r=0.7, r_min=0.2, seed=9)
    assert np.array_equal(a["per_depth_valid"], b["per_depth_valid"])
    assert np.allclose(a["per_depth_loss"], b["per_depth_loss"], atol=1e-12)
    c = O.parallel_forward(model, **inp, K=wl.K, r=0.7, r_min=0.2, seed=9)
    assert (a["per_depth_valid"] <= c["per_depth_valid"]).all()
    assert a["per_depth_valid"].sum() < c["per_depth_valid"].sum()


def test_starting_loss_near_log_vocab():
    # random weights: CE ~ ln V + sigma^2/2 for near-Gaussian logits of std sigma
    wl, model, W, inp = tiny_train(n=60, S_lens=(60,), vocab=1024)
    res = O.parallel_forward(model, **inp, K=wl.K, r=0.7, r_min=0.2, seed=1)
    lg = res["logits"][res["depth"] == 0]
    sigma2 = float(np.var(lg))
    want = math.log(wl.vocab) + sigma2 / 2
    assert abs(res["per_depth_loss"][0] - want) < 0.05 * want


def test_conversation_sampling_is_exact():
    wl, model, W, inp = tiny_train()
    full = O.parallel_forward(model, **inp, K=wl.K, r=0.7, r_min=0.2, seed=9)
    part = O.parallel_forward(model, **inp, K=wl.K, r=0.7, r_min=0.2, seed=9, conversations=[2])
    rows = np.flatnonzero(part["row_argmax"] >= 0)
    assert rows.size > 0
    assert np.array_equal(part["logits"][rows], full["logits"][rows])


def test_masked_row_is_an_anchor_row_fed_mask_hidden_and_ptd():
    # mask_hidden goes through the same fc/fc_norm as the aux states, and
    # ptd_token_id through the same embedding. So with an empty context, an
    # anchor whose aux is mask_hidden and whose token is ptd has the same
    # layer inputs as its masked depth-1 row; both rows then attend to equal
    # values, so every layer keeps them equal and their logits coincide.
    wl = tiny_workload(kv_len=0, kv_len_range=None, K=2, batch=1)
    model, W = tiny_model(wl)
    inp = synth.make_decode_inputs(wl)
    ptd = model.cfg["ptd_token_id"]
    out = O.draft_step(model, W["mask_hidden"], np.array([ptd]), np.array([5]),
                       inp["k_cache"], inp["v_cache"], inp["kv_offsets"], inp["kv_lens"], 2)
    assert np.allclose(out["logits"][0, 0], out["logits"][0, 1], atol=1e-12)
    # a real anchor makes them differ
    out2 = O.draft_step(model, inp["aux"], inp["anchor_tokens"], np.array([5]),
                        inp["k_cache"], inp["v_cache"], inp["kv_offsets"], inp["kv_lens"], 2)
    assert not np.allclose(out2["logits"][0, 0], out2["logits"][0, 1])


def test_row_labels_agree_with_forward():
    wl, model, W, inp = tiny_train()
    res = O.parallel_forward(model, **inp, K=wl.K, r=0.7, r_min=0.2, seed=9)
    lab, counts = O.row_labels(wl.n_tokens, wl.K, 0.7, 0.2, 9, inp["cu_seqlens"], inp["labels"])
    assert counts == res["counts"]
    assert np.array_equal(lab, res["row_label"])


# -------------------------------------------------------- stochastic verify
def _probs(rng, V, sharp=1.0):
    x = rng.standard_normal(V) * sharp
    e = np.exp(x - x.max())
    return (e / e.sum()).astype(np.float32)


def test_verify_sample_one_hot_is_greedy_verify():
    # one-hot target and draft distributions reduce rejection sampling to
    # greedy longest-prefix acceptance, the brute-force-pinned rule
    rng = np.random.default_rng(3)
    B, K, V = 400, 4, 3
    d = rng.integers(0, V, (B, K))
    t = rng.integers(0, V, (B, K + 1))
    t[:, :K] = np.where(rng.random((B, K)) < 0.6, d, t[:, :K])
    q = np.eye(V, dtype=np.float32)[d]
    p = np.eye(V, dtype=np.float32)[t]
    u = rng.random((B, K)).astype(np.float32)
    draws = rng.integers(0, 2 ** 32, B, dtype=np.uint64)
    a, n = O.verify_sample(d, q, p, u, draws)
    ga, gn = O.verify_accept(d, t)
    assert np.array_equal(a, ga) and np.array_equal(n, gn)


def test_verify_sample_first_token_follows_the_target_distribution():
    # the speculative-sampling theorem: whatever the draft distribution q,
    # the first emitted token is distributed as the target's p. Acceptance
    # depends only on u and the resample only on the draw, so each is
    # integrated on its own uniform grid.
    rng = np.random.default_rng(8)
    V, Nu, Nd = 6, 2000, 4000
    for trial in range(3):
        p0 = _probs(rng, V, 1.5)
        q0 = _probs(rng, V, 1.5)
        p = np.stack([p0, _probs(rng, V)])[None]          # [1, K+1=2, V]
        ugrid = ((np.arange(Nu) + 0.5) / Nu).astype(np.float32)
        A = np.zeros(V)
        for x in range(V):
            a, _ = O.verify_sample(np.full((Nu, 1), x), np.broadcast_to(q0, (Nu, 1, V)),
                                   np.broadcast_to(p, (Nu, 2, V)), ugrid[:, None], np.zeros(Nu, np.uint64))
            A[x] = a.mean()
            assert abs(A[x] - min(1.0, p0[x] / q0[x])) <= 1.5 / Nu
        xr = int(np.argmin(p0 / q0))                        # a draft that is rejected at u ~ 1
        assert p0[xr] < 0.99 * q0[xr]
        dgrid = (np.arange(Nd, dtype=np.uint64) * (2 ** 32 // Nd)).astype(np.uint64)
        a, nxt = O.verify_sample(np.full((Nd, 1), xr), np.broadcast_to(q0, (Nd, 1, V)),
                                 np.broadcast_to(p, (Nd, 2, V)), np.full((Nd, 1), 0.999999, np.float32), dgrid)
        assert (a == 0).all()
        R = np.bincount(nxt, minlength=V) / Nd
        resid = np.maximum(p0.astype(np.float64) - q0, 0)
        assert np.allclose(R, resid / resid.sum(), atol=2.0 / Nd)
        first = q0 * A + (1 - np.sum(q0 * A)) * R
        assert np.allclose(first, p0, atol=3e-3), (first, p0)


def test_verify_sample_bonus_token_follows_the_last_target_distribution():
    # drafts drawn from q = p are always kept (u < 1), and the bonus token is
    # then distributed as p_K
    rng = np.random.default_rng(9)
    V, K, Nd = 7, 3, 5000
    p = np.stack([_probs(rng, V) for _ in range(K + 1)])
    q = p[:K]
    d = np.argmax(q, -1)
    dgrid = (np.arange(Nd, dtype=np.uint64) * (2 ** 32 // Nd)).astype(np.uint64)
    a, nxt = O.verify_sample(np.broadcast_to(d, (Nd, K)), np.broadcast_to(q, (Nd, K, V)),
                             np.broadcast_to(p, (Nd, K + 1, V)), np.full((Nd, K), 0.9999, np.float32), dgrid)
    assert (a == K).all()
    assert np.allclose(np.bincount(nxt, minlength=V) / Nd, p[K], atol=2.0 / Nd)


def test_verify_sample_degenerate_residual_takes_the_argmax():
    # a draft with p(x) = q(x) = 0 is rejected (0 < 0 fails); when p == q the
    # residual is empty and the token is the lowest-index argmax of p
    V = 5
    p = np.array([0.1, 0.4, 0.0, 0.4, 0.1], dtype=np.float32)
    a, n = O.verify_sample(np.array([[2]]), p[None, None], np.stack([p, p])[None],
                           np.array([[0.5]], np.float32), np.array([123], np.uint64))
    assert a[0] == 0 and n[0] == 1
    # integer weights: floor(w * 2^40), NaN as 0, clamped to [0, 1]
    W = O.sample_weights(np.array([0.5, np.nan, 2.0, -1.0, 2.0 ** -41], np.float32))
    assert W.tolist() == [2 ** 39, 0, 2 ** 40, 0, 0]


def test_verify_sample_draw_intervals_are_half_open():
    # hand-worked: bonus weights [1/4, 1/4, 0, 1/2] give integer weights
    # [2^38, 2^38, 0, 2^39], S = 2^40 and T = draw * 2^8. Token j owns the
    # draws with prefix(j-1) <= T < prefix(j): [0, 2^30) -> 0,
    # [2^30, 2^31) -> 1, token 2 never, [2^31, 2^32) -> 3
    p = np.array([[0.0, 1.0, 0.0, 0.0], [0.25, 0.25, 0.0, 0.5]], dtype=np.float32)[None]
    q = np.array([[0.0, 1.0, 0.0, 0.0]], dtype=np.float32)[None]
    cases = {0: 0, 2 ** 30 - 1: 0, 2 ** 30: 1, 2 ** 31 - 1: 1, 2 ** 31: 3, 2 ** 32 - 1: 3}
    for draw, want in cases.items():
        a, n = O.verify_sample(np.array([[1]]), q, p, np.array([[0.3]], np.float32), np.array([draw], np.uint64))
        assert a[0] == 1 and n[0] == want, (draw, n[0], want)


# ------------------------------------------------------------ batch of sequences
def test_depth_sums_of_one_sequence_give_its_loss():
    wl, model, W, inp = tiny_train()
    res = O.parallel_forward(model, **inp, K=wl.K, r=0.7, r_min=0.2, seed=9)
    got = O.loss_from_depth_sums(O.depth_sums(res, wl.K))
    assert abs(got["loss"] - res["loss"]) < 1e-12
    assert np.allclose(got["per_depth_loss"], res["per_depth_loss"], atol=1e-12)
    assert np.allclose(got["per_depth_acc"], res["per_depth_acc"], atol=1e-15)
    assert np.array_equal(got["per_depth_valid"], res["per_depth_valid"])


def test_batch_loss_is_library_cross_entropy_over_all_sequences():
    # two packed sequences: each depth's mean is taken over the labelled rows
    # of both, then the depths are weighted by 0.8^d
    wl, model, W, inp = tiny_train()
    wl2, _, _, inp2 = tiny_train(n=17, S_lens=(10, 7), seed=6)
    res = [O.parallel_forward(model, **x, K=wl.K, r=0.7, r_min=0.2, seed=sd)
           for x, sd in ((inp, 9), (inp2, 4))]
    got = O.loss_from_depth_sums(sum(O.depth_sums(r_, wl.K) for r_ in res))
    total = 0.0
    for d in range(wl.K):
        lg = np.concatenate([r_["logits"][(r_["depth"] == d) & (r_["row_label"] >= 0)] for r_ in res])
        lb = np.concatenate([r_["row_label"][(r_["depth"] == d) & (r_["row_label"] >= 0)] for r_ in res])
        ce = float(torch.nn.functional.cross_entropy(torch.from_numpy(lg), torch.from_numpy(lb)))
        assert abs(ce - got["per_depth_loss"][d]) < 1e-12
        assert got["per_depth_valid"][d] == len(lb)
        total += 0.8 ** d * ce
    assert abs(total - got["loss"]) < 1e-12


# ------------------------------------------------------- new context rows
def test_draft_step_ctx_with_one_new_row_is_the_anchor_step():
    wl = tiny_workload()
    model, W = tiny_model(wl)
    inp = synth.make_decode_inputs(wl)
    args = (inp["k_cache"], inp["v_cache"], inp["kv_offsets"], inp["kv_lens"], wl.K)
    a = O.draft_step(model, inp["aux"], inp["anchor_tokens"], inp["anchor_pos"], *args, append_anchor_kv=True)
    b = O.draft_step_ctx(model, [inp["aux"][i:i + 1] for i in range(wl.batch)],
                         [[t] for t in inp["anchor_tokens"]], [[p] for p in inp["anchor_pos"]], *args)
    assert np.array_equal(a["logits"], b["logits"]) and np.array_equal(a["draft_tokens"], b["draft_tokens"])
    for l in range(wl.num_layers):
        for r in range(wl.batch):
            assert np.array_equal(a["appended"][l][r][0], b["appended"][l][r][0][0])


def test_draft_step_ctx_equals_the_training_layout():
    # a conversation prefix fed as new rows over an empty cache is the
    # training layout's anchor: the depth logits equal parallel_forward's
    # rows (i, d) (pinned against expanded decode), and the new rows' K/V
    # equal its depth-0 K/V
    wl, model, W, inp = tiny_train()
    res = O.parallel_forward(model, **inp, K=wl.K, r=1.0, r_min=1.0, seed=3, keep_kv=True)
    n = wl.n_tokens
    cu = inp["cu_seqlens"]
    empty = [np.zeros((1, wl.num_kv_heads, wl.head_dim))] * wl.num_layers
    for i in (0, 5, 8, 9, 12, 22):
        s = int(cu[np.searchsorted(cu, i, side="right") - 1])
        out = O.draft_step_ctx(model, [inp["aux"][s:i + 1]], [inp["input_ids"][s:i + 1]],
                               [inp["position_ids"][s:i + 1]], empty, empty, [0], [0], wl.K)
        for d in range(wl.K):
            assert np.allclose(out["logits"][0, d], res["logits"][d * n + i], atol=1e-12, rtol=0)
        for l in range(wl.num_layers):
            assert np.allclose(out["appended"][l][0][0], res["kv"][l][0][s:i + 1], atol=1e-12)


def test_draft_step_ctx_split_over_two_calls_matches_one_call():
    # feeding new rows in two steps (the first appending its rows to the
    # cache) drafts what one step over all of them drafts
    wl = tiny_workload(kv_len_range=(2, 5))
    model, W = tiny_model(wl)
    inp = synth.make_decode_inputs(wl, spare=8)
    rng = np.random.default_rng(12)
    B = wl.batch
    n = [3, 1, 4]
    aux = [rng.standard_normal((k, wl.num_aux * wl.target_hidden)) for k in n]
    tok = [rng.integers(0, wl.vocab, k) for k in n]
    pos = [list(range(int(inp["kv_lens"][b]), int(inp["kv_lens"][b]) + n[b])) for b in range(B)]
    one = O.draft_step_ctx(model, aux, tok, pos, inp["k_cache"], inp["v_cache"], inp["kv_offsets"],
                           inp["kv_lens"], wl.K)
    m = [1, 0, 2]   # rows of the first call (a request needs at least one: b=1 takes all in call 2)
    kc = [k.copy() for k in inp["k_cache"]]
    vc = [v.copy() for v in inp["v_cache"]]
    first = [b for b in range(B) if m[b] > 0]
    o1 = O.draft_step_ctx(model, [aux[b][:m[b]] for b in first], [tok[b][:m[b]] for b in first],
                          [pos[b][:m[b]] for b in first], kc, vc, inp["kv_offsets"][first],
                          inp["kv_lens"][first], wl.K)
    lens = inp["kv_lens"].copy()
    for i, b in enumerate(first):
        for l in range(wl.num_layers):
            k, v = o1["appended"][l][i]
            o = int(inp["kv_offsets"][b] + lens[b])
            kc[l][o:o + m[b]] = k
            vc[l][o:o + m[b]] = v
        lens[b] += m[b]
    two = O.draft_step_ctx(model, [aux[b][m[b]:] for b in range(B)], [tok[b][m[b]:] for b in range(B)],
                           [pos[b][m[b]:] for b in range(B)], kc, vc, inp["kv_offsets"], lens, wl.K)
    assert np.allclose(one["logits"], two["logits"], atol=1e-12)
    assert np.array_equal(one["draft_tokens"], two["draft_tokens"])


def test_next_context_hand_worked():
    drafts = np.array([[5, 6, 7], [8, 9, 1]])
    toks, pos = O.next_context(drafts, np.array([2, 0]), np.array([40, 41]), np.array([10, 20]))
    assert toks == [[5, 6, 40], [41]] and pos == [[11, 12, 13], [21]]


# ------------------------------------------------------------------- gradients
def _grad_case(nbr=True, **kw):
    wl, model, W, inp = tiny_train(**kw)
    if not nbr:
        model = O.DraftModel(dict(model.cfg, norm_before_residual=False), W)
    return wl, model, W, inp


@pytest.mark.parametrize("nbr", [True, False])
def test_autograd_loss_is_the_forward_loss(nbr):
    wl, model, W, inp = _grad_case(nbr)
    res = O.parallel_forward(model, **inp, K=wl.K, r=0.7, r_min=0.2, seed=9)
    loss, _ = O.parallel_loss_torch(model, **inp, K=wl.K, r=0.7, r_min=0.2, seed=9)
    assert abs(float(loss.detach()) - res["loss"]) < 1e-12


@pytest.mark.parametrize("nbr", [True, False])
def test_gradients_match_central_differences(nbr):
    # central differences of the (pinned) forward loss, in float64, on a few
    # coordinates of every weight that has a gradient
    wl, model, W, inp = _grad_case(nbr)
    kw = dict(**inp, K=wl.K, r=0.7, r_min=0.2, seed=9)
    _, grads = O.parallel_grads(model, **kw)
    rng = np.random.default_rng(3)
    h = 1e-6

    def loss_with(path, idx, delta):
        W2 = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in W.items()}
        W2["layers"] = [{k: (None if v is None else np.asarray(v, dtype=np.float64).copy()) for k, v in L.items()}
                        for L in W["layers"]]
        for k in ("fc_w", "fc_norm_w", "mask_hidden", "final_norm_w", "lm_head_w"):
            W2[k] = np.asarray(W2[k], dtype=np.float64)
        arr = W2[path[0]] if len(path) == 1 else W2["layers"][path[0]][path[1]]
        arr[idx] += delta
        return O.parallel_forward(O.DraftModel(model.cfg, W2), **kw)["loss"]

    paths = [(k,) for k in O.GRAD_KEYS] + [(l, k) for l in range(wl.num_layers) for k in O.LAYER_GRAD_KEYS
                                           if W["layers"][l].get(k) is not None]
    for path in paths:
        g = grads[path[0]] if len(path) == 1 else grads["layers"][path[0]][path[1]]
        for _ in range(3):
            idx = tuple(int(rng.integers(0, s)) for s in g.shape)
            fd = (loss_with(path, idx, h) - loss_with(path, idx, -h)) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(g).max()), (path, idx, fd, g[idx])


def test_loss_decreases_along_the_negative_gradient():
    wl, model, W, inp = _grad_case()
    kw = dict(**inp, K=wl.K, r=0.7, r_min=0.2, seed=9)
    loss0, grads = O.parallel_grads(model, **kw)
    W2 = dict(W)
    lr = 0.05
    for k in O.GRAD_KEYS:
        W2[k] = np.asarray(W[k], dtype=np.float64) - lr * grads[k].reshape(np.shape(W[k]))
    W2["layers"] = [{k: (None if v is None else np.asarray(v, dtype=np.float64) - lr * grads["layers"][l][k])
                     if k in grads["layers"][l] else v for k, v in L.items()} for l, L in enumerate(W["layers"])]
    loss1 = O.parallel_forward(O.DraftModel(model.cfg, W2), **kw)["loss"]
    assert loss1 < loss0 - 1e-4, (loss0, loss1)
