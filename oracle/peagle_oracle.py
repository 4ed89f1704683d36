"""Plain float64 CPU oracle of the P-EAGLE parallel-drafting step.

TEST INFRASTRUCTURE ONLY. This module is the parity reference for the CUDA
library and the timed CPU baseline. Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the product path never does.
It shares no code with the CUDA path: no kernels, helpers, tables or
constants. It computes every step directly from its definition, in float64,
on float64 copies of the (already bf16- or fp32-valued) inputs.

Sources (page title, then section):
  [UG]   "P-EAGLE" user guide page: How It Works / Architecture,
         COD Sampling, Inference Process, Key Parameters.
  [PR]   "feat(speculative): add P-EAGLE parallel-drafting training for
         EAGLE-3 drafts - #2376": PR description, Changelog, Checkpoint
         contract, Equivalence to vLLM inference (parity), Validation,
         and the RoPE fix commit message ("Gather cos/sin by the actual
         position values ...").
  [RM]   "P_Eagle" README: the "How Speculative Decoding Works" table
         (EAGLE-3 injection concatenates [embeddings (+) hidden]) and the
         variable-length attention note (cu_seqlens isolation).

Readings taken where the pages are silent:
  * layer-0 input is [RMSNorm_in(embedding) (+) RMSNorm_hidden(hidden)]
    (2H wide); later layers take RMSNorm_in(h) (H wide);
  * norm_before_residual (default on) makes the layer-0 residual the
    normalised hidden state;
  * fc_norm and the final norm are RMSNorms with a gain;
  * RoPE is Llama rotate-half with inv_freq[j] = theta^(-2j/hd);
  * decode context = cache rows of the request; the anchor row is chain
    element 0; depth d also sees chain elements 1..d;
  * training depth-d row at anchor i sees depth-0 rows s(i)..i of its own
    conversation and its own chain rows (i,1..d);
  * depth-d label of anchor i is labels[i+d] when i+d is inside the
    conversation (and unmasked, and inside the draft vocab);
  * COD counts: c_0 = n, c_d = min(c_{d-1}, max(floor(n r^d), floor(n r_min)));
    S_d = the c_d positions with the smallest SplitMix64 keys (nested);
  * argmax takes the lowest index among equal maxima;
  * loss = sum_d decay^d * mean_d(CE); an empty depth contributes 0.
"""
import functools
import math

import numpy as np

MASK64 = (1 << 64) - 1
SPLITMIX_GAMMA = 0x9E3779B97F4A7C15


# --------------------------------------------------------------------------
# SplitMix64 (Steele, Lea, Flood: "Fast splittable pseudorandom number
# generators", OOPSLA 2014), the generator behind COD's random subsets.
# Output i of a generator seeded with s is mix(s + (i+1)*gamma mod 2^64).
# --------------------------------------------------------------------------
def splitmix64(seed: int, count: int) -> np.ndarray:
    """The first ``count`` outputs of SplitMix64 seeded with ``seed``."""
    with np.errstate(over="ignore"):
        i = np.arange(1, count + 1, dtype=np.uint64)
        z = np.uint64(seed & MASK64) + i * np.uint64(SPLITMIX_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


# --------------------------------------------------------------------------
# COD (Conditional Drop-token) sampling  [UG: COD Sampling, Key Parameters]
# Depth 0 keeps all n positions, depth d keeps about n*r^d, never fewer than
# the floor n*r_min. Subsets are nested so that every kept depth-d row has
# its chain rows at depths 1..d-1.
# --------------------------------------------------------------------------
def cod_counts(n: int, K: int, r: float, r_min: float) -> list:
    counts = [n]
    rd = 1.0
    floor_min = math.floor(n * r_min)
    for _ in range(1, K):
        rd = rd * r
        c = max(math.floor(n * rd), floor_min)
        counts.append(min(counts[-1], c))
    return counts


def cod_select(n: int, K: int, r: float, r_min: float, seed: int):
    """Return (counts, sets): sets[d] = ascending int64 positions kept at d."""
    counts = cod_counts(n, K, r, r_min)
    keys = splitmix64(seed, n)
    order = np.argsort(keys, kind="stable")        # keys are distinct
    sets = [np.arange(n, dtype=np.int64)]
    for d in range(1, K):
        sets.append(np.sort(order[:counts[d]]).astype(np.int64))
    return counts, sets


# --------------------------------------------------------------------------
# Greedy verification  [UG: Inference Process]
# --------------------------------------------------------------------------
def verify_accept(drafts: np.ndarray, targets: np.ndarray):
    """accept[b] = longest prefix of drafts[b] equal to targets[b];
    next[b] = targets[b, accept[b]] (the correction or bonus token)."""
    drafts = np.asarray(drafts)
    targets = np.asarray(targets)
    B, K = drafts.shape
    accept = np.zeros(B, dtype=np.int32)
    nxt = np.zeros(B, dtype=np.int32)
    for b in range(B):
        a = 0
        while a < K and drafts[b, a] == targets[b, a]:
            a += 1
        accept[b] = a
        nxt[b] = targets[b, a]
    return accept, nxt


# --------------------------------------------------------------------------
# Stochastic verification  ["P_Eagle" README, "How Speculative Decoding
# Works" row 6: accepted tokens are used, rejected ones resampled; output
# quality "probabilistically same" as the target]
# The published speculative-sampling rule (Leviathan, Kalman, Matias, ICML
# 2023; Chen et al., 2023): draft token x at depth i is kept with probability
# min(1, p_i(x) / q_i(x)); at the first rejection the next token is drawn
# from the normalised residual max(0, p_i - q_i); when all K drafts are kept
# it is drawn from p_K (the bonus token). The random numbers are inputs:
#   accept_u[b, i] in [0, 1): keep x iff fl32(u * q_i(x)) < p_i(x), in fp32;
#   draws[b]: a uniform 32-bit integer for the one inverse-CDF draw.
# The draw is exact integer arithmetic: each weight (the fp32 residual or
# p_K, clamped to [0, 1], NaN as 0) becomes W_j = floor(w_j * 2^40) (int64),
# S = sum W_j, T = (draw * S) >> 32, and the token is the smallest j whose
# inclusive prefix sum of W exceeds T. Weights below 2^-40 thus count as 0.
# If S == 0 (the draft was rejected where p and q agree to 2^-40), the token
# is the lowest-index argmax of p_i.
# --------------------------------------------------------------------------
SAMPLE_SCALE = 2.0 ** 40


def sample_weights(w):
    """Integer weights of the inverse-CDF draw from fp32 weights w."""
    w = np.asarray(w, dtype=np.float32).astype(np.float64)
    w = np.where(np.isnan(w), 0.0, np.clip(w, 0.0, 1.0))
    return np.floor(w * SAMPLE_SCALE).astype(np.int64)


def verify_sample(drafts, draft_probs, target_probs, accept_u, draws):
    """drafts [B, K] target ids; draft_probs q [B, K, V] and target_probs
    p [B, K+1, V] (fp32 values); accept_u [B, K] fp32; draws [B] uint32.
    Returns (accept_len [B], next_token [B])."""
    drafts = np.asarray(drafts, dtype=np.int64)
    q = np.asarray(draft_probs, dtype=np.float32)
    p = np.asarray(target_probs, dtype=np.float32)
    u = np.asarray(accept_u, dtype=np.float32)
    B, K = drafts.shape
    accept = np.zeros(B, dtype=np.int32)
    nxt = np.zeros(B, dtype=np.int32)
    for b in range(B):
        a = 0
        while a < K:
            x = int(drafts[b, a])
            if not (np.float32(u[b, a] * q[b, a, x]) < p[b, a, x]):
                break
            a += 1
        if a < K:
            w = np.maximum(p[b, a] - q[b, a], np.float32(0.0))
        else:
            w = p[b, K]
        W = sample_weights(w)
        S = int(W.sum())
        if S == 0:
            nxt[b] = int(argmax_lowest(p[b, a]))
        else:
            T = (int(draws[b]) * S) >> 32
            nxt[b] = int(np.searchsorted(np.cumsum(W), T, side="right"))
        accept[b] = a
    return accept, nxt


# --------------------------------------------------------------------------
# Dense pieces
# --------------------------------------------------------------------------
def rms_norm(x, gain, eps):
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gain


def silu(x):
    return x / (1.0 + np.exp(-x))


def argmax_lowest(x):
    """Row argmax, lowest index among equal maxima (first NaN wins)."""
    return np.argmax(x, axis=-1)


def logsumexp(x):
    m = np.max(x, axis=-1, keepdims=True)
    return (m + np.log(np.sum(np.exp(x - m), axis=-1, keepdims=True)))[..., 0]


# --------------------------------------------------------------------------
# RoPE gathered by position value  [PR: RoPE fix commit]
# cos/sin rows are looked up at the actual position values (anchor + d,
# packed restarts), from a table sized to the highest requested position.
# --------------------------------------------------------------------------
@functools.lru_cache(maxsize=16)
def rope_table(max_pos: int, head_dim: int, theta: float):
    half = head_dim // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / head_dim)
    ang = np.arange(max_pos + 1, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang), np.sin(ang)


def apply_rope(x, pos, theta):
    """x: [rows, heads, hd]; pos: [rows] integer positions (any values)."""
    pos = np.asarray(pos, dtype=np.int64)
    hd = x.shape[-1]
    half = hd // 2
    top = int(pos.max()) if pos.size else 0
    size = 1 << max(top, 1).bit_length()       # table covers the highest position
    cos_t, sin_t = rope_table(size, hd, float(theta))
    c = cos_t[pos][:, None, :]
    s = sin_t[pos][:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# --------------------------------------------------------------------------
# Masked attention: softmax(q k^T / sqrt(hd)) v over an allowed-key set.
# --------------------------------------------------------------------------
def masked_attention(q, k, v, allowed):
    """q [Rq, nq, hd], k/v [Rk, nkv, hd], allowed [Rq, Rk] bool.
    Query head h reads KV head h // (nq/nkv)."""
    Rq, nq, hd = q.shape
    nkv = k.shape[1]
    g = nq // nkv
    out = np.zeros((Rq, nq, hd), dtype=np.float64)
    scale = 1.0 / math.sqrt(hd)
    for h in range(nq):
        kh = k[:, h // g, :]
        vh = v[:, h // g, :]
        s = (q[:, h, :] @ kh.T) * scale
        s = np.where(allowed, s, -np.inf)
        m = np.max(s, axis=-1, keepdims=True)
        p = np.where(allowed, np.exp(s - m), 0.0)
        p = p / np.sum(p, axis=-1, keepdims=True)
        out[:, h, :] = p @ vh
    return out


# --------------------------------------------------------------------------
# The draft model
# --------------------------------------------------------------------------
class DraftModel:
    """float64 copy of a P-EAGLE draft (EAGLE-3 layout plus mask_hidden).

    cfg keys: hidden, target_hidden, num_aux, num_layers, num_q_heads,
    num_kv_heads, head_dim, intermediate, target_vocab, draft_vocab,
    ptd_token_id, rope_theta, rms_eps, norm_before_residual.
    W keys: embed, fc_w, fc_norm_w, mask_hidden, final_norm_w, lm_head_w,
    d2t, t2d, layers[l]{in_norm_w, hidden_norm_w, qkv_w, o_w, post_norm_w,
    gate_up_w, down_w}.
    """

    def __init__(self, cfg: dict, W: dict):
        self.cfg = dict(cfg)
        f = lambda a: None if a is None else np.asarray(a, dtype=np.float64)
        self.embed = f(W["embed"])
        self.fc_w = f(W["fc_w"])
        self.fc_norm_w = f(W["fc_norm_w"])
        # mask_hidden is one learnable row of width num_aux * target_hidden
        # [PR: Changelog, Checkpoint contract]
        self.mask_hidden = f(W["mask_hidden"]).reshape(1, -1)
        self.final_norm_w = f(W["final_norm_w"])
        self.lm_head_w = f(W["lm_head_w"])
        self.d2t = None if W.get("d2t") is None else np.asarray(W["d2t"], dtype=np.int64)
        self.t2d = None if W.get("t2d") is None else np.asarray(W["t2d"], dtype=np.int64)
        self.layers = [{k: f(v) for k, v in L.items()} for L in W["layers"]]
        c = self.cfg
        assert self.mask_hidden.shape == (1, c["num_aux"] * c["target_hidden"])
        assert 0 <= c["ptd_token_id"] < c["target_vocab"]

    # fc + fc_norm over the concatenated aux hidden states  [UG: Architecture]
    def project_hidden(self, aux):
        u = np.asarray(aux, dtype=np.float64) @ self.fc_w.T
        return rms_norm(u, self.fc_norm_w, self.cfg["rms_eps"])

    # the masked depths' hidden input: mask_hidden through the same fc/fc_norm
    # [PR: Changelog, masked_projected_hidden()]
    def masked_hidden(self):
        return self.project_hidden(self.mask_hidden)[0]

    def layer(self, l, h, tok_emb, pos, attend):
        """One decoder layer over a set of rows.

        Layer 0: h = fc-projected hidden rows, tok_emb = token embeddings.
        Layers >= 1: h = residual stream, tok_emb unused.
        attend(q, k, v) -> o performs the depth-masked attention.
        Returns the new residual stream.
        """
        c = self.cfg
        L = self.layers[l]
        eps = c["rms_eps"]
        nq, nkv, hd = c["num_q_heads"], c["num_kv_heads"], c["head_dim"]
        if l == 0:
            e = rms_norm(tok_emb, L["in_norm_w"], eps)
            hn = rms_norm(h, L["hidden_norm_w"], eps)
            x = np.concatenate([e, hn], axis=-1)
            resid = hn if c["norm_before_residual"] else h
        else:
            x = rms_norm(h, L["in_norm_w"], eps)
            resid = h
        qkv = x @ L["qkv_w"].T
        R = x.shape[0]
        q = qkv[:, :nq * hd].reshape(R, nq, hd)
        k = qkv[:, nq * hd:(nq + nkv) * hd].reshape(R, nkv, hd)
        v = qkv[:, (nq + nkv) * hd:].reshape(R, nkv, hd)
        q = apply_rope(q, pos, c["rope_theta"])
        k = apply_rope(k, pos, c["rope_theta"])
        o = attend(q, k, v)
        h1 = resid + o.reshape(R, nq * hd) @ L["o_w"].T
        y = rms_norm(h1, L["post_norm_w"], eps)
        I = c["intermediate"]
        gu = y @ L["gate_up_w"].T
        m = silu(gu[:, :I]) * gu[:, I:]
        h2 = h1 + m @ L["down_w"].T
        return h2, k, v

    def head(self, h):
        z = rms_norm(h, self.final_norm_w, self.cfg["rms_eps"])
        return z @ self.lm_head_w.T

    def to_target(self, draft_ids):
        return draft_ids if self.d2t is None else self.d2t[draft_ids]


# --------------------------------------------------------------------------
# Decode: one parallel draft step  [UG: Architecture, Inference Process;
# PR: Equivalence to vLLM inference -- the flat [context, mask_1..mask_{K-1}]
# layout]. All K depths of each request come out of one pass.
# --------------------------------------------------------------------------
def decode_allowed(L_ctx: int, K: int):
    """Allowed keys of the K depth rows of one request over
    [context (L_ctx rows), chain 0..K-1]: all context, chain j <= d."""
    m = np.zeros((K, L_ctx + K), dtype=bool)
    m[:, :L_ctx] = True
    for d in range(K):
        m[d, L_ctx:L_ctx + d + 1] = True
    return m


def draft_step(model: DraftModel, aux, anchor_tokens, anchor_pos, k_cache, v_cache,
               kv_offsets, kv_lens, K, append_anchor_kv=False, requests=None,
               dense_attention=False, keep_hidden=False):
    """Returns dict(draft_tokens [B,K], logits [B,K,Vd], and optionally the
    appended anchor K/V rows and pre-head hidden states).

    ``requests`` restricts the computation to a subset of requests (they are
    independent); rows of other requests are left zero.
    ``dense_attention`` switches to one brute-force boolean mask over all
    requests' rows (tiny inputs only)."""
    c = model.cfg
    B = len(anchor_tokens)
    req = list(range(B)) if requests is None else list(requests)
    Vd = c["draft_vocab"]
    ptd = c["ptd_token_id"]
    h_mask = model.masked_hidden()
    out_tok = np.zeros((B, K), dtype=np.int64)
    out_logits = np.zeros((B, K, Vd), dtype=np.float64)
    hidden = np.zeros((B, K, c["hidden"])) if keep_hidden else None
    appended = [dict() for _ in range(c["num_layers"])]

    if dense_attention:
        return _draft_step_dense(model, aux, anchor_tokens, anchor_pos, k_cache, v_cache,
                                 kv_offsets, kv_lens, K, append_anchor_kv, req, keep_hidden)

    for b in req:
        h_anchor = model.project_hidden(np.asarray(aux[b:b + 1], dtype=np.float64))[0]
        toks = np.array([anchor_tokens[b]] + [ptd] * (K - 1), dtype=np.int64)
        h = np.stack([h_anchor] + [h_mask] * (K - 1))
        emb = model.embed[toks]
        pos = int(anchor_pos[b]) + np.arange(K)
        off, Lb = int(kv_offsets[b]), int(kv_lens[b])
        allowed = decode_allowed(Lb, K)
        for l in range(c["num_layers"]):
            ck = np.asarray(k_cache[l][off:off + Lb], dtype=np.float64)
            cv = np.asarray(v_cache[l][off:off + Lb], dtype=np.float64)

            def attend(q, k, v, ck=ck, cv=cv):
                return masked_attention(q, np.concatenate([ck, k]), np.concatenate([cv, v]), allowed)

            h, k, v = model.layer(l, h, emb, pos, attend)
            if append_anchor_kv:
                appended[l][b] = (k[0].copy(), v[0].copy())
        logits = model.head(h)
        out_logits[b] = logits
        out_tok[b] = model.to_target(argmax_lowest(logits))
        if keep_hidden:
            hidden[b] = h
    res = {"draft_tokens": out_tok, "logits": out_logits, "appended": appended}
    if keep_hidden:
        res["hidden"] = hidden
    return res


def _draft_step_dense(model, aux, anchor_tokens, anchor_pos, k_cache, v_cache,
                      kv_offsets, kv_lens, K, append_anchor_kv, req, keep_hidden):
    """All requests' rows in one batch with one brute-force mask built key by
    key from the definition: a query (b, d) may read key x iff x belongs to
    request b and x is a context row, or x is chain row (b, j) with j <= d."""
    c = model.cfg
    B = len(anchor_tokens)
    ptd = c["ptd_token_id"]
    h_mask = model.masked_hidden()
    rows = [(b, d) for b in req for d in range(K)]
    R = len(rows)
    toks = np.array([anchor_tokens[b] if d == 0 else ptd for b, d in rows], dtype=np.int64)
    hanc = {b: model.project_hidden(np.asarray(aux[b:b + 1], dtype=np.float64))[0] for b in req}
    h = np.stack([hanc[b] if d == 0 else h_mask for b, d in rows])
    emb = model.embed[toks]
    pos = np.array([int(anchor_pos[b]) + d for b, d in rows])
    ctx_keys = [(b, t) for b in req for t in range(int(kv_lens[b]))]
    keys = [("ctx", b, t) for b, t in ctx_keys] + [("chain", b, d) for b, d in rows]
    allowed = np.zeros((R, len(keys)), dtype=bool)
    for qi, (qb, qd) in enumerate(rows):
        for ki, key in enumerate(keys):
            if key[0] == "ctx":
                allowed[qi, ki] = key[1] == qb
            else:
                allowed[qi, ki] = key[1] == qb and key[2] <= qd
    appended = [dict() for _ in range(c["num_layers"])]
    for l in range(c["num_layers"]):
        ck = np.stack([np.asarray(k_cache[l][int(kv_offsets[b]) + t], dtype=np.float64)
                       for b, t in ctx_keys]) if ctx_keys else np.zeros((0, c["num_kv_heads"], c["head_dim"]))
        cv = np.stack([np.asarray(v_cache[l][int(kv_offsets[b]) + t], dtype=np.float64)
                       for b, t in ctx_keys]) if ctx_keys else np.zeros_like(ck)

        def attend(q, k, v, ck=ck, cv=cv):
            return masked_attention(q, np.concatenate([ck, k]), np.concatenate([cv, v]), allowed)

        h, k, v = model.layer(l, h, emb, pos, attend)
        if append_anchor_kv:
            for qi, (b, d) in enumerate(rows):
                if d == 0:
                    appended[l][b] = (k[qi].copy(), v[qi].copy())
    logits = model.head(h)
    Vd = c["draft_vocab"]
    out_logits = np.zeros((B, K, Vd))
    out_tok = np.zeros((B, K), dtype=np.int64)
    for qi, (b, d) in enumerate(rows):
        out_logits[b, d] = logits[qi]
        out_tok[b, d] = model.to_target(argmax_lowest(logits[qi:qi + 1]))[0]
    res = {"draft_tokens": out_tok, "logits": out_logits, "appended": appended}
    if keep_hidden:
        hid = np.zeros((B, K, c["hidden"]))
        for qi, (b, d) in enumerate(rows):
            hid[b, d] = h[qi]
        res["hidden"] = hid
    return res


# --------------------------------------------------------------------------
# Decode over new context rows  [PR: Equivalence to vLLM inference -- the
# flat [context, new rows, mask_1..mask_{K-1}] layout; UG: Inference Process]
# Each request brings n_b >= 1 new rows (token, aux state, position); the
# last is the anchor. Row j of a request (its new rows, then its masked
# depths 1..K-1) attends to the request's cached context and to its rows
# 0..j. The new rows' K/V join the context.
# --------------------------------------------------------------------------
def draft_step_ctx(model: DraftModel, new_aux, new_tokens, new_pos, k_cache, v_cache, kv_offsets,
                   kv_lens, K):
    """new_aux / new_tokens / new_pos: per request, a list (or array) of its
    new rows. Returns draft_tokens [B, K], logits [B, K, Vd] (depth rows:
    the anchor, then the masked rows) and appended[l][b] = (k, v) of the
    request's new rows."""
    c = model.cfg
    B = len(new_tokens)
    ptd = c["ptd_token_id"]
    h_mask = model.masked_hidden()
    out_tok = np.zeros((B, K), dtype=np.int64)
    out_logits = np.zeros((B, K, c["draft_vocab"]))
    appended = [dict() for _ in range(c["num_layers"])]
    for b in range(B):
        n = len(new_tokens[b])
        assert n >= 1
        hp = model.project_hidden(np.asarray(new_aux[b], dtype=np.float64).reshape(n, -1))
        toks = np.array(list(new_tokens[b]) + [ptd] * (K - 1), dtype=np.int64)
        h = np.concatenate([hp, np.stack([h_mask] * (K - 1))]) if K > 1 else hp
        emb = model.embed[toks]
        anchor = int(new_pos[b][n - 1])
        pos = np.array(list(new_pos[b]) + [anchor + d for d in range(1, K)], dtype=np.int64)
        off, Lb = int(kv_offsets[b]), int(kv_lens[b])
        rows = n + K - 1
        allowed = np.zeros((rows, Lb + rows), dtype=bool)
        allowed[:, :Lb] = True
        for j in range(rows):
            allowed[j, Lb:Lb + j + 1] = True
        for l in range(c["num_layers"]):
            ck = np.asarray(k_cache[l][off:off + Lb], dtype=np.float64)
            cv = np.asarray(v_cache[l][off:off + Lb], dtype=np.float64)

            def attend(q, k, v, ck=ck, cv=cv):
                return masked_attention(q, np.concatenate([ck, k]), np.concatenate([cv, v]), allowed)

            h, k, v = model.layer(l, h, emb, pos, attend)
            appended[l][b] = (k[:n].copy(), v[:n].copy())
        logits = model.head(h[n - 1:])
        out_logits[b] = logits
        out_tok[b] = model.to_target(argmax_lowest(logits))
    return {"draft_tokens": out_tok, "logits": out_logits, "appended": appended}


def next_context(drafts, accept, nxt, anchor_pos):
    """The next step's new rows after verification [UG: Inference Process,
    steps 3-4]: request b continues with its a_b accepted drafts and the
    target's token, at the positions after its anchor. Returns per request
    (tokens, positions)."""
    out_tok, out_pos = [], []
    for b in range(len(accept)):
        a = int(accept[b])
        toks = [int(t) for t in drafts[b, :a]] + [int(nxt[b])]
        out_tok.append(toks)
        out_pos.append([int(anchor_pos[b]) + 1 + j for j in range(a + 1)])
    return out_tok, out_pos


# --------------------------------------------------------------------------
# Training-shaped parallel forward  [PR: description, Changelog (core:
# PEagleTrainerModule), Equivalence to vLLM inference; UG: COD Sampling;
# RM: cu_seqlens isolation]
# --------------------------------------------------------------------------
def train_rows(n, counts, sets):
    """Row list in depth-major order: depth 0 anchors 0..n-1, then each
    depth's kept anchors ascending. Returns (anchor [R], depth [R])."""
    anchors = np.concatenate([sets[d] for d in range(len(counts))]) if counts else np.zeros(0, np.int64)
    depths = np.concatenate([np.full(counts[d], d, dtype=np.int64) for d in range(len(counts))]) \
        if counts else np.zeros(0, np.int64)
    return anchors.astype(np.int64), depths


def conversation_bounds(cu_seqlens, n):
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    conv = np.zeros(n, dtype=np.int64)
    for c in range(len(cu) - 1):
        conv[cu[c]:cu[c + 1]] = c
    return conv, cu[conv], cu[conv + 1]


def train_allowed(anchor, depth, start):
    """Brute-force allowed mask over rows: row (i,d) reads row (j,d') iff
    (d' == 0 and start(i) <= j <= i) or (j == i and 1 <= d' <= d)."""
    a_q = anchor[:, None]
    a_k = anchor[None, :]
    d_q = depth[:, None]
    d_k = depth[None, :]
    s_q = start[anchor][:, None]
    ctx = (d_k == 0) & (a_k >= s_q) & (a_k <= a_q)
    chain = (a_k == a_q) & (d_k >= 1) & (d_k <= d_q)
    return ctx | chain


def train_attention_structured(q, k, v, a, d):
    """Depth-masked attention of one conversation's rows, per the definition:
    row (i, d) reads the depth-0 rows j <= i (all in this conversation) and
    its own chain rows (i, 1..d). Depth-0 keys are scored as one causal
    block; chain keys are gathered per row."""
    Rq, nq, hd = q.shape
    nkv = k.shape[1]
    g = nq // nkv
    scale = 1.0 / math.sqrt(hd)
    idx0 = np.flatnonzero(d == 0)
    a0 = a[idx0]
    Kmax = int(d.max()) + 1 if d.size else 1
    where = {(int(a[t]), int(d[t])): t for t in range(Rq)}
    # chain slot c (depth c+1) of row t, or -1
    chain = np.full((Rq, max(Kmax - 1, 1)), -1, dtype=np.int64)
    for t in range(Rq):
        for dd in range(1, int(d[t]) + 1):
            chain[t, dd - 1] = where[(int(a[t]), dd)]
    causal = a0[None, :] <= a[:, None]                       # [Rq, m]
    has_chain = chain >= 0
    out = np.zeros((Rq, nq, hd))
    for h in range(nq):
        kh, vh = k[:, h // g, :], v[:, h // g, :]
        s0 = np.where(causal, (q[:, h, :] @ kh[idx0].T) * scale, -np.inf)
        kc = kh[np.maximum(chain, 0)]                          # [Rq, C, hd]
        vc = vh[np.maximum(chain, 0)]
        sc = np.where(has_chain, np.einsum("rd,rcd->rc", q[:, h, :], kc) * scale, -np.inf)
        m = np.maximum(s0.max(-1), sc.max(-1))[:, None]
        p0 = np.where(causal, np.exp(s0 - m), 0.0)
        pc = np.where(has_chain, np.exp(sc - m), 0.0)
        z = p0.sum(-1, keepdims=True) + pc.sum(-1, keepdims=True)
        out[:, h, :] = (p0 @ vh[idx0] + np.einsum("rc,rcd->rd", pc, vc)) / z
    return out


def row_labels(n, K, r, r_min, seed, cu_seqlens, labels, loss_mask=None, t2d=None):
    """Draft-vocab label of every training row (depth-major order), -1 where
    the row has none: labels[i+d] if i+d is inside anchor i's conversation,
    not masked out, and mapped into the draft vocab."""
    counts, sets = cod_select(n, K, r, r_min, seed)
    anchor, depth = train_rows(n, counts, sets)
    _, _, end = conversation_bounds(cu_seqlens, n)
    labels = np.asarray(labels, dtype=np.int64)
    out = np.full(len(anchor), -1, dtype=np.int64)
    for t in range(len(anchor)):
        p = int(anchor[t] + depth[t])
        if p >= end[anchor[t]]:
            continue
        if loss_mask is not None and not loss_mask[p]:
            continue
        lab = int(labels[p]) if t2d is None else int(t2d[int(labels[p])])
        if lab >= 0:
            out[t] = lab
    return out, counts


def parallel_forward(model: DraftModel, aux, input_ids, position_ids, cu_seqlens, labels,
                     loss_mask, K, r, r_min, seed, depth_decay=0.8,
                     conversations=None, keep_logits=True, keep_kv=False, dense_rows=False):
    """Training-shaped forward over one packed sequence.

    Returns dict with counts, sets, row anchors/depths (all R rows), and for
    the computed rows: row_ce (nan where the row has no label), row_label
    (-1 where none), row_argmax, logits; and, when every conversation was
    computed, per-depth loss / accuracy / valid counts and the total loss.
    ``conversations`` restricts the computation to whole conversations
    (exact: conversations never attend to one another).
    ``keep_kv`` also returns each layer's post-RoPE (k, v) of every row.
    ``dense_rows`` runs all rows as one batch under one brute-force boolean
    mask (tiny inputs only)."""
    c = model.cfg
    n = len(input_ids)
    counts, sets = cod_select(n, K, r, r_min, seed)
    anchor, depth = train_rows(n, counts, sets)
    R = len(anchor)
    conv, start, end = conversation_bounds(cu_seqlens, n)
    S = len(cu_seqlens) - 1
    todo = list(range(S)) if conversations is None else list(conversations)
    ptd = c["ptd_token_id"]
    Vd = c["draft_vocab"]
    nkv, hd = c["num_kv_heads"], c["head_dim"]
    h_mask = model.masked_hidden()
    aux = np.asarray(aux, dtype=np.float64)
    ids = np.asarray(input_ids, dtype=np.int64)
    posn = np.asarray(position_ids, dtype=np.int64)
    labels = np.asarray(labels, dtype=np.int64)

    row_ce = np.full(R, np.nan)
    row_label = np.full(R, -1, dtype=np.int64)
    row_argmax = np.full(R, -1, dtype=np.int64)
    logits_all = np.zeros((R, Vd)) if keep_logits else None
    kv = [(np.zeros((R, nkv, hd)), np.zeros((R, nkv, hd))) for _ in range(c["num_layers"])] \
        if keep_kv else None

    if dense_rows:
        groups = [np.arange(R)]
    else:
        groups = []
        for cv in todo:
            s_, e_ = int(cu_seqlens[cv]), int(cu_seqlens[cv + 1])
            groups.append(np.flatnonzero((anchor >= s_) & (anchor < e_)))

    for sel in groups:
        if sel.size == 0:
            continue
        a = anchor[sel]
        d = depth[sel]
        toks = np.where(d == 0, ids[a], ptd)
        hproj = model.project_hidden(aux[a])
        h = np.where((d == 0)[:, None], hproj, h_mask[None, :])
        emb = model.embed[toks]
        pos = posn[a] + d
        if dense_rows:
            allowed = train_allowed(a, d, start)
            attend = lambda q, k, v: masked_attention(q, k, v, allowed)
        else:
            attend = lambda q, k, v: train_attention_structured(q, k, v, a, d)
        for l in range(c["num_layers"]):
            h, kl, vl = model.layer(l, h, emb, pos, attend)
            if keep_kv:
                kv[l][0][sel] = kl
                kv[l][1][sel] = vl
        logits = model.head(h)
        am = argmax_lowest(logits)
        p = a + d
        e = end[a]
        lab = np.full(sel.size, -1, dtype=np.int64)
        for t in range(sel.size):
            pi = int(p[t])
            if pi >= e[t]:
                continue                       # label past the conversation end
            if loss_mask is not None and not loss_mask[pi]:
                continue
            tl = int(labels[pi])
            tl = tl if model.t2d is None else int(model.t2d[tl])
            if tl >= 0:                        # inside the draft vocab
                lab[t] = tl
        lse = logsumexp(logits)
        ce = np.full(sel.size, np.nan)
        ok = np.flatnonzero(lab >= 0)
        ce[ok] = lse[ok] - logits[ok, lab[ok]]
        row_ce[sel] = ce
        row_label[sel] = lab
        row_argmax[sel] = am
        if keep_logits:
            logits_all[sel] = logits

    res = {"counts": counts, "sets": sets, "anchor": anchor, "depth": depth,
           "row_ce": row_ce, "row_label": row_label, "row_argmax": row_argmax,
           "logits": logits_all}
    if keep_kv:
        res["kv"] = kv
    if conversations is None:
        loss_d = np.zeros(K)
        acc_d = np.zeros(K)
        valid_d = np.zeros(K, dtype=np.int64)
        for dd in range(K):
            m = (depth == dd) & (row_label >= 0)
            valid_d[dd] = int(m.sum())
            if valid_d[dd]:
                loss_d[dd] = float(np.mean(row_ce[m]))
                acc_d[dd] = float(np.mean(row_argmax[m] == row_label[m]))
        # 0.8^d-weighted sum of per-depth means  [PR: Changelog]
        res["per_depth_loss"] = loss_d
        res["per_depth_acc"] = acc_d
        res["per_depth_valid"] = valid_d
        res["loss"] = float(sum(depth_decay ** dd * loss_d[dd] for dd in range(K)))
    return res


# --------------------------------------------------------------------------
# A batch of packed sequences  [PR: Validation (8-GPU training), Changelog
# (0.8**d weighted-mean schedule)]: the loss of a batch averages each depth's
# CE over the labelled rows of every sequence, then weights the depths.
# --------------------------------------------------------------------------
def depth_sums(res, K):
    """[3, K] of one forward's result: sum of CE over labelled rows, labelled
    rows whose argmax is the label, labelled rows -- per depth."""
    out = np.zeros((3, K))
    for d in range(K):
        m = (res["depth"] == d) & (res["row_label"] >= 0)
        out[0, d] = float(np.sum(res["row_ce"][m]))
        out[1, d] = float(np.sum(res["row_argmax"][m] == res["row_label"][m]))
        out[2, d] = float(np.sum(m))
    return out


def loss_from_depth_sums(sums, decay=0.8):
    """Per-depth mean CE, accuracy and count, and sum_d decay^d * mean_d (a
    depth without labelled rows contributes 0)."""
    sums = np.asarray(sums, dtype=np.float64)
    K = sums.shape[1]
    C = sums[2]
    loss_d = np.where(C > 0, sums[0] / np.maximum(C, 1), 0.0)
    acc_d = np.where(C > 0, sums[1] / np.maximum(C, 1), 0.0)
    loss = float(sum(decay ** d * loss_d[d] for d in range(K)))
    return {"per_depth_loss": loss_d, "per_depth_acc": acc_d, "per_depth_valid": C.astype(np.int64),
            "loss": loss}


# --------------------------------------------------------------------------
# Gradients of the training loss  [PR: description and Changelog -- the
# trainer runs the parallel masked-depth loss; "loss decreases" test]
# The loss of parallel_forward written once more with float64 torch tensors,
# and differentiated by autograd. The embedding is frozen (the draft reuses
# the target's token embedding); every other weight gets a gradient:
# fc_w, fc_norm_w, mask_hidden, final_norm_w, lm_head_w and every layer's
# weights. All rows attend under one dense mask (train_allowed), so this is
# for small inputs.
# --------------------------------------------------------------------------
GRAD_KEYS = ("fc_w", "fc_norm_w", "mask_hidden", "final_norm_w", "lm_head_w")
LAYER_GRAD_KEYS = ("in_norm_w", "hidden_norm_w", "qkv_w", "o_w", "post_norm_w", "gate_up_w", "down_w")


def parallel_loss_torch(model: DraftModel, aux, input_ids, position_ids, cu_seqlens, labels, loss_mask,
                        K, r, r_min, seed, depth_decay=0.8, params=None):
    """Returns (loss, params): loss a float64 torch scalar, params the dict of
    leaf tensors (requires_grad) it was computed from, named like the weights
    (params["layers"][l][key])."""
    import torch
    t = lambda a: torch.tensor(np.asarray(a, dtype=np.float64))
    c = model.cfg
    if params is None:
        params = {k: t(getattr(model, k)).requires_grad_() for k in GRAD_KEYS}
        params["layers"] = [{k: t(L[k]).requires_grad_() for k in LAYER_GRAD_KEYS if L.get(k) is not None}
                            for L in model.layers]
    eps = c["rms_eps"]
    nq, nkv, hd, I = c["num_q_heads"], c["num_kv_heads"], c["head_dim"], c["intermediate"]
    n = len(input_ids)
    counts, sets = cod_select(n, K, r, r_min, seed)
    anchor, depth = train_rows(n, counts, sets)
    R = len(anchor)
    _, start, end = conversation_bounds(cu_seqlens, n)

    def norm(x, g):
        return x / torch.sqrt(torch.mean(x * x, dim=-1, keepdim=True) + eps) * g

    def project(a):
        return norm(a @ params["fc_w"].T, params["fc_norm_w"])

    def rope(x, pos):
        half = hd // 2
        inv = c["rope_theta"] ** (-(2.0 * np.arange(half)) / hd)
        ang = torch.tensor(np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :])
        cs, sn = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
        x1, x2 = x[..., :half], x[..., half:]
        return torch.cat([x1 * cs - x2 * sn, x2 * cs + x1 * sn], dim=-1)

    d0 = torch.tensor(depth == 0)
    hid = torch.where(d0[:, None], project(t(np.asarray(aux)[anchor])),
                      project(params["mask_hidden"].reshape(1, -1)).expand(R, -1))
    toks = np.where(depth == 0, np.asarray(input_ids)[anchor], c["ptd_token_id"])
    emb = t(model.embed[toks])
    pos = np.asarray(position_ids)[anchor] + depth
    allowed = torch.tensor(train_allowed(anchor, depth, start))
    scale = 1.0 / math.sqrt(hd)
    h = hid
    for l, L in enumerate(params["layers"]):
        if l == 0:
            hn = norm(hid, L["hidden_norm_w"])
            x = torch.cat([norm(emb, L["in_norm_w"]), hn], dim=-1)
            resid = hn if c["norm_before_residual"] else hid
        else:
            x = norm(h, L["in_norm_w"])
            resid = h
        qkv = x @ L["qkv_w"].T
        q = rope(qkv[:, :nq * hd].reshape(R, nq, hd), pos)
        k = rope(qkv[:, nq * hd:(nq + nkv) * hd].reshape(R, nkv, hd), pos)
        v = qkv[:, (nq + nkv) * hd:].reshape(R, nkv, hd)
        g = nq // nkv
        kk = k.repeat_interleave(g, dim=1)
        vv = v.repeat_interleave(g, dim=1)
        sc = torch.einsum("rhd,khd->hrk", q, kk) * scale
        sc = sc.masked_fill(~allowed[None], float("-inf"))
        o = torch.einsum("hrk,khd->rhd", torch.softmax(sc, dim=-1), vv).reshape(R, nq * hd)
        h1 = resid + o @ L["o_w"].T
        y = norm(h1, L["post_norm_w"])
        gu = y @ L["gate_up_w"].T
        a = torch.nn.functional.silu(gu[:, :I]) * gu[:, I:]
        h = h1 + a @ L["down_w"].T
    logits = norm(h, params["final_norm_w"]) @ params["lm_head_w"].T
    lab, _ = row_labels(n, K, r, r_min, seed, cu_seqlens, labels, loss_mask, model.t2d)
    lse = torch.logsumexp(logits, dim=-1)
    loss = torch.zeros((), dtype=torch.float64)
    for d in range(K):
        m = np.flatnonzero((depth == d) & (lab >= 0))
        if m.size:
            ce = lse[m] - logits[m, lab[m]]
            loss = loss + depth_decay ** d * ce.mean()
    return loss, params


def parallel_grads(model: DraftModel, **kw):
    """(loss, gradients) of parallel_loss_torch as float64 numpy arrays,
    named like the weights (grads["layers"][l][key])."""
    loss, params = parallel_loss_torch(model, **kw)
    loss.backward()
    grads = {k: params[k].grad.numpy() for k in GRAD_KEYS}
    grads["layers"] = [{k: v.grad.numpy() for k, v in L.items()} for L in params["layers"]]
    return float(loss.detach()), grads


def model_config(wl, norm_before_residual=True) -> dict:
    """Config dict for a synthetic workload description (attribute access)."""
    return {
        "hidden": wl.hidden, "target_hidden": wl.target_hidden, "num_aux": wl.num_aux,
        "num_layers": wl.num_layers, "num_q_heads": wl.num_q_heads,
        "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
        "intermediate": wl.intermediate, "target_vocab": wl.vocab, "draft_vocab": wl.vocab,
        "ptd_token_id": wl.ptd_token_id, "rope_theta": wl.rope_theta, "rms_eps": wl.rms_eps,
        "norm_before_residual": norm_before_residual,
    }
