"""Seeded generators for weights and per-call inputs.

Every tensor is drawn from its own NumPy PCG64 stream keyed by
(workload seed, tag, ...), so any one tensor (or one request's KV cache) can
be regenerated alone, in any order. Floating-point arrays come back as
float32; for bf16 workloads their values are already rounded to bf16
(round-to-nearest-even), so uploading them as bf16 is exact and the oracle
can upcast the very same values to float64.

Distributions (the plainest reading of the workload text):
  * linear weights, embedding, mask_hidden: N(0, 0.02^2)
  * RMSNorm gains: 1 + N(0, 0.02^2) (a pure N(0, 0.02) gain would make every
    norm degenerate)
  * aux hidden states and context K/V: N(0, 1)
  * token ids and labels: uniform over the vocabulary
"""
import zlib

import numpy as np

from .workloads import Workload


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _tag(s: str) -> int:
    return zlib.crc32(s.encode())


def _rng(wl: Workload, *key) -> np.random.Generator:
    parts = [wl.seed]
    for k in key:
        parts.append(_tag(k) if isinstance(k, str) else int(k))
    return np.random.default_rng(parts)


def _normal(wl, shape, std, *key):
    x = _rng(wl, *key).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return bf16_round(x) if wl.dtype == "bf16" else x


def _gain(wl, n, *key):
    x = np.float32(1.0) + _rng(wl, *key).standard_normal(n, dtype=np.float32) * np.float32(0.02)
    return bf16_round(x) if wl.dtype == "bf16" else x


def make_weights(wl: Workload) -> dict:
    """Random-init draft weights in nn.Linear layout ([out, in], row-major)."""
    H, A, Ht = wl.hidden, wl.num_aux, wl.target_hidden
    I, V = wl.intermediate, wl.vocab
    W = {
        "embed": _normal(wl, (V, H), 0.02, "embed"),
        "fc_w": _normal(wl, (H, A * Ht), 0.02, "fc_w"),
        "fc_norm_w": _gain(wl, H, "fc_norm_w"),
        "mask_hidden": _normal(wl, (1, A * Ht), 0.02, "mask_hidden"),
        "final_norm_w": _gain(wl, H, "final_norm_w"),
        "lm_head_w": _normal(wl, (V, H), 0.02, "lm_head_w"),
        "d2t": None,
        "t2d": None,
        "layers": [],
    }
    for l in range(wl.num_layers):
        in_dim = 2 * H if l == 0 else H
        L = {
            "in_norm_w": _gain(wl, H, "in_norm_w", l),
            "hidden_norm_w": _gain(wl, H, "hidden_norm_w", l) if l == 0 else None,
            "qkv_w": _normal(wl, (wl.qkv_out, in_dim), 0.02, "qkv_w", l),
            "o_w": _normal(wl, (H, wl.num_q_heads * wl.head_dim), 0.02, "o_w", l),
            "post_norm_w": _gain(wl, H, "post_norm_w", l),
            "gate_up_w": _normal(wl, (2 * I, H), 0.02, "gate_up_w", l),
            "down_w": _normal(wl, (H, I), 0.02, "down_w", l),
        }
        W["layers"].append(L)
    return W


def _kv_lens(wl: Workload) -> np.ndarray:
    if wl.kv_len_range is not None:
        lo, hi = wl.kv_len_range
        return _rng(wl, "kv_lens").integers(lo, hi + 1, size=wl.batch).astype(np.int32)
    return np.full(wl.batch, wl.kv_len, dtype=np.int32)


def make_request_cache(wl: Workload, layer: int, b: int, length: int):
    """Post-RoPE context K and V of one request at one layer: [length, nkv, hd]."""
    shape = (length, wl.num_kv_heads, wl.head_dim)
    k = _normal(wl, shape, 1.0, "k_cache", layer, b)
    v = _normal(wl, shape, 1.0, "v_cache", layer, b)
    return k, v


def make_decode_inputs(wl: Workload, with_cache: bool = True, spare: int = None) -> dict:
    """Per-call inputs of one draft step.

    Each request b owns cache rows [kv_offsets[b], kv_offsets[b+1]); its
    first kv_lens[b] rows hold context K/V, the rest (``spare`` rows, K by
    default) are free for appended anchor rows. anchor_pos = kv_lens.
    """
    B, K, V = wl.batch, wl.K, wl.vocab
    spare = K if spare is None else spare
    lens = _kv_lens(wl)
    cap = lens.astype(np.int64) + spare
    offsets = np.zeros(B + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(cap)
    out = {
        "aux": _normal(wl, (B, wl.num_aux * wl.target_hidden), 1.0, "aux"),
        "anchor_tokens": _rng(wl, "anchor_tokens").integers(0, V, size=B).astype(np.int32),
        "anchor_pos": lens.copy(),
        "kv_lens": lens,
        "kv_offsets": offsets,
        "kv_capacity": int(offsets[-1]),
    }
    if with_cache:
        total = int(offsets[-1])
        kc, vc = [], []
        for l in range(wl.num_layers):
            kl = np.zeros((total, wl.num_kv_heads, wl.head_dim), dtype=np.float32)
            vl = np.zeros_like(kl)
            for b in range(B):
                k, v = make_request_cache(wl, l, b, int(lens[b]))
                o = int(offsets[b])
                kl[o:o + lens[b]] = k
                vl[o:o + lens[b]] = v
            kc.append(kl)
            vc.append(vl)
        out["k_cache"] = kc
        out["v_cache"] = vc
    return out


def draw_accept_lengths(wl: Workload, B: int, K: int, salt: int = 0) -> np.ndarray:
    """Accept lengths in {0..K}: truncated geometric (each draft kept with
    probability accept_p until the first miss) or uniform."""
    rng = _rng(wl, "accept", salt)
    if wl.accept_uniform:
        return rng.integers(0, K + 1, size=B).astype(np.int32)
    keep = rng.random((B, K)) < wl.accept_p
    a = np.full(B, K, dtype=np.int32)
    for b in range(B):
        miss = np.flatnonzero(~keep[b])
        if miss.size:
            a[b] = miss[0]
    return a


def make_targets_with_accept(wl: Workload, drafts: np.ndarray, accept: np.ndarray,
                             salt: int = 0) -> np.ndarray:
    """Target tokens [B, K+1] that agree with ``drafts`` on exactly the first
    accept[b] depths: column accept[b] (if < K) differs from the draft, later
    columns and the bonus column are uniform."""
    drafts = np.asarray(drafts, dtype=np.int64)
    B, K = drafts.shape
    V = wl.vocab
    rng = _rng(wl, "targets", salt)
    t = rng.integers(0, V, size=(B, K + 1)).astype(np.int64)
    shift = rng.integers(1, V, size=B)
    for b in range(B):
        a = int(accept[b])
        t[b, :a] = drafts[b, :a]
        if a < K:
            t[b, a] = (drafts[b, a] + shift[b]) % V
    return t.astype(np.int32)


def _conv_lengths(wl: Workload) -> np.ndarray:
    rng = _rng(wl, "conv_lens")
    n = wl.n_tokens
    lens = []
    total = 0
    while total < n:
        if wl.conv_len_uniform is not None:
            lo, hi = wl.conv_len_uniform
            x = int(rng.integers(lo, hi + 1))
        else:
            med, sig = wl.conv_len_lognormal
            x = max(1, int(round(rng.lognormal(np.log(med), sig))))
        x = min(x, n - total)
        lens.append(x)
        total += x
    return np.asarray(lens, dtype=np.int32)


def make_train_inputs(wl: Workload) -> dict:
    """One packed sequence of n tokens split into conversations by cu_seqlens.

    Position ids restart at 0 in every conversation; labels are uniform
    token ids; every position is a loss position (no loss mask)."""
    n, V = wl.n_tokens, wl.vocab
    lens = _conv_lengths(wl)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    pos = np.concatenate([np.arange(l, dtype=np.int32) for l in lens])
    return {
        "aux": _normal(wl, (n, wl.num_aux * wl.target_hidden), 1.0, "aux_train"),
        "input_ids": _rng(wl, "input_ids").integers(0, V, size=n).astype(np.int32),
        "position_ids": pos,
        "cu_seqlens": cu,
        "labels": _rng(wl, "labels").integers(0, V, size=n).astype(np.int32),
        "loss_mask": None,
        "K": wl.K,
        "r": wl.cod_r,
        "r_min": wl.cod_r_min,
        "seed": 0x5EED0000 + wl.seed,
        "depth_decay": wl.depth_decay,
    }
