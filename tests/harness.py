"""Glue shared by the GPU tests, smoke() and the benchmark: upload seeded
synthetic inputs, call the library through its C ABI, and run the CPU
oracle on the very same values."""
import numpy as np
import torch

import eagle_speculative_drafting_gb300 as pe
from oracle import peagle_oracle as O


def tdtype(wl):
    return torch.bfloat16 if wl.dtype == "bf16" else torch.float32


def dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def weights_to_device(wl, W):
    dt = tdtype(wl)
    out = {}
    for k, v in W.items():
        if k == "layers":
            out["layers"] = [{kk: (None if vv is None else dev(vv, dt)) for kk, vv in L.items()}
                             for L in v]
        elif k in ("d2t", "t2d"):
            out[k] = None if v is None else dev(np.asarray(v, dtype=np.int32))
        else:
            out[k] = dev(v, dt)
    return out


def config_of(wl, norm_before_residual=1):
    return pe.make_config(wl.hidden, wl.target_hidden, wl.num_aux, wl.num_layers, wl.num_q_heads,
                          wl.num_kv_heads, wl.head_dim, wl.intermediate, wl.vocab, wl.vocab,
                          wl.ptd_token_id, wl.dtype, norm_before_residual, wl.max_position,
                          wl.rope_theta, wl.rms_eps)


def make_model(wl, W, norm_before_residual=1):
    return pe.Model(config_of(wl, norm_before_residual), weights_to_device(wl, W))


def oracle_model(wl, W, norm_before_residual=True):
    cfg = O.model_config(wl, norm_before_residual)
    return O.DraftModel(cfg, W)


def upload_decode(wl, inp):
    dt = tdtype(wl)
    return {
        "aux": dev(inp["aux"], dt),
        "anchor_tokens": dev(inp["anchor_tokens"].astype(np.int32)),
        "anchor_pos": dev(inp["anchor_pos"].astype(np.int32)),
        "kv_offsets": dev(inp["kv_offsets"].astype(np.int64)),
        "kv_lens": dev(inp["kv_lens"].astype(np.int32)),
        "k_cache": [dev(k, dt) for k in inp["k_cache"]],
        "v_cache": [dev(v, dt) for v in inp["v_cache"]],
    }


def run_decode(wl, model, inp, want_logits=False, append=False, K=None, d=None):
    K = wl.K if K is None else K
    d = upload_decode(wl, inp) if d is None else d
    B = len(inp["anchor_tokens"])
    logits = torch.empty((B, K, wl.vocab), dtype=torch.float32, device="cuda") if want_logits else None
    toks = model.draft_step(K, d["aux"], d["anchor_tokens"], d["anchor_pos"], d["k_cache"],
                            d["v_cache"], d["kv_offsets"], d["kv_lens"], int(inp["kv_capacity"]),
                            int(np.max(inp["kv_lens"])) if B else 0, append, logits=logits)
    torch.cuda.synchronize()
    out = {"draft_tokens": toks.cpu().numpy(), "dev": d}
    if want_logits:
        out["logits"] = logits.cpu().numpy().astype(np.float64)
    return out


def oracle_decode(wl, W, inp, K=None, requests=None, append=False):
    m = oracle_model(wl, W)
    K = wl.K if K is None else K
    return O.draft_step(m, inp["aux"], inp["anchor_tokens"], inp["anchor_pos"], inp["k_cache"],
                        inp["v_cache"], inp["kv_offsets"], inp["kv_lens"], K,
                        append_anchor_kv=append, requests=requests)


def run_verify(drafts, targets):
    d = torch.from_numpy(np.ascontiguousarray(drafts, dtype=np.int32)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(targets, dtype=np.int32)).cuda()
    B, K = d.shape
    a = torch.empty(B, dtype=torch.int32, device="cuda")
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    pe.peagle_verify_accept(B, K, d, t, a, n)
    torch.cuda.synchronize()
    return a.cpu().numpy(), n.cpu().numpy()


def upload_train(wl, inp):
    dt = tdtype(wl)
    d = {
        "aux": dev(inp["aux"], dt),
        "input_ids": dev(np.asarray(inp["input_ids"], dtype=np.int32)),
        "position_ids": dev(np.asarray(inp["position_ids"], dtype=np.int32)),
        "cu_seqlens": dev(np.asarray(inp["cu_seqlens"], dtype=np.int32)),
        "labels": dev(np.asarray(inp["labels"], dtype=np.int32)),
        "loss_mask": None if inp.get("loss_mask") is None else dev(np.asarray(inp["loss_mask"], dtype=np.uint8)),
    }
    return d


def run_train(wl, model, inp, K, r, r_min, seed, decay=0.8, want_logits=False, d=None):
    d = upload_train(wl, inp) if d is None else d
    n = len(inp["input_ids"])
    counts = pe.peagle_cod_counts(n, K, r, r_min)
    R = sum(counts)
    row_am = torch.empty(max(R, 1), dtype=torch.int32, device="cuda")
    row_ce = torch.empty(max(R, 1), dtype=torch.float32, device="cuda")
    logits = torch.empty((max(R, 1), wl.vocab), dtype=torch.float32, device="cuda") if want_logits else None
    out = model.parallel_forward(d["aux"], d["input_ids"], d["position_ids"], d["cu_seqlens"],
                                 d["labels"], K, r, r_min, seed, decay, loss_mask=d["loss_mask"],
                                 row_argmax=row_am, row_ce=row_ce, logits=logits)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["row_argmax"] = row_am.cpu().numpy()[:R]
    res["row_ce"] = row_ce.cpu().numpy()[:R].astype(np.float64)
    if want_logits:
        res["logits"] = logits.cpu().numpy()[:R].astype(np.float64)
    res["counts"] = counts
    return res


def max_abs_rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = float(np.max(np.abs(ref))) if ref.size else 1.0
    return float(np.max(np.abs(got - ref))) / max(scale, 1e-30) if ref.size else 0.0


def token_mismatches_explained(got_tokens, ref_logits, tol_frac=2e-2):
    """Draft tokens may differ from the oracle's only where the oracle's own
    top-1/top-2 margin is below tol_frac * max|logit| (near-ties under bf16)."""
    ref_tok = np.argmax(ref_logits, axis=-1)
    bad = []
    flat_got = np.asarray(got_tokens).reshape(-1)
    flat_ref = ref_tok.reshape(-1)
    flat_log = ref_logits.reshape(-1, ref_logits.shape[-1])
    scale = float(np.max(np.abs(ref_logits)))
    for i in np.flatnonzero(flat_got != flat_ref):
        row = np.sort(flat_log[i])
        margin = row[-1] - row[-2]
        if margin >= tol_frac * scale:
            bad.append((int(i), float(margin)))
    return bad
