"""Host-side marshalling for the library's callers: move numpy arrays to
device tensors, build the config and weight structs, call the ABI entry
points and bring results back as numpy arrays.

Nothing here computes any step of the method; every step runs in the
library's CUDA kernels. ``wl`` is any object with the attributes of a draft
configuration (hidden, target_hidden, num_aux, num_layers, num_q_heads,
num_kv_heads, head_dim, intermediate, vocab, ptd_token_id, dtype,
max_position, rope_theta, rms_eps).
"""
import numpy as np
import torch

from . import (peagle_cod_counts, peagle_draft_step_ctx, peagle_draft_step_ctx_workspace_size,
               peagle_verify_accept)
from .model import Model, make_config


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


def config_of(wl, norm_before_residual=1, draft_vocab=None):
    return make_config(wl.hidden, wl.target_hidden, wl.num_aux, wl.num_layers, wl.num_q_heads,
                       wl.num_kv_heads, wl.head_dim, wl.intermediate, wl.vocab,
                       wl.vocab if draft_vocab is None else draft_vocab, wl.ptd_token_id, wl.dtype,
                       norm_before_residual, wl.max_position, wl.rope_theta, wl.rms_eps)


def make_model(wl, W, norm_before_residual=1, draft_vocab=None):
    """A created model over device copies of the weight arrays in W."""
    if draft_vocab is None:
        draft_vocab = int(np.asarray(W["lm_head_w"]).shape[0])
    return Model(config_of(wl, norm_before_residual, draft_vocab), weights_to_device(wl, W))


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
    """One draft step; returns draft tokens (and logits) as numpy arrays and
    the device tensors used (key ``dev``)."""
    K = wl.K if K is None else K
    d = upload_decode(wl, inp) if d is None else d
    B = len(inp["anchor_tokens"])
    Vd = model.cfg.draft_vocab
    logits = torch.empty((B, K, Vd), dtype=torch.float32, device="cuda") if want_logits else None
    toks = model.draft_step(K, d["aux"], d["anchor_tokens"], d["anchor_pos"], d["k_cache"],
                            d["v_cache"], d["kv_offsets"], d["kv_lens"], int(inp["kv_capacity"]),
                            int(np.max(inp["kv_lens"])) if B else 0, append, logits=logits)
    torch.cuda.synchronize()
    out = {"draft_tokens": toks.cpu().numpy(), "dev": d}
    if want_logits:
        out["logits"] = logits.cpu().numpy().astype(np.float64)
    return out


def run_verify(drafts, targets):
    d = torch.from_numpy(np.ascontiguousarray(drafts, dtype=np.int32)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(targets, dtype=np.int32)).cuda()
    B, K = d.shape
    a = torch.empty(B, dtype=torch.int32, device="cuda")
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    peagle_verify_accept(B, K, d, t, a, n)
    torch.cuda.synchronize()
    return a.cpu().numpy(), n.cpu().numpy()


def upload_train(wl, inp):
    dt = tdtype(wl)
    return {
        "aux": dev(inp["aux"], dt),
        "input_ids": dev(np.asarray(inp["input_ids"], dtype=np.int32)),
        "position_ids": dev(np.asarray(inp["position_ids"], dtype=np.int32)),
        "cu_seqlens": dev(np.asarray(inp["cu_seqlens"], dtype=np.int32)),
        "labels": dev(np.asarray(inp["labels"], dtype=np.int32)),
        "loss_mask": None if inp.get("loss_mask") is None else dev(np.asarray(inp["loss_mask"], dtype=np.uint8)),
    }


def run_train(wl, model, inp, K, r, r_min, seed, decay=0.8, want_logits=False, d=None,
              logit_rows=None):
    """One training-shaped forward; per-depth outputs and per-row results as
    numpy arrays. ``logit_rows`` (row indices) limits the logits copied back
    to those rows, in that order."""
    d = upload_train(wl, inp) if d is None else d
    n = len(inp["input_ids"])
    counts = peagle_cod_counts(n, K, r, r_min)
    R = sum(counts)
    Vd = model.cfg.draft_vocab
    row_am = torch.empty(max(R, 1), dtype=torch.int32, device="cuda")
    row_ce = torch.empty(max(R, 1), dtype=torch.float32, device="cuda")
    logits = torch.empty((max(R, 1), Vd), dtype=torch.float32, device="cuda") if want_logits else None
    out = model.parallel_forward(d["aux"], d["input_ids"], d["position_ids"], d["cu_seqlens"],
                                 d["labels"], K, r, r_min, seed, decay, loss_mask=d["loss_mask"],
                                 row_argmax=row_am, row_ce=row_ce, logits=logits)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["row_argmax"] = row_am.cpu().numpy()[:R]
    res["row_ce"] = row_ce.cpu().numpy()[:R].astype(np.float64)
    if want_logits:
        if logit_rows is not None:
            sel = torch.as_tensor(np.asarray(logit_rows, dtype=np.int64), device="cuda")
            res["logits"] = logits.index_select(0, sel).cpu().numpy().astype(np.float64)
        else:
            res["logits"] = logits.cpu().numpy()[:R].astype(np.float64)
    res["counts"] = counts
    return res


def run_decode_ctx(wl, model, new_aux, new_tokens, new_pos, d, kv_lens, kv_capacity, max_kv_len,
                   want_logits=False, K=None):
    """One draft step over new context rows: per request b, new_aux[b]
    [n_b, A*Ht], new_tokens[b] and new_pos[b] (n_b each). ``d`` holds the
    device caches and kv_offsets (as upload_decode returns); kv_lens is a
    host array. The new rows' K/V are appended to the caches."""
    K = wl.K if K is None else K
    B = len(new_tokens)
    n = np.array([len(t) for t in new_tokens], dtype=np.int32)
    off = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    total, max_new = int(off[-1]), int(n.max())
    aux = dev(np.concatenate([np.asarray(a, dtype=np.float32).reshape(len(t), -1)
                              for a, t in zip(new_aux, new_tokens)]), tdtype(wl))
    tok = dev(np.concatenate([np.asarray(t, dtype=np.int32) for t in new_tokens]))
    pos = dev(np.concatenate([np.asarray(p, dtype=np.int32) for p in new_pos]))
    Vd = model.cfg.draft_vocab
    drafts = torch.empty((B, K), dtype=torch.int32, device="cuda")
    logits = torch.empty((B, K, Vd), dtype=torch.float32, device="cuda") if want_logits else None
    nbytes = peagle_draft_step_ctx_workspace_size(model.handle, B, K, total, max_new, max_kv_len)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    peagle_draft_step_ctx(model.handle, B, K, total, max_new, dev(off), aux, tok, pos, d["k_cache"], d["v_cache"],
                          d["kv_offsets"], dev(np.asarray(kv_lens, dtype=np.int32)), int(kv_capacity), max_kv_len,
                          1, drafts, logits, ws, nbytes)
    torch.cuda.synchronize()
    out = {"draft_tokens": drafts.cpu().numpy()}
    if want_logits:
        out["logits"] = logits.cpu().numpy().astype(np.float64)
    return out
