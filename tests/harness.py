"""Test glue: the library's marshalling helpers (re-exported from the
package, which never imports the oracle) plus the oracle-side helpers the
parity tests and smoke() compare against."""
import numpy as np

from eagle_speculative_drafting_gb300.marshal import (  # noqa: F401  (re-exported for the tests)
    config_of, dev, make_model, run_decode, run_decode_ctx, run_train, run_verify, tdtype, upload_decode,
    upload_train, weights_to_device)
from oracle import peagle_oracle as O


def oracle_model(wl, W, norm_before_residual=True, draft_vocab=None):
    cfg = O.model_config(wl, norm_before_residual)
    cfg["draft_vocab"] = int(np.asarray(W["lm_head_w"]).shape[0]) if draft_vocab is None else draft_vocab
    return O.DraftModel(cfg, W)


def oracle_decode(wl, W, inp, K=None, requests=None, append=False, norm_before_residual=True):
    m = oracle_model(wl, W, norm_before_residual)
    K = wl.K if K is None else K
    return O.draft_step(m, inp["aux"], inp["anchor_tokens"], inp["anchor_pos"], inp["k_cache"],
                        inp["v_cache"], inp["kv_offsets"], inp["kv_lens"], K,
                        append_anchor_kv=append, requests=requests)


def max_abs_rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = float(np.max(np.abs(ref))) if ref.size else 1.0
    return float(np.max(np.abs(got - ref))) / max(scale, 1e-30) if ref.size else 0.0


def token_mismatches_explained(got_tokens, ref_logits, tol_frac=2e-2, d2t=None):
    """Draft tokens may differ from the oracle's only where the oracle's own
    top-1/top-2 margin is below tol_frac * max|logit| (near-ties under bf16).
    ``d2t`` maps draft ids to the token ids ``got_tokens`` holds."""
    ref_tok = np.argmax(ref_logits, axis=-1)
    if d2t is not None:
        ref_tok = np.asarray(d2t)[ref_tok]
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
