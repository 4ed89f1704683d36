"""Parity at the workloads' full sizes, in the launch configuration the
benchmark uses (the same draft_step / verify / parallel_forward calls).

Where the oracle cannot run the whole workload in seconds it computes a
sample that is exact on its own: whole requests (decode requests are
independent) or whole conversations (packed conversations never attend to
one another). Row-wise outputs of the sample are compared element by
element; per-depth label counts are compared for every row.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import peagle_oracle as O

pytestmark = pytest.mark.gpu
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


def test_decode_b1_ctx2048_k4_full():
    wl = synth.WORKLOADS["decode_b1_ctx2048_k4"]
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl)
    model = H().make_model(wl, W)
    got = H().run_decode(wl, model, inp, want_logits=True)
    ref = H().oracle_decode(wl, W, inp)
    err = H().max_abs_rel(got["logits"], ref["logits"])
    assert err <= BF16_TOL, err
    assert np.array_equal(got["draft_tokens"], np.argmax(got["logits"], -1))
    assert not H().token_mismatches_explained(got["draft_tokens"], ref["logits"])
    # greedy verify of the GPU's own drafts against geometric-accept targets,
    # on the GPU and in the oracle (the same drafts go to both)
    acc = synth.draw_accept_lengths(wl, wl.batch, wl.K)
    tgt = synth.make_targets_with_accept(wl, got["draft_tokens"], acc)
    a, n = H().run_verify(got["draft_tokens"], tgt)
    ra, rn = O.verify_accept(got["draft_tokens"], tgt)
    assert np.array_equal(a, ra) and np.array_equal(n, rn)
    assert np.array_equal(a, acc)
    import eagle_speculative_drafting_gb300 as pe
    assert pe.peagle_get_device_status(model.handle) == 0
    model.close()


def test_decode_b64_ragged_k8_sampled_requests():
    wl = synth.WORKLOADS["decode_b64_ragged_k8"]
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl)
    model = H().make_model(wl, W)
    got = H().run_decode(wl, model, inp, want_logits=True)
    lens = inp["kv_lens"]
    sample = sorted({0, int(np.argmax(lens)), int(np.argmin(lens)), wl.batch - 1})
    ref = H().oracle_decode(wl, W, inp, requests=sample)
    for b in sample:
        err = H().max_abs_rel(got["logits"][b], ref["logits"][b])
        assert err <= BF16_TOL, (b, err)
        assert not H().token_mismatches_explained(got["draft_tokens"][b], ref["logits"][b]), b
    assert np.array_equal(got["draft_tokens"], np.argmax(got["logits"], -1))
    import eagle_speculative_drafting_gb300 as pe
    assert pe.peagle_get_device_status(model.handle) == 0
    model.close()


def check_train_conversations(wl, convs):
    """Full-size forward on the GPU; the oracle on whole conversations
    (exact on their own: conversations never attend to one another)."""
    W = synth.make_weights(wl)
    inp = synth.make_train_inputs(wl)
    model = H().make_model(wl, W)
    K, r, rmin, seed = inp["K"], inp["r"], inp["r_min"], inp["seed"]
    cu = inp["cu_seqlens"]
    n = wl.n_tokens
    counts, sets = O.cod_select(n, K, r, rmin, seed)
    anchor, depth = O.train_rows(n, counts, sets)
    conv_of_anchor = np.searchsorted(cu, anchor, side="right") - 1
    rows = np.flatnonzero(np.isin(conv_of_anchor, convs))
    got = H().run_train(wl, model, inp, K, r, rmin, seed, want_logits=True, logit_rows=rows)
    fwd_in = {k: inp[k] for k in ("aux", "input_ids", "position_ids", "cu_seqlens", "labels", "loss_mask")}
    ref = O.parallel_forward(H().oracle_model(wl, W), **fwd_in, K=K, r=r, r_min=rmin, seed=seed,
                             conversations=list(convs), keep_logits=True)
    assert np.array_equal(np.flatnonzero(ref["row_argmax"] >= 0), rows)
    assert H().max_abs_rel(got["logits"], ref["logits"][rows]) <= BF16_TOL
    lab = ref["row_label"][rows] >= 0
    lrows = rows[lab]
    assert H().max_abs_rel(got["row_ce"][lrows], ref["row_ce"][lrows]) <= BF16_TOL
    assert not H().token_mismatches_explained(got["row_argmax"][rows], ref["logits"][rows])
    # per-depth mean CE over the sampled conversations' rows: GPU rows against
    # the oracle's CE of the same rows
    for d in range(K):
        m = lrows[depth[lrows] == d]
        if m.size:
            g, o = float(np.mean(got["row_ce"][m])), float(np.mean(ref["row_ce"][m]))
            assert abs(g - o) <= BF16_TOL * max(1.0, abs(o)), (d, g, o)
    # every row's label presence, for the whole packed sequence
    labels, counts2 = O.row_labels(n, K, r, rmin, seed, cu, inp["labels"])
    assert got["counts"] == counts2 == counts
    want_valid = [int(np.sum((depth == d) & (labels >= 0))) for d in range(K)]
    assert got["per_depth_valid"].tolist() == want_valid
    assert np.all(np.isnan(got["row_ce"][labels < 0]))
    assert np.all(np.isfinite(got["row_ce"][labels >= 0]))
    # loss = sum_d 0.8^d * mean CE_d, from the GPU's own per-row values
    ce = got["row_ce"]
    means = [float(np.mean(ce[(depth == d) & (labels >= 0)])) for d in range(K)]
    assert np.allclose(got["per_depth_loss"], means, rtol=1e-4)
    assert abs(float(got["loss"][0]) - sum(0.8 ** d * means[d] for d in range(K))) < 1e-3
    import eagle_speculative_drafting_gb300 as pe
    assert pe.peagle_get_device_status(model.handle) == 0
    model.close()
    return rows


def test_train_n4096_k4_shortest_and_longest_conversations():
    # the shortest conversation (132 tokens: about one 128-key tile) and the
    # longest (889 tokens: many 128-key tiles of the tensor-core attention)
    wl = synth.WORKLOADS["train_n4096_k4"]
    cu = synth.make_train_inputs(wl)["cu_seqlens"]
    lens = np.diff(cu)
    rows = check_train_conversations(wl, [int(np.argmin(lens)), int(np.argmax(lens))])
    assert rows.size > 2000


def test_train_n32768_k8_sampled_conversation():
    # the long-context training workload: n = 32768, K = 8, H = 4096, four
    # layers; the oracle computes the shortest conversation (670 tokens)
    wl = synth.WORKLOADS["train_n32768_k8"]
    cu = synth.make_train_inputs(wl)["cu_seqlens"]
    check_train_conversations(wl, [int(np.argmin(np.diff(cu)))])
