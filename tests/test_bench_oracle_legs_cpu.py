"""The oracle legs of bench.py on the host: the training baseline and the
reference arm time the oracle on a bounded sample of the workload (the
forward of the shortest conversation, or the gradients of its first 128
tokens as a packed sequence of their own). Checked here on a scaled-down
training workload, so a break in either leg shows without a GPU."""
import numpy as np

import bench
import synth
from oracle import peagle_oracle as O


def _small_train():
    wl = synth.WORKLOADS["train_n4096_k4"].scaled(
        hidden=64, target_hidden=32, num_aux=3, num_layers=2, num_q_heads=4, num_kv_heads=2, head_dim=16,
        intermediate=128, vocab=300, n_tokens=400, conv_len_uniform=(130, 200))
    return wl, synth.make_weights(wl), synth.make_train_inputs(wl)


def test_forward_leg_counts_the_rows_of_the_shortest_conversation():
    wl, W, inp = _small_train()
    v, steps, el, cores, sample = bench.oracle_train_leg(wl, W, inp, seconds=0.0, max_steps=1)
    cu = inp["cu_seqlens"]
    conv = int(np.argmin(np.diff(cu)))
    L = int(cu[conv + 1] - cu[conv])
    assert steps == 1 and el > 0 and cores >= 1
    rows = round(v * el / steps)
    # the conversation's rows: its tokens at depth 0 and the COD-selected
    # deeper rows that fall in it (at most K per token)
    assert L <= rows <= inp["K"] * L
    assert f"conversation {conv} ({L} tokens" in sample


def test_backward_leg_takes_the_first_128_tokens_as_their_own_sequence():
    wl, W, inp = _small_train()
    v, steps, el, cores, sample = bench.oracle_train_leg(wl, W, inp, seconds=0.0, max_steps=1, backward=True)
    cu = inp["cu_seqlens"]
    conv = int(np.argmin(np.diff(cu)))
    L = min(128, int(cu[conv + 1] - cu[conv]))
    rows = int(sum(O.cod_counts(L, inp["K"], inp["r"], inp["r_min"])))
    assert steps == 1 and el > 0
    assert abs(v * el - rows) < 1e-6 * rows
    assert f"first {L} tokens of conversation {conv}" in sample and f"({rows} rows)" in sample
