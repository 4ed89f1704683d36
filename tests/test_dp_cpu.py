"""The data-parallel training split on two gloo ranks (CPU): each rank runs
its shard of a batch of packed sequences, the ranks exchange only their
per-depth sums in one all-reduce, and the combined loss must equal the
single-process result over the whole batch. The per-sequence forward here
is the CPU oracle; the sharding, the per-sequence COD seeds and the
exchange are the library's data-parallel code."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch():
    """Four tiny packed sequences (conversation lengths differ per sequence)."""
    wl = synth.WORKLOADS["tiny_f32_decode"].scaled(
        hidden=32, target_hidden=16, num_aux=3, num_layers=2, num_q_heads=4, num_kv_heads=2, head_dim=8,
        intermediate=48, vocab=64, K=4, kind="train", seed=77)
    seqs = []
    for i, lens in enumerate([(9, 1, 13), (17,), (5, 6, 7, 2), (30, 3)]):
        rng = np.random.default_rng(100 + i)
        n = sum(lens)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        seqs.append(dict(aux=rng.standard_normal((n, wl.num_aux * wl.target_hidden)),
                         input_ids=rng.integers(0, wl.vocab, n),
                         position_ids=np.concatenate([np.arange(l) for l in lens]).astype(np.int32),
                         cu_seqlens=cu, labels=rng.integers(0, wl.vocab, n), loss_mask=None))
    return wl, seqs


def _sums(wl, seqs, indices, base_seed):
    from eagle_speculative_drafting_gb300 import dp
    from oracle import peagle_oracle as O
    model = O.DraftModel(O.model_config(wl), synth.make_weights(wl))
    total = np.zeros((3, wl.K))
    for i in indices:
        res = O.parallel_forward(model, **seqs[i], K=wl.K, r=0.7, r_min=0.2, seed=dp.sequence_seed(base_seed, i))
        total += O.depth_sums(res, wl.K)
    return total


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import __graft_entry__
    __graft_entry__.build()
    from eagle_speculative_drafting_gb300 import dp
    from oracle import peagle_oracle as O
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl, seqs = _batch()
    mine = dp.shard(len(seqs), rank, world)
    sums = torch.from_numpy(_sums(wl, seqs, mine, 1234).reshape(-1)).clone()
    dp.allreduce_depth_sums(sums, dist)
    got = O.loss_from_depth_sums(sums.numpy().reshape(3, wl.K))
    q.put((rank, mine, got["loss"], got["per_depth_loss"].tolist(), got["per_depth_valid"].tolist()))
    dist.destroy_process_group()


def test_two_gloo_ranks_give_the_single_process_batch_loss():
    import __graft_entry__
    __graft_entry__.build()
    from oracle import peagle_oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl, seqs = _batch()
    ref = O.loss_from_depth_sums(_sums(wl, seqs, range(len(seqs)), 1234))
    assert sorted(out[0][1] + out[1][1]) == list(range(len(seqs)))    # a partition
    assert not set(out[0][1]) & set(out[1][1])
    for rank, mine, loss, loss_d, valid in out:
        assert loss == pytest.approx(ref["loss"], abs=1e-12)
        assert np.allclose(loss_d, ref["per_depth_loss"], atol=1e-12)
        assert valid == ref["per_depth_valid"].tolist()


def test_shards_and_seeds():
    import __graft_entry__
    __graft_entry__.build()
    from eagle_speculative_drafting_gb300 import dp
    assert dp.shard(5, 0, 2) == [0, 2, 4] and dp.shard(5, 1, 2) == [1, 3]
    assert dp.shard(3, 2, 4) == [2] and dp.shard(3, 3, 4) == []
    with pytest.raises(ValueError):
        dp.shard(3, 2, 2)
    seeds = {dp.sequence_seed(7, i) for i in range(1000)}
    assert len(seeds) == 1000 and all(0 <= s < 2 ** 64 for s in seeds)
    t = torch.arange(6, dtype=torch.float64)
    assert dp.allreduce_depth_sums(t) is t   # no process group: identity
