"""Data-parallel training-shaped forward over several GPUs ("feat(speculative)
... #2376", Validation: the drafter trained on 8 GPUs).

Packed sequences never attend to one another (cu_seqlens isolation), so the
batch splits by whole sequences: rank r runs sequences r, r + W, r + 2W, ...
of the global batch, each through peagle_parallel_forward, which adds that
sequence's per-depth sums (sum of CE, correct rows, labelled rows) to one
[3, K] float64 buffer. The ranks exchange that buffer in one all-reduce
(sum) -- the only data exchanged -- and peagle_combine_depth_sums turns it
into the per-depth means and the decay-weighted loss on every rank.

Each sequence's COD draw is seeded by its global index, so the result does
not depend on how many ranks share the batch.
"""
import torch

from . import peagle_combine_depth_sums

SEED_STRIDE = 0x9E3779B97F4A7C15


def shard(num_sequences: int, rank: int, world: int) -> list:
    """Global indices of the sequences rank `rank` of `world` runs."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    return list(range(rank, num_sequences, world))


def sequence_seed(base_seed: int, index: int) -> int:
    """COD seed of global sequence `index` of a batch."""
    return (base_seed + index * SEED_STRIDE) & ((1 << 64) - 1)


def allreduce_depth_sums(sums: torch.Tensor, dist=None) -> torch.Tensor:
    """Adds every rank's [3, K] depth sums in place (identity without a
    process group): the one collective of a data-parallel step."""
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(sums, op=dist.ReduceOp.SUM)
    return sums


class DataParallelForward:
    """One rank's share of a data-parallel training-shaped forward.

    ``model`` is a created eagle_speculative_drafting_gb300.Model; every
    sequence is a dict of device tensors (aux, input_ids, position_ids,
    cu_seqlens, labels, loss_mask or None)."""

    def __init__(self, model, K, r, r_min, base_seed, depth_decay=0.8, dist=None):
        self.model, self.K, self.r, self.r_min = model, K, r, r_min
        self.base_seed, self.decay, self.dist = base_seed, depth_decay, dist
        dev = dict(device="cuda")
        self.sums = torch.zeros(3 * K, dtype=torch.float64, **dev)
        self.out = {"per_depth_loss": torch.empty(K, dtype=torch.float32, **dev),
                    "per_depth_acc": torch.empty(K, dtype=torch.float32, **dev),
                    "per_depth_valid": torch.empty(K, dtype=torch.int32, **dev),
                    "loss": torch.empty(1, dtype=torch.float32, **dev)}

    def step(self, sequences, stream=None) -> dict:
        """sequences: list of (global index, sequence dict) this rank runs.
        Returns the batch's per-depth loss / accuracy / counts and the loss
        (device tensors, identical on every rank)."""
        self.sums.zero_()
        for index, sq in sequences:
            self.model.parallel_forward(sq["aux"], sq["input_ids"], sq["position_ids"], sq["cu_seqlens"],
                                        sq["labels"], self.K, self.r, self.r_min,
                                        sequence_seed(self.base_seed, index), self.decay,
                                        loss_mask=sq.get("loss_mask"), stream=stream, depth_sums=self.sums)
        allreduce_depth_sums(self.sums, self.dist)
        o = self.out
        peagle_combine_depth_sums(self.K, self.decay, self.sums, o["per_depth_loss"], o["per_depth_acc"],
                                  o["per_depth_valid"], o["loss"], stream)
        return o
