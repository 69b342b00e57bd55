"""Vocab-parallel (tensor-parallel) LM head over torch.distributed ranks.

The SkyRL pull request "Triton backend for fused LM-head log-prob" (its
chunked distributed log-prob) splits the vocabulary over tensor-parallel ranks
and exchanges per-row statistics between them. Here:

Forward. Each rank runs ``lmhead_logprob_fwd_partials`` on its shard, giving
the base-2 (max, sum, entropy accumulator) of every 1024-column vocabulary
chunk it holds and the label logit of the rows whose label it holds (0 for the
others). The ranks all-gather those chunk planes in rank order, which rebuilds
the whole vocabulary's planes, and sum the label logits (every row has exactly
one nonzero term, so the sum is exact in any order). ``lmhead_logprob_merge``
then folds the chunks in ascending order on every rank. Every rank gets the
same logprob, entropy and lse, bit-identical to ``lmhead_logprob_fwd`` on the
whole weight.

Backward. Each rank runs ``lmhead_logprob_bwd_shard`` with the merged lse: its
fp32 share of grad_hidden and its own rows of grad_weight (which need no
exchange). The ranks all-gather the grad_hidden shares in rank order and
``lmhead_sum_ranks_bf16`` adds them in that order and rounds once, so every rank
holds the same grad_hidden bits.

Shards: rank r holds rows [v_offset_r, v_offset_r + V_r) of the weight, in
rank order, each starting on a 1024-column chunk boundary (``shard_bounds``
gives such a split). This module only moves data between ranks and calls the
library; the arithmetic runs in the library's kernels. With the gloo backend
the exchanged tensors go through host memory; with NCCL they stay on the
device.
"""

from __future__ import annotations

from . import (lmhead_logprob_bwd_shard, lmhead_logprob_fwd_partials, lmhead_logprob_merge,
               lmhead_sum_ranks_bf16)

CHUNK = 1024  # vocabulary columns per forward partial


def _dist():
    import torch.distributed as dist

    return dist


def shard_bounds(V_total: int, world: int, rank: int) -> tuple[int, int]:
    """Rows [begin, end) of rank's shard: the 1024-column chunks dealt out in
    rank order, as evenly as they go (the first ranks take one more)."""
    n = -(-int(V_total) // CHUNK)
    if not 0 <= rank < world or world > n:
        raise ValueError(f"{world} ranks cannot each hold a {CHUNK}-column chunk of {V_total}")
    per, extra = divmod(n, world)
    c0 = rank * per + min(rank, extra)
    c1 = c0 + per + (1 if rank < extra else 0)
    return min(V_total, c0 * CHUNK), min(V_total, c1 * CHUNK)


def _comm_device(group, local_device):
    """Where the exchanged tensors live: host memory for gloo, else the device."""
    return "cpu" if _dist().get_backend(group) == "gloo" else local_device


def exchange_layout(v_offset: int, V_shard: int, V_total: int, group=None) -> list[int]:
    """Every rank's chunk count, after checking that the shards tile the
    vocabulary in rank order on chunk boundaries (raises ValueError if not)."""
    import torch

    dist = _dist()
    world = dist.get_world_size(group)
    mine = torch.tensor([int(v_offset), int(V_shard)], dtype=torch.int64)
    allv = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
    if dist.get_backend(group) != "gloo":
        mine = mine.cuda()
        allv = [a.cuda() for a in allv]
    dist.all_gather(allv, mine, group=group)
    pairs = [(int(a[0]), int(a[1])) for a in allv]
    expect = 0
    for r, (off, n) in enumerate(pairs):
        if off != expect or off % CHUNK != 0 or n < 1:
            raise ValueError(f"rank {r} holds rows [{off}, {off + n}); the shards must tile the "
                             f"vocabulary in rank order from 0, each starting on a multiple of "
                             f"{CHUNK}")
        expect = off + n
    if expect != V_total:
        raise ValueError(f"the shards cover {expect} vocabulary rows, not {V_total}")
    return [-(-n // CHUNK) for _, n in pairs]


def gather_chunks(planes, counts: list[int], group=None):
    """All-gather [P, n_r, T] chunk planes, concatenated along the chunk axis
    in rank order: [P, sum(counts), T], on the device of ``planes``."""
    import torch

    dist = _dist()
    dev = planes.device
    cdev = _comm_device(group, dev)
    P, n, T = planes.shape
    width = max(counts)
    buf = torch.zeros(P, width, T, dtype=planes.dtype, device=cdev)
    buf[:, :n].copy_(planes)
    got = [torch.empty_like(buf) for _ in counts]
    dist.all_gather(got, buf, group=group)
    whole = torch.cat([g[:, :c] for g, c in zip(got, counts)], dim=1)
    return whole.to(dev).contiguous()


def gather_ranks(x, group=None):
    """All-gather a tensor of the same shape from every rank: [world, ...] in
    rank order, on the device of ``x``."""
    import torch

    dist = _dist()
    dev = x.device
    cdev = _comm_device(group, dev)
    src = x.to(cdev).contiguous()
    got = [torch.empty_like(src) for _ in range(dist.get_world_size(group))]
    dist.all_gather(got, src, group=group)
    return torch.stack(got).to(dev)


def sum_label_logits(label_logit, group=None):
    """The label logits summed over ranks: each row has one nonzero term."""
    dist = _dist()
    dev = label_logit.device
    x = label_logit.to(_comm_device(group, dev)).clone()
    dist.all_reduce(x, op=dist.ReduceOp.SUM, group=group)
    return x.to(dev)


def vocab_parallel_logprob_fwd(hidden, weight_shard, labels, v_offset: int, V_total: int,
                               inv_temperature: float = 1.0, *, group=None):
    """(logprob, entropy, lse) f32 [T] of the whole vocabulary, the same bits
    on every rank and as lmhead_logprob_fwd on the whole weight.

    hidden bf16 [T, H] and labels int32 [T] (whole-vocabulary indices) are the
    same on every rank; weight_shard bf16 [V_r, H] is rows [v_offset,
    v_offset + V_r) of the head."""
    import torch

    T = hidden.shape[0]
    V = weight_shard.shape[0]
    counts = exchange_layout(v_offset, V, V_total, group)
    dev = hidden.device
    planes = torch.empty(3, -(-V // CHUNK), T, dtype=torch.float32, device=dev)
    label_logit = torch.empty(T, dtype=torch.float32, device=dev)
    lmhead_logprob_fwd_partials(hidden, weight_shard, labels, v_offset, inv_temperature,
                                part_m=planes[0], part_s=planes[1], part_u=planes[2],
                                label_logit=label_logit)
    whole = gather_chunks(planes, counts, group)
    label_logit = sum_label_logits(label_logit, group)
    return lmhead_logprob_merge(whole[0], whole[1], whole[2], label_logit, labels, V_total)


def vocab_parallel_logprob_bwd(hidden, weight_shard, labels, grad_logprob, lse, v_offset: int,
                               inv_temperature: float = 1.0, *, grad_entropy=None, entropy=None,
                               group=None):
    """(grad_hidden bf16 [T, H], the same bits on every rank; this rank's
    grad_weight rows f32 [V_r, H]). lse (and entropy, with grad_entropy) are
    the merged forward's."""
    part, grad_weight = lmhead_logprob_bwd_shard(hidden, weight_shard, labels, grad_logprob, lse,
                                                 v_offset, inv_temperature,
                                                 grad_entropy=grad_entropy, entropy=entropy)
    parts = gather_ranks(part, group)
    return lmhead_sum_ranks_bf16(parts), grad_weight
