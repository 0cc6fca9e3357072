"""Multi-GPU layouts.

Replicas: decode rows of different requests never interact, so the batch
partitions by request with no data-path collective: rank k of N decodes requests
[start_k, end_k).  Timing across ranks takes the maximum (the slowest rank ends
the step); that reduction is the only collective and it sits outside the path.

Decode context parallelism (the kv_balanced_mla kernel page: cp_world, cp_rank,
cp_interleave_size): every sequence's keys are dealt to the ranks in runs of
cp_interleave positions; each rank decodes its own keys under the whole
sequence's bounds (PagedMlaDecoder with cp_* set, its global_seq_lens given),
the ranks exchange their (O, LSE) shares with one all-gather (dcp_exchange), and
mla_merge combines them (api.merge_ranks, dcp_decode).
"""

from __future__ import annotations

import torch


def shard_rows(B: int, world: int, rank: int) -> tuple:
    """Contiguous, balanced request range [start, end) of `rank` among `world` ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world / rank")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def rank_seed(seed: int, rank: int) -> int:
    """Seed of rank's own batch when every rank decodes a full batch (weak scaling)."""
    return seed + 1000003 * rank


def max_over_ranks(value: float) -> float:
    """Maximum of a host scalar over all ranks (identity when not distributed)."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dcp_exchange(out: torch.Tensor, lse: torch.Tensor, group=None):
    """All-gather this rank's share of a context-parallel decode.

    out [B, Sq, H, 512] and lse [B, Sq, H] (natural log, -inf where the rank saw no
    visible key) become o_parts [world, B, Sq, H, 512] and lse_parts [world, B, Sq, H]
    in rank order, the layout mla_merge takes.  Works on any backend (NCCL on GPUs,
    gloo on CPU tensors).
    """
    import torch.distributed as dist

    world = dist.get_world_size(group)
    o_parts = torch.empty((world,) + tuple(out.shape), dtype=out.dtype, device=out.device)
    lse_parts = torch.empty((world,) + tuple(lse.shape), dtype=lse.dtype, device=lse.device)
    if out.is_cuda:  # NCCL gathers into one tensor
        dist.all_gather_into_tensor(o_parts, out.contiguous(), group=group)
        dist.all_gather_into_tensor(lse_parts, lse.contiguous(), group=group)
    else:  # gloo gathers into a list (views of the same tensors)
        dist.all_gather(list(o_parts.unbind(0)), out.contiguous(), group=group)
        dist.all_gather(list(lse_parts.unbind(0)), lse.contiguous(), group=group)
    return o_parts, lse_parts


def dcp_decode(decoder, inputs: dict, global_seq_lens: torch.Tensor, group=None, stream=None):
    """One context-parallel decode step on this rank's GPU: the local decode (fp32 out),
    the exchange, and the merge.  Returns (out, lse) of the whole decode, on every rank."""
    from .api import merge_ranks

    out, lse = decoder(inputs["q_latent"], inputs["q_rope"], inputs["ckv"], inputs["kpe"], inputs["page_table"],
                       inputs["seq_lens"], inputs["scale"], stream=stream, global_seq_lens=global_seq_lens)
    o_parts, lse_parts = dcp_exchange(out, lse, group)
    return merge_ranks(o_parts, lse_parts, stream=stream)
