"""Host-side logic for running the attention forward on several GPUs.

Attention heads are independent, so the forward pass partitions with no
data-path exchange: each rank owns whole (batch, head) units or, for weak
scaling, its own batch.  One partitioning does need an exchange: splitting
one long key sequence across ranks (split-KV).  Each rank then returns a
partial (O_r, LSE_r) over its key range and the ranks merge them with
LSE = ln Σ_r exp(LSE_r) and O = Σ_r exp(LSE_r − LSE)·O_r.  The pages describe
single-GPU tiling only; this module holds the plans and the small collectives
(torch.distributed, any backend) and is exercised on CPU ranks with gloo.
"""

from __future__ import annotations

import torch
import torch.distributed as dist


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of a rank's independent batch under weak scaling."""
    return base_seed + 1000 * rank


def shard_range(n: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous [start, stop) share of n units for `rank` (sizes differ by ≤ 1)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_heads(B: int, H: int, world: int, rank: int) -> list[tuple[int, int]]:
    """(batch, head) units owned by `rank` when B·H heads are split across ranks."""
    a, b = shard_range(B * H, world, rank)
    return [(u // H, u % H) for u in range(a, b)]


def split_keys(Sk: int, world: int, rank: int, block: int = 128) -> tuple[int, int]:
    """Key range [start, stop) of `rank` under split-KV, cut at key-block edges."""
    nb = (Sk + block - 1) // block
    a, b = shard_range(nb, world, rank)
    return min(a * block, Sk), min(b * block, Sk)


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank scalar (timings are reported as the slowest rank)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def merge_partials(o_parts: torch.Tensor, lse_parts: torch.Tensor):
    """Merge split-KV partials.

    o_parts [R, ..., n, d] and lse_parts [R, ..., n] (natural-log LSE of each
    part's key range, −inf where the range holds no visible key).  Returns the
    merged (O [..., n, d], LSE [..., n]) in float32/float64 as given.
    """
    m = lse_parts.max(dim=0).values
    finite = torch.isfinite(m)
    shift = torch.where(finite, m, torch.zeros_like(m))
    w = torch.where(torch.isfinite(lse_parts), torch.exp(lse_parts - shift), torch.zeros_like(lse_parts))
    tot = w.sum(dim=0)
    safe = torch.where(tot > 0, tot, torch.ones_like(tot))
    lse = torch.where(finite, shift + torch.log(safe), torch.full_like(m, float("-inf")))
    o = (w / safe).unsqueeze(-1).mul(o_parts).sum(dim=0)
    return o, lse


def gather_merge(o_local: torch.Tensor, lse_local: torch.Tensor):
    """The split-KV exchange: all-gather every rank's partial and merge."""
    world = dist.get_world_size()
    os_ = [torch.empty_like(o_local) for _ in range(world)]
    ls_ = [torch.empty_like(lse_local) for _ in range(world)]
    dist.all_gather(os_, o_local.contiguous())
    dist.all_gather(ls_, lse_local.contiguous())
    return merge_partials(torch.stack(os_), torch.stack(ls_))
