"""One attention problem partitioned across ranks (one process per GPU).

Query rows of different (batch, head) pairs never interact ("IO-aware exact
attention", section "Reference summary": the query blocks are independent), so
the forward needs no exchange when it is split by heads: rank r of `world`
computes heads [h0, h1) of every batch index on its own device and writes its
own slice of O and lse. An all-gather assembles the full O and lse on every rank
only when a caller asks for it.

Only host-side logic lives here: which heads a rank owns, slicing the inputs,
and assembling the gathered slices. The arithmetic of each slice is the caller's
`compute` function, by default the CUDA forward of this package on the rank's
current device.
"""
from __future__ import annotations

import math

import torch


def head_range(H: int, world: int, rank: int) -> tuple[int, int]:
    """Heads [h0, h1) owned by `rank`: contiguous, sizes differ by at most one, and
    together the ranks cover every head exactly once."""
    if world < 1 or not 0 <= rank < world or H < 1:
        raise ValueError("need H >= 1, world >= 1 and 0 <= rank < world")
    return rank * H // world, (rank + 1) * H // world


def max_heads(H: int, world: int) -> int:
    """The largest slice any rank owns (the padded size of a gathered slice)."""
    return max(h1 - h0 for h0, h1 in (head_range(H, world, r) for r in range(world)))


def shard_forward(q, k, v, mask, scale, causal, rank: int, world: int, compute):
    """This rank's slice of the forward: heads [h0, h1) of every batch index.

    q, k, v: [B][H][N][d]; mask: None or [B][N][N] (shared by the heads, so every
    rank reads all of it). `compute(q_s, k_s, v_s, mask, scale, causal)` returns
    (out_s [B][h1-h0][N][d], lse_s [B][h1-h0][N]). Returns (h0, h1, out_s, lse_s);
    a rank that owns no head returns empty slices."""
    B, H, N, d = q.shape
    h0, h1 = head_range(H, world, rank)
    if h1 == h0:
        return h0, h1, q.new_empty((B, 0, N, d)), torch.empty((B, 0, N), dtype=torch.float32, device=q.device)
    qs, ks, vs = (t[:, h0:h1].contiguous() for t in (q, k, v))
    out_s, lse_s = compute(qs, ks, vs, mask, scale, causal)
    return h0, h1, out_s, lse_s


def assemble(parts, B: int, H: int, N: int, d: int, dtype, device, lse_dtype=torch.float32):
    """Full O [B][H][N][d] and lse [B][H][N] from (h0, h1, out_s, lse_s) slices that
    cover every head once."""
    out = torch.empty((B, H, N, d), dtype=dtype, device=device)
    lse = torch.empty((B, H, N), dtype=lse_dtype, device=device)
    seen = torch.zeros(H, dtype=torch.int64)
    for h0, h1, o, l in parts:
        out[:, h0:h1] = o
        lse[:, h0:h1] = l
        seen[h0:h1] += 1
    if not bool((seen == 1).all()):
        raise ValueError("the slices do not cover every head exactly once")
    return out, lse


def gather(h0: int, h1: int, out_s, lse_s, H: int, world: int, group=None):
    """All-gather every rank's slice (padded to the largest slice, as all_gather
    needs equal shapes) and assemble the full O and lse on every rank."""
    import torch.distributed as dist

    B, _, N, d = out_s.shape
    hm = max_heads(H, world)
    o_pad = out_s.new_zeros((B, hm, N, d))
    l_pad = lse_s.new_zeros((B, hm, N))
    o_pad[:, :h1 - h0] = out_s
    l_pad[:, :h1 - h0] = lse_s
    o_all = [torch.empty_like(o_pad) for _ in range(world)]
    l_all = [torch.empty_like(l_pad) for _ in range(world)]
    dist.all_gather(o_all, o_pad, group=group)
    dist.all_gather(l_all, l_pad, group=group)
    parts = []
    for r in range(world):
        a, b = head_range(H, world, r)
        parts.append((a, b, o_all[r][:, :b - a], l_all[r][:, :b - a]))
    return assemble(parts, B, H, N, d, out_s.dtype, out_s.device, lse_s.dtype)


def _cuda_compute(q, k, v, mask, scale, causal):
    from . import fa

    return fa.attention(q, k, v, mask=mask, scale=scale, causal=causal)


def sharded_attention(q, k, v, mask=None, scale=None, causal=False, rank=None, world=None, group=None,
                      gather_result=True, compute=None):
    """The forward of one problem split by heads over the ranks of `group` (the
    default process group when rank/world are not given). Returns the full
    (O, lse) on every rank when `gather_result`, else this rank's
    (h0, h1, O slice, lse slice)."""
    if rank is None or world is None:
        import torch.distributed as dist

        rank, world = dist.get_rank(group), dist.get_world_size(group)
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else scale
    h0, h1, out_s, lse_s = shard_forward(q, k, v, mask, scale, causal, rank, world, compute or _cuda_compute)
    if not gather_result:
        return h0, h1, out_s, lse_s
    return gather(h0, h1, out_s, lse_s, q.shape[1], world, group)
