"""KV-sequence sharding of the cascade decode across devices.

"Attention States and Recursive Attention", section "Applications": since
the merge operator is associative and commutative, the keys of a request can
be cut into parts that different devices attend to, and the parts' states
merged afterwards in any order.  Here every rank holds a contiguous part of
every request's keys -- a slice of each shared prefix and a page-aligned
slice of each request's cached suffix (``kv_shard_range``) -- and

1. computes the float32 state of its part (``cascade_decode_state``: the
   library's cascade, rounded nowhere),
2. all-gathers the states: one collective of B * Hq * (128 + 1) floats per
   rank, the only data that crosses devices,
3. merges the gathered states locally with one n-ary merge that rounds once
   into q's dtype (``merge_states_to``).

Every rank ends with the same final O and LSE.  The binding only marshals
arguments; the device work is the library's kernels and the collective.
"""
from __future__ import annotations

from . import cascade_decode_state, merge_states_to


def kv_shard_range(n_tokens: int, rank: int, world: int, align: int = 1):
    """Tokens [lo, hi) of a sequence of n_tokens that rank `rank` of `world`
    holds: contiguous, balanced in whole units of `align` tokens (a page, so
    that a suffix slice is whole pages of the request's block table), the
    last unit possibly partial.  The ranges of all ranks cover every token
    once, in rank order."""
    if world < 1 or not 0 <= rank < world or align < 1 or n_tokens < 0:
        raise ValueError("kv_shard_range: need 0 <= rank < world, align >= 1, n_tokens >= 0")
    units = (n_tokens + align - 1) // align
    u0, u1 = units * rank // world, units * (rank + 1) // world
    return min(n_tokens, u0 * align), min(n_tokens, u1 * align)


def gather_states(o, lse, group=None):
    """Every rank's state, in rank order: o [W, B, Hq, D], lse [W, B, Hq].

    One all-gather per tensor straight into the slices of the result (no
    staging copy).  Works with any torch.distributed backend (NCCL between
    GPUs, gloo for CPU tensors)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    o_all = torch.empty((world,) + tuple(o.shape), dtype=o.dtype, device=o.device)
    lse_all = torch.empty((world,) + tuple(lse.shape), dtype=lse.dtype, device=lse.device)
    dist.all_gather([o_all[r] for r in range(world)], o.contiguous(), group=group)
    dist.all_gather([lse_all[r] for r in range(world)], lse.contiguous(), group=group)
    return o_all, lse_all


def merge_gathered(o_all, lse_all, out_dtype, o=None, lse=None, stream=None):
    """(+) over the W gathered float32 states [W, B, Hq, D] / [W, B, Hq] into
    O [B, Hq, D] of out_dtype and LSE [B, Hq]: the rank-major layout is read
    as W states of one token with B * Hq heads, so one n-ary merge does it."""
    W, B, Hq, D = o_all.shape
    v = o_all.view(1, W, B * Hq, D)
    s = lse_all.view(1, W, B * Hq)
    vo = None if o is None else o.view(1, B * Hq, D)
    so = None if lse is None else lse.view(1, B * Hq)
    vo, so = merge_states_to(v, s, out_dtype, v_out=vo, s_out=so, stream=stream)
    return vo.view(B, Hq, D), so.view(B, Hq)


def kv_sharded_cascade_decode(q, k_prefix, v_prefix, prefix_kv_indptr, prefix_req_indptr, k_cache,
                              v_cache, block_table, cache_seqlens, sm_scale, workspace, group=None,
                              plan_buf=None, o=None, lse=None):
    """Cascade decode of requests whose keys are sharded over the ranks of
    `group` (the default process group if None; a single process without
    one runs alone).

    Each rank passes the same q [B, Hq, 128] and prefix grouping, and its own
    part of the keys: prefix slices k/v_prefix with their prefix_kv_indptr
    (a group may have no tokens on a rank), and a paged cache whose
    block_table / cache_seqlens list only this rank's suffix tokens (plan_buf,
    if given, is the plan of these lengths, uploaded into `workspace`).
    Returns the final O [B, Hq, 128] of q's dtype and LSE [B, Hq], the same
    on every rank: attention over the union of all ranks' keys."""
    import torch.distributed as dist
    o32, l32 = cascade_decode_state(q, k_prefix, v_prefix, prefix_kv_indptr, prefix_req_indptr,
                                    k_cache, v_cache, block_table, cache_seqlens, sm_scale, workspace,
                                    plan_buf=plan_buf)
    if dist.is_available() and dist.is_initialized():
        o_all, l_all = gather_states(o32, l32, group)
    else:
        o_all, l_all = o32.unsqueeze(0), l32.unsqueeze(0)
    return merge_gathered(o_all, l_all, q.dtype, o=o, lse=lse)
