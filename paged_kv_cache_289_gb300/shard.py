"""Host-side shard plans for running one decode batch on several GPUs.

Decode attention has no exchange between its units (request, KV head): a unit reads
only its own request's pages of its own KV head, and the G query heads of the group
("深入LLM推理：从KV Cache到PD分离的Serving全景解析", "KV Cache：Transformer的循环状态":
grouped query heads share one KV head).  A batch therefore splits with no collective
on the data path, either

  * by requests (data parallel): each rank holds whole requests, their block tables,
    lengths and pages, and computes their output rows; or
  * by KV heads (tensor parallel over heads): each rank holds a contiguous range of KV
    heads of every request's pages, with the G query heads that use them.

Concatenating the ranks' outputs along requests (or along query heads) gives the
whole batch's output.  The plans here are pure arithmetic on host integers.
"""
from __future__ import annotations

import numpy as np


def plan_requests(seq_lens, world: int) -> list[tuple[int, int]]:
    """Contiguous request ranges [start, end), one per rank, balanced by cached tokens.

    A decode step reads every cached token of every request once, so the tokens are
    the work.  Rank k's range ends at the first request boundary where the running
    token count reaches (k + 1) / world of the total; ranges may be empty when there
    are fewer requests than ranks."""
    if world < 1:
        raise ValueError("world must be >= 1")
    lens = np.asarray(seq_lens, dtype=np.int64)
    if np.any(lens < 0):
        raise ValueError("negative sequence length")
    n = int(lens.shape[0])
    csum = np.concatenate([[0], np.cumsum(lens)])
    total = int(csum[-1])
    bounds = [0]
    for k in range(1, world):
        if total == 0:
            cut = (n * k) // world                  # no tokens: split by count
        else:
            target = total * k / world
            cut = int(np.searchsorted(csum, target, side="left"))
            # the boundary nearer the target, never before the previous one
            if 0 < cut <= n and target - csum[cut - 1] < csum[cut] - target:
                cut -= 1
        bounds.append(min(max(cut, bounds[-1]), n))
    bounds.append(n)
    return [(bounds[k], bounds[k + 1]) for k in range(world)]


def plan_kv_heads(num_kv_heads: int, world: int) -> list[tuple[int, int]]:
    """Contiguous KV-head ranges [h0, h1), one per rank, as even as the count allows
    (the first num_kv_heads % world ranks take one more).  A rank holding KV heads
    h0..h1-1 computes query heads h0*G .. h1*G - 1."""
    if world < 1 or num_kv_heads < 1:
        raise ValueError("world and num_kv_heads must be >= 1")
    base, extra = divmod(num_kv_heads, world)
    out, h = [], 0
    for k in range(world):
        w = base + (1 if k < extra else 0)
        out.append((h, h + w))
        h += w
    return out
