"""One long context split across devices: host logic of the sequence split.

"GLM-5.3-Flash on MI300X" (aiholics) contrasts replicating the KV cache on
every device (tensor parallel) with sharding it (data parallel): only the
sharded cache leaves room for long contexts.  Here one sequence's pages are
cut into consecutive shares, one per device.  Every device runs the split
stage of the decode on its own share; the partial outputs and log-sum-exps
(O_s, lse_s) are gathered into one device's memory and merged there by
kv4_split_combine, the same log-sum-exp merge that combines the splits of one
device.  The merge is exact whatever the grouping of the splits, so the result
is the attention over the whole sequence.

The device holding the newest tokens (the query positions of the step, causal
among themselves) calls kv4_decode_partials on its share; every other device
holds tokens that all precede the queries and calls
kv4_decode_partials_prefix.  The only exchange is one gather of
B*T*Hq*S*(D+1) floats per step.  No collective runs inside a kernel.
"""
from __future__ import annotations

import numpy as np
import torch


def share_ranges(context_lens, q_per_seq: int, world_size: int, page_size: int = 16) -> np.ndarray:
    """Token range [t0, t1) of every sequence's share on every device.

    Returns int64 [world_size, B, 2].  Shares are page-aligned and
    consecutive, and cover [0, L_b).  The last device's share holds the
    newest q_per_seq tokens (it starts at or before L_b - q_per_seq).  The
    pages before it are divided as evenly as whole pages allow among the
    other devices; shares may be empty for short sequences."""
    lens = np.asarray(context_lens, dtype=np.int64)
    if world_size < 1 or page_size < 1 or q_per_seq < 1:
        raise ValueError("world_size, page_size and q_per_seq must be positive")
    if (lens < q_per_seq).any():
        raise ValueError("every context must hold the q_per_seq new tokens")
    W, B = world_size, lens.size
    out = np.zeros((W, B, 2), dtype=np.int64)
    n_pages = (lens + page_size - 1) // page_size
    # the tail share starts at the even cut or earlier, so that it holds the new tokens
    tail_page = np.minimum((W - 1) * n_pages // W, (lens - q_per_seq) // page_size)
    for r in range(W - 1):
        p0 = r * tail_page // (W - 1)
        p1 = (r + 1) * tail_page // (W - 1)
        out[r, :, 0] = p0 * page_size
        out[r, :, 1] = p1 * page_size
    out[W - 1, :, 0] = tail_page * page_size
    out[W - 1, :, 1] = lens
    return out


def local_tables(block_tables: np.ndarray, ranges: np.ndarray, page_size: int = 16):
    """A device's page table and context lengths for its share.

    block_tables: int32 [B, max_pages] of the whole sequences; ranges: int64
    [B, 2] of this device's share (one row of share_ranges).  Returns
    (tables int32 [B, max_local_pages] holding the share's pages from column 0,
    lens int32 [B]).  In a deployment each device keeps only its share's pages
    in its own cache; the page ids here index that cache."""
    B = block_tables.shape[0]
    p0 = ranges[:, 0] // page_size
    p1 = (ranges[:, 1] + page_size - 1) // page_size
    width = max(1, int((p1 - p0).max()) if B else 1)
    tab = np.zeros((B, width), dtype=np.int32)
    for b in range(B):
        n = int(p1[b] - p0[b])
        tab[b, :n] = block_tables[b, p0[b]:p0[b] + n]
    return tab, (ranges[:, 1] - ranges[:, 0]).astype(np.int32)


def gather_partials(partial_o: torch.Tensor, partial_lse: torch.Tensor, group=None, dst: int = 0):
    """Gather every device's split partials onto device `dst`.

    partial_o: fp32 [B, T, Hq, S, D], partial_lse: fp32 [B, T, Hq, S] (the
    same S on every device).  On dst returns the partials of all devices
    concatenated along the split axis, device order (fp32 [B, T, Hq, W*S, D]
    and [B, T, Hq, W*S]), ready for kv4_split_combine; elsewhere returns
    (None, None).  One torch.distributed gather per tensor, into dst's own
    memory."""
    import torch.distributed as dist
    W = dist.get_world_size(group)
    rank = dist.get_rank(group)
    po = partial_o.contiguous()
    pl = partial_lse.contiguous()
    bufs_o = [torch.empty_like(po) for _ in range(W)] if rank == dst else None
    bufs_l = [torch.empty_like(pl) for _ in range(W)] if rank == dst else None
    dist.gather(po, bufs_o, dst=dst, group=group)
    dist.gather(pl, bufs_l, dst=dst, group=group)
    if rank != dst:
        return None, None
    return torch.cat(bufs_o, dim=3).contiguous(), torch.cat(bufs_l, dim=3).contiguous()


def sequence_split_decode(q, k_cache, v_cache, tables, lens, num_kv_heads: int, num_pages: int,
                          softmax_scale: float, num_splits: int, holds_newest: bool, group=None, dst: int = 0):
    """One decode step of sequences split across the devices of `group`.

    Each device passes its own share: its cache, its page table and context
    lengths (local_tables).  holds_newest marks the device whose share holds
    the step's query positions.  Returns the attention output fp32 [B, T, Hq, D]
    on device dst, None elsewhere."""
    import bit_kv_cache_rotate_b300 as kv4
    B, T, Hq, D = q.shape
    ws = kv4.workspace(B, T, Hq, D, num_splits, device=q.device)
    fn = kv4.kv4_decode_partials if holds_newest else kv4.kv4_decode_partials_prefix
    fn(q, k_cache, v_cache, tables, lens, num_kv_heads, num_pages, softmax_scale, num_splits, ws)
    po, pl = kv4.split_views(ws, B, T, Hq, D, num_splits)
    po, pl = gather_partials(po, pl, group=group, dst=dst)
    if po is None:
        return None
    return kv4.kv4_split_combine(po, pl)
