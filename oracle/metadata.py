"""Per-row causal rank-local lengths, subpages and splits (oracle; test only).

Definitions followed, each in the plainest reading the pages support:

* Token -> rank interleave. "Context Parallel Guide (PCP & DCP)", DCP Guide,
  ``--dcp-config`` table, ``interleave_size``: token ``p`` lives on rank
  ``(p // S) % W`` (S = interleave size, W = dcp); S = 1 is token round-robin.
* Rank-local index. Same page, section "interleave_size": the local index is
  ``(p // (S*W)) * S + p % S``; it needs ``block_size % S == 0`` when S > 1.
* Shared block ids. Same page, "How it works" item 1: one block-table entry is
  shared by all ranks and names, on each rank, that rank's own physical block of
  ``block_size`` local tokens.
* Row boundary. "[ROCm][MLA][DCP] Support causal multi-token verification",
  section "Implementation", first item: each verification row has its own global
  causal boundary. The pages give no formula; the reading used here (stated in
  the design notes) is that ``seq_len`` counts every token including the
  ``qlen`` verify tokens, so row ``j`` (0-based) sees global positions
  ``[0, seq_len - qlen + j]``, i.e. ``g_j = seq_len - qlen + 1 + j``. The
  "committed-prefix-only" boundary of that page's negative control is
  ``seq_len - qlen + 1`` for every row. With ``causal=False`` (the DSpark
  draft block of "DCP + Speculative Decode", which is bidirectional) every row
  sees the whole sequence, ``g_j = seq_len``.
* Rank-local length. The oracle COUNTS the owned positions below ``g``; the
  closed form of "Support Kimi-K3 DCP with DSpark" (review thread) is written
  out separately and pinned against the count.
* Subpages. "[ROCm][MLA][DCP] Support causal multi-token verification",
  "Implementation" second item and the review thread on the subpage size: the
  subpage is the largest power of two dividing the block size, capped at 128.
  Subpage ``p`` of a sequence lies in block ``p // ppb`` (ppb = blocks'
  subpages) and is numbered ``block_id * ppb + p % ppb``, so that subpage
  ``page`` covers pool rows ``[page*P, (page+1)*P)`` of the flat pool.
* Static bound. Same page, "Implementation" fifth item: row metadata is laid
  out at a maximum DCP-local KV bound; replay masks inactive segments. Inactive
  page entries are -1.
* Splits. Not on the pages (a property of the split-KV kernel): split ``s`` of
  ``NS`` covers subpages ``[floor(s*np/NS), floor((s+1)*np/NS))`` of the
  ``np`` subpages that the longest row of the sequence needs.

Status bits (the numbers are the library's documented ABI values):
bit0 a sequence shorter than qlen (causal) or negative; bit1 a local length
above the static bound (clamped to it); bit2 a block id outside [0, NB) (its
subpages become -1).
"""

from __future__ import annotations

import numpy as np

STATUS_BAD_SEQ_LEN = 1 << 0
STATUS_LOCAL_OVER_BOUND = 1 << 1
STATUS_BAD_BLOCK_ID = 1 << 2


def owner(p, W: int, S: int):
    """Rank that stores global position ``p``."""
    return (np.asarray(p) // S) % W


def local_index(p, W: int, S: int):
    """Index of global position ``p`` inside its owner's local sequence."""
    p = np.asarray(p)
    return (p // (S * W)) * S + p % S


def row_boundary(seq_len: int, qlen: int, j: int, causal: bool = True) -> int:
    """Number of global positions verify row ``j`` attends (its boundary g)."""
    if causal:
        return int(seq_len) - int(qlen) + 1 + int(j)
    return int(seq_len)


def committed_prefix_boundary(seq_len: int, qlen: int, j: int) -> int:
    """The wrong, pre-fix boundary: every row sees only the committed prefix."""
    return int(seq_len) - int(qlen) + 1


def count_local(g: int, r: int, W: int, S: int) -> int:
    """Rank-local length by counting owned positions in [0, g)."""
    if g <= 0:
        return 0
    return int(np.count_nonzero(owner(np.arange(g, dtype=np.int64), W, S) == r))


def local_len_closed_form(g: int, r: int, W: int, S: int) -> int:
    """The closed form from the review thread of the Kimi-K3 DSpark page."""
    span = W * S
    rem = min(max(g % span - r * S, 0), S)
    return (g // span) * S + rem


def subpage_size(block_size: int) -> int:
    """Largest power of two dividing ``block_size``, capped at 128."""
    if block_size <= 0:
        raise ValueError("block_size must be positive")
    low = block_size & (-block_size)
    return min(128, low)


def max_pages(max_local_len: int, block_size: int) -> int:
    """Subpage entries per (rank, sequence) at the static bound."""
    P = subpage_size(block_size)
    return -(-max_local_len // P)


def build_metadata(*, batch, qlen, dcp, interleave, block_size, max_local_len,
                   num_blocks, num_splits, seq_lens, block_table,
                   rank_begin=0, num_ranks=None, causal=True, boundary=None):
    """Metadata for ranks ``[rank_begin, rank_begin + num_ranks)``.

    ``seq_lens`` is ``[batch]`` and ``block_table`` is ``[batch][MB]`` (ints).
    ``boundary`` may replace ``row_boundary`` (used only by the negative
    control). Returns a dict of int32 arrays ``row_len [nr][batch*qlen]``,
    ``page_ids [nr][batch][MP]``, ``split_beg``/``split_end [nr][batch][NS]``
    and the status word.
    """
    W, S, bs = int(dcp), int(interleave), int(block_size)
    nr = W - rank_begin if num_ranks is None else int(num_ranks)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    block_table = np.asarray(block_table, dtype=np.int64)
    P = subpage_size(bs)
    ppb = bs // P
    MP = max_pages(max_local_len, bs)
    NS = int(num_splits)
    R = batch * qlen
    row_len = np.zeros((nr, R), dtype=np.int32)
    page_ids = np.full((nr, batch, MP), -1, dtype=np.int32)
    split_beg = np.zeros((nr, batch, NS), dtype=np.int32)
    split_end = np.zeros((nr, batch, NS), dtype=np.int32)
    status = 0
    for b in range(batch):
        L = int(seq_lens[b])
        if L < 0 or (causal and L < qlen):
            status |= STATUS_BAD_SEQ_LEN
        for k in range(nr):
            r = rank_begin + k
            longest = 0
            for j in range(qlen):
                if boundary is not None:
                    g = boundary(L, qlen, j)
                else:
                    g = row_boundary(L, qlen, j, causal)
                n = count_local(g, r, W, S)
                if n > max_local_len:
                    status |= STATUS_LOCAL_OVER_BOUND
                    n = max_local_len
                row_len[k, b * qlen + j] = n
                longest = max(longest, n)
            npages = -(-longest // P)
            for p in range(npages):
                blk = int(block_table[b, p // ppb])
                if 0 <= blk < num_blocks:
                    page_ids[k, b, p] = blk * ppb + p % ppb
                else:
                    status |= STATUS_BAD_BLOCK_ID
            for s in range(NS):
                split_beg[k, b, s] = (s * npages) // NS
                split_end[k, b, s] = ((s + 1) * npages) // NS
    return dict(row_len=row_len, page_ids=page_ids, split_beg=split_beg,
                split_end=split_end, status=status, subpage=P, max_pages=MP)
