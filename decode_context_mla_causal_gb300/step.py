"""One verify step (metadata -> partial -> merge) over preallocated buffers.

Host-side plumbing around the three C entry points: it sizes and allocates the
device buffers once (torch tensors), then every call launches the three
kernels on one stream with no host synchronisation, so a call can be captured
in a CUDA graph and replayed with new ``seq_lens`` / ``block_table`` / ``q``
contents up to the static bound.
"""

from __future__ import annotations

import math

import torch

from . import binding as B


def num_sms(device=None) -> int:
    return torch.cuda.get_device_properties(device or torch.cuda.current_device()).multi_processor_count


def choose_num_splits(batch: int, qlen: int, num_heads: int, num_ranks: int,
                      max_local_len: int, block_size: int, sms: int = 152) -> int:
    """Static split count for the partial kernel.

    Each work item (rank, sequence, split, 128-row tile) runs on a cluster of two
    CTAs, one CTA per SM, so ``sms // 2`` items run at once. The cost model is
    waves * (64-token tiles per split + 11 tiles of per-item overhead) + 0.5 tile
    per split for the merge's extra partial rows, evaluated at the static bound;
    the per-item overhead (start-up, pipeline fill, epilogue) was fitted to
    measured times over split counts 10-20 of the long-context workload. The
    cheapest split count wins (ties: fewer splits). Uses only static sizes, so the
    choice is graph-safe.
    """
    tiles = max(1, math.ceil(max_local_len / 64))
    row_tiles = math.ceil(qlen * num_heads / 128)
    base = max(1, batch * num_ranks * row_tiles)
    slots = max(1, sms // 2)
    best = None
    for ns in range(1, min(64, tiles) + 1):
        cost = math.ceil(base * ns / slots) * (tiles / ns + 11.0) + 0.5 * ns
        if best is None or cost < best[0] - 1e-9:
            best = (cost, ns)
    return int(best[1])


def concurrent_items() -> int:
    """Work items the partial kernel runs at once on the current device."""
    n = B.dcp_mla_concurrent_items()
    if n < 1:
        raise RuntimeError("no CUDA device to size the split plan for: " + B.dcp_last_error())
    return n


def choose_split_plan(batch: int, qlen: int, num_heads: int, num_ranks: int,
                      max_local_len: int, block_size: int, concurrent: int = 76):
    """``(num_splits, base_splits)`` for the dims: the static split count of
    ``choose_num_splits`` as the base and, when the work items at the static bound
    leave the last wave of ``concurrent`` items at most half full, room for the
    shortest (rank, sequence) pairs to take more splits and fill it (the device's
    wave balancing, ``dcp_mla_metadata``). ``base_splits`` is 0 when there is
    nothing to balance."""
    base = choose_num_splits(batch, qlen, num_heads, num_ranks, max_local_len, block_size,
                             sms=2 * concurrent)
    tiles = max(1, math.ceil(max_local_len / 64))
    per = math.ceil(qlen * num_heads / 128) * base
    rem = batch * num_ranks * per % concurrent
    if rem == 0 or 2 * rem > concurrent:
        return base, 0
    tail = -(-rem // per)
    kf = concurrent // (tail * per)
    hi = (concurrent - kf * tail * per) // per
    ns = min(64, base * (max(1, kf) + (1 if hi > 0 else 0)), max(base, tiles // 8))
    return (ns, base) if ns > base else (base, 0)


def make_dims(*, batch, qlen, num_heads, dcp, interleave, block_size, max_blocks_per_seq,
              max_local_len, num_blocks, num_splits, causal=True, base_splits=0) -> B.Dims:
    return B.Dims(batch, qlen, num_heads, dcp, interleave, block_size, max_blocks_per_seq,
                  max_local_len, num_blocks, num_splits, 1 if causal else 0, base_splits)


class VerifyStep:
    """Buffers + launches for ranks ``[rank_begin, rank_begin + num_ranks)``."""

    def __init__(self, dims: B.Dims, kv_dtype: int, device=None, rank_begin: int = 0,
                 num_ranks: int | None = None, rank_lse: bool = True):
        B.dcp_mla_check_dims(dims, rank_begin, num_ranks)
        self.dims = dims
        self.kv_dtype = kv_dtype
        self.rank_begin = rank_begin
        self.num_ranks = dims.dcp - rank_begin if num_ranks is None else num_ranks
        dev = torch.device(device or "cuda")
        nr, Bt, R, H, NS = self.num_ranks, dims.batch, dims.rows, dims.num_heads, dims.num_splits
        MP = B.dcp_mla_max_pages(dims)
        i32, f32 = torch.int32, torch.float32
        self.row_len = torch.empty((nr, R), dtype=i32, device=dev)
        self.page_ids = torch.empty((nr, Bt, MP), dtype=i32, device=dev)
        self.split_beg = torch.empty((nr, Bt, NS), dtype=i32, device=dev)
        self.split_end = torch.empty((nr, Bt, NS), dtype=i32, device=dev)
        self.part_o = torch.empty((nr, NS, R, H, B.V_DIM), dtype=f32, device=dev)
        self.part_m = torch.empty((nr, NS, R, H), dtype=f32, device=dev)
        self.part_l = torch.empty((nr, NS, R, H), dtype=f32, device=dev)
        self.out = torch.empty((R, H, B.V_DIM), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((R, H), dtype=f32, device=dev)
        self.rank_lse = torch.empty((nr, R, H), dtype=f32, device=dev) if rank_lse else None
        self.status = torch.zeros(1, dtype=i32, device=dev)
        # the partial call's item order (longest first)
        self.workspace = torch.empty(B.dcp_mla_workspace_size(dims, self.num_ranks),
                                     dtype=torch.uint8, device=dev)

    def metadata(self, seq_lens, block_table, stream=None):
        B.dcp_mla_metadata(self.dims, seq_lens, block_table, self.rank_begin, self.num_ranks,
                           self.row_len, self.page_ids, self.split_beg, self.split_end,
                           self.status, stream)

    def partial(self, q, kv, kv_scale, softmax_scale, stream=None):
        B.dcp_mla_partial(self.dims, q, kv, self.kv_dtype, kv_scale, softmax_scale,
                          self.rank_begin, self.num_ranks, self.row_len, self.page_ids,
                          self.split_beg, self.split_end, self.part_o, self.part_m,
                          self.part_l, self.status, stream, workspace=self.workspace)

    def merge(self, stream=None):
        B.dcp_lse_merge(self.dims, self.num_ranks, self.part_o, self.part_m, self.part_l,
                        self.out, self.lse, self.rank_lse, self.status, stream)

    def __call__(self, q, kv, kv_scale, softmax_scale, seq_lens, block_table, stream=None):
        self.metadata(seq_lens, block_table, stream)
        self.partial(q, kv, kv_scale, softmax_scale, stream)
        self.merge(stream)
        return self.out, self.lse

    def read_status(self) -> int:
        return int(self.status.item()) & 0xFFFFFFFF
