"""Shared test helpers: run the CUDA path and the oracle on the same inputs."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads


def dims_of(dm, w, num_splits, causal=True, base_splits=0):
    return dm.make_dims(batch=w.batch, qlen=w.qlen, num_heads=w.num_heads, dcp=w.dcp,
                        interleave=w.interleave, block_size=w.block_size,
                        max_blocks_per_seq=w.max_blocks_per_seq, max_local_len=w.max_local_len,
                        num_blocks=w.num_blocks, num_splits=num_splits, causal=causal,
                        base_splits=base_splits)


def split_plan(dm, w):
    """The product's default (num_splits, base_splits) for a workload on this device."""
    return dm.choose_split_plan(w.batch, w.qlen, w.num_heads, w.dcp, w.max_local_len,
                                w.block_size, dm.concurrent_items())


def kv_dtype_of(dm, w):
    return dm.KV_FP8_E4M3 if w.kv_dtype == "fp8" else dm.KV_BF16


def run_gpu(dm, w, num_splits=None, causal=True, rank_begin=0, num_ranks=None, step=None):
    """Run metadata + partial + merge on the workload's device; returns the step."""
    base = 0
    if num_splits is None:
        num_splits, base = split_plan(dm, w)
    if step is None:
        step = dm.VerifyStep(dims_of(dm, w, num_splits, causal, base), kv_dtype_of(dm, w),
                             w.q.device, rank_begin=rank_begin, num_ranks=num_ranks)
    nr = step.num_ranks
    kv = w.kv[rank_begin:rank_begin + nr].contiguous()
    scale = torch.tensor([w.kv_scale], dtype=torch.float32, device=w.q.device)
    step(w.q, kv, scale, w.softmax_scale, w.seq_lens, w.block_table)
    torch.cuda.synchronize()
    return step


def oracle_metadata(w, num_splits, rank_begin=0, num_ranks=None, causal=True):
    return oracle.metadata.build_metadata(
        batch=w.batch, qlen=w.qlen, dcp=w.dcp, interleave=w.interleave,
        block_size=w.block_size, max_local_len=w.max_local_len, num_blocks=w.num_blocks,
        num_splits=num_splits, seq_lens=w.seq_lens.cpu().numpy(),
        block_table=w.block_table.cpu().numpy(), rank_begin=rank_begin,
        num_ranks=num_ranks, causal=causal)


def sequence_subset(w, b):
    """Host copies of only sequence b's blocks (table remapped), for big workloads."""
    table = w.block_table[b].long()
    pools = w.kv[:, table]  # [W][MB][bs][576]
    sub = workloads.Workload(**{**w.__dict__})
    sub.kv = pools.cpu()
    sub.block_table = torch.arange(table.numel(), dtype=torch.int32).reshape(1, -1)
    sub.seq_lens = w.seq_lens[b:b + 1].cpu()
    sub.q = w.q[b * w.qlen:(b + 1) * w.qlen].cpu()
    sub.batch = 1
    sub.num_blocks = table.numel()
    return sub


def oracle_forward(w, rows=None, heads=None, per_rank=True, causal=True, boundary=None):
    return oracle.attention.forward(
        q_bits=w.q_bits_np(), pools=w.pools_np(), block_table=w.block_table.cpu().numpy(),
        seq_lens=w.seq_lens.cpu().numpy(), qlen=w.qlen, dcp=w.dcp, interleave=w.interleave,
        block_size=w.block_size, kv_dtype=w.kv_dtype, kv_scale=w.kv_scale,
        softmax_scale=w.softmax_scale, rows=rows, heads=heads, per_rank=per_rank,
        causal=causal, boundary=boundary)


def compare(out_gpu, lse_gpu, out_ref, lse_ref):
    """Parity gate: |dO| <= 1e-2 + half a BF16 ulp of the oracle value, |dLSE| <= 1e-3,
    -inf LSE on exactly the same rows. Returns a dict of statistics."""
    o = np.asarray(out_gpu, dtype=np.float64)
    e = np.asarray(out_ref, dtype=np.float64)
    allow = 1e-2 + 0.5 * oracle.fp8.bf16_ulp(e)
    diff = np.abs(o - e)
    bad_o = int((~(diff <= allow)).sum())
    l = np.asarray(lse_gpu, dtype=np.float64)
    le = np.asarray(lse_ref, dtype=np.float64)
    inf_ok = bool(np.array_equal(np.isneginf(l), np.isneginf(le)))
    fin = np.isfinite(le)
    dl = np.abs(l[fin] - le[fin]) if fin.any() else np.zeros(1)
    bad_l = int((~(dl <= 1e-3)).sum())
    # the gate adds half a BF16 spacing to 1e-2 for the output's own rounding; this
    # counts the elements that pass only because of it (strictly above 1e-2)
    over = int((diff > 1e-2).sum())
    return dict(bad_out=bad_o, bad_lse=bad_l, inf_ok=inf_ok, n_out=o.size,
                max_abs_out=float(diff.max()) if diff.size else 0.0,
                n_out_over_1e2=over,
                max_abs_lse=float(dl.max()) if dl.size else 0.0)


def assert_parity(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    st = compare(out_gpu, lse_gpu, out_ref, lse_ref)
    assert st["bad_out"] == 0 and st["bad_lse"] == 0 and st["inf_ok"], (what, st)
    return st


def _local_len(g, rank, dcp, interleave):
    """Local length of a row with global boundary g ("Support Kimi-K3 DCP with
    DSpark", review thread)."""
    if g <= 0:
        return 0
    span = dcp * interleave
    rem = min(max(g % span - rank * interleave, 0), interleave)
    return g // span * interleave + rem


def balanced_split_counts(seq_lens, *, batch, qlen, num_heads, dcp, interleave,
                          max_local_len, num_splits, base_splits, concurrent):
    """Host restatement of the wave-balancing rule documented beside dcp_mla_metadata:
    the number of splits each (rank, sequence) pair takes, ``n[rank][b]``."""
    n = np.full((dcp, batch), num_splits, dtype=np.int64)
    if not 0 < base_splits < num_splits:
        return n
    tiles = np.array([[-(-min(_local_len(max(int(seq_lens[b]), 0), r, dcp, interleave),
                                 max_local_len) // 64) for b in range(batch)]
                      for r in range(dcp)])
    flat = tiles.reshape(-1)                       # rank-major pair index
    live = int((flat > 0).sum())
    per = -(-(qlen * num_heads) // 128) * base_splits
    rem = live * per % concurrent
    for v in range(flat.size):
        t = int(flat[v])
        if t == 0:
            s = 1
        elif rem == 0 or 2 * rem > concurrent:
            s = base_splits
        else:
            tail = -(-rem // per)
            pos = int((flat > t).sum() + (flat[:v] == t).sum())
            if pos < live - tail:
                s = base_splits
            else:
                j = pos - (live - tail)
                kf = concurrent // (tail * per)
                hi = (concurrent - kf * tail * per) // per
                s = min(base_splits * (max(kf, 1) + (1 if j < hi else 0)), num_splits,
                        t // 8)
                s = max(s, base_splits)
        n.reshape(-1)[v] = s
    return n


def expected_split_bounds(n, row_len, *, batch, qlen, num_splits, subpage, rank_begin=0):
    """split_beg/split_end for per-pair split counts ``n[rank][b]`` (all ranks) over
    the call's ranks, from the call's row_len ``[nr][R]``: split s < n of a pair covers
    subpages [s*np/n, (s+1)*np/n), later slots are [np, np)."""
    nr = row_len.shape[0]
    beg = np.zeros((nr, batch, num_splits), dtype=np.int64)
    end = np.zeros_like(beg)
    for k in range(nr):
        for b in range(batch):
            longest = int(row_len[k, b * qlen:(b + 1) * qlen].max())
            np_ = -(-longest // subpage)
            nn = int(n[rank_begin + k, b])
            for s in range(num_splits):
                beg[k, b, s] = s * np_ // nn if s < nn else np_
                end[k, b, s] = (s + 1) * np_ // nn if s < nn else np_
    return beg, end
