"""Shared test helpers: run the CUDA path and the oracle on the same inputs."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads


def dims_of(dm, w, num_splits, causal=True):
    return dm.make_dims(batch=w.batch, qlen=w.qlen, num_heads=w.num_heads, dcp=w.dcp,
                        interleave=w.interleave, block_size=w.block_size,
                        max_blocks_per_seq=w.max_blocks_per_seq, max_local_len=w.max_local_len,
                        num_blocks=w.num_blocks, num_splits=num_splits, causal=causal)


def kv_dtype_of(dm, w):
    return dm.KV_FP8_E4M3 if w.kv_dtype == "fp8" else dm.KV_BF16


def run_gpu(dm, w, num_splits=None, causal=True, rank_begin=0, num_ranks=None, step=None):
    """Run metadata + partial + merge on the workload's device; returns the step."""
    if num_splits is None:
        num_splits = dm.choose_num_splits(w.batch, w.qlen, w.num_heads, w.dcp, w.max_local_len,
                                          w.block_size, dm.num_sms())
    if step is None:
        step = dm.VerifyStep(dims_of(dm, w, num_splits, causal), kv_dtype_of(dm, w), w.q.device,
                             rank_begin=rank_begin, num_ranks=num_ranks)
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
