"""Global causal absorbed-MLA attention over the interleaved cache (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed, from the pages' statement of the method:

* The cache holds one 576-wide latent row per token: 512 latent dims followed by
  64 rope dims. Query and key use all 576 dims; the value is the 512-dim latent
  part of the same row (absorbed MLA: ``kv_lora_rank`` is the value width,
  "Context Parallel Guide (PCP & DCP)", ``enable_project_before_merge``).
* Gather: global position ``p`` of sequence ``b`` is stored on rank
  ``owner(p)``, in that rank's pool at block ``block_table[b][li // bs]``, row
  ``li % bs``, where ``li`` is the rank-local index (same page, "How it works"
  item 1 and ``interleave_size``). For S = 1 this is the slot formula of the
  DSpark section. FP8 codes are decoded exactly and multiplied by the
  per-tensor scale in float64.
* Global causal attention ("[ROCm][MLA][DCP] Support causal multi-token
  verification", "Validation": the merged rank partials are compared against
  global causal attention): for row (b, j, h) with boundary g,
  ``s_t = softmax_scale * q . K[t]`` for t < g,
  ``LSE = ln sum_t exp(s_t)`` (natural log, shifted by the maximum),
  ``O = sum_t exp(s_t - LSE) * K[t][:512]``.
* Per-shard attention: the same restricted to the positions a rank owns
  ("Decode": each rank runs attention over its local KV and returns its LSE).
  A rank with no positions has LSE = -inf and O = 0 ("empty-row and
  natural-log LSE reduction" in the PR's test list).
* Merge: ``LSE = ln sum_r exp(LSE_r)``, ``O = sum_r exp(LSE_r - LSE) O_r``
  (the "LSE-correct + reduce" of the DCP Guide's decode description).

Long sequences are processed in chunks of positions with an exact two-pass
softmax (pass 1: the maximum; pass 2: the sum and the weighted values). This
only bounds memory; it does not change what is computed, and the pins check
the chunked form against the one-shot form on multi-chunk inputs.
"""

from __future__ import annotations

import numpy as np

from . import fp8 as _fp8
from . import metadata as _md

D_QK = 576
D_V = 512
CHUNK = 1 << 16


def decode_pool_rows(pool_rows: np.ndarray, kv_dtype: str, kv_scale: float) -> np.ndarray:
    """Decode raw cache rows (uint8 E4M3 codes or uint16 BF16 bits) to float64."""
    if kv_dtype == "fp8":
        return _fp8.decode_e4m3(pool_rows) * float(kv_scale)
    if kv_dtype == "bf16":
        return _fp8.decode_bf16(pool_rows) * float(kv_scale)
    raise ValueError(kv_dtype)


def gather_rows(pools, block_table_row, positions, *, dcp, interleave, block_size):
    """Raw cache rows of the given global positions of one sequence.

    ``pools`` is ``[W][NB][bs][576]`` (uint8 or uint16); returns
    ``[len(positions)][576]`` of the same dtype.
    """
    p = np.asarray(positions, dtype=np.int64)
    r = _md.owner(p, dcp, interleave)
    li = _md.local_index(p, dcp, interleave)
    blk = np.asarray(block_table_row, dtype=np.int64)[li // block_size]
    return pools[r, blk, li % block_size]


def gather_sequence(pools, block_table_row, length, *, dcp, interleave, block_size,
                    kv_dtype, kv_scale, start=0):
    """Decoded K rows (float64 ``[length - start][576]``) of one sequence."""
    pos = np.arange(start, length, dtype=np.int64)
    raw = gather_rows(pools, block_table_row, pos, dcp=dcp, interleave=interleave,
                      block_size=block_size)
    return decode_pool_rows(raw, kv_dtype, kv_scale)


def attend(q: np.ndarray, K: np.ndarray, limits, softmax_scale: float, token_mask=None):
    """Plain softmax attention of query rows over the first ``limits[i]`` keys.

    ``q`` is float64 ``[n][576]``, ``K`` float64 ``[T][576]``; ``limits[i]`` is
    row i's boundary g (keys ``t < g`` are visible); ``token_mask`` (bool
    ``[T]``) further restricts the visible keys (per-shard attention).
    Returns ``O [n][512]`` and natural-log ``LSE [n]``; a row with no visible
    key gets ``O = 0`` and ``LSE = -inf``.
    """
    q = np.asarray(q, dtype=np.float64)
    n, T = q.shape[0], K.shape[0]
    limits = np.asarray(limits, dtype=np.int64).reshape(n)
    visible = np.arange(T)[None, :] < limits[:, None]
    if token_mask is not None:
        visible &= np.asarray(token_mask, dtype=bool)[None, :]
    s = softmax_scale * (q @ K.T)
    s = np.where(visible, s, -np.inf)
    out = np.zeros((n, D_V), dtype=np.float64)
    lse = np.full(n, -np.inf, dtype=np.float64)
    any_vis = visible.any(axis=1)
    if any_vis.any():
        sv = s[any_vis]
        m = sv.max(axis=1, keepdims=True)
        e = np.exp(sv - m)
        tot = e.sum(axis=1, keepdims=True)
        lse[any_vis] = (m + np.log(tot))[:, 0]
        out[any_vis] = (e / tot) @ K[:, :D_V]
    return out, lse


def attend_chunked(q, key_chunks, limits, softmax_scale, mask_chunks=None):
    """``attend`` over keys given as a re-iterable sequence of position chunks.

    ``key_chunks`` is a callable returning an iterator of ``(start, K_chunk)``;
    ``mask_chunks`` (optional) maps ``(start, count)`` to a bool mask. Exact
    two-pass softmax: pass 1 finds each row's maximum, pass 2 sums.
    """
    q = np.asarray(q, dtype=np.float64)
    n = q.shape[0]
    limits = np.asarray(limits, dtype=np.int64).reshape(n)

    def scores(start, Kc):
        vis = (start + np.arange(Kc.shape[0]))[None, :] < limits[:, None]
        if mask_chunks is not None:
            vis &= mask_chunks(start, Kc.shape[0])[None, :]
        return np.where(vis, softmax_scale * (q @ Kc.T), -np.inf)

    m = np.full(n, -np.inf)
    for start, Kc in key_chunks():
        m = np.maximum(m, scores(start, Kc).max(axis=1))
    tot = np.zeros(n)
    acc = np.zeros((n, D_V))
    has = np.isfinite(m)
    mm = np.where(has, m, 0.0)
    for start, Kc in key_chunks():
        e = np.exp(scores(start, Kc) - mm[:, None])
        tot += e.sum(axis=1)
        acc += e @ Kc[:, :D_V]
    out = np.zeros((n, D_V))
    lse = np.full(n, -np.inf)
    out[has] = acc[has] / tot[has, None]
    lse[has] = mm[has] + np.log(tot[has])
    return out, lse


def merge_shards(outs, lses):
    """LSE merge of per-shard results: ``LSE = ln sum exp(LSE_r)``,
    ``O = sum exp(LSE_r - LSE) O_r``; all-empty rows give O = 0, LSE = -inf."""
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    m = lses.max(axis=0)
    has = np.isfinite(m)
    mm = np.where(has, m, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - mm[None]), 0.0)
    tot = w.sum(axis=0)
    lse = np.where(has, mm + np.log(np.where(has, tot, 1.0)), -np.inf)
    scale = np.where(has, 1.0 / np.where(has, tot, 1.0), 0.0)
    out = np.einsum("r...,r...d->...d", w * scale[None], outs)
    return out, lse


def _row_limits(seq_len, qlen, causal, boundary):
    if boundary is not None:
        return [boundary(seq_len, qlen, j) for j in range(qlen)]
    return [_md.row_boundary(seq_len, qlen, j, causal) for j in range(qlen)]


def forward(*, q_bits, pools, block_table, seq_lens, qlen, dcp, interleave, block_size,
            kv_dtype, kv_scale, softmax_scale, causal=True, rows=None, heads=None,
            boundary=None, per_rank=True, chunk=CHUNK):
    """Oracle outputs for the requested (b, j) rows and heads.

    ``q_bits`` is uint16 ``[B*qlen][H][576]`` (BF16 bits); ``pools``
    ``[W][NB][bs][576]`` uint8/uint16. ``rows`` is a list of ``(b, j)`` (default
    all), ``heads`` a list of head indices (default all). Returns a dict with
    ``out [n_rows][n_heads][512]``, ``lse [n_rows][n_heads]`` (natural log) and,
    if ``per_rank``, ``rank_lse [W][n_rows][n_heads]`` and
    ``rank_out [W][n_rows][n_heads][512]``. Rows are grouped per sequence so
    every sequence's keys are gathered once (in chunks).
    """
    B = len(seq_lens)
    H = q_bits.shape[1]
    if rows is None:
        rows = [(b, j) for b in range(B) for j in range(qlen)]
    if heads is None:
        heads = list(range(H))
    heads = list(heads)
    W = dcp
    n_rows, n_heads = len(rows), len(heads)
    out = np.zeros((n_rows, n_heads, D_V))
    lse = np.full((n_rows, n_heads), -np.inf)
    rank_out = np.zeros((W, n_rows, n_heads, D_V)) if per_rank else None
    rank_lse = np.full((W, n_rows, n_heads), -np.inf) if per_rank else None
    by_seq = {}
    for i, (b, j) in enumerate(rows):
        by_seq.setdefault(b, []).append((i, j))
    for b, items in by_seq.items():
        L = int(seq_lens[b])
        lim_all = _row_limits(L, qlen, causal, boundary)
        qs, lims, where = [], [], []
        for i, j in items:
            qrow = _fp8.decode_bf16(q_bits[b * qlen + j][heads])
            qs.append(qrow)
            lims += [lim_all[j]] * n_heads
            where.append(i)
        qmat = np.concatenate(qs, axis=0)
        top = max(0, max(lims))
        top = min(top, L)

        def chunks():
            for st in range(0, top, chunk):
                yield st, gather_sequence(pools, block_table[b], min(top, st + chunk),
                                          dcp=dcp, interleave=interleave,
                                          block_size=block_size, kv_dtype=kv_dtype,
                                          kv_scale=kv_scale, start=st)

        o, l = attend_chunked(qmat, chunks, lims, softmax_scale)
        o = o.reshape(len(items), n_heads, D_V)
        l = l.reshape(len(items), n_heads)
        for k, i in enumerate(where):
            out[i], lse[i] = o[k], l[k]
        if per_rank:
            for r in range(W):
                def mask(st, cnt, r=r):
                    return _md.owner(np.arange(st, st + cnt), dcp, interleave) == r
                o, l = attend_chunked(qmat, chunks, lims, softmax_scale, mask)
                o = o.reshape(len(items), n_heads, D_V)
                l = l.reshape(len(items), n_heads)
                for k, i in enumerate(where):
                    rank_out[r, i], rank_lse[r, i] = o[k], l[k]
    res = dict(out=out, lse=lse)
    if per_rank:
        res.update(rank_out=rank_out, rank_lse=rank_lse)
    return res
