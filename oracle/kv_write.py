"""New-token KV write into the interleaved rank pools (oracle; test only).

What is computed, from the pages' statement of the method:

* "Context Parallel Guide (PCP & DCP)", "How it works" item 2: new-token KV is
  written interleaved via a slot mapping that holds -1 for the tokens a rank
  does not own; item 4: the FP8 cache has one per-tensor scale.
* The owner and slot of global position ``p`` are those of the gather in
  ``attention`` (owner ``(p // S) % W``, local index ``li``, block
  ``block_table[b][li // bs]``, row ``li % bs``) -- the DSpark slot formula of
  "Support Kimi-K3 DCP with DSpark" for S = 1.
* The new tokens of sequence b are its last qlen positions: token j is at
  ``seq_lens[b] - qlen + j`` (seq_lens counts them, as everywhere here).
* FP8 encoding: the code of ``x / scale`` (the division in IEEE float32, the
  arithmetic the library documents) is the OCP E4M3 value nearest to it, ties to
  the code with an even mantissa, magnitudes above 448 saturating to 448. The
  encoder below finds the nearest value by comparing against every code, which
  is slow and plainly correct.

Status bits follow the library's ABI values (see ``metadata``).
"""

from __future__ import annotations

import numpy as np

from . import fp8 as _fp8
from . import metadata as _md

STATUS_BAD_SEQ_LEN = _md.STATUS_BAD_SEQ_LEN
STATUS_LOCAL_OVER_BOUND = _md.STATUS_LOCAL_OVER_BOUND
STATUS_BAD_BLOCK_ID = _md.STATUS_BAD_BLOCK_ID

# magnitudes of the non-negative finite codes 0x00..0x7E, in code order
_MAGS = _fp8.E4M3_TABLE[:0x7F]


def encode_e4m3(x) -> np.ndarray:
    """E4M3 codes of the values ``x`` (float64 exact values): nearest finite
    code, ties to even mantissa, saturating at 448; NaN -> 0x7F; the sign of a
    zero is kept."""
    x = np.asarray(x, dtype=np.float64)
    flat = x.reshape(-1)
    out = np.zeros(flat.shape, dtype=np.uint8)
    nan = np.isnan(flat)
    mag = np.minimum(np.abs(np.where(nan, 0.0, flat)), 448.0)
    dist = np.abs(mag[:, None] - _MAGS[None, :])            # [n][127]
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best                                       # nearest codes (1 or 2)
    codes = np.arange(0x7F, dtype=np.int64)[None, :]
    even = cand & ((codes & 1) == 0)
    # a tie between two adjacent codes: take the even one; otherwise the unique one
    pick = np.where(even.any(axis=1), np.argmax(even, axis=1), np.argmax(cand, axis=1))
    sign = np.signbit(flat) & ~nan
    out[:] = pick.astype(np.uint8) | np.where(sign, 0x80, 0).astype(np.uint8)
    out[nan] = 0x7F
    return out.reshape(x.shape)


def quantize_rows(bits: np.ndarray, scale: float) -> np.ndarray:
    """BF16 bit patterns (uint16) -> E4M3 codes of x / scale, the division done
    in IEEE float32."""
    x32 = _fp8.decode_bf16(bits).astype(np.float32)
    q = (x32 / np.float32(scale)).astype(np.float32)
    return encode_e4m3(q.astype(np.float64))


def slot_mapping(*, seq_lens, block_table, qlen, dcp, interleave, block_size,
                 max_blocks_per_seq, num_blocks, rank_begin=0, num_ranks=None):
    """``[nr][B*qlen]`` int32 pool rows of the new tokens per rank (-1: not
    owned or invalid) and the status word."""
    W, S, bs = int(dcp), int(interleave), int(block_size)
    nr = W - rank_begin if num_ranks is None else int(num_ranks)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    block_table = np.asarray(block_table, dtype=np.int64)
    B = len(seq_lens)
    out = np.full((nr, B * qlen), -1, dtype=np.int32)
    status = 0
    for b in range(B):
        L = int(seq_lens[b])
        if L < qlen:
            status |= STATUS_BAD_SEQ_LEN
            continue
        for j in range(qlen):
            p = L - qlen + j
            r = int(_md.owner(p, W, S))
            k = r - rank_begin
            if not 0 <= k < nr:
                continue
            li = int(_md.local_index(p, W, S))
            if li // bs >= max_blocks_per_seq:
                status |= STATUS_LOCAL_OVER_BOUND
                continue
            blk = int(block_table[b, li // bs])
            if not 0 <= blk < num_blocks:
                status |= STATUS_BAD_BLOCK_ID
                continue
            out[k, b * qlen + j] = blk * bs + li % bs
    return out, status


def write(pools, slots, new_bits, kv_dtype, scale):
    """A copy of ``pools`` ([nr][NB][bs][576], uint8 codes or uint16 bf16 bits)
    with row ``slots[k][t]`` of rank k replaced by new token t (bits
    ``new_bits[t]``, uint16 [T][576]); -1 entries are skipped."""
    out = np.array(pools, copy=True)
    nr = out.shape[0]
    flat = out.reshape(nr, -1, out.shape[-1])
    rows = (quantize_rows(new_bits, scale) if kv_dtype == "fp8"
            else np.asarray(new_bits, dtype=np.uint16))
    for k in range(nr):
        for t, slot in enumerate(slots[k]):
            if slot >= 0:
                flat[k, slot] = rows[t]
    return out
