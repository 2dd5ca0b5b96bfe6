"""The cross-rank exchange of per-rank results, and project-before-merge (oracle; test only).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed, from the pages' statement of the method:

* "Context Parallel Guide (PCP & DCP)", Decode: every rank attends its local
  KV and returns its output and LSE; the outputs are LSE-corrected and summed so
  that every rank ends with its slice of the heads.
* Same page, ``comm_backend``: the default ``a2a`` does this with ONE
  all-to-all that carries the LSE packed alongside the output, then combines
  locally. The fp32 LSE travels as two 16-bit halves of the BF16 buffer, so it
  arrives bit for bit; the output itself travels as BF16, which is why the
  result is not bitwise identical to an fp32 merge.
* Same page, ``enable_project_before_merge``: the merge is a per-(token, head)
  scalar weighting plus a cross-rank sum and W_V is a per-head linear map, so
  projecting each rank's output by W_V before the exchange gives the same
  merged result and moves v_head_dim instead of kv_lora_rank values per head.

The wire format (the pages fix only the points above; the layout is this
library's, and the oracle states it independently):

* destination rank d receives the heads ``[d*Hg, (d+1)*Hg)``, ``Hg = H / W``;
* the chunk a source rank s sends to d holds ``[R][Hg][P]`` BF16 outputs (P = 512,
  or the projected width), then ``[R][Hg][2]`` LSE halves (the low 16 bits of
  the float32 pattern first, then the high 16 bits), then zero words up to a
  multiple of 8 words (16 bytes);
* the send buffer of rank s is ``[W destinations][chunk]``; the all-to-all
  delivers ``send_s[d]`` as ``recv_d[s]``.

Combine at d: ``LSE = ln sum_s exp(LSE_s)``, ``O = sum_s exp(LSE_s - LSE) O_s``
(empty ranks have LSE_s = -inf and weight 0; all empty gives O = 0, LSE = -inf).
"""

from __future__ import annotations

import numpy as np

from . import attention as _att
from . import fp8 as _fp8


def to_bf16_bits(x) -> np.ndarray:
    """BF16 bit patterns (uint16) of float64 values, rounded as ``fp8.round_to_bf16``."""
    v = _fp8.round_to_bf16(np.asarray(x, dtype=np.float64)).astype(np.float32)
    return (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def lse_halves(lse) -> tuple[np.ndarray, np.ndarray]:
    """The float32 bit pattern of each LSE as (low 16 bits, high 16 bits)."""
    bits = np.asarray(lse, dtype=np.float64).astype(np.float32).view(np.uint32)
    return (bits & np.uint32(0xFFFF)).astype(np.uint16), (bits >> np.uint32(16)).astype(np.uint16)


def lse_from_halves(lo, hi) -> np.ndarray:
    """Inverse of ``lse_halves``: float32 values (as float64)."""
    bits = (np.asarray(hi, dtype=np.uint32) << np.uint32(16)) | np.asarray(lo, dtype=np.uint32)
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def chunk_words(R: int, Hg: int, P: int) -> int:
    """16-bit words of one (source, destination) chunk."""
    lse_words = 2 * R * Hg
    return R * Hg * P + (lse_words + 7) // 8 * 8


def pack(rank_out, rank_lse) -> np.ndarray:
    """Send buffers of every rank: uint16 ``[W][W][chunk_words]``.

    ``rank_out`` is float64 ``[W][R][H][P]`` (each rank's normalised output),
    ``rank_lse`` float64 ``[W][R][H]`` (natural log, -inf for an empty rank).
    """
    rank_out = np.asarray(rank_out, dtype=np.float64)
    rank_lse = np.asarray(rank_lse, dtype=np.float64)
    W, R, H, P = rank_out.shape
    if H % W:
        raise ValueError("heads must divide evenly among the ranks")
    Hg = H // W
    cw = chunk_words(R, Hg, P)
    send = np.zeros((W, W, cw), dtype=np.uint16)
    for s in range(W):
        for d in range(W):
            heads = slice(d * Hg, (d + 1) * Hg)
            o_bits = to_bf16_bits(rank_out[s][:, heads, :])         # [R][Hg][P]
            lo, hi = lse_halves(rank_lse[s][:, heads])              # [R][Hg]
            send[s, d, : R * Hg * P] = o_bits.reshape(-1)
            halves = np.stack([lo, hi], axis=-1).reshape(-1)        # [R][Hg][2]
            send[s, d, R * Hg * P : R * Hg * P + 2 * R * Hg] = halves
    return send


def exchange(send) -> np.ndarray:
    """The all-to-all: ``recv[d][s] = send[s][d]``."""
    send = np.asarray(send)
    return np.ascontiguousarray(np.swapaxes(send, 0, 1))


def unpack(recv_d, R: int, Hg: int, P: int):
    """One destination's received chunks ``[W][chunk_words]`` -> outputs
    float64 ``[W][R][Hg][P]`` (exact BF16 values) and LSE ``[W][R][Hg]``."""
    recv_d = np.asarray(recv_d, dtype=np.uint16)
    W = recv_d.shape[0]
    o = recv_d[:, : R * Hg * P].reshape(W, R, Hg, P)
    halves = recv_d[:, R * Hg * P : R * Hg * P + 2 * R * Hg].reshape(W, R, Hg, 2)
    return _fp8.decode_bf16(o), lse_from_halves(halves[..., 0], halves[..., 1])


def combine(recv, R: int, H: int, P: int):
    """Every destination's combine: float64 ``out [R][H][P]`` and ``lse [R][H]``."""
    recv = np.asarray(recv, dtype=np.uint16)
    W = recv.shape[0]
    Hg = H // W
    out = np.zeros((R, H, P))
    lse = np.full((R, H), -np.inf)
    for d in range(W):
        o, l = unpack(recv[d], R, Hg, P)
        od, ld = _att.merge_shards(o, l)
        out[:, d * Hg : (d + 1) * Hg] = od
        lse[:, d * Hg : (d + 1) * Hg] = ld
    return out, lse


def project(o, w_v) -> np.ndarray:
    """Per-head projection ``o[..., h, :] @ w_v[h]`` (``w_v`` is ``[H][512][P]``)."""
    return np.einsum("...hk,hkp->...hp", np.asarray(o, dtype=np.float64),
                     np.asarray(w_v, dtype=np.float64))


def wire_bound(rank_out, rank_lse, lse) -> np.ndarray:
    """Bound of what the BF16 wire rounding can change in the combined output:
    ``sum_s exp(LSE_s - LSE) * ulp_bf16(O_s)`` per element (a full ulp, which
    also covers a rounding decision that an fp32 producer takes differently)."""
    rank_out = np.asarray(rank_out, dtype=np.float64)
    rank_lse = np.asarray(rank_lse, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    fin = np.isfinite(rank_lse) & np.isfinite(lse)[None]
    w = np.where(fin, np.exp(np.where(fin, rank_lse - lse[None], 0.0)), 0.0)
    return np.einsum("s...,s...p->...p", w, _fp8.bf16_ulp(rank_out))
