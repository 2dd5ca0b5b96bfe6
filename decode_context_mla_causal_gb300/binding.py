"""ctypes binding of libdcpmla.so (argument marshalling only).

Each function has the name of the C entry point it calls and takes torch
tensors in place of raw pointers; it checks dtype, device, contiguity and size,
passes ``data_ptr()`` and the current CUDA stream, and raises ``DcpError`` on a
non-OK return. Every step of the computation runs in the library's kernels.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

QK_DIM = 576
V_DIM = 512

DCP_OK = 0
DCP_ERR_INVALID_ARG = 1
DCP_ERR_UNSUPPORTED = 2
DCP_ERR_CUDA = 3

STATUS_BAD_SEQ_LEN = 0x1
STATUS_LOCAL_OVER_BOUND = 0x2
STATUS_BAD_BLOCK_ID = 0x4
STATUS_BAD_PAGE = 0x8
STATUS_TIMEOUT = 0x10
STATUS_BAD_SPLIT = 0x20
STATUS_Q_RANGE = 0x40

KV_BF16 = 0
KV_FP8_E4M3 = 1


class DcpError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dcp status {code}: {msg}")
        self.code = code


class Dims(ctypes.Structure):
    """Mirror of ``dcp_mla_dims`` (include/dcp_mla.h)."""

    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "qlen", "num_heads", "dcp", "interleave", "block_size",
        "max_blocks_per_seq", "max_local_len", "num_blocks", "num_splits", "causal",
        "base_splits")]

    def __repr__(self):
        return "Dims(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"

    @property
    def rows(self) -> int:
        return self.batch * self.qlen


_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libdcpmla.so; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with __graft_entry__.build() or "
            "python decode_context_mla_causal_gb300/build.py (there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int32
    D = ctypes.POINTER(Dims)
    sig = {
        "dcp_mla_subpage_size": (I, [I]),
        "dcp_mla_max_pages": (I, [D]),
        "dcp_mla_concurrent_items": (I, []),
        "dcp_mla_check_dims": (I, [D, I, I]),
        "dcp_mla_metadata": (I, [D, P, P, I, I, P, P, P, P, P, P]),
        "dcp_mla_partial": (I, [D, P, P, I, P, ctypes.c_float, I, I, P, P, P, P, P, P, P, P, P,
                                P]),
        "dcp_mla_partial_hold_q": (I, [D, P, P, I, P, ctypes.c_float, I, I, P, P, P, P, P, P, P,
                                       P, P, ctypes.c_uint64, P]),
        "dcp_mla_workspace_size": (I, [D, I, ctypes.POINTER(ctypes.c_size_t)]),
        "dcp_lse_merge": (I, [D, I, P, P, P, P, P, P, P, P]),
        "dcp_mla_verify_noalloc": (I, [D, P, P, P, P, I, P, ctypes.c_float, P, P, P, P]),
        "dcp_kv_slot_mapping": (I, [D, P, P, I, I, P, P, P]),
        "dcp_kv_write": (I, [D, P, P, I, P, I, P, P, P]),
        "dcp_mla_partial_packed": (I, [D, P, P, I, P, ctypes.c_float, I, I, P, P, P, P, P, P, P,
                                       P]),
        "dcp_a2a_chunk_words": (ctypes.c_int64, [D, I]),
        "dcp_a2a_pack": (I, [D, I, P, P, P, P, P, P]),
        "dcp_a2a_project": (I, [D, I, P, P, I, P, P, P]),
        "dcp_a2a_combine": (I, [D, I, P, ctypes.c_int64, ctypes.c_int64, I, I, P, P, P, P]),
        "dcp_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def dcp_last_error() -> str:
    return load().dcp_last_error().decode()


def _check(code: int):
    if code != DCP_OK:
        raise DcpError(code, dcp_last_error())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t, dtype, numel, name, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return t.data_ptr()


def dcp_mla_subpage_size(block_size: int) -> int:
    return load().dcp_mla_subpage_size(block_size)


def dcp_mla_max_pages(dims: Dims) -> int:
    return load().dcp_mla_max_pages(ctypes.byref(dims))


def dcp_mla_concurrent_items() -> int:
    """Work items the partial kernel runs at once on the current device (-1: none)."""
    return int(load().dcp_mla_concurrent_items())


def dcp_mla_check_dims(dims: Dims, rank_begin: int = 0, num_ranks: int | None = None):
    nr = dims.dcp - rank_begin if num_ranks is None else num_ranks
    _check(load().dcp_mla_check_dims(ctypes.byref(dims), rank_begin, nr))


def dcp_mla_metadata(dims, seq_lens, block_table, rank_begin, num_ranks, row_len, page_ids,
                     split_beg, split_end, status, stream=None):
    lib = load()
    B, R, NS = dims.batch, dims.rows, dims.num_splits
    MP = lib.dcp_mla_max_pages(ctypes.byref(dims))
    if MP < 0:
        _check(lib.dcp_mla_check_dims(ctypes.byref(dims), rank_begin, num_ranks))
    i32 = torch.int32
    _check(lib.dcp_mla_metadata(
        ctypes.byref(dims), _ptr(seq_lens, i32, B, "seq_lens"),
        _ptr(block_table, i32, B * dims.max_blocks_per_seq, "block_table"),
        rank_begin, num_ranks,
        _ptr(row_len, i32, num_ranks * R, "row_len"),
        _ptr(page_ids, i32, num_ranks * B * MP, "page_ids"),
        _ptr(split_beg, i32, num_ranks * B * NS, "split_beg"),
        _ptr(split_end, i32, num_ranks * B * NS, "split_end"),
        _ptr(status, i32, 1, "status"), _stream(stream)))


def dcp_mla_workspace_size(dims, num_ranks) -> int:
    """Bytes of device workspace ``dcp_mla_partial`` takes (the longest-first item order)."""
    n = ctypes.c_size_t(0)
    _check(load().dcp_mla_workspace_size(ctypes.byref(dims), int(num_ranks), ctypes.byref(n)))
    return int(n.value)


def dcp_mla_partial(dims, q, kv, kv_dtype, kv_scale, softmax_scale, rank_begin, num_ranks,
                    row_len, page_ids, split_beg, split_end, part_o, part_m, part_l, status,
                    stream=None, workspace=None):
    """Partial attention of ranks ``rank_begin ..``; ``workspace`` (a device tensor of at
    least ``dcp_mla_workspace_size`` bytes, optional) lets the call run the work items
    longest first (same results)."""
    lib = load()
    B, R, H, NS = dims.batch, dims.rows, dims.num_heads, dims.num_splits
    MP = lib.dcp_mla_max_pages(ctypes.byref(dims))
    i32 = torch.int32
    f32 = torch.float32
    kv_elem = torch.uint8 if kv_dtype == KV_FP8_E4M3 else torch.bfloat16
    pool = dims.num_blocks * dims.block_size * QK_DIM
    _check(lib.dcp_mla_partial(
        ctypes.byref(dims), _ptr(q, torch.bfloat16, R * H * QK_DIM, "q"),
        _ptr(kv, kv_elem, num_ranks * pool, "kv"), int(kv_dtype),
        _ptr(kv_scale, f32, 1, "kv_scale", allow_none=True), float(softmax_scale),
        rank_begin, num_ranks,
        _ptr(row_len, i32, num_ranks * R, "row_len"),
        _ptr(page_ids, i32, num_ranks * B * max(MP, 0), "page_ids"),
        _ptr(split_beg, i32, num_ranks * B * NS, "split_beg"),
        _ptr(split_end, i32, num_ranks * B * NS, "split_end"),
        _ptr(part_o, f32, num_ranks * NS * R * H * V_DIM, "part_o"),
        _ptr(part_m, f32, num_ranks * NS * R * H, "part_m"),
        _ptr(part_l, f32, num_ranks * NS * R * H, "part_l"),
        _ptr(workspace, None, None, "workspace", allow_none=True),
        _ptr(status, i32, 1, "status"), _stream(stream)))


def dcp_mla_partial_hold_q(dims, q, kv, kv_dtype, kv_scale, softmax_scale, rank_begin,
                           num_ranks, row_len, page_ids, split_beg, split_end, part_o, part_m,
                           part_l, status, q_wait_ns, stream=None, workspace=None):
    """dcp_mla_partial with the q arrival withheld (the failure path's test): the wait
    for q runs out after ``q_wait_ns`` and DCP_STATUS_TIMEOUT is raised."""
    lib = load()
    B, R, H, NS = dims.batch, dims.rows, dims.num_heads, dims.num_splits
    MP = lib.dcp_mla_max_pages(ctypes.byref(dims))
    i32 = torch.int32
    f32 = torch.float32
    kv_elem = torch.uint8 if kv_dtype == KV_FP8_E4M3 else torch.bfloat16
    pool = dims.num_blocks * dims.block_size * QK_DIM
    _check(lib.dcp_mla_partial_hold_q(
        ctypes.byref(dims), _ptr(q, torch.bfloat16, R * H * QK_DIM, "q"),
        _ptr(kv, kv_elem, num_ranks * pool, "kv"), int(kv_dtype),
        _ptr(kv_scale, f32, 1, "kv_scale", allow_none=True), float(softmax_scale),
        rank_begin, num_ranks,
        _ptr(row_len, i32, num_ranks * R, "row_len"),
        _ptr(page_ids, i32, num_ranks * B * max(MP, 0), "page_ids"),
        _ptr(split_beg, i32, num_ranks * B * NS, "split_beg"),
        _ptr(split_end, i32, num_ranks * B * NS, "split_end"),
        _ptr(part_o, f32, num_ranks * NS * R * H * V_DIM, "part_o"),
        _ptr(part_m, f32, num_ranks * NS * R * H, "part_m"),
        _ptr(part_l, f32, num_ranks * NS * R * H, "part_l"),
        _ptr(workspace, None, None, "workspace", allow_none=True),
        _ptr(status, i32, 1, "status"), int(q_wait_ns), _stream(stream)))


def dcp_mla_partial_packed(dims, q, kv, kv_dtype, kv_scale, softmax_scale, rank_begin,
                           num_ranks, row_len, page_ids, split_beg, split_end, send, status,
                           stream=None, workspace=None):
    """Partial attention of ranks ``rank_begin ..`` with one split, each rank's BF16
    output and LSE written straight into ``send`` (the all-to-all wire format, payload
    512) instead of fp32 partials."""
    lib = load()
    B, R, H = dims.batch, dims.rows, dims.num_heads
    MP = lib.dcp_mla_max_pages(ctypes.byref(dims))
    i32 = torch.int32
    f32 = torch.float32
    kv_elem = torch.uint8 if kv_dtype == KV_FP8_E4M3 else torch.bfloat16
    pool = dims.num_blocks * dims.block_size * QK_DIM
    cw = lib.dcp_a2a_chunk_words(ctypes.byref(dims), V_DIM)
    _check(lib.dcp_mla_partial_packed(
        ctypes.byref(dims), _ptr(q, torch.bfloat16, R * H * QK_DIM, "q"),
        _ptr(kv, kv_elem, num_ranks * pool, "kv"), int(kv_dtype),
        _ptr(kv_scale, f32, 1, "kv_scale", allow_none=True), float(softmax_scale),
        rank_begin, num_ranks,
        _ptr(row_len, i32, num_ranks * R, "row_len"),
        _ptr(page_ids, i32, num_ranks * B * max(MP, 0), "page_ids"),
        _ptr(split_beg, i32, num_ranks * B, "split_beg"),
        _ptr(split_end, i32, num_ranks * B, "split_end"),
        _ptr(send, torch.bfloat16, num_ranks * dims.dcp * max(cw, 0), "send"),
        _ptr(workspace, None, None, "workspace", allow_none=True),
        _ptr(status, i32, 1, "status"), _stream(stream)))


def dcp_lse_merge(dims, num_ranks, part_o, part_m, part_l, out, lse, rank_lse=None,
                  status=None, stream=None):
    lib = load()
    R, H, NS = dims.rows, dims.num_heads, dims.num_splits
    f32 = torch.float32
    _check(lib.dcp_lse_merge(
        ctypes.byref(dims), num_ranks,
        _ptr(part_o, f32, num_ranks * NS * R * H * V_DIM, "part_o"),
        _ptr(part_m, f32, num_ranks * NS * R * H, "part_m"),
        _ptr(part_l, f32, num_ranks * NS * R * H, "part_l"),
        _ptr(out, torch.bfloat16, R * H * V_DIM, "out"),
        _ptr(lse, f32, R * H, "lse"),
        _ptr(rank_lse, f32, num_ranks * R * H, "rank_lse", allow_none=True),
        _ptr(status, torch.int32, 1, "status"), _stream(stream)))


def dcp_kv_slot_mapping(dims, seq_lens, block_table, rank_begin, num_ranks, slot_mapping,
                        status, stream=None):
    """Pool row of each new token on each rank (-1 where the rank does not own it)."""
    lib = load()
    i32 = torch.int32
    _check(lib.dcp_kv_slot_mapping(
        ctypes.byref(dims), _ptr(seq_lens, i32, dims.batch, "seq_lens"),
        _ptr(block_table, i32, dims.batch * dims.max_blocks_per_seq, "block_table"),
        int(rank_begin), int(num_ranks),
        _ptr(slot_mapping, i32, num_ranks * dims.rows, "slot_mapping"),
        _ptr(status, i32, 1, "status"), _stream(stream)))


def dcp_kv_write(dims, slot_mapping, kv_new, kv_dtype, kv_scale, num_ranks, pool, status,
                 stream=None):
    """Writes (FP8: quantises) the new tokens' rows into the rank pools."""
    lib = load()
    kv_elem = torch.uint8 if kv_dtype == KV_FP8_E4M3 else torch.bfloat16
    _check(lib.dcp_kv_write(
        ctypes.byref(dims), _ptr(slot_mapping, torch.int32, num_ranks * dims.rows, "slot_mapping"),
        _ptr(kv_new, torch.bfloat16, dims.rows * QK_DIM, "kv_new"), int(kv_dtype),
        _ptr(kv_scale, torch.float32, 1, "kv_scale", allow_none=True), int(num_ranks),
        _ptr(pool, kv_elem, num_ranks * dims.num_blocks * dims.block_size * QK_DIM, "pool"),
        _ptr(status, torch.int32, 1, "status"), _stream(stream)))


def dcp_a2a_chunk_words(dims, payload=V_DIM) -> int:
    """16-bit words of one (source, destination) chunk of the all-to-all wire format."""
    n = load().dcp_a2a_chunk_words(ctypes.byref(dims), int(payload))
    if n < 0:
        raise DcpError(DCP_ERR_INVALID_ARG, "invalid dims or payload for the wire format")
    return int(n)


def dcp_a2a_pack(dims, num_ranks, part_o, part_m, part_l, send, status=None, stream=None):
    """Each rank's merged output and LSE in the all-to-all wire format (``send`` is a
    bf16 tensor of ``num_ranks * dcp * chunk_words`` elements, payload 512)."""
    lib = load()
    R, H = dims.rows, dims.num_heads
    parts = num_ranks * dims.num_splits * R * H
    cw = dcp_a2a_chunk_words(dims, V_DIM)
    _check(lib.dcp_a2a_pack(
        ctypes.byref(dims), int(num_ranks), _ptr(part_o, torch.float32, parts * V_DIM, "part_o"),
        _ptr(part_m, torch.float32, parts, "part_m"), _ptr(part_l, torch.float32, parts, "part_l"),
        _ptr(send, torch.bfloat16, num_ranks * dims.dcp * cw, "send"),
        _ptr(status, torch.int32, 1, "status", allow_none=True), _stream(stream)))


def dcp_a2a_project(dims, num_ranks, send, w_v, payload, send_projected, status=None,
                    stream=None):
    """Project-before-merge of packed send buffers by ``w_v`` (bf16 ``[H][payload][512]``)
    into ``send_projected`` (payload ``payload``)."""
    lib = load()
    H = dims.num_heads
    cw_in = dcp_a2a_chunk_words(dims, V_DIM)
    cw = dcp_a2a_chunk_words(dims, payload)
    _check(lib.dcp_a2a_project(
        ctypes.byref(dims), int(num_ranks),
        _ptr(send, torch.bfloat16, num_ranks * dims.dcp * cw_in, "send"),
        _ptr(w_v, torch.bfloat16, H * payload * V_DIM, "w_v"), int(payload),
        _ptr(send_projected, torch.bfloat16, num_ranks * dims.dcp * cw, "send_projected"),
        _ptr(status, torch.int32, 1, "status", allow_none=True), _stream(stream)))


def dcp_a2a_combine(dims, payload, recv, src_stride, dst_stride, dst_begin, num_dst, out, lse,
                    status=None, stream=None):
    """Combine at destination ranks ``dst_begin .. dst_begin+num_dst-1`` of the chunks
    they received (strides in 16-bit words); writes their heads of ``out`` (bf16
    ``[R][H][payload]``) and ``lse`` (float ``[R][H]``)."""
    lib = load()
    R, H = dims.rows, dims.num_heads
    cw = dcp_a2a_chunk_words(dims, payload)
    need = (num_dst - 1) * dst_stride + (dims.dcp - 1) * src_stride + cw
    _check(lib.dcp_a2a_combine(
        ctypes.byref(dims), int(payload), _ptr(recv, torch.bfloat16, need, "recv"),
        int(src_stride), int(dst_stride), int(dst_begin), int(num_dst),
        _ptr(out, torch.bfloat16, R * H * payload, "out"), _ptr(lse, torch.float32, R * H, "lse"),
        _ptr(status, torch.int32, 1, "status", allow_none=True), _stream(stream)))


def dcp_mla_verify_noalloc(dims, seq_lens, block_table, q, kv, kv_dtype, kv_scale,
                           softmax_scale, out, lse, status, stream=None):
    """The whole verify step over the library's fixed device scratch (no allocation)."""
    lib = load()
    B, R, H = dims.batch, dims.rows, dims.num_heads
    i32, f32 = torch.int32, torch.float32
    kv_elem = torch.uint8 if kv_dtype == KV_FP8_E4M3 else torch.bfloat16
    pool = dims.num_blocks * dims.block_size * QK_DIM
    _check(lib.dcp_mla_verify_noalloc(
        ctypes.byref(dims), _ptr(seq_lens, i32, B, "seq_lens"),
        _ptr(block_table, i32, B * dims.max_blocks_per_seq, "block_table"),
        _ptr(q, torch.bfloat16, R * H * QK_DIM, "q"),
        _ptr(kv, kv_elem, dims.dcp * pool, "kv"), int(kv_dtype),
        _ptr(kv_scale, f32, 1, "kv_scale", allow_none=True), float(softmax_scale),
        _ptr(out, torch.bfloat16, R * H * V_DIM, "out"), _ptr(lse, f32, R * H, "lse"),
        _ptr(status, i32, 1, "status"), _stream(stream)))
