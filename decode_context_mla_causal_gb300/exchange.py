"""The cross-rank exchange of a verify step's per-rank results (the a2a backend).

"Context Parallel Guide (PCP & DCP)", ``comm_backend`` a2a: one all-to-all
carries every rank's output with its LSE packed alongside (the float32 LSE as
two 16-bit halves of the BF16 buffer) and each destination combines locally, so
that every rank ends with its slice of the heads; ``enable_project_before_merge``
projects each rank's output by the head's W_V first, which shrinks the payload.
The packing, projection and combine run in ``libdcpmla.so``; this module only
owns the buffers and, with one rank per process, the collective call.
"""

from __future__ import annotations

import torch

from . import binding as B


def a2a_exchange(send: torch.Tensor, group=None) -> torch.Tensor:
    """One rank's all-to-all of equal chunks: ``send`` holds ``dcp`` chunks (one per
    destination, in order); the result holds the chunk each source sent to this
    rank, in source order. Runs on whatever backend ``group`` uses (NCCL for CUDA
    tensors, gloo for host tensors); the chunks are moved, never interpreted."""
    recv = torch.empty_like(send)
    torch.distributed.all_to_all_single(recv, send, group=group)
    return recv


class A2AExchange:
    """Send buffers and combine outputs for a ``VerifyStep``'s ranks.

    ``w_v`` (bf16 ``[H][P][512]``, optional) turns on project-before-merge with
    payload P; without it the payload is the 512 latent dims.
    """

    def __init__(self, step, w_v: torch.Tensor | None = None):
        dims = step.dims
        self.step = step
        self.w_v = w_v
        self.payload = B.V_DIM if w_v is None else int(w_v.shape[1])
        self.chunk_words = B.dcp_a2a_chunk_words(dims, self.payload)
        dev = step.part_o.device
        R, H = dims.rows, dims.num_heads
        n = step.num_ranks * dims.dcp
        # what is exchanged; with a projection, the per-rank BF16 outputs come first
        self.send = torch.empty(n * self.chunk_words, dtype=torch.bfloat16, device=dev)
        self.packed = self.send if w_v is None else torch.empty(
            n * B.dcp_a2a_chunk_words(dims, B.V_DIM), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((R, H, self.payload), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((R, H), dtype=torch.float32, device=dev)

    def pack(self, stream=None):
        """Each rank's merged (optionally projected) output and LSE into its send buffer."""
        self.pack_ranks(stream)
        if self.w_v is not None:
            self.project(stream)

    def partial_packed(self, q, kv, kv_scale, softmax_scale, stream=None):
        """One split: the step's partial attention writing each rank's BF16 output and
        LSE straight into the send buffer (payload 512; the step's fp32 partials are
        not written), in place of ``step.partial`` followed by ``pack_ranks``."""
        s = self.step
        B.dcp_mla_partial_packed(s.dims, q, kv, s.kv_dtype, kv_scale, softmax_scale,
                                 s.rank_begin, s.num_ranks, s.row_len, s.page_ids, s.split_beg,
                                 s.split_end, self.packed, s.status, stream,
                                 workspace=s.workspace)

    def pack_ranks(self, stream=None):
        """Each rank's merged BF16 output and LSE (payload 512)."""
        s = self.step
        B.dcp_a2a_pack(s.dims, s.num_ranks, s.part_o, s.part_m, s.part_l, self.packed,
                       status=s.status, stream=stream)

    def project(self, stream=None):
        """Project-before-merge of the packed outputs into the send buffer."""
        s = self.step
        B.dcp_a2a_project(s.dims, s.num_ranks, self.packed, self.w_v, self.payload, self.send,
                          status=s.status, stream=stream)

    def combine_local(self, stream=None):
        """All dcp ranks live on this device: every destination's combine, reading
        the send buffers in place (the all-to-all is a change of strides)."""
        s = self.step
        if s.rank_begin != 0 or s.num_ranks != s.dims.dcp:
            raise ValueError("combine_local needs every rank of the group in this step")
        cw = self.chunk_words
        B.dcp_a2a_combine(s.dims, self.payload, self.send, s.dims.dcp * cw, cw, 0, s.dims.dcp,
                          self.out, self.lse, status=s.status, stream=stream)
        return self.out, self.lse

    def combine(self, recv: torch.Tensor, rank: int, stream=None):
        """This process's destination combine after ``a2a_exchange`` (its heads only)."""
        s = self.step
        B.dcp_a2a_combine(s.dims, self.payload, recv, self.chunk_words, 0, rank, 1, self.out,
                          self.lse, status=s.status, stream=stream)
        return self.out, self.lse
