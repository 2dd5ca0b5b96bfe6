"""The no-allocation verify step: same results as the allocating entry points.

dcp_mla_verify_noalloc is for callers that cannot call cudaMalloc (code inside
an allocator callback, or a runtime that owns the device heap): it keeps every
intermediate in a fixed device array inside the library. This file is named to
be collected last; it also passes when run on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import workloads
from tests import _helpers as h


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__

    __graft_entry__.build()
    import decode_context_mla_causal_gb300 as mod

    return mod


@pytest.mark.gpu
@pytest.mark.parametrize("name,num_splits", [("c1", 2), ("c2", 3)])
def test_noalloc_matches_allocating_path_twice(dm, name, num_splits):
    w = workloads.generate(name, device="cuda")
    dims = h.dims_of(dm, w, num_splits)
    kvt = h.kv_dtype_of(dm, w)
    scale = torch.tensor([w.kv_scale], dtype=torch.float32, device="cuda")
    ref = dm.VerifyStep(dims, kvt, "cuda")
    ref(w.q, w.kv, scale, w.softmax_scale, w.seq_lens, w.block_table)
    torch.cuda.synchronize()
    assert ref.read_status() == 0
    bufs = [(torch.full_like(ref.out, float("nan")), torch.full_like(ref.lse, float("nan")),
             torch.zeros(1, dtype=torch.int32, device="cuda")) for _ in range(2)]
    torch.cuda.synchronize()

    def device_memory():
        # the driver's free bytes (cudaMemGetInfo) and torch's allocator counters
        st = torch.cuda.memory_stats()
        return (torch.cuda.mem_get_info()[0], st.get("allocated_bytes.all.current", 0),
                st.get("reserved_bytes.all.current", 0))

    for call, (out, lse, status) in enumerate(bufs):
        before = device_memory()
        dm.dcp_mla_verify_noalloc(dims, w.seq_lens, w.block_table, w.q, w.kv, kvt, scale,
                                  w.softmax_scale, out, lse, status)
        torch.cuda.synchronize()
        if call == 1:
            # the first call has looked up the static array's address; a later call
            # takes no device memory at all
            assert device_memory() == before
        assert int(status.item()) == 0, call
        st = h.compare(out.float().cpu().numpy(), lse.cpu().numpy(),
                       ref.out.float().cpu().numpy().astype(np.float64),
                       ref.lse.cpu().numpy().astype(np.float64))
        assert st["bad_out"] == 0 and st["bad_lse"] == 0 and st["inf_ok"], (call, st)


@pytest.mark.gpu
def test_noalloc_rejects_dims_beyond_its_scratch(dm):
    w = workloads.generate("c1", device="cuda")
    dims = h.dims_of(dm, w, 2)
    dims.num_splits = 4096  # partial buffers far beyond the fixed scratch
    out = torch.empty((w.rows, w.num_heads, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.rows, w.num_heads), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(dm.DcpError) as ei:
        dm.dcp_mla_verify_noalloc(dims, w.seq_lens, w.block_table, w.q, w.kv,
                                  h.kv_dtype_of(dm, w), None, w.softmax_scale, out, lse, status)
    assert ei.value.code == dm.DCP_ERR_UNSUPPORTED
    assert "scratch" in dm.dcp_last_error()
