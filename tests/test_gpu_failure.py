"""The failure path of the partial kernel, without a GPU fault: a wait that nothing will
satisfy (the q arrival is withheld) runs out after a short limit, the kernel raises
DCP_STATUS_TIMEOUT and stops in order, and the next normal call on the same context
still matches the oracle."""

import time

import pytest
import torch

import workloads
from tests import _helpers as h

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import decode_context_mla_causal_gb300 as mod

    return mod


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_withheld_q_times_out_and_the_context_stays_usable(dm, name):
    w = workloads.generate(name, device="cuda")
    ns = 2
    step = dm.VerifyStep(h.dims_of(dm, w, ns), h.kv_dtype_of(dm, w), "cuda")
    scale = torch.tensor([w.kv_scale], dtype=torch.float32, device="cuda")
    step.metadata(w.seq_lens, w.block_table)
    torch.cuda.synchronize()
    assert step.read_status() == 0
    t0 = time.perf_counter()
    dm.dcp_mla_partial_hold_q(step.dims, w.q, w.kv, step.kv_dtype, scale, w.softmax_scale, 0,
                              step.num_ranks, step.row_len, step.page_ids, step.split_beg,
                              step.split_end, step.part_o, step.part_m, step.part_l,
                              step.status, 1_000_000, workspace=step.workspace)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert step.read_status() & dm.STATUS_TIMEOUT
    assert elapsed < 2.0  # the 1 ms limit, not the 4 s default, ended the waits
    # the same context, a normal step: status clean, parity with the oracle
    step.status.zero_()
    h.run_gpu(dm, w, step=step)
    assert step.read_status() == 0
    ref = h.oracle_forward(w)
    h.assert_parity(step.out.float().cpu().numpy(), step.lse.cpu().numpy(), ref["out"],
                    ref["lse"], name)


def test_hold_q_rejects_a_limit_outside_range(dm):
    w = workloads.generate("c1", device="cuda")
    step = dm.VerifyStep(h.dims_of(dm, w, 2), h.kv_dtype_of(dm, w), "cuda")
    scale = torch.tensor([w.kv_scale], dtype=torch.float32, device="cuda")
    for bad in (0, 5_000_000_000):
        with pytest.raises(dm.DcpError):
            dm.dcp_mla_partial_hold_q(step.dims, w.q, w.kv, step.kv_dtype, scale,
                                      w.softmax_scale, 0, step.num_ranks, step.row_len,
                                      step.page_ids, step.split_beg, step.split_end, step.part_o,
                                      step.part_m, step.part_l, step.status, bad)
