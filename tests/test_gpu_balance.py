"""Wave balancing (dims.base_splits): the split plan on the device, the items the
order kernel drops, and parity of the balanced step with the oracle.

The plan is a schedule, not arithmetic: it is compared bit for bit with its host
restatement (tests/_helpers.balanced_split_counts), and the balanced step's output
with the oracle under the same gate as every other parity test (|dO| <= 1e-2 + half
a BF16 ulp, |dLSE| <= 1e-3, -inf on the same rows).
"""

import numpy as np
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


def _expected_bounds(dm, w, ns, base, row_len, rank_begin=0):
    n = h.balanced_split_counts(
        w.seq_lens.cpu().numpy(), batch=w.batch, qlen=w.qlen, num_heads=w.num_heads,
        dcp=w.dcp, interleave=w.interleave, max_local_len=w.max_local_len, num_splits=ns,
        base_splits=base, concurrent=dm.concurrent_items())
    return n, h.expected_split_bounds(n, row_len, batch=w.batch, qlen=w.qlen, num_splits=ns,
                                      subpage=dm.dcp_mla_subpage_size(w.block_size),
                                      rank_begin=rank_begin)


def _metadata(dm, w, ns, base, rank_begin=0, num_ranks=None):
    step = dm.VerifyStep(h.dims_of(dm, w, ns, base_splits=base), h.kv_dtype_of(dm, w), "cuda",
                         rank_begin=rank_begin, num_ranks=num_ranks)
    step.metadata(w.seq_lens, w.block_table)
    torch.cuda.synchronize()
    return step


def _small(seq_lens=None):
    # two decode sequences over 8 ranks: 16 (rank, sequence) pairs, one 128-row tile
    # each, so one split per pair leaves most of the device idle and balancing cuts
    # every pair into 4 or 5
    return workloads.generate("c3", device="cuda", overrides=dict(batch=2), seq_lens=seq_lens)


@pytest.mark.parametrize("lens", [None, "mixed"])
def test_device_plan_matches_host_rule(dm, lens):
    """Full decode workload (and a mixed-length copy): split bounds bit for bit."""
    seq = None
    if lens == "mixed":  # equal lengths in groups, a few very short (ties and dead pairs)
        seq = np.repeat([32768, 30000, 20000, 12000, 700, 9, 3, 1], 4)
    w = workloads.generate("c3", device="cuda", seq_lens=seq)
    ns, base = 3, 1
    step = _metadata(dm, w, ns, base)
    n, (beg, end) = _expected_bounds(dm, w, ns, base, step.row_len.cpu().numpy())
    assert np.array_equal(step.split_beg.cpu().numpy(), beg)
    assert np.array_equal(step.split_end.cpu().numpy(), end)
    if lens is None:  # 228 pairs keep one split, 28 share the last wave
        assert int((n == 1).sum()) == 256 - 28 and int(n.max()) == 3
    # a one-rank call cuts its pairs exactly as the call for the whole group
    one = _metadata(dm, w, ns, base, rank_begin=5, num_ranks=1)
    assert torch.equal(one.split_beg[0], step.split_beg[5])
    assert torch.equal(one.split_end[0], step.split_end[5])


def test_order_lists_live_items_only(dm):
    """The order kernel lists every group of slot 0 and every non-empty slot, nothing
    else, longest first, and stores how many items it listed."""
    w = _small()
    ns, base = 5, 1
    step = dm.VerifyStep(h.dims_of(dm, w, ns, base_splits=base), h.kv_dtype_of(dm, w), "cuda")
    h.run_gpu(dm, w, step=step)
    assert step.read_status() == 0
    beg, end = step.split_beg.cpu().numpy(), step.split_end.cpu().numpy()
    rt = -(-(w.qlen * w.num_heads) // 128)
    groups = beg.size
    live = [g for g in range(groups) if g % ns == 0 or end.reshape(-1)[g] > beg.reshape(-1)[g]]
    ws = step.workspace.view(torch.int32).cpu().numpy()
    items = groups * rt
    assert ws[items] == len(live) * rt
    listed = ws[: len(live) * rt]
    assert sorted(listed.tolist()) == sorted(g * rt + t for g in live for t in range(rt))
    # every pair has at least 5 subpages, so its n splits are all non-empty: the
    # listed groups are exactly the host rule's split counts, and some slots are dropped
    n, _ = _expected_bounds(dm, w, ns, base, step.row_len.cpu().numpy())
    assert len(live) == int(n.sum()) < groups


@pytest.mark.parametrize("seq", [None, [32768, 3]])
def test_balanced_step_matches_oracle(dm, seq):
    """Every row and head of the balanced step against the oracle. [32768, 3]: the
    second sequence has tokens on 3 of 8 ranks only (dead pairs, all of whose later
    slots are dropped). part_o is poisoned with NaN first: no reader may touch the
    output of a dropped slot."""
    w = _small(seq)
    ns, base = 5, 1
    step = dm.VerifyStep(h.dims_of(dm, w, ns, base_splits=base), h.kv_dtype_of(dm, w), "cuda")
    step.part_o.fill_(float("nan"))
    h.run_gpu(dm, w, step=step)
    assert step.read_status() == 0
    beg, end = step.split_beg.cpu().numpy(), step.split_end.cpu().numpy()
    assert ((end > beg).sum(axis=2) >= 2).any()  # balancing did cut pairs
    m = step.part_m.cpu().numpy()
    l = step.part_l.cpu().numpy()
    dropped = (end <= beg)
    dropped[:, :, 0] = False
    for k, b, s in zip(*np.nonzero(dropped)):  # m and l written by slot 0's item
        rows = slice(b * w.qlen, (b + 1) * w.qlen)
        assert np.isneginf(m[k, s, rows]).all() and (l[k, s, rows] == 0).all()
    ref = h.oracle_forward(w)
    h.assert_parity(step.out.float().cpu().numpy(), step.lse.cpu().numpy(), ref["out"],
                    ref["lse"], "balanced")
    # the exchange's pack reads only live splits too
    ex = dm.A2AExchange(step)
    ex.pack()
    ex.combine_local()
    torch.cuda.synchronize()
    assert not torch.isnan(ex.out.float()).any()


def test_balanced_per_rank_calls_equal_one_call(dm):
    """Each rank's metadata + partial on its own (the one-rank-per-GPU form) gives the
    merged output of the all-rank call bit for bit: the plan does not depend on the
    ranks a call covers."""
    w = _small()
    ns, base = 5, 1
    full = dm.VerifyStep(h.dims_of(dm, w, ns, base_splits=base), h.kv_dtype_of(dm, w), "cuda")
    h.run_gpu(dm, w, step=full)
    step = dm.VerifyStep(h.dims_of(dm, w, ns, base_splits=base), h.kv_dtype_of(dm, w), "cuda")
    scale = torch.tensor([w.kv_scale], dtype=torch.float32, device="cuda")
    for r in range(w.dcp):
        dm.dcp_mla_metadata(step.dims, w.seq_lens, w.block_table, r, 1, step.row_len[r],
                            step.page_ids[r], step.split_beg[r], step.split_end[r], step.status)
        dm.dcp_mla_partial(step.dims, w.q, w.kv[r], h.kv_dtype_of(dm, w), scale,
                           w.softmax_scale, r, 1, step.row_len[r], step.page_ids[r],
                           step.split_beg[r], step.split_end[r], step.part_o[r],
                           step.part_m[r], step.part_l[r], step.status)
    step.merge()
    torch.cuda.synchronize()
    assert step.read_status() == 0
    assert torch.equal(step.split_beg, full.split_beg)
    assert torch.equal(step.out, full.out) and torch.equal(step.lse, full.lse)
