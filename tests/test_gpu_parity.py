"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Metadata is compared bit-exactly (padding included). Outputs are compared
element by element: |dO| <= 1e-2 + half a BF16 ulp of the oracle value,
|dLSE| <= 1e-3 (natural log), and -inf LSE on exactly the same rows.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _helpers as h

pytestmark = pytest.mark.gpu

_CACHE = {}


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import decode_context_mla_causal_gb300 as mod

    return mod


def workload(name, **kw):
    key = (name, tuple(sorted(kw.items())))
    if key not in _CACHE:
        if name in ("c3", "c4", "c5"):
            for k in [k for k in _CACHE if k[0] in ("c3", "c4", "c5")]:
                del _CACHE[k]
            torch.cuda.empty_cache()
        _CACHE[key] = workloads.generate(name, device="cuda", **kw)
    return _CACHE[key]


def _gpu_metadata(dm, w, num_splits, causal=True):
    step = dm.VerifyStep(h.dims_of(dm, w, num_splits, causal), h.kv_dtype_of(dm, w), "cuda")
    step.metadata(w.seq_lens, w.block_table)
    torch.cuda.synchronize()
    return step


def _check_metadata(dm, w, num_splits, causal=True):
    step = _gpu_metadata(dm, w, num_splits, causal)
    ref = h.oracle_metadata(w, num_splits, causal=causal)
    for f in ("row_len", "page_ids", "split_beg", "split_end"):
        got = getattr(step, f).cpu().numpy()
        assert np.array_equal(got, ref[f]), f
    assert step.read_status() == ref["status"]


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_metadata_bit_exact(dm, name):
    w = workload(name)
    for ns in (1, 3, dm.choose_num_splits(w.batch, w.qlen, w.num_heads, w.dcp,
                                          w.max_local_len, w.block_size, dm.num_sms())):
        _check_metadata(dm, w, ns)


@pytest.mark.parametrize("W,S,bs,qlen", [
    (2, 1, 16, 3), (8, 1, 64, 1), (8, 64, 64, 5), (4, 16, 96, 3), (2, 2, 256, 2), (3, 1, 96, 4)])
@pytest.mark.parametrize("causal", [True, False])
def test_metadata_edge_sweep(dm, W, S, bs, qlen, causal):
    lens = list(range(qlen, 4 * W * S + qlen + 1))
    bound = -(-(4 * W * S + qlen) // W) + S
    w = workloads.generate("c1", device="cuda", seq_lens=lens, overrides=dict(
        batch=len(lens), num_heads=1, qlen=qlen, dcp=W, interleave=S, block_size=bs,
        max_local_len=bound, kv_dtype="bf16"))
    for ns in (1, 2, 5):
        _check_metadata(dm, w, ns, causal)


def _full_parity(dm, w, num_splits=None, per_rank=True, causal=True):
    step = h.run_gpu(dm, w, num_splits=num_splits, causal=causal)
    assert step.read_status() == 0
    ref = h.oracle_forward(w, per_rank=per_rank, causal=causal)
    R, H = w.rows, w.num_heads
    st = h.assert_parity(step.out.float().cpu().numpy(), step.lse.cpu().numpy(),
                         ref["out"].reshape(R, H, -1), ref["lse"].reshape(R, H), w.name)
    if per_rank:
        rl = step.rank_lse.cpu().numpy()
        exp = ref["rank_lse"].reshape(w.dcp, R, H)
        assert np.array_equal(np.isneginf(rl), np.isneginf(exp))
        fin = np.isfinite(exp)
        assert np.abs(rl[fin] - exp[fin]).max(initial=0) <= 1e-3
    return st


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_parity_full(dm, name):
    w = workload(name)
    _full_parity(dm, w)


# Sampled (sequence, verify row) pairs, every head of each. At H = 128 each verify row
# is one 128-row tile of the partial kernel, so every row tile is covered, and every
# row sees every split of its (rank, sequence) pairs. Spec-verify covers a long
# sequence in full and the short ones (5, 70, 300, 511 tokens) that leave ranks empty.
ALL_HEADS = list(range(128))


@pytest.mark.parametrize("name,rows,heads", [
    ("c3", [(0, 0), (17, 0), (31, 0)], ALL_HEADS),
    ("c4", [(0, 0), (0, 1), (0, 2), (0, 3), (0, 4), (13, 2), (28, 0), (28, 4), (29, 1),
            (30, 3), (31, 4)], ALL_HEADS),
    ("c5", [(0, 0), (0, 1), (0, 2), (3, 1)], ALL_HEADS),
])
def test_parity_sampled_full_size(dm, name, rows, heads):
    w = workload(name)
    step = h.run_gpu(dm, w)
    assert step.read_status() == 0
    out = step.out.float().cpu().numpy()
    lse = step.lse.cpu().numpy()
    for b in sorted({b for b, _ in rows}):
        sub = h.sequence_subset(w, b)
        js = [j for bb, j in rows if bb == b]
        ref = h.oracle_forward(sub, rows=[(0, j) for j in js], heads=heads, per_rank=False)
        got_o = np.stack([out[b * w.qlen + j][heads] for j in js])
        got_l = np.stack([lse[b * w.qlen + j][heads] for j in js])
        h.assert_parity(got_o, got_l, ref["out"], ref["lse"], (name, b))
    assert np.isfinite(out).all()


SMALL = [
    dict(batch=2, num_heads=8, qlen=1, dcp=2, interleave=1, block_size=16, kv_dtype="fp8",
         max_local_len=256, lengths=("uniform", 1, 500)),
    dict(batch=3, num_heads=16, qlen=2, dcp=3, interleave=1, block_size=96, kv_dtype="bf16",
         max_local_len=400, lengths=("uniform", 2, 1100)),
    dict(batch=2, num_heads=96, qlen=3, dcp=2, interleave=2, block_size=64, kv_dtype="fp8",
         max_local_len=700, lengths=("uniform", 3, 1300)),
    dict(batch=2, num_heads=128, qlen=5, dcp=8, interleave=64, block_size=64, kv_dtype="fp8",
         max_local_len=1024, lengths=("uniform", 5, 6000)),
    dict(batch=3, num_heads=128, qlen=4, dcp=4, interleave=16, block_size=256, kv_dtype="bf16",
         max_local_len=600, lengths=("uniform", 4, 2000)),
    dict(batch=1, num_heads=40, qlen=3, dcp=1, interleave=1, block_size=64, kv_dtype="fp8",
         max_local_len=900, lengths=("fixed", 777)),
    dict(batch=4, num_heads=128, qlen=3, dcp=8, interleave=1, block_size=64, kv_dtype="fp8",
         max_local_len=64, lengths=("uniform", 3, 40)),
]


@pytest.mark.parametrize("idx", range(len(SMALL)))
@pytest.mark.parametrize("num_splits", [1, 3])
def test_parity_small_grid(dm, idx, num_splits):
    w = workloads.generate("c2", device="cuda", seed_index=50 + idx, overrides=SMALL[idx])
    _full_parity(dm, w, num_splits=num_splits)


def test_parity_non_causal(dm):
    w = workloads.generate("c2", device="cuda", seed_index=70, overrides=dict(
        batch=2, num_heads=32, qlen=4, max_local_len=2048))
    _full_parity(dm, w, num_splits=2, causal=False)


def test_negative_control_boundary_mutation(dm):
    # Only the row boundary changes (as in the PR's negative control): the GPU
    # result must fail against the mutated oracle while passing the real one.
    w = workloads.generate("c2", device="cuda", seed_index=71, overrides=dict(batch=1),
                           seq_lens=[3001])
    step = h.run_gpu(dm, w, num_splits=2)
    out = step.out.float().cpu().numpy()
    lse = step.lse.cpu().numpy()
    good = h.oracle_forward(w, per_rank=False)
    h.assert_parity(out, lse, good["out"].reshape(out.shape), good["lse"].reshape(lse.shape))
    for mut in (dict(boundary=oracle.metadata.committed_prefix_boundary), dict(causal=False)):
        bad = h.oracle_forward(w, per_rank=False, **mut)
        st = h.compare(out, lse, bad["out"].reshape(out.shape), bad["lse"].reshape(lse.shape))
        assert st["bad_out"] > 0 or st["bad_lse"] > 0, st


def _used_rows(w):
    md = h.oracle_metadata(w, 1)
    P = md["subpage"]
    used = np.zeros((w.dcp, w.num_blocks * w.block_size), dtype=bool)
    for r in range(w.dcp):
        for b in range(w.batch):
            n = md["row_len"][r, b * w.qlen + w.qlen - 1]
            li = np.arange(n)
            used[r, md["page_ids"][r, b][li // P] * P + li % P] = True
    return used


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
def test_nan_poison_outside_valid_tokens(dm, kv):
    w = workloads.generate("c2", device="cuda", seed_index=72, overrides=dict(
        batch=3, num_heads=96, kv_dtype=kv, max_local_len=2100), seq_lens=[1025, 2049, 131])
    ref_step = h.run_gpu(dm, w, num_splits=3)
    ref_out = ref_step.out.clone()
    used = torch.from_numpy(_used_rows(w)).to("cuda")
    flat = w.kv.view(w.dcp, -1, 576)
    if kv == "fp8":
        flat[~used] = 0x7F
    else:
        flat.view(torch.int16)[~used] = 0x7FC0
    step = h.run_gpu(dm, w, num_splits=3)
    assert torch.isfinite(step.out.float()).all()
    assert torch.equal(step.out, ref_out)


def test_graph_capture_replay_at_static_bound(dm):
    wa = workload("c2")
    ns = 4
    step = dm.VerifyStep(h.dims_of(dm, wa, ns), h.kv_dtype_of(dm, wa), "cuda")
    scale = torch.tensor([wa.kv_scale], dtype=torch.float32, device="cuda")
    seq = wa.seq_lens.clone()
    table = wa.block_table.clone()
    q = wa.q.clone()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        step(q, wa.kv, scale, wa.softmax_scale, seq, table)  # warm up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(q, wa.kv, scale, wa.softmax_scale, seq, table)
    rng = np.random.default_rng(5)
    for trial in range(3):
        lens = rng.integers(wa.qlen, 4097, size=wa.batch)
        lens[trial % wa.batch] = wa.qlen  # a row with nothing before it
        seq.copy_(torch.as_tensor(lens, dtype=torch.int32))
        q.copy_(torch.randn_like(q, dtype=torch.float32).to(torch.bfloat16))
        graph.replay()
        torch.cuda.synchronize()
        got_o, got_l = step.out.clone(), step.lse.clone()
        fresh = dm.VerifyStep(h.dims_of(dm, wa, ns), h.kv_dtype_of(dm, wa), "cuda")
        fresh(q, wa.kv, scale, wa.softmax_scale, seq, table)
        torch.cuda.synchronize()
        assert torch.equal(got_o, fresh.out) and torch.equal(got_l, fresh.lse)


def test_per_rank_calls_equal_one_call(dm):
    w = workload("c2")
    ns = 2
    full = h.run_gpu(dm, w, num_splits=ns)
    step = dm.VerifyStep(h.dims_of(dm, w, ns), h.kv_dtype_of(dm, w), "cuda")
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
    assert torch.equal(step.out, full.out) and torch.equal(step.lse, full.lse)


def _item_tiles(step, w, subpage):
    """Tile counts of the work items in natural order (rank, sequence, split, row tile)."""
    R = w.rows
    rt = -(-(w.qlen * w.num_heads) // 128)
    row_len = step.row_len.cpu().numpy()
    beg, end = step.split_beg.cpu().numpy(), step.split_end.cpu().numpy()
    tiles = []
    for k in range(step.num_ranks):
        for b in range(w.batch):
            for s in range(step.dims.num_splits):
                for t in range(rt):
                    r0 = t * 128
                    r1 = min(w.qlen * w.num_heads, r0 + 128) - 1
                    js = range(r0 // w.num_heads, r1 // w.num_heads + 1)
                    max_l = max(int(row_len[k, b * w.qlen + j]) for j in js)
                    t0 = int(beg[k, b, s]) * subpage
                    t1 = min(int(end[k, b, s]) * subpage, max_l)
                    tiles.append(-(-(t1 - t0) // 64) if t1 > t0 else 0)
    return np.array(tiles)


def test_item_order_is_longest_first_and_changes_nothing(dm):
    """The order kernel sorts groups of row tiles longest first; results are unchanged."""
    w = workload("c4")  # sequence lengths from 5 to 131072: very uneven work items
    step = h.run_gpu(dm, w)
    assert step.read_status() == 0
    tiles = _item_tiles(step, w, dm.dcp_mla_subpage_size(w.block_size))
    order = step.workspace.view(torch.int32)[: tiles.size].cpu().numpy()
    assert np.array_equal(np.sort(order), np.arange(tiles.size))
    # groups (rank, sequence, split) longest first, each group's row tiles adjacent
    rt = -(-(w.qlen * w.num_heads) // 128)
    groups = order.reshape(-1, rt)
    assert (groups == groups[:, :1] + np.arange(rt)[None]).all()
    assert (groups[:, 0] % rt == 0).all()
    group_max = np.minimum(tiles.reshape(-1, rt).max(axis=1), 4095)
    assert (np.diff(group_max[groups[:, 0] // rt]) <= 0).all()
    ordered = [x.clone() for x in (step.part_o, step.part_m, step.part_l, step.out, step.lse)]
    scale = torch.tensor([w.kv_scale], dtype=torch.float32, device="cuda")
    dm.dcp_mla_partial(step.dims, w.q, w.kv, step.kv_dtype, scale, w.softmax_scale, 0,
                       step.num_ranks, step.row_len, step.page_ids, step.split_beg,
                       step.split_end, step.part_o, step.part_m, step.part_l, step.status)
    step.merge()
    torch.cuda.synchronize()
    assert step.read_status() == 0
    for a, b in zip(ordered, (step.part_o, step.part_m, step.part_l, step.out, step.lse)):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                           b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16))


def test_device_errors_set_status_and_stay_safe(dm):
    w = workloads.generate("c2", device="cuda", seed_index=73, overrides=dict(
        batch=3, num_heads=16, max_local_len=512), seq_lens=[2, 900, 5000])
    table = w.block_table.clone()
    table[1, 3] = w.num_blocks + 1000  # out of range block id
    table[1, 4] = -7
    w.block_table = table
    step = h.run_gpu(dm, w, num_splits=2)
    st = step.read_status()
    assert st & dm.STATUS_BAD_SEQ_LEN
    assert st & dm.STATUS_LOCAL_OVER_BOUND
    assert st & dm.STATUS_BAD_BLOCK_ID
    assert torch.isfinite(step.out.float()).all()
    assert (step.row_len <= 512).all()
