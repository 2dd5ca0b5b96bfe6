"""Parity of the all-to-all exchange path and of project-before-merge (CUDA, through
the C ABI) with the oracle.

The combined output is compared with the oracle's unsharded global attention (or
its projection) element by element: |dO| <= 1e-2 + half a BF16 ulp of the oracle
value + what the BF16 wire can change (``oracle.exchange.wire_bound``) + for the
projected form what rounding each rank's output to BF16 before the projection
can change (sum_k ulp(O_r[k]) |W_V[h][p][k]|, weighted like the merge);
|dLSE| <= 1e-3 and -inf on exactly the same rows. The LSE each rank sends is
compared with the oracle's per-rank LSE the same way.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import exchange as X
from tests import _helpers as h

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import decode_context_mla_causal_gb300 as mod

    return mod


def _send_np(ex, W, G):
    return ex.send.view(torch.int16).cpu().numpy().view(np.uint16).reshape(W, G, -1)


def _check(dm, w, ref, rows_idx, heads, ex, w_v=None):
    """Compare the combined output (rows ``rows_idx`` of the step, ``heads``) and the
    sent per-rank LSE with the oracle result ``ref`` of those rows and heads."""
    W, G = w.dcp, w.dcp
    n, nh = len(rows_idx), len(heads)
    rank_out = ref["rank_out"].reshape(W, n, nh, -1)
    rank_lse = ref["rank_lse"].reshape(W, n, nh)
    out_ref = ref["out"].reshape(n, nh, -1)
    lse_ref = ref["lse"].reshape(n, nh)
    extra = 0.0
    if w_v is not None:
        wv = oracle.fp8.decode_bf16(w_v.view(torch.int16).cpu().numpy().view(np.uint16))
        wv = wv[heads].transpose(0, 2, 1)                      # [nh][512][P]
        proj_err = np.einsum("snhk,hkp->snhp", oracle.fp8.bf16_ulp(rank_out), np.abs(wv))
        rank_out, out_ref = X.project(rank_out, wv), X.project(out_ref, wv)
        fin = np.isfinite(rank_lse) & np.isfinite(lse_ref)[None]
        wgt = np.where(fin, np.exp(np.where(fin, rank_lse - lse_ref[None], 0.0)), 0.0)
        extra = np.einsum("snh,snhp->nhp", wgt, proj_err)
    out = ex.out.float().cpu().numpy()[rows_idx][:, heads]
    lse = ex.lse.cpu().numpy()[rows_idx][:, heads]
    allow = (1e-2 + 0.5 * oracle.fp8.bf16_ulp(out_ref)
             + X.wire_bound(rank_out, rank_lse, lse_ref) + extra)
    bad = ~(np.abs(out - out_ref) <= allow)
    assert not bad.any(), (w.name, int(bad.sum()), float(np.abs(out - out_ref).max()))
    assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    assert np.abs(lse[fin] - lse_ref[fin]).max(initial=0) <= 1e-3
    # the LSE each source rank sent for these rows and heads
    R, Hg, P = w.rows, w.num_heads // G, ex.payload
    send = _send_np(ex, W, G)
    for s in range(W):
        for hi, hh in enumerate(heads):
            d, hl = divmod(hh, Hg)
            _, l = X.unpack(send[s, d][None], R, Hg, P)
            got = l[0][rows_idx, hl]
            exp = rank_lse[s][:, hi]
            assert np.array_equal(np.isneginf(got), np.isneginf(exp))
            f = np.isfinite(exp)
            assert np.abs(got[f] - exp[f]).max(initial=0) <= 1e-3


def _run(dm, w, w_v=None, num_splits=None):
    step = h.run_gpu(dm, w, num_splits=num_splits)
    assert step.read_status() == 0
    ex = dm.A2AExchange(step, w_v=w_v)
    ex.pack()
    ex.combine_local()
    torch.cuda.synchronize()
    assert step.read_status() == 0
    return step, ex


@pytest.mark.parametrize("name", ["c1", "c2"])
@pytest.mark.parametrize("projected", [False, True])
def test_a2a_full_matches_oracle(dm, name, projected):
    w = workloads.generate(name, device="cuda")
    w_v = workloads.generate_w_v(w.num_heads, 128, device="cuda") if projected else None
    for ns in (1, 3):
        step, ex = _run(dm, w, w_v, num_splits=ns)
        ref = h.oracle_forward(w, per_rank=True)
        _check(dm, w, ref, list(range(w.rows)), list(range(w.num_heads)), ex, w_v)


@pytest.mark.parametrize("name,rows,heads", [
    ("c3", [(0, 0), (31, 0)], [0, 17, 127]),
    ("c4", [(0, 4), (28, 0), (28, 4), (29, 2), (31, 4)], [0, 64, 127]),
    ("c5", [(1, 2)], [5, 127]),
])
@pytest.mark.parametrize("projected", [False, True])
def test_a2a_sampled_full_size(dm, name, rows, heads, projected):
    w = workloads.generate(name, device="cuda")
    w_v = workloads.generate_w_v(w.num_heads, 128, device="cuda") if projected else None
    step, ex = _run(dm, w, w_v)
    for b in sorted({b for b, _ in rows}):
        sub = h.sequence_subset(w, b)
        js = [j for bb, j in rows if bb == b]
        ref = h.oracle_forward(sub, rows=[(0, j) for j in js], heads=heads, per_rank=True)
        _check(dm, w, ref, [b * w.qlen + j for j in js], heads, ex, w_v)
    del step, ex, w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("payload", [16, 48, 256])
def test_projected_payload_widths(dm, payload):
    w = workloads.generate("c2", device="cuda")
    w_v = workloads.generate_w_v(w.num_heads, payload, seed=payload, device="cuda")
    step, ex = _run(dm, w, w_v, num_splits=2)
    ref = h.oracle_forward(w, per_rank=True)
    _check(dm, w, ref, list(range(w.rows)), list(range(w.num_heads)), ex, w_v)


def test_per_process_layout_equals_one_device_combine(dm):
    """What each rank would receive from a real all-to-all (its column of chunks,
    source order) gives, through the per-rank combine, bit for bit the one-device
    result; and a one-rank step packs exactly that rank's send buffer."""
    w = workloads.generate("c2", device="cuda")
    G = w.dcp
    step, ex = _run(dm, w, num_splits=3)
    cw = ex.chunk_words
    send = ex.send.view(G, G, cw)
    for d in range(G):
        recv = send[:, d].contiguous().view(-1)
        one = dm.A2AExchange(step)
        one.out.zero_()
        one.combine(recv, d)
        torch.cuda.synchronize()
        Hg = w.num_heads // G
        hs = slice(d * Hg, (d + 1) * Hg)
        assert torch.equal(one.out[:, hs].view(torch.int16), ex.out[:, hs].view(torch.int16))
        assert torch.equal(one.lse[:, hs], ex.lse[:, hs])
    for r in range(G):
        st = h.run_gpu(dm, w, num_splits=3, rank_begin=r, num_ranks=1)
        mine = dm.A2AExchange(st)
        mine.pack()
        torch.cuda.synchronize()
        assert torch.equal(mine.send.view(torch.int16), send[r].reshape(-1).view(torch.int16))


def test_a2a_matches_the_fp32_merge_within_the_wire(dm):
    """The same step merged both ways: the a2a result stays within the wire bound of
    the fp32 merge (LSE equal to float rounding)."""
    w = workloads.generate("c2", device="cuda")
    step, ex = _run(dm, w, num_splits=3)
    a = ex.out.float().cpu().numpy().astype(np.float64)
    b = step.out.float().cpu().numpy().astype(np.float64)
    assert np.abs(a - b).max() <= 2 * oracle.fp8.bf16_ulp(b).max()
    la, lb = ex.lse.cpu().numpy(), step.lse.cpu().numpy()
    fin = np.isfinite(lb)
    assert np.array_equal(np.isneginf(la), np.isneginf(lb))
    assert np.abs(la[fin] - lb[fin]).max(initial=0) <= 1e-5


def test_graph_capture_of_step_and_exchange(dm):
    """The verify step plus pack, projection and combine captured in one CUDA graph and
    replayed with new lengths and queries equals fresh eager calls bit for bit."""
    w = workloads.generate("c2", device="cuda")
    w_v = workloads.generate_w_v(w.num_heads, 128, device="cuda")
    ns = 3
    step = dm.VerifyStep(h.dims_of(dm, w, ns), h.kv_dtype_of(dm, w), "cuda")
    ex = dm.A2AExchange(step, w_v=w_v)
    scale = torch.tensor([w.kv_scale], dtype=torch.float32, device="cuda")
    seq, q = w.seq_lens.clone(), w.q.clone()
    stream = torch.cuda.Stream()

    def run():
        step(q, w.kv, scale, w.softmax_scale, seq, w.block_table)
        ex.pack()
        ex.combine_local()

    with torch.cuda.stream(stream):
        run()  # warm up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        run()
    rng = np.random.default_rng(9)
    for trial in range(2):
        seq.copy_(torch.as_tensor(rng.integers(w.qlen, 4097, size=w.batch), dtype=torch.int32))
        q.copy_(torch.randn_like(q, dtype=torch.float32).to(torch.bfloat16))
        graph.replay()
        torch.cuda.synchronize()
        got = (ex.out.clone(), ex.lse.clone(), ex.send.clone())
        fresh = dm.VerifyStep(h.dims_of(dm, w, ns), h.kv_dtype_of(dm, w), "cuda")
        fex = dm.A2AExchange(fresh, w_v=w_v)
        fresh(q, w.kv, scale, w.softmax_scale, seq, w.block_table)
        fex.pack()
        fex.combine_local()
        torch.cuda.synchronize()
        assert torch.equal(got[0].view(torch.int16), fex.out.view(torch.int16))
        assert torch.equal(got[1], fex.lse)
        assert torch.equal(got[2].view(torch.int16), fex.send.view(torch.int16))


# One split: the partial kernel writes the wire format itself (dcp_mla_partial_packed).
# Its send buffer must hold the very bits of dcp_mla_partial followed by dcp_a2a_pack,
# the zero words at the end of every chunk included; the combine of it then passes the
# oracle checks above (test_a2a_*), so it is compared bit for bit here.
PACKED = [
    ("c1", None),
    ("c2", dict(batch=3, num_heads=96, qlen=3, dcp=2, interleave=2, block_size=64,
                kv_dtype="fp8", max_local_len=700, lengths=("uniform", 3, 1300))),
    ("c2", dict(batch=2, num_heads=128, qlen=5, dcp=8, interleave=64, block_size=64,
                kv_dtype="fp8", max_local_len=1024, lengths=("uniform", 5, 6000))),
    ("c2", dict(batch=2, num_heads=16, qlen=2, dcp=4, interleave=1, block_size=96,
                kv_dtype="bf16", max_local_len=400, lengths=("uniform", 2, 1100))),
    ("c3", None),
]


@pytest.mark.parametrize("idx", range(len(PACKED)))
def test_partial_packed_equals_partial_then_pack(dm, idx):
    name, ov = PACKED[idx]
    w = workloads.generate(name, device="cuda", seed_index=None if ov is None else 90 + idx,
                           overrides=ov)
    step = dm.VerifyStep(h.dims_of(dm, w, 1), h.kv_dtype_of(dm, w), "cuda")
    scale = torch.tensor([w.kv_scale], dtype=torch.float32, device="cuda")
    step.metadata(w.seq_lens, w.block_table)
    step.partial(w.q, w.kv, scale, w.softmax_scale)
    ex = dm.A2AExchange(step)
    ex.pack_ranks()
    torch.cuda.synchronize()
    want = ex.send.clone()
    ex.send.fill_(float("nan"))  # every word must be written again
    ex.partial_packed(w.q, w.kv, scale, w.softmax_scale)
    torch.cuda.synchronize()
    assert step.read_status() == 0
    assert torch.equal(ex.send.view(torch.int16), want.view(torch.int16))


def test_partial_packed_rejects_more_than_one_split(dm):
    w = workloads.generate("c1", device="cuda")
    step = dm.VerifyStep(h.dims_of(dm, w, 2), h.kv_dtype_of(dm, w), "cuda")
    ex = dm.A2AExchange(step)
    scale = torch.tensor([w.kv_scale], dtype=torch.float32, device="cuda")
    with pytest.raises(dm.DcpError) as ei:
        ex.partial_packed(w.q, w.kv, scale, w.softmax_scale)
    assert ei.value.code == dm.DCP_ERR_UNSUPPORTED


@pytest.mark.parametrize("P,offset", [(12, 0), (40, 0), (40, 4), (512, 0), (512, 4)])
def test_combine_matches_oracle_combine_on_wire_buffers(dm, P, offset):
    """dcp_a2a_combine on wire buffers written by the oracle's pack: each destination's
    merge of the BF16 values it received, within one BF16 ulp of the oracle's fp64
    combine of the same bits (LSE within float rounding). Payloads that are not a
    multiple of 8, and outputs that start 8 bytes past a 16-byte boundary (offset 4),
    take the kernel's 8-byte chunks; the rest its 16-byte chunks."""
    Bt, S, H, G = 3, 2, 16, 4
    R = Bt * S
    dims = dm.make_dims(batch=Bt, qlen=S, num_heads=H, dcp=G, interleave=1, block_size=64,
                        max_blocks_per_seq=4, max_local_len=256, num_blocks=16, num_splits=1)
    rng = np.random.default_rng(P + offset)
    rank_out = rng.standard_normal((G, R, H, P))
    rank_lse = rng.normal(0.0, 3.0, (G, R, H))
    rank_lse[rng.random((G, R, H)) < 0.2] = -np.inf       # empty ranks
    rank_lse[:, 0, 0] = -np.inf                            # an entry no rank reaches
    rank_out[np.isneginf(rank_lse)] = 0.0
    recv = X.exchange(X.pack(rank_out, rank_lse))          # [d][s][cw]
    out_ref, lse_ref = X.combine(recv, R, H, P)
    cw = X.chunk_words(R, H // G, P)
    assert cw == dm.dcp_a2a_chunk_words(dims, P)
    dev_recv = torch.from_numpy(recv.reshape(-1).view(np.int16)).cuda().view(torch.bfloat16)
    buf = torch.full((offset + R * H * P,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[offset:]
    lse = torch.full((R, H), float("nan"), dtype=torch.float32, device="cuda")
    dm.dcp_a2a_combine(dims, P, dev_recv, cw, G * cw, 0, G, out, lse)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64).reshape(R, H, P)
    assert not np.isnan(got).any()
    assert np.all(np.abs(got - out_ref) <= oracle.fp8.bf16_ulp(out_ref)), P
    gl = lse.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(gl), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    assert np.abs(gl[fin] - lse_ref[fin]).max() <= 1e-5 * (1 + np.abs(lse_ref[fin]).max())
