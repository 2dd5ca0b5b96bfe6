"""Host-side logic of the package that needs no GPU: the static split count and the
wave-balancing plan."""

import math

import numpy as np
import pytest

from decode_context_mla_causal_gb300.step import choose_num_splits


def _cost(ns, batch, qlen, heads, ranks, bound, slots=76):
    # the model stated in choose_num_splits' docstring, for the brute-force check
    tiles = max(1, math.ceil(bound / 64))
    base = max(1, batch * ranks * math.ceil(qlen * heads / 128))
    return math.ceil(base * ns / slots) * (tiles / ns + 11.0) + 0.5 * ns


@pytest.mark.parametrize("shape,want", [
    ((1, 3, 8, 2, 100, 16), 2),         # tiny
    ((4, 3, 96, 2, 2048, 64), 3),       # small
    ((32, 1, 128, 8, 4096, 64), 1),     # decode: 256 items already fill 3.4 waves
    ((32, 5, 128, 8, 16384, 64), 1),    # spec-verify: 1280 items
    ((4, 3, 128, 8, 131072, 64), 7),    # long-context: 96 items of 2048 tiles
])
def test_split_choices_of_the_workloads(shape, want):
    assert choose_num_splits(*shape, sms=152) == want


@pytest.mark.parametrize("shape", [
    (1, 1, 8, 1, 64, 16), (1, 3, 128, 8, 1 << 20, 64), (64, 5, 128, 8, 512, 64),
    (3, 2, 40, 3, 999, 96), (128, 1, 128, 8, 131072, 64)])
def test_split_choice_is_the_cheapest_in_range(shape):
    ns = choose_num_splits(*shape, sms=152)
    tiles = max(1, math.ceil(shape[4] / 64))
    assert 1 <= ns <= min(64, tiles)
    best = min(_cost(k, *shape[:5]) for k in range(1, min(64, tiles) + 1))
    assert _cost(ns, *shape[:5]) == pytest.approx(best)


def test_one_long_item_is_split_and_many_items_are_not():
    # one (rank, sequence, row tile) of 2048 tiles: split until the SMs are busy
    assert choose_num_splits(1, 1, 128, 1, 131072, 64, sms=152) >= 32
    # thousands of items already fill many waves: no split
    assert choose_num_splits(1024, 1, 128, 8, 4096, 64, sms=152) == 1


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_algorithmic_counts_follow_their_definitions(name):
    """bench.py's per-step counts: every global token read once (by the rank that
    owns it, counted rank by rank), 2 * (576 + 512) flops per (row, head, visible
    token) with the visible tokens counted per row, the cache bytes of those tokens
    plus q once and the BF16 output once."""
    import bench
    import workloads
    from oracle import metadata as M

    w = workloads.generate(name, device="cpu")
    tokens, flops, nbytes = bench.algorithmic(w)
    lens = [int(x) for x in w.seq_lens.numpy()]
    owned = sum(M.count_local(L, r, w.dcp, w.interleave) for L in lens for r in range(w.dcp))
    assert tokens == owned == sum(lens)
    visible = sum(M.row_boundary(L, w.qlen, j, True) for L in lens for j in range(w.qlen))
    assert flops == w.num_heads * visible * 2 * (576 + 512)
    elem = 1 if w.kv_dtype == "fp8" else 2
    rows = w.batch * w.qlen
    assert nbytes == owned * 576 * elem + rows * w.num_heads * (576 + 512) * 2


def test_long_context_counts():
    # B4 H128 qlen3 L = 2^20, FP8: the figures the roofline of the bench line rests on
    import types

    import torch

    import bench

    w = types.SimpleNamespace(seq_lens=torch.full((4,), 1 << 20), num_heads=128, qlen=3,
                              causal=True, kv_dtype="fp8", batch=4)
    tokens, flops, nbytes = bench.algorithmic(w)
    assert tokens == 4 << 20
    assert flops == 4 * 128 * 2176 * (3 * (1 << 20) - 3)
    assert nbytes == (4 << 20) * 576 + 12 * 128 * 1088 * 2 == 2419261440


def test_nvml_sampler_summary_decodes_reason_bits():
    """The bench's clock summary: median SM clock, maximum, and the clocks-event reason
    bits of the NVML API mapped to names (samples injected; no GPU or NVML needed)."""
    import bench

    s = bench.NvmlSampler.__new__(bench.NvmlSampler)
    s.samples = [(2070, 2070, 900.0, 0), (2070, 2070, 1000.0, 0x4),
                 (1900, 2070, 1100.0, 0x4 | 0x40), (2070, 2070, 950.0, 0x1)]
    out = s.summary()
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070 and out["samples"] == 4
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert out["power_w_max"] == 1100.0
    s.samples = []
    assert s.summary()["reasons"] == ["no samples"]


def test_split_plan_of_the_workloads():
    from decode_context_mla_causal_gb300.step import choose_split_plan

    # decode: 256 items of 64 tiles leave 28 of 76 slots busy in the 4th wave; the 28
    # shortest pairs may take up to 3 splits to fill it
    assert choose_split_plan(32, 1, 128, 8, 4096, 64, concurrent=76) == (3, 1)
    # spec-verify (1280 items: 64 of 76 in the last wave) and long-context (672
    # items: 64 of 76) have nothing to balance
    assert choose_split_plan(32, 5, 128, 8, 16384, 64, concurrent=76) == (1, 0)
    assert choose_split_plan(4, 3, 128, 8, 131072, 64, concurrent=76) == (7, 0)
    # short sequences are not cut below 8 tiles a piece
    assert choose_split_plan(1, 3, 8, 2, 100, 16, concurrent=76) == (2, 0)


def _makespan(costs, slots):
    """List scheduling in the given order (the hardware hands each next cluster to
    the first free slot): the finish time of the last item."""
    import heapq

    free = [0.0] * slots
    heapq.heapify(free)
    end = 0.0
    for c in costs:
        t = heapq.heappop(free) + c
        end = max(end, t)
        heapq.heappush(free, t)
    return end


def test_balanced_plan_shortens_the_decode_schedule():
    """The decode shape (32 sequences x 8 ranks, 4096 local tokens each): with the
    per-item cost of the split model (tiles + 11), longest first on 76 slots, the
    balanced counts finish the step earlier than one split per pair."""
    from tests._helpers import balanced_split_counts

    seq = np.full(32, 32768)
    kw = dict(batch=32, qlen=1, num_heads=128, dcp=8, interleave=1, max_local_len=4096)
    n = balanced_split_counts(seq, num_splits=3, base_splits=1, concurrent=76, **kw)
    assert sorted(np.unique(n).tolist()) == [1, 2, 3]
    assert int((n == 1).sum()) == 228 and int(n.sum()) == 228 + 76
    costs = sorted((64 / k + 11.0 for k in n.reshape(-1) for _ in range(k)), reverse=True)
    plain = _makespan([64 + 11.0] * 256, 76)
    balanced = _makespan(costs, 76)
    assert plain == pytest.approx(4 * 75.0)
    assert balanced < 0.9 * plain


def test_balanced_plan_keeps_uneven_batches_whole():
    """Lengths that already spread over the waves (spec-verify's log-uniform mix) or
    a last wave more than half full: every pair keeps base_splits."""
    from tests._helpers import balanced_split_counts

    rng = np.random.default_rng(3)
    seq = rng.integers(8192, 131072, size=32)
    kw = dict(batch=32, qlen=5, num_heads=128, dcp=8, interleave=1, max_local_len=16384)
    n = balanced_split_counts(seq, num_splits=2, base_splits=1, concurrent=76, **kw)
    assert (n == 1).all()
