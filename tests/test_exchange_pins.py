"""Pins for the oracle of the cross-rank exchange and of project-before-merge.

Each check ties ``oracle.exchange`` to something other than itself: IEEE-754
binary32 bit patterns that are facts of the format, torch's BF16 cast (a library
routine), the permutation an all-to-all must be, the unsharded global attention
of ``oracle.attention`` (pinned by its own tests) and the linearity of the
projection. One test plants a plausible mistake (the two LSE halves swapped)
and checks that a pin catches it.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import exchange as X
from tests.test_oracle_pins import _tiny_workload


def test_lse_halves_known_patterns():
    # binary32: 1.0 = 0x3F800000, -inf = 0xFF800000, -0.0 = 0x80000000,
    # float32(pi) = 0x40490FDB, largest finite = 0x7F7FFFFF, least subnormal = 0x00000001
    cases = [(1.0, 0x0000, 0x3F80), (-np.inf, 0x0000, 0xFF80), (-0.0, 0x0000, 0x8000),
             (float(np.float32(np.pi)), 0x0FDB, 0x4049), (3.4028234663852886e38, 0xFFFF, 0x7F7F),
             (2.0 ** -149, 0x0001, 0x0000)]
    for v, lo, hi in cases:
        l, h = X.lse_halves(np.array([v]))
        assert (int(l[0]), int(h[0])) == (lo, hi), v
        back = X.lse_from_halves(l, h)[0]
        assert back == v and np.signbit(back) == np.signbit(v)


def test_lse_halves_round_trip_is_bit_exact():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    keep = ~np.isnan(vals)
    lo, hi = X.lse_halves(vals[keep].astype(np.float64))
    back = X.lse_from_halves(lo, hi).astype(np.float32)
    assert np.array_equal(back.view(np.uint32), bits[keep])


def test_bf16_bits_match_torch_cast():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-6, 6, 5000),
                        [0.0, -0.0, np.inf, -np.inf, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
    assert np.array_equal(X.to_bf16_bits(x), ref.numpy().view(np.uint16))


@pytest.mark.parametrize("R,Hg,P", [(3, 4, 512), (12, 16, 512), (1, 1, 128), (5, 3, 128)])
def test_chunk_words_aligned_and_minimal(R, Hg, P):
    cw = X.chunk_words(R, Hg, P)
    need = R * Hg * (P + 2)
    assert cw % 8 == 0 and need <= cw < need + 8


def test_exchange_is_the_all_to_all_permutation():
    W, cw = 3, 8
    send = np.zeros((W, W, cw), dtype=np.uint16)
    for s in range(W):
        for d in range(W):
            send[s, d] = 100 * s + 10 * d + np.arange(cw)
    recv = X.exchange(send)
    for d in range(W):
        for s in range(W):
            assert np.array_equal(recv[d, s], 100 * s + 10 * d + np.arange(cw))
    assert np.array_equal(X.exchange(recv), send)


def _check_combine(wl, w_v=None):
    res = A.forward(**wl)
    rank_out, out = res["rank_out"], res["out"]
    if w_v is not None:
        rank_out, out = X.project(rank_out, w_v), X.project(out, w_v)
    W, R, H, P = rank_out.shape
    got_out, got_lse = X.combine(X.exchange(X.pack(rank_out, res["rank_lse"])), R, H, P)
    fin = np.isfinite(res["lse"])
    assert np.array_equal(np.isneginf(got_lse), ~fin)
    # the LSE travels as float32: its only change is that rounding
    assert np.abs(got_lse[fin] - res["lse"][fin]).max() <= 1e-6 * max(1.0, np.abs(res["lse"][fin]).max())
    bound = X.wire_bound(rank_out, res["rank_lse"], res["lse"]) + 1e-9
    assert (np.abs(got_out - out) <= bound).all()
    return res, got_out, got_lse


@pytest.mark.parametrize("W,S,H", [(2, 1, 4), (4, 2, 8), (8, 64, 8), (1, 1, 3)])
def test_combine_of_packed_shards_matches_unsharded(W, S, H):
    wl = _tiny_workload(31 + W, L=150, W=W, S=S, bs=8 if S < 8 else 64, qlen=4, H=H)
    _check_combine(wl)


def test_single_nonempty_rank_passes_through_exactly():
    wl = _tiny_workload(21, L=30, W=4, S=64, bs=64, qlen=2, H=4)
    res, got_out, got_lse = _check_combine(wl)
    assert np.isneginf(res["rank_lse"][1:]).all()
    assert np.array_equal(X.to_bf16_bits(got_out), X.to_bf16_bits(res["rank_out"][0]))
    assert np.array_equal(got_lse, res["rank_lse"][0].astype(np.float32).astype(np.float64))


def test_all_empty_rows_give_zero_and_neg_inf():
    W, R, H, P = 2, 3, 4, 512
    send = X.pack(np.zeros((W, R, H, P)), np.full((W, R, H), -np.inf))
    out, lse = X.combine(X.exchange(send), R, H, P)
    assert (out == 0).all() and np.isneginf(lse).all()


@pytest.mark.parametrize("W,S", [(2, 1), (8, 64)])
def test_projection_commutes_with_the_merge(W, S):
    wl = _tiny_workload(41 + W, L=120, W=W, S=S, bs=8 if S < 8 else 64, qlen=3, H=8)
    rng = np.random.default_rng(W)
    w_v = rng.standard_normal((8, A.D_V, 128)) / np.sqrt(A.D_V)
    res = A.forward(**wl)
    # merge then project == project then merge (linear map, per-(row, head) weights)
    o1 = X.project(res["out"], w_v)
    o2, l2 = A.merge_shards(X.project(res["rank_out"], w_v), res["rank_lse"])
    assert np.abs(o1 - o2).max() < 1e-12 and np.abs(l2 - res["lse"]).max() < 1e-12
    # and through the wire, with a quarter of the output payload per head
    _check_combine(wl, w_v)
    assert X.chunk_words(4, 2, 512) - X.chunk_words(4, 2, 128) == 4 * 2 * (512 - 128)


def test_planted_swapped_halves_is_caught(monkeypatch):
    wl = _tiny_workload(51, L=150, W=2, S=1, bs=8, qlen=4, H=4)
    good = X.lse_halves

    def swapped(lse):
        lo, hi = good(lse)
        return hi, lo

    monkeypatch.setattr(X, "lse_halves", swapped)
    with pytest.raises(AssertionError):
        _check_combine(wl)
