"""Pins for the two tolerance helpers every parity gate uses.

``oracle.fp8.bf16_ulp`` is tied to the spacing of torch's BF16 numbers (a library
type): for BF16 values across the whole exponent range, subnormals included, the
distance to the next larger BF16 number, read off the bit patterns. A few spacings
are facts of the format and are checked literally.

``oracle.exchange.wire_bound`` bounds what rounding each rank's output to BF16 can
change in the combined output. It is checked against the exact change on random
cases (the bound must hold), against the closed form it must not exceed (the merge
weights sum to 1, so the bound is at most the largest spacing among the rank
outputs), and for tightness (the realised change reaches a fair share of it).
Each helper also has a planted mistake that a pin must catch.
"""

import numpy as np
import pytest
import torch

from oracle import exchange as X
from oracle import fp8 as F


def _bf16_from_bits(bits):
    return torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16).float().numpy().astype(np.float64)


def _torch_spacing_at(bits):
    """Distance from the positive BF16 number with these bits to the next one up."""
    b = np.asarray(bits, dtype=np.uint32)
    return _bf16_from_bits(b + 1) - _bf16_from_bits(b)


def _all_positive_finite_bits():
    return np.arange(0x0001, 0x7F80, dtype=np.uint32)  # 0x7F80 is +inf


def test_bf16_ulp_equals_torch_spacing_on_every_positive_bf16_number():
    bits = _all_positive_finite_bits()[:-1]  # the largest finite has no finite successor
    vals = _bf16_from_bits(bits)
    assert np.array_equal(F.bf16_ulp(vals), _torch_spacing_at(bits))
    assert np.array_equal(F.bf16_ulp(-vals), _torch_spacing_at(bits))


def test_bf16_ulp_is_constant_between_neighbours():
    # any real value between two BF16 neighbours of one binade has their spacing
    rng = np.random.default_rng(11)
    bits = rng.integers(0x0080, 0x7F7F, size=20000).astype(np.uint32)
    lo, hi = _bf16_from_bits(bits), _bf16_from_bits(bits + 1)
    same_binade = np.floor(np.log2(lo)) == np.floor(np.log2(hi))
    t = rng.uniform(0.0, 1.0, size=bits.size)
    x = lo + t * (hi - lo)
    x = np.where(x < hi, x, lo)
    assert np.array_equal(F.bf16_ulp(x[same_binade]), (hi - lo)[same_binade])


def test_bf16_ulp_format_facts():
    # 8 significant bits: spacing 2^-7 in [1, 2), 2^-5 in [4, 8), 2^-8 in [0.5, 1);
    # subnormal spacing 2^-133 below 2^-126; zero takes the subnormal spacing
    assert F.bf16_ulp(np.array([1.0]))[0] == 2.0 ** -7
    assert F.bf16_ulp(np.array([1.9921875]))[0] == 2.0 ** -7
    assert (F.bf16_ulp(np.array([4.0, 5.5, 7.96875])) == 2.0 ** -5).all()
    assert F.bf16_ulp(np.array([0.75]))[0] == 2.0 ** -8
    assert F.bf16_ulp(np.array([2.0 ** -130, 0.0]))[0] == 2.0 ** -133
    assert F.bf16_ulp(np.array([0.0]))[0] == 2.0 ** -133


def test_planted_wrong_bf16_spacing_is_caught():
    def wrong(x):  # one bit too coarse: 2^(e-6)
        return 2.0 * F.bf16_ulp(x)
    bits = _all_positive_finite_bits()[:-1]
    vals = _bf16_from_bits(bits)
    assert not np.array_equal(wrong(vals), _torch_spacing_at(bits))


def _random_shards(rng, W, R, H, P, spread):
    rank_out = rng.standard_normal((W, R, H, P)) * 10.0 ** rng.uniform(-2, 1, (W, R, H, 1))
    rank_lse = rng.standard_normal((W, R, H)) * spread
    if W > 1:
        rank_lse[rng.integers(0, W), 0, 0] = -np.inf  # an empty rank
    m = np.max(rank_lse, axis=0)
    lse = m + np.log(np.sum(np.exp(rank_lse - m), axis=0))
    return rank_out, rank_lse, lse


def _exact_wire_change(rank_out, rank_lse, lse):
    """|combine(BF16(O_s)) - combine(O_s)| in fp64, with the exact merge weights."""
    w = np.exp(rank_lse - lse[None])
    rounded = F.round_to_bf16(rank_out)
    return np.abs(np.einsum("s...,s...p->...p", w, rounded - rank_out))


@pytest.mark.parametrize("W,spread", [(2, 0.5), (4, 3.0), (8, 1.0), (1, 1.0)])
def test_wire_bound_holds_and_is_not_vacuous(W, spread):
    rng = np.random.default_rng(100 + W)
    rank_out, rank_lse, lse = _random_shards(rng, W, 3, 5, 64, spread)
    bound = X.wire_bound(rank_out, rank_lse, lse)
    change = _exact_wire_change(rank_out, rank_lse, lse)
    assert (change <= bound * (1 + 1e-12)).all()
    # the merge weights sum to 1: never above the largest spacing among the shards
    assert (bound <= F.bf16_ulp(rank_out).max(axis=0) * (1 + 1e-12)).all()
    # tight: RNE moves a value by half its spacing on average, so the realised change
    # is a fair share of a full-spacing bound
    assert change.sum() >= 0.05 * bound.sum()


def test_wire_bound_is_zero_weight_for_empty_ranks():
    rank_out = np.full((2, 1, 1, 4), 1000.0)
    rank_lse = np.array([[[0.0]], [[-np.inf]]])
    lse = np.array([[0.0]])
    assert np.array_equal(X.wire_bound(rank_out, rank_lse, lse), F.bf16_ulp(rank_out[0]))


def test_planted_inverted_merge_weights_are_caught():
    rng = np.random.default_rng(7)
    rank_out, rank_lse, lse = _random_shards(rng, 4, 3, 5, 64, 3.0)

    def wrong(ro, rl, ls):  # weights exp(LSE - LSE_s) instead of exp(LSE_s - LSE)
        fin = np.isfinite(rl)
        w = np.where(fin, np.exp(np.where(fin, ls[None] - rl, 0.0)), 0.0)
        return np.einsum("s...,s...p->...p", w, F.bf16_ulp(ro))

    bad = wrong(rank_out, rank_lse, lse)
    assert (bad > F.bf16_ulp(rank_out).max(axis=0) * (1 + 1e-12)).any()
