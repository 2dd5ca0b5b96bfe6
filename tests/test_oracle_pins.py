"""Pins for the CPU oracle: each check ties it to something other than itself.

Pins used: printed examples from the pages (golden fixtures), a second printed
formula (the DSpark slot map), brute force on tiny inputs, library routines for
special cases (torch's E4M3/BF16 casts, torch SDPA and logsumexp in float64),
closed forms and invariants. The last group plants plausible mistakes in the
oracle (on the CPU) and checks that some pin catches each of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as A
from oracle import fp8 as F
from oracle import metadata as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# element decoders


def test_e4m3_table_matches_torch_cast():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    ours = F.decode_e4m3(codes.numpy())
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])
    assert np.nanmax(ours) == 448.0 and np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    x = torch.from_numpy(rng.standard_normal(4096).astype(np.float32) * 10).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(F.decode_bf16(bits), x.to(torch.float64).numpy())


def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(10000) * 3
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(F.round_to_bf16(x.astype(np.float32).astype(np.float64)), ref)


# --------------------------------------------------------------------------
# interleave, local lengths, slots


def test_golden_dcp2_round_robin():
    g = _golden("dcp2_round_robin.json")
    W, S = g["dcp"], g["interleave"]
    p = np.arange(g["num_tokens"])
    for r, toks in g["rank_tokens"].items():
        assert list(p[M.owner(p, W, S) == int(r)]) == toks
        # local indices of a rank's tokens are 0, 1, 2, ... in order
        assert list(M.local_index(np.array(toks), W, S)) == list(range(len(toks)))


@pytest.mark.parametrize("W", [1, 2, 3, 8])
@pytest.mark.parametrize("S", [1, 2, 16, 64])
def test_closed_form_equals_count(W, S):
    for g in range(0, 4 * W * S + 3):
        tot = 0
        for r in range(W):
            n = M.count_local(g, r, W, S)
            assert M.local_len_closed_form(g, r, W, S) == n, (g, r)
            tot += n
        assert tot == g  # every position covered exactly once


@pytest.mark.parametrize("W", [2, 5, 8])
def test_interleave_one_reduces_to_dspark_ceil(W):
    # DSpark section: a sequence of L global tokens has ceil((L - rank)/dcp) local rows
    for L in range(0, 200):
        for r in range(W):
            assert M.count_local(L, r, W, 1) == max(0, -(-(L - r) // W))


@pytest.mark.parametrize("W,S", [(2, 1), (3, 2), (8, 64), (4, 16)])
def test_local_index_is_a_bijection_per_rank(W, S):
    p = np.arange(W * S * 7 + 5)
    own = M.owner(p, W, S)
    li = M.local_index(p, W, S)
    for r in range(W):
        mine = li[own == r]
        assert list(mine) == list(range(len(mine)))


@pytest.mark.parametrize("W,bs", [(2, 16), (8, 64), (3, 4)])
def test_slot_map_matches_dspark_formula(W, bs):
    # DSpark section: owner p % dcp, slot block_table[p // (bs*dcp)]*bs + (p % (bs*dcp)) // dcp
    rng = np.random.default_rng(W * 100 + bs)
    table = rng.permutation(64)
    for p in range(W * bs * 5):
        li = int(M.local_index(p, W, 1))
        ours = table[li // bs] * bs + li % bs
        theirs = table[p // (bs * W)] * bs + (p % (bs * W)) // W
        assert int(M.owner(p, W, 1)) == p % W
        assert ours == theirs


def test_row_boundary_monotone_and_last_row_sees_everything():
    for L in range(3, 50):
        gs = [M.row_boundary(L, 3, j) for j in range(3)]
        assert gs == sorted(gs) and gs[-1] == L and gs[0] == L - 2
        for r in range(4):
            ns = [M.count_local(g, r, 4, 1) for g in gs]
            assert ns == sorted(ns)


def test_subpage_golden():
    for bs, want in _golden("subpage_review.json")["cases"]:
        assert M.subpage_size(bs) == want


@pytest.mark.parametrize("bs,S,W", [(16, 1, 2), (64, 64, 8), (96, 1, 3), (256, 2, 2), (64, 16, 4)])
def test_pages_cover_the_same_rows_as_slots(bs, S, W):
    rng = np.random.default_rng(bs + S)
    B, qlen = 3, 4
    bound = 300
    MB = -(-bound // bs)
    NB = B * MB + 5
    table = rng.permutation(NB)[: B * MB].reshape(B, MB)
    seq_lens = rng.integers(qlen, W * bound // 2, size=B)
    md = M.build_metadata(batch=B, qlen=qlen, dcp=W, interleave=S, block_size=bs,
                          max_local_len=bound, num_blocks=NB, num_splits=3,
                          seq_lens=seq_lens, block_table=table)
    assert md["status"] == 0
    P = md["subpage"]
    for r in range(W):
        for b in range(B):
            n = md["row_len"][r, b * qlen + qlen - 1]
            pages = md["page_ids"][r, b]
            npg = -(-n // P)
            assert (pages[:npg] >= 0).all() and (pages[npg:] == -1).all()
            for li in range(n):
                flat = pages[li // P] * P + li % P
                assert flat == table[b, li // bs] * bs + li % bs
            beg, end = md["split_beg"][r, b], md["split_end"][r, b]
            assert beg[0] == 0 and end[-1] == npg
            assert (beg[1:] == end[:-1]).all()
            sizes = end - beg
            assert sizes.max() - sizes.min() <= 1


def test_metadata_status_bits():
    table = np.arange(8).reshape(2, 4)
    md = M.build_metadata(batch=2, qlen=3, dcp=2, interleave=1, block_size=16,
                          max_local_len=64, num_blocks=8, num_splits=1,
                          seq_lens=[2, 20], block_table=table)
    assert md["status"] & M.STATUS_BAD_SEQ_LEN
    md = M.build_metadata(batch=1, qlen=1, dcp=2, interleave=1, block_size=16,
                          max_local_len=16, num_blocks=8, num_splits=1,
                          seq_lens=[100], block_table=table[:1])
    assert md["status"] & M.STATUS_LOCAL_OVER_BOUND and md["row_len"].max() == 16
    bad = table[:1].copy()
    bad[0, 1] = 99
    md = M.build_metadata(batch=1, qlen=1, dcp=2, interleave=1, block_size=16,
                          max_local_len=64, num_blocks=8, num_splits=1,
                          seq_lens=[100], block_table=bad)
    assert md["status"] & M.STATUS_BAD_BLOCK_ID and md["page_ids"][0, 0, 1] == -1


# --------------------------------------------------------------------------
# attention


def _brute(q, K, g, scale):
    """Triple loop with exactly rounded sums (math.fsum)."""
    n = q.shape[0]
    out = np.zeros((n, A.D_V))
    lse = np.full(n, -math.inf)
    for i in range(n):
        if g[i] <= 0:
            continue
        s = [scale * math.fsum(q[i, d] * K[t, d] for d in range(q.shape[1])) for t in range(g[i])]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        tot = math.fsum(e)
        lse[i] = m + math.log(tot)
        for d in range(A.D_V):
            out[i, d] = math.fsum(e[t] * K[t, d] for t in range(g[i])) / tot
    return out, lse


def _tiny_workload(seed, L=37, W=2, S=1, bs=4, qlen=3, H=2, dtype="fp8"):
    rng = np.random.default_rng(seed)
    bound = -(-L // W) + S
    MB = -(-bound // bs) + 1
    NB = MB + 3
    table = rng.permutation(NB)[:MB].reshape(1, MB)
    if dtype == "fp8":
        pools = rng.integers(0, 256, size=(W, NB, bs, A.D_QK), dtype=np.uint8)
        pools[(pools & 0x7F) == 0x7F] = 0x3C  # avoid NaN codes in random bytes
        scale = 0.01
    else:
        x = torch.from_numpy(rng.standard_normal((W, NB, bs, A.D_QK)).astype(np.float32))
        pools = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        scale = 1.0
    qx = torch.from_numpy(rng.standard_normal((qlen, H, A.D_QK)).astype(np.float32))
    q_bits = qx.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return dict(q_bits=q_bits, pools=pools, block_table=table, seq_lens=np.array([L]),
                qlen=qlen, dcp=W, interleave=S, block_size=bs, kv_dtype=dtype,
                kv_scale=scale, softmax_scale=1 / math.sqrt(192))


@pytest.mark.parametrize("seed,W,S,dtype", [(0, 2, 1, "fp8"), (1, 3, 2, "bf16"), (2, 1, 1, "fp8")])
def test_forward_matches_brute_force(seed, W, S, dtype):
    wl = _tiny_workload(seed, W=W, S=S, dtype=dtype)
    res = A.forward(**wl)
    L, qlen = 37, 3
    K = A.decode_pool_rows(
        A.gather_rows(wl["pools"], wl["block_table"][0], np.arange(L), dcp=W,
                      interleave=S, block_size=4), dtype, wl["kv_scale"])
    for j in range(qlen):
        q = F.decode_bf16(wl["q_bits"][j])
        g = [L - qlen + 1 + j] * q.shape[0]
        o, l = _brute(q, K, g, wl["softmax_scale"])
        assert np.abs(o - res["out"][j]).max() < 1e-12
        assert np.abs(l - res["lse"][j]).max() < 1e-12


def test_gather_is_inverse_of_scatter():
    # scatter a random global sequence by brute-force enumeration of each rank's
    # tokens in order, then gather it back with the oracle
    rng = np.random.default_rng(5)
    for W, S, bs in [(2, 1, 16), (8, 64, 64), (3, 2, 4)]:
        L = 3 * W * S * 2 + 7
        n_loc = -(-L // (W * S)) * S
        MB = -(-n_loc // bs)
        NB = MB + 2
        table = rng.permutation(NB)[:MB]
        pools = np.zeros((W, NB, bs, 2), dtype=np.int64)
        seq = rng.integers(1, 1 << 40, size=(L, 2))
        counters = [0] * W
        for p in range(L):
            r = (p // S) % W
            k = counters[r]
            counters[r] += 1
            pools[r, table[k // bs], k % bs] = seq[p]
        got = A.gather_rows(pools, table, np.arange(L), dcp=W, interleave=S, block_size=bs)
        assert np.array_equal(got, seq)


def test_attend_matches_torch_sdpa_fp64():
    rng = np.random.default_rng(7)
    n, T = 6, 50
    q = rng.standard_normal((n, A.D_QK))
    K = rng.standard_normal((T, A.D_QK))
    g = np.array([1, 5, 17, 33, 49, 50])
    scale = 1 / math.sqrt(192)
    o, l = A.attend(q, K, g, scale)
    mask = torch.from_numpy(np.arange(T)[None, :] < g[:, None])
    qt, kt = torch.from_numpy(q), torch.from_numpy(K)
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt[None], kt[None], kt[None, :, : A.D_V], attn_mask=mask[None], scale=scale)[0]
    assert np.abs(ref.numpy() - o).max() < 1e-12
    s = scale * (qt @ kt.T)
    ref_l = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=1)
    assert np.abs(ref_l.numpy() - l).max() < 1e-12


def test_closed_forms():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((3, A.D_QK))
    K = rng.standard_normal((9, A.D_QK))
    scale = 0.3
    o, l = A.attend(q, K, [1, 1, 1], scale)
    assert np.allclose(o, K[0, : A.D_V][None], atol=0, rtol=0)
    assert np.allclose(l, scale * q @ K[0], atol=1e-13)
    Ks = np.repeat(K[:1], 9, axis=0)
    o, l = A.attend(q, Ks, [9, 4, 2], scale)
    assert np.abs(o - Ks[0, : A.D_V][None]).max() < 1e-13
    assert np.abs(l - (scale * q @ K[0] + np.log([9, 4, 2]))).max() < 1e-12
    o, l = A.attend(q, K, [0, 0, 0], scale)
    assert (o == 0).all() and np.isneginf(l).all()


def test_chunked_equals_one_shot():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((4, A.D_QK))
    K = rng.standard_normal((1000, A.D_QK))
    g = np.array([1, 333, 999, 1000])
    o1, l1 = A.attend(q, K, g, 0.1)

    def chunks():
        for st in range(0, 1000, 128):
            yield st, K[st: st + 128]

    o2, l2 = A.attend_chunked(q, chunks, g, 0.1)
    assert np.abs(o1 - o2).max() < 1e-13 and np.abs(l1 - l2).max() < 1e-12


@pytest.mark.parametrize("W,S", [(2, 1), (4, 2), (8, 64), (1, 1)])
def test_merge_of_shards_equals_unsharded(W, S):
    wl = _tiny_workload(11 + W, L=150, W=W, S=S, bs=8 if S < 8 else 64, qlen=4, H=3)
    res = A.forward(**wl)
    o, l = A.merge_shards(res["rank_out"], res["rank_lse"])
    assert np.abs(o - res["out"]).max() < 1e-12
    assert np.abs(l - res["lse"]).max() < 1e-12
    if W == 1:
        assert np.abs(res["rank_lse"][0] - res["lse"]).max() == 0


def test_interleave_beyond_length_puts_everything_on_rank0():
    wl = _tiny_workload(21, L=30, W=4, S=64, bs=64, qlen=2, H=2)
    res = A.forward(**wl)
    assert np.isneginf(res["rank_lse"][1:]).all()
    assert np.abs(res["rank_lse"][0] - res["lse"]).max() == 0
    assert (res["rank_out"][1:] == 0).all()


def _tolerance_failures(a_out, b_out, a_lse, b_lse):
    allow = 1e-2 + 0.5 * F.bf16_ulp(b_out)
    bad_o = int((np.abs(F.round_to_bf16(a_out) - b_out) > allow).sum())
    bad_l = int((np.abs(a_lse - b_lse) > 1e-3).sum())
    return bad_o, bad_l


@pytest.mark.parametrize("wrong", ["committed_prefix", "whole_sequence"])
def test_negative_control_boundaries_fail(wrong):
    # Like the PR's negative control: only the row boundary changes; parity must fail.
    rng = np.random.default_rng(3)
    W, qlen, H, bs, L = 2, 3, 96, 64, 1500
    MB = -(-(-(-L // W)) // bs)
    NB = MB + 2
    table = rng.permutation(NB)[:MB].reshape(1, MB)
    x = rng.standard_normal((W, NB, bs, A.D_QK)).astype(np.float32)
    scale = float(np.abs(x).max()) / 448
    pools = torch.from_numpy(x / scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    qx = torch.from_numpy(rng.standard_normal((qlen, H, A.D_QK)).astype(np.float32))
    q_bits = qx.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    args = dict(q_bits=q_bits, pools=pools, block_table=table, seq_lens=np.array([L]),
                qlen=qlen, dcp=W, interleave=1, block_size=bs, kv_dtype="fp8",
                kv_scale=scale, softmax_scale=1 / math.sqrt(192), per_rank=False)
    good = A.forward(**args)
    if wrong == "committed_prefix":
        bad = A.forward(boundary=M.committed_prefix_boundary, **args)
    else:
        bad = A.forward(causal=False, **args)
    bad_o, bad_l = _tolerance_failures(bad["out"], good["out"], bad["lse"], good["lse"])
    assert bad_o > 0 or bad_l > 0
    # the one row whose boundary the mutation leaves alone is unchanged: j = 0 for
    # the committed prefix, j = qlen - 1 for the whole sequence
    same = 0 if wrong == "committed_prefix" else -1
    assert np.abs(bad["out"][same] - good["out"][same]).max() < 1e-12


# --------------------------------------------------------------------------
# the pins have teeth: plant plausible mistakes in the oracle and see them caught


def test_planted_dropped_rope_dims_is_caught(monkeypatch):
    wl = _tiny_workload(30, W=2, dtype="fp8")
    good = A.forward(**wl)
    orig = A.attend_chunked

    def no_rope(q, key_chunks, limits, scale, mask_chunks=None):
        q = q.copy()
        q[:, A.D_V:] = 0.0
        return orig(q, key_chunks, limits, scale, mask_chunks)

    monkeypatch.setattr(A, "attend_chunked", no_rope)
    bad = A.forward(**wl)
    assert np.abs(bad["lse"] - good["lse"]).max() > 1e-6


def test_planted_wrong_owner_is_caught(monkeypatch):
    # ignoring the interleave size in the owner breaks the per-rank bijection
    monkeypatch.setattr(M, "owner", lambda p, W, S: np.asarray(p) % W)
    p = np.arange(64)
    own = M.owner(p, 4, 2)
    li = M.local_index(p, 4, 2)
    broken = any(list(li[own == r]) != list(range((own == r).sum())) for r in range(4))
    assert broken


def test_planted_off_by_one_boundary_is_caught():
    # a boundary one short on every row changes the covered-once invariant
    g = 40
    short = sum(M.local_len_closed_form(g - 1, r, 4, 1) for r in range(4))
    assert short != g
