"""Pins of the new-token KV write oracle (slot mapping, E4M3 encoding, write).

Each pin checks the oracle against something other than itself: the OCP
definition through its decode table, a library conversion
(torch.float8_e4m3fn), the DSpark slot formula written out here, the gather of
``oracle.attention`` (a different function), and counting.
"""

import numpy as np
import pytest
import torch

from oracle import attention, fp8
from oracle import kv_write as kw

pytestmark = pytest.mark.filterwarnings("ignore")


def test_encode_roundtrips_every_finite_code():
    codes = np.arange(256, dtype=np.uint8)
    vals = fp8.decode_e4m3(codes)
    fin = ~np.isnan(vals)
    assert np.array_equal(kw.encode_e4m3(vals[fin]), codes[fin])
    assert kw.encode_e4m3(np.array([np.nan]))[0] == 0x7F


def test_encode_ties_go_to_even_like_the_library():
    mags = fp8.E4M3_TABLE[:0x7F]
    mids = (mags[:-1] + mags[1:]) / 2.0          # every midpoint of adjacent codes
    x = np.concatenate([mids, -mids])
    lib = torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = kw.encode_e4m3(x.astype(np.float32).astype(np.float64))
    assert np.array_equal(got, lib)
    assert all(int(c) & 1 == 0 for c in got[: len(mids)])   # the even code wins each tie


def test_encode_saturates_and_keeps_signed_zero():
    got = kw.encode_e4m3(np.array([448.0, 449.0, 464.0, 1e30, -1e30, 0.0, -0.0]))
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x00, 0x80]


def test_encode_matches_library_on_random_values():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(20000) * 40, rng.standard_normal(5000) * 0.01])
    x32 = np.clip(x, -448, 448).astype(np.float32)
    lib = torch.tensor(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(kw.encode_e4m3(x32.astype(np.float64)), lib)


def test_quantize_divides_in_float32():
    bits = np.array([[0x3F80, 0x4000, 0xC2C8]], dtype=np.uint16)   # 1, 2, -100 in bf16
    scale = 0.3
    q = np.float32(np.array([1.0, 2.0, -100.0], dtype=np.float32) / np.float32(scale))
    expect = torch.tensor(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(kw.quantize_rows(bits, scale)[0], expect)


def _table(rng, B, MB, NB):
    perm = rng.permutation(NB)
    return perm[: B * MB].reshape(B, MB).astype(np.int64)


def test_slot_mapping_matches_dspark_slot_formula_for_s1():
    # DSpark: owner of p is p % dcp; its slot is block_table[(p // dcp) // bs]*bs + (p // dcp) % bs
    rng = np.random.default_rng(3)
    W, bs, B, qlen, MB = 4, 8, 3, 5, 6
    NB = B * MB + 2
    table = _table(rng, B, MB, NB)
    lens = np.array([5, 37, 180])
    sm, st = kw.slot_mapping(seq_lens=lens, block_table=table, qlen=qlen, dcp=W, interleave=1,
                             block_size=bs, max_blocks_per_seq=MB, num_blocks=NB)
    assert st == 0
    for b, L in enumerate(lens):
        for j in range(qlen):
            p = L - qlen + j
            r, li = p % W, p // W
            for k in range(W):
                want = table[b, li // bs] * bs + li % bs if k == r else -1
                assert sm[k, b * qlen + j] == want


@pytest.mark.parametrize("W,S,bs", [(2, 1, 16), (3, 2, 4), (8, 64, 64), (4, 4, 8)])
def test_written_tokens_are_gathered_back(W, S, bs):
    # all positions of each sequence written as "new" tokens, then gathered by
    # oracle.attention's independent addressing: identity
    rng = np.random.default_rng(W * 100 + S)
    B = 3
    lens = np.array([1, 2 * W * S + 3, 5 * W * S + 1])
    MB = int(max(-(-(L // (W * S) * S + S) // bs) for L in lens)) + 1
    NB = B * MB + 3
    table = _table(rng, B, MB, NB)
    pools = np.zeros((W, NB, bs, 576), dtype=np.uint16)
    for b, L in enumerate(lens):
        ids = (np.arange(L, dtype=np.uint16)[:, None] + 1000 * (b + 1) + np.zeros((1, 576), dtype=np.uint16))
        sm, st = kw.slot_mapping(seq_lens=[L], block_table=table[b:b + 1], qlen=L, dcp=W,
                                 interleave=S, block_size=bs, max_blocks_per_seq=MB, num_blocks=NB)
        assert st == 0
        assert np.array_equal((sm >= 0).sum(axis=0), np.ones(L))   # exactly one owner each
        pools = kw.write(pools, sm, ids, "bf16", 1.0)
        got = attention.gather_rows(pools, table[b], np.arange(L), dcp=W, interleave=S,
                                    block_size=bs)
        assert np.array_equal(got, ids)


def test_write_touches_only_mapped_rows_and_quantises():
    rng = np.random.default_rng(11)
    W, bs, NB = 2, 4, 6
    pools = rng.integers(0, 256, size=(W, NB, bs, 576), dtype=np.uint8)
    sm = np.array([[5, -1, 0], [-1, 22, -1]], dtype=np.int32)
    x = torch.randn(3, 576).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    out = kw.write(pools, sm, bits, "fp8", 0.05)
    flat_in, flat_out = pools.reshape(W, -1, 576), out.reshape(W, -1, 576)
    q = kw.quantize_rows(bits, 0.05)
    assert np.array_equal(flat_out[0, 5], q[0]) and np.array_equal(flat_out[0, 0], q[2])
    assert np.array_equal(flat_out[1, 22], q[1])
    mask = np.ones((W, NB * bs), dtype=bool)
    mask[0, [5, 0]] = False
    mask[1, 22] = False
    assert np.array_equal(flat_out[mask], flat_in[mask])


def test_slot_mapping_status_bits():
    table = np.array([[0, 1, 99]])
    _, st = kw.slot_mapping(seq_lens=[2], block_table=table, qlen=3, dcp=1, interleave=1,
                            block_size=4, max_blocks_per_seq=3, num_blocks=4)
    assert st == kw.STATUS_BAD_SEQ_LEN
    sm, st = kw.slot_mapping(seq_lens=[10], block_table=table, qlen=2, dcp=1, interleave=1,
                             block_size=4, max_blocks_per_seq=3, num_blocks=4)
    assert st == kw.STATUS_BAD_BLOCK_ID and list(sm[0]) == [-1, -1]
    sm, st = kw.slot_mapping(seq_lens=[14], block_table=table, qlen=3, dcp=1, interleave=1,
                             block_size=4, max_blocks_per_seq=3, num_blocks=4)
    assert st == kw.STATUS_LOCAL_OVER_BOUND | kw.STATUS_BAD_BLOCK_ID
    assert list(sm[0]) == [-1, -1, -1]
