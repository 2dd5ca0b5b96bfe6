"""GPU parity of the new-token KV write (slot mapping + write) against the oracle.

Bit-exact: the slot mapping (int) and every byte of the pools after the write
(FP8 codes decided by x / scale in IEEE float32 on both sides). End to end: the
verify attention over pools written by the GPU equals the oracle's attention
over pools written by the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import kv_write as okw
from tests import _helpers as h


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import decode_context_mla_causal_gb300 as mod

    return mod


def _new_rows(w, seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn((w.rows, 576), generator=g, dtype=torch.float32) * 2.0
    return x.to(torch.bfloat16)


def _gpu_mapping(dm, w, dims, rank_begin=0, num_ranks=None):
    nr = w.dcp - rank_begin if num_ranks is None else num_ranks
    sm = torch.full((nr, w.rows), 12345, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dm.dcp_kv_slot_mapping(dims, w.seq_lens, w.block_table, rank_begin, nr, sm, st)
    torch.cuda.synchronize()
    return sm.cpu().numpy(), int(st.item())


def _oracle_mapping(w, rank_begin=0, num_ranks=None):
    return okw.slot_mapping(seq_lens=w.seq_lens.cpu().numpy(), block_table=w.block_table.cpu().numpy(),
                            qlen=w.qlen, dcp=w.dcp, interleave=w.interleave,
                            block_size=w.block_size, max_blocks_per_seq=w.max_blocks_per_seq,
                            num_blocks=w.num_blocks, rank_begin=rank_begin, num_ranks=num_ranks)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4"])
def test_slot_mapping_bit_exact(dm, name):
    w = workloads.generate(name, device="cuda")
    dims = h.dims_of(dm, w, 1)
    got, st = _gpu_mapping(dm, w, dims)
    exp, est = _oracle_mapping(w)
    assert st == est == 0
    assert np.array_equal(got, exp)
    # one rank per call gives the same rows
    for r in range(w.dcp):
        g1, _ = _gpu_mapping(dm, w, dims, rank_begin=r, num_ranks=1)
        assert np.array_equal(g1[0], exp[r])


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["c1", "c2", "c4"])
def test_write_bit_exact(dm, name):
    w = workloads.generate(name, device="cuda")
    dims = h.dims_of(dm, w, 1)
    new = _new_rows(w, 5)
    sm, _ = _gpu_mapping(dm, w, dims)
    kvt = h.kv_dtype_of(dm, w)
    pool = w.kv.clone()
    scale = torch.tensor([w.kv_scale], dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dm.dcp_kv_write(dims, torch.as_tensor(sm, device="cuda"), new.cuda(), kvt, scale, w.dcp,
                    pool, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bits = new.view(torch.int16).numpy().view(np.uint16)
    exp = okw.write(w.pools_np(), sm, bits, w.kv_dtype, w.kv_scale)
    got = pool.cpu()
    got = got.numpy().view(np.uint8) if w.kv_dtype == "fp8" else got.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, exp)


@pytest.mark.gpu
def test_write_then_attend_end_to_end(dm):
    # the verify tokens are written by the GPU, then the verify step reads them
    w = workloads.generate("c2", device="cuda")
    dims = h.dims_of(dm, w, 3)
    new = _new_rows(w, 9)
    sm, _ = _gpu_mapping(dm, w, dims)
    scale = torch.tensor([w.kv_scale], dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dm.dcp_kv_write(dims, torch.as_tensor(sm, device="cuda"), new.cuda(), h.kv_dtype_of(dm, w),
                    scale, w.dcp, w.kv, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    step = h.run_gpu(dm, w, num_splits=3)
    assert step.read_status() == 0
    bits = new.view(torch.int16).numpy().view(np.uint16)
    pools = okw.write(w.pools_np(), sm, bits, "fp8", w.kv_scale)  # equal to the GPU's pools
    ref = oracle.attention.forward(q_bits=w.q_bits_np(), pools=pools,
                                   block_table=w.block_table.cpu().numpy(),
                                   seq_lens=w.seq_lens.cpu().numpy(), qlen=w.qlen, dcp=w.dcp,
                                   interleave=w.interleave, block_size=w.block_size,
                                   kv_dtype="fp8", kv_scale=w.kv_scale,
                                   softmax_scale=w.softmax_scale, per_rank=False)
    R, H = w.rows, w.num_heads
    h.assert_parity(step.out.float().cpu().numpy(), step.lse.cpu().numpy(),
                    ref["out"].reshape(R, H, -1), ref["lse"].reshape(R, H), "c2 after write")


@pytest.mark.gpu
def test_bad_inputs_set_status(dm):
    w = workloads.generate("c1", device="cuda", overrides=dict(batch=3),
                           seq_lens=[2, 200, 60])
    bt = w.block_table.clone()
    bt[2, 1] = w.num_blocks + 7           # the block holding sequence 2's new tokens
    w.block_table = bt
    dims = h.dims_of(dm, w, 1)
    got, st = _gpu_mapping(dm, w, dims)
    exp, est = _oracle_mapping(w)
    assert np.array_equal(got, exp)
    assert st == est
    assert st & dm.STATUS_BAD_SEQ_LEN and st & dm.STATUS_BAD_BLOCK_ID
    # an out-of-range entry in a hand-made mapping is skipped and reported
    sm = torch.as_tensor(got, device="cuda").clone()
    sm[0, 3] = 1 << 30
    pool = w.kv.clone()
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    dm.dcp_kv_write(dims, sm, _new_rows(w, 1).cuda(), h.kv_dtype_of(dm, w), None, w.dcp, pool, st2)
    torch.cuda.synchronize()
    assert int(st2.item()) & dm.STATUS_BAD_PAGE
