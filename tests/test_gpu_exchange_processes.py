"""The exchange with one dcp rank per process, on the GPU: two processes (both on
cuda:0) each run the library's metadata, partial and merge kernels for their own rank
only, pack their send buffer, exchange it through a gloo all-to-all of host copies and
combine their head slice with the library's combine kernel.

Each process's result must equal, bit for bit, the one-device step that holds every
rank (its combine reads all ranks' send buffers in place), and match the oracle's
unsharded attention for its heads within the BF16 wire bound. The two processes' kernels
never wait on each other: the collective runs on the host, between launches.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, num_splits):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import decode_context_mla_causal_gb300 as dm
        import oracle
        import workloads
        from oracle import exchange as X
        from tests import _helpers as h

        torch.cuda.set_device(0)
        w = workloads.generate("c2", device="cuda")
        assert w.dcp == world
        G, Hg = w.dcp, w.num_heads // w.dcp
        hs = slice(rank * Hg, (rank + 1) * Hg)

        # this process's rank: its own pool, its own partials, its own send buffer
        step = h.run_gpu(dm, w, num_splits=num_splits, rank_begin=rank, num_ranks=1)
        ex = dm.A2AExchange(step)
        ex.pack()
        torch.cuda.synchronize()
        recv = dm.a2a_exchange(ex.send.cpu()).cuda()  # gloo: host tensors
        out, lse = ex.combine(recv, rank)
        torch.cuda.synchronize()
        assert step.read_status() == 0

        # the one-device form with every rank of the group
        full = h.run_gpu(dm, w, num_splits=num_splits)
        exf = dm.A2AExchange(full)
        exf.pack()
        exf.combine_local()
        torch.cuda.synchronize()
        assert torch.equal(out[:, hs].view(torch.int16), exf.out[:, hs].view(torch.int16)), rank
        assert torch.equal(lse[:, hs], exf.lse[:, hs]), rank

        # the oracle, for this process's heads
        ref = h.oracle_forward(w, per_rank=True)
        R, H = w.rows, w.num_heads
        rank_out = ref["rank_out"].reshape(G, R, H, -1)[:, :, hs]
        rank_lse = ref["rank_lse"].reshape(G, R, H)[:, :, hs]
        out_ref = ref["out"].reshape(R, H, -1)[:, hs]
        lse_ref = ref["lse"].reshape(R, H)[:, hs]
        o = out[:, hs].float().cpu().numpy()
        allow = (1e-2 + 0.5 * oracle.fp8.bf16_ulp(out_ref)
                 + X.wire_bound(rank_out, rank_lse, lse_ref))
        assert (np.abs(o - out_ref) <= allow).all(), (rank, float(np.abs(o - out_ref).max()))
        l = lse[:, hs].cpu().numpy()
        assert np.array_equal(np.isneginf(l), np.isneginf(lse_ref))
        fin = np.isfinite(lse_ref)
        assert np.abs(l[fin] - lse_ref[fin]).max(initial=0) <= 1e-3
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("num_splits", [1, 3])
def test_two_processes_pack_exchange_combine(num_splits):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    mp.spawn(_rank_main, args=(2, _free_port(), num_splits), nprocs=2, join=True)
