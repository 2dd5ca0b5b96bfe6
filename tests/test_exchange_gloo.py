"""The multi-process form of the exchange on CPU: two gloo ranks run the library's
``a2a_exchange`` on send buffers packed by the oracle; each must receive exactly
the chunks the all-to-all permutation assigns it, and the oracle's combine of
what it received must equal the unsharded attention for its heads."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from decode_context_mla_causal_gb300.exchange import a2a_exchange
        from oracle import attention as A
        from oracle import exchange as X
        from tests.test_oracle_pins import _tiny_workload

        wl = _tiny_workload(61, L=150, W=world, S=1, bs=8, qlen=3, H=4)
        res = A.forward(**wl)
        R, H = res["out"].shape[:2]
        Hg = H // world
        send_all = X.pack(res["rank_out"], res["rank_lse"])            # [W][W][cw] uint16
        mine = torch.from_numpy(send_all[rank].reshape(-1).view(np.int16).copy())
        recv = a2a_exchange(mine.view(torch.bfloat16))
        got = recv.view(torch.int16).numpy().view(np.uint16).reshape(world, -1)
        want = X.exchange(send_all)[rank]
        assert np.array_equal(got, want), rank
        o, l = X.unpack(got, R, Hg, 512)
        out, lse = A.merge_shards(o, l)
        hs = slice(rank * Hg, (rank + 1) * Hg)
        bound = X.wire_bound(res["rank_out"][:, :, hs], res["rank_lse"][:, :, hs],
                             res["lse"][:, hs]) + 1e-9
        assert (np.abs(out - res["out"][:, hs]) <= bound).all()
        fin = np.isfinite(res["lse"][:, hs])
        assert np.abs(lse[fin] - res["lse"][:, hs][fin]).max() <= 1e-5
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_exchange_and_combine():
    import __graft_entry__

    __graft_entry__.build()  # the package loads the library at import
    mp.spawn(_rank_main, args=(2, _free_port()), nprocs=2, join=True)
