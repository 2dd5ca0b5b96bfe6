"""Parity on inputs that stress the cross-CTA factor exchange of the partial kernel.

The kernel splits each q.k dot product between two CTAs (dims [0, 256) and
[256, 576)), exchanges per-token factors relative to each CTA's own maximum over a
group of 32 tokens, and bounds the group's largest score by the sum of the two
maxima. When the two partial scores of a row disagree (one token large on the first
span only, another on the second only), that bound lies far above the true maximum.
These inputs make the gap 15 to 21 binades in most groups; the outputs must still
match the oracle within the usual tolerance.
"""

import math

import numpy as np
import pytest
import torch

import workloads
from tests import _helpers as h

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import decode_context_mla_causal_gb300 as mod

    return mod


def bound_gaps(w):
    """Per (sequence, rank, group of 32 rank-local tokens, head) of verify row 0: the
    sum of the two spans' maximum partial scores minus the largest full score (log2
    units). Interleave 1: rank r holds the tokens p with p mod dcp == r, in order."""
    assert w.interleave == 1
    kv = w.kv.cpu().view(torch.float8_e4m3fn).float().numpy().astype(np.float64) * w.kv_scale
    q = w.q.float().cpu().numpy().astype(np.float64)
    sc = w.softmax_scale / math.log(2.0)
    table = w.block_table.cpu().numpy()
    out = []
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        for r in range(w.dcp):
            li = np.arange(len(range(r, L, w.dcp)))
            slots = table[b][li // w.block_size] * w.block_size + li % w.block_size
            k = kv[r].reshape(-1, 576)[slots]
            qq = q[b * w.qlen]
            a = sc * (qq[:, :256] @ k[:, :256].T)
            c = sc * (qq[:, 256:] @ k[:, 256:].T)
            for g0 in range(0, len(li) - 31, 32):
                sa, sb = a[:, g0:g0 + 32], c[:, g0:g0 + 32]
                out.append(sa.max(1) + sb.max(1) - (sa + sb).max(1))
    return np.concatenate(out)


def anticorrelated(seed):
    base = workloads.generate("c2", device="cpu", seed_index=80, overrides=dict(
        batch=2, num_heads=16, qlen=3, dcp=2, interleave=1, max_local_len=512,
        lengths=("fixed", 900)))
    return workloads.make_anticorrelated(base, seed=seed).to("cuda")


@pytest.mark.parametrize("seed", [5, 6])
@pytest.mark.parametrize("num_splits", [1, 3])
def test_parity_anticorrelated_partial_scores(dm, seed, num_splits):
    w = anticorrelated(seed)
    gaps = bound_gaps(w)
    assert gaps.max() >= 18.0 and (gaps >= 15.0).mean() > 0.3, (gaps.max(), (gaps >= 15).mean())
    step = h.run_gpu(dm, w, num_splits=num_splits)
    assert step.read_status() == 0
    ref = h.oracle_forward(w, per_rank=True)
    R, H = w.rows, w.num_heads
    h.assert_parity(step.out.float().cpu().numpy(), step.lse.cpu().numpy(),
                    ref["out"].reshape(R, H, -1), ref["lse"].reshape(R, H), ("anti", seed))
    rl = step.rank_lse.cpu().numpy()
    exp = ref["rank_lse"].reshape(w.dcp, R, H)
    assert np.array_equal(np.isneginf(rl), np.isneginf(exp))
    fin = np.isfinite(exp)
    assert np.abs(rl[fin] - exp[fin]).max(initial=0) <= 1e-3
