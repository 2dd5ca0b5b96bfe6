"""Seeded synthetic inputs for DCP causal MLA verification.

This module is the ONLY code shared by the CUDA library's callers (tests,
bench) and the CPU oracle. It draws random inputs and holds none of the
method's arithmetic: no token->rank mapping, no local lengths, no attention.
Pools are filled completely (every slot of every block on every rank) so no
knowledge of which slots hold which tokens is needed to build them.

Workload recipe (the five shapes the method is exercised on):

* ``c1`` tiny: batch 1, 8 heads, qlen 3, 200 tokens, dcp 2, interleave 1,
  block 16, BF16 cache.
* ``c2``: batch 4, 96 heads, qlen 3, lengths uniform in [1024, 4096], dcp 2,
  interleave 1, block 64, FP8 cache.
* ``c3`` single-token decode: batch 32, 128 heads, qlen 1, 32768 tokens each,
  dcp 8, interleave 1, block 64, FP8 cache.
* ``c4`` speculative verify: batch 32, 128 heads, qlen 5, 28 lengths
  log-uniform in [8192, 131072] plus the four short lengths 5, 70, 300, 511
  (shorter than dcp*interleave = 512, so some rank-local lengths are 0),
  dcp 8, interleave 64, block 64, FP8 cache.
* ``c5`` long context: batch 4, 128 heads, qlen 3, 1,048,576 tokens each,
  dcp 8, interleave 1, block 64, FP8 cache.

All use softmax scale 1/sqrt(192). q and the cache values are N(0, 1) float32,
rounded to BF16 (ties to even); for FP8 the per-tensor scale is
``max|x| / 448`` over every generated cache value of the workload and the codes
are ``E4M3(clamp(x / scale, -448, 448))`` (ties to even). Seeds: a NumPy
``SeedSequence(1000 + k)`` for workload k spawns children for lengths (0), the
block-table permutation (1), q (2) and each rank's pool (3 + r); pool values are
drawn in chunks of blocks, each chunk from its own derived seed, so the FP8 scale
pass and the quantisation pass draw identical numbers.

Every sequence is given ``MB = ceil(max_local_len / block_size)`` distinct
blocks (the static bound of the workload, a config constant), taken from a
random permutation of the ``NB = batch * MB + 8`` blocks of each rank's pool
("random/shuffled physical pages"); the eight spare blocks are never listed.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

D_QK = 576
D_V = 512

CONFIGS = {
    "c1": dict(batch=1, num_heads=8, qlen=3, dcp=2, interleave=1, block_size=16,
               kv_dtype="bf16", max_local_len=100, lengths=("fixed", 200)),
    "c2": dict(batch=4, num_heads=96, qlen=3, dcp=2, interleave=1, block_size=64,
               kv_dtype="fp8", max_local_len=2048, lengths=("uniform", 1024, 4096)),
    "c3": dict(batch=32, num_heads=128, qlen=1, dcp=8, interleave=1, block_size=64,
               kv_dtype="fp8", max_local_len=4096, lengths=("fixed", 32768)),
    "c4": dict(batch=32, num_heads=128, qlen=5, dcp=8, interleave=64, block_size=64,
               kv_dtype="fp8", max_local_len=16384,
               lengths=("loguniform+short", 8192, 131072, (5, 70, 300, 511))),
    "c5": dict(batch=4, num_heads=128, qlen=3, dcp=8, interleave=1, block_size=64,
               kv_dtype="fp8", max_local_len=131072, lengths=("fixed", 1048576)),
}

CONFIG_INDEX = {"c1": 0, "c2": 1, "c3": 2, "c4": 3, "c5": 4}

DESCRIPTIONS = {
    "c1": "tiny: B1 H8 qlen3 L200 dcp2 S1 bs16 bf16-KV",
    "c2": "B4 H96 qlen3 L~U[1024,4096] dcp2 S1 bs64 fp8-KV",
    "c3": "decode: B32 H128 qlen1 L32768 dcp8 S1 bs64 fp8-KV",
    "c4": "spec-verify: B32 H128 qlen5 L~logU[8192,131072]+{5,70,300,511} dcp8 S64 bs64 fp8-KV",
    "c5": "long-context: B4 H128 qlen3 L1048576 dcp8 S1 bs64 fp8-KV",
}

SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)
CHUNK_BLOCKS = 512


@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    num_heads: int
    qlen: int
    dcp: int
    interleave: int
    block_size: int
    kv_dtype: str               # "fp8" or "bf16"
    max_local_len: int
    max_blocks_per_seq: int
    num_blocks: int
    softmax_scale: float
    kv_scale: float
    seq_lens: torch.Tensor      # int32 [B]
    block_table: torch.Tensor   # int32 [B][MB]
    q: torch.Tensor             # bf16 [B*qlen][H][576]
    kv: torch.Tensor            # uint8 (E4M3 codes) or bf16, [W][NB][bs][576]
    causal: bool = True

    @property
    def rows(self) -> int:
        return self.batch * self.qlen

    def to(self, device) -> "Workload":
        d = dataclasses.replace(self)
        for f in ("seq_lens", "block_table", "q", "kv"):
            setattr(d, f, getattr(self, f).to(device))
        return d

    # Views for the oracle (host NumPy arrays of raw bits).
    def q_bits_np(self) -> np.ndarray:
        return self.q.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    def pools_np(self) -> np.ndarray:
        kv = self.kv.detach().cpu().contiguous()
        if self.kv_dtype == "fp8":
            return kv.numpy().view(np.uint8)
        return kv.view(torch.int16).numpy().view(np.uint16)


def _seed(*parts) -> int:
    return int(np.random.SeedSequence(list(parts)).generate_state(1, dtype=np.uint64)[0]
               & 0x7FFF_FFFF_FFFF)


def draw_lengths(spec, batch: int, rng: np.random.Generator) -> np.ndarray:
    kind = spec[0]
    if kind == "fixed":
        return np.full(batch, spec[1], dtype=np.int64)
    if kind == "uniform":
        return rng.integers(spec[1], spec[2] + 1, size=batch, dtype=np.int64)
    if kind == "loguniform+short":
        lo, hi, short = spec[1], spec[2], spec[3]
        n_long = batch - len(short)
        u = rng.uniform(math.log(lo), math.log(hi), size=n_long)
        longs = np.floor(np.exp(u)).astype(np.int64)
        return np.concatenate([longs, np.asarray(short, dtype=np.int64)])
    raise ValueError(kind)


def _normal(shape, seed: int, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def generate(name: str = "c1", *, device="cpu", seed_index: Optional[int] = None,
             overrides: Optional[dict] = None, seq_lens=None) -> Workload:
    """Build workload ``name`` on ``device`` (tensors created there).

    ``overrides`` replaces config fields (used by tests for small variants);
    ``seq_lens`` replaces the drawn lengths.
    """
    cfg = dict(CONFIGS[name])
    if overrides:
        cfg.update(overrides)
    k = CONFIG_INDEX.get(name, 9) if seed_index is None else seed_index
    ss = np.random.SeedSequence(1000 + k)
    W = cfg["dcp"]
    kids = ss.spawn(3 + W)
    B, H, qlen, bs = cfg["batch"], cfg["num_heads"], cfg["qlen"], cfg["block_size"]
    if seq_lens is None:
        lens = draw_lengths(cfg["lengths"], B, np.random.default_rng(kids[0]))
    else:
        lens = np.asarray(seq_lens, dtype=np.int64)
    MB = max(1, -(-cfg["max_local_len"] // bs))
    NB = B * MB + 8
    perm = np.random.default_rng(kids[1]).permutation(NB)
    table = perm[: B * MB].reshape(B, MB)
    q = _normal((B * qlen, H, D_QK), _seed(int(kids[2].generate_state(1)[0])), device)
    q = q.to(torch.bfloat16)

    def pool_chunks(r):
        base = int(kids[3 + r].generate_state(1)[0])
        for c0 in range(0, NB, CHUNK_BLOCKS):
            n = min(CHUNK_BLOCKS, NB - c0)
            yield c0, n, _normal((n, bs, D_QK), _seed(base, c0), device)

    if cfg["kv_dtype"] == "bf16":
        kv = torch.empty((W, NB, bs, D_QK), dtype=torch.bfloat16, device=device)
        for r in range(W):
            for c0, n, x in pool_chunks(r):
                kv[r, c0:c0 + n] = x.to(torch.bfloat16)
        kv_scale = 1.0
    elif cfg["kv_dtype"] == "fp8":
        amax = torch.zeros((), dtype=torch.float32, device=device)
        for r in range(W):
            for _, _, x in pool_chunks(r):
                amax = torch.maximum(amax, x.abs().max())
        kv_scale = float(amax.item()) / 448.0
        kv = torch.empty((W, NB, bs, D_QK), dtype=torch.uint8, device=device)
        for r in range(W):
            for c0, n, x in pool_chunks(r):
                codes = (x / kv_scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
                kv[r, c0:c0 + n] = codes.view(torch.uint8)
    else:
        raise ValueError(cfg["kv_dtype"])
    return Workload(
        name=name, batch=B, num_heads=H, qlen=qlen, dcp=W, interleave=cfg["interleave"],
        block_size=bs, kv_dtype=cfg["kv_dtype"], max_local_len=cfg["max_local_len"],
        max_blocks_per_seq=MB, num_blocks=NB, softmax_scale=SOFTMAX_SCALE,
        kv_scale=kv_scale,
        seq_lens=torch.as_tensor(lens, dtype=torch.int32).to(device),
        block_table=torch.as_tensor(table, dtype=torch.int32).to(device),
        q=q, kv=kv)


def generate_w_v(num_heads: int, payload: int = 128, seed: int = 7, device="cpu") -> torch.Tensor:
    """Synthetic per-head value projection for project-before-merge: bf16
    ``[H][payload][512]`` (row p of head h holds the 512 weights of projected
    value p), N(0, 1/512) so that projected values keep the scale of the latent
    ones. Drawn on the host, so every device sees the same weights."""
    x = _normal((num_heads, payload, 512), _seed(9100, seed), "cpu") / math.sqrt(512)
    return x.to(torch.bfloat16).to(device)


def make_anticorrelated(w: Workload, *, seed: int = 5, frac: float = 1.0 / 16,
                        kappa: float = 12.0, noise: float = 0.1) -> Workload:
    """Rewrite an FP8 workload so that the partial scores over dims [0, 256) and
    [256, 576) of one row disagree strongly (input construction only).

    q is constant on each span: c_h / 16 on both, with c_h in {0.75, 0.85, 0.95, 1.0}
    by head. Every cache row (every slot of every rank's pool) independently becomes
    "first-span dominant" (value ~kappa on dims [0, 256), ~0 on the rest) with
    probability frac, "second-span dominant" (~0 on [0, 256), ~kappa * 0.8 on the rest)
    with probability frac, or small (~0 everywhere); N(0, noise) is added to every
    value before the E4M3 cast, and kv_scale is 1. Where a group of tokens holds one
    row of each kind, the sum of the two spans' maxima lies far above the largest
    score of the group.
    """
    if w.kv_dtype != "fp8":
        raise ValueError("FP8 workloads only")
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    W, NB, bs, D = w.kv.shape
    u = torch.rand((W, NB, bs), generator=g)
    x = torch.randn((W, NB, bs, D), generator=g) * noise
    first = (u < frac).unsqueeze(-1)
    second = ((u >= frac) & (u < 2 * frac)).unsqueeze(-1)
    span0 = torch.zeros(D, dtype=torch.bool)
    span0[:256] = True
    x = x + torch.where(first & span0, torch.tensor(kappa), torch.tensor(0.0))
    x = x + torch.where(second & ~span0, torch.tensor(0.8 * kappa), torch.tensor(0.0))
    codes = x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    c = torch.tensor([0.75, 0.85, 0.95, 1.0])[torch.arange(w.num_heads) % 4] / 16.0
    q = c.view(1, -1, 1).expand(w.rows, w.num_heads, D).clone()
    out = dataclasses.replace(w)
    out.kv = codes.to(w.kv.device)
    out.q = q.to(torch.bfloat16).to(w.q.device)
    out.kv_scale = 1.0
    return out
