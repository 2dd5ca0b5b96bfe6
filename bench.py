#!/usr/bin/env python3
"""Throughput of one DCP causal MLA verify step on GB300.

A step is the whole hot path for all dcp virtual ranks of one batch:
metadata (row lengths, subpages, splits) -> split-KV partial attention ->
LSE merge into the BF16 output. Inputs are seeded synthetic tensors resident
in HBM; the default workload is the long-context one (batch 4, 128 heads,
qlen 3, 1,048,576 tokens, dcp 8, FP8 cache), whose cache (2.4 GB) is far larger
than L2, so no flush is needed between steps (smaller workloads flush L2 with a
512 MB write before every timed step, outside the timed events).

Prints ONE JSON line (rank 0). ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead (test infrastructure only).
With ``--gpus N`` under torchrun every rank runs an independent replica of the
workload (weak scaling; the dcp shards of a replica stay on its GPU).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV-tokens/s and TFLOP/s per verify step vs roofline fraction; μs per step"
UNIT = "KV-tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic(w):
    """Per-step KV tokens, flops and bytes (causal work only).

    KV tokens = sum_b L_b (each token read once by its owner);
    flops = sum_b sum_j H * g_j * 2 * (576 + 512);
    bytes = sum_b L_b * 576 * elem + R*H*576*2 (q) + R*H*512*2 (out).
    """
    lens = [int(x) for x in w.seq_lens.cpu().tolist()]
    H, qlen = w.num_heads, w.qlen
    tokens = sum(lens)
    flops = 0
    for L in lens:
        for j in range(qlen):
            g = L - qlen + 1 + j if w.causal else L
            flops += H * max(g, 0) * 2 * (576 + 512)
    elem = 1 if w.kv_dtype == "fp8" else 2
    R = w.batch * qlen
    nbytes = tokens * 576 * elem + R * H * 576 * 2 + R * H * 512 * 2
    return tokens, flops, nbytes


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 50 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, path):
        self.index, self.path, self.proc = index, path, None

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


class NvmlSampler:
    """The same clock fields read through NVML (ctypes, read-only queries) every 5 ms
    from a thread, so a timed region of a few tens of ms still gets many samples.
    ``ok`` is False when NVML cannot be loaded; the caller then uses nvidia-smi."""

    # clocks-event-reason bits of the NVML API
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index, period_s=0.005):
        import ctypes
        import threading
        self.ctypes, self.threading = ctypes, threading
        self.period, self.samples, self.ok = period_s, [], False
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
                return
            self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.lib, self.h, self.ok = lib, h, True
        except (OSError, AttributeError):
            self.ok = False

    def _read(self):
        c = self.ctypes
        mhz, mx, mw, rs = c.c_uint(), c.c_uint(), c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, c.byref(mhz)) != 0:  # 1: SM clock
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, c.byref(mx))
        self.lib.nvmlDeviceGetPowerUsage(self.h, c.byref(mw))
        self.reason_fn(self.h, c.byref(rs))
        return mhz.value, mx.value, mw.value / 1000.0, rs.value

    def __enter__(self):
        self.stop = False

        def loop():
            import time as _t
            while not self.stop:
                r = self._read()
                if r is not None:
                    self.samples.append(r)
                _t.sleep(self.period)
        self.th = self.threading.Thread(target=loop, daemon=True)
        self.th.start()
        return self

    def __exit__(self, *exc):
        self.stop = True
        self.th.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = set()
        for *_, rs in self.samples:
            for bit, name in self.REASONS.items():
                if rs & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x[0] for x in self.samples),
                "sm_max_mhz": max(x[1] for x in self.samples), "reasons": sorted(reasons),
                "samples": len(self.samples), "source": "nvml every 5 ms",
                "power_w_max": max(x[2] for x in self.samples)}


def clock_sampler(local, rank):
    """NVML sampler if NVML loads, else nvidia-smi every 50 ms (raw samples to
    DCP_CLOCKS_DIR when set)."""
    s = NvmlSampler(local)
    if s.ok:
        return s
    clocks_dir = os.environ.get("DCP_CLOCKS_DIR")
    return ClockSampler(local, os.path.join(clocks_dir, f"clocks_rank{rank}.csv")
                        if clocks_dir and os.path.isdir(clocks_dir)
                        else f"/tmp/dcp_clocks_{os.getpid()}.csv")


def kernel_source_hash():
    import glob
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "decode_context_mla_causal_gb300", "csrc", "*"))):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """DRAM traffic per launch from the committed ncu summary, only if it was
    taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel}:{workload}")
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def oracle_prepare(w, b=0):
    """Host copy of sequence b's blocks only (block table remapped)."""
    import torch

    import workloads

    table = w.block_table[b].long()
    sub = workloads.Workload(**{**w.__dict__})
    sub.kv = w.kv[:, table].cpu()
    sub.block_table = torch.arange(table.numel(), dtype=torch.int32).reshape(1, -1)
    sub.seq_lens = w.seq_lens[b:b + 1].cpu()
    sub.q = w.q[b * w.qlen:(b + 1) * w.qlen].cpu()
    sub.batch, sub.num_blocks = 1, table.numel()
    return dict(q_bits=sub.q_bits_np(), pools=sub.pools_np(),
                block_table=sub.block_table.numpy(), seq_lens=sub.seq_lens.numpy(),
                qlen=w.qlen, dcp=w.dcp, interleave=w.interleave, block_size=w.block_size,
                kv_dtype=w.kv_dtype, kv_scale=w.kv_scale, softmax_scale=w.softmax_scale)


def oracle_sample(w, prepared, heads_sample, rows_sample=None):
    """Time the CPU oracle on sequence 0 for a subset of heads and rows; returns the
    timing and the oracle's output and LSE of the sample."""
    import oracle

    heads = list(range(heads_sample))
    rows = [(0, j) for j in range(w.qlen)] if rows_sample is None else rows_sample
    t0 = time.perf_counter()
    ref = oracle.attention.forward(rows=rows, heads=heads, per_rank=False, **prepared)
    dt = time.perf_counter() - t0
    L = int(prepared["seq_lens"][0])
    equiv_tokens = L * (len(heads) * len(rows)) / (w.num_heads * w.qlen)
    return dict(value=equiv_tokens / dt, seconds=dt, ref=ref, heads=heads, rows=rows,
                sample=(f"sequence 0 ({L} tokens), {len(rows)} of {w.qlen} verify rows, "
                        f"{len(heads)} of {w.num_heads} heads; value = KV tokens x "
                        f"(sampled rows*heads / all rows*heads) / seconds"))


def oracle_cores():
    try:
        import numpy as np  # noqa: F401
        return os.cpu_count()
    except Exception:
        return None


# Heads of the oracle sample (all verify rows of sequence 0): the same sample for
# the cpu_baseline leg and the reference arm, sized for a few seconds of CPU work.
SAMPLE_HEADS = {"c1": 8, "c2": 96, "c3": 128, "c4": 32, "c5": 32}
BASELINE_SECONDS = 8.0  # the cpu_baseline leg repeats the sample to about this long


def cpu_baseline(w, out, lse):
    """The cpu_baseline leg: time the oracle on the sample (repeated to about
    BASELINE_SECONDS) and compare the GPU's output on the same rows and heads."""
    import numpy as np

    prepared = oracle_prepare(w)
    runs = [oracle_sample(w, prepared, SAMPLE_HEADS[w.name])]
    while sum(r["seconds"] for r in runs) < BASELINE_SECONDS and len(runs) < 16:
        runs.append(oracle_sample(w, prepared, SAMPLE_HEADS[w.name]))
    secs = sum(r["seconds"] for r in runs)
    value = len(runs) / sum(1.0 / r["value"] for r in runs)
    r0 = runs[0]
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    got_o = np.stack([o[b * w.qlen + j][r0["heads"]] for b, j in r0["rows"]])
    got_l = np.stack([l[b * w.qlen + j][r0["heads"]] for b, j in r0["rows"]])
    exp_o, exp_l = r0["ref"]["out"], r0["ref"]["lse"]
    d = np.abs(got_o - exp_o)
    fin = np.isfinite(exp_l)
    dl = np.abs(got_l[fin] - exp_l[fin]) if fin.any() else np.zeros(1)
    parity = {"sample": "the cpu_baseline sample", "max_abs_out": float(d.max()),
              "n_out": int(d.size), "n_out_over_1e-2": int((d > 1e-2).sum()),
              "max_abs_lse": float(dl.max()),
              "neg_inf_lse_match": bool(np.array_equal(np.isneginf(got_l), np.isneginf(exp_l)))}
    return ({"value": value, "unit": UNIT, "cores": oracle_cores(), "kind": "oracle",
             "sample": r0["sample"], "seconds": secs, "repeats": len(runs)}, parity)


def setup(config, dev, splits=0, batch=0):
    import torch

    import decode_context_mla_causal_gb300 as dm
    import workloads

    # batch: fewer sequences of the same shape (a small case for profiler captures)
    w = workloads.generate(config, device=dev, overrides=dict(batch=batch) if batch else None)
    if splits:
        ns, base = splits, 0
    else:  # the static split count, with room for wave balancing where it helps
        ns, base = dm.choose_split_plan(w.batch, w.qlen, w.num_heads, w.dcp, w.max_local_len,
                                        w.block_size, dm.concurrent_items())
    dims = dm.make_dims(batch=w.batch, qlen=w.qlen, num_heads=w.num_heads, dcp=w.dcp,
                        interleave=w.interleave, block_size=w.block_size,
                        max_blocks_per_seq=w.max_blocks_per_seq, max_local_len=w.max_local_len,
                        num_blocks=w.num_blocks, num_splits=ns, base_splits=base)
    kvt = dm.KV_FP8_E4M3 if w.kv_dtype == "fp8" else dm.KV_BF16
    step = dm.VerifyStep(dims, kvt, dev)
    scale = torch.tensor([w.kv_scale], dtype=torch.float32, device=dev)
    kv_bytes = w.kv.numel() * w.kv.element_size()
    flush = None
    if kv_bytes < 4 * 129 * 2**20:
        flush = torch.empty(512 * 2**20 // 4, dtype=torch.float32, device=dev)
    return dict(w=w, ns=ns, base=base, dims=dims, kvt=kvt, step=step, scale=scale, flush=flush,
                kv_bytes=kv_bytes)


def time_steps(env, K, warmup, stream):
    """W untimed steps, then K steps timed with CUDA events on the launch stream
    (metadata, partial with its item order, merge). Returns per-step lists in ms."""
    import torch

    w, step, scale, flush = env["w"], env["step"], env["scale"], env["flush"]

    def run():
        step.metadata(w.seq_lens, w.block_table)
        step.partial(w.q, w.kv, scale, w.softmax_scale)
        step.merge()

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    if step.read_status() != 0:
        raise RuntimeError(f"device status {step.read_status():#x}")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        if flush is not None:
            flush.fill_(float(i))
        ev[i][0].record(stream)
        step.metadata(w.seq_lens, w.block_table)
        ev[i][1].record(stream)
        step.partial(w.q, w.kv, scale, w.softmax_scale)
        ev[i][2].record(stream)
        step.merge()
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    return dict(step=[ev[i][0].elapsed_time(ev[i][3]) for i in range(K)],
                meta=[ev[i][0].elapsed_time(ev[i][1]) for i in range(K)],
                part=[ev[i][1].elapsed_time(ev[i][2]) for i in range(K)],
                merge=[ev[i][2].elapsed_time(ev[i][3]) for i in range(K)])


def time_packed(env, K, warmup, stream):
    """One split: the exchange's send buffer made two ways, each timed over K calls
    after W untimed ones: the partial kernel (fp32 partials) then the pack kernel,
    and the partial kernel writing the wire format itself (dcp_mla_partial_packed)."""
    import torch

    import decode_context_mla_causal_gb300 as dm

    w, step, scale = env["w"], env["step"], env["scale"]
    if env["ns"] != 1:  # the fused epilogue takes one split: a one-split step of the same dims
        d = env["dims"]
        step = dm.VerifyStep(dm.make_dims(
            batch=d.batch, qlen=d.qlen, num_heads=d.num_heads, dcp=d.dcp, interleave=d.interleave,
            block_size=d.block_size, max_blocks_per_seq=d.max_blocks_per_seq,
            max_local_len=d.max_local_len, num_blocks=d.num_blocks, num_splits=1,
            causal=bool(d.causal)), env["kvt"], w.q.device)
    ex = dm.A2AExchange(step)
    step.metadata(w.seq_lens, w.block_table)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    for i in range(warmup + K):
        e = ev[i - warmup] if i >= warmup else None
        if e:
            e[0].record(stream)
        step.partial(w.q, w.kv, scale, w.softmax_scale)
        if e:
            e[1].record(stream)
        ex.pack_ranks(stream)
        if e:
            e[2].record(stream)
        ex.partial_packed(w.q, w.kv, scale, w.softmax_scale, stream)
        if e:
            e[3].record(stream)
    torch.cuda.synchronize()
    if step.read_status() != 0:
        raise RuntimeError(f"packed status {step.read_status():#x}")
    avg = [1e3 * sum(e[j].elapsed_time(e[j + 1]) for e in ev) / K for j in range(3)]
    return {"partial_us": avg[0], "pack_us": avg[1], "partial_packed_us": avg[2],
            "saved_us": avg[0] + avg[1] - avg[2],
            "note": "send buffer of the all-to-all (payload 512): partial + pack, or the "
                    "partial kernel writing it directly (one split); not part of ms_per_step"}


def time_a2a(env, K, warmup, stream):
    """The step after the path: each rank's result in the all-to-all wire format
    (pack), then the combine with every rank on this device; plain (512 latent dims
    per head) and with project-before-merge (synthetic W_V, 512 -> 128). Each kernel
    timed over K rounds after W untimed ones, with its HBM bytes per launch."""
    import torch

    import decode_context_mla_causal_gb300 as dm
    import workloads

    w, step, ns = env["w"], env["step"], env["ns"]
    if w.num_heads % w.dcp != 0:
        return None
    dev = w.q.device
    a2a = {}
    w_v = workloads.generate_w_v(w.num_heads, 128, device=dev)
    nr, R, H = w.dcp, w.rows, w.num_heads
    for label, wv in (("plain", None), ("project_before_merge", w_v)):
        ex = dm.A2AExchange(step, w_v=wv)
        a_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
        for i in range(warmup + K):
            e = a_ev[i - warmup] if i >= warmup else None
            if e:
                e[0].record(stream)
            ex.pack_ranks(stream)
            if e:
                e[1].record(stream)
            if wv is not None:
                ex.project(stream)
            if e:
                e[2].record(stream)
            ex.combine_local(stream)
            if e:
                e[3].record(stream)
        torch.cuda.synchronize()
        if step.read_status() != 0:
            raise RuntimeError(f"a2a status {step.read_status():#x}")
        avg = [1e3 * sum(e[j].elapsed_time(e[j + 1]) for e in a_ev) / K for j in range(3)]
        packed_bytes = ex.packed.numel() * 2
        send_bytes = ex.send.numel() * 2
        # partials whose output the pack reads: every slot, or with wave balancing
        # the live ones (slot 0 and the non-empty slots; their m and l are read for all)
        slots = nr * w.batch * ns
        if env["base"]:
            beg, end = step.split_beg.cpu(), step.split_end.cpu()
            live = (end > beg)
            live[:, :, 0] = True
            slots = int(live.sum())
        pack_bytes = (slots * w.qlen * H * 4 * 512 + nr * ns * R * H * 8) + packed_bytes
        comb_bytes = send_bytes + R * H * (2 * ex.payload + 4)
        a2a[label] = {"payload": ex.payload, "send_bytes": send_bytes,
                      "kernel_us": {"pack": avg[0], "combine": avg[2]},
                      "pack_hbm_gbs": pack_bytes / (avg[0] / 1e6) / 1e9,
                      "combine_hbm_gbs": comb_bytes / (avg[2] / 1e6) / 1e9}
        if wv is not None:
            a2a[label]["kernel_us"]["project"] = avg[1]
            a2a[label]["project_tflops"] = 2.0 * nr * R * H * 512 * ex.payload / (avg[1] / 1e6) / 1e12
            a2a[label]["project_hbm_gbs"] = (
                packed_bytes + wv.numel() * 2 + send_bytes) / (avg[1] / 1e6) / 1e9
        del ex
    a2a["note"] = ("all-to-all wire format (BF16 output + float32 LSE as two 16-bit "
                   "halves), combined on this device; timed separately, not part of "
                   "ms_per_step")
    return a2a


def roofline(flops, nbytes, part_ms, peaks):
    tensor_peak = float(peaks["bf16_tflops"])
    hbm_peak = float(peaks["hbm_gbs"])
    achieved = flops / (part_ms / 1e3) / 1e12
    return achieved, tensor_peak, hbm_peak, max(nbytes / (hbm_peak * 1e9),
                                                flops / (tensor_peak * 1e12)) * 1e3


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c5", choices=["c1", "c2", "c3", "c4", "c5"])
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences of the headline workload (0: the workload's own); a "
                         "smaller case for profiler captures, not a bench line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    import torch
    import torch.distributed as dist

    import workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        return run_reference(args, rank, world)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import decode_context_mla_causal_gb300 as dm

    env = setup(args.config, dev, args.splits, args.batch)
    w, dims, step, scale, kvt, ns, flush = (env[k] for k in
                                            ("w", "dims", "step", "scale", "kvt", "ns", "flush"))
    tokens, flops, nbytes = algorithmic(w)
    stream = torch.cuda.current_stream(dev)
    K = args.steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = clock_sampler(local, rank)
    for _ in range(args.warmup):  # untimed, before the sampler starts
        step.metadata(w.seq_lens, w.block_table)
        step.partial(w.q, w.kv, scale, w.softmax_scale)
        step.merge()
    with sampler:
        tm = time_steps(env, K, 0, stream)
    if world > 1:
        dist.barrier()
    step_ms, part_ms, meta_ms, merge_ms = tm["step"], tm["part"], tm["meta"], tm["merge"]
    total_ms = sum(step_ms)
    t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    total_ms = float(t.item())
    ms_per_step = total_ms / K
    value = tokens * world * K / (total_ms / 1e3)
    out_keep, lse_keep = step.out.clone(), step.lse.clone()

    # end to end through the C ABI with host buffers: per step H2D of q, seq_lens,
    # block_table from pinned memory, the three calls, D2H of out and lse
    hq = w.q.cpu().pin_memory()
    hs = w.seq_lens.cpu().pin_memory()
    ht = w.block_table.cpu().pin_memory()
    ho = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    hl = torch.empty(step.lse.shape, dtype=step.lse.dtype).pin_memory()
    dq, dsq, dt_ = torch.empty_like(w.q), torch.empty_like(w.seq_lens), torch.empty_like(w.block_table)
    h2d = hq.numel() * hq.element_size() + hs.numel() * 4 + ht.numel() * 4
    d2h = ho.numel() * ho.element_size() + hl.numel() * 4

    def run_e2e():
        dq.copy_(hq, non_blocking=True)
        dsq.copy_(hs, non_blocking=True)
        dt_.copy_(ht, non_blocking=True)
        step.metadata(dsq, dt_)
        step.partial(dq, w.kv, scale, w.softmax_scale)
        step.merge()
        ho.copy_(step.out, non_blocking=True)
        hl.copy_(step.lse, non_blocking=True)

    for _ in range(args.warmup):
        run_e2e()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    for i in range(K):
        if flush is not None:
            flush.fill_(float(i))
        e0.record(stream)
        run_e2e()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    te = torch.tensor([e2e_ms], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(te, op=dist.ReduceOp.MAX)
    e2e_value = tokens * world * K / (float(te.item()) / 1e3)

    # the step before the path: the new tokens' slot mapping and KV write (FP8:
    # quantisation), timed on its own after the verify step (it overwrites the
    # new tokens' cache rows with synthetic values)
    new_rows = torch.randn((w.rows, 576), generator=torch.Generator(device=dev).manual_seed(17),
                           device=dev).to(torch.bfloat16)
    slots = torch.empty((w.dcp, w.rows), dtype=torch.int32, device=dev)
    kv_status = torch.zeros(1, dtype=torch.int32, device=dev)
    kw_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    kv_copy = w.kv.clone()
    for i in range(args.warmup + K):
        if i >= args.warmup:
            kw_ev[i - args.warmup][0].record(stream)
        dm.dcp_kv_slot_mapping(dims, w.seq_lens, w.block_table, 0, w.dcp, slots, kv_status)
        if i >= args.warmup:
            kw_ev[i - args.warmup][1].record(stream)
        dm.dcp_kv_write(dims, slots, new_rows, kvt, scale, w.dcp, kv_copy, kv_status)
        if i >= args.warmup:
            kw_ev[i - args.warmup][2].record(stream)
    torch.cuda.synchronize()
    del kv_copy
    if int(kv_status.item()) != 0:
        raise RuntimeError(f"kv write status {int(kv_status.item()):#x}")
    kv_map_us = 1e3 * sum(e[0].elapsed_time(e[1]) for e in kw_ev) / K
    kv_write_us = 1e3 * sum(e[1].elapsed_time(e[2]) for e in kw_ev) / K

    a2a = time_a2a(env, K, args.warmup, stream)

    peaks, src = load_peaks()
    part_avg = sum(part_ms) / K
    achieved_tf, tensor_peak, hbm_peak, roof_ms = roofline(flops, nbytes, part_avg, peaks)
    clocks = sampler.summary()
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dm.COMPUTE_DTYPE,
        "data": "synthetic (seeded N(0,1) q and cache, FP8 E4M3 per-tensor scale)",
        "config": {"workload": f"{args.config} {workloads.DESCRIPTIONS[args.config]}",
                   "global_batch": w.batch * world, "seq_len": int(w.seq_lens.max()),
                   "qlen": w.qlen, "num_heads": w.num_heads, "dcp": w.dcp,
                   "interleave": w.interleave, "num_splits": ns,
                   "base_splits": env["base"],
                   "parallelism": f"dcp{w.dcp} virtual shards per GPU; replicas x{world}",
                   "l2": ("flushed with a 512 MB write before each timed step" if flush is not None
                          else f"inputs larger than L2 (cache {env['kv_bytes'] / 1e9:.2f} GB)")},
        "us_per_step": ms_per_step * 1e3,
        "tflops": flops / (ms_per_step / 1e3) / 1e12,
        "kernel_us": {"metadata": 1e3 * sum(meta_ms) / K, "partial": 1e3 * part_avg,
                      "merge": 1e3 * sum(merge_ms) / K},
        "roofline": {"bound": "tensor", "achieved": achieved_tf, "peak": tensor_peak,
                     "unit": "TFLOP/s", "frac": achieved_tf / tensor_peak,
                     "traffic": profiled_traffic("partial", args.config),
                     "peak_source": f"{src} bf16 dense (burst), MEASURED_PEAKS.json"
                     if src == "measured" else "fallback 1.9 PFLOP/s bf16",
                     "kernel": "dcp_mla_partial",
                     "step_frac": roof_ms / ms_per_step,
                     "hbm_bytes_algorithmic": nbytes,
                     "hbm_frac_of_partial": nbytes / (part_avg / 1e3) / (hbm_peak * 1e9)},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "kv_write": {"kernel_us": {"slot_mapping": kv_map_us, "write": kv_write_us},
                     "rows": w.rows, "ranks": w.dcp,
                     "note": "new-token KV write (the step before the verify path), timed "
                             "separately; not part of ms_per_step"},
        "a2a": a2a,
        "gpu_launches": 4 * K,  # metadata, item order, partial, merge
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"], res["parity"] = cpu_baseline(w, out_keep, lse_keep)
    del env, w, step, out_keep, lse_keep, hq, ho, dq
    torch.cuda.empty_cache()

    # every other workload of the path at N=1: the same step, timed the same way
    # (K steps after W untimed ones), with its roofline fraction, the oracle timed on
    # its sample and the parity of that sample
    if world == 1 and not args.no_per_config:
        per = {}
        sampler2 = clock_sampler(local, rank)
        with sampler2:
            for cfg in ("c1", "c2", "c3", "c4", "c5"):
                if cfg == args.config:
                    continue
                e = setup(cfg, dev)
                cw = e["w"]
                ctok, cfl, cby = algorithmic(cw)
                ct = time_steps(e, K, args.warmup, stream)
                cms = sum(ct["step"]) / K
                cpart = sum(ct["part"]) / K
                ach, tp, hp, croof = roofline(cfl, cby, cpart, peaks)
                entry = {"workload": f"{cfg} {workloads.DESCRIPTIONS[cfg]}",
                         "num_splits": e["ns"], "base_splits": e["base"], "ms_per_step": cms,
                         "value": ctok * K / (sum(ct["step"]) / 1e3), "unit": UNIT,
                         "tflops": cfl / (cms / 1e3) / 1e12,
                         "kernel_us": {"metadata": 1e3 * sum(ct["meta"]) / K,
                                       "partial": 1e3 * cpart,
                                       "merge": 1e3 * sum(ct["merge"]) / K},
                         "roofline": {"bound": "tensor", "achieved": ach, "peak": tp,
                                      "unit": "TFLOP/s", "frac": ach / tp,
                                      "traffic": profiled_traffic("partial", cfg),
                                      "step_frac": croof / cms,
                                      "hbm_frac_of_partial":
                                          cby / (cpart / 1e3) / (hp * 1e9)},
                         "l2": ("flushed with a 512 MB write before each timed step"
                                if e["flush"] is not None else "inputs larger than L2")}
                if cfg in ("c3", "c4"):  # the exchange at the sizes where HBM rate means something
                    entry["a2a"] = time_a2a(e, K, args.warmup, stream)
                if cfg in ("c3", "c4") and cw.num_heads % cw.dcp == 0:
                    entry["a2a_one_split"] = time_packed(e, K, args.warmup, stream)
                if not args.no_cpu_baseline:
                    entry["cpu_baseline"], entry["parity"] = cpu_baseline(
                        cw, e["step"].out, e["step"].lse)
                per[cfg] = entry
                del e, cw
                torch.cuda.empty_cache()
        res["per_config"] = per
        res["per_config_clocks"] = sampler2.summary()
        res["gpu_launches_per_config"] = 4 * K * len(per)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm (rank 0 only): one step = the oracle on
    the same sample the cpu_baseline leg of the other arm times."""
    if rank != 0:
        return
    import torch

    import workloads

    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    w = workloads.generate(args.config, device=dev)
    heads = SAMPLE_HEADS[args.config]
    prepared = oracle_prepare(w)
    for _ in range(args.warmup):  # untimed (the oracle keeps no state)
        oracle_sample(w, prepared, heads)
    vals, secs = [], 0.0
    cb = None
    for _ in range(args.steps):
        cb = oracle_sample(w, prepared, heads)
        vals.append(cb["value"])
        secs += cb["seconds"]
    value = len(vals) / sum(1.0 / v for v in vals)
    res = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "config": {"workload": f"{args.config} {workloads.DESCRIPTIONS[args.config]}"},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_cores(),
                            "kind": "oracle", "sample": cb["sample"]},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
