#!/usr/bin/env python3
"""Benchmark of one paged decode step (copy-on-write copy + slot-mapped append
+ paged decode attention with its split-K merge) on synthetic inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--partition P] [--impl ours|reference]

Prints one JSON line.  ``value`` is the step's algorithmic bytes (KV gathered
through the block tables + q + out + tables + lens, the append's rows and the
block copies) over the device time of exactly K steps (CUDA events, inputs
resident in HBM), summed over ranks and divided by the slowest rank's time.
``e2e`` is the same metric through the public API with every step's inputs
copied from pinned host memory and the output copied back inside the timed
region.  ``roofline`` is the decode kernel's achieved bandwidth against the
measured HBM copy peak.  ``cpu_baseline`` times the float64 oracle on a
bounded sample of the same workload.  ``--impl reference`` times that oracle
alone, as the reference arm.  The default run (the Llama-7B-shaped MHA
workload on one GPU) also times every other decode config under ``configs``
and the chunked prefill (bf16 and fp8 pools), the host prefix cache and block
swap under ``next``; ``--workload prefill_*`` times a prefill step instead.

With ``--gpus N`` (torchrun) every rank runs its own replica of the workload
on its own GPU (the path has no exchange step; no collective touches the
data), so scaling is weak.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode-attention KV GB/s (% of GB300 HBM peak) and µs/step, 1 GPU"
DEFAULT_WORKLOAD = "llama7b_mha"
_CSRC = "paged_kv_cache_10_gb300/csrc/"
# Sources of the decode kernel a workload runs (CUDA-core kernel for one
# query head per KV head or head_size 64; tensor-core kernel for GQA at 128).
KERNEL_SOURCES = {
    "cuda_core": [_CSRC + "pkv_decode_impl.cuh", _CSRC + "pkv_device.cuh", _CSRC + "pkv_append.cuh"],
    "tensor_core": [_CSRC + "pkv_decode_impl.cuh", _CSRC + "pkv_device.cuh", _CSRC + "pkv_decode_mma.cuh",
                    _CSRC + "pkv_append.cuh"],
    "cascade": [_CSRC + "pkv_decode_impl.cuh", _CSRC + "pkv_device.cuh", _CSRC + "pkv_decode_mma.cuh",
                _CSRC + "pkv_append.cuh",
                _CSRC + "pkv_cascade.cu", _CSRC + "pkv_prefill.cu", _CSRC + "pkv_tcgen05.cuh", _CSRC + "pkv_merge.cuh"],
    "prefill": [_CSRC + "pkv_prefill.cu", _CSRC + "pkv_tcgen05.cuh", _CSRC + "pkv_device.cuh",
                _CSRC + "pkv_decode_mma.cuh"],
}


# ------------------------------------------------------------------ helpers
def decode_kernel_kind(wl) -> str:
    return "tensor_core" if (wl.Hq // wl.Hkv >= 2 and wl.D == 128) else "cuda_core"


def code_only(src: str) -> str:
    """Source text without // comments, trailing blanks and empty lines, so
    an edit to comments alone leaves the hash (and recorded counters) valid."""
    out = []
    for line in src.splitlines():
        line = re.sub(r"//.*$", "", line).rstrip()
        if line:
            out.append(line)
    return "\n".join(out)


def kernel_hash(kind: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        h.update(code_only(open(os.path.join(ROOT, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:12]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def recorded_traffic(workload: str, kind: str):
    """dram read+write bytes per decode launch from the committed ncu summary,
    valid only for the kernel sources it was taken on."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    kh = kernel_hash(kind)
    for line in open(p):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == kh:
            return float(parts[2])
    return None


def step_bytes(step) -> dict:
    """Algorithmic bytes of one step of a DecodeStep."""
    wl = step.wl
    ke = wl.kv_elem_bytes()
    qe = 2
    lens = step.seq_lens.astype(np.int64)
    kv = int(lens.sum()) * 2 * wl.Hkv * wl.D * ke
    q_out = 2 * wl.S * wl.Hq * wl.D * qe
    tables = int(((lens + wl.b - 1) // wl.b).sum()) * 4 + wl.S * 4
    decode = kv + q_out + tables
    # distinct KV bytes: every distinct (block, token) the batch gathers, counted
    # once -- the least any method must read when sequences share blocks
    ids, valid = [], []
    for r in range(wl.S):
        L = int(lens[r])
        nb = (L + wl.b - 1) // wl.b
        if nb:
            ids.append(step.tables[r, :nb].astype(np.int64))
            valid.append(np.minimum(wl.b, L - wl.b * np.arange(nb)))
    if ids:
        ids, valid = np.concatenate(ids), np.concatenate(valid)
        best = np.zeros(int(ids.max()) + 1, np.int64)
        np.maximum.at(best, ids, valid)
        unique_tokens = int(best.sum())
    else:
        unique_tokens = 0
    unique_kv = unique_tokens * 2 * wl.Hkv * wl.D * ke
    n_app = int((step.slots >= 0).sum())
    in_e = 2
    append = n_app * 2 * wl.Hkv * wl.D * (in_e + ke) + wl.S * 8
    block_bytes = wl.Hkv * wl.b * wl.D * ke
    copy = len(step.pairs) * (2 * 2 * block_bytes + 8)
    return {"kv": kv, "decode": decode, "append": append, "copy": copy, "total": decode + append + copy,
            "unique_kv": unique_kv, "decode_unique": unique_kv + q_out + tables}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, stamped on arrival."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.samples = []
        self.proc = None
        ident = []
        try:
            ident = ["-i", "GPU-" + str(torch.cuda.get_device_properties(device).uuid)]
        except Exception:
            ident = []
        cmd = ["nvidia-smi", *ident, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                self.samples.append((time.monotonic(), float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                pass

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4) if s[3][i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside)}


def aggregate(value_bytes: float, seconds: float, group=None):
    """Whole-job bytes (sum over ranks) and time (max over ranks)."""
    import torch.distributed as dist
    if group is None and not (dist.is_available() and dist.is_initialized()):
        return value_bytes, seconds
    t = torch.tensor([value_bytes, seconds], dtype=torch.float64)
    if dist.get_backend(group) == "nccl":
        t = t.cuda()
    b = t[0:1].clone()
    s = t[1:2].clone()
    dist.all_reduce(b, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(s, op=dist.ReduceOp.MAX, group=group)
    return float(b.item()), float(s.item())


E2E_COPIES = ("every step: its inputs host->device in one upload from a pinned staging buffer on an upload "
              "stream, its result device->host into pinned memory on a download stream; two device buffer sets, "
              "so the copies of one step overlap the kernels of its neighbours")


def e2e_pipelined(h, launch, out, steps, stream, flush_buf=None):
    """Times `steps` steps end to end as a serving loop runs them: every step
    copies its inputs `h` (host tensors, staged in one pinned buffer) to the
    device in one upload, launches its
    kernels (`launch(device_inputs, device_out)`) and copies the result back
    into pinned host memory.  Two device buffer sets let step i + 1's
    host->device copies (on an upload stream) overlap step i's kernels, and
    step i's device->host copy (on a download stream) overlap step i + 1.
    Returns the elapsed ms on `stream` from before the first copy to after
    the last result has landed, minus the L2 flushes (`flush_buf` written
    before each step's kernels, each timed by its own events), and the bytes
    one upload moves."""
    dev = out.device
    # the step's inputs staged in one pinned buffer (256-byte aligned fields),
    # so a step is one upload; the device copies are views of one buffer
    offs, n = {}, 0
    for k, t in h.items():
        offs[k] = n
        n += -(-(t.numel() * t.element_size()) // 256) * 256
    staged = torch.empty(n, dtype=torch.uint8).pin_memory()
    for k, t in h.items():
        nb = t.numel() * t.element_size()
        staged[offs[k]:offs[k] + nb].copy_(t.reshape(-1).view(torch.uint8))
    packed = [torch.empty(n, dtype=torch.uint8, device=dev) for _ in range(2)]
    ds = [{k: packed[i][offs[k]:offs[k] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
           for k, t in h.items()} for i in range(2)]
    outs = [out, torch.empty_like(out)]
    out_hs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(2)]   # inputs of the buffer's step on the device
    done = [torch.cuda.Event() for _ in range(2)]    # its kernels finished (inputs free, output written)
    landed = [torch.cuda.Event() for _ in range(2)]  # its output copied to the host
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fl = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps if flush_buf is not None else 0)]
    torch.cuda.synchronize()
    e0.record(stream)
    up.wait_stream(stream)
    down.wait_stream(stream)
    for i in range(steps):
        b = i & 1
        if i >= 2:
            up.wait_event(done[b])
        with torch.cuda.stream(up):
            packed[b].copy_(staged, non_blocking=True)
        ready[b].record(up)
        if flush_buf is not None:
            fl[i][0].record(stream)
            flush_buf.zero_()
            fl[i][1].record(stream)
        stream.wait_event(ready[b])
        if i >= 2:
            stream.wait_event(landed[b])
        launch(ds[b], outs[b])
        done[b].record(stream)
        down.wait_event(done[b])
        with torch.cuda.stream(down):
            out_hs[b].copy_(outs[b], non_blocking=True)
        landed[b].record(down)
    stream.wait_stream(up)
    stream.wait_stream(down)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) - sum(a.elapsed_time(b) for a, b in fl), n


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------- oracle leg
# The float64 oracle runs only in this leg (and in the reference arm below):
# it times the oracle on bounded samples of the workload (cpu_baseline) and,
# outside every timed region, recomputes the whole measured step to report
# the GPU output's error.  Nothing it computes feeds the GPU path.
TOL = {"f16": 2e-3, "bf16": 1e-2, "e4m3": 1e-2}  # max-abs bounds on the attention output
_MANT = {"f16": 10, "bf16": 7}
FP32_TERM = 2.0 ** -14


def error_bound(ref: np.ndarray, out_dtype: str, tol: float, vmax: float) -> np.ndarray:
    """Per-element bound on |out - oracle|: `tol`, except where half a unit in
    the last place of the 16-bit output format at the oracle value exceeds
    it (bf16 |out| >= 4, f16 |out| >= 8), where no value of that format can
    meet it: there half that unit plus twice the float32 term 2^-14 * max|V|."""
    a = np.maximum(np.abs(ref), np.finfo(np.float64).tiny)
    half = 0.5 * np.exp2(np.floor(np.log2(a)) - _MANT[out_dtype])
    return np.where(half > tol, half + 2.0 * FP32_TERM * vmax, tol)


def oracle_host_step(wl):
    """Slots, copy-on-write pairs, block tables and lengths of the step from
    the oracle's own allocator model (the workload's script replayed)."""
    from oracle.allocator_model import AllocatorModel
    m = AllocatorModel(wl.NB, wl.b, wl.free_order)
    for op in wl.setup:
        if op[0] == "new":
            m.seq_new(op[1], op[2])
        elif op[0] == "fork":
            m.fork(op[1], op[2])
        elif op[0] == "extend":
            for _ in range(op[2]):
                m.append_slot(op[1])
        elif op[0] == "free":
            m.free_seq(op[1])
    slots = np.full(wl.S, -1, np.int64)
    pairs = []
    for s in wl.step_seqs:
        slot, cow = m.append_slot(s)
        slots[s] = slot
        if cow:
            pairs.append(cow)
    tables = np.full((wl.S, wl.max_blocks), -1, np.int32)
    lens = np.zeros(wl.S, np.int32)
    for s in range(wl.S):
        t = m.block_table(s)
        tables[s, :len(t)] = t
        lens[s] = m.lens[s]
    return slots, np.array(pairs, np.int32).reshape(-1, 2), tables, lens


class HostStep:
    """The host bookkeeping of one decode step (no device state)."""

    def __init__(self, wl, slots, pairs, tables, lens):
        self.wl, self.slots, self.pairs, self.tables, self.seq_lens = wl, slots, pairs, tables, lens


def oracle_rows_step(wl, step, rows, pools):
    """The float64 oracle on rows of the workload: their append and their
    decode (plus the copy-on-write copies of the step).  ``pools`` = (k, v)
    numpy pools updated in place (idempotent).  Returns the decode output."""
    import oracle
    kp, vp = pools
    if len(step.pairs):
        oracle.copy_blocks(kp, vp, wl.kv_dtype, step.pairs)
    sl = np.full(wl.S, -1, np.int64)
    sl[rows] = step.slots[rows]
    oracle.append(wl.k_new, wl.v_new, wl.in_dtype, sl, kp, vp, wl.kv_dtype, wl.k_scale, wl.v_scale)
    return oracle.paged_decode(np.ascontiguousarray(wl.q[rows]), wl.q_dtype, kp, vp, wl.kv_dtype,
                               np.ascontiguousarray(step.tables[rows]), np.ascontiguousarray(step.seq_lens[rows]),
                               wl.scale, wl.k_scale, wl.v_scale)


def rows_bytes(step, rows) -> int:
    wl = step.wl
    ke = wl.kv_elem_bytes()
    lens = step.seq_lens[rows].astype(np.int64)
    kv = int(lens.sum()) * 2 * wl.Hkv * wl.D * ke
    other = 2 * len(rows) * wl.Hq * wl.D * 2 + int(((lens + 15) // 16).sum()) * 4
    app = int((step.slots[rows] >= 0).sum()) * 2 * wl.Hkv * wl.D * (2 + ke)
    return kv + other + app


def _time_oracle(wl, step, pools, budget_s):
    """Whole sequences (all heads) through the oracle, repeated over the
    batch until ~budget_s of CPU time: (GB/s, reps, sequences per rep, s)."""
    t = time.perf_counter()
    oracle_rows_step(wl, step, np.array([0]), pools)
    one = max(time.perf_counter() - t, 1e-3)
    n = int(max(1, min(wl.S, budget_s / one)))
    done, dt, reps = 0, 0.0, 0
    while dt < budget_s and reps < 1000:
        rows = (np.arange(n) + reps * n) % wl.S
        t = time.perf_counter()
        oracle_rows_step(wl, step, rows, pools)
        dt += time.perf_counter() - t
        done += rows_bytes(step, rows)
        reps += 1
    return done / dt / 1e9, reps, n, dt


def cpu_baseline(wl, step, budget_s=10.0, single_s=3.0):
    """The oracle on whole-sequence samples of the workload, on all host
    cores (about budget_s of CPU time) and on one core (about single_s)."""
    import oracle
    pools = (wl.k_pool.copy(), wl.v_pool.copy())
    cores = oracle.num_threads()
    gbs, reps, n, dt = _time_oracle(wl, step, pools, budget_s)
    out = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
           "sample": f"{reps} x {n} of {wl.S} sequences of {wl.name} (all heads): their append + float64 "
                     f"decode, {dt:.1f} s"}
    if single_s > 0:
        oracle.set_num_threads(1)
        try:
            g1, r1, n1, d1 = _time_oracle(wl, step, pools, single_s)
        finally:
            oracle.set_num_threads(cores)
        out["single_thread"] = {"value": round(g1, 4), "unit": "GB/s", "cores": 1,
                                "sample": f"{r1} x {n1} sequences, {d1:.1f} s"}
    return out


def _host_bits(t) -> np.ndarray:
    """A device tensor's raw bits on the host (uint16 or uint8)."""
    t = t.detach().cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if t.element_size() == 2 else t.view(torch.uint8).numpy()


def oracle_parity(step) -> dict:
    """Untimed: the whole step (copy-on-write copies, appends, every row's
    decode) recomputed by the oracle from its own allocator model, against
    the GPU's host bookkeeping, pools and output."""
    import oracle
    wl = step.wl
    t0 = time.perf_counter()
    slots, pairs, tables, lens = oracle_host_step(wl)
    host_ok = (np.array_equal(step.slots, slots) and np.array_equal(np.asarray(step.pairs).reshape(-1, 2), pairs)
               and np.array_equal(step.tables, tables) and np.array_equal(step.seq_lens, lens))
    hs = HostStep(wl, slots, pairs, tables, lens)
    pools = (wl.k_pool.copy(), wl.v_pool.copy())
    ref = oracle_rows_step(wl, hs, np.arange(wl.S), pools)

    pools_ok = bool(np.array_equal(_host_bits(step.k_cache), pools[0])
                    and np.array_equal(_host_bits(step.v_cache), pools[1]))
    got = oracle.dequantize(_host_bits(step.out), wl.q_dtype)
    tol = TOL[wl.kv_dtype]
    vmax = float(np.max(np.abs(oracle.dequantize(pools[1], wl.kv_dtype)))) * (wl.v_scale if wl.kv_dtype == "e4m3"
                                                                               else 1.0)
    err = np.abs(got - ref)
    over = float(np.max(err - error_bound(ref, wl.q_dtype, tol, vmax))) if ref.size else -tol
    return {"rows": int(wl.S), "max_abs_err": float(err.max()) if ref.size else 0.0,
            "max_abs_oracle": float(np.abs(ref).max()) if ref.size else 0.0, "tol": tol,
            "within_tolerance": bool(over <= 0 and np.all(np.isfinite(got))),
            "max_err_minus_bound": over, "pools_bit_exact": pools_ok, "host_bookkeeping_exact": bool(host_ok),
            "oracle_s": round(time.perf_counter() - t0, 2),
            "basis": "every row and head of the step against the float64 oracle; bound: max-abs tol, or half an "
                     "ulp of the output format + 2^-13 max|V| where that half ulp exceeds tol"}


def kv_utilisation(step) -> dict:
    """Share of the block slots the batch holds that carry a token (distinct
    blocks, a shared block counted once) and the largest per-sequence waste
    (slots of its last block past its length; at most block_size - 1)."""
    wl = step.wl
    lens = step.seq_lens.astype(np.int64)
    nb = (lens + wl.b - 1) // wl.b
    ids, valid = [], []
    for r in range(wl.S):
        if nb[r]:
            ids.append(step.tables[r, :nb[r]].astype(np.int64))
            valid.append(np.minimum(wl.b, lens[r] - wl.b * np.arange(nb[r])))
    if not ids:
        return {"utilisation": 1.0, "max_waste_tokens_per_seq": 0, "distinct_blocks": 0}
    ids, valid = np.concatenate(ids), np.concatenate(valid)
    best = np.zeros(int(ids.max()) + 1, np.int64)
    np.maximum.at(best, ids, valid)
    used = np.unique(ids)
    return {"utilisation": round(float(best[used].sum()) / (len(used) * wl.b), 5),
            "max_waste_tokens_per_seq": int((nb * wl.b - lens).max()), "distinct_blocks": int(len(used)),
            "bound": f"waste <= block_size - 1 = {wl.b - 1} tokens per sequence"}


# ----------------------------------------------------------------- our arm
# every decode config of the benchmark, in the order the default run times them
DECODE_CONFIGS = [
    ("tiny_fp16", False, False),
    ("llama7b_mha", False, False),
    ("llama3_8b_gqa", False, False),
    ("longctx_fp8", False, False),
    ("prefix_share", False, False),
    ("prefix_share", True, True),  # shared-prefix (cascade) decode, each step one CUDA-graph replay
]


def measure_decode(args, rank, world, local_rank, name, cascade=False, graph=False, steps=None, sampler=None,
                   oracle_leg=True, cpu_budget=10.0):
    """Times one decode workload (K device-timed steps, the decode call's
    launches, the e2e loop) and, on rank 0 of a single-GPU run, the oracle
    leg.  Returns the JSON line of the workload (rank 0) or None."""
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = workloads.NAMED[name]()
    step = DecodeStep(wl, device=dev, partition_tokens=args.partition, cascade=cascade,
                      fused=not args.unfused, plan={"auto": "auto", "on": True, "off": False}[args.decode_plan])
    nbytes = step_bytes(step)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    working_set = nbytes["total"]
    flush = working_set < 4 * l2
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev) if flush else None

    for _ in range(max(args.warmup, 3)):
        step.run()
    torch.cuda.synchronize()

    K = steps or args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    g = step.capture() if graph else None
    if g is not None:
        for _ in range(max(args.warmup, 3)):
            g.replay()
    barrier()
    torch.cuda.synchronize()
    t_load0 = time.monotonic()
    for i in range(K):
        if flush:
            flush_buf.zero_()
        a, b, c = ev[i]
        a.record(stream)
        if g is not None:
            g.replay()  # the whole step, one launch
        else:
            step.copy()
            step.append()
            b.record(stream)
            step.decode()
        c.record(stream)
    torch.cuda.synchronize()
    t_load1 = time.monotonic()
    barrier()
    if flush:
        step_ms = [a.elapsed_time(c) for a, _, c in ev]
        total_ms = sum(step_ms)
    else:
        total_ms = ev[0][0].elapsed_time(ev[-1][2])
    if g is None:
        decode_ms = [b.elapsed_time(c) for _, b, c in ev]
    else:
        # kernel roofline from replays of a graph holding the decode call
        # alone (its kernels without the host's launch work, which a graph
        # removes; re-running a step's append and copies is idempotent)
        gdec = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(gdec):
            step.decode()
        torch.cuda.synchronize()
        dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            if flush:
                flush_buf.zero_()
            dev_ev[i][0].record(stream)
            gdec.replay()
            dev_ev[i][1].record(stream)
        torch.cuda.synchronize()
        decode_ms = [x.elapsed_time(y) for x, y in dev_ev]
    # extend the load window (same steps, untimed) if it was too short for clock samples
    if sampler and not args.profile and t_load1 - t_load0 < 1.0:
        t_ext = time.monotonic()
        while time.monotonic() - t_ext < 1.5:
            for _ in range(20):
                step.run()
            torch.cuda.synchronize()
        t_load1 = time.monotonic()

    tot_bytes, tot_s = aggregate(nbytes["total"] * K, total_ms / 1e3)
    value = tot_bytes / tot_s / 1e9

    # ---- end to end through the public API from pinned host buffers
    h = {
        "q": step.q.cpu().pin_memory(), "k": step.k_new.cpu().pin_memory(), "v": step.v_new.cpu().pin_memory(),
        "slots": step.d_slots.cpu().pin_memory(), "tables": step.d_tables.cpu().pin_memory(),
        "lens": step.d_lens.cpu().pin_memory(),
    }
    if len(step.pairs):  # the step's copy-on-write: per-row sources (fused) or the pair list
        h["cow"] = (step.d_cow_src if step.fused else step.d_pairs).cpu().pin_memory()
    if step.work is not None:  # the host plan, rebuilt from the host arrays every step
        h["work"] = torch.from_numpy(step.work_host.copy())
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = step.out.numel() * step.out.element_size()
    Ke = 0 if args.profile else max(1, min(K, 200))
    barrier()

    def launch_decode(dd, o):
        from paged_kv_cache_10_gb300 import pagedkv as pk
        if len(step.pairs) and not step.fused:
            pk.copy_blocks(step.k_cache, step.v_cache, step.desc, dd["cow"])
        step.append(k=dd["k"], v=dd["v"], slots=dd["slots"])
        if "work" in dd:  # planning is host work of the step; the batch (so the plan) never changes here
            wk = pk.decode_plan(step.seq_lens, wl.Hkv, step.max_seq_len, step.partition_tokens)
            if not np.array_equal(wk, step.work_host):
                raise RuntimeError("decode plan changed between steps")
        step.decode(q=dd["q"], tables=dd["tables"], lens=dd["lens"], k=dd["k"], v=dd["v"], slots=dd["slots"],
                    cow_src=dd["cow"] if (len(step.pairs) and step.fused) else None, out=o, work=dd.get("work"))

    # the flushes are not part of the step: e2e_pipelined subtracts each one's time
    e2e_ms, h2d = (e2e_pipelined(h, launch_decode, step.out, Ke, stream, flush_buf if flush else None) if Ke
                   else (0.0, h2d))
    e2e_bytes, e2e_s = aggregate(nbytes["total"] * Ke, max(e2e_ms, 1e-6) / 1e3)

    from paged_kv_cache_10_gb300 import pagedkv as pk
    assert pk.get_device_error() == 0, "device error word set during the benchmark"

    if rank != 0:
        return None
    clocks = sampler.summary(t_load0, t_load1) if sampler else None
    peak, peak_kind = measured_peaks()
    dec_ms = statistics.mean(decode_ms)
    # Where sequences share blocks the kernel need only read each distinct
    # byte once, so the roofline counts distinct bytes (logical bytes would
    # credit L2 hits or skipped re-reads as HBM bandwidth).
    shared = nbytes["unique_kv"] < nbytes["kv"]
    roof_bytes = nbytes["decode_unique"] if shared else nbytes["decode"]
    if step.fused:  # the timed decode launch also writes the step's new tokens and copy-on-write copies
        roof_bytes += nbytes["append"] + nbytes["copy"]
    achieved = roof_bytes / (dec_ms / 1e3) / 1e9
    kind = decode_kernel_kind(wl) if not cascade else "cascade"
    traffic = recorded_traffic(name, kind)  # the kind's source hash tells the cascade row from the plain one
    ms_per_step = total_ms / K
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "us_per_step": round(ms_per_step * 1e3, 2),
        "median_us_per_step": round(1e3 * statistics.median(a.elapsed_time(c) for a, _, c in ev), 2),
        "tokens_per_s": round(world * wl.S / (tot_s / K), 1),
        "pct_of_hbm_peak": round(100 * value / world / peak, 2),
        "pct_of_nominal_8tbs": round(100 * value / world / 8000.0, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"e4m3": "e4m3 KV, bf16 q"}.get(wl.kv_dtype, wl.kv_dtype) + ", fp32 accumulate",
        "data": "synthetic",
        "config": {
            "workload": wl.name, "num_seqs": wl.S, "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_size": wl.D,
            "block_size": wl.b, "kv_dtype": wl.kv_dtype, "num_blocks": wl.NB, "max_seq_len": step.max_seq_len,
            "mean_seq_len": float(step.seq_lens.mean()), "partition_tokens": step.effective_partition(),
            "cow_pairs": int(len(step.pairs)), "appended_tokens": int((step.slots >= 0).sum()),
            "decode": ("cascade: %d groups, prefix up to %d blocks" % (step.groups.num_groups, step.groups.max_blocks)
                       if step.cascade else "plain"),
            "bytes_per_step": nbytes, "l2": ("flushed between steps (2x L2 write)" if flush else
                                             f"inputs larger than L2 ({working_set / 2**20:.0f} MiB vs "
                                             f"{l2 / 2**20:.0f} MiB), no flush"),
            "parallelism": f"replicas x{world}",
            "launch": ("CUDA graph replay per step" if graph else "eager launches")
                      + ("; append fused into the decode kernel" if step.fused else ""),
            "cta_order": ("host plan, longest unit first" if step.work is not None else "grid order"),
        },
        "e2e": {"value": round(e2e_bytes / e2e_s / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": Ke, "copies": E2E_COPIES},
        "gpu_launches": K * step.kernel_launches(),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "frac_of_nominal_8tbs": round(achieved / 8000.0, 4),
                     "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": {"tensor_core": "decode_mma_kernel (+ merge when split)",
                                "cuda_core": "decode_kernel (+ merge when split)",
                                "cascade": "prefill_tc_kernel prefix pass + decode kernel + merge"}[kind]
                               + (", with the step's append fused in" if step.fused else ""),
                     "kernel_sources_hash": kernel_hash(kind),
                     "mean_launch_us": round(dec_ms * 1e3, 2),
                     "median_launch_us": round(statistics.median(decode_ms) * 1e3, 2),
                     "launch_timing": ("decode call replayed as a CUDA graph" if g is not None
                                       else "eager decode call inside the timed steps"),
                     "algorithmic_bytes_per_launch": roof_bytes,
                     "bytes_basis": ("distinct KV bytes (blocks shared between sequences counted once)" if shared
                                     else "KV bytes gathered through the block tables"),
                     "logical_gbs": round(nbytes["decode"] / (dec_ms / 1e3) / 1e9, 1)},
        "clocks": clocks,
        "kv_utilisation": kv_utilisation(step),
    }
    if world == 1 and oracle_leg and not (args.no_cpu_baseline or args.profile):
        line["parity"] = oracle_parity(step)
        line["cpu_baseline"] = cpu_baseline(wl, step, budget_s=cpu_budget, single_s=min(3.0, cpu_budget))
    del step, g
    torch.cuda.empty_cache()
    return line


def config_summary(line) -> dict:
    """The per-config fields of a workload's line."""
    r = line["roofline"]
    keep = ("us_per_step", "median_us_per_step", "tokens_per_s", "value", "unit", "pct_of_hbm_peak",
            "pct_of_nominal_8tbs", "dtype", "steps", "gpu_launches", "clocks", "kv_utilisation", "parity",
            "cpu_baseline")
    out = {k: line[k] for k in keep if k in line}
    out["kv_gbs"] = line["value"]
    out["e2e"] = {k: line["e2e"][k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step")}
    out["roofline"] = {k: r[k] for k in ("bound", "achieved", "peak", "unit", "frac", "frac_of_nominal_8tbs",
                                        "traffic", "mean_launch_us", "median_launch_us", "kernel", "bytes_basis",
                                        "logical_gbs", "algorithmic_bytes_per_launch")}
    c = line["config"]
    out["config"] = {k: c[k] for k in ("workload", "num_seqs", "q_heads", "kv_heads", "head_size", "kv_dtype",
                                       "mean_seq_len", "partition_tokens", "cow_pairs", "decode", "l2", "launch",
                                       "cta_order")}
    return out


def run_ours(args, rank, world, local_rank):
    sampler = ClockSampler(local_rank) if rank == 0 else None
    try:
        line = measure_decode(args, rank, world, local_rank, args.workload, args.cascade, args.graph,
                              sampler=sampler)
        if args.configs == "all" and world == 1:
            # every decode config timed in the same run (the headline's fields stay its own)
            configs = {}
            for name, casc, graph in DECODE_CONFIGS:
                key = name + ("_cascade" if casc else "")
                if (name, casc, graph) == (args.workload, args.cascade, args.graph):
                    configs[key] = config_summary(line)
                    continue
                ln = measure_decode(args, rank, world, local_rank, name, casc, graph,
                                    steps=min(args.steps, 100), sampler=sampler, cpu_budget=4.0)
                configs[key] = config_summary(ln)
            line["configs"] = configs
            line["next"] = measure_next(args, rank, world, local_rank, sampler=sampler)
    finally:
        if sampler:
            sampler.stop()
    return line


# ------------------------------------------------------------ prefill step
PREFILL_METRIC = "paged prefill attention TFLOP/s (causal, % of GB300 dense bf16 peak) and us/step, 1 GPU"


def prefill_flops(wl) -> float:
    """Algorithmic flops of causal attention for the step's new tokens: each
    row at position p does q.k and p.v over p + 1 keys, 4 * D flops per key
    and query head."""
    tot = 0
    for c, n in zip(wl.ctx, wl.qlens):
        tot += n * c + n * (n + 1) // 2  # sum over the chunk of (position + 1)
    return 4.0 * wl.D * wl.Hq * tot


def prefill_bytes(wl) -> int:
    """Least bytes the step must move: q and out, every key / value of each
    sequence once per KV head, the appended k / v (read in q's type, written
    in the pool's)."""
    e = 1 if wl.kv_dtype == "e4m3" else 2
    kv = sum(wl.seq_lens) * 2 * wl.Hkv * wl.D * e
    return 2 * wl.T * wl.Hq * wl.D * 2 + kv + wl.T * 2 * wl.Hkv * wl.D * (2 + e)


def measured_tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    return 1900.0, "fallback"


def oracle_prefill_host(wl):
    """Slots of the chunk's tokens, block tables and lengths of a prefill
    step from the oracle's own allocator model."""
    from oracle.allocator_model import AllocatorModel
    m = AllocatorModel(wl.NB, wl.b, wl.free_order)
    for s, c in enumerate(wl.ctx):
        m.seq_new(s, int(c))
    slots = []
    for s, n in enumerate(wl.qlens):
        for _ in range(int(n)):
            slots.append(m.append_slot(s)[0])
    tables = np.full((wl.S, wl.max_blocks), -1, np.int32)
    lens = np.zeros(wl.S, np.int32)
    for s in range(wl.S):
        t = m.block_table(s)
        tables[s, :len(t)] = t
        lens[s] = m.lens[s]
    return np.array(slots, np.int64), tables, lens


def prefill_cpu_baseline(wl, budget_s=10.0):
    """The float64 oracle on the first tokens of each chunk in turn (all
    heads, each with every key it sees), about budget_s of CPU time."""
    import oracle
    slots, tables, lens = oracle_prefill_host(wl)
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.append(wl.k_new, wl.v_new, wl.dtype, slots, kp, vp, wl.kv_dtype, wl.k_scale, wl.v_scale)
    qs = np.concatenate([[0], np.cumsum(wl.qlens)]).astype(np.int64)
    m, flops, dt, reps = 8, 0.0, 0.0, 0
    while dt < budget_s and reps < 10000:
        s = reps % wl.S
        n = min(m, wl.qlens[s])
        if n == 0:
            reps += 1
            continue
        ctx = int(lens[s]) - wl.qlens[s]
        q = np.ascontiguousarray(wl.q[qs[s]:qs[s] + n])
        t = time.perf_counter()
        oracle.paged_prefill(q, wl.dtype, np.array([0, n], np.int32), kp, vp, wl.kv_dtype, tables[s:s + 1],
                             np.array([ctx + n], np.int32), wl.scale, wl.k_scale, wl.v_scale)
        dt += time.perf_counter() - t
        flops += 4.0 * wl.D * wl.Hq * (n * ctx + n * (n + 1) // 2)
        if reps == 0 and dt < budget_s / 50:
            m = min(4096, m * 4)
        reps += 1
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{reps} chunk heads of {wl.name} (first <= {m} tokens of a chunk, all heads, every key "
                      f"they see): float64 causal attention, {dt:.1f} s"}


def run_prefill(args, rank, world, local_rank):
    sampler = ClockSampler(local_rank) if rank == 0 else None
    try:
        return measure_prefill(args, rank, world, local_rank, args.workload, sampler=sampler)
    finally:
        if sampler:
            sampler.stop()


def measure_prefill(args, rank, world, local_rank, name, steps=None, sampler=None, cpu_budget=10.0):
    """Times one prefill workload (K device-timed steps, the attention call,
    the e2e loop) and, on rank 0 of a single-GPU run, the oracle leg.
    Returns the JSON line of the workload (rank 0) or None."""
    from paged_kv_cache_10_gb300 import pagedkv as pk
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import PrefillStep

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = workloads.PREFILL[name]()
    step = PrefillStep(wl, device=dev, plan=not args.no_plan)
    flops = prefill_flops(wl)
    nbytes = prefill_bytes(wl)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = nbytes < 4 * l2
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev) if flush else None
    for _ in range(max(args.warmup, 3)):
        step.run()
    torch.cuda.synchronize()
    K = steps or args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    t_load0 = time.monotonic()
    for i in range(K):
        if flush:
            flush_buf.zero_()
        ev[i][0].record(stream)
        step.append()
        ev[i][1].record(stream)
        step.attend()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    t_load1 = time.monotonic()
    barrier()
    total_ms = sum(a.elapsed_time(c) for a, _, c in ev)
    attn_ms = [b.elapsed_time(c) for _, b, c in ev]
    if sampler and not args.profile and t_load1 - t_load0 < 1.0:
        t_ext = time.monotonic()
        while time.monotonic() - t_ext < 1.5:
            for _ in range(20):
                step.run()
            torch.cuda.synchronize()
        t_load1 = time.monotonic()
    tot_flops, tot_s = aggregate(flops * K, total_ms / 1e3)
    value = tot_flops / tot_s / 1e12

    # end to end through the public API: inputs from pinned host memory, output back
    h = {"q": step.q.cpu().pin_memory(), "k": step.k_new.cpu().pin_memory(), "v": step.v_new.cpu().pin_memory(),
         "slots": step.d_slots.cpu().pin_memory(), "tables": step.d_tables.cpu().pin_memory(),
         "lens": step.d_lens.cpu().pin_memory(), "qs": step.d_query_start.cpu().pin_memory()}
    if step.work is not None:  # the host plan, rebuilt from the host arrays every step
        h["work"] = torch.from_numpy(step.work_host.copy()).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = step.out.numel() * step.out.element_size()
    Ke = 0 if args.profile else max(1, min(K, 100))
    barrier()

    def launch_prefill(dd, o):
        if "work" in dd:  # planning is host work of the step; the batch (so the plan) never changes here
            wk = pk.prefill_plan(step.query_start, step.seq_lens, wl.Hq, wl.Hkv, wl.max_query_len)
            if not np.array_equal(wk, step.work_host):
                raise RuntimeError("prefill plan changed between steps")
        pk.paged_kv_append(dd["k"], dd["v"], dd["slots"], step.k_cache, step.v_cache, step.desc, in_dtype=wl.dtype)
        pk.paged_attention_prefill(dd["q"], step.k_cache, step.v_cache, step.desc, dd["qs"], wl.max_query_len,
                                   dd["tables"], dd["lens"], wl.scale, o, q_dtype=wl.dtype,
                                   work_units=dd.get("work"), workspace=step.workspace)

    e2e_ms, h2d = (e2e_pipelined(h, launch_prefill, step.out, Ke, stream, flush_buf if flush else None) if Ke
                   else (0.0, h2d))
    e2e_flops, e2e_s = aggregate(flops * Ke, max(e2e_ms, 1e-6) / 1e3)
    assert pk.get_device_error() == 0, "device error word set during the benchmark"
    if rank != 0:
        return None
    clocks = sampler.summary(t_load0, t_load1) if sampler else None
    peak, peak_kind = measured_tensor_peak()
    a_ms = statistics.mean(attn_ms)
    achieved = flops / (a_ms / 1e3) / 1e12
    line = {
        "metric": PREFILL_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_ms / K, 5), "us_per_step": round(1e3 * total_ms / K, 2),
        "median_us_per_step": round(1e3 * statistics.median(a.elapsed_time(c) for a, _, c in ev), 2),
        "tokens_per_s": round(world * wl.T / (tot_s / K), 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": (f"e4m3 KV, {wl.dtype} q" if wl.kv_dtype == "e4m3" else wl.dtype) + ", fp32 accumulate",
        "data": "synthetic",
        "config": {"workload": wl.name, "num_seqs": wl.S, "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_size": wl.D,
                   "kv_dtype": wl.kv_dtype, "new_tokens": wl.T, "chunk_tokens": wl.qlens, "context_tokens": wl.ctx, "num_blocks": wl.NB,
                   "flops_per_step": flops, "min_bytes_per_step": nbytes,
                   "l2": ("flushed between steps (2x L2 write)" if flush else "inputs larger than L2, no flush"),
                   "cta_order": ("host plan, longest causal key range first" if step.work is not None
                                 else "grid order"),
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": round(e2e_flops / e2e_s / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": Ke, "copies": E2E_COPIES},
        "gpu_launches": K * step.kernel_launches(),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": recorded_traffic(wl.name, "prefill"),
                     "peak_kind": peak_kind,
                     "kernel": ("stage_fp8_kernel + prefill_tc_kernel (timed together)" if step.workspace is not None
                                else "prefill_tc_kernel"),
                     "kernel_sources_hash": kernel_hash("prefill"), "mean_launch_us": round(a_ms * 1e3, 2),
                     "median_launch_us": round(statistics.median(attn_ms) * 1e3, 2),
                     "algorithmic_flops_per_launch": flops,
                     "hbm_gbs_at_min_bytes": round(nbytes / (a_ms / 1e3) / 1e9, 1)},
        "clocks": clocks,
    }
    if world == 1 and not (args.no_cpu_baseline or args.profile):
        line["parity"] = prefill_parity(step)
        line["cpu_baseline"] = prefill_cpu_baseline(wl, budget_s=cpu_budget)
    del step
    torch.cuda.empty_cache()
    return line


def prefill_summary(line) -> dict:
    """The per-workload fields of a prefill line."""
    r = line["roofline"]
    keep = ("metric", "us_per_step", "median_us_per_step", "tokens_per_s", "value", "unit", "dtype", "steps",
            "gpu_launches", "clocks", "parity", "cpu_baseline")
    out = {k: line[k] for k in keep if k in line}
    out["e2e"] = {k: line["e2e"][k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step")}
    out["roofline"] = {k: r[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic", "peak_kind",
                                        "kernel", "mean_launch_us", "median_launch_us",
                                        "algorithmic_flops_per_launch")}
    c = line["config"]
    out["config"] = {k: c[k] for k in ("workload", "num_seqs", "q_heads", "kv_heads", "head_size", "kv_dtype",
                                       "new_tokens", "l2", "cta_order")}
    return out


# the rows beyond the decode configs that the default run also measures
NEXT_PREFILL = ("prefill_chunked_gqa", "prefill_chunked_gqa_fp8")


def measure_next(args, rank, world, local_rank, sampler=None) -> dict:
    """Chunked prefill over a bf16 and an fp8 pool (device-timed, with e2e,
    sampled oracle parity and the oracle's timing), the host prefix cache on
    a request stream, and block swap to and from a pinned host pool."""
    out = {}
    for name in NEXT_PREFILL:
        ln = measure_prefill(args, rank, world, local_rank, name, steps=min(args.steps, 50), sampler=sampler,
                             cpu_budget=4.0)
        out[name] = prefill_summary(ln)
    out["prefix_cache_host"] = run_apc(argparse.Namespace(steps=50))
    out["swap_blocks"] = run_swap(argparse.Namespace(workload="llama3_8b_gqa", steps=20, warmup=3), local_rank)
    return out


# ------------------------------------------- prefill per-unit cost sweep
def run_prefill_unit_sweep(args, local_rank):
    """Separates the prefill kernel's cost per key tile from its fixed cost
    per unit: batches of equal units (each sequence appends 64 tokens, 32/8
    heads, D 128, bf16, so one unit per (sequence, KV head)) with 0, 1024 or
    3072 tokens of context (1, 9 or 25 key tiles per unit), sized to 2 and 4
    units per SM; times the attention call with CUDA events.  A linear fit of
    time per unit round against key tiles gives both costs."""
    import numpy as np
    from paged_kv_cache_10_gb300 import pagedkv as pk
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import PrefillStep
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    points = []
    for rounds in (2, 4):
        S = sms * rounds // 8
        for ctx in (0, 1024, 3072):
            wl = workloads.prefill(f"unit_sweep_{ctx}", 5000 + ctx, [ctx] * S, [64] * S, 32, 8)
            st = PrefillStep(wl, device=dev)
            st.run()
            for _ in range(max(args.warmup, 3)):
                st.attend()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(args.steps, 10)
            e0.record()
            for _ in range(reps):
                st.attend()
            e1.record()
            torch.cuda.synchronize()
            assert pk.get_device_error() == 0, "device error word set during the sweep"
            us = e0.elapsed_time(e1) * 1e3 / reps
            tiles = -(-(ctx + 64) // 128)
            points.append({"rounds": rounds, "context": ctx, "key_tiles": tiles, "us": round(us, 2),
                           "us_per_round": round(us / rounds, 2)})
            del st
            torch.cuda.empty_cache()
    big = [q for q in points if q["rounds"] == 4]
    slope, icpt = np.polyfit([q["key_tiles"] for q in big], [q["us_per_round"] for q in big], 1)
    return {"metric": "prefill cost per unit round (equal units)", "unit": "us", "points": points,
            "fit_4_rounds": {"us_per_key_tile": round(float(slope), 3), "us_per_unit": round(float(icpt), 2)},
            "sms": sms}


def prefill_parity(step, per_seq=8) -> dict:
    """Untimed: the step's host bookkeeping and pools against the oracle's
    own allocator model and append, and the first and last ``per_seq`` new
    tokens of every chunk (all heads, every key each sees) against the
    float64 oracle."""
    import oracle
    wl = step.wl
    t0 = time.perf_counter()
    slots, tables, lens = oracle_prefill_host(wl)
    host_ok = (np.array_equal(step.slots, slots) and np.array_equal(step.tables, tables)
               and np.array_equal(step.seq_lens, lens))
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.append(wl.k_new, wl.v_new, wl.dtype, slots, kp, vp, wl.kv_dtype, wl.k_scale, wl.v_scale)
    pools_ok = bool(np.array_equal(_host_bits(step.k_cache), kp) and np.array_equal(_host_bits(step.v_cache), vp))
    got_all = oracle.dequantize(_host_bits(step.out), wl.dtype)
    tol = TOL[wl.kv_dtype]
    vmax = float(np.max(np.abs(oracle.dequantize(vp, wl.kv_dtype)))) * (wl.v_scale if wl.kv_dtype == "e4m3" else 1.0)
    qs = step.query_start
    err_max = ref_max = 0.0
    over = -tol
    tokens = 0
    finite = True
    for s in range(wl.S):
        n = int(wl.qlens[s])
        ctx = int(lens[s]) - n
        spans = sorted({(0, min(per_seq, n)), (max(0, n - per_seq), n)})
        for a, b in spans:
            if b <= a:
                continue
            # the oracle takes the rows as the last b - a tokens of a sequence of ctx + b
            ref = oracle.paged_prefill(np.ascontiguousarray(wl.q[qs[s] + a:qs[s] + b]), wl.dtype,
                                       np.array([0, b - a], np.int32), kp, vp, wl.kv_dtype, tables[s:s + 1],
                                       np.array([ctx + b], np.int32), wl.scale, wl.k_scale, wl.v_scale)
            got = got_all[qs[s] + a:qs[s] + b]
            err = np.abs(got - ref)
            finite = finite and bool(np.all(np.isfinite(got)))
            err_max = max(err_max, float(err.max()))
            ref_max = max(ref_max, float(np.abs(ref).max()))
            over = max(over, float(np.max(err - error_bound(ref, wl.dtype, tol, vmax))))
            tokens += b - a
    return {"tokens": tokens, "of_tokens": int(wl.T), "max_abs_err": err_max, "max_abs_oracle": ref_max, "tol": tol,
            "within_tolerance": bool(over <= 0 and finite), "max_err_minus_bound": over,
            "pools_bit_exact": pools_ok, "host_bookkeeping_exact": bool(host_ok),
            "oracle_s": round(time.perf_counter() - t0, 2),
            "basis": f"first and last {per_seq} new tokens of every chunk (all heads) against the float64 oracle "
                     "(every token at full size in the GPU tests); bound as for the decode"}


# ------------------------------------------------------ prefix-cache timing
def run_apc(args):
    """Host-side automatic prefix caching on a request stream: 16 system
    prompts of 2048 tokens, each request one of them plus U[64, 1024] own
    tokens; per request: block hashes, lookup + touch + allocation,
    commit of its full blocks, release.  Times the library's C++ allocator
    and reports the share of full blocks served from the cache."""
    from paged_kv_cache_10_gb300 import pagedkv as pk
    rng = np.random.default_rng(2024)
    systems = [rng.integers(0, 128000, size=2048).astype(np.int32) for _ in range(16)]
    reqs = []
    for _ in range(max(args.steps, 1) * 20):
        own = rng.integers(0, 128000, size=int(rng.integers(64, 1024, endpoint=True))).astype(np.int32)
        reqs.append(np.concatenate([systems[int(rng.integers(0, 16))], own]))
    NB = 40000
    a = pk.Allocator(NB, 16)
    live = []
    hits = blocks = 0

    def one(i, t):
        nonlocal hits, blocks
        h = pk.prefix_block_hashes(t)
        hits += a.seq_new_prefix(i, h, len(t))
        blocks += len(h)
        a.commit(i, h)
        live.append(i)
        if len(live) > 64:  # 64 requests in flight; the oldest finishes
            a.free(live.pop(0))

    for i, t in enumerate(reqs[:50]):
        one(i, t)
    hits = blocks = 0
    t0 = time.perf_counter()
    for i, t in enumerate(reqs[50:], start=50):
        one(i, t)
    dt = time.perf_counter() - t0
    n = len(reqs) - 50
    toks = sum(len(t) for t in reqs[50:])
    return {"metric": "automatic prefix caching, host allocator (hash + lookup + touch + allocate + commit + free)",
            "value": round(n / dt, 1), "unit": "requests/s", "us_per_request": round(1e6 * dt / n, 2),
            "blocks_per_s": round(blocks / dt, 1), "tokens_per_s": round(toks / dt, 1),
            "cached_block_fraction": round(hits / max(blocks, 1), 4), "requests": n, "cores": 1,
            "config": {"system_prompts": 16, "system_tokens": 2048, "own_tokens": "U[64,1024]",
                       "in_flight": 64, "num_blocks": NB}}


# ------------------------------------------------------------ swap timing
def run_swap(args, local_rank):
    """Times pkv_swap_blocks on the workload's pool: all blocks of the first
    half of the batch out to a pinned host pool and back (CUDA events)."""
    from paged_kv_cache_10_gb300 import pagedkv as pk
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = workloads.NAMED[args.workload]()
    st = DecodeStep(wl, device=dev)
    rows = list(range(max(1, wl.S // 2)))
    blocks = sorted({b for r in rows for b in st.alloc.block_table(r)})
    n = len(blocks)
    pairs = torch.tensor([[b, i] for i, b in enumerate(blocks)], dtype=torch.int32, device=dev)
    shape = (n,) + tuple(st.k_cache.shape[1:])
    k_host = torch.empty(shape, dtype=st.k_cache.dtype).pin_memory()
    v_host = torch.empty(shape, dtype=st.v_cache.dtype).pin_memory()
    nbytes = 2 * n * st.k_cache[0].numel() * st.k_cache.element_size()
    res = {}
    for name, direction in (("device_to_host", pk.SWAP_OUT), ("host_to_device", pk.SWAP_IN)):
        for _ in range(max(args.warmup, 3)):
            pk.swap_blocks(st.k_cache, st.v_cache, st.desc, k_host, v_host, pairs, direction)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            pk.swap_blocks(st.k_cache, st.v_cache, st.desc, k_host, v_host, pairs, direction)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
        res[name] = {"us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms / 1e3) / 1e9, 1)}
    assert pk.get_device_error() == 0
    return {"metric": "KV block swap bandwidth (pkv_swap_blocks, pinned mapped host pool)", "unit": "GB/s",
            "workload": wl.name, "blocks": n, "bytes_per_swap": nbytes, "steps": args.steps, **res}


# ----------------------------------------------------------- reference arm
def run_reference_prefill(args, wl):
    """The oracle as the reference arm of a prefill workload: per step, the
    float64 causal attention of the first tokens of one chunk (all heads,
    every key they see), rotating through the sequences."""
    import oracle
    slots, tables, lens = oracle_prefill_host(wl)
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.append(wl.k_new, wl.v_new, wl.dtype, slots, kp, vp, wl.kv_dtype, wl.k_scale, wl.v_scale)
    qs = np.concatenate([[0], np.cumsum(wl.qlens)]).astype(np.int64)
    m = 4

    def one(i):
        s = i % wl.S
        n = min(m, wl.qlens[s])
        ctx = int(lens[s]) - wl.qlens[s]
        oracle.paged_prefill(np.ascontiguousarray(wl.q[qs[s]:qs[s] + n]), wl.dtype, np.array([0, n], np.int32), kp, vp,
                             wl.kv_dtype, tables[s:s + 1], np.array([ctx + n], np.int32), wl.scale,
                             wl.k_scale, wl.v_scale)
        return 4.0 * wl.D * wl.Hq * (n * ctx + n * (n + 1) // 2)

    K, W = args.steps, args.warmup
    for i in range(W):
        one(i)
    flops, t = 0.0, 0.0
    for i in range(K):
        t0 = time.perf_counter()
        flops += one(W + i)
        t += time.perf_counter() - t0
    value = flops / t / 1e12
    return {
        "impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": K, "warmup": W, "ms_per_step": round(1e3 * t / K, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "num_seqs": wl.S, "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_size": wl.D,
                   "kv_dtype": wl.kv_dtype},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"the first {m} tokens of one chunk of {wl.name} per step (all heads), rotating: "
                                   f"float64 causal attention"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    from paged_kv_cache_10_gb300 import workloads

    oracle.build()
    if args.workload in workloads.PREFILL:
        return run_reference_prefill(args, workloads.PREFILL[args.workload]())
    wl = workloads.NAMED[args.workload]()
    # the host bookkeeping of the step from the oracle's allocator model
    st = HostStep(wl, *oracle_host_step(wl))
    pools = (wl.k_pool.copy(), wl.v_pool.copy())
    K, W = args.steps, args.warmup
    # one sequence (all heads) per step, rotating through the batch
    for i in range(W):
        oracle_rows_step(wl, st, np.array([i % wl.S]), pools)
    nbytes, t = 0, 0.0
    for i in range(K):
        rows = np.array([(W + i) % wl.S])
        t0 = time.perf_counter()
        oracle_rows_step(wl, st, rows, pools)
        t += time.perf_counter() - t0
        nbytes += rows_bytes(st, rows)
    value = nbytes / t / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(1e3 * t / K, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "num_seqs": wl.S, "q_heads": wl.Hq, "kv_heads": wl.Hkv,
                   "head_size": wl.D, "kv_dtype": wl.kv_dtype},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"one sequence of {wl.name} (all heads) per step, rotating: its append + "
                                   f"float64 decode"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--partition", type=int, default=None, help="tokens per split-K partition (0 = auto)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--apc", action="store_true",
                    help="time host-side automatic prefix caching on a request stream (no GPU work)")
    ap.add_argument("--swap", action="store_true",
                    help="time block swap to / from a pinned host pool instead of the decode step")
    ap.add_argument("--graph", action="store_true",
                    help="time steps as CUDA-graph replays (one launch per step)")
    ap.add_argument("--unfused", action="store_true",
                    help="append with its own kernel before the decode (default: fused into the decode kernel)")
    ap.add_argument("--cascade", action="store_true",
                    help="shared-prefix decode: blocks shared by a group of sequences are read once per group")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle leg (cpu_baseline timing and the untimed parity check)")
    ap.add_argument("--configs", choices=["all", "none"], default=None,
                    help="also time every decode config in the same run and report each under 'configs', "
                         "and the chunked prefill, prefix cache and block swap under 'next' "
                         "(default: all for the default workload on one GPU, none otherwise)")
    ap.add_argument("--decode-plan", choices=["auto", "on", "off"], default="auto",
                    help="decode: CTAs in the host plan's longest-first order (auto: when unit lengths differ "
                         "and no blocks are shared)")
    ap.add_argument("--no-plan", action="store_true",
                    help="prefill: CTAs in grid order instead of the host plan's longest-first order")
    ap.add_argument("--prefill-unit-sweep", action="store_true",
                    help="prefill kernel cost per key tile and per unit, from batches of equal units")
    ap.add_argument("--profile", action="store_true",
                    help="timed steps only (no e2e loop, clock-window extension or CPU baseline): for ncu runs")
    args = ap.parse_args(argv)

    if args.configs is None:
        args.configs = ("all" if (args.workload == DEFAULT_WORKLOAD and not args.cascade and not args.graph
                                  and not args.profile and args.partition is None) else "none")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.apc:
        line = run_apc(args) if rank == 0 else None
    elif args.swap:
        line = run_swap(args, local_rank) if rank == 0 else None
    elif args.prefill_unit_sweep:
        line = run_prefill_unit_sweep(args, local_rank) if rank == 0 else None
    elif args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        from paged_kv_cache_10_gb300 import workloads
        if args.workload in workloads.PREFILL:
            line = run_prefill(args, rank, world, local_rank)
        else:
            line = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
