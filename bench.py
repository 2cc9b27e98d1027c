"""Benchmark of the fused attention forward pass on GB300 (sm_103a).

One step = one call of the whole hot path on one batch of synthetic input
(for the BF16 workloads: the fused forward kernel; for the FP8 workload: the
prep of Q, K, V (one launch) plus the FP8 forward).  Default workload: BF16,
non-causal, B=4, H=16, Nq=Nk=4096, d=128, scale 1/sqrt(128).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

Prints one JSON line (rank 0).  Timing: W untimed warm-up steps, then K steps
bracketed by a barrier and torch.cuda.synchronize() on both sides, CUDA
events on the launching stream, max over ranks.  The working set (Q, K, V, O)
is larger than the 129 MB L2, so no extra flush is made between steps.
N > 1 (torchrun, one rank per GPU) runs N independent replicas of the same
workload: the path has no exchange step, so there is no collective on the
data path (weak scaling).
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOADS = {
    # name: (B, Hq, Hkv, Nq, Nk, d, causal, kind)
    "bf16_mha_B4_H16_N4096_d128": (4, 16, 16, 4096, 4096, 128, False, "bf16"),
    "bf16_mha_B4_H16_N4096_d64": (4, 16, 16, 4096, 4096, 64, False, "bf16"),
    "bf16_mha_B4_H16_N4096_d256": (4, 16, 16, 4096, 4096, 256, False, "bf16"),
    "bf16_causal_gqa_B1_Hq64_Hkv8_N32768_d128": (1, 64, 8, 32768, 32768, 128, True, "bf16"),
    "bf16_causal_gqa_B1_Hq64_Hkv8_N131072_d128": (1, 64, 8, 131072, 131072, 128, True, "bf16"),
    "fp8_e4m3_B4_H16_N4096_d128": (4, 16, 16, 4096, 4096, 128, False, "fp8"),
    "fp8_e4m3_hadamard_B4_H16_N4096_d128": (4, 16, 16, 4096, 4096, 128, False, "fp8h"),
    "fp8_e4m3_B4_H16_N4096_d64": (4, 16, 16, 4096, 4096, 64, False, "fp8"),
    "fp8_e4m3_B4_H16_N4096_d256": (4, 16, 16, 4096, 4096, 256, False, "fp8"),
    "fp8_e4m3_causal_gqa_B1_Hq64_Hkv8_N32768_d128": (1, 64, 8, 32768, 32768, 128, True, "fp8"),
    # rotary embedding fused into the Q / K prep (tables built once, outside the steps)
    "fp8_e4m3_rope_hadamard_B4_H16_N4096_d128": (4, 16, 16, 4096, 4096, 128, False, "fp8hr"),
    # one query per head against a long key cache: split key ranges + LSE merge
    "bf16_decode_splitkv_B1_Hq64_Hkv8_Nq1_Nk131072_d128": (1, 64, 8, 1, 131072, 128, False,
                                                          "decode"),
    # a batch of sequences, one new query each, against 8192 cached keys
    "bf16_decode_batched_B32_Hq64_Hkv8_Nq1_Nk8192_d128": (32, 64, 8, 1, 8192, 128, False,
                                                          "decode"),
}
DEFAULT_WORKLOAD = "bf16_mha_B4_H16_N4096_d128"
METRIC = "attention fwd TFLOPS (BF16, FP8) at 1 GB300 and % of dense tensor-core peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def attention_flops(B, Hq, Nq, Nk, d, causal):
    """Algorithmic FLOPs: Q K^T and P V, 2 flops per multiply-add, 4*d per
    score; the causal mask halves the count."""
    f = 4.0 * B * Hq * Nq * Nk * d
    return f / 2 if causal else f


# CUDA sources each timed kernel is built from (its launch set-up included)
FWD_SOURCES = ("attn_fwd_kernel.cuh", "fwd_launch.cuh", "ptx.cuh", "internal.h", "api.cu",
               "attn_fwd_f16.cu", "attn_fwd_bf16.cu", "attn_fwd_e4m3.cu")
MERGE_SOURCES = FWD_SOURCES + ("splitkv_merge.cu",)


def kernel_source_hash(names=FWD_SOURCES) -> str:
    """Hash of the CUDA sources of a kernel: ncu counters taken on other
    sources are stale."""
    csrc = os.path.join(ROOT, "tiled_attention_forward_02_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(names):
        path = os.path.join(csrc, name)
        if os.path.exists(path):
            with open(path, "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    e = rec.get(f"{kernel}|{workload}")
    names = MERGE_SOURCES if "merge" in kernel else FWD_SOURCES
    if not e or e.get("source_hash") != kernel_source_hash(names):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5:
            time.sleep(0.05)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1]
        if not rows:
            rows = [s for (_, s) in self.samples]
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            parts = [x.strip() for x in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ distributed
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- CPU oracle
class OracleSampler:
    """Times the FP64 oracle (as it stands, never tuned for this) on bounded
    samples of query rows of a workload, on this host's cores."""

    def __init__(self, workload):
        import numpy as np
        import torch

        import oracle
        import synth
        B, Hq, Hkv, Nq, Nk, d, causal, kind = WORKLOADS[workload]
        self.Hq, self.Nq, self.Nk, self.d, self.causal = Hq, Nq, Nk, d, causal
        # keys/values of batch element 0 only (the oracle decodes them in full per call)
        q, k, v = synth.attn_inputs(1, Nq, Nk, Hq, Hkv, d, dtype=torch.bfloat16, seed=0,
                                    outlier_frac=1e-3 if kind.startswith("fp8") else 0.0)
        self.q, self.kb, self.vb = q, synth.raw_bits(k), synth.raw_bits(v)
        self.threads = oracle.default_threads()
        self.rng = np.random.default_rng(0)
        self._np, self._oracle, self._synth = np, oracle, synth

    def rows(self, n):
        np = self._np
        idx = self.rng.integers(0, self.Hq * self.Nq, size=n)
        return np.stack([np.zeros(n, np.int64), idx % self.Hq, idx // self.Hq],
                        axis=1).astype(np.int64)

    def flops(self, rows):
        np = self._np
        keys = np.minimum(rows[:, 2] + 1, self.Nk) if self.causal else np.full(len(rows), self.Nk)
        return float(np.sum(4.0 * keys * self.d))

    def run(self, rows):
        qr = self._synth.raw_bits(self.q[0, rows[:, 2], rows[:, 1]])
        t0 = time.perf_counter()
        self._oracle.attention_rows(qr, self.kb, self.vb, Hq=self.Hq, causal=self.causal,
                                    scale=1 / math.sqrt(self.d), rows=rows,
                                    elem=self._oracle.ELEM_BF16, nthreads=self.threads)
        return time.perf_counter() - t0

    def rows_for(self, seconds):
        """Rows that take about `seconds`: after one warm-up call (the first
        call also pages in the decoded keys and values), the sample doubles
        until one call takes at least 0.25 s, and the count scales linearly
        from that call (its fixed cost included, so the estimate errs short).
        Bounded: at most 48 times the calibrated sample."""
        self.run(self.rows(self.threads))
        n = self.threads * 4
        while True:
            t = self.run(self.rows(n))
            if t >= 0.25 or n >= (1 << 22):
                break
            n *= 2
        return max(self.threads, min(int(n * seconds / max(t, 1e-3)), 48 * n))


def time_oracle(workload, budget_s=12.0):
    """(TFLOPS-equivalent, rows, seconds, threads) of one bounded oracle sample."""
    s = OracleSampler(workload)
    rows = s.rows(s.rows_for(budget_s))
    t = s.run(rows)
    return s.flops(rows) / t / 1e12, len(rows), t, s.threads


def reference_arm(args, rank, world):
    """--impl reference: the oracle timed on host cores (rank 0 only); every
    step is a bounded sample sized so that the whole run takes about two
    minutes whatever K and W are."""
    if rank != 0:
        return
    wl = args.workload
    s = OracleSampler(wl)
    per_step_s = max(0.02, 120.0 / (args.steps + args.warmup))
    n = s.rows_for(per_step_s)
    flops_total, secs_total = 0.0, 0.0
    for i in range(args.warmup + args.steps):
        rows = s.rows(n)
        t = s.run(rows)
        if i >= args.warmup:
            flops_total += s.flops(rows)
            secs_total += t
    value = flops_total / secs_total / 1e12
    sample = (f"{n} random query rows of batch 0 per step, {args.steps} steps, "
              f"{secs_total:.1f} s of FP64 oracle time; TFLOPS-equivalent = 4*keys*d per row")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs_total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": s.threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(wl):
    B, Hq, Hkv, Nq, Nk, d, causal, kind = WORKLOADS[wl]
    return {"workload": wl, "B": B, "Hq": Hq, "Hkv": Hkv, "Nq": Nq, "Nk": Nk, "d": d,
            "causal": causal, "scale": "1/sqrt(d)", "parallelism": "replicas",
            "l2": "inputs larger than L2 (Q+K+V+O > 129 MB), no flush between steps",
            "inputs": "iid N(0,1) BSHD, seed 0" + (", 0.1% outliers x50"
                                                  if kind.startswith("fp8") else ""),
            "prep": {"fp8": "per-block E4M3", "fp8h": "Hadamard + per-block E4M3",
                     "fp8hr": "rotary (rotate-half, base 10000) + Hadamard + per-block E4M3 "
                              "on Q and K in one pass"}.get(kind, "none")}


# ------------------------------------------------------------------ GPU arm
def make_step(wl, dev):
    """Return (step_fn, hot_fn, meta) for the workload; inputs resident.

    hot_fn(q, k, v, o, lse) runs the whole path on the given device buffers
    (the end-to-end leg alternates two buffer sets); step_fn runs it on the
    resident set, with CUDA events around the dominant kernel when asked."""
    import torch

    import synth
    from tiled_attention_forward_02_gb300 import attn
    B, Hq, Hkv, Nq, Nk, d, causal, kind = WORKLOADS[wl]
    scale = 1.0 / math.sqrt(d)
    outl = 1e-3 if kind.startswith("fp8") else 0.0
    q, k, v = synth.attn_inputs(B, Nq, Nk, Hq, Hkv, d, dtype=torch.bfloat16, seed=0, device=dev,
                                outlier_frac=outl)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    meta = {"flops": attention_flops(B, Hq, Nq, Nk, d, causal), "kernel": "attn_fwd_kernel"}
    # pinned host copies for the end-to-end leg
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    meta["h2d"] = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    meta["d2h"] = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    meta["host"] = (hq, hk, hv, ho, hl)
    meta["device"] = (q, k, v, o, lse)

    if kind == "decode":
        splits = attn.splitkv_default_splits(B, Hq, Hkv, Nq, Nk, d)
        ws = torch.empty(attn.splitkv_workspace_bytes(B, Hq, Nq, d, splits), dtype=torch.uint8,
                         device=dev)

        def hot(q, k, v, o, lse):
            attn.attn_fwd_splitkv(q, k, v, num_splits=splits, scale=scale, out=o, lse=lse,
                                  workspace=ws)

        def step(kernel_events=None):
            if kernel_events:
                kernel_events[0].record()
            hot(q, k, v, o, lse)
            if kernel_events:
                kernel_events[1].record()
        rows = splits * B * Hq * Nq if splits > 1 else 0
        # K and V once, Q, O, LSE, and (with several splits) the FP32 partial
        # rows written and read back
        meta["bytes"] = (2 * B * Nk * Hkv * d * 2 + 2 * B * Nq * Hq * d * 2 + B * Hq * Nq * 4
                         + 2 * rows * (d + 1) * 4)
        meta["launches_per_step"] = 2 if splits > 1 else 1
        meta["kernel"] = (f"attn_fwd_kernel<split> + splitkv_merge ({splits} splits)" if splits > 1
                          else "attn_fwd_kernel<split> (GQA group packed, one split)")
        return step, hot, meta

    if kind == "bf16":
        def hot(q, k, v, o, lse):
            attn.attn_fwd(q, k, v, causal=causal, scale=scale, out=o, lse=lse)

        def step(kernel_events=None):
            if kernel_events:
                kernel_events[0].record()
            hot(q, k, v, o, lse)
            if kernel_events:
                kernel_events[1].record()
        meta["launches_per_step"] = 1
        return step, hot, meta

    had = kind in ("fp8h", "fp8hr")
    rope = kind == "fp8hr"
    signs = synth.hadamard_signs(Hkv, d, seed=0).to(dev) if had else None
    if rope:
        # one table for Q and K (Nq == Nk here), built on the device once
        assert Nq == Nk
        rcos, rsin = attn.attn_rope_table(Nk, d, device=dev)
    npad = (Nk + 15) // 16 * 16
    q8 = torch.empty((B, Nq, Hq, d), dtype=torch.uint8, device=dev)
    k8 = torch.empty((B, Nk, Hkv, d), dtype=torch.uint8, device=dev)
    v8 = torch.empty((B, Hkv, d, npad), dtype=torch.uint8, device=dev)
    qd = torch.empty((B, Hq, (Nq + 127) // 128), dtype=torch.float32, device=dev)
    kd = torch.empty((B, Hkv, (Nk + 127) // 128), dtype=torch.float32, device=dev)
    vd = torch.empty_like(kd)

    prep_ev = []   # (start, end) events around the three prep calls of each timed step

    def hot(q, k, v, o, lse, kernel_events=None):
        if kernel_events:
            pe = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            pe[0].record()
        # Q, K (rotated and / or transformed) and V (transposed) in one launch
        attn.attn_prep_fp8_qkv(q, k, v, signs=signs, rope=(rcos, rsin) if rope else None,
                               out=(q8, qd, k8, kd, v8, vd))
        if kernel_events:
            pe[1].record()
            prep_ev.append(pe)
        if kernel_events:
            kernel_events[0].record()
        attn.attn_fwd_fp8(q8, k8, v8, qd, kd, vd, causal=causal, scale=scale, hadamard=had,
                          out=o, lse=lse)
        if kernel_events:
            kernel_events[1].record()

    def step(kernel_events=None):
        hot(q, k, v, o, lse, kernel_events)
    meta["launches_per_step"] = 2
    meta["kernel"] = "attn_fwd_kernel<e4m3>"
    meta["prep_events"] = prep_ev
    # prep: every bf16 element read once, one E4M3 byte written, one descale per block
    meta["prep_bytes"] = sum(t.numel() * 3 for t in (q, k, v)) + 4 * (qd.numel() + 2 * kd.numel())
    if rope:
        # the cos / sin tables, read once for Q and once for K
        meta["prep_bytes"] += 2 * (rcos.numel() + rsin.numel()) * 4
    return step, hot, meta


class E2EPipeline:
    """End-to-end steps through the public API with host buffers: each step
    copies its inputs from pinned host memory to the device, runs the whole
    path, and copies the output and LSE back.  Two device buffer sets and
    separate copy streams let step i+1's upload and step i-1's download
    overlap step i's kernels; every step's copies stay inside the timed
    region, which ends after the last download."""

    def __init__(self, hot, host, device, stream):
        import torch
        self.torch = torch
        self.hot = hot
        self.host = host
        q, k, v, o, lse = device
        self.sets = [device, tuple(torch.empty_like(t) for t in (q, k, v, o, lse))]
        self.comp = stream
        self.up = torch.cuda.Stream(device=q.device)
        self.down = torch.cuda.Stream(device=q.device)

    def run(self, n):
        """Run n steps; return their total time in ms (CUDA events)."""
        torch = self.torch
        hq, hk, hv, ho, hl = self.host
        ev = lambda: torch.cuda.Event(enable_timing=False)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(self.comp)
        self.up.wait_event(start)
        self.down.wait_event(start)
        uploaded, computed, downloaded = [None] * n, [None] * n, [None] * n

        def upload(i):
            q, k, v, _, _ = self.sets[i % 2]
            with torch.cuda.stream(self.up):
                if i >= 2:
                    self.up.wait_event(computed[i - 2])   # set i % 2 no longer read
                q.copy_(hq, non_blocking=True)
                k.copy_(hk, non_blocking=True)
                v.copy_(hv, non_blocking=True)
                uploaded[i] = ev()
                uploaded[i].record(self.up)

        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            q, k, v, o, lse = self.sets[i % 2]
            self.comp.wait_event(uploaded[i])
            if i >= 2:
                self.comp.wait_event(downloaded[i - 2])   # o, lse of this set read back
            with torch.cuda.stream(self.comp):
                self.hot(q, k, v, o, lse)
            computed[i] = ev()
            computed[i].record(self.comp)
            with torch.cuda.stream(self.down):
                self.down.wait_event(computed[i])
                ho.copy_(o, non_blocking=True)
                hl.copy_(lse, non_blocking=True)
                downloaded[i] = ev()
                downloaded[i].record(self.down)
        self.comp.wait_event(downloaded[n - 1])
        end.record(self.comp)
        torch.cuda.synchronize()
        return start.elapsed_time(end)


def timed_region(step, steps, warmup, world, rank, local):
    """W untimed warm-up steps, then `steps` timed steps bracketed by a
    barrier and a synchronize on both sides, with CUDA events on the
    launching stream around every launch of the dominant kernel and around
    the whole region, and nvidia-smi clocks sampled meanwhile.
    Returns (per-launch ms list, total ms, clocks summary, launches)."""
    import torch

    from tiled_attention_forward_02_gb300 import attn
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if attn.get_status() != 0:
        raise RuntimeError("device status reported an error during warm-up")
    sampler = ClockSampler(local if world > 1 else torch.cuda.current_device())
    if rank == 0 or world > 1:
        sampler.start()
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    n0 = attn.launch_count()
    t_wall0 = time.time()
    t_start.record(stream)
    for i in range(steps):
        step(kev[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    launches = attn.launch_count() - n0
    per_launch_ms = [a.elapsed_time(b) for a, b in kev]
    total_ms = t_start.elapsed_time(t_end)
    clocks = sampler.summary(t_wall0, t_wall1)
    sampler.stop()
    return per_launch_ms, total_ms, clocks, launches


def tensor_roofline(wl, meta, per_launch_ms, peaks, peak_src):
    """Roofline of the dominant (tensor-core) kernel: algorithmic FLOPs per
    launch over its mean CUDA-event launch time, against the measured dense
    peak of its input type."""
    avg = sum(per_launch_ms) / len(per_launch_ms)
    achieved = meta["flops"] / (avg * 1e-3) / 1e12
    if WORKLOADS[wl][7] == "bf16":
        peak, note = peaks["bf16_tflops"], f"dense bf16, {peak_src} burst"
    else:
        peak = 2.0 * peaks["bf16_tflops"]
        note = f"dense fp8 = 2 x {peak_src} bf16 burst (nominal fp8:bf16 ratio)"
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "peak_source": note, "kernel": meta["kernel"],
            "traffic": recorded_traffic(meta["kernel"], wl)}


def prep_roofline(meta, peaks):
    if not meta.get("prep_events"):
        return None
    pms = [a.elapsed_time(b) for a, b in meta["prep_events"]]
    pms = sum(pms) / len(pms)
    gbs = meta["prep_bytes"] / (pms * 1e-3) / 1e9
    return {"kernel": "prep_fp8_kernel (Q, K, V in one launch)", "ms_per_step": pms, "bound": "hbm",
            "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / peaks["hbm_gbs"], "bytes_per_step": meta["prep_bytes"]}


def fp8_record(wl, args, world, rank, local, dev, peaks, peak_src):
    """The FP8 workload measured in the same run as the headline line: one
    step = the prep of Q, K, V plus the FP8 forward, timed like the main
    workload (device-resident inputs); kernel-alone times of the forward and
    of the three prep launches from CUDA events on their stream."""
    import torch
    step, _, meta = make_step(wl, dev)
    per_launch_ms, total_ms, clocks, launches = timed_region(step, args.steps, args.warmup,
                                                             world, rank, local)
    ms_step = max_over_ranks(total_ms / args.steps, world)
    rec = {
        "workload": wl, "value": world * meta["flops"] / (ms_step * 1e-3) / 1e12,
        "unit": "TFLOPS", "ms_per_step": ms_step, "steps": args.steps, "warmup": args.warmup,
        "dtype": "e4m3", "config": config_of(wl),
        "roofline": tensor_roofline(wl, meta, per_launch_ms, peaks, peak_src),
        "prep_roofline": prep_roofline(meta, peaks),
        "kernel_ms": {"avg": sum(per_launch_ms) / len(per_launch_ms),
                      "median": statistics.median(per_launch_ms),
                      "min": min(per_launch_ms), "max": max(per_launch_ms)},
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "gpu_launches": launches,
    }
    del step, meta
    torch.cuda.empty_cache()
    return rec


def gpu_arm(args, rank, world, local):
    import torch

    from tiled_attention_forward_02_gb300 import attn
    attn.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = args.workload
    step, hot, meta = make_step(wl, dev)
    stream = torch.cuda.current_stream()
    flops = meta["flops"]

    # ---- timed region: device-resident inputs
    per_launch_ms, total_ms, clocks, launches = timed_region(step, args.steps, args.warmup,
                                                             world, rank, local)
    status = attn.get_status()

    ms_step = max_over_ranks(total_ms / args.steps, world)
    value = world * flops / (ms_step * 1e-3) / 1e12

    # ---- end-to-end: host buffers, copies inside the timed region
    e2e_steps = max(3, min(args.steps, 20))
    pipe = E2EPipeline(hot, meta["host"], meta["device"], stream)
    pipe.run(2)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(pipe.run(e2e_steps) / e2e_steps, world)
    barrier(world)

    peaks, peak_src = load_peaks()
    # the FP8 workload (B4 H16 N4096 d128, x50 outliers), plain and with the
    # transform, measured in the same run beside the headline workload
    fp8 = None
    if wl == DEFAULT_WORKLOAD and not args.no_fp8:
        fp8 = [fp8_record(w, args, world, rank, local, dev, peaks, peak_src)
               for w in ("fp8_e4m3_B4_H16_N4096_d128", "fp8_e4m3_hadamard_B4_H16_N4096_d128")]

    if rank != 0:
        return
    avg_launch_ms = sum(per_launch_ms) / len(per_launch_ms)
    achieved = flops / (avg_launch_ms * 1e-3) / 1e12   # dominant kernel alone
    kind = WORKLOADS[wl][7]
    roof_unit, bound = "TFLOP/s", "tensor"
    if kind == "decode":
        # one query row per head: the path streams K and V once, HBM bound
        achieved = meta["bytes"] / (avg_launch_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        peak_note = f"HBM copy bandwidth, {peak_src}"
        roof_unit, bound = "GB/s", "hbm"
    elif kind == "bf16":
        peak = peaks["bf16_tflops"]
        peak_note = f"dense bf16, {peak_src} burst"
    else:
        peak = 2.0 * peaks["bf16_tflops"]
        peak_note = f"dense fp8 = 2 x {peak_src} bf16 burst (nominal fp8:bf16 ratio)"
    cpu_tf, cpu_rows, cpu_s, cpu_threads = (None, 0, 0.0, 0)
    if not args.no_cpu_baseline:
        cpu_tf, cpu_rows, cpu_s, cpu_threads = time_oracle(wl, budget_s=args.cpu_budget)
    # the second limiter of the softmax: one exp2 per score on the MUFU units,
    # 32 per SM per cycle (4 sub-partitions x 8 lanes) at the sampled SM clock
    B_, Hq_, _, Nq_, Nk_, _, causal_, _ = WORKLOADS[wl]
    exps = B_ * Hq_ * Nq_ * Nk_ * (0.5 if causal_ else 1.0)
    sm_hz = (clocks.get("sm_mhz") or peaks.get("sm_max_mhz", 2070.0)) * 1e6
    exp_peak = torch.cuda.get_device_properties(dev).multi_processor_count * 32 * sm_hz
    exp_roofline = None if kind == "decode" else {
        "bound": "mufu", "achieved": exps / (avg_launch_ms * 1e-3) / 1e9,
        "peak": exp_peak / 1e9, "unit": "Gexp/s",
        "frac": exps / (avg_launch_ms * 1e-3) / exp_peak,
        "peak_source": "SMs x 32 exp2 per cycle x median SM clock"}
    prep = prep_roofline(meta, peaks)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if kind.startswith("fp8") else "bf16", "data": "synthetic",
        "config": config_of(wl),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": roof_unit,
                     "frac": achieved / peak, "peak_source": peak_note,
                     "kernel": meta["kernel"],
                     "traffic": recorded_traffic(meta["kernel"], wl)},
        "cpu_baseline": None if cpu_tf is None else {
            "value": cpu_tf, "unit": "TFLOPS", "cores": cpu_threads, "kind": "oracle",
            "sample": f"{cpu_rows} random query rows of batch 0, FP64 two-pass oracle, "
                      f"{cpu_s:.1f} s; TFLOPS-equivalent = 4*keys*d per row",
            "extrapolated_full_problem_s": flops / (cpu_tf * 1e12)},
        "exp_roofline": exp_roofline,
        "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
                "h2d_bytes_per_step": meta["h2d"], "d2h_bytes_per_step": meta["d2h"]},
        "gpu_launches": launches,
        "prep_roofline": prep,
        "kernel_ms": {"avg": avg_launch_ms, "median": statistics.median(per_launch_ms),
                      "min": min(per_launch_ms), "max": max(per_launch_ms)},
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "status": status,
        "kernel_source_hash": kernel_source_hash(),
    }
    if fp8 is not None:
        line["fp8"] = fp8
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip the FP8 records added to the default workload's line")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of FP64 oracle time for the cpu_baseline sample")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    rank, world, local = dist_setup(args)
    if args.impl == "reference":
        reference_arm(args, rank, world)
    else:
        gpu_arm(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
