#!/usr/bin/env python3
"""Benchmark of the fused attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one attention forward (the whole hot path: one kernel launch; two for causal fp8
with an fp8 P V product, three with key splits) over one batch of seeded synthetic inputs
already resident in HBM.  The default workload is the headline shape
B=2, H=32, N=8192, d=128, bf16, non-causal; every input tensor (134 MB each, 403 MB for Q, K, V)
is larger than the 129 MB L2, so consecutive steps do not find their inputs in L2.

Prints ONE JSON line on rank 0: the metric (attention forward TFLOPS, 4·B·H·N²·d, halved for
the causal mask), the device-timed value, an end-to-end value through the C ABI with host
buffers (H2D of Q, K, V and D2H of O, LSE inside the timed region), the roofline of the kernel
against the measured peak, SM clocks read from NVML during the timed region, a sustained leg
(the same step back to back for about two seconds, with its own clock record, against the
sustained peak), and the fp64 CPU oracle timed on a bounded sample of the same workload, whose
outputs also give the raw errors of the GPU result on that sample.  ``--impl reference`` times that oracle as the
reference arm instead.  Under torchrun every rank runs its own copy of the workload (independent
(batch, head) problems: weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import HEADLINE, WORKLOADS, make_inputs  # noqa: E402

METRIC = "attention fwd TFLOPS and % of GB300 dense BF16/FP8 peak (1 GPU, device-timed)"
UNIT = "TFLOPS"
FP8_OVER_BF16 = 4.5 / 2.25          # nominal dense fp8 : bf16 tensor ratio
EXP_PER_CLK_SM = 32                 # MUFU ex2 results per clock per SM on GB300 (measured)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"bf16": float(p["bf16_tflops"]), "bf16_sustained": float(p["bf16_tflops_sustained"]),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


class NvmlClocks:
    """SM clock, power and clock-event reasons read in-process from NVML every ``period_s`` on a
    background thread while the block runs (read-only queries: no clock, power or other GPU
    setting is changed).  Falls back to ``nvidia-smi`` sampling where NVML cannot be loaded."""

    REASON_BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
                   0x4: "sw_power_cap"}

    def __init__(self, device, period_s: float = 0.001):
        import ctypes
        import threading

        self.period = period_s
        self.rows = []
        self.fallback = None
        self._stop = threading.Event()
        self._thread = None
        self.nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.handle = ctypes.c_void_p()
            import torch

            props = torch.cuda.get_device_properties(device)
            uuid = getattr(props, "uuid", None)
            found = False
            if uuid is not None:
                found = nv.nvmlDeviceGetHandleByUUID(f"GPU-{uuid}".encode(),
                                                     ctypes.byref(self.handle)) == 0
            if not found:
                found = nv.nvmlDeviceGetHandleByIndex_v2(device.index or 0,
                                                         ctypes.byref(self.handle)) == 0
            if not found:
                raise OSError("no NVML handle")
            self.nvml = nv
            self._u = ctypes.c_uint()
            self._ull = ctypes.c_ulonglong()
            nv.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(self._u))
            self.max_mhz = float(self._u.value)
        except (OSError, AttributeError):
            self.nvml = None
            self.fallback = ClockSampler(device.index or 0)

    def _sample(self):
        import ctypes

        nv, h = self.nvml, self.handle
        while not self._stop.is_set():
            mhz = pw = reasons = None
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(self._u)) == 0:
                mhz = float(self._u.value)
            if nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(self._u)) == 0:
                pw = self._u.value / 1000.0
            if nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(self._ull)) == 0:
                reasons = int(self._ull.value)
            if mhz is not None:
                self.rows.append((mhz, pw, reasons))
            self._stop.wait(self.period)

    def __enter__(self):
        import threading

        if self.nvml is None:
            self.fallback.__enter__()
            return self
        self.rows = []
        self._stop.clear()
        self._thread = threading.Thread(target=self._sample, daemon=True)
        self._thread.start()
        return self

    def __exit__(self, *exc):
        if self.nvml is None:
            self.fallback.__exit__(*exc)
            return
        self._stop.set()
        self._thread.join(timeout=5)

    def summary(self):
        if self.nvml is None:
            return self.fallback.summary()
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"],
                    "source": "nvml"}
        names = sorted({name for _, _, r in self.rows if r is not None
                        for bit, name in self.REASON_BITS.items() if r & bit})
        pws = [p for _, p, _ in self.rows if p is not None]
        return {"sm_mhz": statistics.median(m for m, _, _ in self.rows),
                "sm_max_mhz": self.max_mhz, "power_w_max": max(pws) if pws else None,
                "samples": len(self.rows), "period_ms": 1e3 * self.period, "reasons": names,
                "source": "nvml (in-process reads during the timed region)"}


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"exattn_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, busy_fraction: float = 0.5):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        pmax = max(r[2] for r in rows)
        loaded = [r for r in rows if r[2] >= busy_fraction * pmax] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in loaded),
                "power_w_max": pmax, "samples": len(loaded), "reasons": reasons}


def oracle_sample_rate(inp, w, target_s: float, rerun=None, outputs=None):
    """Time the fp64 oracle on a sample of the workload sized for about target_s seconds.

    The sample is a set of query rows (spread over the sequence) of the first heads; the rate is
    the attention-forward flops of those rows (4 * keys * d each) per second, in TFLOPS.  With
    a list as `rerun`, a callable that runs the same sample again (returning TFLOPS, seconds) is
    appended to it; with a dict as `outputs`, the oracle's O and LSE of the timed sample and the
    sample's coordinates are stored in it.
    """
    from oracle import oracle

    orc = oracle.get()
    cores = os.cpu_count() or 1
    bh = w.B * w.H
    stride = max(1, w.N // 4096)
    rows_all = list(range(w.N - 1, -1, -stride))

    def run(heads, nrows):
        b_heads = min(heads, w.H)
        nb = (heads + w.H - 1) // w.H
        sub = type(inp)(inp.q[:nb, :b_heads], inp.k[:nb, :b_heads], inp.v[:nb, :b_heads],
                        inp.descale_q, inp.descale_k, inp.descale_v)
        rows = sorted(rows_all[:nrows])
        t0 = time.perf_counter()
        o_ref, l_ref = orc.attention_fwd(sub.raw("q"), sub.raw("k"), sub.raw("v"), w.scale,
                                         w.causal, sub.dtype,
                                         (sub.descale_q, sub.descale_k, sub.descale_v), rows,
                                         cores)
        dt = time.perf_counter() - t0
        last.update(o=o_ref, lse=l_ref, nb=nb, heads=b_heads, rows=rows)
        keys = sum((r + 1) if w.causal else w.N for r in rows)
        nh = sub.q.shape[0] * sub.q.shape[1]
        return 4.0 * keys * w.d * nh / dt / 1e12, dt, nh, len(rows)

    last = {}
    heads, nrows = min(bh, 2), min(len(rows_all), 256)
    tf, dt, nh, nr = run(heads, nrows)
    # grow rows first, then heads, to reach the target duration; shrink rows if one probe
    # already takes longer than the target
    scale = target_s / max(dt, 1e-3)
    if scale > 1.2:
        nrows = min(len(rows_all), int(nrows * scale))
        scale /= nrows / max(nr, 1)
        heads = min(bh, max(heads, int(heads * max(scale, 1.0))))
        tf, dt, nh, nr = run(heads, nrows)
    elif scale < 0.8:
        heads, nrows = 1, max(1, int(nrows * scale * 2))
        tf, dt, nh, nr = run(heads, nrows)
    sample = (f"{nr} query rows x {nh} heads of {w.name} "
              f"({'causal' if w.causal else 'all'} keys each), fp64 on {cores} threads")
    if rerun is not None:
        rerun.append(lambda: run(heads, nrows)[:2])
    if outputs is not None:
        outputs.update(last)
    return tf, dt, cores, sample


def sample_parity(o, lse, ref, dtype: str):
    """Raw errors of the GPU output against the oracle on the CPU-baseline sample: max |O - O_ref|
    and max |LSE - LSE_ref|, elements over the unwidened O tolerance (1e-2 bf16, 5e-2 fp8), and
    elements over the tolerance widened by half a bf16 ulp of |O_ref| (the rounding of O)."""
    import numpy as np

    nb, nh, rows = ref["nb"], ref["heads"], ref["rows"]
    og = o[:nb, :nh, rows].double().cpu().numpy()
    lg = lse[:nb, :nh, rows].double().cpu().numpy()
    tol_o, tol_l = (5e-2, 5e-3) if dtype == "e4m3" else (1e-2, 1e-3)
    err = np.abs(og - ref["o"])
    a = np.abs(ref["o"])
    half_ulp = np.where(a > 0, np.exp2(np.floor(np.log2(np.where(a > 0, a, 1.0))) - 8), 0.0)
    return {"rows": len(rows), "heads": nb * nh, "max_err_o": float(err.max()),
            "max_err_lse": float(np.abs(lg - ref["lse"]).max()), "tol_o": tol_o, "tol_lse": tol_l,
            "n_over_tol_o": int((err > tol_o).sum()),
            "n_over_tol_o_plus_half_ulp": int((err > tol_o + half_ulp).sum())}


L2_BYTES = 129e6          # GB300 L2 (about 126 MiB usable)
FLUSH_BYTES = 256 << 20   # written between steps to evict inputs that fit in L2

def inputs_fit_in_l2(w) -> bool:
    """Whether the workload's Q, K and V together fit in L2 (then each timed launch is preceded
    by a write that evicts them)."""
    elem = 1 if w.dtype == "e4m3" else 2
    return 3 * w.B * w.H * w.N * w.d * elem <= L2_BYTES


KERNEL_SOURCES = ["exact_attention_13_gb300/csrc/fa_fwd_kernel.cuh",
                  "exact_attention_13_gb300/csrc/sm103_ptx.cuh",
                  "exact_attention_13_gb300/csrc/fa_api.cu"]


def kernel_sources_sha256() -> str:
    import hashlib

    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload: str, override, variant: str = ""):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on these sources
    (entries are keyed by workload, plus ":<variant>" for a non-default kernel variant)."""
    if override is not None:
        return override
    path = os.path.join(ROOT, "profiles", "fa_fwd_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(workload + (f":{variant}" if variant else ""))
    if not ent or ent.get("kernel_sources_sha256") != kernel_sources_sha256():
        return None
    return ent.get("dram_bytes_per_launch")


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (the slowest rank's time); x itself when alone."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, world: int, ms_slowest: float) -> float:
    """Whole-job throughput: every rank's work (weak scaling) over the slowest rank's time."""
    return world * flops_per_rank / (ms_slowest * 1e-3) / 1e12


def init_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if _cuda_ok() else "gloo")
    return world, rank, local


def _cuda_ok():
    import torch

    return torch.cuda.is_available()


def run_reference(args, w, world, rank):
    """Reference arm: the fp64 CPU oracle as it stands, on bounded samples of the workload."""
    if rank != 0:
        return
    inp = make_inputs(w)
    # every step runs the same bounded sample, sized so that the whole run (warm-up included)
    # takes about --ref-budget-s of oracle work
    per_step = max(0.02, min(args.ref_step_s, args.ref_budget_s / (args.warmup + args.steps)))
    rerun = []
    _, _, cores, sample = oracle_sample_rate(inp, w, target_s=per_step, rerun=rerun)
    rates, times = [], []
    for step in range(args.warmup + args.steps):
        tf, dt = rerun[0]()
        if step >= args.warmup:
            rates.append(tf)
            times.append(dt)
    value = statistics.median(rates)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "shape": w.describe(), "parallelism": "host threads"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def launches_per_step(w, args, fp8_pv: bool) -> int:
    """Kernel launches of one attention call: the forward kernel (twice for causal fp8 with an
    fp8 P V product longer than one 256-row query block: its first block runs the f16 P V
    instance), plus the merge kernel with key splits."""
    fwd = 2 if (w.causal and fp8_pv and w.N > 256) else 1
    return fwd + (1 if args.splits > 1 else 0)


def run_ours(args, w, world, rank, local):
    import torch

    import exact_attention_13_gb300 as ea

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = make_inputs(w)
    q, k, v = (getattr(inp, n).to(dev) for n in "qkv")
    descale = (inp.descale_q, inp.descale_k, inp.descale_v)
    # fp8 with block descales: the operands are the bf16 draws quantised on the GPU, one descale
    # per 128-row block (power-of-two descales for V)
    block = w.dtype == "e4m3" and args.fp8_scaling == "block"
    scales = ()
    if block:
        from workloads import random_inputs

        src = random_inputs(w.B, w.H, w.N, w.d, "bf16", w.seed)
        q, dq_b = ea.quantize_e4m3(src.q.to(dev))
        k, dk_b = ea.quantize_e4m3(src.k.to(dev))
        v, dv_b = ea.quantize_e4m3(src.v.to(dev), pow2=True)
        scales = (dq_b, dk_b, dv_b)
        del src
    o = torch.empty(w.B, w.H, w.N, w.d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    splits = args.splits
    workspace = None
    if splits > 1:
        workspace = torch.empty(ea.split_workspace_bytes(w.B, w.H, w.N, w.d, splits),
                                dtype=torch.uint8, device=dev)

    pv16 = args.fp8_pv == "f16"

    def attn(q_, k_, v_, o_, l_, sc_):
        if block:
            ea.fwd_fp8_blockscaled(q_, k_, v_, *sc_, causal=w.causal, scale=w.scale, out=o_,
                                   lse=l_, num_splits=splits, workspace=workspace, pv16=pv16)
        else:
            ea.fwd(q_, k_, v_, causal=w.causal, scale=w.scale, descale=descale, out=o_, lse=l_,
                   num_splits=splits, workspace=workspace, pv16=pv16)

    def step():
        attn(q, k, v, o, lse, scales)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    # ---- device-timed region: K launches back to back on one stream, or, when the inputs fit in
    # L2, each launch timed on its own with a 256 MB write between launches that evicts them
    in_l2 = inputs_fit_in_l2(w)
    clk = NvmlClocks(dev)
    barrier()
    torch.cuda.synchronize()
    if not in_l2:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with clk:
            start.record(stream)
            for _ in range(args.steps):
                step()
            end.record(stream)
            torch.cuda.synchronize()
        ms = start.elapsed_time(end) / args.steps
    else:
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        with clk:
            for e0, e1 in evs:
                flush.fill_(1)
                e0.record(stream)
                step()
                e1.record(stream)
            torch.cuda.synchronize()
        ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / args.steps
        del flush
    barrier()
    clocks = clk.summary()
    ms_max = max_over_ranks(ms, world, dev)
    assert ea.device_status() == 0, "device wait timed out during the bench"

    # ---- end to end: pinned host inputs -> device -> attention -> host outputs, per step.
    # Pipelined the way a serving loop runs it: two device buffer sets, H2D on one stream, the
    # kernel on another, D2H on a third; step i's copies overlap steps i-1 / i+1's kernels, and
    # every step still moves its own inputs in and its own outputs out.
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    sh = [t.cpu().pin_memory() for t in scales]
    dsc = [list(scales), [torch.empty_like(t) for t in scales]]
    oh = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    lh = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    dq = [q, torch.empty_like(q)]
    dk = [k, torch.empty_like(k)]
    dv = [v, torch.empty_like(v)]
    do = [o, torch.empty_like(o)]
    dl = [lse, torch.empty_like(lse)]
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in", "cmp", "out")}
    for b in range(2):  # every buffer starts free
        for name in ("cmp", "out"):
            ev[name][b].record(s_cmp if name == "cmp" else s_out)

    def e2e_step(i):
        b = i % 2
        s_in.wait_event(ev["cmp"][b])          # the kernel that last read buffer b is done
        with torch.cuda.stream(s_in):
            dq[b].copy_(qh, non_blocking=True)
            dk[b].copy_(kh, non_blocking=True)
            dv[b].copy_(vh, non_blocking=True)
            for dst, srcp in zip(dsc[b], sh):
                dst.copy_(srcp, non_blocking=True)
        ev["in"][b].record(s_in)
        s_cmp.wait_event(ev["in"][b])
        s_cmp.wait_event(ev["out"][b])         # the D2H that last read outputs b is done
        with torch.cuda.stream(s_cmp):
            attn(dq[b], dk[b], dv[b], do[b], dl[b], dsc[b])
        ev["cmp"][b].record(s_cmp)
        s_out.wait_event(ev["cmp"][b])
        with torch.cuda.stream(s_out):
            oh[b].copy_(do[b], non_blocking=True)
            lh[b].copy_(dl[b], non_blocking=True)
        ev["out"][b].record(s_out)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(s_in)
    for i in range(args.steps):
        e2e_step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    e_end.record(s_out)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(e_start.elapsed_time(e_end) / args.steps, world, dev)
    assert ea.device_status() == 0, "device wait timed out during the end-to-end run"
    # ---- sustained: the device-timed step back to back for about --sustained-s seconds, with
    # its own clock record (the timed region above is a burst of a few tens of milliseconds); run
    # last, so that the power-capped clocks it settles at do not carry into the other legs
    sustained = None
    if args.sustained_s > 0:
        n_sus = max(args.steps, int(math.ceil(args.sustained_s * 1e3 / ms)))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sclk = NvmlClocks(dev, period_s=0.01)
        barrier()
        torch.cuda.synchronize()
        with sclk:
            s0.record(stream)
            for _ in range(n_sus):
                step()
            s1.record(stream)
            torch.cuda.synchronize()
        barrier()
        s_ms = max_over_ranks(s0.elapsed_time(s1) / n_sus, world, dev)
        sustained = {"steps": n_sus, "seconds": n_sus * s_ms * 1e-3, "ms_per_step": s_ms,
                     "value": job_tflops(w.flops, world, s_ms), "unit": UNIT,
                     "clocks": sclk.summary()}
        assert ea.device_status() == 0, "device wait timed out during the sustained run"

    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh, *sh))
    d2h = oh[0].numel() * oh[0].element_size() + lh[0].numel() * lh[0].element_size()

    flops_rank = w.flops
    value = job_tflops(flops_rank, world, ms_max)
    e2e_value = job_tflops(flops_rank, world, e_ms)

    if rank != 0:
        return
    pk = peaks()
    is_fp8 = w.dtype == "e4m3"
    if is_fp8 and pv16:
        # half the flops (Q K^T) at the fp8 rate, half (P V) at the f16 rate: the time-weighted
        # peak is 1 / (0.5 / (2 P) + 0.5 / P) = 4 P / 3
        dtype_mult = 4.0 / 3.0
        peak_note = " x 4/3 (Q K^T fp8 at 2x, P V f16 at 1x)"
    else:
        dtype_mult = FP8_OVER_BF16 if is_fp8 else 1.0
        peak_note = " x 2 (nominal fp8:bf16)" if is_fp8 else ""
    peak = pk["bf16"] * dtype_mult
    if sustained is not None:
        sustained["peak"] = pk["bf16_sustained"] * dtype_mult
        sustained["frac"] = sustained["value"] / world / sustained["peak"]
        sustained["peak_kind"] = f"{pk['source']} cuBLAS bf16 sustained" + peak_note
    achieved = flops_rank / (ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "traffic": None if args.lib else measured_traffic(
                    w.name, args.traffic_bytes, "_".join(
                        ([("pv16" if pv16 else "")] if is_fp8 else []) +
                        (["block"] if block else [])).strip("_")),
                "peak_kind": f"{pk['source']} cuBLAS bf16 burst" + peak_note,
                "kernel": "exattn::fa_fwd_kernel"}
    # exp-unit bound at the clock seen during the run (informative)
    exps = w.B * w.H * (w.N * (w.N + 1) / 2 if w.causal else w.N * w.N)
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks.get("sm_mhz") or 2070.0
    exp_floor_ms = exps / (EXP_PER_CLK_SM * sm_count * mhz * 1e6) * 1e3
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if is_fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "shape": w.describe(), "global_batch": w.B * world,
                   "heads": w.H, "seq_len": w.N, "head_dim": w.d, "causal": w.causal,
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "key_splits": args.splits,
                   **({"pv_product": args.fp8_pv, "fp8_scaling": args.fp8_scaling}
                      if is_fp8 else {}),
                   **({"library": args.lib} if args.lib else {}),
                   "l2": "inputs larger than L2 (no flush)" if not in_l2 else
                   "inputs fit in L2: 256 MB written between steps, each step timed alone"},
        "pct_of_peak": 100.0 * achieved / peak,
        "exp_bound": {"exp_per_clk_sm": EXP_PER_CLK_SM, "floor_ms": exp_floor_ms,
                      "frac": exp_floor_ms / ms},
        "roofline": roofline,
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
                "pipelining": "2 buffer sets; H2D, kernel, D2H on 3 streams"},
        "gpu_launches": args.steps * launches_per_step(w, args, is_fp8 and not pv16),
        "sustained": sustained,
    }
    if not args.no_cpu_baseline:
        ref = {}
        tf, dt, cores, sample = oracle_sample_rate(inp, w, target_s=args.cpu_s, outputs=ref)
        line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": sample, "seconds": dt}
        # the same sample compared with the GPU's output (block-scaled fp8 quantises other
        # inputs on the GPU, so it has no per-tensor oracle sample here)
        line["parity"] = (sample_parity(o, lse, ref, w.dtype) if not block else
                          {"skipped": "block-scaled inputs differ from the oracle sample"})
    print(json.dumps(line), flush=True)


def run_quantize(args, w, world, rank, local):
    """Time the fp8 block quantiser (fa_quantize_e4m3) on a bf16 operand of the workload's
    shape: bytes moved per launch = 2 (bf16 in) + 1 (e4m3 out) per element, plus the descales."""
    import torch

    import exact_attention_13_gb300 as ea
    from workloads import hadamard_signs, random_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    x = random_inputs(w.B, w.H, w.N, w.d, "bf16", w.seed).q.to(dev)
    codes = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=dev)
    nblk = -(-w.N // 128)
    ds = torch.empty((w.B, w.H, nblk), dtype=torch.float32, device=dev)
    signs = hadamard_signs(w.d, w.seed).to(dev) if args.hadamard else None

    def step():
        ea.quantize_e4m3(x, signs=signs, codes=codes, descales=ds)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with NvmlClocks(dev) as clk:
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end) / args.steps, world, dev)
    if rank != 0:
        return
    nbytes = x.numel() * 3 + ds.numel() * 4 + (w.d * 4 if signs is not None else 0)
    gbs = nbytes / (ms * 1e-3) / 1e9
    pk = peaks()
    line = {
        "metric": "fp8 block quantisation GB/s (1 GPU, device-timed)", "value": gbs * world,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16->e4m3", "data": "synthetic",
        "config": {"workload": w.name, "shape": f"B{w.B} H{w.H} N{w.N} d{w.d}",
                   "hadamard": bool(args.hadamard), "block_rows": 128,
                   "l2": "input larger than L2 (no flush)" if x.numel() * 2 > 129e6
                   else "input smaller than L2"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"], "traffic": None,
                     "peak_kind": f"{pk['source']} copy bandwidth",
                     "kernel": "exattn::quantize_e4m3_kernel"},
        "clocks": clk.summary(),
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def run_backward(args, w, world, rank, local):
    """Time the attention backward (fa_bwd: D, dK/dV and dQ kernels) on the workload's shape,
    with O and LSE from the forward.  Work counted: 10·B·H·N²·d flop (halved causal), the five
    N²d products of the backward (2.5x the forward's)."""
    import torch

    import exact_attention_13_gb300 as ea
    from workloads import random_bwd_inputs

    if w.dtype != "bf16":
        raise SystemExit("the backward takes bf16 operands")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = random_bwd_inputs(w.B, w.H, w.N, w.d, w.seed)
    q, k, v, do = (getattr(inp, n).to(dev) for n in ("q", "k", "v", "do"))
    o, lse = ea.fwd(q, k, v, causal=w.causal)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(ea.bwd_workspace_bytes(w.B, w.H, w.N), dtype=torch.uint8, device=dev)

    def step():
        ea.bwd(q, k, v, o, lse, do, causal=w.causal, dq=dq, dk=dk, dv=dv, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with NvmlClocks(dev) as clk:
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end) / args.steps, world, dev)
    assert ea.device_status() == 0, "device wait timed out during the bench"
    if rank != 0:
        return
    flops = 2.5 * w.flops
    tf = flops / (ms * 1e-3) / 1e12
    pk = peaks()
    line = {
        "metric": "attention bwd TFLOPS (10·B·H·N²·d, halved causal; 1 GPU, device-timed)",
        "value": tf * world, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "shape": w.describe(), "op": "backward"},
        "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16"], "unit": "TFLOP/s",
                     "frac": tf / pk["bf16"], "traffic": None,
                     "peak_kind": f"{pk['source']} cuBLAS bf16 burst",
                     "kernel": "exattn::bwd_dkdv_kernel + bwd_dq_kernel + bwd_delta_kernel"},
        "clocks": clk.summary(),
        "gpu_launches": 3 * args.steps,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--splits", type=int, default=1,
                    help="key splits per query tile (split-KV + merge kernel)")
    ap.add_argument("--cpu-s", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--ref-step-s", type=float, default=4.0,
                    help="reference arm: longest oracle sample per step")
    ap.add_argument("--ref-budget-s", type=float, default=90.0,
                    help="reference arm: oracle seconds for the whole run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sustained-s", type=float, default=2.0,
                    help="seconds of the sustained leg (0 = off)")
    ap.add_argument("--fp8-pv", default="e4m3", choices=["e4m3", "f16"],
                    help="fp8 operands: precision of the P V product")
    ap.add_argument("--fp8-scaling", default="tensor", choices=["tensor", "block"],
                    help="fp8 operands: one descale per tensor, or per 128-row block")
    ap.add_argument("--op", default="attention", choices=["attention", "quantize", "backward"],
                    help="attention forward (default), the fp8 block quantiser alone, or the "
                         "attention backward")
    ap.add_argument("--hadamard", action="store_true",
                    help="--op quantize: apply the incoherent (Hadamard) transform")
    ap.add_argument("--traffic-bytes", type=float, default=None,
                    help="DRAM bytes per launch from an ncu capture of the current kernel")
    ap.add_argument("--lib", default=None,
                    help="time this build of the library (e.g. a compile-time variant of the "
                         "kernel) instead of the package's libexattn.so; the roofline's DRAM "
                         "traffic is then null")
    args = ap.parse_args()
    if args.lib:
        if args.impl == "reference":
            ap.error("--lib applies to --impl ours")
        import exact_attention_13_gb300 as ea

        ea.lib(os.path.abspath(args.lib))
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        # host-only arm: no process group; under torchrun rank 0 alone does the work
        run_reference(args, w, int(os.environ.get("WORLD_SIZE", "1")),
                      int(os.environ.get("RANK", "0")))
        return
    world, rank, local = init_dist()
    if args.op == "quantize":
        run_quantize(args, w, world, rank, local)
    elif args.op == "backward":
        run_backward(args, w, world, rank, local)
    else:
        run_ours(args, w, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
