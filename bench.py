"""Benchmark of libgemmpipe on the named GEMM workloads.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Headline (``value``): INT8 IGEMM M = N = K = 4096 (the pages' benchmark shape),
int8 operands uniform on [-128, 127], int32 C, in TOPS.  A step is one
gemm_s8s8s32 call through the C ABI with inputs resident in HBM.  Because the
inputs (32 MiB) fit in the 126 MiB L2, a 256 MiB buffer is written and
another 256 MiB read between timed steps (no input cached, no dirty lines
left for the timed step to write back), and each step is timed alone with
CUDA events on its stream.

``roofline`` is the GEMM kernel alone: 2 M N K over the mean of the CUDA
events the library records around that kernel on its launch stream, in a
second pass of the same timed steps (those events stop the GEMM's
programmatic early launch, so the first pass, which gives ``value``, runs
without them).  ``peak`` is the measured bf16 burst figure (the fp16
tcgen05 pipe runs at the bf16 rate; INT8 runs on that pipe too), or HBM
copy bandwidth for the skinny shape.  ``traffic`` is the DRAM bytes of one
ncu capture of the same kernel sources (null once they change).

``parity``: every timed output (the C of the last timed step) is compared
with the CPU oracle's whole product -- bit for bit for INT8, max-abs 1e-2 and
relative Frobenius 1e-4 for FP16 -- and the oracle's wall time on all host
cores is each workload's CPU baseline (``cpu_baseline`` for the headline,
``cpu`` in each secondary entry).

``e2e`` is the same headline through the host-buffer call
gemm_s8s8s32_host: page-locked A and B in, C out, inside the timed region.
``int8_step_floor`` puts the step beside its floor (the widening pass at the
in-run copy rate plus the GEMM kernel); ``library_context`` times cuBLAS FP16
and torch._int_mm on the same shape and the pages' own design (warp-level
integer MMA, the legacy INT8 ceiling) -- context, not the hot path.

``secondary`` (last in the line): INT8 512^3 and FP16 1024^3 (launch- and
latency-bound, reported only), the ragged FP16 4093 x 3001 x 4107, the skinny
FP16 16384 x 128 x 16384 (GB/s of algorithmic bytes: A, B and C moved once)
and FP16 4096^3 (TFLOPS), each with its step time, kernel time, fractions of
peak per kernel (``frac``) and per step (``step_frac``), parity and CPU time.

``--impl reference`` times the CPU oracle on the host cores instead, on a
bounded sample of rows of the same workload.

With N > 1 (torchrun, one rank per GPU) every rank runs its own replica of
the workload (the GEMM does not shard across GPUs here); ``value`` is the
total of all ranks' operations over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "INT8 TOPS and FP16 TFLOPS at 4096³ (% of dense tensor peak); GB/s on skinny"
HEADLINE = 2  # index of the INT8 4096^3 workload in inputs.WORKLOADS
FLUSH_BYTES = 256 << 20
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# DRAM bytes (read + write) per launch of a kernel variant, from one
# `ncu --set full` capture of that launch, valid only while the kernel
# sources hash as they did when the counters were taken (else null).
KERNEL_SOURCES = ["gemm_kernel.cuh", "ptx.cuh", "gemm_params.h", "launch_impl.cuh", "gemm_f16.cu", "gemm_s8.cu",
                  "gemmpipe_api.cpp"]
TRAFFIC = {
    # (dtype, M, N, K, cta pair, BN, BK): (bytes per launch, sources hash)
    ("s8", 4096, 4096, 4096, 1, 256, 64): (137_224_448, "1ae595d388cafc61"),
    ("f16", 4096, 4096, 4096, 1, 256, 64): (138_488_576, "1ae595d388cafc61"),
    ("f16", 16384, 128, 16384, 0, 128, 128): (544_418_304, "1ae595d388cafc61"),
    ("f16", 4093, 3001, 4107, 2, 512, 64): (67_333_120, "1ae595d388cafc61"),
}


def kernel_source_hash(csrc: str | None = None) -> str:
    """Hash of the kernel sources' code (in `csrc`, default the package's):
    comments and blank space are left out, so an edit to a comment keeps the
    captured figures valid."""
    import hashlib
    import re
    csrc = csrc or os.path.join(ROOT, "software_pipelined_loop_gb300", "csrc")
    h = hashlib.sha1()
    for f in KERNEL_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)   # block comments
        text = re.sub(r"//[^\n]*", " ", text)               # line comments
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def measured_traffic(dtype: str, plan: dict, shape: tuple) -> int | None:
    """Captured DRAM traffic of the launch this plan runs on this shape, or None."""
    t = TRAFFIC.get((dtype, *shape, plan["cta_pair"], plan["BN"], plan["BK"]))
    if t is None or t[1] != kernel_source_hash():
        return None
    return t[0]


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return dict(PEAKS_FALLBACK), "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (50 Hz) with host timestamps; the bench asks for
    the ones that fall inside its timed window."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples: list[tuple[float, list[str]]] = []
        self.proc = None
        self.thread = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        win = [s for t, s in self.samples if t0 - 0.025 <= t <= t1 + 0.025]
        if not win:
            win = [s for _, s in self.samples]
        sm = [float(s[0]) for s in win if s and s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in win if len(s) > 1 and s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4) if len(s) > 4 + i and s[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win)}


# ---------------------------------------------------------------- helpers

SHAPE = None  # (dtype, M, N, K) from --shape


def workload(index: int):
    from software_pipelined_loop_gb300 import inputs
    if index == HEADLINE and SHAPE is not None:
        dt, M, N, K = SHAPE
        A, B = inputs.make_operands(dt, M, N, K, inputs.SEED_BASE + 7)
        return (f"{dt}_{M}x{N}x{K}", dt, M, N, K, A, B)
    return inputs.workload_operands(index)


def cpu_oracle_rate(A, B, dtype: str, target_s: float, max_rows: int | None = None) -> dict:
    """Times the oracle on the first rows of the workload for about target_s."""
    import oracle
    M, K = A.shape
    N = B.shape[1]
    fn = oracle.gemm_s8s8s32 if dtype == "s8" else oracle.gemm_f16f32
    threads = oracle.default_threads()
    rows = min(M, max(threads, 8))
    t = time.perf_counter()
    fn(A, B, rows=list(range(rows)), threads=threads)
    dt = time.perf_counter() - t
    if dt < target_s:
        rows = int(min(M, max(rows, rows * target_s / max(dt, 1e-3))))
        if max_rows:
            rows = min(rows, max_rows)
        t = time.perf_counter()
        fn(A, B, rows=list(range(rows)), threads=threads)
        dt = time.perf_counter() - t
    ops = 2.0 * rows * N * K
    return {"value": ops / dt / 1e12, "cores": threads, "seconds": dt, "rows": rows}


def run_reference(args) -> int:
    """The CPU oracle as the reference arm (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    name, dtype, M, N, K, A, B = workload(HEADLINE)
    # Each step times a bounded sample of rows: about --ref-seconds of CPU
    # work, less when many steps are asked for, so the whole run stays near
    # two minutes.
    per_step = args.ref_seconds if args.ref_seconds is not None else max(0.2, min(4.0, 120.0 / max(1, args.steps)))
    for _ in range(max(0, args.warmup)):
        cpu_oracle_rate(A, B, dtype, target_s=0.0, max_rows=8)
    vals, secs, rows, cores = [], 0.0, 0, 1
    for _ in range(max(1, args.steps)):
        r = cpu_oracle_rate(A, B, dtype, target_s=per_step)
        vals.append(r["value"])
        secs += r["seconds"]
        rows = r["rows"]
        cores = r["cores"]
    v = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
        "config": bench_config(name, M, N, K, "flushed" if A.nbytes + B.nbytes < FLUSH_BYTES else "inputs > L2"),
        "cpu_baseline": {"value": v, "unit": "TOPS", "cores": cores, "kind": "oracle",
                         "sample": f"first {rows} of {M} rows of C per step (all {N} columns, full K)"},
        "e2e": {"value": v, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def time_steps(call, steps: int, flush=None, stream=None) -> list[float]:
    """Per-step CUDA-event times (ms) on `stream`, L2 flushed before each."""
    import torch
    evs = []
    for _ in range(steps):
        if flush is not None:
            flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def measure_gemm(wl, steps: int, warmup: int, dev, flush, peaks, peak_src):
    """Device-resident timing of one workload (name, dtype, M, N, K, A, B)."""
    import torch

    from software_pipelined_loop_gb300 import gemmpipe
    name, dtype, M, N, K, A, B = wl
    Ad = torch.from_numpy(A).to(dev)
    Bd = torch.from_numpy(B).to(dev)
    C = torch.empty((M, N), dtype=torch.int32 if dtype == "s8" else torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    fn = gemmpipe.gemm_s8s8s32 if dtype == "s8" else gemmpipe.gemm_f16f32
    call = lambda: fn(M, N, K, Ad, Bd, C, stream)
    in_bytes = A.nbytes + B.nbytes
    needs_flush = in_bytes < FLUSH_BYTES
    for _ in range(max(3, warmup)):
        call()
    torch.cuda.synchronize()
    st = gemmpipe.gemmpipe_get_device_status(stream)
    if st != gemmpipe.OK:
        raise RuntimeError(f"{name}: device status {gemmpipe.STATUS.get(st, st)}")
    # Pass 1 times whole steps as a caller runs them.  Pass 2 repeats them
    # with the library's per-kernel events on (events between the widening
    # or padding kernel and the GEMM stop the GEMM's programmatic early
    # launch, so they stay out of pass 1); its GEMM-kernel average is the
    # roofline's duration.
    launches0 = gemmpipe.gemmpipe_launch_count()
    t0 = time.time()
    times = time_steps(call, steps, flush if needs_flush else None, stream)
    launches = gemmpipe.gemmpipe_launch_count() - launches0
    gemmpipe.gemmpipe_timing_read()
    gemmpipe.gemmpipe_timing_enable(True)
    time_steps(call, steps, flush if needs_flush else None, stream)
    t1 = time.time()
    gemm_ms, gemm_n, aux_ms, aux_n = gemmpipe.gemmpipe_timing_read()
    gemmpipe.gemmpipe_timing_enable(False)
    st = gemmpipe.gemmpipe_get_device_status(stream)
    if st != gemmpipe.OK:
        raise RuntimeError(f"{name}: device status {gemmpipe.STATUS.get(st, st)}")
    ms = statistics.mean(times)
    flops = 2.0 * M * N * K
    alg_bytes = in_bytes + C.numel() * C.element_size()
    kernel_ms = gemm_ms / max(1, gemm_n)
    plan = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K, Ad, Bd, C)
    skinny = N <= 128
    traffic = measured_traffic(dtype, plan, (M, N, K))
    if skinny:
        peak = peaks["hbm_gbs"]
        achieved = alg_bytes / kernel_ms / 1e6
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "peak_source": f"hbm_gbs, {peak_src}"}
    else:
        peak = peaks["bf16_tflops"]
        achieved = flops / kernel_ms / 1e9
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic, "peak_source": f"bf16_tflops burst, {peak_src}"}
    return {
        "name": name, "dtype": dtype, "M": M, "N": N, "K": K, "ms": ms, "ms_median": statistics.median(times),
        "ops_per_s": flops / ms / 1e9, "bytes_per_s": alg_bytes / ms / 1e6, "kernel_ms": kernel_ms,
        "aux_ms": aux_ms / max(1, aux_n) if aux_n else 0.0, "launches": launches, "flops": flops,
        "alg_bytes": alg_bytes, "roofline": roof, "plan": plan, "l2": "flushed" if needs_flush else "inputs > L2",
        "window": (t0, t1), "A": A, "B": B, "C": C,
    }


def measure_e2e(res: dict, steps: int, dev) -> dict:
    """Same GEMM through the C ABI's host-buffer call (gemm_s8s8s32_host /
    gemm_f16f32_host): A and B from page-locked host memory to the GPU, the
    GEMM, C back to page-locked host memory, all inside the event-timed
    region (the library overlaps the three by row panels).  Its C is
    compared with the device-resident call's C (exact for INT8; FP16 plans
    differ per panel, so within the FP16 tolerance)."""
    import torch

    from software_pipelined_loop_gb300 import gemmpipe
    A, B, M, N, K = res["A"], res["B"], res["M"], res["N"], res["K"]
    Ah = torch.from_numpy(A).pin_memory()
    Bh = torch.from_numpy(B).pin_memory()
    out_dtype = torch.int32 if res["dtype"] == "s8" else torch.float32
    Ch = torch.empty((M, N), dtype=out_dtype).pin_memory()
    stream = torch.cuda.current_stream(dev)
    fn = gemmpipe.gemm_s8s8s32_host if res["dtype"] == "s8" else gemmpipe.gemm_f16f32_host
    call = lambda: fn(M, N, K, Ah, Bh, Ch, stream)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    times = time_steps(call, steps, None, stream)
    st = gemmpipe.gemmpipe_get_device_status(stream)
    if st != gemmpipe.OK:
        raise RuntimeError(f"e2e: device status {gemmpipe.STATUS.get(st, st)}")
    ms = statistics.mean(times)
    ref = res["C"].cpu()
    if res["dtype"] == "s8":
        same = bool(torch.equal(Ch, ref))
    else:
        same = bool((Ch.double() - ref.double()).abs().max().item() <= 1e-2)
    if not same:
        raise RuntimeError("e2e: the host-buffer call's C differs from the device-resident call's C")
    return {"value": res["flops"] / ms / 1e9, "unit": "TOPS" if res["dtype"] == "s8" else "TFLOPS",
            "ms_per_step": ms, "h2d_bytes_per_step": A.nbytes + B.nbytes,
            "d2h_bytes_per_step": Ch.numel() * Ch.element_size(),
            "call": fn.__name__, "panel_rows": gemmpipe.gemmpipe_host_panel_rows(M)}


def measure_copy_ref(dev, peaks: dict, reps: int = 10) -> dict:
    """The in-run bandwidth reference: the library's plain copy kernel moving
    512 MiB device to device (bytes read + bytes written per second)."""
    import torch

    from software_pipelined_loop_gb300 import gemmpipe
    n = 512 << 20
    src = torch.ones(n, dtype=torch.uint8, device=dev)
    dst = torch.empty(n, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    call = lambda: gemmpipe.gemmpipe_copy(dst, src, n, stream)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ms = statistics.median(time_steps(call, reps, None, stream))
    gbs = 2 * n / ms / 1e6
    return {"kernel": "copy_kernel (16-byte loads and stores, grid-stride)", "bytes_moved": 2 * n,
            "gbs": gbs, "of_measured_hbm_peak": gbs / peaks["hbm_gbs"]}


def parity_check(res: dict) -> dict:
    """The timed call's C (the output of its last timed step) against the
    CPU oracle's whole product, every element: bit-exact for INT8, max-abs
    <= 1e-2 and relative Frobenius <= 1e-4 for FP16.  The oracle's wall time
    on the host cores is this workload's CPU baseline."""
    import numpy as np

    import oracle
    A, B = res["A"], res["B"]
    threads = oracle.default_threads()
    t = time.perf_counter()
    want = oracle.gemm_s8s8s32(A, B, threads=threads) if res["dtype"] == "s8" else \
        oracle.gemm_f16f32(A, B, threads=threads)
    secs = time.perf_counter() - t
    got = res["C"].cpu().numpy()
    if res["dtype"] == "s8":
        bad = int(np.count_nonzero(got != want))
        ok = bad == 0
        verdict = f"bit-exact, all {got.size} elements" if ok else f"FAIL: {bad} of {got.size} elements differ"
    else:
        d = got.astype(np.float64) - want.astype(np.float64)
        err = float(np.abs(d).max()) if d.size else 0.0
        nrm = float(np.linalg.norm(want.astype(np.float64)))
        rel = float(np.linalg.norm(d) / nrm) if nrm > 0 else float(np.linalg.norm(d))
        ok = bool(np.isfinite(got).all()) and err <= 1e-2 and rel <= 1e-4
        verdict = f"{'ok' if ok else 'FAIL'}: all {got.size} elements, max-abs {err:.2e}, rel-fro {rel:.2e}"
    return {"ok": ok, "verdict": verdict, "oracle_s": secs, "cores": threads,
            "oracle_rate": res["flops"] / secs / 1e12}


def library_context(dev, flush, steps: int) -> dict:
    """Library calls on the 4096^3 operands, timed like the steps above
    (L2 flushed, CUDA events): cuBLAS FP16 through torch (fp32 output where
    this torch offers it) and torch._int_mm INT8.  Context only; nothing of
    libgemmpipe runs here."""
    import torch

    from software_pipelined_loop_gb300 import inputs
    out = {}
    M = N = K = 4096
    A, B = inputs.make_operands("f16", M, N, K, inputs.SEED_BASE + 5)
    Ad, Bd = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
    stream = torch.cuda.current_stream(dev)
    try:
        torch.mm(Ad[:8, :8], Bd[:8, :8], out_dtype=torch.float32)
        call, label = (lambda: torch.mm(Ad, Bd, out_dtype=torch.float32)), "cublas_f16_f32out_4096"
    except (TypeError, RuntimeError):
        call, label = (lambda: torch.mm(Ad, Bd)), "cublas_f16_f16out_4096"
    for _ in range(3):
        call()
    ms = statistics.mean(time_steps(call, steps, flush, stream))
    out[label] = {"ms": ms, "tflops": 2.0 * M * N * K / ms / 1e9}
    A8, B8 = inputs.make_operands("s8", M, N, K, inputs.SEED_BASE + 2)
    A8d, B8d = torch.from_numpy(A8).to(dev), torch.from_numpy(B8).to(dev)
    try:
        call = lambda: torch._int_mm(A8d, B8d)
        for _ in range(3):
            call()
        ms = statistics.mean(time_steps(call, steps, flush, stream))
        out["torch_int_mm_s8_4096"] = {"ms": ms, "tops": 2.0 * M * N * K / ms / 1e9}
    except RuntimeError as e:
        out["torch_int_mm_s8_4096"] = {"unavailable": str(e).splitlines()[0][:120]}
    return out


def legacy_int8_ceiling(head: dict, dev, flush, steps: int) -> dict:
    """INT8 4096^3 on the library's comparison path: the pages' own design
    (warp-level mma.sync m16n8k32 s8 -> s32 fed by a cp.async ring),
    recompiled for sm_103a.  Its GEMM-kernel rate is the legacy integer-MMA
    ceiling, the second denominator of the INT8 fraction."""
    import torch

    from software_pipelined_loop_gb300 import gemmpipe
    M, N, K = head["M"], head["N"], head["K"]
    Ad, Bd = torch.from_numpy(head["A"]).to(dev), torch.from_numpy(head["B"]).to(dev)
    C = torch.empty((M, N), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    gemmpipe.gemmpipe_set_plan_override(2, 0, 0, -1, -1)
    try:
        call = lambda: gemmpipe.gemm_s8s8s32(M, N, K, Ad, Bd, C, stream)
        call()
        torch.cuda.synchronize()
        gemmpipe.gemmpipe_timing_read()
        gemmpipe.gemmpipe_timing_enable(True)
        time_steps(call, steps, flush, stream)
        gms, gn, _, _ = gemmpipe.gemmpipe_timing_read()
        gemmpipe.gemmpipe_timing_enable(False)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
    if gemmpipe.gemmpipe_get_device_status(stream) != gemmpipe.OK:
        raise RuntimeError("legacy INT8 path: device status not OK")
    if not torch.equal(C, head["C"]):
        raise RuntimeError("legacy INT8 path: C differs from the tcgen05 path's C")
    kms = gms / max(1, gn)
    return {"kernel_ms": kms, "tops": head["flops"] / kms / 1e9}


def slowest_rank_ms(ms: float, dist=None, device=None) -> float:
    """Max over ranks of a per-step time (the job's step time)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ops_per_rank: float, ms: float, world: int) -> float:
    """Whole-job throughput in T(FL)OPS: every rank's operations over the
    slowest rank's step time (replicas: one copy of the workload per rank)."""
    return world * ops_per_rank / ms / 1e9


def run_gpu(args) -> int:
    import torch

    from software_pipelined_loop_gb300 import build, gemmpipe

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build.build()
    if dist:
        dist.barrier()
    gemmpipe.load()
    peaks, peak_src = load_peaks()
    # L2 flush between timed steps: write a buffer larger than L2, then read
    # another one, so the timed step starts with none of its data cached and
    # with clean lines (the write-back of the flush's own dirty lines is not
    # charged to the timed step).
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean_buf = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    flush_sink = torch.empty((), dtype=torch.int32, device=dev)

    def flush():
        flush_buf.zero_()
        torch.sum(clean_buf, dim=0, dtype=torch.int32, out=flush_sink)  # int32 in and out: a read, no cast

    clock = ClockSampler(local)
    clock.start()
    try:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        head = measure_gemm(workload(HEADLINE), args.steps, args.warmup, dev, flush, peaks, peak_src)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        clocks = clock.summary(*head["window"])
        if clocks["samples"] < 3:
            clocks["window"] = "whole GPU phase (timed region shorter than the sampling period)"
        secondary = []
        if not args.no_secondary:
            # Small cases first, the metric's FP16 4096^3 and skinny last.
            for wl in (workload(0), workload(1), workload(4), workload(3), fp16_4096()):
                secondary.append(measure_gemm(wl, max(10, args.steps // 4), args.warmup, dev, flush, peaks,
                                              peak_src))
        e2e = measure_e2e(head, max(5, args.steps // 4), dev)
        copy_ref = measure_copy_ref(dev, peaks)
        context = None
        if not args.no_secondary and world == 1:
            context = library_context(dev, flush, max(10, args.steps // 4))
            if head["dtype"] == "s8":
                context["int8_legacy_ceiling"] = legacy_int8_ceiling(head, dev, flush, 5)
    finally:
        clock.stop()

    ms = slowest_rank_ms(head["ms"], dist, dev)
    ms_median = slowest_rank_ms(head["ms_median"], dist, dev)
    value = job_throughput(head["flops"], ms, world)
    unit = "TOPS" if head["dtype"] == "s8" else "TFLOPS"
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    # Every timed output against the oracle's whole product (rank 0 at N = 1;
    # the replicas of other ranks compute the same C).
    parity, cpu = {}, None
    if world == 1 and not args.no_parity:
        for r in [head] + secondary:
            r["parity"] = parity_check(r)
            parity[r["name"]] = r["parity"]["verdict"]
        pc = head["parity"]
        cpu = {"value": pc["oracle_rate"], "unit": unit, "cores": pc["cores"], "kind": "oracle",
               "sample": f"the whole workload: all {head['M']} x {head['N']} elements of C, full K, "
                         f"{pc['oracle_s']:.1f} s",
               "parity": pc["verdict"]}

    int8_floor = None
    if head["dtype"] == "s8":
        # The step is the widening pass plus the GEMM kernel: with the pass
        # at the in-run copy rate, the step cannot beat this floor unless
        # the GEMM kernel itself gets faster.
        widen_bytes = 3 * (head["A"].nbytes + head["B"].nbytes)
        widen_ms = widen_bytes / copy_ref["gbs"] / 1e6
        int8_floor = {"widen_ms": head["aux_ms"], "widen_at_copy_rate_ms": widen_ms,
                      "kernel_ms": head["kernel_ms"], "floor_ms": widen_ms + head["kernel_ms"],
                      "step_ms": head["ms"], "step_frac": head["flops"] / head["ms"] / 1e9 / peaks["bf16_tflops"],
                      "kernel_frac": head["roofline"]["frac"]}
        if context and "int8_legacy_ceiling" in context:
            lc = context["int8_legacy_ceiling"]
            int8_floor["step_vs_legacy_ceiling"] = (head["flops"] / head["ms"] / 1e9) / lc["tops"]

    def brief(r):
        skinny = r["N"] <= 128
        unit = "GB/s" if skinny else ("TOPS" if r["dtype"] == "s8" else "TFLOPS")
        val = r["bytes_per_s"] if skinny else r["ops_per_s"]
        peak = r["roofline"]["peak"]
        out = {"value": round(val, 1), "unit": unit, "ms": round(r["ms"], 5), "kernel_ms": round(r["kernel_ms"], 5),
               "frac": round(r["roofline"]["frac"], 3), "step_frac": round(val / peak, 3),
               "traffic": r["roofline"]["traffic"]}
        if "parity" in r:
            out["parity"] = r["parity"]["verdict"]
            out["cpu"] = {"value": round(r["parity"]["oracle_rate"], 4), "unit": "TOPS" if r["dtype"] == "s8"
                          else "TFLOPS", "s": round(r["parity"]["oracle_s"], 2), "cores": r["parity"]["cores"]}
        return out

    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": ms_median,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": head["dtype"],
        "data": "synthetic",
        "config": bench_config(head["name"], head["M"], head["N"], head["K"], head["l2"]),
        "roofline": head["roofline"],
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": head["launches"],
        "clocks": clocks,
        "parity": parity or None,
        "kernel_ms": head["kernel_ms"], "aux_ms": head["aux_ms"],
        "plan": {k: head["plan"][k] for k in ("producer", "BM", "BN", "BK", "stages", "threads", "cta_pair", "grid",
                                              "units", "tiles", "split_tiles", "k_blocks", "operand_copy",
                                              "smem_bytes")},
        "copy_ref_gbs": round(copy_ref["gbs"], 1),
        "int8_step_floor": int8_floor,
        "library_context": context,
        "secondary": {r["name"]: brief(r) for r in secondary},
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def bench_config(name: str, M: int, N: int, K: int, l2: str) -> dict:
    """The `config` object of both arms' lines (the same workload)."""
    return {"workload": name, "M": M, "N": N, "K": K,
            "l2": l2 + " (between timed steps: 256 MiB written, then another 256 MiB read, when inputs < L2)"}


def fp16_4096():
    """FP16 4096^3, operands uniform on [-1, 1]: the fp16 half of the metric."""
    from software_pipelined_loop_gb300 import inputs
    A, B = inputs.make_operands("f16", 4096, 4096, 4096, inputs.SEED_BASE + 5)
    return ("fp16_4096", "f16", 4096, 4096, 4096, A, B)


SQUARE = (4096, 4096, 4096)
RAGGED = (4093, 3001, 4107)
SKINNY = (16384, 128, 16384)
ABLATION = [
    # (label, dtype, shape, producer, bn, stages, cta_pair, split[, k per stage])
    ("pair S=1 (load, wait, compute)", "f16", SQUARE, 0, 256, 1, 1, -1),
    ("pair S=2 (double buffer)", "f16", SQUARE, 0, 256, 2, 1, -1),
    ("pair S=3", "f16", SQUARE, 0, 256, 3, 1, -1),
    ("pair S=4", "f16", SQUARE, 0, 256, 4, 1, -1),
    ("pair S=5", "f16", SQUARE, 0, 256, 5, 1, -1),
    ("pair S=6 (default)", "f16", SQUARE, 0, 256, 6, 1, -1),
    ("pair, 128 k per stage, S=3", "f16", SQUARE, 0, 256, 0, 1, -1, 128),
    ("pair S=6, every tile whole (no stream-K)", "f16", SQUARE, 0, 256, 6, 1, 0),
    ("single CTA 128x256 S=4", "f16", SQUARE, 0, 256, 4, 0, -1),
    ("single CTA 128x128 S=6", "f16", SQUARE, 0, 128, 6, 0, -1),
    ("single CTA bounded-load producer 128x256 S=4", "f16", SQUARE, 1, 256, 4, 0, -1),
    ("int8: widening pass + pair (default)", "s8", SQUARE, -1, 0, 0, -1, -1),
    ("int8: widening pass + pair, every tile whole", "s8", SQUARE, -1, 0, 0, -1, 0),
    ("int8: in-kernel widening, pair", "s8", SQUARE, 0, 256, 4, 1, -1),
    ("int8: in-kernel widening, single CTA", "s8", SQUARE, 0, 256, 2, 0, -1),
    ("int8: the pages' design: mma.sync m16n8k32 + 4-stage cp.async ring", "s8", SQUARE, 2, 0, 0, -1, -1),
    ("int8: the pages' design with their double buffer (S=2)", "s8", SQUARE, 2, 0, 2, -1, -1),
    ("ragged fp16: stream-K (default)", "f16", RAGGED, -1, 0, 0, -1, -1),
    ("ragged fp16: every tile whole", "f16", RAGGED, -1, 0, 0, -1, 0),
    ("skinny fp16: TMA producer (default)", "f16", SKINNY, -1, 0, 0, -1, -1),
    ("skinny fp16: stream-K forced on all 152 SMs", "f16", SKINNY, -1, 0, 0, -1, 1),
    ("skinny fp16: bounded-load producer", "f16", SKINNY, 1, 128, 6, 0, -1),
]


def run_ablation(args) -> int:
    """Ring depth, producer and stream-K ablation (one JSON line)."""
    import torch

    from software_pipelined_loop_gb300 import build, gemmpipe, inputs
    build.build()
    gemmpipe.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean_buf = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    sink = torch.empty((), dtype=torch.int32, device=dev)

    def flush():
        flush_buf.zero_()
        torch.sum(clean_buf, dim=0, dtype=torch.int32, out=sink)

    ops = {}
    rows = []
    for label, dt, shape, producer, bn, stages, pair, split, *rest in ABLATION:
        bk = rest[0] if rest else 0  # k per stage (0: the planner's choice)
        M, N, K = shape
        if (dt, shape) not in ops:
            A, B = inputs.make_operands(dt, M, N, K, inputs.SEED_BASE + 5)
            ops[(dt, shape)] = (torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev),
                                torch.empty((M, N), dtype=torch.int32 if dt == "s8" else torch.float32,
                                            device=dev))
        Ad, Bd, C = ops[(dt, shape)]
        fn = gemmpipe.gemm_s8s8s32 if dt == "s8" else gemmpipe.gemm_f16f32
        stream = torch.cuda.current_stream(dev)
        gemmpipe.gemmpipe_set_plan_override(producer, bn, stages, pair, split)
        gemmpipe.gemmpipe_set_plan_bk(bk)
        try:
            plan = gemmpipe.gemmpipe_plan(0 if dt == "s8" else 1, M, N, K, Ad, Bd, C)
            call = lambda: fn(M, N, K, Ad, Bd, C, stream)
            for _ in range(max(3, args.warmup)):
                call()
            torch.cuda.synchronize()
            gemmpipe.gemmpipe_timing_read()
            gemmpipe.gemmpipe_timing_enable(True)
            times = time_steps(call, max(5, args.steps // 10), flush, stream)
            gms, gn, ams, an = gemmpipe.gemmpipe_timing_read()
            gemmpipe.gemmpipe_timing_enable(False)
        finally:
            gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
            gemmpipe.gemmpipe_set_plan_bk(0)
        st = gemmpipe.gemmpipe_get_device_status(stream)
        ms = statistics.mean(times)
        kms = gms / max(1, gn)
        rows.append({"config": label, "shape": list(shape), "ms_per_step": ms,
                     "per_step": 2.0 * M * N * K / ms / 1e9, "kernel_ms": kms,
                     "per_kernel": 2.0 * M * N * K / kms / 1e9, "status": st,
                     "plan": {k: plan[k] for k in ("producer", "BM", "BN", "BK", "stages", "cta_pair", "units",
                                                   "split_tiles", "operand_copy")}})
    base = rows[0]["ms_per_step"]
    for r in rows:
        r["speedup_vs_S1"] = base / r["ms_per_step"] if r["shape"] == list(SQUARE) and r["plan"]["cta_pair"] \
            and r["config"].startswith("pair") else None
    print(json.dumps({"ablation": "ring depth, producer and stream-K", "unit": "TFLOPS or TOPS",
                      "rows": rows}), flush=True)
    return 0


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-parity", "--no-cpu-baseline", dest="no_parity", action="store_true",
                    help="skip the whole-C oracle comparison (and with it the CPU baselines)")
    ap.add_argument("--ref-seconds", type=float, default=None,
                    help="CPU seconds per reference step (default: 4, or 120 / steps when that is less)")
    ap.add_argument("--shape", default=None,
                    help="time dtype,M,N,K (s8 or f16) as the headline instead of INT8 4096^3 "
                         "(for profiling and sweeps; uniform inputs)")
    ap.add_argument("--force", default=None,
                    help="plan override producer,bn,stages[,cta_pair[,split]] (see gemmpipe_set_plan_override)")
    ap.add_argument("--ablation", action="store_true",
                    help="ring-depth / producer ablation at 4096^3 instead of the benchmark line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.shape:
        global SHAPE
        dt, M, N, K = args.shape.split(",")
        if dt not in ("s8", "f16"):
            ap.error("--shape dtype must be s8 or f16")
        SHAPE = (dt, int(M), int(N), int(K))
    if args.force:
        from software_pipelined_loop_gb300 import build, gemmpipe
        build.build()
        gemmpipe.gemmpipe_set_plan_override(*[int(x) for x in args.force.split(",")])
    if args.impl == "reference":
        return run_reference(args)
    if args.ablation:
        return run_ablation(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
