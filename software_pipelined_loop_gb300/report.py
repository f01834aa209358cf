"""Bottleneck report for one libgemmpipe GEMM launch.

Follows the analysis steps and the report layout of the "Analyze Kernel
Bottleneck" skill page (Steps 1-8 and its report template), redone for
GB300:

* Step 1, baseline: kernel time from CUDA events, effective throughput
  2*M*N*K / t and effective bandwidth = algorithmic bytes / t.
* Step 2, roofline: arithmetic intensity over the unique DRAM bytes (A and
  B read once, C written once), the machine balance = peak compute / peak
  bandwidth, the class (compute-, memory- or latency-bound) and the
  attained fraction of the relevant peak.
* Step 3, occupancy: blocks per SM under each resource limit (registers,
  shared memory, warps, blocks), the limiting one and the active warps.
* Step 4, compute/load ratio: the pages' per-tile flops-per-byte helper and
  the per-k-block ratio of tensor instructions to copy instructions, which
  this library knows from its plan (the pages count them in SASS, which is
  not read here) -- classified with the pages' 5:1 / 20:1 thresholds.
* Step 5, instruction mix and stalls: replaced by ncu counters (tensor-pipe
  activity, SM activity, DRAM and L2 bytes, warp stall reasons) when a raw
  ncu CSV is given.
* Step 6, shared-memory cliff: per-block shared memory against the per-SM
  capacity.
* Step 7, decision matrix: ranked recommendations with a gain estimate from
  the distance to the relevant ceiling.

    python -m software_pipelined_loop_gb300.report --bench bench_line.json \
        [--workload fp16_4096] [--ncu-csv raw.csv]

`--bench` takes the JSON line `bench.py` prints; `--ncu-csv` the output of
`ncu -i <report> --page raw --csv` for the same kernel.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import sys
from dataclasses import dataclass, field

# GB300 (sm_103) per-SM limits; the occupancy formulas are the page's.
GB300_LIMITS = {
    "sms": 152,
    "regs_per_sm": 65536,
    "smem_per_sm": 233472,      # 228 KiB, of which a CTA may take 227 KiB
    "smem_per_block": 232448,
    "warps_per_sm": 64,
    "blocks_per_sm": 32,
}
# The profiling recipe's fallback when no measured peaks are at hand.
FALLBACK_PEAKS = {"tflops": 1900.0, "gbs": 6800.0, "source": "fallback"}
# The page's thresholds on the compute/load ratio (Step 4).
RATIO_LOW, RATIO_HIGH = 5.0, 20.0
# The page's latency-hiding threshold (GA104: 8 warps per SM).
WARPS_ENOUGH = 8


@dataclass
class Launch:
    """What the report needs about one GEMM launch."""
    name: str
    dtype: str                 # "s8" or "f16"
    M: int
    N: int
    K: int
    kernel_ms: float
    plan: dict
    peak_tflops: float
    peak_gbs: float
    peak_source: str = "measured"
    step_ms: float | None = None
    traffic: int | None = None          # DRAM bytes per launch, if captured
    regs_per_thread: int | None = None
    counters: dict = field(default_factory=dict)   # ncu metric name -> value


# ------------------------------------------------------------------ steps

def baseline(L: Launch) -> dict:
    """Step 1: effective throughput and bandwidth of the kernel."""
    flops = 2.0 * L.M * L.N * L.K
    operand = 1 if L.dtype == "s8" else 2  # the caller's operands, read once
    alg_bytes = operand * (L.M * L.K + L.K * L.N) + 4 * L.M * L.N
    t = L.kernel_ms / 1e3
    return {"flops": flops, "alg_bytes": alg_bytes, "tflops": flops / t / 1e12, "gbs": alg_bytes / t / 1e9}


def roofline(L: Launch, base: dict) -> dict:
    """Step 2: arithmetic intensity, balance point, class, attained fraction."""
    ai = base["flops"] / base["alg_bytes"]
    balance = L.peak_tflops * 1e12 / (L.peak_gbs * 1e9)
    bound = "compute" if ai >= balance else "memory"
    attained = base["tflops"] / L.peak_tflops if bound == "compute" else base["gbs"] / L.peak_gbs
    cls = bound
    # Neither ceiling near: the page calls this latency-bound.
    if attained < 0.5:
        cls = "latency"
    return {"ai": ai, "balance": balance, "bound": bound, "class": cls, "attained": attained}


def occupancy(L: Launch, limits: dict = GB300_LIMITS) -> dict:
    """Step 3: blocks per SM under each limit and active warps per SM."""
    threads = int(L.plan["threads"])
    warps = threads // 32
    smem = int(L.plan["smem_bytes"])
    out = {"threads": threads, "warps_per_block": warps, "smem_per_block": smem}
    lim = {}
    if L.regs_per_thread:
        lim["registers"] = limits["regs_per_sm"] // (L.regs_per_thread * threads)
    lim["shared memory"] = limits["smem_per_sm"] // smem if smem else limits["blocks_per_sm"]
    lim["warps"] = limits["warps_per_sm"] // warps
    lim["blocks"] = limits["blocks_per_sm"]
    blocks = min(lim.values())
    limiting = [k for k, v in lim.items() if v == blocks]
    out.update({"limits": lim, "blocks_per_sm": blocks, "limiting": limiting,
                "active_warps": blocks * warps, "enough": blocks * warps >= WARPS_ENOUGH})
    return out


def compute_load(L: Launch) -> dict:
    """Step 4: the per-tile flops-per-byte ratio and the per-k-block ratio
    of tensor instructions to copy instructions."""
    BM, BN, BK = int(L.plan["BM"]), int(L.plan["BN"]), int(L.plan["BK"])
    elem = 2  # the tensor cores read fp16 (INT8 operands are widened)
    flop_per_byte = 2.0 * BM * BN * BK / ((BM * BK + BK * BN) * elem)
    # CTAs per tile: 1 (single CTA), 2 (CTA pair), 4 (quad: two pairs).
    ctas = {0: 1, 1: 2, 2: 4}[int(L.plan.get("cta_pair", 0))]
    pairs = max(1, ctas // 2)
    # One MMA instruction covers a pair's (or a single CTA's) tile columns
    # up to N = 256 for K = 16 (cta_group::2 for a pair: one instruction for
    # both CTAs); a quad's two pairs issue their own.
    mma = pairs * (BK // 16) * max(1, BN // pairs // 256)
    # Copy instructions per CTA: A as 64-k boxes (a quad's CTA loads half of
    # its rows and multicasts them), B as 64-column boxes of BK rows, or one
    # 3-D box per MMA when N is a multiple of 64 on pairs; the bounded-load
    # producer issues 16-byte loads instead.
    cta_bn = BN // ctas
    if int(L.plan.get("producer", 0)) == 0:
        a_boxes = BK // 64
        b_boxes = max(1, BN // pairs // 256) if ctas > 1 and L.N % 64 == 0 else cta_bn // 64
        copies = ctas * (a_boxes + b_boxes)
        copy_unit = "TMA box"
    else:
        copies = ctas * ((128 * BK + BK * cta_bn) * elem // 16)
        copy_unit = "16-byte load"
    ratio = mma / copies
    cls = "high" if ratio > RATIO_HIGH else ("medium" if ratio >= RATIO_LOW else "low")
    advice = {"low": "asynchronous loads strongly beneficial (loads dominate the issue stream)",
              "medium": "asynchronous loads may help: benchmark both",
              "high": "asynchronous loads net negative: warp interleaving already hides DRAM latency"}[cls]
    return {"flop_per_byte": flop_per_byte, "mma_per_kblock": mma, "copies_per_kblock": copies,
            "copy_unit": copy_unit, "ratio": ratio, "class": cls, "advice": advice}


def smem_cliff(L: Launch, occ: dict, limits: dict = GB300_LIMITS) -> dict:
    """Step 6: shared memory per block against the per-SM capacity."""
    smem = occ["smem_per_block"]
    return {"smem_per_block": smem, "per_sm": limits["smem_per_sm"], "blocks_per_sm": occ["blocks_per_sm"],
            "over_half": smem > limits["smem_per_sm"] // 2}


def counter_view(L: Launch, base: dict) -> dict:
    """Step 5 replacement: the ncu counters that locate the time."""
    c = L.counters
    if not c:
        return {}

    def num(k):
        v = c.get(k)
        try:
            return float(str(v).replace(",", ""))
        except (TypeError, ValueError):
            return None

    out = {}
    ta = num("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active")
    if ta is not None:
        out["tensor_active_pct"] = ta
    sa, el = num("sm__cycles_active.avg"), num("gpc__cycles_elapsed.max")
    if sa and el:
        out["sm_active_frac"] = sa / el
    rd, wr = num("dram__bytes_read.sum"), num("dram__bytes_write.sum")
    if rd is not None and wr is not None:
        units = c.get("__units__", {})
        scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
        rd *= scale.get(units.get("dram__bytes_read.sum", "byte"), 1.0)
        wr *= scale.get(units.get("dram__bytes_write.sum", "byte"), 1.0)
        out["dram_bytes"] = rd + wr
        out["dram_over_alg"] = out["dram_bytes"] / base["alg_bytes"]
    l2 = num("l1tex__m_xbar2l1tex_read_bytes.sum.pct_of_peak_sustained_elapsed")
    if l2 is not None:
        out["l2_to_sm_pct"] = l2
    tc = num("l1tex__data_pipe_tc_wavefronts_mem_shared.sum.pct_of_peak_sustained_elapsed")
    if tc is not None:
        out["smem_tensor_read_pct"] = tc
    stalls = []
    pre, suf = "smsp__average_warps_issue_stalled_", "_per_issue_active.ratio"
    for k in c:
        if k.startswith(pre) and k.endswith(suf):
            v = num(k)
            if v:
                stalls.append((v, k[len(pre):-len(suf)]))
    out["stalls"] = sorted(stalls, reverse=True)[:5]
    return out


def recommend(L: Launch, roof: dict, cl: dict, occ: dict, cnt: dict) -> list[tuple[float, str, str]]:
    """Step 7: the decision matrix, ranked by estimated gain (fraction)."""
    recs = []
    ceiling_gap = max(0.0, 1.0 / max(roof["attained"], 1e-9) - 1.0)
    if roof["bound"] == "memory" and cl["class"] == "low":
        recs.append((min(ceiling_gap, 1.0), "Deepen the load pipeline (more ring stages, asynchronous copies)",
                     "memory-bound with a low compute/load ratio: overlapping loads with math is the page's "
                     "first remedy"))
    if roof["bound"] == "memory" and cl["class"] == "high":
        recs.append((min(ceiling_gap, 0.5), "Change the algorithm's data movement (fewer bytes per result)",
                     "memory-bound while loads are already hidden"))
    if roof["bound"] == "compute":
        ta = cnt.get("tensor_active_pct")
        if ta is not None and ta < 90.0:
            recs.append((min(0.9 / (ta / 100.0) - 1.0, ceiling_gap), "Feed the tensor pipe: larger tiles "
                         "(CTA pairs), longer k-loops per accumulator, fewer epilogue stalls",
                         f"the tensor pipe is busy {ta:.0f}% of active cycles"))
    sm = cnt.get("sm_active_frac")
    if sm is not None and sm < 0.95:
        recs.append((1.0 / sm - 1.0, "Balance the last wave (stream-K split of the tail tiles) and shorten "
                     "set-up and teardown", f"SMs are active {100 * sm:.0f}% of the kernel's cycles"))
    over = cnt.get("dram_over_alg")
    if over is not None and over > 1.2 and roof["bound"] == "memory":
        recs.append((over - 1.0, "Remove DRAM re-reads (tile order for L2 reuse, fusion)",
                     f"DRAM traffic is {over:.2f}x the algorithmic bytes"))
    if not occ["enough"] and int(L.plan.get("producer", 0)) != 0:
        recs.append((0.2, "Raise resident warps (fewer registers or less shared memory per block)",
                     f"{occ['active_warps']} warps per SM, below the page's {WARPS_ENOUGH}"))
    if roof["class"] == "latency":
        recs.append((ceiling_gap, "More work per launch (batch calls, larger problems) or fewer launches",
                     "neither ceiling is near: launch and latency bound"))
    recs.sort(key=lambda r: -r[0])
    return recs


# ---------------------------------------------------------------- render

def render(L: Launch) -> str:
    base = baseline(L)
    roof = roofline(L, base)
    occ = occupancy(L)
    cl = compute_load(L)
    sm = smem_cliff(L, occ)
    cnt = counter_view(L, base)
    recs = recommend(L, roof, cl, occ, cnt)
    unit = "TOPS" if L.dtype == "s8" else "TFLOPS"
    lines = [f"## Bottleneck Analysis Report: {L.name}", "", "### Baseline",
             f"- Problem: M={L.M}, N={L.N}, K={L.K} ({'int8 x int8 -> int32' if L.dtype == 's8' else 'fp16 x fp16 -> fp32'})",
             f"- Kernel time: {L.kernel_ms:.4f} ms (CUDA events)"
             + (f"; whole step {L.step_ms:.4f} ms" if L.step_ms else ""),
             f"- Effective {unit}: {base['tflops']:.1f} | Effective bandwidth: {base['gbs']:.1f} GB/s "
             f"of algorithmic bytes ({base['alg_bytes'] / 1e6:.1f} MB)", "",
             "### Roofline Classification",
             f"- Arithmetic intensity: {roof['ai']:.1f} FLOP/byte",
             f"- Balance point: {roof['balance']:.1f} FLOP/byte ({L.peak_tflops:.1f} TFLOP/s over "
             f"{L.peak_gbs:.1f} GB/s, {L.peak_source})",
             f"- Classification: **{roof['class']}-bound**"
             + (f" (intensity says {roof['bound']}-bound)" if roof["class"] != roof["bound"] else ""),
             f"- Attained fraction: {100 * roof['attained']:.1f}% of the "
             f"{'tensor' if roof['bound'] == 'compute' else 'HBM'} peak", "",
             "### Occupancy", "| Resource | Per Block | Limit/SM | Blocks/SM |", "|---|---|---|---|"]
    lim = occ["limits"]
    if "registers" in lim:
        lines.append(f"| Registers | {L.regs_per_thread}/thread x {occ['threads']} | {GB300_LIMITS['regs_per_sm']} "
                     f"| {lim['registers']} |")
    lines += [f"| Shared mem | {occ['smem_per_block'] / 1024:.1f} KiB | {GB300_LIMITS['smem_per_sm'] / 1024:.0f} KiB "
              f"| {lim['shared memory']} |",
              f"| Warps | {occ['warps_per_block']} | {GB300_LIMITS['warps_per_sm']} | {lim['warps']} |",
              f"| Blocks | 1 | {GB300_LIMITS['blocks_per_sm']} | {lim['blocks']} |",
              f"| **Limiting** | {', '.join(occ['limiting'])} | | **{occ['blocks_per_sm']}** |",
              f"- Active warps/SM: {occ['active_warps']} ("
              + ("sufficient" if occ["enough"] else "below the page's 8") + " for latency hiding; the kernel is "
              "warp-specialised, its loads are asynchronous TMA copies tracked by mbarriers)", "",
              "### Compute/Load Ratio",
              f"- Per-tile flops per byte (BM={L.plan['BM']}, BN={L.plan['BN']}, BK={L.plan['BK']}, fp16): "
              f"{cl['flop_per_byte']:.1f}",
              f"- Tensor instructions per k-block: {cl['mma_per_kblock']} (tcgen05.mma, K = 16 each)",
              f"- Copy instructions per k-block: {cl['copies_per_kblock']} ({cl['copy_unit']})",
              f"- Ratio: {cl['ratio']:.2f}:1 -- **{cl['class']}**",
              f"- Recommendation: {cl['advice']}", ""]
    lines.append("### Counters (in place of the SASS instruction mix)")
    if cnt:
        if "tensor_active_pct" in cnt:
            lines.append(f"- Tensor pipe active: {cnt['tensor_active_pct']:.1f}% of SM-active cycles")
        if "sm_active_frac" in cnt:
            lines.append(f"- SMs active: {100 * cnt['sm_active_frac']:.1f}% of elapsed cycles")
        if "dram_bytes" in cnt:
            lines.append(f"- DRAM traffic: {cnt['dram_bytes'] / 1e6:.1f} MB "
                         f"({cnt['dram_over_alg']:.2f}x the algorithmic bytes)")
        if "l2_to_sm_pct" in cnt:
            lines.append(f"- L2 -> SM bytes: {cnt['l2_to_sm_pct']:.1f}% of peak")
        if "smem_tensor_read_pct" in cnt:
            lines.append(f"- Tensor-core shared-memory reads: {cnt['smem_tensor_read_pct']:.1f}% of peak")
        if cnt.get("stalls"):
            lines.append("- Top warp stalls (per issue): "
                         + ", ".join(f"{n} {v:.2f}" for v, n in cnt["stalls"]))
    else:
        lines.append("- no ncu counters given (`--ncu-csv`)")
    lines += ["", "### Smem Cliff",
              f"- Smem/block: {sm['smem_per_block'] / 1024:.1f} KiB of {sm['per_sm'] / 1024:.0f} KiB per SM -- "
              + ("over half the SM: one block per SM by design (the ring depth is traded against tile size)"
                 if sm["over_half"] else "room for more than one block per SM"),
              f"- Blocks/SM: {sm['blocks_per_sm']}", "", "### Recommended Optimizations (ranked)"]
    if recs:
        for i, (g, what, why) in enumerate(recs, 1):
            lines.append(f"{i}. {what} -- estimated up to {100 * g:.0f}% ({why})")
    else:
        lines.append("1. none: within 10% of the relevant ceiling")
    return "\n".join(lines) + "\n"


# ------------------------------------------------------------------- I/O

def parse_ncu_raw_csv(text: str) -> dict:
    """First data row of `ncu --page raw --csv` as {metric: value}, with the
    units row under the key "__units__"."""
    rows = list(csv.reader(io.StringIO(text)))
    rows = [r for r in rows if r and not r[0].startswith("==")]
    if len(rows) < 3:
        return {}
    out = dict(zip(rows[0], rows[2]))
    out["__units__"] = dict(zip(rows[0], rows[1]))
    return out


def load_peaks(root: str) -> tuple[float, float, str]:
    try:
        with open(os.path.join(root, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_PEAKS["tflops"], FALLBACK_PEAKS["gbs"], FALLBACK_PEAKS["source"]


def launch_from_bench(line: dict, workload: str | None, peaks: tuple[float, float, str]) -> Launch:
    """The headline (or a named secondary workload) of a bench JSON line."""
    if workload is None or workload == line["config"]["workload"]:
        cfg = line["config"]
        name, dtype, M, N, K = cfg["workload"], line["dtype"], cfg["M"], cfg["N"], cfg["K"]
        plan = line["plan"] if "plan" in line else cfg["plan"]
        kms, step = line["kernel_ms"], line["ms_per_step"]
        traffic = line["roofline"].get("traffic")
    else:
        sec = line["secondary"][workload]
        if "plan" not in sec:
            raise SystemExit(f"the bench line's entry for {workload} carries no plan: run "
                             f"bench.py --shape <dtype>,M,N,K for that shape and report its headline")
        name, dtype = workload, sec.get("dtype", "f16")
        M, N, K = sec["shape"]
        plan, kms, step = sec["plan"], sec["kernel_ms"], sec["ms_per_step"]
        traffic = sec["roofline"].get("traffic")
    return Launch(name=name, dtype=dtype, M=M, N=N, K=K, kernel_ms=kms, plan=plan, peak_tflops=peaks[0],
                  peak_gbs=peaks[1], peak_source=peaks[2], step_ms=step, traffic=traffic)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--bench", required=True, help="file holding bench.py's JSON line")
    ap.add_argument("--workload", default=None, help="secondary workload name (default: the headline)")
    ap.add_argument("--ncu-csv", default=None, help="ncu -i <report> --page raw --csv output for the kernel")
    ap.add_argument("--regs", type=int, default=None, help="registers per thread at launch (else from ncu)")
    args = ap.parse_args(argv)
    with open(args.bench) as f:
        text = [ln for ln in f.read().splitlines() if ln.strip().startswith("{")]
    line = json.loads(text[-1])
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    L = launch_from_bench(line, args.workload, load_peaks(root))
    if args.ncu_csv:
        with open(args.ncu_csv) as f:
            L.counters = parse_ncu_raw_csv(f.read())
        regs = L.counters.get("launch__registers_per_thread")
        if regs and not args.regs:
            L.regs_per_thread = int(float(regs))
    if args.regs:
        L.regs_per_thread = args.regs
    sys.stdout.write(render(L))
    return 0


if __name__ == "__main__":
    sys.exit(main())
