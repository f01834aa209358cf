"""The bottleneck report's arithmetic and decision logic (no GPU): the
classification and occupancy steps of the "Analyze Kernel Bottleneck" page
redone with GB300 limits, checked on the workloads' own shapes."""
import json

import pytest

from software_pipelined_loop_gb300 import report

PAIR_PLAN = {"producer": 0, "BM": 256, "BN": 256, "BK": 64, "stages": 6, "threads": 384, "cta_pair": 1,
             "grid": 152, "units": 76, "tiles": 256, "split_tiles": 104, "k_blocks": 64, "smem_bytes": 230552,
             "operand_copy": 0}
SKINNY_PLAN = dict(PAIR_PLAN, BM=128, BN=128, cta_pair=0, grid=128, units=128, tiles=128, split_tiles=0,
                   k_blocks=256)


def launch(dtype="f16", shape=(4096, 4096, 4096), kernel_ms=0.0906, plan=PAIR_PLAN, **kw):
    M, N, K = shape
    return report.Launch(name="t", dtype=dtype, M=M, N=N, K=K, kernel_ms=kernel_ms, plan=dict(plan),
                         peak_tflops=1917.5, peak_gbs=6785.2, **kw)


def test_baseline_and_roofline_match_the_workload_table():
    # FP16 4096^3: 2*4096^3 flops over A, B (fp16) and C (fp32) once: AI 1024;
    # INT8 4096^3 over int8 operands: AI 1365.3; skinny: 125.1; balance 282.6.
    L = launch()
    b = report.baseline(L)
    assert b["flops"] == 2 * 4096 ** 3 and b["alg_bytes"] == 134217728
    r = report.roofline(L, b)
    assert r["ai"] == pytest.approx(1024.0) and r["balance"] == pytest.approx(282.6, abs=0.05)
    assert r["bound"] == r["class"] == "compute"
    assert r["attained"] == pytest.approx(2 * 4096 ** 3 / 0.0906e-3 / 1917.5e12)
    r8 = report.roofline(launch("s8"), report.baseline(launch("s8")))
    assert r8["ai"] == pytest.approx(2 * 4096 ** 3 / 100663296)
    sk = launch(shape=(16384, 128, 16384), kernel_ms=0.1027, plan=SKINNY_PLAN)
    rs = report.roofline(sk, report.baseline(sk))
    assert rs["ai"] == pytest.approx(125.07, abs=0.01) and rs["bound"] == "memory"
    assert rs["attained"] == pytest.approx(549453824 / 0.1027e-3 / 6785.2e9)


def test_latency_bound_when_neither_ceiling_is_near():
    L = launch(shape=(512, 512, 512), kernel_ms=0.010)
    r = report.roofline(L, report.baseline(L))
    assert r["bound"] == "memory" and r["class"] == "latency"


def test_occupancy_limits():
    # 384 threads x 168 registers = 64512 of 65536: one block; 225 KiB of
    # shared memory: one block; 12 warps: five blocks; the limit is one.
    o = report.occupancy(launch(regs_per_thread=168))
    assert o["limits"] == {"registers": 1, "shared memory": 1, "warps": 5, "blocks": 32}
    assert o["blocks_per_sm"] == 1 and set(o["limiting"]) == {"registers", "shared memory"}
    assert o["active_warps"] == 12 and o["enough"]
    small = report.occupancy(launch(plan=dict(PAIR_PLAN, threads=128, smem_bytes=4096)))
    assert small["limits"]["shared memory"] == 57 and small["blocks_per_sm"] == 16
    assert small["active_warps"] == 64


def test_compute_load_ratios():
    # Pages' per-tile flops per byte: 2*BM*BN*BK / ((BM*BK + BK*BN) * 2).
    c = report.compute_load(launch())
    assert c["flop_per_byte"] == pytest.approx(128.0)
    # Pair: 4 tcgen05.mma (K = 16) per 64-deep k-block against 2 x (1 A box +
    # one 3-D B box) TMA copies: 1:1, low -> asynchronous loads pay.
    assert (c["mma_per_kblock"], c["copies_per_kblock"]) == (4, 4) and c["class"] == "low"
    # N not a multiple of 64: B as two 64-column 2-D boxes per CTA.
    r = report.compute_load(launch(shape=(4093, 3001, 4107)))
    assert r["copies_per_kblock"] == 6
    # 128 k per stage: 8 MMAs against 2 x (2 A boxes + one 3-D B box).
    b = report.compute_load(launch(plan=dict(PAIR_PLAN, BK=128, stages=3)))
    assert (b["mma_per_kblock"], b["copies_per_kblock"]) == (8, 6)
    # Quad (256 x 512 tile): each pair issues its 4 MMAs; 4 CTAs x (1 A box + 1 B box).
    q = report.compute_load(launch(plan=dict(PAIR_PLAN, BN=512, cta_pair=2)))
    assert (q["mma_per_kblock"], q["copies_per_kblock"]) == (8, 8)
    s = report.compute_load(launch(plan=SKINNY_PLAN))
    assert s["flop_per_byte"] == pytest.approx(64.0) and s["copies_per_kblock"] == 3
    ldg = report.compute_load(launch(plan=dict(SKINNY_PLAN, producer=1)))
    assert ldg["copy_unit"] == "16-byte load" and ldg["copies_per_kblock"] == (128 * 64 + 64 * 128) * 2 // 16


def test_counters_and_recommendations():
    counters = {
        "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active": "73.3",
        "sm__cycles_active.avg": "150497", "gpc__cycles_elapsed.max": "167177",
        "dram__bytes_read.sum": "86.2", "dram__bytes_write.sum": "47.7",
        "__units__": {"dram__bytes_read.sum": "Mbyte", "dram__bytes_write.sum": "Mbyte"},
        "smsp__average_warps_issue_stalled_long_scoreboard_per_issue_active.ratio": "11.2",
        "smsp__average_warps_issue_stalled_barrier_per_issue_active.ratio": "5.4",
    }
    L = launch(counters=counters, regs_per_thread=168)
    b = report.baseline(L)
    cv = report.counter_view(L, b)
    assert cv["tensor_active_pct"] == pytest.approx(73.3)
    assert cv["sm_active_frac"] == pytest.approx(150497 / 167177)
    assert cv["dram_bytes"] == pytest.approx(133.9e6) and cv["dram_over_alg"] == pytest.approx(133.9e6 / 134217728)
    assert [n for _, n in cv["stalls"]] == ["long_scoreboard", "barrier"]
    recs = report.recommend(L, report.roofline(L, b), report.compute_load(L), report.occupancy(L), cv)
    gains = [g for g, _, _ in recs]
    assert gains == sorted(gains, reverse=True) and len(recs) == 2
    assert "tensor pipe" in recs[0][1] and "last wave" in recs[1][1]
    text = report.render(L)
    for h in ("### Baseline", "### Roofline Classification", "### Occupancy", "### Compute/Load Ratio",
              "### Counters", "### Smem Cliff", "### Recommended Optimizations"):
        assert h in text


def test_parse_raw_csv_and_bench_line(tmp_path):
    csv_text = ('"ID","Kernel Name","launch__registers_per_thread","dram__bytes_read.sum"\n'
                '"","","register/thread","Mbyte"\n'
                '"0","gemm","168","85.6"\n')
    c = report.parse_ncu_raw_csv(csv_text)
    assert c["launch__registers_per_thread"] == "168" and c["dram__bytes_read.sum"] == "85.6"
    assert c["__units__"]["dram__bytes_read.sum"] == "Mbyte"
    line = {"dtype": "s8", "kernel_ms": 0.0907, "ms_per_step": 0.1027, "plan": PAIR_PLAN,
            "config": {"workload": "int8_4096", "M": 4096, "N": 4096, "K": 4096},
            "roofline": {"traffic": None},
            "secondary": {"fp16_skinny": {"shape": [16384, 128, 16384], "dtype": "f16", "plan": SKINNY_PLAN,
                                          "kernel_ms": 0.1027, "ms_per_step": 0.1023, "roofline": {}}}}
    L = report.launch_from_bench(line, None, (1917.5, 6785.2, "measured"))
    assert (L.name, L.dtype, L.M, L.step_ms) == ("int8_4096", "s8", 4096, 0.1027)
    S = report.launch_from_bench(line, "fp16_skinny", (1917.5, 6785.2, "measured"))
    assert (S.N, S.plan["BN"]) == (128, 128)
    # Secondary entries of the compact line carry no plan: refused with a hint.
    line["secondary"]["fp16_1024"] = {"value": 150.0, "unit": "TFLOPS", "ms": 0.014}
    with pytest.raises(SystemExit, match="--shape"):
        report.launch_from_bench(line, "fp16_1024", (1917.5, 6785.2, "measured"))
    p = tmp_path / "b.json"
    p.write_text("noise\n" + json.dumps(line) + "\n")
    q = tmp_path / "raw.csv"
    q.write_text(csv_text)
    assert report.main(["--bench", str(p), "--ncu-csv", str(q)]) == 0


def test_balance_points_match_the_pages_ga104_table():
    # The page's worked example: GA104 peaks over 608 GB/s (tests/golden).
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "ga104_balance_points.json")))
    for row in g["peaks"]:
        L = report.Launch(name="ga104", dtype="f16", M=4096, N=4096, K=4096, kernel_ms=1.0, plan=dict(PAIR_PLAN),
                          peak_tflops=row["peak_gflops"] / 1e3, peak_gbs=g["dram_gbs"])
        r = report.roofline(L, report.baseline(L))
        assert round(r["balance"], 1) == row["balance"], row["precision"]
    # The page's effective-throughput formula at 4096^3 and 1 ms.
    b = report.baseline(launch(kernel_ms=1.0))
    assert b["tflops"] * 1e3 == pytest.approx(2 * 4096 ** 3 / (1.0 / 1000) / 1e9)
