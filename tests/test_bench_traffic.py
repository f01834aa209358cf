"""The captured-traffic table of bench.py on CPU.

`roofline.traffic` in a bench line is the DRAM bytes of one ncu capture of
the timed kernel, valid only for the kernel sources it was captured at.  The
table is keyed by the plan's shape and carries a hash of the sources' code
(comments and blank space left out).  These tests check that a comment-only
edit keeps the hash, that a code edit changes it, and that the bench reports
the captured bytes only while the hash matches.
"""
from __future__ import annotations

import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

CSRC = os.path.join(ROOT, "software_pipelined_loop_gb300", "csrc")


def _copy_sources(tmp_path):
    dst = tmp_path / "csrc"
    dst.mkdir()
    for f in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(CSRC, f), dst / f)
    return dst


def test_hash_ignores_comments_and_blank_space(tmp_path):
    dst = _copy_sources(tmp_path)
    before = bench.kernel_source_hash(str(dst))
    assert before == bench.kernel_source_hash()
    p = dst / "gemm_kernel.cuh"
    text = p.read_text(encoding="utf-8")
    p.write_text("// a new line comment\n/* and a\n   block comment */\n\n" + text.replace("\n", "\n\n", 3),
                 encoding="utf-8")
    assert bench.kernel_source_hash(str(dst)) == before


def test_hash_follows_code(tmp_path):
    dst = _copy_sources(tmp_path)
    before = bench.kernel_source_hash(str(dst))
    p = dst / "gemmpipe_api.cpp"
    p.write_text(p.read_text(encoding="utf-8") + "\nstatic int extra_symbol = 1;\n", encoding="utf-8")
    assert bench.kernel_source_hash(str(dst)) != before


def test_traffic_reported_only_at_the_captured_sources(monkeypatch):
    key, (bytes_, digest) = next(iter(bench.TRAFFIC.items()))
    dtype, M, N, K, pair, bn, bk = key
    plan = {"cta_pair": pair, "BN": bn, "BK": bk}
    monkeypatch.setattr(bench, "kernel_source_hash", lambda csrc=None: digest)
    assert bench.measured_traffic(dtype, plan, (M, N, K)) == bytes_
    monkeypatch.setattr(bench, "kernel_source_hash", lambda csrc=None: "0" * 16)
    assert bench.measured_traffic(dtype, plan, (M, N, K)) is None
    # A plan the table has no capture for.
    assert bench.measured_traffic(dtype, dict(plan, BN=bn + 1), (M, N, K)) is None


def test_table_entries_are_plausible():
    # Each capture lies within 1.5x of the workload's compulsory bytes
    # (operands read once, C written once; INT8 operands as their fp16
    # copies), and every entry was taken at one set of sources.
    digests = {d for _, d in bench.TRAFFIC.values()}
    assert len(digests) == 1
    for (dtype, M, N, K, *_), (bytes_, _) in bench.TRAFFIC.items():
        compulsory = 2 * (M * K + K * N) + 4 * M * N
        assert 0.4 * compulsory < bytes_ < 1.5 * compulsory, (dtype, M, N, K, bytes_, compulsory)
