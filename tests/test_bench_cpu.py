"""The benchmark's host-side pieces that need no GPU: the oracle baselines it times beside
every path (on small workloads of the same kinds) and its traffic table lookup."""
import json
import pathlib
import sys

import numpy as np

ROOT = pathlib.Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))

import bench  # noqa: E402
import workloads  # noqa: E402


def _well_formed(line: dict, unit: str) -> None:
    assert line["kind"] == "oracle" and line["unit"] == unit
    assert np.isfinite(line["value"]) and line["value"] > 0
    assert isinstance(line["cores"], int) and line["cores"] >= 1
    assert isinstance(line["sample"], str) and line["sample"]


def test_prefill_baselines():
    c = workloads.tiny_prefill()
    _well_formed(bench.cpu_prefill(c, target_s=0.05), "TFLOP/s")
    _well_formed(bench.cpu_baseline(c, target_s=0.05), "TFLOP/s")


def test_decode_baseline_takes_a_subset_of_the_sequences():
    c = workloads.paged_decode(num_seqs=6, ctx_lo=16, ctx_hi=300, num_pages=160, n_heads=8,
                               n_kv_heads=2, head_dim=64, seed=4)
    line = bench.cpu_decode(c, target_s=0.05)
    _well_formed(line, "GB/s")
    assert " of 6 sequences" in line["sample"]


def test_verify_baselines_cover_both_forms():
    c = workloads.ring(lanes=2, rows=4, window=64, q_heads=4, kv_heads=2, head_dim=128, seed=5)
    chain, fused = bench.cpu_verify(c, 1_000_000, 250_000)
    _well_formed(chain, "GB/s")
    _well_formed(fused, "GB/s")


def test_chunk_baseline_counts_the_flops_of_its_tokens():
    c = workloads.paged_chunk(num_seqs=3, tokens_lo=5, tokens_hi=20, prefix_lo=10, prefix_hi=90,
                              seed=6)
    line = bench.cpu_chunk(c, target_s=0.05)
    _well_formed(line, "TFLOP/s")
    assert "new tokens of one sequence" in line["sample"]


def test_traffic_lookup():
    assert bench.traffic_for("no_such_kernel", "no_such_workload") is None
    table = json.loads((ROOT / "profiles" / "traffic.json").read_text())
    for key, entry in table.items():
        kernel, workload = key.split("@", 1)
        got = bench.traffic_for(kernel, workload)
        # the recorded bytes, or None once the kernel's source has changed since the capture
        assert got is None or got == float(entry["bytes_per_launch"])
