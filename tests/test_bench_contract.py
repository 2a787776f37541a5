"""The benchmark's contract, checked on the CPU: the algorithmic work its rooflines divide by
(closed forms of the workloads' causal pairs and selected slots), the value up-projection's byte
count, and the one JSON line of the reference arm (the float64 oracle on the host cores)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from deepseek_sparse_attention_indexer_gb300 import workloads as W  # noqa: E402


def _closed_form(L, p0, N, K):
    """Causal pairs sum_i min(p0 + i + 1, N) and selected slots sum_i min(p0 + i + 1, K), by the
    arithmetic-series formula in the piecewise ranges (no per-query loop)."""
    def clipped_sum(cap):
        # positions p0 + 1 .. p0 + L, each clipped at cap
        lo, hi = p0 + 1, p0 + L
        if hi <= cap:
            return (lo + hi) * L // 2
        if lo >= cap:
            return cap * L
        n_lin = cap - lo + 1
        return (lo + cap) * n_lin // 2 + cap * (L - n_lin)
    return clipped_sum(N), clipped_sum(K)


@pytest.mark.parametrize("name,pairs,slots", [
    ("prefill_16k", 58_722_304, 8_388_608),     # 4096 queries at 12288.. over 16k keys
    ("first_chunk_4k", 8_390_656, 6_292_480),   # 0..4095: rows below 2048 keep every key
    ("prefill_64k", 260_048_896, 8_388_608),
    ("tiny_1k", 63_520, 16_384),
])
def test_algorithmic_work_matches_the_closed_forms(name, pairs, slots):
    wl = W.WORKLOADS[name]
    work = bench.algorithmic(wl)
    assert (work["pairs"], work["slots"]) == (pairs, slots)
    assert _closed_form(wl.L, wl.p0, wl.N, wl.top_k) == (pairs, slots)
    assert work["indexer_flop"] == pairs * 32 * 128 * 2
    assert work["attn_flop"] == slots * 64 * (576 + 512) * 2
    assert work["topk_bytes"] == pairs * 4 and work["gather_bytes"] == slots * 1152


def test_decode_work_counts_every_sequence():
    wl = W.WORKLOADS["decode_b8"]
    work = bench.algorithmic(wl)
    assert work["pairs"] == 8 * 4096 and work["slots"] == 8 * 2048


def test_value_up_projection_line():
    line = bench.value_proj_line(4096, 0.0785, {"hbm_gbs": 6783.5}, "measured")
    assert line["bytes_per_launch"] == 4096 * 64 * 512 * 2 + 64 * 256 * 512 * 2 + 4096 * 64 * 256 * 2
    assert line["achieved_gbs"] == pytest.approx(419430400 / 0.0785e-3 / 1e9)
    assert line["frac"] == pytest.approx(line["achieved_gbs"] / 6783.5)
    assert line["bound"] == "hbm"


def test_reference_arm_prints_one_json_line():
    """`bench.py --impl reference` times the oracle on the host and prints the contract's line."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_1k", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["higher_is_better"] is True
    assert d["metric"] == bench.metric_name(bench.W.WORKLOADS["tiny_1k"]) and d["unit"] == bench.UNIT
    assert d["value"] > 0
    assert d["config"]["workload"] == "tiny_1k" and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_each_workload_line_names_its_own_context():
    """The headline (16k chunk) keeps the metric string of the benchmark contract; every other
    line states its own context, so a 64k line never reads "16k ctx"."""
    W = bench.W
    assert bench.metric_name(W.WORKLOADS["prefill_16k"]) == bench.METRIC
    assert "at 64k ctx" in bench.metric_name(W.WORKLOADS["prefill_64k"])
    assert "at 4k ctx" in bench.metric_name(W.WORKLOADS["first_chunk_4k"])
    assert "at 1k ctx" in bench.metric_name(W.WORKLOADS["tiny_1k"])
    assert bench.metric_name(W.WORKLOADS["decode_b8"]).startswith("decode us/step")
    names = {bench.metric_name(w) for w in W.WORKLOADS.values() if w.L > 1}
    assert len(names) == len([w for w in W.WORKLOADS.values() if w.L > 1])


def test_resolve_workload_narrows_prefill_and_widens_decode():
    wl = bench.resolve_workload("prefill_16k", queries=1024)
    assert (wl.B, wl.L, wl.p0, wl.N, wl.top_k) == (1, 1024, 16384 - 1024, 16384, 2048)
    wl = bench.resolve_workload("decode_b8", batch=128)
    assert (wl.B, wl.L, wl.p0, wl.N, wl.top_k) == (128, 1, 4095, 4096, 2048)
    assert wl.name == "decode_b8_batch128" and "128 sequences" in wl.desc
    assert bench.metric_name(wl).startswith("decode us/step") and "batch 128" in bench.metric_name(wl)
    paged = bench.resolve_workload("decode_b8_paged", batch=16)
    assert paged.page_size == W.WORKLOADS["decode_b8_paged"].page_size and paged.B == 16
    assert bench.resolve_workload("prefill_16k") == W.WORKLOADS["prefill_16k"]
    with pytest.raises(ValueError):
        bench.resolve_workload("prefill_16k", batch=4)


def test_cpu_baseline_sizes_its_sample_from_a_probe():
    """The CPU baseline (the oracle on the host's cores) times a seeded sample sized from a short
    probe to about the target seconds, and says what it timed."""
    wl = W.custom("cpu_base_small", B=1, L=48, p0=464, N=512, top_k=128, seed=3)
    inputs = bench.make_inputs(wl)
    cb = bench.cpu_baseline(wl, inputs, decode=False, target_s=0.05)
    assert cb["kind"] == "oracle" and cb["unit"] == bench.UNIT and cb["value"] > 0 and cb["cores"] >= 1
    assert "query rows" in cb["sample"]
    wl_d = W.custom("cpu_base_decode", B=2, L=1, p0=255, N=256, top_k=64, seed=4)
    cb = bench.cpu_baseline(wl_d, bench.make_inputs(wl_d), decode=True, target_s=0.05)
    assert cb["unit"] == "us/step" and cb["value"] > 0 and "decode steps" in cb["sample"]


def test_step_roofline_of_the_16k_chunk():
    """The step's ideal: indexer FLOP / peak + score bytes / HBM + attention FLOP / peak."""
    work = bench.algorithmic(W.WORKLOADS["prefill_16k"])
    r = bench.step_roofline(work, 1899.5, 6783.5, 1.8)
    want = 1e3 * (481.1e9 / 1899.5e12 + 234.9e6 / 6783.5e9 + 1168.2e9 / 1899.5e12)
    assert abs(r["ideal_ms"] - want) < 2e-3 and abs(r["frac"] - want / 1.8) < 2e-3
