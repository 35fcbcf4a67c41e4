"""bench.py's host-side helpers (CPU only): algorithmic byte counts, the two
roofline fractions, the kernel the automatic choice names, the traffic gate and
the shared `config` object of both arms."""
from __future__ import annotations

import pytest

import bench
from ragged_attention_token_gb300 import workloads as W

PEAKS = dict(hbm_gbs=6788.6, bf16_tflops=1925.9, bf16_tflops_sustained=1696.8, source="test")


def test_case_bytes_of_the_serving_workload():
    case = W.make_serving(4)
    B, N, H, d, T = case.B, case.N, case.H, case.d, case.kept_tokens
    by = bench.case_bytes(case)
    assert by["fused_min"] == B * N + 3 * T * H * d * 2 + B * N * H * d * 2
    assert by["attend"] == 4 * T * H * d * 2
    assert by["flops"] == 4 * H * d * sum(n * n for n in case.lengths)
    assert sum(case.lengths) == T


def test_roofline_fractions():
    case = W.make_batched(0.8)
    by = bench.case_bytes(case)
    us = 10.0
    r = bench.roofline_obj(by["fused_min"], by["flops"], us, PEAKS)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["frac"] == pytest.approx(by["fused_min"] / (us * 1e-6) / 1e9 / PEAKS["hbm_gbs"], abs=1e-4)
    # The problem's roofline: packed Q/K/V/O bytes (or FLOPs) only, so below the pipeline's own count.
    f = bench.packed_qkvo_frac(case, us, PEAKS)
    assert 0 < f < r["frac"]


def test_kernel_named_for_the_automatic_choice():
    small = "attend_small_kernel"
    assert bench.pipeline_kernel_name(W.make_serving(4), 152).startswith(small)
    assert bench.pipeline_kernel_name(W.make_tiny(), 152).startswith(small)
    assert bench.pipeline_kernel_name(W.make_batched(0.8), 152).startswith("attend_tc_kernel")
    assert bench.pipeline_kernel_name(W.make_hires(0.9), 152).startswith("attend_tc_kernel")   # N > 256


def test_traffic_gate():
    assert bench.measured_traffic("no such workload") is None
    for key, (src, sha, nbytes) in bench.TRAFFIC.items():
        assert len(sha) == 16 and int(sha, 16) >= 0 and nbytes > 0
        full = bench.kernel_source_sha(src)
        assert len(full) == 64
        assert bench.measured_traffic(key) == (nbytes if full.startswith(sha) else None)


def test_both_arms_share_the_config():
    case, desc = bench.make_case("serving")
    a = bench.workload_config(case, desc, 1)
    b = bench.workload_config(case, desc, 1)
    assert a == b and a["workload"] == desc and a["kept_tokens_per_step"] == case.kept_tokens


def test_percentile_nearest_rank():
    xs = list(range(1, 11))            # 1..10
    assert bench.percentile(xs, 0.9) == 10
    assert bench.percentile(xs, 0.5) == 6
    assert bench.percentile(xs, 0.0) == 1
    assert bench.percentile([3.0], 0.9) == 3.0
    assert bench.percentile(list(reversed(xs)), 0.9) == 10   # order of the samples does not matter
