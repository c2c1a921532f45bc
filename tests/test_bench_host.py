"""Host logic of bench.py that needs no GPU: the clock sampler's parsing of
nvidia-smi output (fed by a fake nvidia-smi on PATH), the stored-traffic
lookup that goes stale when the GEMM source changes, the whole-job value and
the peak denominators."""
import json
import os
import stat
import time

import pytest

import bench

FAKE_SMI = """#!/bin/sh
cat <<'EOF'
2070, 2070, 1200.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active
1965, 2070, 1390.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active
2040, 2070, 1385.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active
[N/A], 2070, [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]
garbage line
EOF
exec sleep 30
"""


def test_clock_sampler_parses_samples_and_reasons(tmp_path, monkeypatch):
    smi = tmp_path / "nvidia-smi"
    smi.write_text(FAKE_SMI)
    smi.chmod(smi.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    s = bench.ClockSampler(0)
    time.sleep(0.5)
    t0 = time.time()
    r = s.stop()
    assert time.time() - t0 < 10  # the sampler process is stopped, not awaited
    assert r["samples"] == 4  # the malformed line is dropped, the N/A row kept
    assert r["sm_mhz"] == 2040.0  # median of the three numeric SM clocks
    assert r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_sampler_without_nvidia_smi_reports_nothing(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))
    assert bench.ClockSampler(0).stop() is None


def _fake_root(tmp_path, gemm_src, stored_sha):
    csrc = tmp_path / "nvfp4_mixture_experts_expert_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "gemm.cu").write_bytes(gemm_src)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"l1_gemm_swiglu_quant_prefill": {"bytes_per_launch": 123, "gemm_cu_sha256_16": stored_sha}}))
    return str(tmp_path)


def test_stored_traffic_only_for_the_source_it_was_measured_on(tmp_path, monkeypatch):
    import hashlib
    src = b"// kernel source\n"
    sha = hashlib.sha256(src).hexdigest()[:16]
    monkeypatch.setattr(bench, "ROOT", _fake_root(tmp_path / "a", src, sha))
    assert bench.stored_traffic("l1_gemm_swiglu_quant_prefill") == 123
    assert bench.stored_traffic("l1_gemm_swiglu_quant_decode") is None  # never measured
    monkeypatch.setattr(bench, "ROOT", _fake_root(tmp_path / "b", src + b"// changed\n", sha))
    assert bench.stored_traffic("l1_gemm_swiglu_quant_prefill") is None


def test_measured_peaks_and_fallback(tmp_path, monkeypatch):
    p = bench.measured_peaks()
    if os.path.exists(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")):  # written per machine, not committed
        assert p["source"] == "measured" and p["hbm_gbs"] > 1000 and p["bf16_tflops_sustained"] > 100
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f = bench.measured_peaks()
    assert f["source"] == "fallback" and f["hbm_gbs"] == 6800.0


def test_whole_job_value_and_workload_names():
    assert bench.whole_job_throughput(8192, 4, 1.0) == pytest.approx(8192 * 4 / 1e-3)
    assert "T=8192" in bench.workload_name("prefill") and "E=48" in bench.workload_name("prefill")
    assert "T=128" in bench.workload_name("decode") and "E=32" in bench.workload_name("decode")


@pytest.mark.parametrize("n_pieces", [1, 3, 11])
def test_oracle_pieces_are_one_oracle_forward(n_pieces):
    """The reference arm and the CPU baseline time the oracle's forward as
    consecutive pieces; together they must be exactly one moe_forward call
    (same output, bit for bit) whatever the number of pieces."""
    import numpy as np
    from oracle import nvfp4_oracle as O
    from nvfp4_mixture_experts_expert_gb300 import workloads as W
    wl = W.moe_workload(96, 256, 128, 7, 2, 3, logit_bias_std=1.0)
    hidden = W.bf16_bits_to_f32(wl.hidden)
    st = dict(T=wl.T, H=wl.H, I=wl.I, E=wl.E, k=wl.top_k, hidden=hidden, logits=wl.logits,
              w13q=W.random_nvfp4_codes(wl.E, 2 * wl.I, wl.H, 5), w2q=W.random_nvfp4_codes(wl.E, wl.H, wl.I, 6),
              a1=np.full(wl.E, O.global_scale(np.abs(hidden).max()), np.float32),
              a2=np.full(wl.E, 200.0, np.float32))
    times, cpu_s, out = bench.oracle_timed_pieces(st, n_pieces, warmup=2)
    assert len(times) == n_pieces and cpu_s >= 0
    ref = O.moe_forward(hidden, wl.logits, wl.top_k, st["w13q"], st["w2q"], st["a1"], st["a2"],
                        bench.GATE_LIMIT, bench.UP_LIMIT)
    np.testing.assert_array_equal(out.view(np.uint32), ref.view(np.uint32))


def test_expert_pieces_cover_every_expert_once():
    for E, n in [(48, 20), (48, 400), (32, 1), (5, 5)]:
        groups = bench.expert_pieces(E, n)
        assert len(groups) == n
        assert sum(groups, []) == list(range(E))
