"""Exhaustive device checks of the conversion primitives inside the NVFP4
kernels: the fused-multiply-add division by a block scale equals the IEEE
division for every E4M3 scale and every fp32 mantissa, and the paired E2M1
conversion puts the first element in the low nibble."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "nvfp4_mixture_experts_expert_gb300", "csrc")


@pytest.fixture(scope="module")
def probe():
    import torch  # noqa: F401  (initialises the CUDA context the probe shares)
    build = os.path.join(HERE, "probes", "_build")  # git-ignored, beside the probe source
    os.makedirs(build, exist_ok=True)
    out = os.path.join(build, "fp_probe.so")
    subprocess.run(["nvcc", "-gencode=arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-I", CSRC, os.path.join(HERE, "probes", "fp_probe.cu"), "-o", out],
                   check=True, capture_output=True)
    return ctypes.CDLL(out)


@pytest.mark.parametrize("exp_bias", [-3, -1, 0, 1, 2])
def test_scale_division_is_ieee_exact(probe, exp_bias):
    bad = ctypes.c_ulonglong(12345)
    assert probe.run_div_probe(exp_bias, ctypes.byref(bad)) == 0
    assert bad.value == 0


def test_e2m1_pair_conversion_lane_order(probe):
    grid = [0.0, 0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0, 7.0, 100.0]
    vals = np.array(grid + [-g for g in grid] + [0.3, -2.9, 4.5], np.float32)
    bad = ctypes.c_uint(999)
    assert probe.run_e2m1_pair_probe(vals.ctypes.data_as(ctypes.c_void_p), len(vals), ctypes.byref(bad)) == 0
    assert bad.value == 0


def test_e2m1_word_pack_byte_order(probe):
    rng = np.random.default_rng(9)
    grid = np.array([0.0, 0.25, 0.5, 0.75, 1.0, 1.25, 1.75, 2.5, 3.0, 3.5, 5.0, 6.0, 7.0], np.float32)
    vals = np.concatenate([grid, -grid, rng.uniform(-8, 8, 4000).astype(np.float32)])
    bad = ctypes.c_uint(999)
    assert probe.run_e2m1_word_probe(vals.ctypes.data_as(ctypes.c_void_p), len(vals), ctypes.byref(bad)) == 0
    assert bad.value == 0
