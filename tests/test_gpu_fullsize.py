"""GPU parity at the full sizes of the five workloads, in the launch
configuration the benchmark uses.

- dense GEMM (M=2048, K=3584, N=6144): quantization bit-exact, full GEMM output
  vs the oracle's FP64 GEMM (bf16-rounded relative Frobenius <= 1e-3);
- grouped linear (G=8, T=2048, D=2048, R=1024, strided (T,G,D) input and
  (T,G,R) output): same checks per group;
- decode MoE (T=128, H=4096, I=2048, E=32, k=6): everything of the small MoE
  parity test (bit-exact metadata / weights / L1 activations, end to end
  relative Frobenius <= 2e-2, cosine >= 0.999);
- prefill MoE (T=8192, E=48, Zipf prior): every check of the small MoE parity
  test over all 8,192 tokens and 48 experts (scales calibrated on all rows),
  and the stage-by-stage checks of test_gpu_stages on all 49,152 rows.
"""
import numpy as np
import pytest

from oracle import nvfp4_oracle as O
from nvfp4_mixture_experts_expert_gb300 import workloads as W
from helpers import OracleMoE, bf16_dev, bf16_host, cosine, dev, host, rel_frob

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def check_gemm(got, ref):
    ref_b = O.bf16_round(ref.astype(np.float32))
    assert np.all(np.isfinite(got))
    assert rel_frob(got, ref_b) <= 1e-3
    tol = np.abs(ref) * 2.0 ** -8 + 1e-5 * np.abs(ref).max()
    assert np.all(np.abs(got - ref) <= tol)


def test_dense_gemm_full_size():
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api, binding as B
    wl = W.dense_gemm()
    a = W.bf16_bits_to_f32(wl.a)
    b = W.bf16_bits_to_f32(wl.b)
    gs_a = O.global_scale(np.abs(a).max())
    an, as_ = O.quantize_blocks(a, gs_a)
    bn, bs, gs_b = O.weight_quantize(b)
    # device: quantize A on the fly (global scale from amax), B as a weight
    fa, sfa, ga = api.quantize(bf16_dev(wl.a))
    fb, sfb, gb = api.quantize(bf16_dev(wl.b))
    assert host(ga)[0] == gs_a and host(gb)[0] == gs_b
    np.testing.assert_array_equal(host(fa), O.pack_nibbles(an))
    np.testing.assert_array_equal(host(fb), O.pack_nibbles(bn))
    np.testing.assert_array_equal(host(sfa), O.assemble_scales(as_, np.array([0, wl.M]), np.array([0, wl.M])))
    D = torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device="cuda")
    B.nvfp4_grouped_gemm(fa, sfa, ga, fb, sfb, gb, dev(np.int32([0, wl.M])), None, 1, wl.M, wl.N, wl.K, D, wl.N, 0)
    torch.cuda.synchronize()
    check_gemm(bf16_host(D), O.nvfp4_gemm(an, as_, gs_a, bn, bs, gs_b))


def test_grouped_linear_full_size():
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api, binding as B
    wl = W.grouped_linear()
    T, G, D_, R = wl.T, wl.G, wl.D, wl.R
    x = W.bf16_bits_to_f32(wl.x)
    w = W.bf16_bits_to_f32(wl.w)
    fa, sfa, ga = api.quantize_groups(bf16_dev(wl.x), T, D_, G * D_, D_, G, rows_padded=T)
    fw, sfw, gw = api.quantize_expert_weights(bf16_dev(wl.w), gs=dev(wl.w_gs))
    np.testing.assert_array_equal(host(gw), wl.w_gs)
    out = torch.empty((T, G, R), dtype=torch.bfloat16, device="cuda")
    offs = np.arange(G + 1, dtype=np.int32) * T
    B.nvfp4_grouped_gemm(fa, sfa, ga, fw, sfw, gw, dev(offs), dev(np.full(G, T, np.int32)), G, G * T, R, D_, out,
                         G * R, R)
    torch.cuda.synchronize()
    got = bf16_host(out)
    ga, fa = host(ga), host(fa)
    for g in range(G):
        gs_g = O.global_scale(np.abs(x[:, g, :]).max())
        assert ga[g] == gs_g
        an, as_ = O.quantize_blocks(x[:, g, :], gs_g)
        np.testing.assert_array_equal(fa[g * T:(g + 1) * T], O.pack_nibbles(an))
        bn, bs, _ = O.weight_quantize(w[g], gs=wl.w_gs[g])
        check_gemm(got[:, g, :], O.nvfp4_gemm(an, as_, gs_g, bn, bs, wl.w_gs[g]))


def test_decode_moe_full_size():
    from test_gpu_moe import check_all, run_gpu
    wl = W.decode_moe()
    orc = OracleMoE(wl)
    check_all(wl, orc, *run_gpu(wl, orc))


def test_prefill_moe_full_size_all_tokens():
    """The benchmarked prefill layer, every token and every expert: weights,
    routing and slot metadata, gathered L1 activations bit-exact; activation
    scales calibrated by the oracle on all rows; end to end against the
    oracle's forward over the whole batch (relative Frobenius <= 2e-2,
    cosine >= 0.999); L2 inputs dequantized within 2e-2."""
    from test_gpu_moe import check_all, run_gpu
    wl = W.prefill_moe()
    orc = OracleMoE(wl)
    assert orc.meta["counts"].min() > 0 and orc.meta["P"] == 52096
    check_all(wl, orc, *run_gpu(wl, orc))


def test_prefill_moe_full_size_stages():
    """The same layer stage by stage on the GPU's own operands (see
    test_gpu_stages): L1 GEMM + SwiGLU, bit-exact requantization, L2 GEMM +
    routing-weighted rows, token combine -- all 49,152 assignment rows."""
    from test_gpu_stages import check_stages, oracle_a1_scales, run_forwards
    wl = W.prefill_moe()
    a1, meta = oracle_a1_scales(wl)
    check_stages(wl, a1, meta, *run_forwards(wl, a1))
