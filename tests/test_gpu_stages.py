"""Stage-by-stage GPU parity of the fused MoE kernels, each on the GPU's own
(bit-exact) operands, so that an error in one stage cannot hide behind the
end-to-end tolerance.

One forward with the L2 activation scales taken from the batch (a2_gs NULL:
the L1 GEMM stores its bf16 SwiGLU output h) and one with those same scales
given (the fused L1 requantization); then:

- L1 grouped GEMM + SwiGLU: h against the oracle's SwiGLU (gate clamped
  before the SiLU) of the FP64 GEMM over the same A1 / W13 bytes and scales.
  Per element |h - h_exact| <= tol_h (derivation below); the bf16-rounded
  oracle and h agree to relative Frobenius <= 1e-3.
- requantization: the oracle's quantization of the GPU's h with the scale
  used equals the L2 input (nibbles and tile-layout scales) bit for bit, for
  both the batch-scale quantize pass and the fused L1 epilogue; the batch
  scales equal 2688 / amax(h) bit for bit.
- L2 grouped GEMM + routing-weighted epilogue: the bf16 rows Y against
  w * alpha2 * (A2 . W2^T) in FP64 over the same A2 / W2 bytes: per element
  <= tol_y, relative Frobenius against the bf16-rounded oracle <= 1e-3.
- token combine: out[t] against the FP64 sum of the token's Y rows.

Tolerances (the arithmetic the kernels do):
  GEMM accumulation: FP32 in TMEM, one K=64 block-scaled MMA at a time; with
  round-to-nearest or truncation each of the K/64 accumulations errs by at
  most 2^-23 of the running sum, so |acc - exact| <= (K/64) 2^-23 sum_k|a_k b_k|.
  We allow 4x that, delta = (K/64) 2^-21 alpha ||a|| ||b|| (Cauchy-Schwarz
  bounds sum|a_k b_k|).
  SwiGLU: the kernel's sigmoid is (1 + tanh.approx(g/2)) / 2; tanh.approx.f32
  has a relative error below 2^-10.98 (PTX ISA), so the sigmoid is off by at
  most 2^-11.98 (absolute) and h by |g_c u_c| 2^-11.9; the GEMM error enters
  through dh/dg = u_c (s + g_c s (1 - s)) and dh/du = g_c s (clamps are
  1-Lipschitz), counted twice for second-order slack; a few FP32 roundings
  add 2^-21 |h|; the bf16 rounding of h adds half an ulp, <= 2^-8 |h|.
  L2 rows: bf16(fl(w * alpha) * acc): 2^-8 |Y| for the rounding, w * delta for
  the accumulation, 2^-21 |Y| for the FP32 products.
  Combine: FP32 sum of k bf16 rows in a fixed order, then bf16: 2^-8 |out|
  + k 2^-24 sum_j |Y_j|.
"""
import numpy as np
import pytest

from oracle import nvfp4_oracle as O
from nvfp4_mixture_experts_expert_gb300 import workloads as W
from helpers import bf16_dev, bf16_host, dev, host, rel_frob

pytestmark = pytest.mark.gpu

TANH_SIGMOID_ABS = 2.0 ** -11.9


def oracle_a1_scales(wl):
    """Per-expert L1 activation scales (2688 / amax of the rows routed to the
    expert, 1 for none): inputs of both sides, computed by the oracle."""
    hidden = W.bf16_bits_to_f32(wl.hidden)
    ids, wts = O.route(wl.logits, wl.top_k)
    meta = O.sort_slots(ids, wts, wl.E)
    a1 = np.ones(wl.E, np.float32)
    for e in range(wl.E):
        lo, n = int(meta["offsets"][e]), int(meta["counts"][e])
        if n:
            a1[e] = O.global_scale(np.abs(hidden[meta["sorted_token_ids"][lo:lo + n]]).max())
    return a1, meta


def run_forwards(wl, a1):
    """The a2_gs NULL forward (h kept) and the forward given the scales it derived."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    hidden, logits, a1_d = bf16_dev(wl.hidden), dev(wl.logits), dev(a1)
    f_null = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    out_null = f_null(hidden, logits, w, a1_d, None, wl.gate_limit, wl.up_limit)
    a2 = f_null.batch_l2_scales().clone()
    f_given = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    out_given = f_given(hidden, logits, w, a1_d, a2, wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    assert f_null.status() == 0 and f_given.status() == 0
    return w, f_null, f_given, out_null, out_given, host(a2)


def _norm_rows(x):
    return np.sqrt(np.einsum("ij,ij->i", x, x))


def check_stages(wl, a1, meta, w, f_null, f_given, out_null, out_given, a2):
    """All stage checks; returns the figures (for the log) of the worst stage."""
    import torch
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.top_k
    gl, ul = wl.gate_limit, wl.up_limit
    P = meta["P"]
    # the GPU's own slot metadata equals the oracle's (routing parity is pinned elsewhere too)
    np.testing.assert_array_equal(host(f_given.view("offsets", torch.int32, E + 1)), meta["offsets"])
    np.testing.assert_array_equal(host(f_given.view("sorted_token_ids", torch.int32, P)), meta["sorted_token_ids"])
    inv = host(f_given.view("inverse", torch.int32, T * k)).reshape(T, k)
    row_w = host(f_given.view("row_weight", torch.float32, P)).astype(np.float64)
    np.testing.assert_array_equal(bf16_host(out_null).view(np.uint32), bf16_host(out_given).view(np.uint32))

    a1_nib = O.unpack_nibbles(host(f_given.view("a1", torch.uint8, P * H // 2)).reshape(P, H // 2))
    a1_s = O.unswizzle_scales(host(f_given.view("sfa1", torch.uint8, P * H // 16)), P, H // 16)
    h_gpu = bf16_host(f_null.view("h", torch.bfloat16, P * I)).reshape(P, I)  # bf16 values, exact in FP32
    a2n_nib = O.unpack_nibbles(host(f_null.view("a2", torch.uint8, P * I // 2)).reshape(P, I // 2))
    a2n_s = O.unswizzle_scales(host(f_null.view("sfa2", torch.uint8, P * I // 16)), P, I // 16)
    a2g_nib = O.unpack_nibbles(host(f_given.view("a2", torch.uint8, P * I // 2)).reshape(P, I // 2))
    a2g_s = O.unswizzle_scales(host(f_given.view("sfa2", torch.uint8, P * I // 16)), P, I // 16)
    y_gpu = bf16_host(f_given.view("y", torch.bfloat16, P * H)).reshape(P, H)
    w13, w13_sf, w13_gs = host(w.w13), host(w.w13_sf), host(w.w13_gs)
    w2, w2_sf, w2_gs = host(w.w2), host(w.w2_sf), host(w.w2_gs)

    stats = dict(h_viol=0.0, y_viol=0.0, h_frob_num=0.0, h_frob_den=0.0, y_frob_num=0.0, y_frob_den=0.0,
                 h_frob_exact_num=0.0, h_flips=0, h_count=0)
    for e in range(E):
        lo, n = int(meta["offsets"][e]), int(meta["counts"][e])
        if n == 0:
            continue
        rows = slice(lo, lo + n)
        hg = h_gpu[rows].astype(np.float64)
        yg = y_gpu[rows].astype(np.float64)
        # ---- L1 GEMM + SwiGLU on the GPU's A1 and W13 bytes
        b_nib = O.unpack_nibbles(w13[e])
        b_s = O.unswizzle_scales(w13_sf[e], 2 * I, H // 16)
        G = O.nvfp4_gemm(a1_nib[rows], a1_s[rows], a1[e], b_nib, b_s, w13_gs[e])
        alpha1 = 1.0 / (np.float64(a1[e]) * np.float64(w13_gs[e]))
        na = _norm_rows(O.dequant_blocks(a1_nib[rows], a1_s[rows]))
        nb = _norm_rows(O.dequant_blocks(b_nib, b_s))
        delta = (H / 64) * 2.0 ** -21 * alpha1 * na[:, None] * nb[None, :]
        g, u = G[:, :I], G[:, I:]
        h_exact = O.swiglu_exact(g, u, gl, ul)
        gc = np.minimum(g, gl)
        uc = np.clip(u, -ul, ul)
        s = 1.0 / (1.0 + np.exp(-gc))
        dg = np.abs(uc) * (s + np.abs(gc) * s * (1.0 - s))
        du = np.abs(gc) * s
        pre = (np.abs(gc * uc) * TANH_SIGMOID_ABS + 2.0 * (dg * delta[:, :I] + du * delta[:, I:])
               + 2.0 ** -21 * np.abs(h_exact))
        tol_h = 2.0 ** -8 * np.abs(h_exact) + (1 + 2.0 ** -8) * pre + 1e-30
        err_h = np.abs(hg - h_exact)
        stats["h_viol"] = max(stats["h_viol"], float(np.max(err_h / tol_h)))
        h_ref_b = O.bf16_round(h_exact.astype(np.float32)).astype(np.float64)
        stats["h_frob_num"] += float(np.sum((hg - h_ref_b) ** 2))
        stats["h_frob_den"] += float(np.sum(h_ref_b ** 2))
        stats["h_frob_exact_num"] += float(np.sum((hg - h_exact) ** 2))
        stats["h_flips"] += int(np.count_nonzero(hg != h_ref_b))
        stats["h_count"] += h_exact.size
        # ---- requantization, bit-exact, on the GPU's h
        assert a2[e] == O.global_scale(np.abs(h_gpu[rows]).max()), e
        q_nib, q_s = O.quantize_blocks(h_gpu[rows], a2[e])
        np.testing.assert_array_equal(a2n_nib[rows], q_nib)
        np.testing.assert_array_equal(a2n_s[rows], q_s)
        np.testing.assert_array_equal(a2g_nib[rows], q_nib)
        np.testing.assert_array_equal(a2g_s[rows], q_s)
        # ---- L2 GEMM + routing-weighted epilogue on the GPU's A2 and W2 bytes
        c_nib = O.unpack_nibbles(w2[e])
        c_s = O.unswizzle_scales(w2_sf[e], H, I // 16)
        Y = O.nvfp4_gemm(q_nib, q_s, a2[e], c_nib, c_s, w2_gs[e]) * row_w[rows, None]
        alpha2 = 1.0 / (np.float64(a2[e]) * np.float64(w2_gs[e]))
        na2 = _norm_rows(O.dequant_blocks(q_nib, q_s))
        nc = _norm_rows(O.dequant_blocks(c_nib, c_s))
        delta2 = (I / 64) * 2.0 ** -21 * alpha2 * na2[:, None] * nc[None, :] * row_w[rows, None]
        tol_y = 2.0 ** -8 * np.abs(Y) + (1 + 2.0 ** -8) * (delta2 + 2.0 ** -21 * np.abs(Y)) + 1e-30
        stats["y_viol"] = max(stats["y_viol"], float(np.max(np.abs(yg - Y) / tol_y)))
        Y_b = O.bf16_round(Y.astype(np.float32)).astype(np.float64)
        stats["y_frob_num"] += float(np.sum((yg - Y_b) ** 2))
        stats["y_frob_den"] += float(np.sum(Y_b ** 2))
    # ---- token combine: sum of the token's k weighted rows (token chunks, FP64)
    out_h = bf16_host(out_given)
    c_viol, n_equal = 0.0, 0
    for t0 in range(0, T, 1024):
        t1 = min(T, t0 + 1024)
        parts = y_gpu[inv[t0:t1].reshape(-1)].reshape(t1 - t0, k, H).astype(np.float64)
        ref = parts.sum(axis=1)
        tol_o = 2.0 ** -8 * np.abs(ref) + k * 2.0 ** -24 * np.abs(parts).sum(axis=1) + 1e-30
        got = out_h[t0:t1].astype(np.float64)
        c_viol = max(c_viol, float(np.max(np.abs(got - ref) / tol_o)))
        n_equal += int(np.count_nonzero(got == O.bf16_round(ref.astype(np.float32))))
    c_equal = n_equal / (T * H)
    figs = dict(h_viol=stats["h_viol"], y_viol=stats["y_viol"], c_viol=c_viol, c_equal=c_equal,
                h_frob_bf16=np.sqrt(stats["h_frob_num"] / stats["h_frob_den"]),
                h_frob_exact=np.sqrt(stats["h_frob_exact_num"] / stats["h_frob_den"]),
                h_flip_frac=stats["h_flips"] / max(stats["h_count"], 1),
                y_frob_bf16=np.sqrt(stats["y_frob_num"] / max(stats["y_frob_den"], 1e-300)))
    print("stage figures:", {k_: round(float(v), 6) for k_, v in figs.items()})
    assert figs["h_viol"] <= 1.0, figs
    assert figs["y_viol"] <= 1.0, figs
    assert figs["c_viol"] <= 1.0, figs
    assert figs["h_frob_bf16"] <= 1e-3, figs
    assert figs["y_frob_bf16"] <= 1e-3, figs
    return figs


@pytest.mark.parametrize("T,H,I,E,k,seed", [
    (300, 512, 256, 6, 2, 5),     # several m-tiles per expert, ragged tails
    (150, 256, 384, 5, 3, 6),     # I > H, I/128 odd
    (700, 1024, 256, 8, 2, 7),    # K = 1024 for L1: four K stages per tile
])
def test_fused_stages_match_oracle_on_gpu_operands(T, H, I, E, k, seed):
    wl = W.moe_workload(T, H, I, E, k, seed, logit_bias_std=1.0)
    a1, meta = oracle_a1_scales(wl)
    check_stages(wl, a1, meta, *run_forwards(wl, a1))


def test_fused_stages_with_clamps_active():
    """Small limits, so that many gates and ups are clamped (the clamp
    boundaries are inside the checked range)."""
    wl = W.moe_workload(260, 512, 256, 4, 2, 9)
    wl.gate_limit, wl.up_limit = 0.02, 0.015
    a1, meta = oracle_a1_scales(wl)
    check_stages(wl, a1, meta, *run_forwards(wl, a1))


def test_fused_stages_decode_size():
    """The decode layer (T=128, H=4096, I=2048, E=32, top_k=6), stage by stage."""
    wl = W.decode_moe()
    a1, meta = oracle_a1_scales(wl)
    check_stages(wl, a1, meta, *run_forwards(wl, a1))
