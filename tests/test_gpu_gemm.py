"""GPU parity of the tcgen05 block-scaled grouped GEMM against the oracle's FP64
GEMM on identical quantized operands (both quantized by the oracle).

Tolerance: the kernel accumulates in FP32 and stores bf16, so both sides are
compared after rounding to bf16: relative Frobenius error <= 1e-3 (the bound
for the GEMM); elementwise the kernel may differ from the FP64 result by at
most one bf16 rounding plus FP32 accumulation error."""
import numpy as np
import pytest

from oracle import nvfp4_oracle as O
from nvfp4_mixture_experts_expert_gb300 import workloads as W
from helpers import bf16_host, dev, rel_frob

pytestmark = pytest.mark.gpu


def make_problem(counts, N, K, seed, b_gs=None):
    rng = np.random.default_rng(seed)
    G = len(counts)
    padded = np.concatenate([[0], np.cumsum([(c + 127) // 128 * 128 for c in counts])]).astype(np.int32)
    cap = int(padded[-1]) + 128  # a spare tile of capacity beyond the last group
    A = np.zeros((cap, K // 2), np.uint8)
    s_lin = np.zeros((cap, K // 16), np.uint8)
    a_gs = np.ones(G, np.float32)
    a_deq = []
    for g, c in enumerate(counts):
        x = W.bf16_bits_to_f32(W.f32_to_bf16_bits(
            rng.standard_normal((c, K)).astype(np.float32) * np.exp(rng.standard_normal((c, 1))).astype(np.float32)))
        a_gs[g] = O.global_scale(np.abs(x).max()) if c else np.float32(1)
        nib, s = O.quantize_blocks(x, a_gs[g])
        A[padded[g]:padded[g] + c] = O.pack_nibbles(nib)
        s_lin[padded[g]:padded[g] + c] = s
        a_deq.append((nib, s))
    SFA = O.assemble_scales(s_lin, np.array([0, cap]), np.array([0, cap]))
    w = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((G, N, K)).astype(np.float32) * np.float32(0.02)))
    bn, bs, bg = O.quantize_expert_weights(w, gs=b_gs)
    Bp = np.stack([O.pack_nibbles(bn[g]) for g in range(G)])
    n128 = (N + 127) // 128 * 128  # a group's scales span whole 128-row tiles
    SFB = np.stack([O.assemble_scales(bs[g], np.array([0, N]), np.array([0, n128])) for g in range(G)])
    ref = [O.nvfp4_gemm(a_deq[g][0], a_deq[g][1], a_gs[g], bn[g], bs[g], bg[g]) for g in range(G)]
    return dict(A=A, SFA=SFA, a_gs=a_gs, B=Bp, SFB=SFB, b_gs=bg, padded=padded, counts=np.int32(counts),
                cap=cap, ref=ref, G=G, N=N, K=K)


def run_gpu(pb, use_counts=True):
    import torch
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    G, N, K = pb["G"], pb["N"], pb["K"]
    maxrows = int(np.diff(pb["padded"]).max())
    D = torch.full((G, max(maxrows, 1), N), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.nvfp4_grouped_gemm(dev(pb["A"]), dev(pb["SFA"]), dev(pb["a_gs"]), dev(pb["B"]), dev(pb["SFB"]),
                         dev(pb["b_gs"]), dev(pb["padded"]), dev(pb["counts"]) if use_counts else None, G,
                         pb["cap"], N, K, D, N, max(maxrows, 1) * N)
    torch.cuda.synchronize()
    return bf16_host(D)


def check(pb, D):
    for g, c in enumerate(pb["counts"]):
        if c == 0:
            continue
        ref = pb["ref"][g]
        got = D[g, :c]
        assert np.all(np.isfinite(got))
        ref_b = O.bf16_round(ref.astype(np.float32))
        assert rel_frob(got, ref_b) <= 1e-3, (g, rel_frob(got, ref_b))
        # elementwise: within one bf16 rounding of the FP64 result (+ accumulation slack)
        tol = np.abs(ref) * 2.0 ** -8 + 1e-5 * np.abs(ref).max()
        assert np.all(np.abs(got - ref) <= tol), (g, np.max(np.abs(got - ref) - tol))


@pytest.fixture(params=[True, False], ids=["pair", "single"])
def cta_pair(request):
    """Runs the test with the paired-CTA GEMM (cta_group::2) and with one CTA per tile."""
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    prev = B.nvfp4_gemm_set_cta_pair(request.param)
    yield request.param
    B.nvfp4_gemm_set_cta_pair(prev)


@pytest.mark.parametrize("counts,N,K", [
    ([128], 256, 256),               # one tile, one K stage (a pair whose second tile does not exist)
    ([100, 0, 260], 512, 320),       # ragged groups, an empty group, partial last K stage, odd tile counts
    ([37, 129], 256, 128),           # K = 128: a single half stage
    ([300], 768, 1024),              # several tiles and K stages
    ([256, 384, 1, 640], 256, 512),  # even and odd tile counts side by side
])
def test_grouped_gemm_matches_oracle(counts, N, K, cta_pair):
    pb = make_problem(counts, N, K, seed=sum(counts) + N + K)
    check(pb, run_gpu(pb))


def test_pair_and_single_cta_gemm_are_bit_identical():
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    pb = make_problem([300, 0, 129, 640, 5], 512, 768, seed=11)
    prev = B.nvfp4_gemm_set_cta_pair(True)
    try:
        d_pair = run_gpu(pb)
        B.nvfp4_gemm_set_cta_pair(False)
        d_single = run_gpu(pb)
    finally:
        B.nvfp4_gemm_set_cta_pair(prev)
    for g, c in enumerate(pb["counts"]):
        np.testing.assert_array_equal(d_pair[g, :c], d_single[g, :c])


def test_gemm_rows_beyond_counts_are_not_written():
    pb = make_problem([10, 50], 256, 256, seed=1)
    D = run_gpu(pb)
    assert np.all(np.isnan(D[0, 10:128])) and np.all(np.isnan(D[1, 50:128]))


def test_gemm_identity_weight_returns_dequantized_activation():
    """Closed form: B = identity (exactly representable) -> D = dequant(A)."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    K = N = 256
    rng = np.random.default_rng(3)
    x = rng.standard_normal((128, K)).astype(np.float32)
    gs_a = O.global_scale(np.abs(x).max())
    nib, s = O.quantize_blocks(x, gs_a)
    eye_n, eye_s, eye_gs = O.weight_quantize(np.eye(K, dtype=np.float32))
    D = torch.empty((128, N), dtype=torch.bfloat16, device="cuda")
    B.nvfp4_grouped_gemm(dev(O.pack_nibbles(nib)), dev(O.assemble_scales(s, np.array([0, 128]), np.array([0, 128]))),
                         dev(np.float32([gs_a])), dev(O.pack_nibbles(eye_n)),
                         dev(O.assemble_scales(eye_s, np.array([0, K]), np.array([0, K]))),
                         dev(np.float32([eye_gs])), dev(np.int32([0, 128])), None, 1, 128, N, K, D, N, 0)
    torch.cuda.synchronize()
    expect = O.bf16_round((O.dequant_blocks(nib, s) / np.float64(gs_a)).astype(np.float32))
    np.testing.assert_allclose(bf16_host(D), expect, rtol=2.0 ** -7, atol=0)  # at most one bf16 ulp


def test_gemm_output_only_16_byte_aligned():
    """D at a 16-byte (not 32-byte) offset with a row stride of N + 8 elements:
    the epilogue keeps 16-byte stores there (32-byte stores need 32-byte rows)."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    pb = make_problem([150], 256, 256, seed=7)
    ldd = 256 + 8
    buf = torch.full((8 + 256 * ldd,), float("nan"), dtype=torch.bfloat16, device="cuda")
    D = buf[8:]
    assert D.data_ptr() % 32 == 16
    B.nvfp4_grouped_gemm(dev(pb["A"]), dev(pb["SFA"]), dev(pb["a_gs"]), dev(pb["B"]), dev(pb["SFB"]),
                         dev(pb["b_gs"]), dev(pb["padded"]), dev(pb["counts"]), 1, pb["cap"], 256, 256, D, ldd, 0)
    torch.cuda.synchronize()
    got = bf16_host(D[:150 * ldd].view(150, ldd))
    check(pb, got[None, :, :256])
    assert np.all(np.isnan(got[:, 256:]))  # the gap between rows is not written


def test_gemm_device_status_is_clean():
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    pb = make_problem([64], 256, 256, seed=2)
    run_gpu(pb)
    assert B.nvfp4_device_status(reset=False) == 0


def test_stalled_pipeline_reports_timeout_and_context_survives(cta_pair):
    """Failure detection without a fault: with the TMA producer switched off the
    consumers' bounded waits run out, the kernel reports a device timeout,
    frees its tensor memory and returns; the same process then runs a correct
    GEMM with a clean status."""
    import time
    import torch
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    pb = make_problem([128], 256, 256, seed=4)
    B.nvfp4_device_status(reset=True)
    D = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    t0 = time.time()
    B.nvfp4_debug_gemm_stall(dev(pb["A"]), dev(pb["SFA"]), dev(pb["a_gs"]), dev(pb["B"]), dev(pb["SFB"]),
                             dev(pb["b_gs"]), dev(pb["padded"]), 1, pb["cap"], 256, 256, D, 256, 200)
    torch.cuda.synchronize()
    assert time.time() - t0 < 30
    assert B.nvfp4_device_status(reset=True) == B.NVFP4_ERR_DEVICE_TIMEOUT
    assert not D.any()  # nothing was stored
    check(pb, run_gpu(pb))  # the context still works and the result is right
    assert B.nvfp4_device_status() == 0



@pytest.mark.parametrize("counts,N,K", [
    ([300], 200, 256),            # N not a multiple of 16: the last 8 columns stored alone
    ([100, 0, 260], 136, 320),    # one 128-row B half plus 8 columns of the next
    ([37, 129, 5], 384, 512),     # a tile and a half
    ([64], 8, 128),               # a single 8-column group
])
def test_grouped_gemm_ragged_n_matches_oracle(counts, N, K, cta_pair):
    """N a multiple of 8 only: the columns past N in a group's last tile are
    computed from the next group's B rows (or zeros past the last group) and
    never stored; each group's scales span whole 128-row tiles."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    pb = make_problem(counts, N, K, seed=sum(counts) + N + K)
    G = pb["G"]
    maxrows = int(np.diff(pb["padded"]).max())
    ld = N + 8  # a gap after each row that must stay untouched
    D = torch.full((G, maxrows, ld), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.nvfp4_grouped_gemm(dev(pb["A"]), dev(pb["SFA"]), dev(pb["a_gs"]), dev(pb["B"]), dev(pb["SFB"]),
                         dev(pb["b_gs"]), dev(pb["padded"]), dev(pb["counts"]), G, pb["cap"], N, K, D, ld,
                         maxrows * ld)
    torch.cuda.synchronize()
    got = bf16_host(D)
    check(pb, got[:, :, :N])
    assert np.all(np.isnan(got[:, :, N:]))
