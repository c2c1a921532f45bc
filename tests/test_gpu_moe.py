"""GPU parity of the full NVFP4 MoE forward against the oracle.

Bit-exact: routing ids, slot counts / offsets / sorted token ids / inverse
map, quantized expert weights and the gathered L1 activations (nibbles and
tile-layout scales).  Routing weights: 1e-6 relative.  L1 output
requantization: FP32 (kernel) vs FP64 (oracle) accumulation may flip a
rounding boundary, so the L2 input is compared on its dequantized values.
End-to-end output: relative Frobenius <= 2e-2 and cosine >= 0.999."""
import numpy as np
import pytest

from oracle import nvfp4_oracle as O
from nvfp4_mixture_experts_expert_gb300 import workloads as W
from helpers import OracleMoE, bf16_dev, bf16_host, cosine, dev, host, rel_frob

pytestmark = pytest.mark.gpu


def run_gpu(wl, orc):
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    out = fwd(bf16_dev(wl.hidden), dev(wl.logits), w, dev(orc.a1_gs), dev(orc.a2_gs), wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    return w, fwd, out


def check_all(wl, orc, w, fwd, out, check_a2=True):
    import torch
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.top_k
    # quantized weights (GPU quantizer) == oracle quantizer
    np.testing.assert_array_equal(host(w.w13_gs), orc.w13q[2])
    np.testing.assert_array_equal(host(w.w2_gs), orc.w2q[2])
    for e in range(E):
        np.testing.assert_array_equal(host(w.w13[e]), O.pack_nibbles(orc.w13q[0][e]))
        np.testing.assert_array_equal(host(w.w2[e]), O.pack_nibbles(orc.w2q[0][e]))
        np.testing.assert_array_equal(
            host(w.w13_sf[e]), O.assemble_scales(orc.w13q[1][e], np.array([0, 2 * I]), np.array([0, 2 * I])))
    # routing and slots
    A = T * k
    np.testing.assert_array_equal(host(fwd.view("topk_ids", torch.int32, A)).reshape(T, k), orc.ids)
    wts = host(fwd.view("topk_w", torch.float32, A)).reshape(T, k)
    np.testing.assert_allclose(wts, orc.w, rtol=1e-6, atol=1e-7)
    m = orc.meta
    P = m["P"]
    np.testing.assert_array_equal(host(fwd.view("counts", torch.int32, E)), m["counts"])
    np.testing.assert_array_equal(host(fwd.view("offsets", torch.int32, E + 1)), m["offsets"])
    assert host(fwd.view("meta", torch.int32, 2)).tolist() == [P, P // 128]
    np.testing.assert_array_equal(host(fwd.view("sorted_token_ids", torch.int32, P)), m["sorted_token_ids"])
    np.testing.assert_array_equal(host(fwd.view("inverse", torch.int32, A)), m["inverse"])
    np.testing.assert_allclose(host(fwd.view("row_weight", torch.float32, P)), m["row_weight"], rtol=1e-6, atol=1e-7)
    # gathered + quantized L1 activations
    a1_ref, sfa1_ref = orc.slot_activations()
    real = m["sorted_token_ids"] >= 0  # pad rows: zero scales, nibble bytes unspecified
    np.testing.assert_array_equal(host(fwd.view("a1", torch.uint8, P * H // 2)).reshape(P, H // 2)[real],
                                  a1_ref[real])
    np.testing.assert_array_equal(host(fwd.view("sfa1", torch.uint8, P * H // 16)), sfa1_ref)
    # end to end
    ref, inter = orc.forward()
    got = bf16_host(out)
    assert np.all(np.isfinite(got))
    rf, cs = rel_frob(got, ref), cosine(got, ref)
    assert rf <= 2e-2 and cs >= 0.999, (rf, cs)
    if check_a2:
        # L2 input: compare dequantized requantized activations on real rows
        a2 = host(fwd.view("a2", torch.uint8, P * I // 2)).reshape(P, I // 2)
        sfa2 = host(fwd.view("sfa2", torch.uint8, P * I // 16))
        s_lin = O.unswizzle_scales(sfa2, P, I // 16)
        deq = O.dequant_blocks(O.unpack_nibbles(a2), s_lin)
        for e, d in inter["experts"].items():
            lo, n = int(m["offsets"][e]), int(m["counts"][e])
            nib, s = O.quantize_blocks(d["h"], orc.a2_gs[e])
            ref_deq = O.dequant_blocks(nib, s)
            assert rel_frob(deq[lo:lo + n], ref_deq) <= 2e-2
            assert np.mean(O.unpack_nibbles(a2[lo:lo + n]) != nib) <= 0.02
        # pad rows of the L2 input stay zero
        for e in range(E):
            lo, n, hi = int(m["offsets"][e]), int(m["counts"][e]), int(m["offsets"][e + 1])
            assert not a2[lo + n:hi].any()
    return rf, cs


def test_tiny_moe_matches_oracle():
    wl = W.tiny_moe()
    orc = OracleMoE(wl)
    check_all(wl, orc, *run_gpu(wl, orc))


@pytest.mark.parametrize("case", ["empty_expert", "heavy_expert", "top1", "single_expert", "ragged_T", "K128"])
def test_moe_edge_cases(case):
    kw = dict(T=96, H=256, I=128, E=6, top_k=2, seed=21)
    extra = {}
    if case == "empty_expert":
        extra["dead_experts"] = (1, 4)
    elif case == "heavy_expert":
        kw.update(T=300)
        extra["logit_bias_std"] = 3.0  # one or two experts take well over 128 rows
    elif case == "top1":
        kw.update(top_k=1)
    elif case == "single_expert":
        kw.update(E=1, top_k=1)
    elif case == "ragged_T":
        kw.update(T=133, H=512, I=256, E=5, top_k=3)
    elif case == "K128":
        kw.update(H=256, I=128, E=3)
    wl = W.moe_workload(kw["T"], kw["H"], kw["I"], kw["E"], kw["top_k"], kw["seed"], **extra)
    orc = OracleMoE(wl)
    if case == "heavy_expert":
        assert orc.meta["counts"].max() > 128
    if case == "empty_expert":
        assert orc.meta["counts"][1] == 0 and orc.meta["counts"][4] == 0
    check_all(wl, orc, *run_gpu(wl, orc))


def _forced_routing(wl, first, second=None):
    """Overwrite the router logits so that token t takes expert first[t] (and
    second[t] next, for top_k 2) by a wide margin; the rest stays random."""
    lg = wl.logits.astype(np.float32).copy()
    t = np.arange(wl.T)
    lg[t, first] += np.float32(40.0)
    if second is not None:
        lg[t, second] += np.float32(20.0)
    wl.logits = lg
    return wl


def test_moe_experts_with_exactly_128_and_129_rows():
    """Expert 0 fills exactly one m-tile, expert 1 spills one row into a second
    tile, expert 2 takes 300 rows (three tiles, the last ragged), expert 3 43."""
    wl = W.moe_workload(300, 256, 128, 5, 2, 41)
    first = np.where(np.arange(300) < 128, 0, np.where(np.arange(300) < 257, 1, 2))
    second = np.where(np.arange(300) < 257, 2, 3)
    _forced_routing(wl, first, second)
    orc = OracleMoE(wl)
    assert orc.meta["counts"].tolist() == [128, 129, 300, 43, 0]
    check_all(wl, orc, *run_gpu(wl, orc))


@pytest.mark.parametrize("k", [1, 2])
def test_moe_all_tokens_on_one_expert(k):
    """Every token's first choice is expert 2 (and, for top_k 2, its second
    choice expert 0): the other experts get no row."""
    wl = W.moe_workload(200, 256, 128, 4, k, 43)
    _forced_routing(wl, np.full(200, 2), np.zeros(200, np.int64) if k == 2 else None)
    orc = OracleMoE(wl)
    assert orc.meta["counts"].tolist() == ([0, 0, 200, 0] if k == 1 else [200, 0, 200, 0])
    check_all(wl, orc, *run_gpu(wl, orc))


def test_moe_swiglu_clamps_active():
    """Limits small enough that a fifth of the gate values and a third of the
    up values are clamped in the L1 epilogue (gate from above only, before
    the SiLU; up on both sides)."""
    wl = W.moe_workload(150, 256, 128, 5, 2, 49)
    wl.gate_limit, wl.up_limit = 0.25, 0.3
    orc = OracleMoE(wl)
    ref, inter = orc.forward()
    e = next(iter(inter["experts"]))
    toks = inter["experts"][e]["toks"]
    G = O.dequant_blocks(*O.quantize_blocks(orc.hidden[toks], orc.a1_gs[e])) / orc.a1_gs[e] @ \
        (O.dequant_blocks(orc.w13q[0][e], orc.w13q[1][e]) / orc.w13q[2][e]).T
    assert np.mean(G[:, :wl.I] > wl.gate_limit) > 0.15 and np.mean(np.abs(G[:, wl.I:]) > wl.up_limit) > 0.15
    check_all(wl, orc, *run_gpu(wl, orc))


def test_moe_all_zero_hidden_states():
    """All-zero input: calibration gives every scale 1 (the amax == 0 rule),
    the gathered activations are all zero codes and the output is exactly 0."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.moe_workload(90, 256, 128, 4, 2, 47)
    wl.hidden = np.zeros_like(wl.hidden)
    orc = OracleMoE(wl)
    assert np.all(orc.a1_gs == 1) and np.all(orc.a2_gs == 1)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    a1, a2 = fwd.calibrate(bf16_dev(wl.hidden), dev(wl.logits), w, wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(a1), orc.a1_gs)
    np.testing.assert_array_equal(host(a2), orc.a2_gs)
    out = fwd(bf16_dev(wl.hidden), dev(wl.logits), w, a1, a2, wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    assert not host(out.view(torch.int16)).any()  # +0.0 everywhere
    ref, _ = orc.forward()
    assert not ref.any()
    P = orc.meta["P"]
    real = orc.meta["sorted_token_ids"] >= 0
    assert not host(fwd.view("a1", torch.uint8, P * wl.H // 2)).reshape(P, -1)[real].any()
    assert not host(fwd.view("sfa1", torch.uint8, P * wl.H // 16)).any()


def test_moe_hidden_16_byte_aligned_and_half_chunk_rows():
    """The gather reads each 16-element block with one 32-byte load only where
    the hidden states are 32-byte aligned; a pointer that is 16-byte but not
    32-byte aligned takes the two-load path.  H = 768 also leaves the last
    512-element chunk of every row half filled."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.moe_workload(70, 768, 256, 5, 3, 33)
    orc = OracleMoE(wl)
    flat = bf16_dev(wl.hidden).reshape(-1)
    buf = torch.empty(flat.numel() + 8, dtype=torch.bfloat16, device="cuda")
    hidden = buf[8:].view(wl.T, wl.H)
    hidden.copy_(flat.view(wl.T, wl.H))
    assert hidden.data_ptr() % 32 == 16
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    out = fwd(hidden, dev(wl.logits), w, dev(orc.a1_gs), dev(orc.a2_gs), wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    check_all(wl, orc, w, fwd, out)


def test_moe_pair_and_single_cta_gemms_are_bit_identical():
    """The MoE forward with the paired-CTA GEMMs and with single-CTA GEMMs:
    identical L2 inputs (SwiGLU + requantization epilogue) and outputs
    (routing-weighted combine epilogue), bit for bit."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api, binding as B
    wl = W.moe_workload(300, 512, 256, 5, 3, 41, logit_bias_std=1.5)
    orc = OracleMoE(wl)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    res = {}
    prev = B.nvfp4_gemm_set_cta_pair(True)
    try:
        for pair in (True, False):
            B.nvfp4_gemm_set_cta_pair(pair)
            out = fwd(bf16_dev(wl.hidden), dev(wl.logits), w, dev(orc.a1_gs), dev(orc.a2_gs), wl.gate_limit,
                      wl.up_limit)
            torch.cuda.synchronize()
            P = int(host(fwd.view("meta", torch.int32, 1))[0])
            res[pair] = (host(out.view(torch.int16)), host(fwd.view("a2", torch.uint8, P * wl.I // 2)),
                         host(fwd.view("sfa2", torch.uint8, P * wl.I // 16)))
    finally:
        B.nvfp4_gemm_set_cta_pair(prev)
    counts = orc.meta["counts"]
    assert (np.asarray(counts) > 128).any() and ((np.asarray(counts) + 127) // 128 % 2 == 1).any()
    for a, b in zip(res[True], res[False]):
        np.testing.assert_array_equal(a, b)


def test_host_pipeline_matches_direct_forward():
    """Three batches streamed from pinned host memory (uploads and downloads
    overlapping the forwards) give the same outputs, bit for bit, as direct
    forwards of the same batches."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.moe_workload(200, 512, 256, 6, 2, 51)
    orc = OracleMoE(wl)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    a1, a2 = dev(orc.a1_gs), dev(orc.a2_gs)
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    rng = np.random.default_rng(5)
    batches = []
    for i in range(3):
        h = bf16_dev(wl.hidden) * (1.0 + 0.25 * i)
        lg = dev(wl.logits + rng.standard_normal(wl.logits.shape).astype(np.float32))
        batches.append((h, lg))
    direct = [host(fwd(h, lg, w, a1, a2, wl.gate_limit, wl.up_limit).view(torch.int16)) for h, lg in batches]
    torch.cuda.synchronize()
    pipe = api.HostPipeline(fwd, w, a1, a2, wl.gate_limit, wl.up_limit)
    h_in = [(h.cpu().pin_memory(), lg.cpu().pin_memory()) for h, lg in batches]
    h_out = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory() for _ in batches]
    for (hh, hl), ho in zip(h_in, h_out):
        pipe.submit(hh, hl, ho)
    pipe.synchronize()
    for got, ref in zip(h_out, direct):
        np.testing.assert_array_equal(got.view(torch.int16).numpy(), ref)


def test_forward_captured_in_a_cuda_graph_replays_bit_exactly():
    """The forward (7 kernels with programmatic dependent launch, no host
    synchronisation) captured into a CUDA graph: replays on new inputs written
    into the same buffers give the eager results bit for bit."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.moe_workload(300, 512, 256, 6, 2, 61, logit_bias_std=1.0)
    orc = OracleMoE(wl)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    a1, a2 = dev(orc.a1_gs), dev(orc.a2_gs)
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    hidden, logits = bf16_dev(wl.hidden), dev(wl.logits)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    fwd(hidden, logits, w, a1, a2, wl.gate_limit, wl.up_limit, out=out)  # eager call first
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fwd(hidden, logits, w, a1, a2, wl.gate_limit, wl.up_limit, out=out, stream=s)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    for i in range(2):
        new_h = bf16_dev(wl.hidden) * (1.5 - 0.5 * i)
        new_l = dev(wl.logits + rng.standard_normal(wl.logits.shape).astype(np.float32))
        ref = fwd(new_h, new_l, w, a1, a2, wl.gate_limit, wl.up_limit).clone()
        hidden.copy_(new_h)
        logits.copy_(new_l)
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(out.view(torch.int16)), host(ref.view(torch.int16)))


def _routed_case(T=150, H=512, I=256, E=6, k=3, n_global=16, start=4, seed=71):
    wl = W.moe_workload(T, H, I, E, k, seed)
    orc = OracleMoE(wl)
    rng = np.random.default_rng(seed)
    gids = rng.integers(0, n_global, (T, k)).astype(np.int32)
    gids[7] = [0, 1, n_global - 1]      # no local expert
    gids[8] = [start, start + E - 1, start - 1]  # both ends of the local range and one below
    gw = rng.uniform(0.05, 1.0, (T, k)).astype(np.float32)
    return wl, orc, gids, gw, start


def test_routed_forward_matches_oracle():
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl, orc, gids, gw, start = _routed_case()
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.top_k
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(T, H, I, E, k)
    out = fwd.routed(bf16_dev(wl.hidden), dev(gids), dev(gw), start, w, dev(orc.a1_gs), dev(orc.a2_gs),
                     wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    ids, wts = O.remap_global_ids(gids, gw.astype(np.float64), start, E)
    m = O.sort_slots(ids, wts, E)
    A, P = T * k, m["P"]
    np.testing.assert_array_equal(host(fwd.view("topk_ids", torch.int32, A)).reshape(T, k), ids)
    np.testing.assert_array_equal(host(fwd.view("topk_w", torch.float32, A)).reshape(T, k), wts.astype(np.float32))
    np.testing.assert_array_equal(host(fwd.view("counts", torch.int32, E)), m["counts"])
    np.testing.assert_array_equal(host(fwd.view("offsets", torch.int32, E + 1)), m["offsets"])
    np.testing.assert_array_equal(host(fwd.view("sorted_token_ids", torch.int32, P)), m["sorted_token_ids"])
    np.testing.assert_array_equal(host(fwd.view("inverse", torch.int32, A)), m["inverse"])
    hidden = W.bf16_bits_to_f32(wl.hidden)
    ref = O.moe_forward_routed(hidden, ids, wts.astype(np.float32).astype(np.float64), orc.w13q, orc.w2q,
                               orc.a1_gs, orc.a2_gs, wl.gate_limit, wl.up_limit)
    got = bf16_host(out)
    assert not got[7].any()  # no local expert: zero row
    rf, cs = rel_frob(got, ref), cosine(got, ref)
    assert rf <= 2e-2 and cs >= 0.999, (rf, cs)


def test_routed_forward_matches_oracle_multi_block_routing():
    """T above the single-block routing limit: the routing, scan and scatter
    kernels of large batches, on external ids."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl, orc, gids, gw, start = _routed_case(T=600, seed=77)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.top_k
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(T, H, I, E, k)
    out = fwd.routed(bf16_dev(wl.hidden), dev(gids), dev(gw), start, w, dev(orc.a1_gs), dev(orc.a2_gs),
                     wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    ids, wts = O.remap_global_ids(gids, gw.astype(np.float64), start, E)
    m = O.sort_slots(ids, wts, E)
    np.testing.assert_array_equal(host(fwd.view("offsets", torch.int32, E + 1)), m["offsets"])
    np.testing.assert_array_equal(host(fwd.view("sorted_token_ids", torch.int32, m["P"])), m["sorted_token_ids"])
    np.testing.assert_array_equal(host(fwd.view("inverse", torch.int32, T * k)), m["inverse"])
    ref = O.moe_forward_routed(W.bf16_bits_to_f32(wl.hidden), ids, wts.astype(np.float32).astype(np.float64),
                               orc.w13q, orc.w2q, orc.a1_gs, orc.a2_gs, wl.gate_limit, wl.up_limit)
    got = bf16_host(out)
    rf, cs = rel_frob(got, ref), cosine(got, ref)
    assert rf <= 2e-2 and cs >= 0.999, (rf, cs)


def test_routed_forward_with_the_forward_own_routing_is_bit_identical():
    """The routing the logit forward computed on the device, shifted to global
    ids, gives the routed forward the logit forward's output bit for bit."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.moe_workload(200, 512, 256, 6, 2, 73, logit_bias_std=1.0)
    orc = OracleMoE(wl)
    T, k = wl.T, wl.top_k
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, k)
    a1, a2 = dev(orc.a1_gs), dev(orc.a2_gs)
    ref = fwd(bf16_dev(wl.hidden), dev(wl.logits), w, a1, a2, wl.gate_limit, wl.up_limit).clone()
    ids = fwd.view("topk_ids", torch.int32, T * k).clone() + 37
    wts = fwd.view("topk_w", torch.float32, T * k).clone()
    out = fwd.routed(bf16_dev(wl.hidden), ids, wts, 37, w, a1, a2, wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(out.view(torch.int16)), host(ref.view(torch.int16)))


def test_routed_forward_with_no_local_expert_is_zero():
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl, orc, gids, gw, start = _routed_case(T=40, seed=75)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    out = torch.full((wl.T, wl.H), 1.0, dtype=torch.bfloat16, device="cuda")
    far = np.full_like(gids, start + wl.E + 3)
    fwd.routed(bf16_dev(wl.hidden), dev(far), dev(gw), start, w, dev(orc.a1_gs), dev(orc.a2_gs), wl.gate_limit,
               wl.up_limit, out=out)
    torch.cuda.synchronize()
    assert not bf16_host(out).any()
    assert host(fwd.view("meta", torch.int32, 1))[0] == 0


def test_moe_zero_tokens_is_a_no_op():
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    import torch
    assert B.nvfp4_moe_workspace_size(0, 256, 128, 4, 2) > 0
    B.nvfp4_moe_forward(None, None, 0, 256, 128, 4, 2, None, None, None, None, None, None, None, None, 10.0, 10.0,
                        None, 0, None)
    torch.cuda.synchronize()


def test_device_calibration_matches_oracle_scales():
    """nvfp4_moe_calibrate: L1 scales bit-exact (same amax, same FP32 division);
    L2 scales from the kernel's own FP32 L1 output within 1% of the oracle's."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.moe_workload(150, 256, 128, 6, 2, 33, dead_experts=(3,), outlier_frac=0.02)
    orc = OracleMoE(wl)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    a1, a2 = fwd.calibrate(bf16_dev(wl.hidden), dev(wl.logits), w, wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(a1), orc.a1_gs)
    np.testing.assert_allclose(host(a2), orc.a2_gs, rtol=1e-2)
    assert host(a1)[3] == 1.0 and host(a2)[3] == 1.0  # the expert with no rows


@pytest.mark.parametrize("T", [150, 300])
def test_routed_calibration_matches_oracle_scales(T):
    """nvfp4_moe_calibrate_routed from global ids: L1 scales bit-exact, L2
    scales within 1 %; experts no token chose keep scale 1."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl, orc, gids, gw, start = _routed_case(T=T, seed=73)
    gids[:, :] = np.where(gids == start + 2, start - 1, gids)  # local expert 2 gets no row
    ids, _ = O.remap_global_ids(gids, gw.astype(np.float64), start, wl.E)
    a1_ref, a2_ref = O.calibrate_activation_scales_routed(orc.hidden, ids, orc.w13q, wl.gate_limit, wl.up_limit)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    a1, a2 = fwd.calibrate_routed(bf16_dev(wl.hidden), dev(gids), dev(gw), start, w, wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(a1), a1_ref)
    np.testing.assert_allclose(host(a2), a2_ref, rtol=1e-2)
    assert host(a1)[2] == 1.0 and host(a2)[2] == 1.0


def test_routing_ties_and_signed_zero_match_oracle():
    """Exactly equal logits go to the lower expert; -0 and +0 rank as equal."""
    import torch
    wl = W.moe_workload(40, 256, 128, 40, 8, 5)
    lg = wl.logits.copy()
    lg[0, :] = 1.5                       # all tied
    lg[1, 7] = lg[1, 3] = lg[1, 30] = 4.0  # a three-way tie at the top
    lg[2, :] = 0.0
    lg[2, 5] = -0.0
    lg[2, 9] = -0.0                      # zeros of both signs
    lg[3, 20:] = -np.inf                 # only 20 finite candidates
    wl.logits = np.ascontiguousarray(lg, np.float32)
    orc = OracleMoE(wl)
    w, fwd, out = run_gpu(wl, orc)
    ids = host(fwd.view("topk_ids", torch.int32, wl.T * wl.top_k)).reshape(wl.T, wl.top_k)
    np.testing.assert_array_equal(ids, orc.ids)
    assert ids[0].tolist() == list(range(8)) and ids[1, :3].tolist() == [3, 7, 30]
    wts = host(fwd.view("topk_w", torch.float32, wl.T * wl.top_k)).reshape(wl.T, wl.top_k)
    np.testing.assert_allclose(wts, orc.w, rtol=1e-6, atol=1e-7)


# ----------------------------------------------------------------- L2 scales from the batch

@pytest.mark.parametrize("T,H,I,E,k,dead", [(120, 512, 256, 6, 2, (3,)), (700, 256, 512, 5, 3, ())])
def test_batch_l2_scales_match_oracle(T, H, I, E, k, dead):
    """a2_gs NULL: the L1 GEMM stores bf16 h and per-expert amax, a quantize
    pass derives each expert's L2 scale.  Small and multi-block routing; an
    expert with no rows (scale 1); I > H (the bf16 h rows are wider than the
    output rows they share the workspace region with)."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.moe_workload(T, H, I, E, k, 91, dead_experts=dead)
    orc = OracleMoE(wl)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(T, H, I, E, k)
    out = fwd(bf16_dev(wl.hidden), dev(wl.logits), w, dev(orc.a1_gs), None, wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    ref, inter = O.moe_forward(orc.hidden, wl.logits, k, orc.w13q, orc.w2q, orc.a1_gs, None, wl.gate_limit,
                               wl.up_limit, return_intermediates=True)
    scales = host(fwd.batch_l2_scales())
    want = np.ones(E, np.float32)
    for e, d in inter["experts"].items():
        want[e] = d["a2_gs"]
    for e in dead:
        assert scales[e] == 1.0
    # amax of h from FP32 (kernel) vs FP64 (oracle) accumulation: one bf16 step at most
    np.testing.assert_allclose(scales, want, rtol=8e-3)
    assert np.mean(scales == want) >= 0.5
    got = bf16_host(out)
    rf, cs = rel_frob(got, ref), cosine(got, ref)
    assert rf <= 2e-2 and cs >= 0.999, (rf, cs)


@pytest.mark.parametrize("T", [100, 600])
def test_batch_l2_scales_bit_identical_to_the_same_scales_given(T):
    """The forward with a2_gs NULL and the forward given the scales it derived
    produce the same L2 activations and the same output, bit for bit (the
    separate quantize pass and the fused L1 requantization round alike)."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.moe_workload(T, 512, 256, 6, 2, 93, logit_bias_std=1.0)
    orc = OracleMoE(wl)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    hidden, logits, a1 = bf16_dev(wl.hidden), dev(wl.logits), dev(orc.a1_gs)
    out_dyn = fwd(hidden, logits, w, a1, None, wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    P = orc.meta["P"]
    a2_dyn = fwd.view("a2", torch.uint8, P * wl.I // 2).clone()
    sf_dyn = fwd.view("sfa2", torch.uint8, P * wl.I // 16).clone()
    scales = fwd.batch_l2_scales().clone()
    out_giv = fwd(hidden, logits, w, a1, scales, wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    assert torch.equal(fwd.view("a2", torch.uint8, P * wl.I // 2), a2_dyn)
    assert torch.equal(fwd.view("sfa2", torch.uint8, P * wl.I // 16), sf_dyn)
    assert torch.equal(out_dyn, out_giv)


# ----------------------------------------------------------------- routing at the small/large batch boundary

@pytest.mark.parametrize("T", [1, 31, 33, 255, 256, 257])
def test_routing_metadata_bit_exact_around_the_cluster_path(T):
    """Batches of at most 256 tokens route in one cluster of 8 CTAs of 32
    tokens each (distributed-shared-memory counts); 257 takes the three-kernel
    path.  Ids, weights, counts, offsets, slot order and inverse map match the
    oracle exactly at the CTA boundaries (1, 31, 33 tokens: empty and partial
    CTAs; 255, 256: the last CTA partial and full), and the output matches."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.moe_workload(T, 256, 128, 9, 3, 500 + T, logit_bias_std=1.0)
    orc = OracleMoE(wl)
    w, fwd, out = run_gpu(wl, orc)
    k, E = wl.top_k, wl.E
    A = T * k
    m = orc.meta
    P = m["P"]
    np.testing.assert_array_equal(host(fwd.view("topk_ids", torch.int32, A)).reshape(T, k), orc.ids)
    np.testing.assert_array_equal(host(fwd.view("counts", torch.int32, E)), m["counts"])
    np.testing.assert_array_equal(host(fwd.view("offsets", torch.int32, E + 1)), m["offsets"])
    assert host(fwd.view("meta", torch.int32, 2)).tolist() == [P, P // 128]
    np.testing.assert_array_equal(host(fwd.view("sorted_token_ids", torch.int32, P)), m["sorted_token_ids"])
    np.testing.assert_array_equal(host(fwd.view("inverse", torch.int32, A)), m["inverse"])
    tiles = np.searchsorted(m["offsets"], np.arange(P // 128) * 128, side="right") - 1
    np.testing.assert_array_equal(host(fwd.view("tile_expert", torch.int32, P // 128)), tiles)
    ref, _ = orc.forward()
    got = bf16_host(out)
    rf, cs = rel_frob(got, ref), cosine(got, ref)
    assert rf <= 2e-2 and cs >= 0.999, (rf, cs)


@pytest.mark.parametrize("T", [40, 250])
def test_routed_forward_on_the_cluster_path_matches_oracle(T):
    """External global ids through the cluster routing (non-local experts
    dropped inside each CTA), with the L2 scales taken from the batch."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl, orc, gids, gw, start = _routed_case(T=T, seed=80 + T)
    Tn, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.top_k
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(Tn, H, I, E, k)
    out = fwd.routed(bf16_dev(wl.hidden), dev(gids), dev(gw), start, w, dev(orc.a1_gs), None,
                     wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    ids, wts = O.remap_global_ids(gids, gw.astype(np.float64), start, E)
    m = O.sort_slots(ids, wts, E)
    np.testing.assert_array_equal(host(fwd.view("sorted_token_ids", torch.int32, m["P"])), m["sorted_token_ids"])
    np.testing.assert_array_equal(host(fwd.view("inverse", torch.int32, Tn * k)), m["inverse"])
    ref = O.moe_forward_routed(W.bf16_bits_to_f32(wl.hidden), ids, wts.astype(np.float32).astype(np.float64),
                               orc.w13q, orc.w2q, orc.a1_gs, None, wl.gate_limit, wl.up_limit)
    got = bf16_host(out)
    assert not got[7].any()
    rf, cs = rel_frob(got, ref), cosine(got, ref)
    assert rf <= 2e-2 and cs >= 0.999, (rf, cs)


def test_batch_l2_scale_forward_replays_from_a_cuda_graph():
    """The forward with a2_gs NULL (an amax reset, the bf16 L1 output and the
    quantize pass) captured in a CUDA graph replays bit-exactly."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.moe_workload(300, 512, 256, 6, 2, 62, logit_bias_std=1.0)
    orc = OracleMoE(wl)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    a1 = dev(orc.a1_gs)
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    hidden, logits = bf16_dev(wl.hidden), dev(wl.logits)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    fwd(hidden, logits, w, a1, None, wl.gate_limit, wl.up_limit, out=out)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fwd(hidden, logits, w, a1, None, wl.gate_limit, wl.up_limit, out=out, stream=s)
    torch.cuda.synchronize()
    for i in range(2):
        new_h = bf16_dev(wl.hidden) * (2.0 - 0.75 * i)
        ref = fwd(new_h, logits, w, a1, None, wl.gate_limit, wl.up_limit).clone()
        hidden.copy_(new_h)
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(out.view(torch.int16)), host(ref.view(torch.int16)))


@pytest.mark.parametrize("T,E,k", [(200, 256, 8), (600, 100, 4), (120, 65, 2)])
def test_many_experts_match_oracle(T, E, k):
    """Many experts: 256 (eight 32-expert key slots per lane in the routing,
    the cluster path, the most groups the CTA-pair GEMM takes), 100 on the
    multi-block path and 65 just past two key slots.  Routing metadata
    bit-exact, output within the end-to-end tolerance."""
    import torch
    wl = W.moe_workload(T, 256, 128, E, k, 900 + E, logit_bias_std=0.5)
    orc = OracleMoE(wl)
    w, fwd, out = run_gpu(wl, orc)
    A, m = T * k, orc.meta
    P = m["P"]
    np.testing.assert_array_equal(host(fwd.view("topk_ids", torch.int32, A)).reshape(T, k), orc.ids)
    np.testing.assert_allclose(host(fwd.view("topk_w", torch.float32, A)).reshape(T, k), orc.w, rtol=1e-6, atol=1e-7)
    np.testing.assert_array_equal(host(fwd.view("offsets", torch.int32, E + 1)), m["offsets"])
    np.testing.assert_array_equal(host(fwd.view("sorted_token_ids", torch.int32, P)), m["sorted_token_ids"])
    np.testing.assert_array_equal(host(fwd.view("inverse", torch.int32, A)), m["inverse"])
    ref, _ = orc.forward()
    got = bf16_host(out)
    rf, cs = rel_frob(got, ref), cosine(got, ref)
    assert rf <= 2e-2 and cs >= 0.999, (rf, cs)
    if E == 256:  # the CTA-pair GEMMs at their largest group count give the same bits
        from nvfp4_mixture_experts_expert_gb300 import binding as B
        prev = B.nvfp4_gemm_set_cta_pair(True)
        try:
            out2 = fwd(bf16_dev(wl.hidden), dev(wl.logits), w, dev(orc.a1_gs), dev(orc.a2_gs), wl.gate_limit,
                       wl.up_limit)
            torch.cuda.synchronize()
        finally:
            B.nvfp4_gemm_set_cta_pair(prev)
        np.testing.assert_array_equal(host(out2.view(torch.int16)), host(out.view(torch.int16)))


def test_small_batch_forward_replays_from_a_cuda_graph():
    """Small batches (the routing cluster launch, programmatic dependent launch
    from the first kernel) captured in a CUDA graph: replays on new inputs
    give the eager results bit for bit."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.moe_workload(100, 512, 256, 8, 4, 63, logit_bias_std=0.5)
    orc = OracleMoE(wl)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    a1, a2 = dev(orc.a1_gs), dev(orc.a2_gs)
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    hidden, logits = bf16_dev(wl.hidden), dev(wl.logits)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    fwd(hidden, logits, w, a1, a2, wl.gate_limit, wl.up_limit, out=out)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fwd(hidden, logits, w, a1, a2, wl.gate_limit, wl.up_limit, out=out, stream=s)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    for i in range(3):
        new_h = bf16_dev(wl.hidden) * (1.25 - 0.25 * i)
        new_l = dev(wl.logits + rng.standard_normal(wl.logits.shape).astype(np.float32))
        ref = fwd(new_h, new_l, w, a1, a2, wl.gate_limit, wl.up_limit).clone()
        hidden.copy_(new_h)
        logits.copy_(new_l)
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(out.view(torch.int16)), host(ref.view(torch.int16)))


def test_device_status_belongs_to_the_call_workspace():
    """Two forwards on two streams, each with its own workspace.  The one on
    stream 2 runs its L1 GEMM with the operand loads switched off (the
    failure-detection hook): its bounded waits give up after 300 ms and record
    the timeout in that call's workspace word only.  The forward on stream 1,
    the library-wide word and, afterwards, a normal forward on the stalled
    workspace all read OK; the normal results match the oracle."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api, binding as B
    wl = W.moe_workload(300, 256, 128, 4, 2, 31)
    orc = OracleMoE(wl)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    hidden, logits = bf16_dev(wl.hidden), dev(wl.logits)
    a1, a2 = dev(orc.a1_gs), dev(orc.a2_gs)
    fa = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    fb = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    out_a = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    out_b = torch.empty_like(out_a)
    torch.cuda.synchronize()
    B.nvfp4_device_status(reset=True)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    B.nvfp4_moe_set_debug_stall(300)
    try:
        fb(hidden, logits, w, a1, a2, wl.gate_limit, wl.up_limit, out=out_b, stream=s2)
    finally:
        B.nvfp4_moe_set_debug_stall(0)
    fa(hidden, logits, w, a1, a2, wl.gate_limit, wl.up_limit, out=out_a, stream=s1)
    torch.cuda.synchronize()
    assert fb.status(stream=s2) == B.NVFP4_ERR_DEVICE_TIMEOUT
    assert fa.status(stream=s1) == B.NVFP4_OK
    assert B.nvfp4_device_status() == B.NVFP4_OK
    ref = orc.forward()[0]
    got_a = bf16_host(out_a)
    assert rel_frob(got_a, ref) <= 2e-2 and cosine(got_a, ref) >= 0.999
    # the stalled workspace runs a normal forward next, with a clean status
    fb(hidden, logits, w, a1, a2, wl.gate_limit, wl.up_limit, out=out_b, stream=s2)
    torch.cuda.synchronize()
    assert fb.status(stream=s2) == B.NVFP4_OK
    np.testing.assert_array_equal(bf16_host(out_b).view(np.uint32), got_a.view(np.uint32))


# ----------------------------------------------------------------- L1 -> L2 hand-off per m-tile

@pytest.mark.parametrize("T,E,k", [(300, 5, 3), (128, 32, 6), (1000, 9, 2)])
def test_l1_l2_overlap_is_bit_identical(T, E, k):
    """The L2 GEMM taking the L1 output m-tile by m-tile (each L2 tile waits on
    the device until all of its m-tile's L1 n-tiles are stored) gives exactly
    the forward where it waits for the whole L1 GEMM: L2 input, output, and a
    clean status; repeated forwards reuse the per-m-tile counters."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api, binding as B
    wl = W.moe_workload(T, 1024, 512, E, k, 53, logit_bias_std=1.0)
    orc = OracleMoE(wl)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    args = (bf16_dev(wl.hidden), dev(wl.logits), w, dev(orc.a1_gs), dev(orc.a2_gs), wl.gate_limit, wl.up_limit)
    res = {}
    prev = B.nvfp4_moe_set_overlap(0)
    try:
        for ov in (0, 1, 1):
            B.nvfp4_moe_set_overlap(ov)
            out = fwd(*args)
            torch.cuda.synchronize()
            P = int(host(fwd.view("meta", torch.int32, 1))[0])
            res.setdefault(ov, []).append((host(out.view(torch.int16)).copy(),
                                           host(fwd.view("a2", torch.uint8, P * wl.I // 2)).copy()))
            assert fwd.status() == 0
    finally:
        B.nvfp4_moe_set_overlap(prev)
    for got in res[1]:
        for a, b in zip(got, res[0][0]):
            np.testing.assert_array_equal(a, b)
    P = orc.meta["P"]
    done = host(fwd.view("tile_done", torch.int32, P // 128))
    assert (done == wl.I // 128).all()  # every m-tile counted all of its L1 n-tiles
    ref, _ = orc.forward()
    rf, cs = rel_frob(bf16_host(out), ref), cosine(bf16_host(out), ref)
    assert rf <= 2e-2 and cs >= 0.999, (rf, cs)


@pytest.mark.parametrize("T,H,I,E,k", [(128, 512, 256, 8, 6), (300, 256, 512, 12, 3), (64, 1024, 384, 5, 2)])
def test_swapped_l2_gemm_is_bit_identical(T, H, I, E, k):
    """Small batches: the L2 GEMM with W2 tiles as the MMA's M operand and 64
    slot rows as N stores exactly the routing-weighted rows of the slot-major
    GEMM, with and without the L1 -> L2 hand-off, and the forward matches the
    oracle.  Expert sizes: 128 rows exactly and 78-125 (first case); 276,
    176, 134, 52, 1 and empty experts (second); at most 59 rows with I = 384,
    a partial last K-stage (third)."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api, binding as B
    wl = W.moe_workload(T, H, I, E, k, 71, logit_bias_std=1.5)
    orc = OracleMoE(wl)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    args = (bf16_dev(wl.hidden), dev(wl.logits), w, dev(orc.a1_gs), dev(orc.a2_gs), wl.gate_limit, wl.up_limit)
    res = {}
    prev = B.nvfp4_moe_set_swap_l2(0)
    prev_ov = B.nvfp4_moe_set_overlap(1)
    try:
        for sw, ov in ((0, 1), (1, 1), (1, 0)):
            B.nvfp4_moe_set_swap_l2(sw)
            B.nvfp4_moe_set_overlap(ov)
            out = fwd(*args)
            torch.cuda.synchronize()
            P = int(host(fwd.view("meta", torch.int32, 1))[0])
            real = orc.meta["sorted_token_ids"] >= 0
            y = host(fwd.view("y", torch.int16, P * H)).reshape(P, H)[real].copy()
            res[(sw, ov)] = (host(out.view(torch.int16)).copy(), y)
            assert fwd.status() == 0
    finally:
        B.nvfp4_moe_set_swap_l2(prev)
        B.nvfp4_moe_set_overlap(prev_ov)
    for key in ((1, 1), (1, 0)):
        for a, b in zip(res[key], res[(0, 1)]):
            np.testing.assert_array_equal(a, b)
    ref, _ = orc.forward()
    got = bf16_host(torch.from_numpy(res[(1, 1)][0]).view(torch.bfloat16))
    rf, cs = rel_frob(got, ref), cosine(got, ref)
    assert rf <= 2e-2 and cs >= 0.999, (rf, cs)
    # L2 scales from the batch (device-computed): the same rows either way
    batch = {}
    try:
        for sw in (0, 1):
            B.nvfp4_moe_set_swap_l2(sw)
            out = fwd(bf16_dev(wl.hidden), dev(wl.logits), w, dev(orc.a1_gs), None, wl.gate_limit, wl.up_limit)
            torch.cuda.synchronize()
            batch[sw] = host(out.view(torch.int16)).copy()
            assert fwd.status() == 0
    finally:
        B.nvfp4_moe_set_swap_l2(prev)
    np.testing.assert_array_equal(batch[1], batch[0])


# ----------------------------------------------------------------- FP8 L1 output (reading R20)

@pytest.mark.parametrize("T,H,I,E,k,dead", [(120, 512, 256, 6, 2, (3,)), (700, 256, 512, 5, 3, ())])
def test_fp8_l1_output_matches_oracle(T, H, I, E, k, dead):
    """L2 scales from the batch with the L1 output kept as FP8 blocks.  The L1
    GEMM computes the same bf16 h as in the bf16 mode (read from that mode),
    so every later step is checked bit for bit: the E4M3 codes and block
    exponents against the oracle's encoding of that h, each expert's L2 scale
    against 2688 / amax of the stored values, the requantized L2 input against
    the oracle's quantization of the stored values; then the output end to end."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.moe_workload(T, H, I, E, k, 95, dead_experts=dead)
    orc = OracleMoE(wl)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(T, H, I, E, k)
    hidden, logits, a1 = bf16_dev(wl.hidden), dev(wl.logits), dev(orc.a1_gs)
    fwd(hidden, logits, w, a1, None, wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    m = orc.meta
    P, cap = m["P"], fwd.layout["capacity"]
    h16 = W.bf16_bits_to_f32(host(fwd.view("h", torch.int16, P * I)).view(np.uint16).reshape(P, I))
    out = fwd(hidden, logits, w, a1, None, wl.gate_limit, wl.up_limit, l1_output="fp8")
    torch.cuda.synchronize()
    assert fwd.status() == 0
    region = host(fwd.view("h", torch.uint8, cap * I + cap * I // 16))
    codes = region[:P * I].reshape(P, I)
    kbytes = region[cap * I:cap * I + P * I // 16].reshape(P, I // 16)
    scales = host(fwd.batch_l2_scales())
    a2 = host(fwd.view("a2", torch.uint8, P * I // 2)).reshape(P, I // 2)
    s_lin = O.unswizzle_scales(host(fwd.view("sfa2", torch.uint8, P * I // 16)), P, I // 16)
    for e in range(E):
        lo, n = int(m["offsets"][e]), int(m["counts"][e])
        if n == 0:
            assert scales[e] == 1.0
            continue
        ref_codes, ref_k = O.fp8_block_encode(h16[lo:lo + n])
        np.testing.assert_array_equal(codes[lo:lo + n], ref_codes)
        np.testing.assert_array_equal(kbytes[lo:lo + n].astype(np.int64) - 127, ref_k)
        h8 = O.fp8_block_decode(codes[lo:lo + n], kbytes[lo:lo + n].astype(np.int64) - 127)
        assert scales[e] == O.global_scale(np.max(np.abs(h8))), e
        nib, s = O.quantize_blocks(h8, scales[e])
        np.testing.assert_array_equal(a2[lo:lo + n], O.pack_nibbles(nib))
        np.testing.assert_array_equal(s_lin[lo:lo + n], s)
    for e in dead:
        assert scales[e] == 1.0
    ref = O.moe_forward(orc.hidden, wl.logits, k, orc.w13q, orc.w2q, orc.a1_gs, None, wl.gate_limit, wl.up_limit,
                        l1_fp8=True)
    got = bf16_host(out)
    rf, cs = rel_frob(got, ref), cosine(got, ref)
    assert rf <= 2e-2 and cs >= 0.999, (rf, cs)
    with pytest.raises(ValueError):
        fwd(hidden, logits, w, a1, dev(orc.a2_gs), wl.gate_limit, wl.up_limit, l1_output="fp8")
