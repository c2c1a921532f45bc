"""GPU parity at the full sizes of the five workloads, in the launch
configuration the benchmark uses.

- dense GEMM (M=2048, K=3584, N=6144): quantization bit-exact, full GEMM output
  vs the oracle's FP64 GEMM (bf16-rounded relative Frobenius <= 1e-3);
- grouped linear (G=8, T=2048, D=2048, R=1024, strided (T,G,D) input and
  (T,G,R) output): same checks per group;
- decode MoE (T=128, H=4096, I=2048, E=32, k=6): everything of the small MoE
  parity test (bit-exact metadata / weights / L1 activations, end to end
  relative Frobenius <= 2e-2, cosine >= 0.999);
- prefill MoE (T=8192, E=48, Zipf prior): routing and slot metadata bit-exact
  for all 8,192 tokens, weights of the sampled experts bit-exact, and the
  output of sampled tokens (tokens whose experts are all among the most
  popular ones plus the least popular one) computed one by one by the oracle.
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


def test_prefill_moe_full_size_sampled_tokens():
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl = W.prefill_moe()
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.top_k
    hidden = W.bf16_bits_to_f32(wl.hidden)
    ids, wts = O.route(wl.logits, k)
    meta = O.sort_slots(ids, wts, E)
    order = np.argsort(-meta["counts"], kind="stable")
    experts = set(order[:8].tolist()) | {int(order[-1])}
    cand = [t for t in range(T) if set(ids[t].tolist()) <= experts]
    with_small = [t for t in cand if int(order[-1]) in ids[t]]
    rng = np.random.default_rng(0)
    sample = sorted(set(rng.choice(cand, 20, replace=False).tolist()) | set(with_small[:4]))
    # oracle: weights of the sampled experts, activation scales from the workload
    q13, q2 = {}, {}
    a1 = np.ones(E, np.float32)
    a2 = np.ones(E, np.float32)
    for e in range(E):
        lo, n = int(meta["offsets"][e]), int(meta["counts"][e])
        if n:
            a1[e] = O.global_scale(np.abs(hidden[meta["sorted_token_ids"][lo:lo + n]]).max())
    for e in sorted(experts):
        q13[e] = O.quantize_expert_weights(W.bf16_bits_to_f32(wl.w13[e:e + 1]))
        q2[e] = O.quantize_expert_weights(W.bf16_bits_to_f32(wl.w2[e:e + 1]))
        lo, n = int(meta["offsets"][e]), int(meta["counts"][e])
        x = hidden[meta["sorted_token_ids"][lo:lo + min(n, 256)]]
        h = O.expert_l1(x, a1[e], q13[e][0][0], q13[e][1][0], q13[e][2][0], wl.gate_limit, wl.up_limit)
        a2[e] = O.global_scale(np.abs(h).max())
    # device: the whole layer
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    fwd = api.MoEForward(T, H, I, E, k)
    out = fwd(bf16_dev(wl.hidden), dev(wl.logits), w, dev(a1), dev(a2), wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    # metadata for all tokens, bit-exact
    A = T * k
    np.testing.assert_array_equal(host(fwd.view("topk_ids", torch.int32, A)).reshape(T, k), ids)
    np.testing.assert_allclose(host(fwd.view("topk_w", torch.float32, A)).reshape(T, k), wts, rtol=1e-6, atol=1e-7)
    P = meta["P"]
    np.testing.assert_array_equal(host(fwd.view("offsets", torch.int32, E + 1)), meta["offsets"])
    np.testing.assert_array_equal(host(fwd.view("sorted_token_ids", torch.int32, P)), meta["sorted_token_ids"])
    np.testing.assert_array_equal(host(fwd.view("inverse", torch.int32, A)), meta["inverse"])
    # sampled experts' weights, bit-exact
    for e in sorted(experts):
        assert host(w.w13_gs)[e] == q13[e][2][0] and host(w.w2_gs)[e] == q2[e][2][0]
        np.testing.assert_array_equal(host(w.w13[e]), O.pack_nibbles(q13[e][0][0]))
        np.testing.assert_array_equal(host(w.w2[e]), O.pack_nibbles(q2[e][0][0]))
    # gathered L1 activation rows of the sampled tokens, bit-exact
    a1_dev = fwd.view("a1", torch.uint8, P * H // 2)
    for t in sample[:6]:
        for j in range(k):
            r = int(meta["inverse"][t * k + j])
            nib, _ = O.quantize_blocks(hidden[t:t + 1], a1[ids[t, j]])
            np.testing.assert_array_equal(host(a1_dev[r * H // 2:(r + 1) * H // 2]), O.pack_nibbles(nib)[0])
    # sampled token outputs, one by one
    got = bf16_host(out)
    refs = []
    for t in sample:
        acc = np.zeros(H)
        for j in range(k):
            e = int(ids[t, j])
            h = O.expert_l1(hidden[t:t + 1], a1[e], q13[e][0][0], q13[e][1][0], q13[e][2][0], wl.gate_limit,
                            wl.up_limit)
            acc += wts[t, j] * O.expert_l2(h, a2[e], q2[e][0][0], q2[e][1][0], q2[e][2][0])[0]
        refs.append(O.bf16_round(acc.astype(np.float32)))
    refs = np.stack(refs)
    g = got[sample]
    assert np.all(np.isfinite(got))
    rf, cs = rel_frob(g, refs), cosine(g, refs)
    assert rf <= 2e-2 and cs >= 0.999, (rf, cs)
