"""Pins of the oracle's routing, slot sort, GEMM and MoE forward against brute
force, closed forms and special cases (no GPU)."""
import numpy as np
import pytest

from oracle import nvfp4_oracle as O
from nvfp4_mixture_experts_expert_gb300 import workloads as W


# ----------------------------------------------------------------- routing

def brute_route(logits, k):
    T, E = logits.shape
    ids = np.zeros((T, k), np.int64)
    w = np.zeros((T, k))
    for t in range(T):
        # pick k times the largest remaining logit; ties -> lower expert index
        left = list(range(E))
        for j in range(k):
            best = left[0]
            for e in left[1:]:
                if logits[t, e] > logits[t, best]:
                    best = e
            ids[t, j] = best
            left.remove(best)
        p = np.exp(logits[t].astype(np.float64) - logits[t].max())
        p /= p.sum()                       # softmax over all experts ...
        w[t] = p[ids[t]] / p[ids[t]].sum()  # ... renormalised over the k chosen
    return ids, w


@pytest.mark.parametrize("T,E,k", [(17, 8, 2), (40, 48, 6), (9, 5, 5), (12, 3, 1)])
def test_route_matches_brute_force(T, E, k):
    rng = np.random.default_rng(T * 100 + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[0, :] = 0.5  # all tied: lowest indices win
    logits[1, 0] = logits[1, E - 1] = 9.0  # a tie between two experts
    ids, w = O.route(logits, k)
    bids, bw = brute_route(logits, k)
    np.testing.assert_array_equal(ids, bids)
    np.testing.assert_allclose(w, bw, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-12)
    assert ids[0].tolist() == list(range(k))


def brute_sort(ids, w, E):
    T, k = ids.shape
    rows = []
    off = [0]
    for e in range(E):
        mine = [(t, j) for t in range(T) for j in range(k) if ids[t, j] == e]
        pad = (len(mine) + 127) // 128 * 128
        rows += [(t, w[t, j], t * k + j) for (t, j) in mine] + [(-1, 0.0, -1)] * (pad - len(mine))
        off.append(off[-1] + pad)
    return off, rows


@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (200, 3, 2), (150, 4, 1), (30, 6, 3)])
def test_sort_slots_matches_brute_force(T, E, k):
    rng = np.random.default_rng(T + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    if E == 3:
        logits[:, 0] += 4  # expert 0 takes >128 rows: several 128-row chunks
    if E == 6:
        logits[:, 5] = -np.inf  # an empty expert
    ids, w = O.route(logits, k)
    m = O.sort_slots(ids, w, E)
    off, rows = brute_sort(ids, w, E)
    assert m["offsets"].tolist() == off
    assert m["P"] == len(rows) == off[-1]
    assert m["sorted_token_ids"].tolist() == [r[0] for r in rows]
    np.testing.assert_array_equal(m["row_weight"], [r[1] for r in rows])
    for row, (t, _, f) in enumerate(rows):
        if f >= 0:
            assert m["inverse"][f] == row
    assert np.all(np.asarray(off) % 128 == 0)
    assert m["P"] <= O.slot_capacity(T, k, E)


# ----------------------------------------------------------------- GEMM closed forms

def test_gemm_identity_weight_returns_dequantized_activation():
    rng = np.random.default_rng(7)
    M, K = 40, 64
    x = rng.standard_normal((M, K)).astype(np.float32)
    gs_a = O.global_scale(np.max(np.abs(x)))
    a_nib, a_s = O.quantize_blocks(x, gs_a)
    eye = np.eye(K, dtype=np.float32)  # one 1.0 per row: exactly representable
    b_nib, b_s, b_gs = O.weight_quantize(eye)
    np.testing.assert_array_equal(O.dequant_blocks(b_nib, b_s) / b_gs, eye)
    C = O.nvfp4_gemm(a_nib, a_s, gs_a, b_nib, b_s, b_gs)
    np.testing.assert_array_equal(C, O.dequant_blocks(a_nib, a_s) / np.float64(gs_a))


def test_gemm_permutation_weight_is_a_column_permutation():
    rng = np.random.default_rng(8)
    M, K = 8, 32
    x = rng.standard_normal((M, K)).astype(np.float32)
    gs_a = O.global_scale(np.max(np.abs(x)))
    a_nib, a_s = O.quantize_blocks(x, gs_a)
    perm = rng.permutation(K)
    P = np.zeros((K, K), np.float32)
    P[np.arange(K), perm] = 1.0  # output column n reads input column perm[n]
    b_nib, b_s, b_gs = O.weight_quantize(P)
    C = O.nvfp4_gemm(a_nib, a_s, gs_a, b_nib, b_s, b_gs)
    A = O.dequant_blocks(a_nib, a_s) / np.float64(gs_a)
    np.testing.assert_array_equal(C, A[:, perm])


def test_gemm_equals_plain_matmul_of_dequantized_operands():
    rng = np.random.default_rng(9)
    a = rng.standard_normal((16, 48)).astype(np.float32)
    b = rng.standard_normal((24, 48)).astype(np.float32)
    an, as_ = O.quantize_blocks(a, np.float32(2))
    bn, bs = O.quantize_blocks(b, np.float32(4))
    A = O.dequant_blocks(an, as_) / 2
    B = O.dequant_blocks(bn, bs) / 4
    ref = np.array([[sum(A[i, kk] * B[j, kk] for kk in range(48)) for j in range(24)] for i in range(16)])
    np.testing.assert_allclose(O.nvfp4_gemm(an, as_, 2, bn, bs, 4), ref, rtol=1e-12, atol=1e-12)


def test_grouped_gemm_is_per_group_matmul_with_empty_and_ragged_groups():
    rng = np.random.default_rng(12)
    rows, K, N = [5, 0, 17, 1], 32, 12
    a = rng.standard_normal((sum(rows), K)).astype(np.float32)
    gs_a = np.float32([2.0, 1.0, 0.5, 3.0])
    nib, sc = np.zeros((sum(rows), K), np.uint8), np.zeros((sum(rows), K // 16), np.uint8)
    r0 = 0
    for g, n in enumerate(rows):
        nib[r0:r0 + n], sc[r0:r0 + n] = O.quantize_blocks(a[r0:r0 + n], gs_a[g])
        r0 += n
    bq = [O.weight_quantize(rng.standard_normal((N, K)).astype(np.float32)) for _ in rows]
    out = O.grouped_gemm(nib, sc, gs_a, [b[0] for b in bq], [b[1] for b in bq], [b[2] for b in bq], rows)
    r0 = 0
    for g, n in enumerate(rows):
        A = O.dequant_blocks(nib[r0:r0 + n], sc[r0:r0 + n]) / np.float64(gs_a[g])
        B = O.dequant_blocks(bq[g][0], bq[g][1]) / np.float64(bq[g][2])
        ref = np.array([[sum(A[i, k] * B[j, k] for k in range(K)) for j in range(N)] for i in range(n)])
        assert out[g].shape == (n, N)
        np.testing.assert_allclose(out[g], ref.reshape(n, N), rtol=1e-12, atol=1e-12)
        r0 += n


def test_quantize_tensor_pads_rows_with_zero_codes_and_scales():
    rng = np.random.default_rng(13)
    x = rng.standard_normal((130, 64)).astype(np.float32)
    gs = O.global_scale(np.abs(x).max())
    packed, swz, lin = O.quantize_tensor(x, gs)
    nib, s = O.quantize_blocks(x, gs)
    assert packed.shape == (256, 32) and swz.size == 256 * 4
    np.testing.assert_array_equal(O.unpack_nibbles(packed[:130]), nib)
    assert not packed[130:].any()
    full = O.unswizzle_scales(swz, 256, 4)
    np.testing.assert_array_equal(full[:130], s)
    np.testing.assert_array_equal(lin, s)
    assert not full[130:].any()


# ----------------------------------------------------------------- MoE

def small_layer(T=48, H=64, I=32, E=5, k=2, seed=11):
    wl = W.moe_workload(T, H, I, E, k, seed, zero_block_frac=0.05, tiny_block_frac=0.05)
    hidden = W.bf16_bits_to_f32(wl.hidden)
    w13 = W.bf16_bits_to_f32(wl.w13)
    w2 = W.bf16_bits_to_f32(wl.w2)
    w13q = O.quantize_expert_weights(w13)
    w2q = O.quantize_expert_weights(w2)
    a1, a2 = O.calibrate_activation_scales(hidden, wl.logits, k, w13q)
    return wl, hidden, w13, w2, w13q, w2q, a1, a2


def dense_brute_moe(hidden, logits, k, w13q, w2q, a1, a2, gl, ul):
    """Every expert on every token, then masked by the routing: no slots, no sort."""
    T, H = hidden.shape
    E = w13q[0].shape[0]
    I = w13q[0].shape[1] // 2
    ids, w = brute_route(logits, k)
    out = np.zeros((T, H))
    for e in range(E):
        A = O.dequant_blocks(*O.quantize_blocks(hidden, a1[e])) / np.float64(a1[e])
        B = O.dequant_blocks(w13q[0][e], w13q[1][e]) / np.float64(w13q[2][e])
        G = A @ B.T
        g = np.minimum(G[:, :I], gl)
        u = np.clip(G[:, I:], -ul, ul)
        h = O.bf16_round((g / (1 + np.exp(-g)) * u).astype(np.float32))
        A2 = O.dequant_blocks(*O.quantize_blocks(h, a2[e])) / np.float64(a2[e])
        B2 = O.dequant_blocks(w2q[0][e], w2q[1][e]) / np.float64(w2q[2][e])
        Y = A2 @ B2.T
        mask = np.zeros(T)
        for t in range(T):
            for j in range(k):
                if ids[t, j] == e:
                    mask[t] += w[t, j]
        out += mask[:, None] * Y
    return O.bf16_round(out.astype(np.float32))


def test_sparse_moe_equals_dense_brute_force():
    wl, hidden, w13, w2, w13q, w2q, a1, a2 = small_layer()
    out = O.moe_forward(hidden, wl.logits, wl.top_k, w13q, w2q, a1, a2, 10.0, 10.0)
    ref = dense_brute_moe(hidden, wl.logits, wl.top_k, w13q, w2q, a1, a2, 10.0, 10.0)
    np.testing.assert_allclose(out, ref, rtol=1e-2, atol=1e-6)
    # identical up to the last bf16 rounding of sums formed in a different order
    assert np.mean(out != ref) < 0.01


def test_swiglu_clamps_the_gate_from_above_before_silu_and_up_on_both_sides():
    """SiLU written out with math.exp, bf16 rounding by torch.  Limits 2 (gate)
    and 10 (up) make each wrong reading visible: clamping after the SiLU,
    clamping the gate from below too, or leaving up unclamped."""
    import math
    import torch
    silu = lambda x: x / (1.0 + math.exp(-x))
    g = np.array([12.0, -20.0, 3.0, 0.5, 2.0])
    u = np.array([0.75, 1.0, -15.0, 12.0, -3.0])
    want = [silu(2.0) * 0.75,   # gate clamped to 2 first
            silu(-20.0) * 1.0,  # no lower clamp on the gate
            silu(2.0) * -10.0,  # gate 3 -> 2, up -15 -> -10
            silu(0.5) * 10.0,   # up 12 -> 10
            silu(2.0) * -3.0]   # at the limit: unchanged
    want = torch.tensor(want, dtype=torch.float32).to(torch.bfloat16).float().numpy()
    got = O.swiglu(g, u, 2.0, 10.0)
    np.testing.assert_array_equal(got, want)
    # the readings it rules out give other values
    assert got[0] != min(silu(12.0), 2.0) * 0.75
    assert abs(got[1]) < 1e-7 and abs(silu(-2.0)) > 0.2


def test_single_expert_top1_is_a_dense_swiglu_ffn():
    wl = W.moe_workload(20, 64, 32, 1, 1, 3)
    hidden = W.bf16_bits_to_f32(wl.hidden)
    w13q = O.quantize_expert_weights(W.bf16_bits_to_f32(wl.w13))
    w2q = O.quantize_expert_weights(W.bf16_bits_to_f32(wl.w2))
    a1 = np.float32([O.global_scale(np.abs(hidden).max())])
    a2 = np.float32([7.0])
    out = O.moe_forward(hidden, wl.logits, 1, w13q, w2q, a1, a2, 10.0, 10.0)
    # textbook FFN on the dequantized operands: y = W2 (silu(W1 x) * W3 x)
    xq = O.dequant_blocks(*O.quantize_blocks(hidden, a1[0])) / np.float64(a1[0])
    Wg = O.dequant_blocks(w13q[0][0][:32], w13q[1][0][:32]) / np.float64(w13q[2][0])
    Wu = O.dequant_blocks(w13q[0][0][32:], w13q[1][0][32:]) / np.float64(w13q[2][0])
    gate = np.minimum(xq @ Wg.T, 10.0)
    up = np.clip(xq @ Wu.T, -10.0, 10.0)
    h = O.bf16_round((gate * (1 / (1 + np.exp(-gate))) * up).astype(np.float32))
    hq = O.dequant_blocks(*O.quantize_blocks(h, a2[0])) / np.float64(a2[0])
    W2 = O.dequant_blocks(w2q[0][0], w2q[1][0]) / np.float64(w2q[2][0])
    ref = O.bf16_round((hq @ W2.T).astype(np.float32))
    # same arithmetic up to where 1/gs enters an FP64 product: agree to bf16 rounding
    np.testing.assert_allclose(out, ref, rtol=8e-3, atol=1e-6 * np.abs(ref).max())
    assert np.mean(out == ref) > 0.99


def test_quantized_moe_tracks_unquantized_moe():
    """Sanity against an unquantized FP64 MoE: cosine in the range the pages
    report for NVFP4 layers vs BF16 (about 0.99)."""
    wl, hidden, w13, w2, w13q, w2q, a1, a2 = small_layer(T=64, H=128, I=64, E=4, k=2, seed=12)
    out = O.moe_forward(hidden, wl.logits, 2, w13q, w2q, a1, a2)
    ids, w = O.route(wl.logits, 2)
    ref = np.zeros(out.shape)
    for t in range(wl.T):
        for j in range(2):
            e = ids[t, j]
            G = w13[e].astype(np.float64) @ hidden[t].astype(np.float64)
            g, u = np.minimum(G[:64], 10), np.clip(G[64:], -10, 10)
            ref[t] += w[t, j] * (w2[e].astype(np.float64) @ (g / (1 + np.exp(-g)) * u))
    cos = np.sum(out * ref) / np.linalg.norm(out) / np.linalg.norm(ref)
    assert 0.97 < cos < 0.9999


def test_moe_is_linear_in_w2_scale_and_zero_for_zero_input():
    wl, hidden, w13, w2, w13q, w2q, a1, a2 = small_layer(T=16, H=64, I=32, E=3, k=2, seed=13)
    zero = np.zeros_like(hidden)
    out0 = O.moe_forward(zero, wl.logits, 2, w13q, w2q, np.ones(3, np.float32), a2)
    assert np.all(out0 == 0)
    # halving the W2 global scale (same nibbles and block scales) doubles the output
    w2q_half = (w2q[0], w2q[1], (w2q[2] / 2).astype(np.float32))
    o1 = O.moe_forward(hidden, wl.logits, 2, w13q, w2q, a1, a2)
    o2 = O.moe_forward(hidden, wl.logits, 2, w13q, w2q_half, a1, a2)
    np.testing.assert_allclose(o2, 2 * o1, rtol=8e-3, atol=1e-30)


def test_tiny_workload_exercises_forced_blocks():
    wl = W.tiny_moe()
    hidden = W.bf16_bits_to_f32(wl.hidden)
    gs = O.global_scale(np.abs(hidden).max())
    _, s = O.quantize_blocks(hidden, gs)
    xs = (hidden * gs).reshape(-1, 16)
    b = np.abs(xs).max(1)
    zero_blocks = b == 0
    under = (b > 0) & (b < 6 * 2.0 ** -9)
    assert zero_blocks.sum() >= 40 and under.sum() >= 10
    assert np.all(s.reshape(-1)[zero_blocks | under] == 0)


# ----------------------------------------------------------------- expert parallelism (R18)

def test_remap_global_ids_hand_example():
    # 8 local experts starting at global id 16: [16, 24) are local
    ids = np.array([[16, 23], [15, 24], [40, 17]])
    w = np.array([[0.7, 0.3], [0.6, 0.4], [0.9, 0.1]])
    loc, lw = O.remap_global_ids(ids, w, 16, 8)
    assert loc.tolist() == [[0, 7], [-1, -1], [-1, 1]]
    assert lw.tolist() == [[0.7, 0.3], [0.0, 0.0], [0.0, 0.1]]  # kept, not renormalised


def test_sort_slots_skips_non_local_assignments():
    ids = np.array([[1, -1], [0, 1], [-1, -1], [1, 0]])
    w = np.arange(8, dtype=np.float64).reshape(4, 2) + 1
    m = O.sort_slots(ids, w, 2)
    assert m["counts"].tolist() == [2, 3]
    assert m["offsets"].tolist() == [0, 128, 256]
    # non-local assignments have no row; the rest keep ascending flat order per expert
    assert m["inverse"].tolist() == [128, -1, 0, 129, -1, -1, 130, 1]
    assert m["sorted_token_ids"][[0, 1, 128, 129, 130]].tolist() == [1, 3, 0, 1, 3]
    assert m["row_weight"][[0, 1, 128, 129, 130]].tolist() == [3.0, 8.0, 1.0, 4.0, 7.0]
    assert (m["sorted_token_ids"][2:128] == -1).all() and (m["row_weight"][2:128] == 0).all()


def test_routed_forward_all_local_equals_logit_forward():
    wl, hidden, w13, w2, w13q, w2q, a1, a2 = small_layer()
    ids, w = O.route(wl.logits, wl.top_k)
    gids, gw = O.remap_global_ids(ids + 100, w, 100, w13q[0].shape[0])
    a = O.moe_forward(hidden, wl.logits, wl.top_k, w13q, w2q, a1, a2, 10.0, 10.0)
    b = O.moe_forward_routed(hidden, gids, gw, w13q, w2q, a1, a2, 10.0, 10.0)
    np.testing.assert_array_equal(a, b)


def test_routed_forward_equals_per_assignment_brute_force():
    """Each local assignment's token through its expert alone (rows are
    independent in every step), weighted and summed; non-local assignments and
    tokens with none local contribute exactly zero."""
    wl, hidden, w13, w2, w13q, w2q, a1, a2 = small_layer(T=40, E=5, k=3)
    E = w13q[0].shape[0]
    rng = np.random.default_rng(7)
    T, k = hidden.shape[0], 3
    gids = rng.integers(0, 12, (T, k))  # 12 global experts, local ones are [4, 9)
    gids[5] = [0, 1, 11]               # a token with no local expert
    gw = rng.uniform(0.1, 1.0, (T, k))
    ids, w = O.remap_global_ids(gids, gw, 4, E)
    out, inter = O.moe_forward_routed(hidden, ids, w, w13q, w2q, a1, a2, 10.0, 10.0, return_intermediates=True)
    acc = np.zeros(hidden.shape)
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            if e < 0:
                continue
            h = O.expert_l1(hidden[t:t + 1], a1[e], w13q[0][e], w13q[1][e], w13q[2][e], 10.0, 10.0)
            acc[t] += w[t, j] * O.expert_l2(h, a2[e], w2q[0][e], w2q[1][e], w2q[2][e])[0]
    np.testing.assert_allclose(inter["acc"], acc, rtol=1e-12, atol=1e-12)
    assert not out[5].any()
    assert (ids == -1).any() and (ids >= 0).any()


def test_routed_calibration_all_local_equals_logit_calibration():
    wl, hidden, w13, w2, w13q, w2q, a1, a2 = small_layer()
    ids, _ = O.route(wl.logits, wl.top_k)
    r1, r2 = O.calibrate_activation_scales_routed(hidden, ids, w13q)
    np.testing.assert_array_equal(r1, a1)
    np.testing.assert_array_equal(r2, a2)


def test_routed_calibration_of_one_expert_parallel_rank_by_brute_force():
    """The page's setting: 48 local experts per rank, this rank holding global
    experts [240, 288) of 384.  After the remap every local expert's scales
    come from exactly the tokens that chose its global id; a rank that no
    token chose keeps scale 1 everywhere (never 0)."""
    E, start, G, k = 48, 240, 384, 6
    wl = W.moe_workload(300, 64, 32, E, k, 23)
    hidden = W.bf16_bits_to_f32(wl.hidden)
    w13q = O.quantize_expert_weights(W.bf16_bits_to_f32(wl.w13))
    rng = np.random.default_rng(5)
    gids = np.stack([rng.choice(G, size=k, replace=False) for _ in range(wl.T)])
    ids, _ = O.remap_global_ids(gids, np.ones(gids.shape), start, E)
    a1, a2 = O.calibrate_activation_scales_routed(hidden, ids, w13q)
    seen = 0
    for e in range(E):
        toks = [t for t in range(wl.T) if (gids[t] == start + e).any()]
        if not toks:
            assert a1[e] == 1 and a2[e] == 1
            continue
        seen += 1
        x = hidden[toks]
        assert a1[e] == np.float32(2688.0) / np.float32(np.abs(x).max())
        h = O.expert_l1(x, a1[e], w13q[0][e], w13q[1][e], w13q[2][e], 10.0, 10.0)
        assert a2[e] == np.float32(2688.0) / np.float32(np.abs(h).max())
    assert seen > 30
    # every token routed to global expert 0, held by another rank
    none, _ = O.remap_global_ids(np.zeros_like(gids), np.ones(gids.shape), start, E)
    b1, b2 = O.calibrate_activation_scales_routed(hidden, none, w13q)
    assert np.all(b1 == 1) and np.all(b2 == 1)


# ----------------------------------------------------------------- shared expert

def test_shared_expert_equals_one_expert_top1_moe():
    """With one expert and top_k = 1 every routing weight is exactly 1, so the
    routed layer and the shared-expert FFN compute the same thing."""
    wl, hidden, w13, w2, w13q, w2q, a1, a2 = small_layer(T=70, E=1, k=1)
    moe = O.moe_forward(hidden, wl.logits, 1, w13q, w2q, a1, a2, 10.0, 10.0)
    ffn = O.shared_expert_forward(hidden, w13q, w2q, a1[0], a2[0], 10.0, 10.0)
    np.testing.assert_array_equal(moe, ffn)


# ----------------------------------------------------------------- L2 scales from the batch (R19)

def test_batch_l2_scales_match_brute_force_per_expert_amax():
    """a2_gs None: each expert's L2 scale is 2688/amax of the bf16 SwiGLU
    output of exactly the tokens routed to it.  The scales are rebuilt here
    from the brute-force routing (no slots) and fed to the dense brute-force
    layer."""
    wl, hidden, w13, w2, w13q, w2q, a1, _ = small_layer(T=40, H=64, I=32, E=5, k=2, seed=21)
    E, I, k = 5, 32, 2
    ids, _ = brute_route(wl.logits, k)
    a2 = np.ones(E, np.float32)
    for e in range(E):
        rows = [t for t in range(wl.T) if e in ids[t]]
        if not rows:
            continue
        A = O.dequant_blocks(*O.quantize_blocks(hidden[rows], a1[e])) / np.float64(a1[e])
        B = O.dequant_blocks(w13q[0][e], w13q[1][e]) / np.float64(w13q[2][e])
        G = A @ B.T
        g = np.minimum(G[:, :I], 10.0)
        u = np.clip(G[:, I:], -10.0, 10.0)
        h = O.bf16_round((g / (1 + np.exp(-g)) * u).astype(np.float32))
        amax = np.float32(np.abs(h).max())
        if amax > 0:
            a2[e] = np.float32(2688.0) / amax
    out = O.moe_forward(hidden, wl.logits, k, w13q, w2q, a1, None, 10.0, 10.0)
    ref = dense_brute_moe(hidden, wl.logits, k, w13q, w2q, a1, a2, 10.0, 10.0)
    np.testing.assert_allclose(out, ref, rtol=1e-2, atol=1e-6)
    assert np.mean(out != ref) < 0.01


def test_batch_l2_scales_put_each_experts_amax_on_the_top_code():
    """With the scale taken from the expert's own amax, the largest |h| maps to
    2688 = 6 * 448: its block gets the largest finite E4M3 scale (448, code
    0x7E) and it gets the largest E2M1 magnitude (6, code 7)."""
    wl, hidden, w13, w2, w13q, w2q, a1, _ = small_layer(T=60, H=64, I=32, E=4, k=2, seed=22)
    _, inter = O.moe_forward(hidden, wl.logits, 2, w13q, w2q, a1, None, 10.0, 10.0,
                             return_intermediates=True)
    assert len(inter["experts"]) >= 3
    for e, d in inter["experts"].items():
        h = d["h"]
        nib, s = O.quantize_blocks(h, d["a2_gs"])
        r, c = np.unravel_index(np.argmax(np.abs(h)), h.shape)
        assert s[r, c // 16] == 0x7E
        assert (nib[r, c] & 7) == 7
        assert s.max() == 0x7E


def test_batch_l2_scales_equal_calibrated_scales_forward():
    """The calibration entry computes the same per-expert amax over the same
    rows, so a forward given the calibrated L2 scales is the same forward."""
    wl, hidden, w13, w2, w13q, w2q, a1, a2 = small_layer(T=50, H=64, I=32, E=5, k=2, seed=23)
    dyn = O.moe_forward(hidden, wl.logits, 2, w13q, w2q, a1, None, 10.0, 10.0)
    cal = O.moe_forward(hidden, wl.logits, 2, w13q, w2q, a1, a2, 10.0, 10.0)
    np.testing.assert_array_equal(dyn, cal)


# ----------------------------------------------------------------- slot layout cases from the pages

def _slot_cases():
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "slot_offsets.json")) as f:
        return json.load(f)["cases"]


def test_page_offsets_example_gets_whole_chunks_and_scale_rows():
    """Counts [500, 524] (the page's offsets [0, 500, 1024]): expert 0 gets four
    whole 128-row chunks, so all 500 of its scale rows sit where the GEMM reads
    them, and its 12 pad rows carry zero scales."""
    case = _slot_cases()[0]
    counts = case["counts"]
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int32)[:, None]
    m = O.sort_slots(ids, np.ones(ids.shape), len(counts))
    assert m["counts"].tolist() == counts
    assert m["offsets"].tolist() == case["padded_offsets"]
    rng = np.random.default_rng(3)
    lin = rng.integers(1, 127, (sum(counts), 8), dtype=np.uint8)
    swz = O.assemble_scales(lin, np.concatenate([[0], np.cumsum(counts)]), m["offsets"])
    full = O.unswizzle_scales(swz, m["P"], 8)
    np.testing.assert_array_equal(full[0:500], lin[0:500])
    assert not full[500:512].any()
    np.testing.assert_array_equal(full[512:1036], lin[500:1024])


def test_page_bug9_case_needs_more_than_one_chunk_per_expert():
    case = _slot_cases()[1]
    wl = W.moe_workload(case["T"], 64, 32, case["E"], case["top_k"], 0, zipf_s=1.1, with_weights=False)
    ids, w = O.route(wl.logits, case["top_k"])
    m = O.sort_slots(ids, w, case["E"])
    assert m["P"] > case["min_padded_rows_exclusive"]
    assert m["P"] <= O.slot_capacity(case["T"], case["top_k"], case["E"])
