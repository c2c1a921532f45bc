"""CPU oracle for the NVFP4 mixture-of-experts FFN forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this module: only the tests, the smoke check and the benchmark's
CPU-baseline leg do.  It shares no code, table or constant generator with the
CUDA path.

Sources.  The method is described by three commit-log pages of the
``nvfp4-megamoe-kernel`` project:
  [bridge]  ".../commit/50e9b5da.../cutedsl/bridge.py"  (quantizers)
  [vllm]    ".../commit/bde81b95.../vllm"               (MoE runner, slots)
  [cutedsl] ".../commit/dfd9c10a.../cutedsl"            (grouped linear)
The pages have no numbered sections; citations name the commit paragraph.

Precision.  The quantizer's decisions (scales, nibbles) are taken in FP32,
the precision the pages' quantizer computes in; every contraction,
activation and combine is FP64.  All FP32 steps are single IEEE operations
on numpy float32 arrays (correctly rounded, no fused multiply-add).

Readings where the pages leave a step open (each also listed in the design
notes):
  R1  E2M1 rounding is one round-to-nearest on the grid {0,.5,1,1.5,2,3,4,6},
      ties to the even code, saturating at 6 (the pages' half-step round plus
      an unlisted 13-entry table is read as this).
  R2  global scale gs = 2688 / amax (2688 = 448 * 6), multiplied into x;
      amax == 0 gives gs = 1.
  R3  the underflow test is on the globally scaled block amax b, strict b < 6*2^-9.
  R4  "divide" is an IEEE FP32 division (b/6 and x'/scale).
  R5  an element whose magnitude rounds to 0 gets nibble 0x0 (no -0).
  R6  low nibble of a byte = even K index.
  R7  block scales are stored in the 128x4 tile layout of the Blackwell
      block-scaled MMA (512-byte tiles, row r -> (r%32)*16 + ((r%128)/32)*4).
  R8  routing: top-k by logit (ties -> lower expert), weights = softmax over
      all experts renormalised over the k chosen = exp(l_j)/sum_sel exp(l_i).
  R9  slots: expert e's rows start at off[e], a multiple of 128; rows within
      an expert in ascending flat index t*k+j; empty experts get 0 rows;
      pad rows carry token -1 and weight 0.
  R10 SwiGLU: g = min(G,gate_limit), u = clamp(U,-up_limit,up_limit),
      h = bf16(g*sigmoid(g)*u) (rounded through FP32) before requantization.
  R11 combine: FP64 sum of w * Y over the token's k rows, rounded to bf16.
  R12 activation global scales are inputs (calibrated beforehand).
  R13 W13 rows 0..I-1 are gate, rows I..2I-1 are up.
  R14 weights are K-major [N][K/2] per expert.
  R18 expert parallelism: top-k ids from the model's router are global; the
      local expert of global id g is g - experts_start when that lies in
      [0, E), else the assignment is not local: it gets weight 0, occupies
      no slot row and contributes nothing; local assignments keep the
      router's weights (no renormalisation after the drop).
  R19 L2 scales from the batch: when no calibrated L2 activation scale is
      given, expert e's L2 global scale is 2688 / amax of its own bf16 L1
      output h in this forward (1 when that amax is 0); h is quantized with it
      exactly as with a given scale.
  R20 FP8 L1 output (the survey's FP8/BF16 L1-output option when no
      calibrated L2 scale exists; the pages name the option, not a format):
      the bf16 h is stored as OCP E4M3 values in blocks of 16 consecutive
      features of a row, each block with a power-of-two scale 2^k, k the least
      integer with max|h_block| <= 448 * 2^k (clamped to [-126, 126]; k = 0
      for an all-zero block): code = E4M3(h / 2^k), round to nearest even, a
      zero magnitude without sign.  h8 = dec(code) * 2^k replaces h from there
      on: the L2 scale is 2688 / amax(h8) of the expert's rows (R19) and h8 is
      quantized with it.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32

# E2M1 magnitudes by code 0..7 (sign is bit 3).  [bridge] "13-byte lookup table"
# paragraph maps values onto these codes; spec list of the FP4 grid.
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)

# 6 * 2^-9: the smallest block amax whose scale amax/6 is representable in E4M3.
# [bridge] "Bug #4 fix": blocks with amax < 6*2^-9 are forced to scale 0, nibble 0.
UNDERFLOW_AMAX = F32(6.0 * 2.0 ** -9)
E4M3_MAX = 448.0
GS_NUMERATOR = F32(2688.0)  # 448 * 6, [vllm] checkpoint input_scale paragraph


# --------------------------------------------------------------------------- formats

def e2m1_encode(q) -> np.ndarray:
    """Nibble of the E2M1 value nearest to q (R1, R5).

    Nearest grid value; on an exact midpoint the even code wins; |q| > 6
    saturates to 6; a magnitude that rounds to zero has no sign.
    The midpoints between consecutive grid values are
    0.25 .75 1.25 1.75 2.5 3.5 5; at each the even code is on the side the
    comparison ``<=`` / ``<`` below puts it.
    """
    q = np.asarray(q, dtype=np.float32)
    a = np.abs(q).astype(np.float64)
    idx = np.full(a.shape, 7, dtype=np.uint8)
    idx[a <= 5.0] = 6
    idx[a < 3.5] = 5
    idx[a <= 2.5] = 4
    idx[a < 1.75] = 3
    idx[a <= 1.25] = 2
    idx[a < 0.75] = 1
    idx[a <= 0.25] = 0
    neg = (np.signbit(q)) & (idx != 0)
    return (idx | (neg.astype(np.uint8) << 3)).astype(np.uint8)


def e2m1_decode(nib) -> np.ndarray:
    nib = np.asarray(nib, dtype=np.uint8)
    v = E2M1_GRID[nib & 7]
    return np.where(nib & 8, -v, v)


def e4m3_encode(v) -> np.ndarray:
    """OCP E4M3FN code of a non-negative value: round to nearest, ties to even,
    saturating at 448 (code 0x7E).  Bias 7, subnormal step 2^-9, no infinity."""
    v = np.asarray(v, dtype=np.float64)
    if np.any(v < 0) or np.any(~np.isfinite(v)):
        raise ValueError("e4m3_encode expects finite non-negative values")
    code = np.zeros(v.shape, dtype=np.int64)
    sub = v < 2.0 ** -6
    # subnormals (and zero): multiples of 2^-9; rint is round-half-even.
    code[sub] = np.rint(v[sub] * 2.0 ** 9).astype(np.int64)  # 8 -> 0x08 == 2^-6, still right
    nrm = ~sub
    f, ex = np.frexp(v[nrm])            # v = f * 2^ex, f in [0.5, 1)
    e = ex.astype(np.int64) - 1          # v = (2f) * 2^e, 2f in [1, 2)
    m = np.rint((2.0 * f - 1.0) * 8.0).astype(np.int64)
    carry = m == 8
    e[carry] += 1
    m[carry] = 0
    code[nrm] = ((e + 7) << 3) | m
    code = np.minimum(code, 0x7E)        # satfinite: never the NaN pattern 0x7F
    return code.astype(np.uint8)


def e4m3_decode(code) -> np.ndarray:
    """Value of an E4M3FN code (0x7F / 0xFF are NaN)."""
    c = np.asarray(code, dtype=np.int64)
    e = (c >> 3) & 0xF
    m = c & 7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return np.where(c & 0x80, -val, val)


def global_scale(amax) -> np.float32:
    """R2: encode-form global scale 2688 / amax in FP32; amax == 0 gives 1."""
    amax = F32(amax)
    if amax == 0:
        return F32(1.0)
    return F32(GS_NUMERATOR / amax)


# --------------------------------------------------------------------------- block quantization

def quantize_blocks(x, gs):
    """NVFP4 quantization of rows of x along the last axis, 16-element blocks.

    [bridge] "Bug #3 fix" / "Bug #4 fix" / "13-byte lookup table" paragraphs:
      x' = fl32(x * gs)                         (gs per row, FP32)
      b  = max |x'| over the block
      b < 6*2^-9  -> scale code 0 and all nibbles 0   (zero and underflow blocks)
      else s = E4M3(fl32(b / 6)),  q = fl32(x' / dec(s)),  nibble = E2M1(q)
    Returns (nibbles uint8 [..., K], scale codes uint8 [..., K/16]).
    """
    x = np.asarray(x, dtype=np.float32)
    K = x.shape[-1]
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    gs = np.asarray(gs, dtype=np.float32)
    if gs.ndim == 0:
        xs = x * gs
    else:
        xs = x * gs.reshape(gs.shape + (1,) * (x.ndim - gs.ndim))
    xs = xs.astype(np.float32)
    blk = xs.reshape(xs.shape[:-1] + (K // 16, 16))
    b = np.max(np.abs(blk), axis=-1)                      # FP32, exact
    forced = b < UNDERFLOW_AMAX
    s = e4m3_encode(np.where(forced, F32(0), b / F32(6.0)).astype(np.float32))
    s[forced] = 0
    d = e4m3_decode(s).astype(np.float32)
    d_safe = np.where(forced, F32(1.0), d).astype(np.float32)
    q = (blk / d_safe[..., None]).astype(np.float32)
    nib = e2m1_encode(q)
    nib[forced] = 0
    return nib.reshape(x.shape), s


def dequant_blocks(nib, s):
    """e2m1(nib) * dec(s) per element (exact in FP64); the 1/gs factor is not applied."""
    nib = np.asarray(nib, dtype=np.uint8)
    s = np.asarray(s, dtype=np.uint8)
    v = e2m1_decode(nib)
    K = nib.shape[-1]
    d = np.repeat(e4m3_decode(s), 16, axis=-1).reshape(nib.shape[:-1] + (K,))
    return v * d


def pack_nibbles(nib) -> np.ndarray:
    """R6: byte j = nib[2j] | nib[2j+1] << 4 ([bridge] packing paragraph: two values per byte, along K)."""
    nib = np.asarray(nib, dtype=np.uint8)
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


# --------------------------------------------------------------------------- scale layout

def sf_tile_offset(r, c, sf_cols_padded):
    """R7: byte offset of scale (row r, scale column c) in the 128x4 tile layout.

    Tiles of 128 rows x 4 scale columns take 512 bytes; tiles follow each other
    along the scale columns first, then along the row tiles.
    """
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    return (((r // 128) * (sf_cols_padded // 4) + c // 4) * 512
            + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4)


def padded_sf_cols(sf_cols):
    return (sf_cols + 3) // 4 * 4


def assemble_scales(sf_linear, offsets, padded_offsets):
    """[vllm] "Root cause of garbage output" / "Bug 9" / ".item() fallback" paragraphs:
    per-group linear scales (rows offsets[g]..offsets[g+1]) are placed at rows
    padded_offsets[g].. of a buffer whose groups start on 128-row boundaries,
    then laid out in the 128x4 tile layout.  Pad rows and pad columns are 0."""
    sf_linear = np.asarray(sf_linear, dtype=np.uint8)
    C = sf_linear.shape[1]
    Cp = padded_sf_cols(C)
    total = int(padded_offsets[-1])
    if total % 128:
        raise ValueError("padded rows must be a multiple of 128")
    out = np.zeros(total * Cp, dtype=np.uint8)
    for g in range(len(offsets) - 1):
        n = int(offsets[g + 1] - offsets[g])
        if n > int(padded_offsets[g + 1] - padded_offsets[g]):
            raise ValueError("group does not fit its padded slot")
        rows = np.arange(n, dtype=np.int64) + int(padded_offsets[g])
        rr, cc = np.meshgrid(rows, np.arange(C), indexing="ij")
        out[sf_tile_offset(rr, cc, Cp)] = sf_linear[int(offsets[g]):int(offsets[g]) + n]
    return out


def unswizzle_scales(sf_swz, rows, sf_cols):
    """Inverse of the tile layout: linear [rows, sf_cols] view of a swizzled buffer."""
    Cp = padded_sf_cols(sf_cols)
    rr, cc = np.meshgrid(np.arange(rows), np.arange(sf_cols), indexing="ij")
    return np.asarray(sf_swz, dtype=np.uint8)[sf_tile_offset(rr, cc, Cp)]


def quantize_tensor(x, gs, rows_padded=None):
    """Quantize rows of x [R, K] with one global scale, returning the packed bytes
    [Rp, K/2] (pad rows zero), the swizzled scales and the linear scales."""
    x = np.asarray(x, dtype=np.float32)
    R, K = x.shape
    Rp = rows_padded if rows_padded is not None else (R + 127) // 128 * 128
    nib, s = quantize_blocks(x, gs)
    packed = np.zeros((Rp, K // 2), dtype=np.uint8)
    packed[:R] = pack_nibbles(nib)
    swz = assemble_scales(s, np.array([0, R]), np.array([0, Rp]))
    return packed, swz, s


def weight_quantize(w, gs=None):
    """[bridge] "quantize_weight_to_nvfp4" paragraph: weights quantized along K
    (here K-major rows, R14).  gs defaults to 2688/amax of the whole tensor."""
    w = np.asarray(w, dtype=np.float32)
    if gs is None:
        gs = global_scale(np.max(np.abs(w)))
    nib, s = quantize_blocks(w, F32(gs))
    return nib, s, F32(gs)


# --------------------------------------------------------------------------- routing and slots

def route(logits, top_k):
    """R8: expert ids [T,k] in descending logit order (ties -> lower expert),
    weights [T,k] FP64 = softmax renormalised over the chosen experts."""
    logits = np.asarray(logits, dtype=np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")
    ids = order[:, :top_k].astype(np.int32)
    sel = np.take_along_axis(logits, ids.astype(np.int64), axis=1).astype(np.float64)
    z = np.exp(sel - sel[:, :1])
    w = z / z.sum(axis=1, keepdims=True)
    return ids, w


def sort_slots(ids, weights, num_experts, row_align=128):
    """R9: per-expert padded slots.  [vllm] "Root cause of garbage output" and
    "Bug 9" paragraphs (128-row slots, multi-chunk for >128 rows), and the
    cudagraph list (bincount + cumsum offsets, padding slots with zero weight).

    Returns dict with counts [E], offsets [E+1] (padded, multiples of 128),
    P, sorted_token_ids [P] (-1 = pad), row_weight [P] (0 = pad),
    inverse [T*k] (flat assignment -> row)."""
    ids = np.asarray(ids, dtype=np.int64)
    T, k = ids.shape
    flat = ids.reshape(-1)
    local = flat >= 0  # R18: non-local assignments (-1) get no row; inverse -1
    counts = np.bincount(flat[local], minlength=num_experts).astype(np.int64)
    padded = (counts + row_align - 1) // row_align * row_align
    offsets = np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)
    P = int(offsets[-1])
    sorted_ids = np.full(P, -1, dtype=np.int64)
    row_w = np.zeros(P, dtype=np.float64)
    inverse = np.full(T * k, -1, dtype=np.int64)
    order = np.argsort(flat, kind="stable")  # ascending expert, then ascending flat index
    order = order[local[order]]
    starts = np.concatenate([[0], np.cumsum(counts)])
    for e in range(num_experts):
        fs = order[starts[e]:starts[e + 1]]
        rows = offsets[e] + np.arange(len(fs))
        sorted_ids[rows] = fs // k
        row_w[rows] = np.asarray(weights, dtype=np.float64).reshape(-1)[fs]
        inverse[fs] = rows
    return dict(counts=counts, offsets=offsets, P=P, sorted_token_ids=sorted_ids,
                row_weight=row_w, inverse=inverse)


def slot_capacity(T, top_k, num_experts):
    """Upper bound on the padded row count: sum_e ceil(c_e/128)*128."""
    A = T * top_k
    return (A + 127 * min(num_experts, A) + 127) // 128 * 128


# --------------------------------------------------------------------------- GEMMs

def nvfp4_gemm(a_nib, a_s, a_gs, b_nib, b_s, b_gs):
    """D = alpha * dq(A) . dq(B)^T with dq = e2m1 * dec(scale), FP64 accumulation,
    alpha = 1 / (a_gs * b_gs).  A [M,K] nibbles, B [N,K] nibbles (R14)."""
    A = dequant_blocks(a_nib, a_s)
    B = dequant_blocks(b_nib, b_s)
    return (A @ B.T) / (np.float64(a_gs) * np.float64(b_gs))


def swiglu_exact(g, u, gate_limit, up_limit):
    """R10, [cutedsl] SwiGLU clamp fix (the gate is clamped before the SiLU):
    silu(min(g, gate_limit)) * clamp(u, -up_limit, up_limit) in FP64, before
    any rounding."""
    g = np.minimum(g, gate_limit)
    u = np.clip(u, -up_limit, up_limit)
    return g / (1.0 + np.exp(-g)) * u


def swiglu(g, u, gate_limit, up_limit):
    """R10: the SwiGLU value of swiglu_exact rounded to FP32 then to bf16 (the
    fused epilogue emits bf16 on the bridge page); returned as FP32 values."""
    return bf16_round(swiglu_exact(g, u, gate_limit, up_limit).astype(np.float32))


def bf16_round(x):
    """FP32 -> bf16 (nearest, ties to even), returned as FP32 values."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


def fp8_block_exponent(amax) -> np.ndarray:
    """R20: the least k with amax <= 448 * 2^k, clamped to [-126, 126]; 0 for
    amax == 0.  448 = 1.75 * 2^8, so with amax = m * 2^E (m in [1, 2)):
    k = E - 8, plus 1 when m > 1.75."""
    a = np.asarray(amax, dtype=np.float64)
    f, ex = np.frexp(a)                      # a = f * 2^ex, f in [0.5, 1)
    k = (ex.astype(np.int64) - 1) - 8 + (2.0 * f > 1.75)
    k = np.clip(k, -126, 126)
    return np.where(a > 0, k, 0).astype(np.int64)


def fp8_block_encode(h):
    """R20: h [n, I] (bf16 values, I % 16 == 0) -> E4M3 codes uint8 [n, I] and
    block exponents k int64 [n, I/16]."""
    h = np.asarray(h, dtype=np.float64)
    n, I = h.shape
    blk = h.reshape(n, I // 16, 16)
    k = fp8_block_exponent(np.max(np.abs(blk), axis=2))
    scaled = blk / np.exp2(k)[:, :, None]     # exact: a power of two
    mag = e4m3_encode(np.abs(scaled)).astype(np.uint8)
    sign = np.where((scaled < 0) & (mag != 0), 0x80, 0).astype(np.uint8)
    return (mag | sign).reshape(n, I), k


def fp8_block_decode(codes, k):
    """R20: dec(code) * 2^k as FP32 values [n, I]."""
    codes = np.asarray(codes)
    n, I = codes.shape
    v = e4m3_decode(codes).reshape(n, I // 16, 16) * np.exp2(np.asarray(k, dtype=np.float64))[:, :, None]
    return v.reshape(n, I).astype(np.float32)


# --------------------------------------------------------------------------- the MoE forward

def quantize_expert_weights(w, gs=None):
    """Per-expert weight quantization: w [E, N, K] -> nibbles [E,N,K], scales
    [E,N,K/16], gs [E] (default 2688/amax per expert, [vllm] per-expert l1_gs/l2_gs)."""
    w = np.asarray(w, dtype=np.float32)
    E = w.shape[0]
    nibs = np.empty(w.shape, dtype=np.uint8)
    scs = np.empty(w.shape[:-1] + (w.shape[-1] // 16,), dtype=np.uint8)
    gss = np.empty(E, dtype=np.float32)
    for e in range(E):
        g = global_scale(np.max(np.abs(w[e]))) if gs is None else F32(gs[e])
        nibs[e], scs[e] = quantize_blocks(w[e], g)
        gss[e] = g
    return nibs, scs, gss


def expert_l1(x, a1_gs, w13_nib, w13_s, w13_gs, gate_limit, up_limit):
    """One expert's L1 + SwiGLU on rows x [n, H] (FP32 values): returns h [n, I]
    (bf16 values as FP32)."""
    I = w13_nib.shape[0] // 2
    a_nib, a_s = quantize_blocks(x, a1_gs)
    G1 = nvfp4_gemm(a_nib, a_s, a1_gs, w13_nib, w13_s, w13_gs)
    return swiglu(G1[:, :I], G1[:, I:], gate_limit, up_limit)


def expert_l2(h, a2_gs, w2_nib, w2_s, w2_gs):
    a_nib, a_s = quantize_blocks(h, a2_gs)
    return nvfp4_gemm(a_nib, a_s, a2_gs, w2_nib, w2_s, w2_gs)


def remap_global_ids(topk_ids, topk_weights, experts_start, num_experts):
    """R18, [vllm] "Root cause of CUDA_ERROR_ASSERT index out of bounds"
    paragraph (fixes 1-2: experts_start_idx; remap global -> local ids and
    zero the weights of non-local experts): local id g - start where it lies
    in [0, E), else -1 with weight 0."""
    g = np.asarray(topk_ids, dtype=np.int64)
    loc = g - int(experts_start)
    is_local = (loc >= 0) & (loc < num_experts)
    ids = np.where(is_local, loc, -1).astype(np.int32)
    w = np.where(is_local, np.asarray(topk_weights, dtype=np.float64), 0.0)
    return ids, w


def moe_forward(hidden, logits, top_k, w13q, w2q, a1_gs, a2_gs,
                gate_limit=10.0, up_limit=10.0, return_intermediates=False, l1_fp8=False):
    """The sparse MoE forward: route -> slots -> per expert (quantize, L1,
    SwiGLU, requantize, L2) -> routing-weighted combine.  hidden [T,H] FP32
    values (bf16-exact); w13q/w2q = (nibbles, scales, gs) per expert.
    Returns bf16 values as FP32 [T, H]."""
    ids, w = route(logits, top_k)
    return moe_forward_routed(hidden, ids, w, w13q, w2q, a1_gs, a2_gs, gate_limit, up_limit,
                              return_intermediates, l1_fp8)


def moe_forward_routed(hidden, ids, w, w13q, w2q, a1_gs, a2_gs,
                       gate_limit=10.0, up_limit=10.0, return_intermediates=False, l1_fp8=False):
    """The MoE forward from given routing: local expert ids [T,k] (-1 = not
    local, R18) and weights [T,k]; otherwise as moe_forward.
    a2_gs None (R19): each expert's L2 global scale is 2688/amax of its own
    bf16 L1 output in this batch ([vllm] warm-up paragraph: the L2 scale is
    measured on the L1 GEMM's output; [cutedsl] BF16 L1 output when no
    calibrated L2 scale exists).  l1_fp8 (with a2_gs None, R20): h is first
    stored as FP8 blocks and the L2 input is taken from those values."""
    if l1_fp8 and a2_gs is not None:
        raise ValueError("the FP8 L1 output applies when the L2 scales come from the batch")
    hidden = np.asarray(hidden, dtype=np.float32)
    T, H = hidden.shape
    E = w13q[0].shape[0]
    ids = np.asarray(ids)
    meta = sort_slots(ids, w, E)
    acc = np.zeros((T, H), dtype=np.float64)
    inter = {}
    for e in range(E):
        lo = int(meta["offsets"][e])
        n = int(meta["counts"][e])
        if n == 0:
            continue
        toks = meta["sorted_token_ids"][lo:lo + n]
        h = expert_l1(hidden[toks], a1_gs[e], w13q[0][e], w13q[1][e], w13q[2][e],
                      gate_limit, up_limit)
        if l1_fp8:
            h = fp8_block_decode(*fp8_block_encode(h))
        a2e = global_scale(np.max(np.abs(h))) if a2_gs is None else a2_gs[e]
        Y = expert_l2(h, a2e, w2q[0][e], w2q[1][e], w2q[2][e])
        np.add.at(acc, toks, meta["row_weight"][lo:lo + n, None] * Y)
        if return_intermediates:
            inter[e] = dict(h=h, Y=Y, toks=toks, a2_gs=a2e)
    out = bf16_round(acc.astype(np.float32))
    if return_intermediates:
        return out, dict(ids=ids, w=w, meta=meta, experts=inter, acc=acc)
    return out


def shared_expert_forward(hidden, w13q, w2q, a1_gs, a2_gs, gate_limit=10.0, up_limit=10.0):
    """The shared expert: one NVFP4 SwiGLU FFN over every token, no routing
    ([cutedsl] shared-expert runner paragraph: a single group, no scatter
    and no routing; the fused L1+SiLU+L2 paragraph).  w13q / w2q hold one
    expert: (nibbles [1,2I,H], scales, gs [1]); a1_gs / a2_gs scalars.
    Returns bf16 values as FP32 [T, H]."""
    hidden = np.asarray(hidden, dtype=np.float32)
    h = expert_l1(hidden, a1_gs, w13q[0][0], w13q[1][0], w13q[2][0], gate_limit, up_limit)
    Y = expert_l2(h, a2_gs, w2q[0][0], w2q[1][0], w2q[2][0])
    return bf16_round(Y.astype(np.float32))


def calibrate_activation_scales(hidden, logits, top_k, w13q, gate_limit=10.0, up_limit=10.0,
                                row_limit=None):
    """[vllm] "compute_activation_global_scales" paragraphs: per local expert,
    L1 gs = 2688/amax of the rows routed to it, L2 gs = 2688/amax of that
    expert's L1 output (SwiGLU, bf16).  Experts with no rows get gs 1.
    row_limit: calibrate L2 on at most this many rows per expert (the first
    ones in slot order); None uses all rows."""
    ids, _ = route(logits, top_k)
    return calibrate_activation_scales_routed(hidden, ids, w13q, gate_limit, up_limit, row_limit)


def calibrate_activation_scales_routed(hidden, ids, w13q, gate_limit=10.0, up_limit=10.0, row_limit=None):
    """The same calibration from given routing: local expert ids [T,k], -1 for
    an assignment to an expert this layer does not hold ([vllm] "Root cause of
    CUDA_ERROR_ASSERT index out of bounds" paragraph:
    compute_activation_global_scales expects local ids; with global ids no row
    matched a local expert).  Only the ids matter, not the weights."""
    hidden = np.asarray(hidden, dtype=np.float32)
    E = w13q[0].shape[0]
    ids = np.asarray(ids)
    meta = sort_slots(ids, np.ones(ids.shape), E)
    a1 = np.ones(E, dtype=np.float32)
    a2 = np.ones(E, dtype=np.float32)
    for e in range(E):
        lo = int(meta["offsets"][e])
        n = int(meta["counts"][e])
        if n == 0:
            continue
        x = hidden[meta["sorted_token_ids"][lo:lo + n]]
        a1[e] = global_scale(np.max(np.abs(x)))
        if row_limit is not None:
            x = x[:row_limit]
        h = expert_l1(x, a1[e], w13q[0][e], w13q[1][e], w13q[2][e], gate_limit, up_limit)
        a2[e] = global_scale(np.max(np.abs(h)))
    return a1, a2


def grouped_gemm(a_nib, a_s, a_gs, b_nib, b_s, b_gs, group_rows):
    """[cutedsl] grouped-GEMM offsets paragraph: group g's rows of A (given as
    group_rows[g] consecutive rows) times group g's weight; FP64 results per group."""
    out = []
    r0 = 0
    for g, n in enumerate(group_rows):
        out.append(nvfp4_gemm(a_nib[r0:r0 + n], a_s[r0:r0 + n], a_gs[g],
                              b_nib[g], b_s[g], b_gs[g]))
        r0 += n
    return out
