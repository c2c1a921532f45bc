// NVFP4 quantization kernels: per-group amax -> global scale, strided
// quantization with scales written straight into the 128x4 tile layout,
// scale assembly into 128-row padded slots, and the MoE gather+quantize.
//
// All kernels are streaming kernels.  The quantizers give one lane one
// 16-element block, so each warp load and store is contiguous, and write 4
// scale codes per aligned 32-bit word of the tile layout (see
// gather_quantize_kernel and quantize_kernel).
#include <cuda_runtime.h>

#include "internal.h"
#include "nvfp4_format.cuh"
#include "ptx.cuh"

namespace nvfp4 {

namespace {

__device__ __forceinline__ uint4 ldg_nc(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// ---------------------------------------------------------------- amax
// Partial max |x| of group blockIdx.y over the blocks of the x grid: the
// group's rows are read as one sequence of 16-byte vectors (row r, vector c
// at index r*K/8 + c), strided over the whole grid, kAmaxUnroll independent
// loads in flight per thread.  Thread i's vector pointer advances by the
// grid stride with additions (no division in the loop), and the maxima of
// the two bf16 halves of a word are kept packed (one vmax per word).
constexpr int kAmaxThreads = 256;
constexpr int kAmaxUnroll = 8;   // 128 bytes in flight per thread
constexpr int kAmaxBlocksPerSm = 4;

__global__ void __launch_bounds__(kAmaxThreads, kAmaxBlocksPerSm)
    group_amax_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t K, int64_t ld_x, int64_t gstride_x,
                      float* __restrict__ partial, int partial_stride) {
  pdl_trigger();
  pdl_wait();
  const int g = blockIdx.y;
  const int64_t vpr = K / 8;
  const int64_t total = rows * vpr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t sr = stride / vpr, sc = stride - sr * vpr;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t r0 = i / vpr;
  int64_t c = i - r0 * vpr;
  // the thread's next vector, advanced by the grid stride with pointer adds
  const uint16_t* ptr = x + (int64_t)g * gstride_x + r0 * ld_x + c * 8;
  const int64_t step_elems = sr * ld_x + sc * 8, wrap_elems = ld_x - vpr * 8;
  uint32_t m = 0;  // max of |bf16| bit patterns per half (monotone for non-negative floats)
  for (; i < total; i += kAmaxUnroll * stride) {
    uint4 v[kAmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) {
      v[u] = i + u * stride < total ? ldg_nc(ptr) : make_uint4(0u, 0u, 0u, 0u);
      ptr += step_elems;
      c += sc;
      if (c >= vpr) {
        c -= vpr;
        ptr += wrap_elems;
      }
    }
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) {
      m = __vmaxu2(m, v[u].x & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].y & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].z & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].w & 0x7FFF7FFFu);
    }
  }
  m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0u;
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) partial[(int64_t)g * partial_stride + blockIdx.x] = __uint_as_float(m << 16);
  }
}

// gs = 2688 / amax (IEEE division), 1 when the group is all zero.
__device__ __forceinline__ float gs_from_group_amax(float a) { return a > 0.f ? __fdiv_rn(kGsNumerator, a) : 1.0f; }

// quantize_kernel: up to this many groups' global scales are reduced per
// block into shared memory.
constexpr int kSharedGsGroups = 1024;

// The global scale of group g from its nb partial maxima, reduced by one warp
// (max is exact and order-free, so every warp gets the same bits).
__device__ __forceinline__ float warp_group_gs(const float* __restrict__ partial, int partial_stride, int nb,
                                               int64_t g, int lane) {
  float a = 0.f;
  for (int i = lane; i < nb; i += 32) a = fmaxf(a, partial[g * partial_stride + i]);
#pragma unroll
  for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  return gs_from_group_amax(a);
}

__global__ void group_gs_kernel(const float* __restrict__ partial, int partial_stride, int nb, int groups,
                                float* __restrict__ gs) {
  pdl_trigger();
  pdl_wait();
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  float a = 0.f;
  for (int i = 0; i < nb; ++i) a = fmaxf(a, partial[(int64_t)g * partial_stride + i]);
  gs[g] = gs_from_group_amax(a);
}

// ---------------------------------------------------------------- scale assembly
__global__ void assemble_scales_kernel(const uint8_t* __restrict__ lin, int64_t sf_cols,
                                       const int32_t* __restrict__ offsets,
                                       const int32_t* __restrict__ padded_offsets, int groups,
                                       int64_t rows_capacity, uint8_t* __restrict__ out) {
  extern __shared__ int32_t s_off[];  // [groups+1] padded, then [groups+1] real
  for (int i = threadIdx.x; i <= groups; i += blockDim.x) {
    s_off[i] = padded_offsets[i];
    s_off[groups + 1 + i] = offsets[i];
  }
  __syncthreads();
  const int64_t cols4 = (sf_cols + 3) / 4 * 4;
  const int64_t words = rows_capacity * (cols4 / 4);
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < words;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = it / (cols4 / 4), c4 = (it - r * (cols4 / 4)) * 4;
    uint32_t v = 0;
    if (r < s_off[groups]) {
      int lo = 0, hi = groups;  // largest g with padded_offsets[g] <= r
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= r) lo = mid; else hi = mid;
      }
      const int64_t local = r - s_off[lo];
      const int64_t n = (int64_t)s_off[groups + 1 + lo + 1] - s_off[groups + 1 + lo];
      if (local < n) {
        const uint8_t* src = lin + ((int64_t)s_off[groups + 1 + lo] + local) * sf_cols;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (c4 + j < sf_cols) v |= (uint32_t)src[c4 + j] << (8 * j);
      }
    }
    *reinterpret_cast<uint32_t*>(out + sf_offset(r, c4, cols4)) = v;
  }
}

// ---------------------------------------------------------------- MoE gather + quantize
// Token-major gather + quantize of the L1 activations.  One warp owns one
// (token, segment of up to kGatherChunks x 512 elements) item: lane l owns
// the 16-element block at element 512*c + 16*l of each 512-element chunk c,
// loads it once with one 32-byte access (the warp reads 1 KB contiguous),
// and takes the block's max |x| from the bf16 bit patterns (x*gs rounds
// monotonically in |x|, so max|x*gs| = fl(max|x| * gs)).  It then quantizes
// the block for each of the token's top_k slot rows with that expert's
// global scale: 8 bytes of nibbles per lane (256 contiguous bytes per warp)
// and one 32-bit word of 4 block scales per group of 4 lanes.  The hidden row
// is read from memory once instead of once per slot.  The trailing warps
// give the pad rows of every expert's slot range zero block scales, which
// makes every value in them exactly 0 whatever their nibble bytes hold
// (E2M1 codes are all finite); the nibble bytes are not written.
// Large batches take 2 chunks (1,024 elements) per warp; batches of at most
// kSmallRouteTokens tokens take 1, for twice the warps on few tokens.
constexpr int kGatherChunks = 2;

// One 16-element bf16 block (32 bytes): a single 32-byte load where the
// address is 32-byte aligned, else two 16-byte loads (the entry points only
// promise 16-byte alignment of the hidden states).
template <bool kAligned32>
__device__ __forceinline__ void ld_block32(const uint16_t* p, uint32_t (&w)[8]) {
  if constexpr (kAligned32) {
    asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
        : "l"(p));
  } else {
    const uint4 a = ldg_nc(p), b = ldg_nc(p + 8);
    w[0] = a.x, w[1] = a.y, w[2] = a.z, w[3] = a.w, w[4] = b.x, w[5] = b.y, w[6] = b.z, w[7] = b.w;
  }
}

// max |x| over the 16 bf16 values of a block, as an FP32 value.
__device__ __forceinline__ float block_amax_bf16(const uint32_t (&w)[8]) {
  uint32_t m = 0u;
#pragma unroll
  for (int q = 0; q < 8; ++q) m = __vmaxu2(m, w[q] & 0x7FFF7FFFu);
  return __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
}

// Quantize one block of 16 bf16 values (raw bits) with global scale gs; the
// same arithmetic as quant_block16_pairs, with the scale pair from a table: tab[s] holds
// (dec(s), RN(1/dec(s))) for every scale code s.
__device__ __forceinline__ uint32_t quant_block16_bf16(const uint32_t (&w)[8], float amax, float gs, float rcp6,
                                                       const float2* tab, uint32_t& lo, uint32_t& hi) {
  lo = hi = 0u;
  const float b = __fmul_rn(amax, gs);
  if (!(b >= kUnderflowAmax)) return 0u;
  // b / 6 with the same exact correction as the element quotients (6 is an E4M3 value)
  const uint32_t s = e4m3_code(div_by_scale(fminf(b, 3.40282347e38f), 6.0f, rcp6));
  const float2 dy = tab[s];
  const uint64_t gs2 = f2_pack(gs, gs), y2 = f2_pack(dy.y, dy.y), nd2 = f2_pack(-dy.x, -dy.x);
  float q[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint64_t xs = f2_mul(f2_pack(bf16_lo(w[j]), bf16_hi(w[j])), gs2);
    const uint64_t q0 = f2_mul(xs, y2);
    const uint64_t r = f2_fma(q0, nd2, xs);
    f2_unpack(f2_fma(r, y2, q0), q[2 * j], q[2 * j + 1]);
  }
  lo = drop_negative_zero(e2m1x8_word(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]));
  hi = drop_negative_zero(e2m1x8_word(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]));
  return s;
}

template <bool kAligned32, int kChunks>
__global__ void __launch_bounds__(256, 4) gather_quantize_kernel(const uint16_t* __restrict__ hidden, int64_t H,
                                                              int64_t T, int top_k,
                                                              const int32_t* __restrict__ topk_ids,
                                                              const int32_t* __restrict__ inverse,
                                                              const int32_t* __restrict__ counts,
                                                              const int32_t* __restrict__ offsets, int E,
                                                              const float* __restrict__ a1_gs, int64_t capacity,
                                                              uint8_t* __restrict__ a1, uint8_t* __restrict__ sfa1,
                                                              int* __restrict__ tile_done) {
  pdl_trigger();
  __shared__ float2 tab[128];
  if (threadIdx.x < 128) {
    const float d = e4m3_value(threadIdx.x);
    tab[threadIdx.x] = make_float2(d, threadIdx.x ? __frcp_rn(d) : 0.f);
  }
  __syncthreads();
  pdl_wait();
  if (tile_done && blockIdx.x == 0)  // the L1 -> L2 per-m-tile counters of this forward start at 0
    for (int64_t i = threadIdx.x; i < capacity / 128; i += blockDim.x) tile_done[i] = 0;
  const float rcp6 = __frcp_rn(6.0f);
  const int lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t seg_elems = 512 * kChunks;
  const int64_t segs = (H + seg_elems - 1) / seg_elems;
  const int64_t sf_cols = H / 16;
  if (item < T * segs) {
    const int64_t t = item < (1ll << 31) ? (int64_t)((uint32_t)item / (uint32_t)segs) : item / segs;
    const int64_t e0 = (item - t * segs) * seg_elems;
    uint32_t raw[kChunks][8];
    float amax[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const int64_t el = e0 + c * 512 + lane * 16;
      if (el < H) {
        ld_block32<kAligned32>(hidden + t * H + el, raw[c]);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) raw[c][q] = 0u;
      }
    }
#pragma unroll
    for (int c = 0; c < kChunks; ++c) amax[c] = block_amax_bf16(raw[c]);
    int my_row = 0;
    float my_gs = 1.f;
    if (lane < top_k) {
      my_row = inverse[t * top_k + lane];  // -1: not a local expert (no row)
      const int e = topk_ids[t * top_k + lane];
      my_gs = e >= 0 ? a1_gs[e] : 1.f;
    }
    // the column part of each lane's scale byte offset in the tile layout (the
    // row part is added per slot row): each lane stores its own scale byte
    int64_t sf_col_off[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) sf_col_off[c] = sf_offset(0, (e0 + c * 512 + lane * 16) / 16, sf_cols);
#pragma unroll 2  // two slots' blocks in flight per lane (independent dependency chains)
    for (int j = 0; j < top_k; ++j) {
      const int64_t r = __shfl_sync(0xffffffffu, my_row, j);
      const float gs = __shfl_sync(0xffffffffu, my_gs, j);
      const bool row_ok = r >= 0 && r < capacity;
      const int64_t sf_row_off = sf_offset(r, 0, sf_cols);
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const int64_t el = e0 + c * 512 + lane * 16;
        uint32_t lo, hi;
        const uint32_t sc = quant_block16_bf16(raw[c], amax[c], gs, rcp6, tab, lo, hi);
        if (row_ok && el < H) {
          *reinterpret_cast<uint2*>(a1 + r * (H / 2) + el / 2) = make_uint2(lo, hi);
          sfa1[sf_row_off + sf_col_off[c]] = (uint8_t)sc;
        }
      }
    }
    return;
  }
  // pad rows: item -> (expert, j-th row past the expert's last token)
  const int64_t p = item - T * segs;
  if (p >= (int64_t)E * 128) return;
  const int e = (int)(p >> 7), j = (int)(p & 127);
  const int64_t r = (int64_t)offsets[e] + counts[e] + j;
  if (r >= offsets[e + 1] || r >= capacity) return;
  for (int64_t m = lane; m < sf_cols / 4; m += 32)
    *reinterpret_cast<uint32_t*>(sfa1 + sf_offset(r, 4 * m, sf_cols)) = 0u;
}

// ---------------------------------------------------------------- quantize
// Strided groups of rows -> NVFP4 (rows [rows, rows_padded) of every group are
// zero blocks).  Same layout as the MoE gather: one warp per (group, row,
// 1024-element segment), lane l owns the 16-element block at 512*c + 16*l of
// the segment's two chunks, one 32-byte load per block, 8 bytes of nibbles
// per lane and a 32-bit scale word per 4 lanes.  K is a multiple of 64, so the
// 4 lanes of a scale word are all inside or all outside the row.
// The global scale of group g is gs[g], or, with amax_partial given, reduced
// by the warp from the amax kernel's nb partial maxima (once per group a warp
// meets; the warp on a group's first item stores it to gs_copy).
template <bool kAligned32>
__global__ void __launch_bounds__(256) quantize_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                                                       int64_t ld_x, int64_t gstride_x, int groups,
                                                       const float* __restrict__ gs, float* __restrict__ gs_copy,
                                                       const float* __restrict__ amax_partial, int partial_stride,
                                                       int nb, uint8_t* __restrict__ fp4, uint8_t* __restrict__ sf,
                                                       int64_t rows_padded, int* __restrict__ status_reset) {
  pdl_trigger();
  __shared__ float2 tab[128];
  __shared__ float s_gs[kSharedGsGroups];
  __shared__ float s_red[8];
  if (threadIdx.x < 128) {
    const float d = e4m3_value(threadIdx.x);
    tab[threadIdx.x] = make_float2(d, threadIdx.x ? __frcp_rn(d) : 0.f);
  }
  __syncthreads();
  pdl_wait();  // the global scales may come from the amax kernels just before
  if (!amax_partial && gs_copy && blockIdx.x == 0)
    for (int i = threadIdx.x; i < groups; i += blockDim.x) gs_copy[i] = gs[i];
  if (status_reset && blockIdx.x == 0 && threadIdx.x == 0) *status_reset = 0;
  const float rcp6 = __frcp_rn(6.0f);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Global scales from the amax kernel's partial maxima: with few groups the
  // block reduces each group's partials once into shared memory (max is
  // exact and order-free: every block gets the same bits), instead of every
  // warp reducing its group's partials.
  const bool shared_gs = amax_partial && groups <= kSharedGsGroups;
  if (shared_gs) {
    if (groups == 1) {
      float a = 0.f;
      for (int i = threadIdx.x; i < nb; i += blockDim.x) a = fmaxf(a, amax_partial[i]);
#pragma unroll
      for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      if (lane == 0) s_red[warp] = a;
      __syncthreads();
      if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) a = fmaxf(a, s_red[w]);
        s_gs[0] = gs_from_group_amax(a);
      }
    } else {
      for (int gg = warp; gg < groups; gg += blockDim.x >> 5) {
        const float v = warp_group_gs(amax_partial, partial_stride, nb, gg, lane);
        if (lane == 0) s_gs[gg] = v;
      }
    }
    __syncthreads();
  }
  const int64_t segs = (K + 1023) / 1024;
  const int64_t per_group = rows_padded * segs;
  const int64_t items = per_group * groups;
  const int64_t sf_cols = K / 16;
  int64_t have_g = -1;
  float gsv = 0.f;
  // item = (g * rows_padded + r) * segs + sg, stepped by the grid's warp
  // count with additions and at most one carry per level (no division in the
  // loop; the start and the step are split with 32-bit divisions when the
  // item count allows)
  const int64_t first = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;
  const int64_t step = (int64_t)gridDim.x * (blockDim.x >> 5);
  int64_t g, r, sg, dg, dr, ds;
  if (items + step < (1ll << 31)) {
    const uint32_t pg = (uint32_t)per_group, ns = (uint32_t)segs;
    const uint32_t f = (uint32_t)first, st = (uint32_t)step;
    const uint32_t g32 = f / pg, f_in = f - g32 * pg, r32 = f_in / ns;
    const uint32_t dg32 = st / pg, st_in = st - dg32 * pg, dr32 = st_in / ns;
    g = g32, r = r32, sg = f_in - r32 * ns;
    dg = dg32, dr = dr32, ds = st_in - dr32 * ns;
  } else {
    g = first / per_group, r = (first - g * per_group) / segs;
    sg = first - g * per_group - r * segs;
    dg = step / per_group, dr = (step - dg * per_group) / segs;
    ds = step - dg * per_group - dr * segs;
  }
  for (int64_t item = first; item < items; item += step) {
    const int64_t rem = r * segs + sg, e0 = sg * 1024;
    const int64_t orow = g * rows_padded + r;
    uint32_t raw[2][8];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int64_t el = e0 + c * 512 + lane * 16;
      if (r < rows && el < K) ld_block32<kAligned32>(x + g * gstride_x + r * ld_x + el, raw[c]);
    }
    if (g != have_g) {
      gsv = shared_gs ? s_gs[g] : amax_partial ? warp_group_gs(amax_partial, partial_stride, nb, g, lane) : gs[g];
      have_g = g;
    }
    if (amax_partial && gs_copy && rem == 0 && lane == 0) gs_copy[g] = gsv;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int64_t el = e0 + c * 512 + lane * 16;
      uint32_t lo = 0u, hi = 0u, sc = 0u;
      if (r < rows && el < K) sc = quant_block16_bf16(raw[c], block_amax_bf16(raw[c]), gsv, rcp6, tab, lo, hi);
      const uint32_t word = sc | (__shfl_down_sync(0xffffffffu, sc, 1) << 8) |
                            (__shfl_down_sync(0xffffffffu, sc, 2) << 16) |
                            (__shfl_down_sync(0xffffffffu, sc, 3) << 24);
      if (el < K) {
        *reinterpret_cast<uint2*>(fp4 + orow * (K / 2) + el / 2) = make_uint2(lo, hi);
        if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(sf + sf_offset(orow, el / 16, sf_cols)) = word;
      }
    }
    sg += ds;
    if (sg >= segs) {
      sg -= segs;
      ++r;
    }
    r += dr;
    if (r >= rows_padded) {
      r -= rows_padded;
      ++g;
    }
    g += dg;
  }
}

// One warp per slot row: max |x| of the token's hidden row, folded into its
// expert's amax with an order-independent atomicMax on the float bits.
__global__ void __launch_bounds__(256) gather_amax_kernel(const uint16_t* __restrict__ hidden, int64_t H,
                                                          const int32_t* __restrict__ sorted_ids,
                                                          const int32_t* __restrict__ tile_expert,
                                                          const int32_t* __restrict__ meta, int64_t capacity,
                                                          uint32_t* __restrict__ amax_bits) {
  const int lane = threadIdx.x & 31;
  const int64_t P = min((int64_t)meta[0], capacity);
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < P; r += warps) {
    const int t = sorted_ids[r];
    if (t < 0) continue;
    uint32_t m = 0;
    for (int64_t c = lane; c < H / 8; c += 32) {
      const uint4 v = ldg_nc(hidden + (int64_t)t * H + c * 8);
      const uint32_t u[4] = {v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu, v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu};
#pragma unroll
      for (int q = 0; q < 4; ++q) m = max(m, max(u[q] & 0xFFFFu, u[q] >> 16));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0 && m) atomicMax(&amax_bits[tile_expert[r >> 7]], m << 16);
  }
}

// gs = 2688 / amax (IEEE division) from amax float bits; 1 for amax 0.
__device__ __forceinline__ float gs_of_amax_bits(uint32_t bits) {
  const float a = __uint_as_float(bits);
  return a > 0.f ? __fdiv_rn(kGsNumerator, a) : 1.0f;
}

__global__ void gs_from_amax_kernel(const uint32_t* __restrict__ amax_bits, int n, float* __restrict__ gs) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  gs[i] = gs_of_amax_bits(amax_bits[i]);
}

// L2 activations with global scales taken from the batch: slot rows [0, P) of
// the bf16 SwiGLU output h [capacity, K] (row-major, 32-byte aligned rows) ->
// NVFP4 nibbles and tile-layout scales, each row with its expert's
// gs = 2688 / amax(h of that expert).  Block 0 also stores the E global scales
// (the L2 GEMM's alpha needs them).  Warp layout as quantize_kernel.
__global__ void __launch_bounds__(256) slot_quantize_kernel(const uint16_t* __restrict__ h, int64_t K,
                                                            const int32_t* __restrict__ meta,
                                                            const int32_t* __restrict__ tile_expert,
                                                            int64_t capacity, const uint32_t* __restrict__ amax_bits,
                                                            int E, float* __restrict__ gs_out,
                                                            uint8_t* __restrict__ fp4, uint8_t* __restrict__ sf) {
  pdl_trigger();
  __shared__ float2 tab[128];
  if (threadIdx.x < 128) {
    const float d = e4m3_value(threadIdx.x);
    tab[threadIdx.x] = make_float2(d, threadIdx.x ? __frcp_rn(d) : 0.f);
  }
  __syncthreads();
  pdl_wait();  // h, the amax words and the slot table come from the kernels before
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < E; i += blockDim.x) gs_out[i] = gs_of_amax_bits(amax_bits[i]);
  const float rcp6 = __frcp_rn(6.0f);
  const int lane = threadIdx.x & 31;
  const int64_t P = min((int64_t)meta[0], capacity);
  const int64_t segs = (K + 1023) / 1024;
  const int64_t sf_cols = K / 16;
  // item = r * segs + sg, stepped with additions (no division in the loop)
  const int64_t first = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t step = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t dr = step / segs, ds = step - dr * segs;
  int64_t r = first / segs, sg = first - r * segs;
  for (int64_t item = first; item < P * segs; item += step, r += dr) {
    const int64_t e0 = sg * 1024;
    const float gsv = gs_of_amax_bits(amax_bits[tile_expert[r >> 7]]);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int64_t el = e0 + c * 512 + lane * 16;
      uint32_t lo = 0u, hi = 0u, sc = 0u;
      if (el < K) {
        uint32_t raw[8];
        ld_block32<true>(h + r * K + el, raw);
        sc = quant_block16_bf16(raw, block_amax_bf16(raw), gsv, rcp6, tab, lo, hi);
      }
      const uint32_t word = sc | (__shfl_down_sync(0xffffffffu, sc, 1) << 8) |
                            (__shfl_down_sync(0xffffffffu, sc, 2) << 16) |
                            (__shfl_down_sync(0xffffffffu, sc, 3) << 24);
      if (el < K) {
        *reinterpret_cast<uint2*>(fp4 + r * (K / 2) + el / 2) = make_uint2(lo, hi);
        if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(sf + sf_offset(r, el / 16, sf_cols)) = word;
      }
    }
    sg += ds;
    if (sg >= segs) {
      sg -= segs;
      ++r;
    }
  }
}

// slot_quantize_kernel from the FP8 block form of h: a lane's 16-element
// block is 16 code bytes and one exponent byte; the values dec(code) * 2^k
// are exact in FP32 and quantized exactly as the bf16 values are.
__global__ void __launch_bounds__(256) slot_quantize_fp8_kernel(const uint8_t* __restrict__ h8,
                                                                const uint8_t* __restrict__ h8_k, int64_t K,
                                                                const int32_t* __restrict__ meta,
                                                                const int32_t* __restrict__ tile_expert,
                                                                int64_t capacity,
                                                                const uint32_t* __restrict__ amax_bits, int E,
                                                                float* __restrict__ gs_out, uint8_t* __restrict__ fp4,
                                                                uint8_t* __restrict__ sf) {
  pdl_trigger();
  pdl_wait();  // h8, the amax words and the slot table come from the kernels before
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < E; i += blockDim.x) gs_out[i] = gs_of_amax_bits(amax_bits[i]);
  const float rcp6 = __frcp_rn(6.0f);
  const int lane = threadIdx.x & 31;
  const int64_t P = min((int64_t)meta[0], capacity);
  const int64_t segs = (K + 1023) / 1024;
  const int64_t sf_cols = K / 16;
  const int64_t first = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t step = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t dr = step / segs, ds = step - dr * segs;
  int64_t r = first / segs, sg = first - r * segs;
  for (int64_t item = first; item < P * segs; item += step, r += dr) {
    const int64_t e0 = sg * 1024;
    const float gsv = gs_of_amax_bits(amax_bits[tile_expert[r >> 7]]);
    const uint64_t gs2 = f2_pack(gsv, gsv);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int64_t el = e0 + c * 512 + lane * 16;
      uint32_t lo = 0u, hi = 0u, sc = 0u;
      if (el < K) {
        const uint4 cw = __ldg(reinterpret_cast<const uint4*>(h8 + r * K + el));
        const float scale = pow2f((int)h8_k[r * sf_cols + el / 16] - 127);
        const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
        uint64_t xs2[8];
        float b = 0.f;
        const uint64_t scale2 = f2_pack(scale, scale);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float v0, v1;
          e4m3x2_value(words[q >> 1] >> (16 * (q & 1)), v0, v1);
          xs2[q] = f2_mul(f2_mul(f2_pack(v0, v1), scale2), gs2);
          float x0, x1;
          f2_unpack(xs2[q], x0, x1);
          b = fmaxf(b, fmaxf(fabsf(x0), fabsf(x1)));
        }
        sc = quant_block16_pairs(xs2, b, rcp6, lo, hi);
      }
      const uint32_t word = sc | (__shfl_down_sync(0xffffffffu, sc, 1) << 8) |
                            (__shfl_down_sync(0xffffffffu, sc, 2) << 16) |
                            (__shfl_down_sync(0xffffffffu, sc, 3) << 24);
      if (el < K) {
        *reinterpret_cast<uint2*>(fp4 + r * (K / 2) + el / 2) = make_uint2(lo, hi);
        if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(sf + sf_offset(r, el / 16, sf_cols)) = word;
      }
    }
    sg += ds;
    if (sg >= segs) {
      sg -= segs;
      ++r;
    }
  }
}

int grid_for(int64_t items, int threads, int num_sms, int per_sm) {
  const int64_t need = (items + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms * per_sm;
  return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

}  // namespace

int amax_blocks_per_group(int groups, int num_sms) {
  const int want = (kAmaxBlocksPerSm * num_sms + groups - 1) / groups;
  return want < 1 ? 1 : (want < kAmaxBlocksPerGroup ? want : kAmaxBlocksPerGroup);
}

cudaError_t launch_group_amax(const uint16_t* x, int64_t rows, int64_t K, int64_t ld_x, int64_t gstride_x,
                              int groups, float* partial, float* gs_out, int num_sms, cudaStream_t s) {
  const int nb = amax_blocks_per_group(groups, num_sms);
  cudaError_t e = launch_kernel(group_amax_kernel, dim3(nb, groups), dim3(kAmaxThreads), 0, s, true, x, rows, K, ld_x,
                                gstride_x, partial, (int)kAmaxBlocksPerGroup);
  if (e != cudaSuccess || !gs_out) return e;
  return launch_kernel(group_gs_kernel, dim3((groups + 127) / 128), dim3(128), 0, s, true, (const float*)partial,
                       (int)kAmaxBlocksPerGroup, nb, groups, gs_out);
}

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t K, int64_t ld_x, int64_t gstride_x,
                            int groups, const float* gs, float* gs_copy, uint8_t* fp4, uint8_t* sf,
                            int64_t rows_padded, int num_sms, cudaStream_t s, int* status_reset,
                            const float* amax_partial) {
  const int64_t warps = rows_padded * ((K + 1023) / 1024) * groups;
  const int grid = grid_for(warps * 32, 256, num_sms, 8);
  const bool a32 = (reinterpret_cast<uintptr_t>(x) & 31u) == 0 && ld_x % 16 == 0 && gstride_x % 16 == 0;
  auto* kernel = a32 ? quantize_kernel<true> : quantize_kernel<false>;
  return launch_kernel(kernel, dim3(grid), dim3(256), 0, s, true, x, rows, K, ld_x, gstride_x, groups, gs, gs_copy,
                       amax_partial, (int)kAmaxBlocksPerGroup, amax_blocks_per_group(groups, num_sms), fp4, sf,
                       rows_padded, status_reset);
}

cudaError_t launch_assemble_scales(const uint8_t* sf_linear, int64_t sf_cols, const int32_t* offsets,
                                   const int32_t* padded_offsets, int groups, int64_t rows_capacity,
                                   uint8_t* sf_swz, int num_sms, cudaStream_t s) {
  const int64_t words = rows_capacity * ((sf_cols + 3) / 4);
  const int grid = grid_for(words, 256, num_sms, 8);
  const size_t smem = sizeof(int32_t) * 2 * (groups + 1);
  assemble_scales_kernel<<<grid, 256, smem, s>>>(sf_linear, sf_cols, offsets, padded_offsets, groups,
                                                 rows_capacity, sf_swz);
  return cudaGetLastError();
}

cudaError_t launch_gather_quantize(const uint16_t* hidden, int64_t H, int64_t T, int top_k,
                                   const int32_t* topk_ids, const int32_t* inverse, const int32_t* counts,
                                   const int32_t* offsets, int E, const float* a1_gs, int64_t capacity, uint8_t* a1,
                                   uint8_t* sfa1, cudaStream_t s, bool pdl, int* tile_done) {
  const int chunks = T <= kSmallRouteTokens ? 1 : kGatherChunks;
  const int64_t segs = (H + 512 * chunks - 1) / (512 * chunks);
  const int64_t warps = T * segs + (int64_t)E * 128;
  const int64_t grid = (warps + 7) / 8;
  const bool a32 = (reinterpret_cast<uintptr_t>(hidden) & 31u) == 0;
  auto* kernel = chunks == 1 ? (a32 ? gather_quantize_kernel<true, 1> : gather_quantize_kernel<false, 1>)
                             : (a32 ? gather_quantize_kernel<true, kGatherChunks>
                                    : gather_quantize_kernel<false, kGatherChunks>);
  return launch_kernel(kernel, dim3((unsigned)grid), dim3(256), 0, s, pdl, hidden, H, T, top_k, topk_ids, inverse,
                       counts, offsets, E, a1_gs, capacity, a1, sfa1, tile_done);
}

cudaError_t launch_gather_amax(const uint16_t* hidden, int64_t H, const int32_t* sorted_ids,
                               const int32_t* tile_expert, const int32_t* meta, int64_t capacity,
                               uint32_t* amax_bits, int num_sms, cudaStream_t s) {
  const int grid = grid_for(capacity * 32, 256, num_sms, 8);
  gather_amax_kernel<<<grid, 256, 0, s>>>(hidden, H, sorted_ids, tile_expert, meta, capacity, amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_gs_from_amax(const uint32_t* amax_bits, int n, float* gs, cudaStream_t s) {
  gs_from_amax_kernel<<<(n + 127) / 128, 128, 0, s>>>(amax_bits, n, gs);
  return cudaGetLastError();
}

cudaError_t launch_slot_quantize(const uint16_t* h, int64_t K, const int32_t* meta, const int32_t* tile_expert,
                                 int64_t capacity, const uint32_t* amax_bits, int E, float* gs_out, uint8_t* fp4,
                                 uint8_t* sf, int num_sms, cudaStream_t s, bool pdl) {
  const int grid = grid_for(capacity * ((K + 1023) / 1024) * 32, 256, num_sms, 8);
  return launch_kernel(slot_quantize_kernel, dim3(grid), dim3(256), 0, s, pdl, h, K, meta, tile_expert, capacity,
                       amax_bits, E, gs_out, fp4, sf);
}

cudaError_t launch_slot_quantize_fp8(const uint8_t* h8, const uint8_t* h8_k, int64_t K, const int32_t* meta,
                                     const int32_t* tile_expert, int64_t capacity, const uint32_t* amax_bits, int E,
                                     float* gs_out, uint8_t* fp4, uint8_t* sf, int num_sms, cudaStream_t s, bool pdl) {
  const int grid = grid_for(capacity * ((K + 1023) / 1024) * 32, 256, num_sms, 8);
  return launch_kernel(slot_quantize_fp8_kernel, dim3(grid), dim3(256), 0, s, pdl, h8, h8_k, K, meta, tile_expert,
                       capacity, amax_bits, E, gs_out, fp4, sf);
}

}  // namespace nvfp4
