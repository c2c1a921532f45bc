// Routing and slot construction for the MoE forward, all on the device with
// no host synchronisation (vllm page, cudagraph paragraph: GPU-only expert
// offsets, no .item(), padding slots with zero weight).
//
//  route_topk     one warp per token: top-k of the FP32 logits (ties -> lower
//                 expert) by packed (logit, expert) keys held in registers,
//                 weights = exp(l_j - l_max) / sum over the chosen
//                 (softmax renormalised over the top-k); per-block expert
//                 histogram in shared memory.
//  slot_scan      one block: per-expert exclusive scan of the (expert-major)
//                 block histograms (a warp per expert), padded offsets
//                 (multiples of 128, multi-chunk experts -- vllm page "Bug 9")
//                 by a warp scan, the m-tile -> expert table (a thread per
//                 m-tile), pad rows.
//  slot_scatter   per block, the stable rank of each assignment inside its
//                 expert (ascending flat index t*k+j) via warp match/ballot,
//                 giving the slot row; writes sorted_token_ids, row weights and
//                 the inverse map.  Deterministic: no atomics decide a row.
//  route_external expert-parallel routing from the caller's global top-k ids
//                 (remap to local, weight 0 / no row for other ranks' experts).
//  token_combine  out[t] = bf16(sum over the token's top_k rows of the
//                 routing-weighted L2 output), rows in j order: deterministic.
#include <cuda_runtime.h>

#include "internal.h"
#include "nvfp4_format.cuh"
#include "ptx.cuh"

namespace nvfp4 {

namespace {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kRouteWarps = 8;

// Order-preserving key of a (logit, expert) pair: larger logit first, equal
// logits -> lower expert first.  Lanes with no expert get key 0, below every
// real key (also below -inf logits).
__device__ __forceinline__ uint64_t route_key(float v, int e) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;  // -0 ranks equal to +0
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)ord << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)e);
}
__device__ __forceinline__ float key_value(uint64_t key) {
  const uint32_t ord = (uint32_t)(key >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}
__device__ __forceinline__ int key_expert(uint64_t key) { return (int)(0xFFFFFFFFu - (uint32_t)key); }

// One warp per token, all selection state in registers (NK keys per lane,
// expert e in lane e % 32, slot e / 32).  Each of the k rounds takes the
// lane-local best key and two warp reductions: the max of the logit bits,
// then, among lanes holding that logit, the max of the low (inverted
// expert) bits, i.e. the lowest expert.  Lane j keeps the j-th selection;
// then lane j < k computes exp(l_j - l_max) and the warp sum gives the
// renormalised weights.
// s_ids / s_w (may be null): shared-memory copies of the token's k ids and
// weights, at [lane] of the given base.
template <int NK>
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int64_t t, int E, int k, int lane,
                                            int32_t* __restrict__ ids, float* __restrict__ w, int32_t* hist,
                                            int32_t* s_ids = nullptr, float* s_w = nullptr) {
  uint64_t key[NK];
#pragma unroll
  for (int i = 0; i < NK; ++i) {
    const int e = i * 32 + lane;
    key[i] = e < E ? route_key(__ldg(logits + t * E + e), e) : 0ull;
  }
  uint64_t mine = 0ull;  // lane j keeps the j-th selected key
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j >= k) break;
    uint64_t best = key[0];
#pragma unroll
    for (int i = 1; i < NK; ++i) best = key[i] > best ? key[i] : best;
    const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32));
    const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32) == hi ? (uint32_t)best : 0u);
    const uint64_t win = ((uint64_t)hi << 32) | lo;
#pragma unroll
    for (int i = 0; i < NK; ++i)
      if (key[i] == win) key[i] = 0ull;  // keys are unique: only the winner's lane matches
    if (lane == j) mine = win;
  }
  const uint64_t top = __shfl_sync(0xffffffffu, mine, 0);
  const float z = lane < k ? expf(key_value(mine) - key_value(top)) : 0.f;
  float sum = z;
#pragma unroll
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    const int e = key_expert(mine);
    const float wt = z / sum;
    ids[t * k + lane] = e;
    w[t * k + lane] = wt;
    if (s_ids) {
      s_ids[lane] = e;
      s_w[lane] = wt;
    }
    atomicAdd(&hist[e], 1);
  }
}

template <int NK>
__global__ void __launch_bounds__(kRouteWarps * 32) route_topk_kernel(
    const float* __restrict__ logits, int64_t T, int E, int k, int32_t* __restrict__ ids, float* __restrict__ w,
    int32_t* __restrict__ block_counts, int* __restrict__ status_reset) {
  pdl_trigger();
  __shared__ int32_t hist[kMaxExperts];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  pdl_wait();  // the logits may come from the kernel just before
  if (status_reset && blockIdx.x == 0 && threadIdx.x == 0) *status_reset = 0;
  const int64_t t0 = (int64_t)blockIdx.x * kRouteTokensPerBlock;
  const int64_t t1 = min(T, t0 + kRouteTokensPerBlock);
  for (int64_t t = t0 + warp; t < t1; t += kRouteWarps) route_token<NK>(logits, t, E, k, lane, ids, w, hist);
  __syncthreads();
  // expert-major: block_counts[e][block]
  for (int e = threadIdx.x; e < E; e += blockDim.x) block_counts[(int64_t)e * gridDim.x + blockIdx.x] = hist[e];
}

// Expert-parallel routing: the caller's top-k ids are global; global id g is
// local expert g - start when that lies in [0, E), else the assignment is not
// local (id -1, weight 0, no slot row).  vllm page, "Root cause of
// CUDA_ERROR_ASSERT index out of bounds", fixes 1-2.  Same block histograms
// as route_topk_kernel.
__global__ void __launch_bounds__(kRouteWarps * 32) route_external_kernel(
    const int32_t* __restrict__ topk_ids, const float* __restrict__ topk_w, int32_t start, int64_t T, int E, int k,
    int32_t* __restrict__ ids, float* __restrict__ w, int32_t* __restrict__ block_counts,
    int* __restrict__ status_reset) {
  pdl_trigger();
  __shared__ int32_t hist[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  pdl_wait();  // the ids may come from the kernel just before
  if (status_reset && blockIdx.x == 0 && threadIdx.x == 0) *status_reset = 0;
  const int64_t f0 = (int64_t)blockIdx.x * kRouteTokensPerBlock * k;
  const int64_t f1 = min(T, (int64_t)(blockIdx.x + 1) * kRouteTokensPerBlock) * k;
  for (int64_t f = f0 + threadIdx.x; f < f1; f += blockDim.x) {
    const int64_t e = (int64_t)topk_ids[f] - start;
    const bool local = e >= 0 && e < E;
    ids[f] = local ? (int32_t)e : -1;
    w[f] = local ? topk_w[f] : 0.f;
    if (local) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) block_counts[(int64_t)e * gridDim.x + blockIdx.x] = hist[e];
}

__global__ void __launch_bounds__(1024) slot_scan_kernel(int32_t* __restrict__ block_counts, int nblocks, int E,
                                                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ meta,
                                                         int32_t* __restrict__ tile_expert,
                                                         int32_t* __restrict__ sorted_ids,
                                                         float* __restrict__ row_w,
                                                         uint32_t* __restrict__ zero_words, int n_zero_words) {
  pdl_trigger();
  pdl_wait();
  __shared__ int32_t s_cnt[kMaxExperts];
  for (int i = threadIdx.x; i < n_zero_words; i += blockDim.x) zero_words[i] = 0u;
  __shared__ int32_t s_off[kMaxExperts + 1];
  // one warp per expert: exclusive scan over the route blocks, in place, on the
  // expert-major histograms.  Lane l takes entries l, l+32, ... of each
  // 512-entry chunk, so every load and store instruction covers one 128-byte
  // line; the chunk's 16 columns are scanned across the warp one after the
  // other (independent shuffle chains, a running carry).
  constexpr int kScanPerLane = 16;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int e = warp; e < E; e += nwarps) {
    int32_t* row = block_counts + (int64_t)e * nblocks;
    int carry = 0;
    for (int base = 0; base < nblocks; base += 32 * kScanPerLane) {
      int v[kScanPerLane];
#pragma unroll
      for (int i = 0; i < kScanPerLane; ++i) {
        const int b = base + i * 32 + lane;
        v[i] = b < nblocks ? row[b] : 0;
      }
#pragma unroll
      for (int i = 0; i < kScanPerLane; ++i) {
        int incl = v[i];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int x = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += x;
        }
        const int excl = carry + incl - v[i];
        carry += __shfl_sync(0xffffffffu, incl, 31);
        v[i] = excl;
      }
#pragma unroll
      for (int i = 0; i < kScanPerLane; ++i) {
        const int b = base + i * 32 + lane;
        if (b < nblocks) row[b] = v[i];
      }
    }
    if (lane == 0) {
      s_cnt[e] = carry;
      counts[e] = carry;
    }
  }
  __syncthreads();
  if (warp == 0) {  // padded offsets: exclusive scan of the 128-rounded counts
    int off = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? (s_cnt[e] + 127) / 128 * 128 : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      if (e < E) s_off[e] = off + incl - c;
      off += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      s_off[E] = off;
      meta[0] = off;
      meta[1] = off / 128;
      meta[2] = 0;
      meta[3] = 0;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = s_off[e];
  // m-tile -> expert: the last expert whose slot range starts at or before the tile
  for (int mt = threadIdx.x; mt < s_off[E] / 128; mt += blockDim.x) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= mt * 128) lo = mid;
      else hi = mid;
    }
    tile_expert[mt] = lo;
  }
  // pad rows of every slot: token -1, weight 0
  for (int i = threadIdx.x; i < E * 128; i += blockDim.x) {
    const int e = i >> 7, j = i & 127;
    const int r = s_off[e] + s_cnt[e] + j;
    if (r < s_off[e + 1]) {
      sorted_ids[r] = -1;
      row_w[r] = 0.f;
    }
  }
}

__global__ void __launch_bounds__(256) slot_scatter_kernel(const int32_t* __restrict__ ids,
                                                           const float* __restrict__ w, int64_t T, int E, int k,
                                                           const int32_t* __restrict__ block_base,
                                                           const int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ sorted_ids,
                                                           float* __restrict__ row_w, int32_t* __restrict__ inverse) {
  pdl_trigger();
  pdl_wait();
  __shared__ int32_t running[kMaxExperts];
  __shared__ int32_t warp_cnt[8][kMaxExperts];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    running[e] = block_base[(int64_t)e * gridDim.x + blockIdx.x] + offsets[e];
#pragma unroll
    for (int q = 0; q < 8; ++q) warp_cnt[q][e] = 0;
  }
  __syncthreads();
  const int64_t f0 = (int64_t)blockIdx.x * kRouteTokensPerBlock * k;
  const int64_t f1 = min(T, (int64_t)(blockIdx.x + 1) * kRouteTokensPerBlock) * k;
  for (int64_t base = f0; base < f1; base += blockDim.x) {
    const int64_t f = base + threadIdx.x;
    const bool valid = f < f1;
    const int e = valid ? ids[f] : -1;
    const bool local = e >= 0;  // -1: an expert-parallel assignment to another rank
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (local && rank == 0) warp_cnt[warp][e] = __popc(peers);
    __syncthreads();
    if (valid && !local) inverse[f] = -1;
    if (local) {
      int pre = running[e] + rank;
      for (int q = 0; q < warp; ++q) pre += warp_cnt[q][e];
      sorted_ids[pre] = (int32_t)(f / k);
      row_w[pre] = w[f];
      inverse[f] = pre;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
      int add = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        add += warp_cnt[q][x];
        warp_cnt[q][x] = 0;
      }
      running[x] += add;
    }
    __syncthreads();
  }
}

// One 256-thread block per token; thread i owns 8 consecutive features per
// 2048-feature stripe and adds the token's k rows (16-byte loads) in j order.
__global__ void __launch_bounds__(256) token_combine_kernel(const uint16_t* __restrict__ y,
                                                            const int32_t* __restrict__ inverse, int64_t H, int k,
                                                            uint16_t* __restrict__ out) {
  pdl_trigger();  // the next forward's first kernel may start its prologue
  pdl_wait();
  // gridDim.y blocks share a token's columns (several per token for small batches)
  const int64_t t = blockIdx.x;
  const int64_t c0 = H * blockIdx.y / gridDim.y, c1 = H * (blockIdx.y + 1) / gridDim.y;
  __shared__ int32_t rows[kMaxTopK];
  __shared__ int n_rows;
  if (threadIdx.x == 0) {  // the token's local rows in j order (non-local ones contribute nothing)
    int n = 0;
    for (int j = 0; j < k; ++j) {
      const int r = inverse[t * k + j];
      if (r >= 0) rows[n++] = r;
    }
    n_rows = n;
  }
  __syncthreads();
  const int n = n_rows;
  for (int64_t c = c0 + (int64_t)threadIdx.x * 8; c < c1; c += (int64_t)blockDim.x * 8) {
    // all of the token's rows in flight at once, then summed in j order
    uint4 v[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < n) v[j] = __ldg(reinterpret_cast<const uint4*>(y + (int64_t)rows[j] * H + c));
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j >= n) break;
      const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += bf16_lo(u[q]);
        acc[2 * q + 1] += bf16_hi(u[q]);
      }
    }
    *reinterpret_cast<uint4*>(out + t * H + c) = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                                           pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

// Small batches (T <= kSmallRouteTokens): routing, padded offsets, tile
// table, pad rows and the stable slot permutation in one launch of a cluster
// of kSmallCtas CTAs (the same arithmetic as route_topk / route_external,
// slot_scan and slot_scatter, without their launch boundaries).  CTA r routes
// tokens [32r, 32r + 32), a warp per token; the CTAs read each other's
// per-expert counts through distributed shared memory, so each knows the
// totals (padded offsets) and how many rows of every expert the lower-ranked
// CTAs' tokens take (its first slot per expert), and ranks its own
// assignments from there.
constexpr int kSmallWarps = 32;
constexpr int kSmallCtas = 8;
static_assert(kSmallWarps * kSmallCtas == kSmallRouteTokens, "one token per warp");

template <int NK>
__global__ void __cluster_dims__(kSmallCtas, 1, 1) __launch_bounds__(kSmallWarps * 32) route_small_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ ext_ids, const float* __restrict__ ext_w,
    int32_t start, int64_t T, int E, int k, int32_t* __restrict__ ids, float* __restrict__ w,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ meta,
    int32_t* __restrict__ tile_expert, int32_t* __restrict__ sorted_ids, float* __restrict__ row_w,
    int32_t* __restrict__ inverse, int* __restrict__ status_reset) {
  pdl_trigger();
  __shared__ int32_t hist[kMaxExperts];     // this CTA's tokens' rows per expert
  __shared__ int32_t total[kMaxExperts];    // all CTAs' rows per expert
  __shared__ int32_t s_off[kMaxExperts + 1];
  __shared__ int32_t running[kMaxExperts];  // next slot of this CTA per expert
  __shared__ int32_t warp_cnt[kSmallWarps][kMaxExperts];
  __shared__ int32_t s_ids[kSmallWarps * kMaxTopK];  // this CTA's assignments, flat index - f0
  __shared__ float s_w[kSmallWarps * kMaxTopK];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t rank = cluster_ctarank();
  const int64_t t0 = (int64_t)rank * kSmallWarps, t1 = min(T, t0 + kSmallWarps);
  const int64_t f0 = t0 * k, f1 = t1 > t0 ? t1 * k : f0;  // this CTA's assignments
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  pdl_wait();  // the logits or ids may come from the kernel just before
  if (status_reset && rank == 0 && threadIdx.x == 0) *status_reset = 0;
  // phase 1: routing of this CTA's tokens and their per-expert counts
  if (logits) {
    if (t0 + warp < t1)
      route_token<NK>(logits, t0 + warp, E, k, lane, ids, w, hist, s_ids + warp * k, s_w + warp * k);
  } else {
    for (int64_t f = f0 + threadIdx.x; f < f1; f += blockDim.x) {
      const int64_t e = (int64_t)ext_ids[f] - start;
      const bool local = e >= 0 && e < E;
      const int32_t id = local ? (int32_t)e : -1;
      const float wt = local ? ext_w[f] : 0.f;
      ids[f] = id;
      w[f] = wt;
      s_ids[f - f0] = id;
      s_w[f - f0] = wt;
      if (local) atomicAdd(&hist[e], 1);
    }
  }
  cluster_sync_all();  // every CTA's counts are final
  // phase 2: totals and this CTA's first slot per expert (rows of the
  // lower-ranked CTAs come first: ascending flat index), padded offsets
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const uint32_t a = smem_u32(&hist[e]);
    int sum = 0, below = 0;
#pragma unroll
    for (int q = 0; q < kSmallCtas; ++q) {
      const int c = (int)ld_shared_cluster_u32(mapa_shared(a, (uint32_t)q));
      sum += c;
      below += q < (int)rank ? c : 0;
    }
    total[e] = sum;
    running[e] = below;
  }
  __syncthreads();
  // the remote reads above have completed (their values are stored): this
  // CTA's part of the closing rendezvous, awaited just before it exits
  cluster_arrive_relaxed();
  if (warp == 0) {
    int off = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? (total[e] + 127) / 128 * 128 : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      if (e < E) s_off[e] = off + incl - c;
      off += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      s_off[E] = off;
      if (rank == 0) {
        meta[0] = off;
        meta[1] = off / 128;
        meta[2] = 0;
        meta[3] = 0;
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) running[e] += s_off[e];
  if (rank == 0) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = s_off[e];
    for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = total[e];
    for (int mt = threadIdx.x; mt < s_off[E] / 128; mt += blockDim.x) {
      int lo = 0, hi = E;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= mt * 128) lo = mid;
        else hi = mid;
      }
      tile_expert[mt] = lo;
    }
  }
  // pad rows, spread over the cluster
  for (int i = (int)rank * blockDim.x + threadIdx.x; i < E * 128; i += kSmallCtas * blockDim.x) {
    const int e = i >> 7, j = i & 127;
    const int r = s_off[e] + total[e] + j;
    if (r < s_off[e + 1]) {
      sorted_ids[r] = -1;
      row_w[r] = 0.f;
    }
  }
  for (int i = threadIdx.x; i < kSmallWarps * E; i += blockDim.x) warp_cnt[i / E][i % E] = 0;
  __syncthreads();
  // phase 3: stable rank of every assignment of this CTA inside its expert
  for (int64_t base = f0; base < f1; base += blockDim.x) {
    const int64_t f = base + threadIdx.x;
    const bool valid = f < f1;
    const int e = valid ? s_ids[f - f0] : -1;
    const bool local = e >= 0;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rk = __popc(peers & ((1u << lane) - 1u));
    if (local && rk == 0) warp_cnt[warp][e] = __popc(peers);
    __syncthreads();
    if (valid && !local) inverse[f] = -1;
    if (local) {
      int pre = running[e] + rk;
      for (int q = 0; q < warp; ++q) pre += warp_cnt[q][e];
      sorted_ids[pre] = (int32_t)(f / k);
      row_w[pre] = s_w[f - f0];
      inverse[f] = pre;
    }
    if (base + (int64_t)blockDim.x >= f1) break;  // last pass: the running starts are not needed again
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
      int add = 0;
      for (int q = 0; q < kSmallWarps; ++q) {
        add += warp_cnt[q][x];
        warp_cnt[q][x] = 0;
      }
      running[x] += add;
    }
    __syncthreads();
  }
  cluster_wait();  // no CTA leaves while another may still read its counts
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w,
                              int32_t* block_counts, int* status_reset, cudaStream_t s) {
  const int64_t nb = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  const dim3 grid((unsigned)nb), block(kRouteWarps * 32);
  auto* kernel = E <= 32 ? route_topk_kernel<1> : E <= 64 ? route_topk_kernel<2> : E <= 128 ? route_topk_kernel<4>
                                                                                            : route_topk_kernel<8>;
  return launch_kernel(kernel, grid, block, 0, s, true, logits, T, E, k, ids, w, block_counts, status_reset);
}

cudaError_t launch_route_external(const int32_t* topk_ids, const float* topk_w, int32_t start, int64_t T, int E,
                                  int k, int32_t* ids, float* w, int32_t* block_counts, int* status_reset,
                                  cudaStream_t s) {
  const int64_t nb = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  return launch_kernel(route_external_kernel, dim3((unsigned)nb), dim3(kRouteWarps * 32), 0, s, true, topk_ids, topk_w,
                       start, T, E, k, ids, w, block_counts, status_reset);
}

cudaError_t launch_route_small(const float* logits, const int32_t* ext_ids, const float* ext_w, int32_t start,
                               int64_t T, int E, int k, int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                               int32_t* meta, int32_t* tile_expert, int32_t* sorted_ids, float* row_w,
                               int32_t* inverse, int* status_reset, cudaStream_t s) {
  auto* kernel = (!logits || E <= 32) ? route_small_kernel<1>
                 : E <= 64            ? route_small_kernel<2>
                 : E <= 128           ? route_small_kernel<4>
                                      : route_small_kernel<8>;
  // one cluster (the kernel's compile-time cluster shape)
  return launch_kernel(kernel, dim3(kSmallCtas), dim3(kSmallWarps * 32), 0, s, true, logits, ext_ids, ext_w, start,
                       T, E, k, ids, w, counts, offsets, meta, tile_expert, sorted_ids, row_w, inverse, status_reset);
}

cudaError_t launch_slot_scan(int32_t* block_counts, int nblocks, int E, int32_t* counts, int32_t* offsets,
                             int32_t* meta, int32_t* tile_expert, int32_t* sorted_ids, float* row_w,
                             uint32_t* zero_words, int n_zero_words, cudaStream_t s, bool pdl) {
  return launch_kernel(slot_scan_kernel, dim3(1), dim3(1024), 0, s, pdl, block_counts, nblocks, E, counts, offsets,
                       meta, tile_expert, sorted_ids, row_w, zero_words, n_zero_words);
}

cudaError_t launch_slot_scatter(const int32_t* ids, const float* w, int64_t T, int E, int k,
                                const int32_t* block_base, const int32_t* offsets, int32_t* sorted_ids,
                                float* row_w, int32_t* inverse, cudaStream_t s, bool pdl) {
  const int64_t nb = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  return launch_kernel(slot_scatter_kernel, dim3((unsigned)nb), dim3(256), 0, s, pdl, ids, w, T, E, k, block_base,
                       offsets, sorted_ids, row_w, inverse);
}

cudaError_t launch_token_combine(const uint16_t* y, const int32_t* inverse, int64_t T, int64_t H, int k,
                                 uint16_t* out, cudaStream_t s, bool pdl) {
  if (T == 0) return cudaSuccess;
  // small batches: 4 blocks per token (column quarters, multiples of 8) for more loads in flight
  const unsigned split = T <= kSmallRouteTokens && H % 32 == 0 ? 4u : 1u;
  return launch_kernel(token_combine_kernel, dim3((unsigned)T, split), dim3(256), 0, s, pdl, y, inverse, H, k, out);
}

}  // namespace nvfp4
