// Rate of the bare block-scaled FP4 MMA stream on this GPU: the ceiling the
// grouped GEMMs are measured against, for each tile shape they could use.
//
// Every CTA (or CTA pair) stages four operand sets -- A (128 rows x 256 K
// elements), its B rows and the matching UE4M3 scale tiles, taken from the
// caller's quantized buffers -- once into shared memory and TMEM, then one
// thread issues `iters` x 4 back-to-back
//   tcgen05.mma.cta_group::{1,2}.kind::mxf4nvf4.block_scale.scale_vec::4X
// (K = 64 each) into one FP32 accumulator, cycling over the four sets, with
// no waits in between, and commits once.  No ring hand-offs, no epilogue:
// what remains is the tensor pipe's own rate for that instruction shape.
// The single wait for completion is bounded (status word on timeout).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/nvfp4moe.h"
#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kSets = 4;                 // operand sets cycled by the MMA stream
constexpr int kABytes = 128 * 128;       // 128 rows x 128 bytes (256 FP4 per row)
// warps: 0 operand copier (flag 4), 1 MMA issuer, 2-3 idle, 4-7 scale
// re-staging (flag 2), 8-11 accumulator readers (flag 8)
constexpr int kThreads = 384;
constexpr int kFlagCommitEachStage = 1;  // commit to an mbarrier after every 4 MMAs, as the GEMM's ring does
constexpr int kFlagRestageScales = 2;    // re-stage the scale tiles into TMEM continuously (tcgen05.st)
constexpr int kFlagCopyOperands = 4;     // re-copy the operand sets into shared memory continuously (bulk copies)
constexpr int kFlagReadAccumulator = 8;  // read the accumulator continuously (tcgen05.ld + FP32 work)
constexpr int kFlagFenceEachStage = 16;  // tcgen05.fence::after_thread_sync before each stage's MMAs
constexpr int kFlagWaitEachStage = 32;   // an mbarrier wait (on a completed phase) before each stage's MMAs
constexpr int kFlagCopyScales = 64;      // the MMA thread copies the set's scale tiles into TMEM (tcgen05.cp) each stage
constexpr int kFlagWarpIssue = 128;      // the whole warp runs the MMA loop (warp-uniform operands), one elected lane issues
constexpr int kFlagRing = 256;           // with 128: a 4-slot ring protocol (MMA waits full[s], commits empty[s]; warp 2 turns empty into full)
constexpr int kFlagScaleHop = 512;       // with 384: warps 4-7 also wait empty[s] and arrive on a second barrier the MMA waits for
constexpr int kFlagHopFences = 1024;     // with 896: those warps also execute tcgen05 fences around their arrival
constexpr uint64_t kTimeoutNs = 10000000000ull;  // far above the longest allowed stream (iters <= 2^21)

__host__ __device__ constexpr uint32_t idesc_nvf4_rate(int M, int N) {
  // E2M1 x E2M1, UE4M3 scales, K-major A and B, dense K = 64 (as the GEMM's)
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 7) << 27);
}

template <int N, bool PAIR>
struct RateCfg {
  static constexpr int B_ROWS = PAIR ? N / 2 : N;  // B rows staged by this CTA
  static constexpr int B_BYTES = B_ROWS * 128;
  static constexpr int SET_BYTES = kABytes + B_BYTES;
  static constexpr int SFB_COLS = N / 32;             // TMEM columns of one K-step's B scales
  static constexpr int SF_COLS = 4 * (4 + SFB_COLS);  // per operand set: 4 K-steps
  static constexpr int ACC_COLS = N;
  static constexpr int TMEM_COLS = 512;
  static_assert(ACC_COLS + kSets * SF_COLS <= TMEM_COLS, "TMEM budget");
  // at least 120 KB, so that one CTA fits per SM (two CTAs of different
  // pairs on one SM would share its tensor core and TMEM)
  static constexpr int SF_TILES = 4 + 4 * (N / 128);  // scale tiles per set (flag 64 keeps them in shared memory)
  static constexpr size_t SMEM_USED = 1024 + (size_t)kSets * SET_BYTES + (size_t)kSets * SF_TILES * 512 + 64 + 24 * kSets;
  static constexpr size_t SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
};

template <int N, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1) mma_rate_kernel(const uint8_t* __restrict__ A,
                                                               const uint8_t* __restrict__ SFA,
                                                               const uint8_t* __restrict__ B,
                                                               const uint8_t* __restrict__ SFB, int iters,
                                                               int flags, int* status,
                                                               unsigned long long* trace, int trace_stages) {
  using C = RateCfg<N, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sets = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sf_smem = sets + kSets * C::SET_BYTES;  // kSets x SF_TILES scale tiles (flag 64)
  uint64_t* done_bar = reinterpret_cast<uint64_t*>(sf_smem + kSets * C::SF_TILES * 512);
  uint64_t* stage_bar = done_bar + 1;  // per-stage commits (flag 1); nobody waits on it
  uint64_t* copy_bar = done_bar + 2;   // operand re-copies (flag 4)
  uint64_t* ready_bar = done_bar + 3;  // completed once at set-up (flag 32)
  uint64_t* ring_full = done_bar + 4;  // [kSets] (flag 256)
  uint64_t* ring_empty = done_bar + 4 + kSets;
  uint64_t* ring_sf = done_bar + 4 + 2 * kSets;  // [kSets] (flag 512), 4 arrivals
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 4 + 3 * kSets);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* stream_done = abort_flag + 1;  // set once the MMA stream has completed
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;

  // operand sets: A from the caller's A bytes, this CTA's B rows from B
  // (the pair's second CTA takes the second half of each set's B rows)
  for (int s = 0; s < kSets; ++s) {
    const uint4* a_src = reinterpret_cast<const uint4*>(A + (size_t)s * kABytes);
    const uint4* b_src = reinterpret_cast<const uint4*>(B + (size_t)s * N * 128 + (size_t)rank * C::B_BYTES);
    uint4* a_dst = reinterpret_cast<uint4*>(sets + s * C::SET_BYTES);
    uint4* b_dst = reinterpret_cast<uint4*>(sets + s * C::SET_BYTES + kABytes);
    for (int i = threadIdx.x; i < kABytes / 16; i += kThreads) a_dst[i] = a_src[i];
    for (int i = threadIdx.x; i < C::B_BYTES / 16; i += kThreads) b_dst[i] = b_src[i];
    // scale tiles of the set, in the order the MMAs read them: SFA of K-steps
    // 0-3, then per K-step the N/128 B tiles
    uint4* sf_dst = reinterpret_cast<uint4*>(sf_smem + s * C::SF_TILES * 512);
    for (int i = threadIdx.x; i < C::SF_TILES * 32; i += kThreads) {
      const int tile = i >> 5, line = i & 31;
      const uint8_t* src = tile < 4 ? SFA + (size_t)(s * 4 + tile) * 512
                                    : SFB + (size_t)((s * 4 + (tile - 4) / (N / 128)) * 2 + (tile - 4) % (N / 128)) * 512;
      sf_dst[i] = *reinterpret_cast<const uint4*>(src + 16 * line);
    }
  }
  fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core's reads
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(done_bar), 1);
    mbar_init(smem_u32(stage_bar), 1);
    mbar_init(smem_u32(copy_bar), 1);
    mbar_init(smem_u32(ready_bar), 1);
    for (int i = 0; i < kSets; ++i) {
      mbar_init(smem_u32(&ring_full[i]), 1);
      mbar_init(smem_u32(&ring_empty[i]), 1);
      mbar_init(smem_u32(&ring_sf[i]), 4);
    }
    *abort_flag = 0;
    *stream_done = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) mbar_arrive(smem_u32(ready_bar));  // phase 0 of ready_bar completes
  const uint32_t tmem = *tmem_slot;
  {
    // scale tiles -> TMEM: warp q writes 16-byte line `lane` of every 512-byte
    // tile of a set into its lane quarter (the layout the MMA reads, as the
    // GEMM's scale staging does): SFA of K-steps 0-3 (4 columns each), then per
    // K-step the B scale tiles (N/128 tiles of 4 columns)
    const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    for (int s = 0; s < kSets && warp < 4; ++s) {
      uint32_t r[48];
#pragma unroll
      for (int i = 0; i < 48; ++i) r[i] = 0u;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 a = *reinterpret_cast<const uint4*>(SFA + (size_t)(s * 4 + i) * 512 + 16 * lane);
        r[4 * i + 0] = a.x, r[4 * i + 1] = a.y, r[4 * i + 2] = a.z, r[4 * i + 3] = a.w;
#pragma unroll
        for (int t = 0; t < N / 128; ++t) {
          const uint4 b = *reinterpret_cast<const uint4*>(SFB + (size_t)((s * 4 + i) * 2 + t) * 512 + 16 * lane);
          const int c = 16 + C::SFB_COLS * i + 4 * t;
          r[c + 0] = b.x, r[c + 1] = b.y, r[c + 2] = b.z, r[c + 3] = b.w;
        }
      }
      const uint32_t col = t_lane + C::ACC_COLS + s * C::SF_COLS;
      tmem_store_32(col, r);
      if constexpr (C::SF_COLS > 32) tmem_store_16_hi(col + 32, r);
      tmem_store_wait();
    }
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync_all();  // both CTAs' operands and scales in place, TMEM allocated
  else __syncthreads();
  tc_fence_after();

  if (warp == 1 && rank == 0 && (flags & kFlagWarpIssue)) {
    // every lane computes the (warp-uniform) operands; one elected lane issues
    const uint32_t idesc = idesc_nvf4_rate(PAIR ? 256 : 128, N);
    const uint64_t a0 = smem_desc(smem_u32(sets), 16, 1024, 2);
    const uint64_t b0 = smem_desc(smem_u32(sets) + kABytes, 16, 1024, 2);
    constexpr uint64_t kSetDesc = C::SET_BYTES >> 4;
    const bool ring = (flags & kFlagRing) != 0;
    for (int it = 0; it < iters; ++it) {
      const uint32_t s = it & (kSets - 1);
      const uint64_t ad = a0 + s * kSetDesc, bd = b0 + s * kSetDesc;
      const uint32_t sf_col = tmem + C::ACC_COLS + s * C::SF_COLS;
      if (ring) {
        int ok = 1;
        if (lane == 0) ok = wait_bounded_spin(smem_u32(&ring_full[s]), (it / kSets) & 1, abort_flag, status, kTimeoutNs);
        if (lane == 0 && ok && (flags & kFlagScaleHop))
          ok = wait_bounded_spin(smem_u32(&ring_sf[s]), (it / kSets) & 1, abort_flag, status, kTimeoutNs);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        tc_fence_after();
      }
      if (elect_one()) {
        if constexpr (PAIR) {
          tc_mma_nvf4_pair(tmem, ad, bd, idesc, sf_col, sf_col + 16, it != 0);
          tc_mma_nvf4_pair(tmem, ad + 2, bd + 2, idesc, sf_col + 4, sf_col + 16 + C::SFB_COLS, 1u);
          tc_mma_nvf4_pair(tmem, ad + 4, bd + 4, idesc, sf_col + 8, sf_col + 16 + 2 * C::SFB_COLS, 1u);
          tc_mma_nvf4_pair(tmem, ad + 6, bd + 6, idesc, sf_col + 12, sf_col + 16 + 3 * C::SFB_COLS, 1u);
        } else {
          tc_mma_nvf4(tmem, ad, bd, idesc, sf_col, sf_col + 16, it != 0);
          tc_mma_nvf4(tmem, ad + 2, bd + 2, idesc, sf_col + 4, sf_col + 16 + C::SFB_COLS, 1u);
          tc_mma_nvf4(tmem, ad + 4, bd + 4, idesc, sf_col + 8, sf_col + 16 + 2 * C::SFB_COLS, 1u);
          tc_mma_nvf4(tmem, ad + 6, bd + 6, idesc, sf_col + 12, sf_col + 16 + 3 * C::SFB_COLS, 1u);
        }
        if (ring) {
          if constexpr (PAIR) tc_commit_pair_mc(smem_u32(&ring_empty[s]), 3);
          else tc_commit(smem_u32(&ring_empty[s]));
        } else if (flags & kFlagCommitEachStage) {
          if constexpr (PAIR) tc_commit_pair_mc(smem_u32(stage_bar), 3);
          else tc_commit(smem_u32(stage_bar));
        }
      }
      __syncwarp();
    }
    if (elect_one()) {
      if constexpr (PAIR) tc_commit_pair_mc(smem_u32(done_bar), 3);
      else tc_commit(smem_u32(done_bar));
    }
    __syncwarp();
  } else if (warp == 1 && lane == 0 && rank == 0) {
    const uint32_t idesc = idesc_nvf4_rate(PAIR ? 256 : 128, N);
    for (int it = 0; it < iters; ++it) {
      const int s = it & (kSets - 1);
      const uint32_t a_s = smem_u32(sets + s * C::SET_BYTES);
      const uint32_t b_s = a_s + kABytes;
      const uint32_t sf_col = tmem + C::ACC_COLS + s * C::SF_COLS;
      if (flags & kFlagWaitEachStage) {
        volatile int no_abort = 0;
        wait_bounded(smem_u32(ready_bar), 0, &no_abort, nullptr, kTimeoutNs);
      }
      if (flags & kFlagFenceEachStage) tc_fence_after();
      if (trace && blockIdx.x == 0 && it < trace_stages) trace[(int64_t)it * 8 + 5] = clock64();
      if (flags & kFlagCopyScales) {
        const uint32_t sf_s = smem_u32(sf_smem + s * C::SF_TILES * 512);
#pragma unroll
        for (int t = 0; t < C::SF_TILES; ++t) {
          const uint64_t d = smem_desc(sf_s + 512 * t, 16, 128, 0);
          if constexpr (PAIR) tc_cp_scale_tile_pair(tmem + C::ACC_COLS + s * C::SF_COLS + 4 * t, d);
          else tc_cp_scale_tile(tmem + C::ACC_COLS + s * C::SF_COLS + 4 * t, d);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint64_t ad = smem_desc(a_s + 32 * i, 16, 1024, 2);
        const uint64_t bd = smem_desc(b_s + 32 * i, 16, 1024, 2);
        if constexpr (PAIR)
          tc_mma_nvf4_pair(tmem, ad, bd, idesc, sf_col + 4 * i, sf_col + 16 + C::SFB_COLS * i, (it | i) != 0);
        else
          tc_mma_nvf4(tmem, ad, bd, idesc, sf_col + 4 * i, sf_col + 16 + C::SFB_COLS * i, (it | i) != 0);
      }
      if (trace && blockIdx.x == 0 && it < trace_stages) trace[(int64_t)it * 8 + 6] = clock64();
      if (flags & kFlagCommitEachStage) {
        if constexpr (PAIR) tc_commit_pair_mc(smem_u32(stage_bar), 3);
        else tc_commit(smem_u32(stage_bar));
      }
    }
    if constexpr (PAIR) tc_commit_pair_mc(smem_u32(done_bar), 3);
    else tc_commit(smem_u32(done_bar));
  }
  // concurrent activities of the real pipeline (each runs until the stream
  // has completed; every loop is also capped by a time limit)
  const uint64_t t_start = global_timer_ns();
  if ((flags & kFlagScaleHop) && (flags & kFlagRing) && (flags & kFlagWarpIssue) && warp >= 4 && warp < 8 &&
      rank == 0) {
    // the scale warps' hop: wait for the slot's previous MMAs, then publish it
    for (int it = 0; it < iters; ++it) {
      const int s = it & (kSets - 1);
      int ok = 1;
      if (lane == 0)
        ok = wait_bounded_spin(smem_u32(&ring_empty[s]), ((it / kSets) & 1) ^ 1u, abort_flag, status, kTimeoutNs);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (flags & kFlagHopFences) {
        tc_fence_after();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ring_sf[s]));
    }
  }
  if ((flags & kFlagRing) && (flags & kFlagWarpIssue) && warp == 2 && lane == 0 && rank == 0) {
    // turn each committed slot back into a full one (no data moves)
    for (int it = 0; it < iters; ++it) {
      const int s = it & (kSets - 1);
      if (!wait_bounded_spin(smem_u32(&ring_empty[s]), ((it / kSets) & 1) ^ 1u, abort_flag, status, kTimeoutNs)) break;
      mbar_arrive(smem_u32(&ring_full[s]));
    }
  }
  if ((flags & kFlagCopyOperands) && warp == 0 && lane == 0) {
    // re-copy operand sets (the same bytes) into shared memory, one set at a time
    uint32_t ph = 0;
    int it = 0;
    const uint64_t c0 = clock64();
    for (; !*stream_done && global_timer_ns() - t_start < kTimeoutNs; ++it) {
      const int s = it & (kSets - 1);
      mbar_arrive_expect_tx(smem_u32(copy_bar), C::SET_BYTES);
      bulk_load(smem_u32(sets + s * C::SET_BYTES), A + (size_t)s * kABytes, kABytes, smem_u32(copy_bar));
      bulk_load(smem_u32(sets + s * C::SET_BYTES + kABytes), B + (size_t)s * N * 128 + (size_t)rank * C::B_BYTES,
                C::B_BYTES, smem_u32(copy_bar));
      volatile int no_abort = 0;
      if (!wait_bounded(smem_u32(copy_bar), ph, &no_abort, nullptr, kTimeoutNs)) break;
      ph ^= 1u;
    }
    // copies completed and SM cycles spent (first CTA, trace word 7 of stages 0 and 1)
    if (trace && blockIdx.x == 0 && trace_stages > 1) {
      trace[7] = (unsigned long long)it;
      trace[15] = clock64() - c0;
    }
  } else if ((flags & kFlagRestageScales) && warp >= 4 && warp < 8) {
    // rewrite the scale columns with the values they already hold (the loop
    // condition is taken by lane 0 and shared: tcgen05.st needs the whole warp)
    const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    for (int it = 0;; ++it) {
      int go = lane == 0 ? (!*stream_done && global_timer_ns() - t_start < kTimeoutNs) : 0;
      if (!__shfl_sync(0xffffffffu, go, 0)) break;
      const int s = it & (kSets - 1);
      uint32_t r[48];
#pragma unroll
      for (int i = 0; i < 48; ++i) r[i] = 0u;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 a = *reinterpret_cast<const uint4*>(SFA + (size_t)(s * 4 + i) * 512 + 16 * lane);
        r[4 * i + 0] = a.x, r[4 * i + 1] = a.y, r[4 * i + 2] = a.z, r[4 * i + 3] = a.w;
#pragma unroll
        for (int t = 0; t < N / 128; ++t) {
          const uint4 b = *reinterpret_cast<const uint4*>(SFB + (size_t)((s * 4 + i) * 2 + t) * 512 + 16 * lane);
          const int c = 16 + C::SFB_COLS * i + 4 * t;
          r[c + 0] = b.x, r[c + 1] = b.y, r[c + 2] = b.z, r[c + 3] = b.w;
        }
      }
      const uint32_t col = t_lane + C::ACC_COLS + s * C::SF_COLS;
      const uint64_t c0 = clock64();
      tmem_store_32(col, r);
      if constexpr (C::SF_COLS > 32) tmem_store_16_hi(col + 32, r);
      tmem_store_wait();
      if (trace && blockIdx.x == 0 && warp == 4 && lane == 0 && it < trace_stages) {
        trace[(int64_t)it * 8 + 0] = c0;
        trace[(int64_t)it * 8 + 1] = clock64();
      }
      __syncwarp();
    }
  } else if ((flags & kFlagReadAccumulator) && warp >= 8) {
    // load 128 accumulator columns per pass and do FP32 work on them
    const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    float acc = 0.f;
    for (int it = 0;; ++it) {
      int go = lane == 0 ? (!*stream_done && global_timer_ns() - t_start < kTimeoutNs) : 0;
      if (!__shfl_sync(0xffffffffu, go, 0)) break;
      uint32_t v[2][32];
      const uint64_t c0 = clock64();
      tmem_load_64(t_lane + (it & 1) * 64, v[0], v[1]);
      tmem_load_wait();
      if (trace && blockIdx.x == 0 && warp == 8 && lane == 0 && it < trace_stages) {
        trace[(int64_t)it * 8 + 2] = c0;
        trace[(int64_t)it * 8 + 3] = clock64();
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) acc = __fmaf_rn(__uint_as_float(v[0][j]), __uint_as_float(v[1][j]), acc);
    }
    if (acc == 12345.f) *abort_flag = 0;  // keeps the work alive
  }
  // wait (bounded) until the stream has completed
  if (warp == 1 && lane == 0) {
    if (iters > 0) wait_bounded<PAIR>(smem_u32(done_bar), 0, abort_flag, status, kTimeoutNs);
    *stream_done = 1;
  }
  __syncwarp();
  tc_fence_before();
  if constexpr (PAIR) cluster_sync_all();  // no CTA frees TMEM while its peer's MMAs may read it
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, C::TMEM_COLS);
    else tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int N, bool PAIR>
cudaError_t launch_rate(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB, int units,
                        int iters, int flags, int* status, cudaStream_t s) {
  using C = RateCfg<N, PAIR>;
  cudaError_t e = cudaFuncSetAttribute(mma_rate_kernel<N, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)C::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(PAIR ? 2 * units : units);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  if (PAIR) {
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
  }
  unsigned long long* trace = nullptr;
  int trace_stages = 0, trace_kind = -1;
  gemm_get_trace(&trace, &trace_stages, &trace_kind);
  if (trace_kind != 4) trace = nullptr;
  return cudaLaunchKernelEx(&cfg, mma_rate_kernel<N, PAIR>, A, SFA, B, SFB, iters, flags, status, trace,
                           trace_stages);
}

}  // namespace
}  // namespace nvfp4

extern "C" int nvfp4_debug_mma_rate(const void* A, size_t a_bytes, const void* SFA, size_t sfa_bytes, const void* B,
                                    size_t b_bytes, const void* SFB, size_t sfb_bytes, int shape, int units, int iters,
                                    int flags, void* stream) {
  using namespace nvfp4;
  set_last_error("");
  auto bad = [](const char* m) {
    set_last_error(m);
    return (int)NVFP4_ERR_INVALID_ARG;
  };
  if (shape < 0 || shape > 3) return bad("shape must be 0 (128x256), 1 (pair 256x256), 2 (pair 256x128), 3 (128x128)");
  if (units < 1 || units > 4096) return bad("units must be in [1, 4096]");
  if (iters < 0 || iters > (1 << 21)) return bad("iters must be in [0, 2^21]");
  if (flags < 0 || flags > 2047) return bad("flags must be in [0, 2047]");
  if (!A || !SFA || !B || !SFB) return bad("null pointer");
  // the kernel reads 4 operand sets: A 4 x 16 KB, B 4 x N x 128 bytes, 16 A and
  // 16 * N / 128 B scale tiles of 512 bytes
  if (a_bytes < 65536 || b_bytes < 131072 || sfa_bytes < 8192 || sfb_bytes < 16384)
    return bad("buffers too small: A >= 64 KB, B >= 128 KB, SFA >= 8 KB, SFB >= 16 KB");
  for (const void* p : {A, SFA, B, SFB})
    if (reinterpret_cast<uintptr_t>(p) & 15u) return bad("pointers must be 16-byte aligned");
  int dev = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return NVFP4_ERR_CUDA;
  }
  if (major != 10 || minor != 3) {
    set_last_error("this library is built for sm_103a");
    return NVFP4_ERR_DEVICE;
  }
  int* status = nullptr;
  if ((e = gemm_status_ptr(&status)) != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return NVFP4_ERR_CUDA;
  }
  const auto* a = static_cast<const uint8_t*>(A);
  const auto* sa = static_cast<const uint8_t*>(SFA);
  const auto* b = static_cast<const uint8_t*>(B);
  const auto* sb = static_cast<const uint8_t*>(SFB);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (shape) {
    case 0: e = launch_rate<256, false>(a, sa, b, sb, units, iters, flags, status, s); break;
    case 1: e = launch_rate<256, true>(a, sa, b, sb, units, iters, flags, status, s); break;
    case 2: e = launch_rate<128, true>(a, sa, b, sb, units, iters, flags, status, s); break;
    default: e = launch_rate<128, false>(a, sa, b, sb, units, iters, flags, status, s); break;
  }
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return NVFP4_ERR_CUDA;
  }
  return NVFP4_OK;
}
