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
constexpr int kThreads = 128;
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
  static constexpr size_t SMEM_USED = 1024 + (size_t)kSets * SET_BYTES + 64;
  static constexpr size_t SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
};

template <int N, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1) mma_rate_kernel(const uint8_t* __restrict__ A,
                                                               const uint8_t* __restrict__ SFA,
                                                               const uint8_t* __restrict__ B,
                                                               const uint8_t* __restrict__ SFB, int iters,
                                                               int* status) {
  using C = RateCfg<N, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sets = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* done_bar = reinterpret_cast<uint64_t*>(sets + kSets * C::SET_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
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
  }
  fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core's reads
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(done_bar), 1);
    *abort_flag = 0;
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
  const uint32_t tmem = *tmem_slot;
  {
    // scale tiles -> TMEM: warp q writes 16-byte line `lane` of every 512-byte
    // tile of a set into its lane quarter (the layout the MMA reads, as the
    // GEMM's scale staging does): SFA of K-steps 0-3 (4 columns each), then per
    // K-step the B scale tiles (N/128 tiles of 4 columns)
    const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    for (int s = 0; s < kSets; ++s) {
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

  if (warp == 1 && lane == 0 && rank == 0) {
    const uint32_t idesc = idesc_nvf4_rate(PAIR ? 256 : 128, N);
    for (int it = 0; it < iters; ++it) {
      const int s = it & (kSets - 1);
      const uint32_t a_s = smem_u32(sets + s * C::SET_BYTES);
      const uint32_t b_s = a_s + kABytes;
      const uint32_t sf_col = tmem + C::ACC_COLS + s * C::SF_COLS;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint64_t ad = smem_desc(a_s + 32 * i, 16, 1024, 2);
        const uint64_t bd = smem_desc(b_s + 32 * i, 16, 1024, 2);
        if constexpr (PAIR)
          tc_mma_nvf4_pair(tmem, ad, bd, idesc, sf_col + 4 * i, sf_col + 16 + C::SFB_COLS * i, (it | i) != 0);
        else
          tc_mma_nvf4(tmem, ad, bd, idesc, sf_col + 4 * i, sf_col + 16 + C::SFB_COLS * i, (it | i) != 0);
      }
    }
    if constexpr (PAIR) tc_commit_pair_mc(smem_u32(done_bar), 3);
    else tc_commit(smem_u32(done_bar));
  }
  // every thread waits (bounded) until the stream has completed
  if (lane == 0) {
    if (iters > 0)
      wait_bounded<PAIR>(smem_u32(done_bar), 0, abort_flag, status, kTimeoutNs);
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
                        int iters, int* status, cudaStream_t s) {
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
  return cudaLaunchKernelEx(&cfg, mma_rate_kernel<N, PAIR>, A, SFA, B, SFB, iters, status);
}

}  // namespace
}  // namespace nvfp4

extern "C" int nvfp4_debug_mma_rate(const void* A, size_t a_bytes, const void* SFA, size_t sfa_bytes, const void* B,
                                    size_t b_bytes, const void* SFB, size_t sfb_bytes, int shape, int units, int iters,
                                    void* stream) {
  using namespace nvfp4;
  set_last_error("");
  auto bad = [](const char* m) {
    set_last_error(m);
    return (int)NVFP4_ERR_INVALID_ARG;
  };
  if (shape < 0 || shape > 3) return bad("shape must be 0 (128x256), 1 (pair 256x256), 2 (pair 256x128), 3 (128x128)");
  if (units < 1 || units > 4096) return bad("units must be in [1, 4096]");
  if (iters < 0 || iters > (1 << 21)) return bad("iters must be in [0, 2^21]");
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
    case 0: e = launch_rate<256, false>(a, sa, b, sb, units, iters, status, s); break;
    case 1: e = launch_rate<256, true>(a, sa, b, sb, units, iters, status, s); break;
    case 2: e = launch_rate<128, true>(a, sa, b, sb, units, iters, status, s); break;
    default: e = launch_rate<128, false>(a, sa, b, sb, units, iters, status, s); break;
  }
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return NVFP4_ERR_CUDA;
  }
  return NVFP4_OK;
}
