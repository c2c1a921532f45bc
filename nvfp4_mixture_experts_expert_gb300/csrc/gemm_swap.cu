// MoE L2 GEMM for small batches with the operands swapped: the MMA's A
// operand is a 128-row tile of the expert's W2 (128 output features), its
// B operand 64 slot rows of the L1 output, so the accumulator holds
// features x slots and each MMA covers only the 64 slot rows a decode-sized
// expert has, instead of a 128-row slot tile of which most rows are padding
// (vllm page, "Bug 9" paragraph: decode batches still get 128-row slots per
// expert).  The epilogue is the routing-weighted one of the L2 GEMM:
//   Y[row] = bf16(w_row * alpha_g * acc) for the expert's real slot rows,
// alpha_g = 1 / (a2_gs[g] * w2_gs[g]), rows stored in slot order for the
// token combine (vllm page: scatter_add paragraph).
//
// Work items: (expert g, 64-row slot block j, 128-feature tile t), the slot
// blocks of an expert counted from its real rows (counts[g]); t minor, so
// the CTAs on one slot block share its rows through L2 and each streams a
// different weight tile.  Warps: 0 operand producer (TMA: 16 KB of weights
// + 8 KB of slot rows per K-stage of 256, 7-stage ring), 1 TMEM allocator
// and MMA issuer (tcgen05.mma kind::mxf4nvf4 block_scale scale_vec::4X,
// M = 128, N = 64, two 64-column accumulators), 2 scale producer (bulk
// copies into a ring of their own), 4-7 epilogue (one per TMEM lane
// quarter: 32 features x 64 slots), 8-11 scale staging into TMEM with
// tcgen05.st.  The slot rows' scales come from the 128-row tile layout:
// word c of line l is row 32c + l, so a 64-row block at an odd multiple of
// 64 takes words 2 and 3.  The MMA reads the B scales of N = 64 from two
// columns.
// Every wait is bounded (timeout -> device status word, abort, drain of
// copies / MMAs in flight, TMEM freed, return).  With the L1 -> L2 hand-off
// the producers wait for the L1 output of their slot block's m-tile.
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "nvfp4_format.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kSwM = 128;                       // weight rows (features) per tile
constexpr int kSwN = 64;                        // slot rows per tile
constexpr int kSwBk = 128;                      // bytes per row per K-stage (256 FP4)
constexpr int kSwWBytes = kSwM * kSwBk;         // 16 KB
constexpr int kSwXBytes = kSwN * kSwBk;         // 8 KB
constexpr int kSwStageBytes = kSwWBytes + kSwXBytes;
constexpr int kSwStages = 7;
constexpr int kSwSfSlotBytes = 2 * 4 * 512;     // 4 weight + 4 slot scale tiles
constexpr int kSwAccBufs = 2;
constexpr int kSwSfCol0 = kSwAccBufs * kSwN;    // scale columns after the accumulators
constexpr int kSwSfCols = 32;                   // per stage: 4 x 4 weight + 4 x 4 slot (2 used)
constexpr int kSwTmemCols = 512;
constexpr int kSwThreads = 12 * 32;
constexpr int kSwEpiWarp0 = 4, kSwSfWarp0 = 8;
constexpr int kSwMaxGroups = 256;
static_assert(kSwSfCol0 + kSwStages * kSwSfCols <= kSwTmemCols, "TMEM budget");
static_assert(kSwStageBytes % 1024 == 0, "stage alignment");

struct SwLayout {
  uint8_t* stages;
  uint8_t* sf_slots;
  uint64_t* full;       // [kSwStages] operands landed
  uint64_t* empty;      // [kSwStages] MMAs of the stage committed
  uint64_t* sf_data;    // [kSwStages] scale slot landed
  uint64_t* sf_empty;   // [kSwStages] scale slot read
  uint64_t* sf_full;    // [kSwStages] scales of the stage in TMEM
  uint64_t* acc_full;   // [kSwAccBufs]
  uint64_t* acc_empty;  // [kSwAccBufs]
  uint64_t* drain;
  uint32_t* tmem_slot;
  int* abort_flag;
  int* offsets;   // [G+1]
  int* counts;    // [G]
  int* unit_off;  // [G+1] first slot block of each group
};

__device__ __forceinline__ SwLayout sw_carve(uint8_t* raw, int G) {
  SwLayout L;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  L.stages = base;
  L.sf_slots = base + kSwStages * kSwStageBytes;
  uint64_t* b = reinterpret_cast<uint64_t*>(L.sf_slots + kSwStages * kSwSfSlotBytes);
  L.full = b;
  L.empty = L.full + kSwStages;
  L.sf_data = L.empty + kSwStages;
  L.sf_empty = L.sf_data + kSwStages;
  L.sf_full = L.sf_empty + kSwStages;
  L.acc_full = L.sf_full + kSwStages;
  L.acc_empty = L.acc_full + kSwAccBufs;
  L.drain = L.acc_empty + kSwAccBufs;
  L.tmem_slot = reinterpret_cast<uint32_t*>(L.drain + 1);
  L.abort_flag = reinterpret_cast<int*>(L.tmem_slot + 1);
  L.offsets = L.abort_flag + 1;
  L.counts = L.offsets + G + 1;
  L.unit_off = L.counts + G;
  return L;
}

constexpr size_t sw_smem_bytes(int G) {
  return 1024 + (size_t)kSwStages * kSwStageBytes + (size_t)kSwStages * kSwSfSlotBytes +
         8 * (5 * kSwStages + 2 * kSwAccBufs + 1) + 8 + 4 * (3 * (size_t)G + 2) + 16;
}

__device__ __forceinline__ int sw_find_group(const int* off, int G, int u) {
  int lo = 0, hi = G;  // largest g in [0, G) with off[g] <= u
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= u) lo = mid; else hi = mid;
  }
  return lo;
}

struct SwWork {
  int g, t;
  int row0;   // first slot row of the block
  int nrows;  // real rows in it (1..64)
};

__device__ __forceinline__ SwWork sw_decode(const SwLayout& L, const SwapArgs& p, int it) {
  const int u = it / p.n_wtiles;
  SwWork w;
  w.t = it - u * p.n_wtiles;
  w.g = sw_find_group(L.unit_off, p.G, u);
  const int j = u - L.unit_off[w.g];
  w.row0 = L.offsets[w.g] + j * kSwN;
  w.nrows = min(kSwN, L.counts[w.g] - j * kSwN);
  return w;
}

// Bounded wait (one lane) until a counter another kernel increments reaches target.
__device__ __forceinline__ bool sw_wait_count(const int* counter, int target, volatile int* abort, int* status,
                                              uint64_t timeout_ns) {
  if (ld_acquire_gpu(counter) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (ld_acquire_gpu(counter) >= target) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > timeout_ns) {
      *abort = 1;
      if (status) atomicExch(status, 6 /* NVFP4_ERR_DEVICE_TIMEOUT */);
      return false;
    }
  }
}

// Operand producer (SCALES = false) or scale producer (SCALES = true).
template <bool SCALES>
__device__ void sw_producer(const SwapArgs& p, const SwLayout& L, int total, int start, int step) {
  volatile int* abort = L.abort_flag;
  const int lane = threadIdx.x & 31;
  const bool leader = elect_one();
  constexpr uint32_t kSlotBytes = SCALES ? kSwSfSlotBytes : kSwStageBytes;
  const uint32_t empty0 = smem_u32(SCALES ? L.sf_empty : L.empty);
  const uint32_t done0 = smem_u32(SCALES ? L.sf_data : L.full);
  const uint32_t slot0 = smem_u32(SCALES ? L.sf_slots : L.stages);
  const int kt = p.K / 64;  // scale tiles per 128-row band
  const bool per_tile = p.tile_done && p.tile_done_target > 0;
  uint32_t issued = 0, issued_parity = 0;
  uint32_t stage = 0, phase = 0;
  int ok = 1, ready_mt = -1;
  for (int it = start; it < total && ok && !*abort; it += step) {
    const SwWork w = sw_decode(L, p, it);
    const int mt = w.row0 / 128;
    if (per_tile && mt != ready_mt) {
      if (lane == 0) ok = sw_wait_count(p.tile_done + mt, p.tile_done_target, abort, p.status, p.timeout_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      (void)ld_acquire_gpu(p.tile_done + mt);  // every lane, then the copies may read the m-tile
      fence_proxy_async_global();
      ready_mt = mt;
    }
    const uint8_t* sfw = p.sfw + (int64_t)w.g * p.sfw_group_bytes + (int64_t)w.t * kt * 512;
    const uint8_t* sfx = p.sfx + (int64_t)mt * kt * 512;
    for (int kb = 0; kb < p.num_kb; ++kb) {
      if (lane == 0) ok = wait_bounded_spin(empty0 + 8 * stage, phase ^ 1u, abort, p.status, p.timeout_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const uint32_t st = slot0 + stage * kSlotBytes;
      const uint32_t bar = done0 + 8 * stage;
      if (leader) {
        if constexpr (SCALES) {
          const uint32_t bytes = (uint32_t)min(4, (p.K - kb * 256) / 64) * 512;
          mbar_arrive_expect_tx(bar, 2 * bytes);
          bulk_load(st, sfw + kb * 2048, bytes, bar);
          bulk_load(st + 2048, sfx + kb * 2048, bytes, bar);
        } else {
          mbar_arrive_expect_tx(bar, kSwStageBytes);
          tma_load_2d(st, &p.tmap_w, kb * kSwBk, w.g * p.H + w.t * kSwM, bar);
          tma_load_2d(st + kSwWBytes, &p.tmap_x, kb * kSwBk, w.row0, bar);
        }
      }
      __syncwarp();
      issued |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == kSwStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (lane == 0 && (*abort || !ok)) {  // let copies already issued land before the CTA exits
    for (int s = 0; s < kSwStages; ++s)
      if (issued & (1u << s)) {
        volatile int no_abort = 0;
        wait_bounded(done0 + 8 * s, (issued_parity >> s) & 1u, &no_abort, nullptr, p.timeout_ns);
      }
  }
  __syncwarp();
}

// Scale staging: lane l of the warp for lane quarter q writes line l of the
// stage's weight scale tiles (4 columns each) and the two words of the slot
// block's rows of the slot scale tiles into TMEM lane 32q + l.
__device__ void sw_sf_loop(const SwapArgs& p, const SwLayout& L, int total, int start, int step, uint32_t tmem) {
  volatile int* abort = L.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  uint32_t stage = 0, phase = 0, slot = 0, sphase = 0;
  int ok = 1;
  for (int it = start; it < total && ok; it += step) {
    const SwWork w = sw_decode(L, p, it);
    const int half = (w.row0 >> 6) & 1;  // which 64 rows of its 128-row scale tile
    for (int kb = 0; kb < p.num_kb; ++kb) {
      if (lane == 0) ok = wait_bounded_spin(smem_u32(&L.sf_data[slot]), sphase, abort, p.status, p.timeout_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const uint8_t* sf = L.sf_slots + slot * kSwSfSlotBytes + 16 * lane;
      uint32_t r[48];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 a = *reinterpret_cast<const uint4*>(sf + 512 * i);
        const uint4 b = *reinterpret_cast<const uint4*>(sf + 2048 + 512 * i);
        r[4 * i + 0] = a.x, r[4 * i + 1] = a.y, r[4 * i + 2] = a.z, r[4 * i + 3] = a.w;
        r[16 + 4 * i + 0] = half ? b.z : b.x;
        r[16 + 4 * i + 1] = half ? b.w : b.y;
        r[16 + 4 * i + 2] = 0u;
        r[16 + 4 * i + 3] = 0u;
      }
#pragma unroll
      for (int i = 32; i < 48; ++i) r[i] = 0u;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&L.sf_empty[slot]));
      // the stage's TMEM scale columns are free once its previous MMAs committed
      if (lane == 0) ok = wait_bounded_spin(smem_u32(&L.empty[stage]), phase ^ 1u, abort, p.status, p.timeout_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      tmem_store_32(t_lane + kSwSfCol0 + stage * kSwSfCols, r);
      tmem_store_wait();
      tc_fence_before();
      if (lane == 0) mbar_arrive(smem_u32(&L.sf_full[stage]));
      if (++stage == kSwStages) {
        stage = 0;
        phase ^= 1u;
      }
      if (++slot == kSwStages) {
        slot = 0;
        sphase ^= 1u;
      }
    }
  }
}

__device__ void sw_mma_loop(const SwapArgs& p, const SwLayout& L, int total, int start, int step, uint32_t tmem) {
  volatile int* abort = L.abort_flag;
  const int lane = threadIdx.x & 31;
  const bool leader = elect_one();
  const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(kSwN >> 3) << 17) | ((uint32_t)(kSwM >> 7) << 27);
  const uint64_t w_desc0 = smem_desc(smem_u32(L.stages), 16, 1024, 2);
  const uint64_t x_desc0 = smem_desc(smem_u32(L.stages) + kSwWBytes, 16, 1024, 2);
  constexpr uint64_t kSlotDesc = kSwStageBytes >> 4;
  uint32_t stage = 0, phase = 0;
  bool issued_any = false;
  int ok = 1, tile = 0;
  for (int it = start; it < total && ok && !*abort; it += step, ++tile) {
    const uint32_t buf = (uint32_t)(tile & 1), acc_phase = (uint32_t)(tile >> 1) & 1u;
    if (lane == 0)
      ok = wait_bounded_spin(smem_u32(&L.acc_empty[buf]), acc_phase ^ 1u, abort, p.status, p.timeout_ns);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    for (int kb = 0; kb < p.num_kb; ++kb) {
      if (lane == 0) {
        ok = wait_bounded_spin(smem_u32(&L.sf_full[stage]), phase, abort, p.status, p.timeout_ns);
        if (ok) ok = wait_bounded_spin(smem_u32(&L.full[stage]), phase, abort, p.status, p.timeout_ns);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int nk = min(4, (p.K - kb * 256) / 64);
      if (leader) {
        const uint32_t sf_col = tmem + kSwSfCol0 + stage * kSwSfCols;
        for (int i = 0; i < nk; ++i)
          tc_mma_nvf4(tmem + buf * kSwN, w_desc0 + stage * kSlotDesc + 2 * i, x_desc0 + stage * kSlotDesc + 2 * i,
                      idesc, sf_col + 4 * i, sf_col + 16 + 4 * i, (kb | i) ? 1u : 0u);
        tc_commit(smem_u32(&L.empty[stage]));
      }
      __syncwarp();
      issued_any = true;
      if (++stage == kSwStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
    if (leader) tc_commit(smem_u32(&L.acc_full[buf]));
    __syncwarp();
  }
  if (*abort && issued_any) {  // every MMA issued must finish before TMEM is freed
    if (leader) tc_commit(smem_u32(L.drain));
    __syncwarp();
    if (lane == 0) {
      volatile int no_abort = 0;
      wait_bounded(smem_u32(L.drain), 0, &no_abort, nullptr, p.timeout_ns);
    }
    __syncwarp();
  }
}

// One warp per TMEM lane quarter: 32 features x the 64 slot columns of the
// tile; each column's 32 features are 64 contiguous bytes of one Y row.
__device__ void sw_epilogue(const SwapArgs& p, const SwLayout& L, int total, int start, int step, uint32_t tmem) {
  volatile int* abort = L.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const uint32_t t_base = tmem + ((uint32_t)(quarter * 32) << 16);
  int tile = 0;
  for (int it = start; it < total; it += step, ++tile) {
    const SwWork w = sw_decode(L, p, it);
    const float alpha = 1.0f / (p.x_gs[w.g] * p.w_gs[w.g]);
    // routing weight of the row in this lane's column pair (c = lane, lane + 32)
    const float w0 = lane < w.nrows ? p.row_w[w.row0 + lane] * alpha : 0.f;
    const float w1 = lane + 32 < w.nrows ? p.row_w[w.row0 + 32 + lane] * alpha : 0.f;
    const uint32_t buf = (uint32_t)(tile & 1), acc_phase = (uint32_t)(tile >> 1) & 1u;
    int ok = 1;
    if (lane == 0) ok = wait_bounded_spin(smem_u32(&L.acc_full[buf]), acc_phase, abort, p.status, p.timeout_ns);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    __syncwarp();
    tc_fence_after();
    uint32_t v[2][32];
    tmem_load_64(t_base + buf * kSwN, v[0], v[1]);
    tmem_load_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&L.acc_empty[buf]));
    uint16_t* ycol = p.y + (int64_t)w.row0 * p.H + w.t * kSwM + quarter * 32 + lane;
#pragma unroll
    for (int c = 0; c < kSwN; ++c) {
      const float wc = __shfl_sync(0xffffffffu, c < 32 ? w0 : w1, c & 31);
      if (c < w.nrows) {
        const float y = __uint_as_float(v[c >> 5][c & 31]) * wc;  // as the slot-major epilogue: bf16(acc * (w * alpha))
        ycol[(int64_t)c * p.H] = (uint16_t)(pack_bf16x2(y, 0.f) & 0xFFFFu);
      }
    }
  }
}

__global__ void __launch_bounds__(kSwThreads, 1) nvfp4_gemm_swap_kernel(const __grid_constant__ SwapArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const SwLayout L = sw_carve(smem_raw, p.G);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSwStages; ++s) {
      mbar_init(smem_u32(&L.full[s]), 1);
      mbar_init(smem_u32(&L.empty[s]), 1);
      mbar_init(smem_u32(&L.sf_data[s]), 1);
      mbar_init(smem_u32(&L.sf_empty[s]), 4);
      mbar_init(smem_u32(&L.sf_full[s]), 4);
    }
    for (int b = 0; b < kSwAccBufs; ++b) {
      mbar_init(smem_u32(&L.acc_full[b]), 1);
      mbar_init(smem_u32(&L.acc_empty[b]), 4);
    }
    mbar_init(smem_u32(L.drain), 1);
    *L.abort_flag = 0;
    fence_mbar_init();
  }
  // fed per m-tile by the L1 GEMM: no dependency wait (the producers wait
  // for each m-tile; the routing metadata was complete before L1 started)
  if (!(p.tile_done && p.tile_done_target > 0)) pdl_wait();
  for (int i = threadIdx.x; i <= p.G; i += blockDim.x) L.offsets[i] = p.offsets[i];
  for (int i = threadIdx.x; i < p.G; i += blockDim.x) L.counts[i] = p.counts[i];
  __syncthreads();
  if (warp == 0) {  // slot blocks of 64 real rows per group, exclusive prefix
    int carry = 0;
    for (int base = 0; base < p.G; base += 32) {
      const int g = base + lane;
      const int c = g < p.G ? (L.counts[g] + kSwN - 1) / kSwN : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      if (g < p.G) L.unit_off[g] = carry + incl - c;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      L.unit_off[p.G] = carry;
      prefetch_tmap(&p.tmap_w);
      prefetch_tmap(&p.tmap_x);
    }
  } else if (warp == 1) {
    tmem_alloc(smem_u32(L.tmem_slot), kSwTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *L.tmem_slot;
  const int total = L.unit_off[p.G] * p.n_wtiles;
  const int start = (int)blockIdx.x, step = (int)gridDim.x;
  if (warp == 0) {
    sw_producer<false>(p, L, total, start, step);
  } else if (warp == 1) {
    sw_mma_loop(p, L, total, start, step, tmem);
  } else if (warp == 2) {
    sw_producer<true>(p, L, total, start, step);
  } else if (warp >= kSwEpiWarp0 && warp < kSwSfWarp0) {
    sw_epilogue(p, L, total, start, step, tmem);
  } else if (warp >= kSwSfWarp0) {
    sw_sf_loop(p, L, total, start, step, tmem);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kSwTmemCols);
  }
}

}  // namespace

size_t gemm_swap_smem_bytes(int G) { return sw_smem_bytes(G); }

cudaError_t launch_gemm_swap(const SwapArgs& a, int num_sms, cudaStream_t s, bool pdl) {
  if (a.G < 1 || a.G > kSwMaxGroups || a.H % kSwM || a.K % 64) return cudaErrorInvalidValue;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(nvfp4_gemm_swap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sw_smem_bytes(kSwMaxGroups));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kSwThreads);
  cfg.dynamicSmemBytes = sw_smem_bytes(a.G);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? at : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, nvfp4_gemm_swap_kernel, a);
}

}  // namespace nvfp4
