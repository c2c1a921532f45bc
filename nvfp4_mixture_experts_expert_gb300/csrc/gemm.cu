// Block-scaled NVFP4 grouped GEMM for sm_103a on the 5th-generation tensor
// cores (tcgen05.mma kind::mxf4nvf4, 16-element UE4M3 block scales), with
// three fused epilogues:
//   kEpiBf16         D = alpha_g * acc as bf16 (grouped / dense linear)
//   kEpiSwigluQuant  MoE L1: h = bf16(silu(min(alpha*gate, gl)) * clamp(alpha*up, +-ul)),
//                    requantized to NVFP4 with the expert's L2 activation scale,
//                    nibbles and tile-layout scales written for the L2 GEMM
//                    (bridge.py page: fused SwiGLU epilogue; cutedsl page: gate
//                    clamped before SiLU)
//   kEpiCombine      MoE L2: Y[row] = bf16(w_row * alpha * acc) for real slot rows,
//                    in slot order; the token combine then sums each token's
//                    top_k rows (vllm page: scatter_add with zero-weight pads)
//   kEpiSwigluAmax   MoE calibration: per-expert amax of the bf16 SwiGLU output
//                    (vllm page: L2 global scale from the actual L1 output)
//
// Design (one CTA per SM, persistent over output tiles, warp-specialised):
//   warp 0   TMA producer: per K-stage of 256 elements, one 128x128-byte A box,
//            two 128x128-byte B boxes (SWIZZLE_128B) and the matching 512-byte
//            scale tiles (plain bulk copies), into a 4-deep shared-memory ring.
//   warp 1   TMEM allocator and MMA issuer: 4 MMAs of 128x256x64 per stage
//            into a 128-lane x 256-column FP32 accumulator in TMEM.
//   warp 10  scale copier: moves each stage's scale tiles into TMEM
//            (tcgen05.cp 32x128b.warpx4) ahead of the MMAs that read them.
//   warps 2-9 epilogue: each warp owns the 32 TMEM lanes of its quarter
//            (warp % 4), i.e. 32 output rows, and one half of the tile's
//            columns; it reads the accumulator with tcgen05.ld.
// A tile is 128 rows x 256 MMA columns.  For the SwiGLU epilogue the two B
// boxes are the gate rows [n0, n0+128) and the up rows [I+n0, I+n0+128) of the
// expert's W13, so gate and up of one output feature sit in the same TMEM lane
// 128 columns apart, and the 16-wide requantization blocks are in-register.
// Tiles are ordered m-tile major, n-tile minor (n-major is available); m-tiles
// map to groups through the 128-aligned group offsets read from device memory
// (no host sync).
// Every mbarrier wait is bounded (timeout -> device status word, abort, drain
// of copies/MMAs in flight, TMEM freed, return).
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "nvfp4_format.cuh"
#include "ptx.cuh"

namespace nvfp4 {

__device__ int g_device_status;

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK_BYTES = 128;  // 256 FP4 elements per stage
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK_BYTES;
constexpr int B_BYTES = BN * BK_BYTES;
constexpr int SFA_BYTES = 4 * 512;
constexpr int SFB_BYTES = 8 * 512;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int SF_COL0 = 256;         // scale columns start after the accumulator
constexpr int SF_COLS_PER_STAGE = 48;  // 4 x (4 SFA + 8 SFB)
constexpr int NUM_EPI_WARPS = 8;  // two per TMEM lane quarter, each owning half of the columns
constexpr int COPIER_WARP = 2 + NUM_EPI_WARPS;
constexpr int NUM_THREADS = 32 * (COPIER_WARP + 1);
constexpr int MAX_GROUPS = 1024;
static_assert(SF_COL0 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");
static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");

// Instruction descriptor: E2M1 x E2M1, UE4M3 scales, K-major A and B, dense K=64.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 7) << 27);
}

struct SmemLayout {
  uint8_t* stages;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* acc_full;
  uint64_t* acc_empty;
  uint64_t* drain;
  uint64_t* sf_full;     // [STAGES] scale tiles of a stage are in TMEM
  uint64_t* drain_cp;    // copier's own drain on abort
  uint32_t* tmem_slot;
  int* abort_flag;
  int* offsets;
};

__device__ __forceinline__ SmemLayout carve(uint8_t* raw) {
  SmemLayout L;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  L.stages = base;
  uint8_t* p = base + STAGES * STAGE_BYTES;
  L.full = reinterpret_cast<uint64_t*>(p);
  L.empty = L.full + STAGES;
  L.acc_full = L.empty + STAGES;
  L.acc_empty = L.acc_full + 1;
  L.drain = L.acc_empty + 1;
  L.sf_full = L.drain + 1;
  L.drain_cp = L.sf_full + STAGES;
  L.tmem_slot = reinterpret_cast<uint32_t*>(L.drain_cp + 1);
  L.abort_flag = reinterpret_cast<int*>(L.tmem_slot + 1);
  L.offsets = reinterpret_cast<int*>(L.abort_flag + 3);
  return L;
}

__device__ __forceinline__ int find_group(const int* off, int G, int row) {
  int lo = 0, hi = G;  // largest g in [0, G) with off[g] <= row
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= row) lo = mid; else hi = mid;
  }
  return lo;
}

// Tile index -> (m-tile, n-tile).  m-major keeps consecutive CTAs on one
// activation tile (and one expert's weights); n-major keeps every CTA on one
// output column slice, which bounds the live part of a scattered output.
__device__ __forceinline__ void decode_tile(int tile, int num_mtiles, int n_tiles, int n_major, int& mt, int& nt) {
  if (n_major) {
    nt = tile / num_mtiles;
    mt = tile - nt * num_mtiles;
  } else {
    mt = tile / n_tiles;
    nt = tile - mt * n_tiles;
  }
}

// ------------------------------------------------------------------ producer
__device__ void producer_loop(const GemmArgs& p, const SmemLayout& L, int total) {
  volatile int* abort = L.abort_flag;
  int issued_parity[STAGES];
#pragma unroll
  for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
  uint32_t stage = 0, phase = 0;
  const int kt = p.K / 64;  // scale tiles per 128-row band
  if (!p.debug_no_loads) {
    const int num_mtiles = L.offsets[p.G] / BM;
    for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
      int mt, nt;
      decode_tile(tile, num_mtiles, p.n_tiles, p.n_major, mt, nt);
      const int g = find_group(L.offsets, p.G, mt * BM);
      const int b_r0 = nt * p.b_tile_stride;
      const int b_r1 = b_r0 + p.b_second_offset;
      const int64_t b_row0 = (int64_t)g * p.b_rows_per_group + b_r0;
      const int64_t b_row1 = (int64_t)g * p.b_rows_per_group + b_r1;
      const uint8_t* sfa = p.sfa + (int64_t)mt * kt * 512;
      const uint8_t* sfb0 = p.sfb + g * p.sfb_group_bytes + (int64_t)(b_r0 >> 7) * kt * 512;
      const uint8_t* sfb1 = p.sfb + g * p.sfb_group_bytes + (int64_t)(b_r1 >> 7) * kt * 512;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        const int nmma = min(4, (p.K - kb * 256) / 64);
        if (!wait_bounded(smem_u32(&L.empty[stage]), phase ^ 1u, abort, p.status, p.timeout_ns)) break;
        uint8_t* st = L.stages + stage * STAGE_BYTES;
        const uint32_t bar = smem_u32(&L.full[stage]);
        mbar_arrive_expect_tx(bar, A_BYTES + B_BYTES + 3 * nmma * 512);
        tma_load_2d(smem_u32(st), &p.tmap_a, kb * BK_BYTES, mt * BM, bar);
        tma_load_2d(smem_u32(st + A_BYTES), &p.tmap_b, kb * BK_BYTES, (int32_t)b_row0, bar);
        tma_load_2d(smem_u32(st + A_BYTES + B_BYTES / 2), &p.tmap_b, kb * BK_BYTES, (int32_t)b_row1, bar);
        bulk_load(smem_u32(st + A_BYTES + B_BYTES), sfa + kb * 2048, nmma * 512, bar);
        bulk_load(smem_u32(st + A_BYTES + B_BYTES + SFA_BYTES), sfb0 + kb * 2048, nmma * 512, bar);
        bulk_load(smem_u32(st + A_BYTES + B_BYTES + SFA_BYTES + 2048), sfb1 + kb * 2048, nmma * 512, bar);
        issued_parity[stage] = (int)phase;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }
  if (*abort) {  // let copies already issued land before the CTA exits
#pragma unroll
    for (int s = 0; s < STAGES; ++s)
      if (issued_parity[s] >= 0) {
        volatile int no_abort = 0;
        wait_bounded(smem_u32(&L.full[s]), (uint32_t)issued_parity[s], &no_abort, nullptr, p.timeout_ns);
      }
  }
}

// ------------------------------------------------------------------ scale copier
// Copies each stage's scale tiles from shared memory into that stage's TMEM
// columns and signals sf_full[stage].  Issuing these copies from their own
// warp lets them overlap the MMA stream of the previous stages.  A stage's
// TMEM columns are rewritten only after its shared-memory slot was refilled,
// i.e. after the MMAs that read them committed.
__device__ void copier_loop(const GemmArgs& p, const SmemLayout& L, int total, uint32_t tmem) {
  volatile int* abort = L.abort_flag;
  uint32_t stage = 0, phase = 0;
  bool issued_any = false;
  for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
    for (int kb = 0; kb < p.num_kb; ++kb) {
      const int nmma = min(4, (p.K - kb * 256) / 64);
      if (!wait_bounded(smem_u32(&L.full[stage]), phase, abort, p.status, p.timeout_ns)) break;
      tc_fence_after();
      const uint32_t sfa_s = smem_u32(L.stages + stage * STAGE_BYTES) + A_BYTES + B_BYTES;
      const uint32_t sfb_s = sfa_s + SFA_BYTES;
      const uint32_t sf_col = tmem + SF_COL0 + stage * SF_COLS_PER_STAGE;
      for (int i = 0; i < nmma; ++i) {
        tc_cp_sf(sf_col + 4 * i, smem_desc(sfa_s + 512 * i, 0, 128, 0));
        tc_cp_sf(sf_col + 16 + 8 * i, smem_desc(sfb_s + 512 * i, 0, 128, 0));
        tc_cp_sf(sf_col + 16 + 8 * i + 4, smem_desc(sfb_s + 2048 + 512 * i, 0, 128, 0));
      }
      issued_any = true;
      tc_commit(smem_u32(&L.sf_full[stage]));
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (*abort && issued_any) {  // copies in flight must land before TMEM is freed
    tc_commit(smem_u32(L.drain_cp));
    volatile int no_abort = 0;
    wait_bounded(smem_u32(L.drain_cp), 0, &no_abort, nullptr, p.timeout_ns);
  }
}

// ------------------------------------------------------------------ MMA issuer
__device__ void mma_loop(const GemmArgs& p, const SmemLayout& L, int total, uint32_t tmem) {
  volatile int* abort = L.abort_flag;
  const uint32_t idesc = idesc_nvf4(BM, BN);
  uint32_t stage = 0, phase = 0, acc_phase = 0;
  bool issued_any = false;
  for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
    if (!wait_bounded(smem_u32(L.acc_empty), acc_phase ^ 1u, abort, p.status, p.timeout_ns)) break;
    tc_fence_after();
    bool ok = true;
    for (int kb = 0; kb < p.num_kb; ++kb) {
      const int nmma = min(4, (p.K - kb * 256) / 64);
      // sf_full[stage] implies full[stage]: the copier waited for the stage's data first
      if (!wait_bounded(smem_u32(&L.sf_full[stage]), phase, abort, p.status, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_s = smem_u32(L.stages + stage * STAGE_BYTES);
      const uint32_t b_s = a_s + A_BYTES;
      const uint32_t sf_col = tmem + SF_COL0 + stage * SF_COLS_PER_STAGE;
      for (int i = 0; i < nmma; ++i) {
        const uint64_t ad = smem_desc(a_s + 32 * i, 16, 1024, 2);
        const uint64_t bd = smem_desc(b_s + 32 * i, 16, 1024, 2);
        tc_mma_nvf4(tmem, ad, bd, idesc, sf_col + 4 * i, sf_col + 16 + 8 * i, (kb | i) != 0);
      }
      issued_any = true;
      tc_commit(smem_u32(&L.empty[stage]));
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
    tc_commit(smem_u32(L.acc_full));
    acc_phase ^= 1u;
  }
  if (*abort && issued_any) {  // every MMA / copy issued must finish before TMEM is freed
    tc_commit(smem_u32(L.drain));
    volatile int no_abort = 0;
    wait_bounded(smem_u32(L.drain), 0, &no_abort, nullptr, p.timeout_ns);
  }
}

// ------------------------------------------------------------------ epilogues
__device__ __forceinline__ float silu_clamped_product(float g, float u, float gl, float ul) {
  g = fminf(g, gl);
  u = fminf(fmaxf(u, -ul), ul);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Each epilogue thread first copies its 128 accumulator columns (one row)
// from TMEM into registers and releases the accumulator, so the MMAs of the
// next tile overlap all of the epilogue arithmetic and stores below.
template <int EPI>
__device__ void epilogue_loop(const GemmArgs& p, const SmemLayout& L, int total, uint32_t tmem) {
  volatile int* abort = L.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;        // TMEM lanes this warp may access
  const int half = (warp - 2) >> 2;    // which half of the tile's columns it owns
  const int row_in_tile = quarter * 32 + lane;
  const uint32_t t_base = tmem + ((uint32_t)(quarter * 32) << 16);
  const int num_mtiles = L.offsets[p.G] / BM;
  uint32_t acc_phase = 0;
  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    int ok = 1;
    if (lane == 0) ok = wait_bounded(smem_u32(L.acc_full), acc_phase, abort, p.status, p.timeout_ns);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    __syncwarp();
    tc_fence_after();
    // SwiGLU kinds: gate columns [half*64, +64) and up columns 128 + [half*64, +64);
    // other kinds: columns [half*128, +128).
    uint32_t v[4][32];
    if constexpr (EPI == kEpiSwigluQuant || EPI == kEpiSwigluAmax) {
      tmem_load_32(t_base + half * 64, v[0]);
      tmem_load_32(t_base + half * 64 + 32, v[1]);
      tmem_load_32(t_base + 128 + half * 64, v[2]);
      tmem_load_32(t_base + 128 + half * 64 + 32, v[3]);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_load_32(t_base + half * 128 + c * 32, v[c]);
    }
    tmem_load_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(L.acc_empty));
    acc_phase ^= 1u;

    int mt, nt;
    decode_tile(tile, num_mtiles, p.n_tiles, p.n_major, mt, nt);
    const int g = find_group(L.offsets, p.G, mt * BM);
    const int64_t row = (int64_t)mt * BM + row_in_tile;
    const float alpha = 1.0f / (p.a_gs[g] * p.b_gs[g]);

    if constexpr (EPI == kEpiBf16) {
      const int64_t i_local = row - L.offsets[g];
      const bool valid = p.counts ? i_local < p.counts[g] : true;
      if (valid) {
        uint16_t* drow = p.D + g * p.gstride_d + i_local * p.ldd + (int64_t)nt * BN + half * (BN / 2);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = pack_bf16x2(__uint_as_float(v[c][2 * j]) * alpha, __uint_as_float(v[c][2 * j + 1]) * alpha);
          if (p.d_vec32) {
            st_global_v8(drow + c * 32, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
            st_global_v8(drow + c * 32 + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(drow + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
      }
    } else if constexpr (EPI == kEpiSwigluQuant) {
      // output features [nt*128 + half*64, +64) of one row = 4 quantization blocks
      const float qgs = p.q_gs[g];
      uint32_t scales = 0;
      uint32_t words[8];
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        float xs[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int f = blk * 16 + i;
          const float h = silu_clamped_product(__uint_as_float(v[f >> 5][f & 31]) * alpha,
                                               __uint_as_float(v[2 + (f >> 5)][f & 31]) * alpha, p.gate_limit,
                                               p.up_limit);
          xs[i] = __fmul_rn(__uint_as_float(f32_to_bf16_rn(h) << 16), qgs);
        }
        uint32_t lo, hi;
        scales |= quant_block16(xs, lo, hi) << (8 * blk);
        words[blk * 2] = lo;
        words[blk * 2 + 1] = hi;
      }
      const int64_t f0 = (int64_t)nt * 128 + half * 64;  // first output feature of this thread
      // workspace rows: 32-byte aligned (I/2 and f0/2 are multiples of 32 bytes)
      st_global_v8(p.q_out + row * (p.I / 2) + f0 / 2, words[0], words[1], words[2], words[3], words[4], words[5],
                   words[6], words[7]);
      *reinterpret_cast<uint32_t*>(p.q_sf + sf_offset(row, f0 / 16, p.I / 16)) = scales;
    } else if constexpr (EPI == kEpiSwigluAmax) {
      // calibration: amax of the bf16 SwiGLU output of this row's features
      uint32_t m = 0;
#pragma unroll
      for (int f = 0; f < 64; ++f) {
        const float h = silu_clamped_product(__uint_as_float(v[f >> 5][f & 31]) * alpha,
                                             __uint_as_float(v[2 + (f >> 5)][f & 31]) * alpha, p.gate_limit,
                                             p.up_limit);
        m = max(m, f32_to_bf16_rn(h) & 0x7FFFu);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0 && m) atomicMax(&p.amax_bits[g], m << 16);
    } else {  // kEpiCombine: routing-weighted rows, stored in slot order for the token combine
      if (p.sorted_ids[row] >= 0) {
        const float wgt = p.row_w[row] * alpha;
        uint16_t* dst = p.y + row * p.H + (int64_t)nt * BN + half * (BN / 2);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = pack_bf16x2(__uint_as_float(v[c][2 * j]) * wgt, __uint_as_float(v[c][2 * j + 1]) * wgt);
          // workspace rows: 32-byte aligned (H is a multiple of 256)
          st_global_v8(dst + c * 32, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
          st_global_v8(dst + c * 32 + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
        }
      }
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1) nvfp4_gemm_kernel(const __grid_constant__ GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const SmemLayout L = carve(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&L.full[s]), 1);
      mbar_init(smem_u32(&L.empty[s]), 1);
    }
    mbar_init(smem_u32(L.acc_full), 1);
    mbar_init(smem_u32(L.acc_empty), NUM_EPI_WARPS);
    mbar_init(smem_u32(L.drain), 1);
    mbar_init(smem_u32(L.drain_cp), 1);
    for (int st = 0; st < STAGES; ++st) mbar_init(smem_u32(&L.sf_full[st]), 1);
    *L.abort_flag = 0;
    fence_mbar_init();
  }
  pdl_wait();  // everything below reads what earlier kernels wrote
  for (int i = threadIdx.x; i <= p.G; i += blockDim.x) L.offsets[i] = p.padded_offsets[i];
  if (warp == 1) {
    tmem_alloc(smem_u32(L.tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tmap_a);
    prefetch_tmap(&p.tmap_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *L.tmem_slot;
  const int total = (L.offsets[p.G] / BM) * p.n_tiles;

  if (warp == 0) {
    if (lane == 0) producer_loop(p, L, total);
  } else if (warp == 1) {
    if (lane == 0) mma_loop(p, L, total, tmem);
  } else if (warp < COPIER_WARP) {
    epilogue_loop<EPI>(p, L, total, tmem);
  } else {
    if (lane == 0) copier_loop(p, L, total, tmem);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int EPI>
cudaError_t launch_one(const GemmArgs& a, int grid, cudaStream_t s, bool pdl) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const size_t smem = gemm_smem_bytes(MAX_GROUPS);
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(nvfp4_gemm_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return launch_kernel(nvfp4_gemm_kernel<EPI>, dim3(grid), dim3(NUM_THREADS), gemm_smem_bytes(a.G), s, pdl, a);
}

}  // namespace

size_t gemm_smem_bytes(int G) {
  return 1024 + (size_t)STAGES * STAGE_BYTES + 8 * (3 * STAGES + 4) + 16 + 4 * (size_t)(G + 1) + 16;
}

cudaError_t launch_gemm(int kind, const GemmArgs& args, int grid, cudaStream_t s, bool pdl) {
  if (args.G < 1 || args.G > MAX_GROUPS) return cudaErrorInvalidValue;
  switch (kind) {
    case kEpiBf16: return launch_one<kEpiBf16>(args, grid, s, pdl);
    case kEpiSwigluQuant: return launch_one<kEpiSwigluQuant>(args, grid, s, pdl);
    case kEpiCombine: return launch_one<kEpiCombine>(args, grid, s, pdl);
    case kEpiSwigluAmax: return launch_one<kEpiSwigluAmax>(args, grid, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_status_ptr(int** ptr) { return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_device_status); }

cudaError_t gemm_read_status(int* out, int reset) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (reset) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
  }
  return e;
}

}  // namespace nvfp4
