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
//                    (vllm page: L2 global scale from the actual L1 output);
//                    optionally stores that output, as bf16 or as FP8 blocks
//                    (forward with L2 scales taken from the batch, the FP8/BF16
//                    L1-output option)
//
// Design (persistent over output tiles, warp-specialised, one CTA per SM):
//   warp 0   operand producer: per K-stage of 256 elements, the A box (128
//            rows x 128 bytes) and the B box(es) (SWIZZLE_128B) by TMA, into
//            an operand ring.
//   warp 2   scale producer: the stage's 512-byte scale tiles (plain bulk
//            copies) into a scale ring of their own.
//   warp 1   TMEM allocator and MMA issuer: 4 MMAs of K=64 per stage into a
//            128-lane x 256-column FP32 accumulator in TMEM, issued by one
//            elected lane from a warp-uniform loop.
//   warps 4-11 epilogue: each warp owns the 32 TMEM lanes of its quarter
//            (warp % 4), i.e. 32 output rows, and one half of the tile's
//            columns; it reads the accumulator with tcgen05.ld.
//   warps 12-15 scale staging: shared memory -> TMEM scale columns with
//            tcgen05.st, one warp per lane quarter (see sf_loop).
//   Registers are re-balanced per warpgroup with setmaxnreg (the epilogue
//   holds a 128-column accumulator row per thread).
// Two variants:
//   single   one CTA computes a 128 x 256 tile; 4-stage operand ring of 48 KB
//            stages, 4-slot scale ring of 6 KB.
//   pair     a cluster of two CTAs on two SMs computes a 256 x 256 tile with
//            tcgen05 cta_group::2: each CTA holds 128 rows of A and one
//            128-row half of the B tile (the gate or up half for SwiGLU) plus
//            all of the stage's scale tiles, so an SM reads 8 KB of operands
//            per 128x256x64 MMA instead of 12 KB; 5-stage operand ring of
//            32 KB stages, 5-slot scale ring of 6 KB.
//            The leader CTA (rank 0) issues the MMAs; its commits are
//            multicast to both CTAs' barriers.  The peer's scale warps arrive
//            on the leader's sf_full (its scales are in its TMEM), its warp 3
//            relays the arrival of its operands to the leader's peer_full, and
//            its epilogue warps release the accumulator on the leader's
//            barrier.  An expert's m-tiles are paired in order;
//            an odd last tile is paired with a copy of itself whose rows the
//            peer does not store.
// A tile is 128 (per CTA) rows x 256 MMA columns.  For the SwiGLU epilogue the
// two B boxes are the gate rows [n0, n0+128) and the up rows [I+n0, I+n0+128)
// of the expert's W13, so gate and up of one output feature sit in the same
// TMEM lane 128 columns apart, and the 16-wide requantization blocks are
// in-register.  Work units (m-tiles or m-tile pairs) are ordered unit major,
// n-tile minor (n-major is available); units map to groups through the
// 128-aligned group offsets read from device memory (no host sync).
// What bounds this pipeline was measured (a scratch copy with per-role
// timelines, and the bare MMA stream of nvfp4_debug_mma_rate with each
// pipeline activity added in turn): one thread issues every MMA and the
// tensor pipe queues few, so the issuing loop is warp-uniform and short; a
// stage's chain of hand-offs (slot freed by the MMA commit -> copies ->
// scale staging -> MMA) must fit in the ring, so the scale warps stage from a
// ring of their own as soon as the TMEM columns are free, and the waits on
// that chain poll instead of suspending.
// Every mbarrier wait is bounded (timeout -> device status word, abort, drain
// of copies/MMAs in flight, TMEM freed, return); in the pair variant every
// CTA runs to the final cluster barrier before the collective TMEM release,
// and each producer first waits for the leader's last multicast releases.
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
constexpr int A_BYTES = BM * BK_BYTES;
constexpr int SFA_BYTES = 4 * 512;
constexpr int SFB_BYTES = 8 * 512;
constexpr int TMEM_COLS = 512;
constexpr int SF_COL0 = 256;         // scale columns start after the accumulator
constexpr int SF_COLS_PER_STAGE = 48;  // 4 x (4 SFA + 8 SFB)
// Warp roles, by warpgroup (setmaxnreg re-balances registers per warpgroup):
//   WG0  warp 0 operand producer, warp 1 TMEM allocator + MMA issuer, warp 2
//        scale producer, warp 3 (pair variant, peer CTA) operand-arrival relay
//   WG1-2 warps 4-11 epilogue: two per TMEM lane quarter, each owning half of the columns
//   WG3  warps 12-15 scale staging: one per TMEM lane quarter
constexpr int EPI_WARP0 = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int SF_WARP0 = EPI_WARP0 + NUM_EPI_WARPS;
constexpr int NUM_THREADS = 32 * (SF_WARP0 + 4);
constexpr int REGS_LAUNCH = 128;  // per thread at launch (the kernel's register allocation)
constexpr int REGS_SMALL = 72;    // WG0 and WG3 after setmaxnreg.dec
constexpr int REGS_EPI = 184;     // WG1 and WG2 after setmaxnreg.inc
static_assert(128 * (2 * REGS_SMALL + 2 * REGS_EPI) <= NUM_THREADS * REGS_LAUNCH,
              "the register split must fit the launch allocation");
constexpr int MAX_GROUPS = 1024;
constexpr int MAX_GROUPS_PAIR = 256;        // the pair variant's shared memory also holds the staging buffers
constexpr int EPI_STAGE_BYTES = 32 * 128;   // per epilogue warp (pair): 32 rows x 64 bf16 columns

template <bool PAIR>
struct Cfg {
  static constexpr int STAGES = PAIR ? 5 : 4;
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK_BYTES;  // B rows this CTA loads per stage
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // operand ring slot (A and this CTA's B rows)
  static constexpr int SF_STAGES = STAGES;                // scale ring slots (its own ring, see sf_loop)
  static constexpr int SF_SLOT_BYTES = SFA_BYTES + SFB_BYTES;
  static constexpr int EPI_BYTES = PAIR ? NUM_EPI_WARPS * EPI_STAGE_BYTES : 0;
  static_assert(SF_COL0 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
};

// Instruction descriptor: E2M1 x E2M1, UE4M3 scales, K-major A and B, dense K=64.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 7) << 27);
}

struct SmemLayout {
  uint8_t* stages;
  uint8_t* sf_slots;   // scale ring: SF_STAGES slots of the stage's 512-byte scale tiles
  uint8_t* epi_stage;  // pair variant: per-warp output staging for coalesced stores
  uint64_t* full;
  uint64_t* empty;
  uint64_t* acc_full;
  uint64_t* acc_empty;
  uint64_t* drain;
  uint64_t* peer_full;  // [STAGES] pair variant, leader: the peer CTA's operands of a stage have landed
  uint64_t* sf_data;     // [SF_STAGES] a scale slot has landed in shared memory
  uint64_t* sf_empty;    // [SF_STAGES] the scale warps have read a scale slot
  uint64_t* sf_full;     // [STAGES] scale tiles of a stage are in TMEM
  uint32_t* tmem_slot;
  int* abort_flag;
  int* stored;    // [2] L1 -> L2 hand-off: epilogue warps done storing the tile of that parity
  int* offsets;   // [G+1] padded row offsets
  int* unit_off;  // [G+1] first work unit (m-tile or m-tile pair) of each group
};

template <bool PAIR>
__device__ __forceinline__ SmemLayout carve(uint8_t* raw, int G) {
  using C = Cfg<PAIR>;
  SmemLayout L;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  L.stages = base;
  L.sf_slots = base + C::STAGES * C::STAGE_BYTES;
  L.epi_stage = L.sf_slots + C::SF_STAGES * C::SF_SLOT_BYTES;
  uint8_t* p = L.epi_stage + C::EPI_BYTES;
  L.full = reinterpret_cast<uint64_t*>(p);
  L.empty = L.full + C::STAGES;
  L.sf_data = L.empty + C::STAGES;
  L.sf_empty = L.sf_data + C::SF_STAGES;
  L.sf_full = L.sf_empty + C::SF_STAGES;
  L.acc_full = L.sf_full + C::STAGES;
  L.acc_empty = L.acc_full + 1;
  L.drain = L.acc_empty + 1;
  L.peer_full = L.drain + 1;
  L.tmem_slot = reinterpret_cast<uint32_t*>(L.peer_full + C::STAGES);
  L.abort_flag = reinterpret_cast<int*>(L.tmem_slot + 1);
  L.stored = L.abort_flag + 1;
  L.offsets = reinterpret_cast<int*>(L.abort_flag + 3);
  L.unit_off = L.offsets + G + 1;
  return L;
}

template <bool PAIR>
constexpr size_t smem_bytes_for(int G) {
  return 1024 + (size_t)Cfg<PAIR>::STAGES * Cfg<PAIR>::STAGE_BYTES +
         (size_t)Cfg<PAIR>::SF_STAGES * Cfg<PAIR>::SF_SLOT_BYTES + Cfg<PAIR>::EPI_BYTES +
         8 * (4 * Cfg<PAIR>::STAGES + 2 * Cfg<PAIR>::SF_STAGES + 4) + 16 + 8 * (size_t)(G + 1) + 16;
}

// Debug timeline (nvfp4_debug_gemm_trace): SM clock (%clock64) stamps of
// one CTA's roles (trace_cta), per ring stage g (count of stages since the
// kernel started) and per tile t.
//   stage words: 0 producer slot free, 1 producer copies issued, 2 scale warp
//     saw the data, 3 scale warp staged, 4 MMA starts waiting, 5 MMA may issue,
//     6 MMA instructions issued, 7 stage committed
//   tile words:  0 MMA waits for the accumulator, 1 accumulator free, 2 epilogue
//     saw it full, 3 epilogue released it, 4 epilogue finished the tile
// Compiled in only with -DNVFP4_GEMM_TRACE: even switched off at run time the
// checks cost the hot loops about 15 % (measured on the prefill L1 GEMM).
#ifdef NVFP4_GEMM_TRACE
__device__ __forceinline__ void trace_stage(const GemmArgs& p, int g, int ev) {
  if (p.trace && (int)blockIdx.x == p.trace_cta && g < p.trace_stages) p.trace[(int64_t)g * 8 + ev] = clock64();
}
__device__ __forceinline__ void trace_tile(const GemmArgs& p, int t, int ev) {
  if (p.trace && (int)blockIdx.x == p.trace_cta && t < p.trace_tiles)
    p.trace[(int64_t)p.trace_stages * 8 + (int64_t)t * 8 + ev] = clock64();
}
constexpr bool kTraceBuild = true;
#else
__device__ __forceinline__ void trace_stage(const GemmArgs&, int, int) {}
__device__ __forceinline__ void trace_tile(const GemmArgs&, int, int) {}
constexpr bool kTraceBuild = false;
#endif

__device__ __forceinline__ int find_group(const int* off, int G, int row) {
  int lo = 0, hi = G;  // largest g in [0, G) with off[g] <= row
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= row) lo = mid; else hi = mid;
  }
  return lo;
}

// Work item -> (group, m-tile of this CTA, n-tile).  Unit-major order keeps
// consecutive CTAs on one activation tile (and one expert's weights);
// n-major keeps every CTA on one output column slice.  In the pair variant a
// unit is two consecutive m-tiles of one group (rank 0 takes the first); the
// second of an odd group's last pair does not exist (valid = false) and that
// CTA reloads the first tile so every copy stays inside the operands.
struct Work {
  int g, mt, nt;
  bool valid;
};

template <bool PAIR>
__device__ __forceinline__ Work decode_work(const SmemLayout& L, const GemmArgs& p, int it, uint32_t rank) {
  const int nu = L.unit_off[p.G];
  int u, nt;
  if (p.n_major) {
    nt = it / nu;
    u = it - nt * nu;
  } else {
    u = it / p.n_tiles;
    nt = it - u * p.n_tiles;
  }
  Work w;
  w.g = find_group(L.unit_off, p.G, u);
  w.nt = nt;
  const int t0 = L.offsets[w.g] / BM, k = u - L.unit_off[w.g];
  if constexpr (PAIR) {
    const int mt = t0 + 2 * k + (int)rank;
    w.valid = mt < L.offsets[w.g + 1] / BM;
    w.mt = w.valid ? mt : mt - 1;
  } else {
    w.mt = t0 + k;
    w.valid = true;
  }
  return w;
}

// Bounded wait (one lane) until a counter another kernel increments reaches
// target; same give-up rules as the barrier waits.
__device__ __forceinline__ bool wait_count_bounded(const int* counter, int target, volatile int* abort, int* status,
                                                   uint64_t timeout_ns) {
  if (ld_acquire_gpu(counter) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i) {
      __nanosleep(100);
      if (ld_acquire_gpu(counter) >= target) return true;
    }
    if (*abort) return false;
    if (global_timer_ns() - t0 > timeout_ns) {
      *abort = 1;
      if (status) atomicExch(status, 6 /* NVFP4_ERR_DEVICE_TIMEOUT */);
      return false;
    }
  }
}

// ------------------------------------------------------------------ producers
// Work items it = start, start + step, ... (step = CTAs, or CTA pairs).
// Two producer warps: SCALES == false copies a stage's A and B boxes with TMA
// into the operand ring once the MMAs that read the slot have committed
// (empty); SCALES == true copies the stage's 512-byte scale tiles with bulk
// copies into the scale ring once the scale warps have read the slot
// (sf_empty), so it runs ahead.  Each runs on its whole warp: addresses are
// warp-uniform and one elected lane issues; lane 0 polls the barriers.  The
// parity each slot was last issued with is kept in registers (a bitmask),
// for the drain after an abort.
template <bool PAIR, bool SCALES>
__device__ void producer_loop(const GemmArgs& p, const SmemLayout& L, int total, int start, int step,
                              uint32_t rank) {
  using C = Cfg<PAIR>;
  constexpr int kSlots = SCALES ? C::SF_STAGES : C::STAGES;
  constexpr uint32_t kSlotBytes = SCALES ? C::SF_SLOT_BYTES : C::STAGE_BYTES;
  volatile int* abort = L.abort_flag;
  const int lane = threadIdx.x & 31;
  const bool leader = elect_one();
  uint32_t issued = 0, issued_parity = 0;  // bit s: slot s issued at least once / with parity 1
  uint32_t stage = 0, phase = 0;
  int ok = 1;
  int gstage = 0;  // stages issued so far (debug timeline)
  const bool tr = kTraceBuild && !SCALES && leader;
  const int kt = p.K / 64;  // scale tiles per 128-row band
  const uint32_t empty0 = smem_u32(SCALES ? L.sf_empty : L.empty);
  const uint32_t done0 = smem_u32(SCALES ? L.sf_data : L.full);
  const uint32_t slot0 = smem_u32(SCALES ? L.sf_slots : L.stages);
  const bool per_tile = p.tile_done && p.tile_done_target > 0;  // L2 fed per m-tile by L1
  int ready_mt = -1;
  if (!p.debug_no_loads) {
    for (int it = start; it < total && ok && !*abort; it += step) {
      const Work w = decode_work<PAIR>(L, p, it, rank);
      if (per_tile && w.mt != ready_mt) {
        if (lane == 0) ok = wait_count_bounded(p.tile_done + w.mt, p.tile_done_target, abort, p.status, p.timeout_ns);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        (void)ld_acquire_gpu(p.tile_done + w.mt);  // every lane, then the copies may read the m-tile
        fence_proxy_async_global();
        ready_mt = w.mt;
      }
      const int b_r0 = w.nt * p.b_tile_stride;
      const int b_r1 = b_r0 + p.b_second_offset;
      const int32_t a_row = w.mt * BM;
      const int32_t b_row0 = w.g * p.b_rows_per_group + b_r0;
      const int32_t b_row1 = w.g * p.b_rows_per_group + b_r1;
      const uint8_t* sfa = p.sfa + (int64_t)w.mt * kt * 512;
      const uint8_t* sfb0 = p.sfb + w.g * p.sfb_group_bytes + (int64_t)(b_r0 >> 7) * kt * 512;
      const int sf_t1 = p.sfb_tiles > 0 && (b_r1 >> 7) >= p.sfb_tiles ? (b_r0 >> 7) : (b_r1 >> 7);
      const uint8_t* sfb1 = p.sfb + w.g * p.sfb_group_bytes + (int64_t)sf_t1 * kt * 512;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (lane == 0) ok = wait_bounded_spin(empty0 + 8 * stage, phase ^ 1u, abort, p.status, p.timeout_ns);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (tr) trace_stage(p, gstage, 0);
        const uint32_t st = slot0 + stage * kSlotBytes;
        const uint32_t bar = done0 + 8 * stage;
        if (leader) {
          if constexpr (SCALES) {
            const uint32_t bytes = (uint32_t)min(4, (p.K - kb * 256) / 64) * 512;
            mbar_arrive_expect_tx(bar, 3 * bytes);
            bulk_load(st, sfa + kb * 2048, bytes, bar);
            bulk_load(st + SFA_BYTES, sfb0 + kb * 2048, bytes, bar);
            bulk_load(st + SFA_BYTES + 2048, sfb1 + kb * 2048, bytes, bar);
          } else {
            mbar_arrive_expect_tx(bar, A_BYTES + C::B_BYTES);
            tma_load_2d(st, &p.tmap_a, kb * BK_BYTES, a_row, bar);
            if constexpr (PAIR) {  // this CTA's half of the B tile
              tma_load_2d(st + A_BYTES, &p.tmap_b, kb * BK_BYTES, rank ? b_row1 : b_row0, bar);
            } else {
              tma_load_2d(st + A_BYTES, &p.tmap_b, kb * BK_BYTES, b_row0, bar);
              tma_load_2d(st + A_BYTES + C::B_BYTES / 2, &p.tmap_b, kb * BK_BYTES, b_row1, bar);
            }
          }
        }
        __syncwarp();
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (tr) trace_stage(p, gstage, 1);
        ++gstage;
        if (++stage == kSlots) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }
  if (lane == 0) {
    if (*abort || !ok) {  // let copies already issued land before the CTA exits
#pragma unroll
      for (int s = 0; s < kSlots; ++s)
        if (issued & (1u << s)) {
          volatile int no_abort = 0;
          wait_bounded(done0 + 8 * s, (issued_parity >> s) & 1u, &no_abort, nullptr, p.timeout_ns);
        }
    } else if constexpr (PAIR && !SCALES) {
      // the leader's last multicast releases land in this CTA before it may exit
      for (int i = 0; i < C::STAGES; ++i) {
        if (!wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort, p.status, p.timeout_ns)) break;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ scale staging
// Warps 12-15 (one per TMEM lane quarter) move each stage's scale tiles from
// shared memory into that stage's TMEM columns with tcgen05.st: lane l of the
// warp for quarter q writes 16-byte line l of every 512-byte tile into TMEM
// lane 32q + l, 4 columns per tile -- the layout the block-scaled MMA reads
// (each quarter holds the same 32 lines; SFB tiles cover all N rows).  Two
// store instructions per warp per stage replace 12 tcgen05.cp copies, which
// would occupy the tensor pipe ahead of the MMAs.
// The scale tiles come through their own shared-memory ring: a warp reads a
// slot into registers and frees it (sf_empty), so the scale producer runs
// ahead.  A stage's TMEM columns are rewritten once the MMAs that read them
// have committed (empty[stage]); the stores (a few hundred cycles) run while
// the stage's operands are still in flight.  sf_full[stage] tells the MMA
// issuer the scales are in TMEM; it counts the 4 warps (8 in the pair variant:
// the peer's warps arrive on the leader's barrier).  The operands of a stage
// are on the full barrier of each CTA; the leader sees the peer's through
// peer_full, arrived on by the peer's relay warp (relay_loop).
template <bool PAIR>
__device__ void sf_loop(const GemmArgs& p, const SmemLayout& L, int total, int start, int step, uint32_t tmem,
                        uint32_t rank) {
  using C = Cfg<PAIR>;
  volatile int* abort = L.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  uint32_t stage = 0, phase = 0;  // operand / TMEM stage
  uint32_t slot = 0, sphase = 0;  // scale ring slot
  int gstage = 0;
  const bool tracer = kTraceBuild && warp == SF_WARP0 && lane == 0;
  for (int it = start; it < total; it += step) {
    int ok = 1;
    for (int kb = 0; kb < p.num_kb; ++kb) {
      if (lane == 0) ok = wait_bounded_spin(smem_u32(&L.sf_data[slot]), sphase, abort, p.status, p.timeout_ns);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      // columns of a stage: SFA of K-steps 0-3 (4 each), then per K-step the
      // SFB tiles of B rows 0-127 and 128-255 (4 each); unused K-steps of a
      // partial last stage carry stale scales that no MMA reads
      const uint8_t* sf = L.sf_slots + slot * C::SF_SLOT_BYTES + 16 * lane;
      uint32_t r[48];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 a = *reinterpret_cast<const uint4*>(sf + 512 * i);
        const uint4 b0 = *reinterpret_cast<const uint4*>(sf + SFA_BYTES + 512 * i);
        const uint4 b1 = *reinterpret_cast<const uint4*>(sf + SFA_BYTES + 2048 + 512 * i);
        r[4 * i + 0] = a.x, r[4 * i + 1] = a.y, r[4 * i + 2] = a.z, r[4 * i + 3] = a.w;
        r[16 + 8 * i + 0] = b0.x, r[16 + 8 * i + 1] = b0.y, r[16 + 8 * i + 2] = b0.z, r[16 + 8 * i + 3] = b0.w;
        r[16 + 8 * i + 4] = b1.x, r[16 + 8 * i + 5] = b1.y, r[16 + 8 * i + 6] = b1.z, r[16 + 8 * i + 7] = b1.w;
      }
      if (tracer) trace_stage(p, gstage, 2);
      // the stage's TMEM scale columns are free once its previous MMAs committed
      if (lane == 0) ok = wait_bounded_spin(smem_u32(&L.empty[stage]), phase ^ 1u, abort, p.status, p.timeout_ns);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      tc_fence_after();
      const uint32_t col = t_lane + SF_COL0 + stage * SF_COLS_PER_STAGE;
      tmem_store_32(col, r);
      tmem_store_16_hi(col + 32, r);
      __syncwarp();  // every lane's reads of the slot are done (its registers went to the stores)
      if (lane == 0) mbar_arrive(smem_u32(&L.sf_empty[slot]));
      tmem_store_wait();
      tc_fence_before();
      if (lane == 0) {
        if (PAIR && rank) mbar_arrive_remote(mapa_shared(smem_u32(&L.sf_full[stage]), 0));
        else mbar_arrive(smem_u32(&L.sf_full[stage]));
      }
      if (tracer) trace_stage(p, gstage, 3);
      ++gstage;
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
      if (++slot == C::SF_STAGES) {
        slot = 0;
        sphase ^= 1u;
      }
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) break;
  }
}

// ------------------------------------------------------------------ MMA issuer
// One thread issues every MMA of the CTA (or CTA pair), and the tensor pipe
// queues few of them: a cycle spent elsewhere is a cycle the pipe may idle.
// The loop therefore runs on the whole warp, so that every operand (slot
// descriptors built once -- a slot adds STAGE_BYTES, a K-step 32 bytes, in
// the 16-byte units of the start-address field -- TMEM addresses, stage and
// phase) is warp-uniform, and one elected lane issues the MMAs and commits
// (a commit tracks the MMAs of the thread that issues it).  A full stage's 4
// MMAs are unrolled, and the next stage's barriers are tested without
// blocking while this stage's MMAs issue; lane 0 polls when they were not
// ready.  A stage may issue once its scales are in TMEM (sf_full) and its
// operands have landed (full; in the pair variant also the peer's, relayed
// to peer_full).
template <bool PAIR>
__device__ __forceinline__ void issue_stage(uint32_t tmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t sf_col,
                                            uint32_t first_acc, int nmma, bool full, uint32_t next_bar,
                                            uint32_t next_bar2, uint32_t next_bar3, uint32_t next_parity,
                                            uint32_t& next_ready) {
  uint32_t r1 = 1u, r2 = 1u, r3 = 1u;
  if (full) {
    if constexpr (PAIR) {
      tc_mma_nvf4_pair(tmem, ad, bd, idesc, sf_col, sf_col + 16, first_acc);
      if (next_bar) r1 = mbar_test_wait(next_bar, next_parity);
      tc_mma_nvf4_pair(tmem, ad + 2, bd + 2, idesc, sf_col + 4, sf_col + 24, 1u);
      if (next_bar2) r2 = mbar_test_wait(next_bar2, next_parity);
      tc_mma_nvf4_pair(tmem, ad + 4, bd + 4, idesc, sf_col + 8, sf_col + 32, 1u);
      if (next_bar3) r3 = mbar_test_wait(next_bar3, next_parity);
      tc_mma_nvf4_pair(tmem, ad + 6, bd + 6, idesc, sf_col + 12, sf_col + 40, 1u);
    } else {
      tc_mma_nvf4(tmem, ad, bd, idesc, sf_col, sf_col + 16, first_acc);
      if (next_bar) r1 = mbar_test_wait(next_bar, next_parity);
      tc_mma_nvf4(tmem, ad + 2, bd + 2, idesc, sf_col + 4, sf_col + 24, 1u);
      if (next_bar2) r2 = mbar_test_wait(next_bar2, next_parity);
      tc_mma_nvf4(tmem, ad + 4, bd + 4, idesc, sf_col + 8, sf_col + 32, 1u);
      tc_mma_nvf4(tmem, ad + 6, bd + 6, idesc, sf_col + 12, sf_col + 40, 1u);
    }
  } else {
    for (int i = 0; i < nmma; ++i) {
      const uint32_t acc = i ? 1u : first_acc;
      if constexpr (PAIR)
        tc_mma_nvf4_pair(tmem, ad + 2 * i, bd + 2 * i, idesc, sf_col + 4 * i, sf_col + 16 + 8 * i, acc);
      else
        tc_mma_nvf4(tmem, ad + 2 * i, bd + 2 * i, idesc, sf_col + 4 * i, sf_col + 16 + 8 * i, acc);
    }
    if (next_bar) r1 = mbar_test_wait(next_bar, next_parity);
    if (next_bar2) r2 = mbar_test_wait(next_bar2, next_parity);
    if (next_bar3) r3 = mbar_test_wait(next_bar3, next_parity);
  }
  next_ready = r1 & r2 & r3;
}

template <bool PAIR>
__device__ void mma_loop(const GemmArgs& p, const SmemLayout& L, int total, int start, int step, uint32_t tmem) {
  using C = Cfg<PAIR>;
  volatile int* abort = L.abort_flag;
  const int lane = threadIdx.x & 31;
  const bool leader = elect_one();
  const int leader_lane = __ffs(__ballot_sync(0xffffffffu, leader)) - 1;
  const uint32_t idesc = idesc_nvf4(PAIR ? 2 * BM : BM, BN);
  const uint64_t a_desc0 = smem_desc(smem_u32(L.stages), 16, 1024, 2);
  const uint64_t b_desc0 = smem_desc(smem_u32(L.stages) + A_BYTES, 16, 1024, 2);
  constexpr uint64_t kSlotDesc = C::STAGE_BYTES >> 4;
  const uint32_t sf_full0 = smem_u32(L.sf_full), empty0 = smem_u32(L.empty), full0 = smem_u32(L.full);
  const uint32_t peer0 = smem_u32(L.peer_full);  // pair variant: the peer's operands (relayed)
  const int num_kb = p.num_kb;
  const bool tr = kTraceBuild && p.trace != nullptr && (int)blockIdx.x == p.trace_cta && leader;
  uint32_t stage = 0, phase = 0, acc_phase = 0;
  bool issued_any = false;
  int gstage = 0, tile = 0;
  int ok = 1;
  for (int it = start; it < total && ok && !*abort; it += step, ++tile) {
    if (tr) trace_tile(p, tile, 0);
    if (lane == 0) ok = wait_bounded_spin(smem_u32(L.acc_empty), acc_phase ^ 1u, abort, p.status, p.timeout_ns);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    if (tr) trace_tile(p, tile, 1);
    if (lane == 0) {
      ok = wait_bounded_spin(sf_full0 + 8 * stage, phase, abort, p.status, p.timeout_ns);
      if (ok) ok = wait_bounded_spin(full0 + 8 * stage, phase, abort, p.status, p.timeout_ns);
      if (PAIR && ok) ok = wait_bounded_spin(peer0 + 8 * stage, phase, abort, p.status, p.timeout_ns);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    for (int kb = 0; ok && kb < num_kb; ++kb) {
      if (tr) trace_stage(p, gstage, 5);
      tc_fence_after();
      const int rem = p.K - kb * 256;
      const uint32_t next_stage = stage + 1 == C::STAGES ? 0u : stage + 1;
      const uint32_t next_phase = stage + 1 == C::STAGES ? phase ^ 1u : phase;
      const bool more = kb + 1 < num_kb;
      uint32_t next_ready = 1;
      if (leader) {
        issue_stage<PAIR>(tmem, a_desc0 + stage * kSlotDesc, b_desc0 + stage * kSlotDesc, idesc,
                          tmem + SF_COL0 + stage * SF_COLS_PER_STAGE, kb != 0, min(4, rem / 64), rem >= 256,
                          more ? sf_full0 + 8 * next_stage : 0u, more ? full0 + 8 * next_stage : 0u,
                          more && PAIR ? peer0 + 8 * next_stage : 0u,
                          next_phase, next_ready);
        if (tr) trace_stage(p, gstage, 6);
        if constexpr (PAIR) tc_commit_pair_mc(empty0 + 8 * stage, 3);
        else tc_commit(empty0 + 8 * stage);
        if (tr) trace_stage(p, gstage, 7);
      }
      next_ready = __shfl_sync(0xffffffffu, next_ready, leader_lane);
      issued_any = true;
      ++gstage;
      stage = next_stage;
      phase = next_phase;
      if (!next_ready) {
        if (tr) trace_stage(p, gstage, 4);
        if (lane == 0) {
          ok = wait_bounded_spin(sf_full0 + 8 * stage, phase, abort, p.status, p.timeout_ns);
          if (ok) ok = wait_bounded_spin(full0 + 8 * stage, phase, abort, p.status, p.timeout_ns);
          if (PAIR && ok) ok = wait_bounded_spin(peer0 + 8 * stage, phase, abort, p.status, p.timeout_ns);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
    if (!ok) break;
    if (leader) {
      if constexpr (PAIR) tc_commit_pair_mc(smem_u32(L.acc_full), 3);
      else tc_commit(smem_u32(L.acc_full));
    }
    __syncwarp();
    acc_phase ^= 1u;
  }
  if (*abort && issued_any) {  // every MMA / copy issued must finish before TMEM is freed
    if (leader) {
      if constexpr (PAIR) tc_commit_pair(smem_u32(L.drain));
      else tc_commit(smem_u32(L.drain));
    }
    __syncwarp();
    if (lane == 0) {
      volatile int no_abort = 0;
      wait_bounded(smem_u32(L.drain), 0, &no_abort, nullptr, p.timeout_ns);
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ epilogues
// bf16 pair of two accumulator words each multiplied by s (one packed multiply).
__device__ __forceinline__ uint32_t scaled_bf16x2(uint32_t a, uint32_t b, uint64_t s2) {
  float x0, x1;
  f2_unpack(f2_mul(f2_pack(__uint_as_float(a), __uint_as_float(b)), s2), x0, x1);
  return pack_bf16x2(x0, x1);
}

__device__ __forceinline__ float tanh_approx(float x) {
  float r;
  asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// SiLU(min(g, gl)) * clamp(u, -ul, ul) = g * sigmoid(g) * u with
// sigmoid(g) = (1 + tanh(g / 2)) / 2: one hardware tanh approximation
// (relative error about 2^-11, well below the bf16 rounding of h) instead of
// an exponential and a reciprocal.
__device__ __forceinline__ float silu_clamped_product(float g, float u, float gl, float ul) {
  g = fminf(g, gl);
  u = fminf(fmaxf(u, -ul), ul);
  const float sig = __fmaf_rn(0.5f, tanh_approx(0.5f * g), 0.5f);
  return g * sig * u;
}

// The same for two features at once (packed pairs, each half rounded exactly
// as the scalar form: bit-identical results with fewer instructions).
__device__ __forceinline__ void silu_clamped_product2(float g0, float g1, float u0, float u1, float gl, float ul,
                                                      float& h0, float& h1) {
  g0 = fminf(g0, gl);
  g1 = fminf(g1, gl);
  u0 = fminf(fmaxf(u0, -ul), ul);
  u1 = fminf(fmaxf(u1, -ul), ul);
  const uint64_t g2 = f2_pack(g0, g1);
  float t0, t1;
  f2_unpack(f2_mul(g2, f2_pack(0.5f, 0.5f)), t0, t1);
  const uint64_t sig2 = f2_fma(f2_pack(0.5f, 0.5f), f2_pack(tanh_approx(t0), tanh_approx(t1)), f2_pack(0.5f, 0.5f));
  f2_unpack(f2_mul(f2_mul(g2, sig2), f2_pack(u0, u1)), h0, h1);
}

// Each epilogue thread first copies its 128 accumulator columns (one row)
// from TMEM into registers and releases the accumulator, so the MMAs of the
// next tile overlap all of the epilogue arithmetic and stores below.
template <int EPI, bool PAIR>
__device__ void epilogue_loop(const GemmArgs& p, const SmemLayout& L, int total, int start, int step, uint32_t tmem,
                              uint32_t rank) {
  volatile int* abort = L.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;        // TMEM lanes this warp may access
  const int half = (warp - EPI_WARP0) >> 2;  // which half of the tile's columns it owns
  const int row_in_tile = quarter * 32 + lane;
  const uint32_t t_base = tmem + ((uint32_t)(quarter * 32) << 16);
  // the accumulator is released on the leader's barrier (remote for the peer)
  const uint32_t acc_empty = PAIR && rank ? mapa_shared(smem_u32(L.acc_empty), 0) : smem_u32(L.acc_empty);
  uint32_t acc_phase = 0;
  const bool tracer = kTraceBuild && warp == EPI_WARP0 && lane == 0;
  int tile = 0;
  for (int it = start; it < total; it += step, ++tile) {
    // the tile and its per-tile parameters, loaded while the MMAs run
    const Work w = decode_work<PAIR>(L, p, it, rank);
    const int g = w.g, nt = w.nt;
    const int64_t row = (int64_t)w.mt * BM + row_in_tile;
    const float gs_a = p.a_gs[g], gs_b = p.b_gs[g];
    float tile_param = 0.f;  // SwiGLU requant: the L2 activation scale; combine: the row's weight
    int row_id = 0;          // single-CTA combine: the row's token (-1: pad row)
    if constexpr (EPI == kEpiSwigluQuant) tile_param = p.q_gs[g];
    if constexpr (EPI == kEpiCombine) {
      tile_param = p.row_w[row];
      if constexpr (!PAIR) row_id = p.sorted_ids[row];
    }
    int ok = 1;
    // polled (a suspending wait, or 128 ns sleeps between polls, timed the
    // same or slower: the spinning lanes do not slow the MMA warp measurably)
    if (lane == 0) ok = wait_bounded_spin(smem_u32(L.acc_full), acc_phase, abort, p.status, p.timeout_ns);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    if (tracer) trace_tile(p, tile, 2);
    __syncwarp();
    tc_fence_after();
    // SwiGLU kinds: gate columns [half*64, +64) and up columns 128 + [half*64, +64);
    // other kinds: columns [half*128, +128).
    uint32_t v[4][32];
    if constexpr (EPI == kEpiSwigluQuant || EPI == kEpiSwigluAmax) {
      tmem_load_64(t_base + half * 64, v[0], v[1]);
      tmem_load_64(t_base + 128 + half * 64, v[2], v[3]);
    } else {  // (a 128-column load needs more registers than the kernel is compiled with)
      tmem_load_64(t_base + half * 128, v[0], v[1]);
      tmem_load_64(t_base + half * 128 + 64, v[2], v[3]);
    }
    tmem_load_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (PAIR && rank) mbar_arrive_remote(acc_empty);
      else mbar_arrive(acc_empty);
    }
    acc_phase ^= 1u;
    if (tracer) trace_tile(p, tile, 3);

    if (!w.valid) continue;  // the pair's second tile does not exist: nothing to store
    const float alpha = 1.0f / (gs_a * gs_b);

    if constexpr (EPI == kEpiBf16) {
      const uint64_t alpha2 = f2_pack(alpha, alpha);
      const int64_t i_local = row - L.offsets[g];
      const bool valid = p.counts ? i_local < p.counts[g] : (p.host_count <= 0 || i_local < p.host_count);
      // columns of this thread's 32-column chunks that exist (a ragged N ends
      // inside a tile; the stores stop at the last 8-column group below it)
      const int col0 = nt * BN + half * (BN / 2);
      const int ncols = p.n_valid > 0 ? min(BN / 2, p.n_valid - col0) : BN / 2;
      if (valid && ncols > 0) {
        uint16_t* drow = p.D + g * p.gstride_d + i_local * p.ldd + col0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = scaled_bf16x2(v[c][2 * j], v[c][2 * j + 1], alpha2);
          if (c * 32 + 32 <= ncols) {
            if (p.d_vec32) {
              st_global_v8(drow + c * 32, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
              st_global_v8(drow + c * 32 + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(drow + c * 32);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            }
          } else {
            uint4* dst = reinterpret_cast<uint4*>(drow + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (c * 32 + 8 * j + 8 <= ncols) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
      }
    } else if constexpr (EPI == kEpiSwigluQuant) {
      // output features [nt*128 + half*64, +64) of one row = 4 quantization blocks
      // (pairs of features per instruction where the arithmetic allows it;
      // every value is rounded exactly as by the scalar operations)
      const float qgs = tile_param;
      const float rcp6 = __frcp_rn(6.0f);
      const uint64_t alpha2 = f2_pack(alpha, alpha), qgs2 = f2_pack(qgs, qgs);
      uint32_t scales = 0;
      uint32_t words[8];
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        uint64_t xs2[8];
        float b = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int f = blk * 16 + 2 * q;  // features f, f+1: same 32-column load
          float g0, g1, u0, u1;
          f2_unpack(f2_mul(f2_pack(__uint_as_float(v[f >> 5][f & 31]), __uint_as_float(v[f >> 5][(f & 31) + 1])),
                           alpha2),
                    g0, g1);
          f2_unpack(f2_mul(f2_pack(__uint_as_float(v[2 + (f >> 5)][f & 31]),
                                   __uint_as_float(v[2 + (f >> 5)][(f & 31) + 1])),
                           alpha2),
                    u0, u1);
          float h0, h1;
          silu_clamped_product2(g0, g1, u0, u1, p.gate_limit, p.up_limit, h0, h1);
          const uint32_t hb = pack_bf16x2(h0, h1);
          xs2[q] = f2_mul(f2_pack(bf16_lo(hb), bf16_hi(hb)), qgs2);
          float x0, x1;
          f2_unpack(xs2[q], x0, x1);
          b = fmaxf(b, fmaxf(fabsf(x0), fabsf(x1)));
        }
        uint32_t lo, hi;
        scales |= quant_block16_pairs(xs2, b, rcp6, lo, hi) << (8 * blk);
        words[blk * 2] = lo;
        words[blk * 2 + 1] = hi;
      }
      const int64_t f0 = (int64_t)nt * 128 + half * 64;  // first output feature of this thread
      // workspace rows: 32-byte aligned (I/2 and f0/2 are multiples of 32 bytes)
      st_global_v8(p.q_out + row * (p.I / 2) + f0 / 2, words[0], words[1], words[2], words[3], words[4], words[5],
                   words[6], words[7]);
      *reinterpret_cast<uint32_t*>(p.q_sf + sf_offset(row, f0 / 16, p.I / 16)) = scales;
      if (p.tile_done) {  // the last of the eight epilogue warps done storing publishes the tile
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          int* slot = L.stored + (tile & 1);
          if (atomicAdd_block(slot, 1) == NUM_EPI_WARPS - 1) {
            *slot = 0;  // reused two tiles on: no warp reaches that tile before every warp left this one
            __threadfence();
            atomicAdd(p.tile_done + w.mt, 1);
          }
        }
      }
    } else if constexpr (EPI == kEpiSwigluAmax) {
      // amax of the bf16 SwiGLU output of this row's 64 features; with D set,
      // the bf16 values themselves too (row-major, ldd elements per row); with
      // h8 set, their FP8 block form instead (and the amax of what is stored)
      uint32_t m = 0;
      uint32_t hw[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int f = 2 * q;  // features f, f+1: same 32-column load
        const float h0 = silu_clamped_product(__uint_as_float(v[f >> 5][f & 31]) * alpha,
                                              __uint_as_float(v[2 + (f >> 5)][f & 31]) * alpha, p.gate_limit,
                                              p.up_limit);
        const float h1 = silu_clamped_product(__uint_as_float(v[f >> 5][(f & 31) + 1]) * alpha,
                                              __uint_as_float(v[2 + (f >> 5)][(f & 31) + 1]) * alpha, p.gate_limit,
                                              p.up_limit);
        hw[q] = pack_bf16x2(h0, h1);
        m = max(m, max(hw[q] & 0x7FFFu, (hw[q] >> 16) & 0x7FFFu));
      }
      m <<= 16;  // float bits of the largest |h|
      if (p.h8) {
        // FP8 blocks: per 16 features the least power-of-two scale that fits the
        // block into E4M3, the codes of h / 2^k, and the largest stored value
        const int64_t f0 = (int64_t)nt * 128 + half * 64;
        uint32_t codes[16], kword = 0, top = 0;
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          uint32_t bm = 0;
#pragma unroll
          for (int q = 0; q < 8; ++q) bm = __vmaxu2(bm, hw[8 * blk + q] & 0x7FFF7FFFu);
          const float a = __uint_as_float(max(bm & 0xFFFFu, bm >> 16) << 16);
          const int k = fp8_block_k(a);
          const float inv = pow2f(-k);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t w0 = hw[8 * blk + 2 * q], w1 = hw[8 * blk + 2 * q + 1];
            codes[4 * blk + q] = drop_negative_zero_bytes(
                e4m3x2_code(bf16_lo(w0) * inv, bf16_hi(w0) * inv) |
                (e4m3x2_code(bf16_lo(w1) * inv, bf16_hi(w1) * inv) << 16));
          }
          top = max(top, __float_as_uint(e4m3_value(e4m3_code(a * inv)) * pow2f(k)));
          kword |= (uint32_t)(k + 127) << (8 * blk);
        }
        // 64-byte aligned: I is a multiple of 128 and f0 of 64
        uint8_t* dst = p.h8 + row * p.I + f0;
        st_global_v8(dst, codes[0], codes[1], codes[2], codes[3], codes[4], codes[5], codes[6], codes[7]);
        st_global_v8(dst + 32, codes[8], codes[9], codes[10], codes[11], codes[12], codes[13], codes[14],
                     codes[15]);
        *reinterpret_cast<uint32_t*>(p.h8_k + row * (p.I / 16) + f0 / 16) = kword;
        m = top;
      } else if (p.D) {
        // 32-byte aligned: the caller passes a 32-byte aligned D and ldd a multiple of 16
        uint16_t* drow = p.D + row * p.ldd + (int64_t)nt * 128 + half * 64;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          st_global_v8(drow + c * 16, hw[8 * c], hw[8 * c + 1], hw[8 * c + 2], hw[8 * c + 3], hw[8 * c + 4],
                       hw[8 * c + 5], hw[8 * c + 6], hw[8 * c + 7]);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0 && m) atomicMax(&p.amax_bits[g], m);
    } else if constexpr (PAIR) {  // kEpiCombine through the warp's staging buffer
      // Routing-weighted rows in slot order for the token combine; pad rows
      // carry weight 0 and are written as zeros (nothing reads them).  Each
      // 64-column chunk of the warp's 32 rows goes through its 4 KB of shared
      // memory in the 128-byte-swizzled layout (16-byte unit u of row r at
      // unit u ^ (r % 8): conflict-free) and leaves with one bulk tensor
      // store; the buffer is rewritten once that store has read it.
      uint8_t* buf = L.epi_stage + (warp - EPI_WARP0) * EPI_STAGE_BYTES;
      const float wgt = tile_param * alpha;
      const uint64_t wgt2 = f2_pack(wgt, wgt);
      const int32_t y_row = (int32_t)(w.mt * BM + quarter * 32), y_col = nt * BN + half * (BN / 2);
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          pk[j] = scaled_bf16x2(v[2 * c2][2 * j], v[2 * c2][2 * j + 1], wgt2);
          pk[16 + j] = scaled_bf16x2(v[2 * c2 + 1][2 * j], v[2 * c2 + 1][2 * j + 1], wgt2);
        }
        if (lane == 0) bulk_wait_read_all();  // the previous store from this buffer has read it
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(buf + lane * 128 + ((u ^ (lane & 7)) << 4)) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&p.tmap_y, smem_u32(buf), y_col + c2 * 64, y_row);
          bulk_commit();
        }
      }
    } else {  // kEpiCombine: routing-weighted rows, stored in slot order for the token combine
      if (row_id >= 0) {
        const float wgt = tile_param * alpha;
        const uint64_t wgt2 = f2_pack(wgt, wgt);
        uint16_t* dst = p.y + row * p.H + (int64_t)nt * BN + half * (BN / 2);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = scaled_bf16x2(v[c][2 * j], v[c][2 * j + 1], wgt2);
          // workspace rows: 32-byte aligned (H is a multiple of 256)
          st_global_v8(dst + c * 32, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
          st_global_v8(dst + c * 32 + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
        }
      }
    }
    if (tracer) trace_tile(p, tile, 4);
  }
  if constexpr (PAIR && EPI == kEpiCombine) {
    if (lane == 0) bulk_wait_all();  // the warp's bulk stores are complete before its CTA exits
    __syncwarp();
  }
}

// Pair variant, warp 3 of the peer CTA: relays the arrival of its stage
// operands (its own full barrier) to the leader's peer_full barrier, so that
// the leader's MMA waits for both CTAs' operands without the scale warps
// standing in the chain (they only report their scales, and run ahead).
template <bool PAIR>
__device__ void relay_loop(const GemmArgs& p, const SmemLayout& L, int total, int start, int step) {
  using C = Cfg<PAIR>;
  volatile int* abort = L.abort_flag;
  const int lane = threadIdx.x & 31;
  uint32_t stage = 0, phase = 0;
  int ok = 1;
  for (int it = start; it < total && ok; it += step) {
    for (int kb = 0; kb < p.num_kb; ++kb) {
      if (lane == 0) {
        ok = wait_bounded_spin(smem_u32(&L.full[stage]), phase, abort, p.status, p.timeout_ns);
        if (ok) mbar_arrive_remote(mapa_shared(smem_u32(&L.peer_full[stage]), 0));
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  __syncwarp();
}

template <int EPI, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1) nvfp4_gemm_kernel(const __grid_constant__ GemmArgs p) {
  using C = Cfg<PAIR>;
  extern __shared__ uint8_t smem_raw[];
  const SmemLayout L = carve<PAIR>(smem_raw, p.G);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  if (!p.late_trigger) pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&L.full[s]), 1);
      mbar_init(smem_u32(&L.empty[s]), 1);
      mbar_init(smem_u32(&L.sf_full[s]), PAIR ? 8 : 4);  // scale warps of this CTA (and of the peer)
      mbar_init(smem_u32(&L.peer_full[s]), 1);          // the peer's relay warp
    }
    for (int s = 0; s < C::SF_STAGES; ++s) {
      mbar_init(smem_u32(&L.sf_data[s]), 1);
      mbar_init(smem_u32(&L.sf_empty[s]), 4);  // this CTA's scale warps
    }
    mbar_init(smem_u32(L.acc_full), 1);
    mbar_init(smem_u32(L.acc_empty), PAIR ? 2 * NUM_EPI_WARPS : NUM_EPI_WARPS);
    mbar_init(smem_u32(L.drain), 1);
    *L.abort_flag = 0;
    L.stored[0] = L.stored[1] = 0;
    fence_mbar_init();
  }
  // everything below reads what earlier kernels wrote; an L2 GEMM fed per
  // m-tile by the L1 GEMM before it instead waits for each m-tile (producers),
  // and was launched only once every kernel before L1 had completed
  if (!(EPI == kEpiCombine && p.tile_done && p.tile_done_target > 0)) pdl_wait();
  if (p.late_trigger) pdl_trigger();
  if (p.host_rows > 0) {  // one group of host-known size
    if (threadIdx.x == 0) {
      L.offsets[0] = 0;
      L.offsets[1] = p.host_rows;
    }
  } else {
    for (int i = threadIdx.x; i <= p.G; i += blockDim.x) L.offsets[i] = p.padded_offsets[i];
  }
  __syncthreads();
  if (warp == 0) {  // work units per group (m-tiles, or pairs of m-tiles), exclusive prefix
    int carry = 0;
    for (int base = 0; base < p.G; base += 32) {
      const int g = base + lane;
      int c = 0;
      if (g < p.G) {
        const int tiles = (L.offsets[g + 1] - L.offsets[g]) / BM;
        c = PAIR ? (tiles + 1) >> 1 : tiles;
      }
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
      prefetch_tmap(&p.tmap_a);
      prefetch_tmap(&p.tmap_b);
    }
  } else if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(L.tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(L.tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync_all();  // both CTAs' barriers initialised, TMEM allocated
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *L.tmem_slot;
  const int total = L.unit_off[p.G] * p.n_tiles;
  const int start = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int step = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  // each warpgroup changes its register budget first thing in its own branch
  if (warp < EPI_WARP0) {
    regs_dec<REGS_SMALL>();
    if (warp == 0) {
      producer_loop<PAIR, false>(p, L, total, start, step, rank);
    } else if (warp == 1) {
      if (rank == 0) mma_loop<PAIR>(p, L, total, start, step, tmem);
    } else if (warp == 2) {
      producer_loop<PAIR, true>(p, L, total, start, step, rank);
    } else if (PAIR && rank == 1) {
      relay_loop<PAIR>(p, L, total, start, step);
    }
  } else if (warp < SF_WARP0) {
    regs_inc<REGS_EPI>();
    epilogue_loop<EPI, PAIR>(p, L, total, start, step, tmem, rank);
  } else {
    regs_dec<REGS_SMALL>();
    sf_loop<PAIR>(p, L, total, start, step, tmem, rank);
  }
  __syncwarp();
  tc_fence_before();
  if constexpr (PAIR) cluster_sync_all();  // no CTA frees TMEM or exits while its peer may still touch it
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, TMEM_COLS);
    else tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Raises the kernel's dynamic shared-memory limit (once per device).
// Also checks that the kernel was allocated exactly REGS_LAUNCH registers per
// thread: setmaxnreg.inc waits for registers the other warpgroups release,
// and the split above is sized for that allocation (a smaller one would make
// the increase wait for ever), so the kernel is never launched otherwise.
template <int EPI, bool PAIR>
cudaError_t configure(int dev) {
  static int configured_device = -1;
  if (configured_device == dev) return cudaSuccess;
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, nvfp4_gemm_kernel<EPI, PAIR>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != REGS_LAUNCH || fa.maxThreadsPerBlock < NUM_THREADS) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(nvfp4_gemm_kernel<EPI, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_bytes_for<PAIR>(PAIR ? MAX_GROUPS_PAIR : MAX_GROUPS));
  if (e == cudaSuccess) configured_device = dev;
  return e;
}

// Largest number of co-resident CTA pairs for one kernel instance (cached per
// device); 0 when pairs cannot be launched.
template <int EPI>
int max_pairs(int dev) {
  static int cached_dev = -1, cached = 0;
  if (cached_dev == dev) return cached;
  if (configure<EPI, true>(dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem_bytes_for<true>(MAX_GROUPS_PAIR);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, nvfp4_gemm_kernel<EPI, true>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 0;
  }
  cached_dev = dev;
  cached = n;
  return n;
}

// grid = number of CTAs (single) or of CTA pairs (pair).
template <int EPI, bool PAIR>
cudaError_t launch_one(const GemmArgs& a, int grid, cudaStream_t s, bool pdl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = configure<EPI, PAIR>(dev)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(PAIR ? 2 * grid : grid);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem_bytes_for<PAIR>(a.G);
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int n = 0;
  if (PAIR) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = 2;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = n ? at : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, nvfp4_gemm_kernel<EPI, PAIR>, a);
}

template <int EPI>
cudaError_t launch_kind(const GemmArgs& a, int units_upper, int num_sms, cudaStream_t s, bool pdl) {
  if (gemm_pair_enabled(EPI, a.pair_hint != 0) && a.G <= MAX_GROUPS_PAIR) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int pairs = max_pairs<EPI>(dev);
    if (pairs > 0) {
      const int want = (units_upper + 1) / 2;
      return launch_one<EPI, true>(a, want < pairs ? (want < 1 ? 1 : want) : pairs, s, pdl);
    }
  }
  return launch_one<EPI, false>(a, units_upper < num_sms ? (units_upper < 1 ? 1 : units_upper) : num_sms, s, pdl);
}

}  // namespace

size_t gemm_smem_bytes(int G) { return smem_bytes_for<false>(G); }

namespace {
int g_gemm_pair_mode = 2;
}

// Mode 2 pairs only the routing-weighted L2 epilogue, whose output stores go
// through the pair variant's staging buffers, and only for large batches; the
// SwiGLU L1 GEMM measured faster as single CTAs.
bool gemm_pair_enabled(int kind, bool hint) {
  return g_gemm_pair_mode == 1 || (g_gemm_pair_mode == 2 && kind == kEpiCombine && hint);
}
int gemm_set_pair_mode(int mode) {
  const int prev = g_gemm_pair_mode;
  g_gemm_pair_mode = mode;
  return prev;
}

namespace {
unsigned long long* g_trace_buf = nullptr;
int g_trace_stages = 0, g_trace_tiles = 0, g_trace_kind = -1;
}  // namespace

bool gemm_trace_built() { return kTraceBuild; }

void gemm_set_trace(unsigned long long* buf, int stages, int tiles, int kind) {
  g_trace_buf = buf;
  g_trace_stages = stages;
  g_trace_tiles = tiles;
  g_trace_kind = buf ? kind : -1;
}
void gemm_get_trace(unsigned long long** buf, int* stages, int* kind) {
  *buf = g_trace_buf;
  *stages = g_trace_stages;
  *kind = g_trace_kind;
}

cudaError_t launch_gemm(int kind, const GemmArgs& args_in, int units_upper, int num_sms, cudaStream_t s, bool pdl) {
  if (args_in.G < 1 || args_in.G > MAX_GROUPS) return cudaErrorInvalidValue;
  GemmArgs args = args_in;
  if (kind == (g_trace_kind & 0xFF)) {  // bits 8 and up of the traced kind: the CTA
    args.trace = g_trace_buf;
    args.trace_stages = g_trace_stages;
    args.trace_tiles = g_trace_tiles;
    args.trace_cta = g_trace_kind >> 8;
  }
  switch (kind) {
    case kEpiBf16: return launch_kind<kEpiBf16>(args, units_upper, num_sms, s, pdl);
    case kEpiSwigluQuant: return launch_kind<kEpiSwigluQuant>(args, units_upper, num_sms, s, pdl);
    case kEpiCombine: return launch_kind<kEpiCombine>(args, units_upper, num_sms, s, pdl);
    case kEpiSwigluAmax: return launch_kind<kEpiSwigluAmax>(args, units_upper, num_sms, s, pdl);
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
