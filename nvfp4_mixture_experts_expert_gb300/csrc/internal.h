// Internal launch interface between the C ABI (abi.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace nvfp4 {

// Launch with optional programmatic stream serialization (the kernel must call
// pdl_wait() before touching global memory when pdl is set).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? at : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- quant.cu
// Per-group amax of bf16 rows into partial maxima (groups x kAmaxBlocksPerGroup
// floats, amax_blocks_per_group(groups, num_sms) of each group's slots
// written), then, when gs_out is given, gs = 2688/amax by a second kernel.
constexpr int kAmaxBlocksPerGroup = 1024;
int amax_blocks_per_group(int groups, int num_sms);
cudaError_t launch_group_amax(const uint16_t* x, int64_t rows, int64_t K, int64_t ld_x, int64_t gstride_x,
                              int groups, float* partial, float* gs_out, int num_sms, cudaStream_t s);
// status_reset (may be null): a per-call device status word the kernel clears
// before anything later in the stream can record into it.  amax_partial (may
// be null): the amax kernel's partial maxima; the kernel then derives each
// group's gs from them (gs unused) and writes it to gs_copy.
cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t K, int64_t ld_x, int64_t gstride_x,
                            int groups, const float* gs, float* gs_copy, uint8_t* fp4, uint8_t* sf,
                            int64_t rows_padded, int num_sms, cudaStream_t s, int* status_reset = nullptr,
                            const float* amax_partial = nullptr);
cudaError_t launch_assemble_scales(const uint8_t* sf_linear, int64_t sf_cols, const int32_t* offsets,
                                   const int32_t* padded_offsets, int groups, int64_t rows_capacity,
                                   uint8_t* sf_swz, int num_sms, cudaStream_t s);
// MoE: gather hidden rows into expert slots and quantize them (one slot row per thread group).
cudaError_t launch_gather_quantize(const uint16_t* hidden, int64_t H, int64_t T, int top_k,
                                   const int32_t* topk_ids, const int32_t* inverse, const int32_t* counts,
                                   const int32_t* offsets, int E, const float* a1_gs, int64_t capacity, uint8_t* a1,
                                   uint8_t* sfa1, cudaStream_t s, bool pdl = false, int* tile_done = nullptr);
// Calibration: per-expert amax of the gathered hidden rows (as float bits, atomicMax
// into a zeroed array), and gs = 2688/amax (1 for an empty / all-zero expert).
cudaError_t launch_gather_amax(const uint16_t* hidden, int64_t H, const int32_t* sorted_ids,
                               const int32_t* tile_expert, const int32_t* meta, int64_t capacity,
                               uint32_t* amax_bits, int num_sms, cudaStream_t s);
cudaError_t launch_gs_from_amax(const uint32_t* amax_bits, int n, float* gs, cudaStream_t s);
// MoE L2 activations with global scales from the batch: slot rows of the bf16
// SwiGLU output h [capacity, K] quantized with gs = 2688/amax of their expert
// (amax as float bits); gs_out receives the E global scales.
cudaError_t launch_slot_quantize(const uint16_t* h, int64_t K, const int32_t* meta, const int32_t* tile_expert,
                                 int64_t capacity, const uint32_t* amax_bits, int E, float* gs_out, uint8_t* fp4,
                                 uint8_t* sf, int num_sms, cudaStream_t s, bool pdl = false);
// The same from the FP8 block form of h (codes [rows][K], exponents [rows][K/16]).
cudaError_t launch_slot_quantize_fp8(const uint8_t* h8, const uint8_t* h8_k, int64_t K, const int32_t* meta,
                                     const int32_t* tile_expert, int64_t capacity, const uint32_t* amax_bits, int E,
                                     float* gs_out, uint8_t* fp4, uint8_t* sf, int num_sms, cudaStream_t s, bool pdl);

// ---------------------------------------------------------------- route.cu
constexpr int kRouteTokensPerBlock = 16;
// The routing kernels open a forward: each clears the call's device status
// word (status_reset, may be null) before any later kernel of the call runs.
cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w,
                              int32_t* block_counts, int* status_reset, cudaStream_t s);
// Expert-parallel routing from given global top-k ids / weights (see route.cu).
cudaError_t launch_route_external(const int32_t* topk_ids, const float* topk_w, int32_t start, int64_t T, int E,
                                  int k, int32_t* ids, float* w, int32_t* block_counts, int* status_reset,
                                  cudaStream_t s);
// Small batches: routing (logits, or external ids when logits is null),
// offsets, tile table, pad rows and slot permutation in one block.
constexpr int64_t kSmallRouteTokens = 256;
cudaError_t launch_route_small(const float* logits, const int32_t* ext_ids, const float* ext_w, int32_t start,
                               int64_t T, int E, int k, int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                               int32_t* meta, int32_t* tile_expert, int32_t* sorted_ids, float* row_w,
                               int32_t* inverse, int* status_reset, cudaStream_t s);
cudaError_t launch_slot_scan(int32_t* block_counts, int nblocks, int E, int32_t* counts, int32_t* offsets,
                             int32_t* meta, int32_t* tile_expert, int32_t* sorted_ids, float* row_w,
                             uint32_t* zero_words, int n_zero_words, cudaStream_t s, bool pdl = false);
cudaError_t launch_slot_scatter(const int32_t* ids, const float* w, int64_t T, int E, int k,
                                const int32_t* block_base, const int32_t* offsets, int32_t* sorted_ids,
                                float* row_w, int32_t* inverse, cudaStream_t s, bool pdl = false);
// out[t] = bf16( sum_j Y[inverse[t*k + j]] ), j ascending, FP32 sum.
cudaError_t launch_token_combine(const uint16_t* y, const int32_t* inverse, int64_t T, int64_t H, int k,
                                 uint16_t* out, cudaStream_t s, bool pdl = false);

// ---------------------------------------------------------------- gemm.cu
enum EpilogueKind { kEpiBf16 = 0, kEpiSwigluQuant = 1, kEpiCombine = 2, kEpiSwigluAmax = 3 };

struct GemmArgs {
  CUtensorMap tmap_a;  // A: [rows][K/2] bytes, box 128 B x 128 rows, 128-byte swizzle
  CUtensorMap tmap_b;  // B: [G * b_rows_per_group][K/2] bytes, same box
  CUtensorMap tmap_y;  // kEpiCombine, pair variant: y as bf16 [rows][H], box 64 x 32, 128-byte swizzle
  const uint8_t* sfa;  // tile-layout scales of A (rows x K/16)
  const uint8_t* sfb;  // tile-layout scales of B, sfb_group_bytes per group
  const int32_t* padded_offsets;  // [G+1]
  const int32_t* counts;          // [G] or null (plain epilogue)
  const float* a_gs;              // [G]
  const float* b_gs;              // [G]
  int G;
  int K;
  int num_kb;            // ceil(K / 256)
  int b_rows_per_group;  // N (plain / combine) or 2I (SwiGLU)
  int n_tiles;           // output tiles per 128-row m-tile
  int b_second_offset;   // rows from the first to the second 128-row B box
  int b_tile_stride;     // B rows between consecutive n-tiles
  int n_major;           // tile order: 0 = m-tile major, 1 = n-tile major
  int64_t sfb_group_bytes;
  // kEpiBf16 with a ragged N (0: every column of every tile is stored): the
  // columns stored per group, and the 128-row scale tiles a group has (a
  // tile's second B half beyond them takes the first half's scales; those
  // columns are not stored)
  int n_valid;
  int sfb_tiles;
  // kEpiBf16
  uint16_t* D;
  int64_t ldd;
  int64_t gstride_d;
  int d_vec32;  // D, ldd and gstride_d allow 32-byte stores
  int pair_hint;  // mode 2: the caller expects most groups to span at least two m-tiles
  // One group whose sizes the host knows (no device metadata): host_rows > 0
  // replaces padded_offsets by [0, host_rows]; host_count > 0 (kEpiBf16, no
  // counts array) keeps rows at or beyond it from being stored.
  int host_rows;
  int host_count;
  // kEpiSwigluQuant
  uint8_t* q_out;
  uint8_t* q_sf;
  const float* q_gs;
  int I;
  float gate_limit;
  float up_limit;
  // kEpiSwigluAmax: per-group amax of h (float bits, atomicMax).  With h8
  // set, h is stored as FP8 blocks instead of bf16 in D: E4M3 codes
  // [rows][I] in h8 and, per 16 features, the block exponent k + 127 in
  // h8_k [rows][I/16]; the amax is then that of the stored values.
  uint32_t* amax_bits;
  uint8_t* h8;
  uint8_t* h8_k;
  // kEpiCombine
  uint16_t* y;  // bf16 [rows][H], routing-weighted L2 rows in slot order
  const int32_t* sorted_ids;
  const float* row_w;
  int H;
  // Hand-off of the MoE forward's L1 output to the L2 GEMM per m-tile, so
  // that the L2 GEMM runs on the SMs the L1 GEMM's last partial round leaves
  // idle.  L1 (kEpiSwigluQuant): tile_done[mt] += 1 once a tile's A2 rows and
  // scales are stored; late_trigger: its dependent launch is released only
  // after its own dependency wait (so the L2 kernel starts after every kernel
  // before L1 completed).  L2 (kEpiCombine, tile_done_target > 0): no
  // dependency wait; before it loads m-tile mt it waits until
  // tile_done[mt] == tile_done_target.  tile_done is zeroed by the gather.
  int* tile_done;
  int tile_done_target;
  int late_trigger;
  // bounded waits
  int* status;
  unsigned long long timeout_ns;
  int debug_no_loads;  // test hook: the producer issues nothing, so consumers time out
  // optional timeline of CTA 0 (nvfp4_debug_gemm_trace): 8 words per ring
  // stage for trace_stages stages, then 8 words per tile for trace_tiles tiles
  unsigned long long* trace;
  int trace_stages;
  int trace_tiles;
  int trace_cta;  // the CTA whose roles are recorded
};

size_t gemm_smem_bytes(int G);

// gemm_swap.cu: the MoE L2 GEMM for small batches with W2 tiles as the MMA's
// M = 128 operand and 64 slot rows as N (see there); same output as the
// routing-weighted epilogue of launch_gemm(kEpiCombine).
struct SwapArgs {
  CUtensorMap tmap_w;  // W2: [G * H][K/2] bytes, box 128 B x 128 rows, 128-byte swizzle
  CUtensorMap tmap_x;  // L1 output (A2): [rows][K/2] bytes, box 128 B x 64 rows, 128-byte swizzle
  const uint8_t* sfw;  // W2 tile-layout scales, sfw_group_bytes per group
  const uint8_t* sfx;  // A2 tile-layout scales (slot rows)
  const int32_t* offsets;  // [G+1] 128-aligned slot offsets
  const int32_t* counts;   // [G] real rows per group
  const float* x_gs;       // [G] A2 global scales
  const float* w_gs;       // [G] W2 global scales
  const float* row_w;      // [rows] routing weights in slot order
  uint16_t* y;             // bf16 [rows][H]
  int G;
  int K;        // I
  int num_kb;   // ceil(K / 256)
  int H;        // output features (W2 rows per group), a multiple of 128
  int n_wtiles; // H / 128
  int64_t sfw_group_bytes;
  int* tile_done;  // as GemmArgs (L1 -> L2 hand-off per m-tile)
  int tile_done_target;
  int* status;
  unsigned long long timeout_ns;
};
size_t gemm_swap_smem_bytes(int G);
cudaError_t launch_gemm_swap(const SwapArgs& args, int num_sms, cudaStream_t s, bool pdl);

// abi.cu: sets the text nvfp4_last_error() returns on the calling thread.
void set_last_error(const char* msg);
// units_upper: an upper bound on the work items (128-row m-tiles x n-tiles);
// the grid is sized from it and from the SM count / co-resident CTA pairs.
cudaError_t launch_gemm(int kind, const GemmArgs& args, int units_upper, int num_sms, cudaStream_t s,
                        bool pdl = false);
// Whether a GEMM with this epilogue runs as CTA pairs (cta_group::2) or single
// CTAs.  Mode: 0 single, 1 pair, 2 pair for the routing-weighted L2 epilogue
// when the caller's hint says most groups span at least two m-tiles (a group
// of one m-tile would leave half of its pair idle); set returns the previous
// mode.
bool gemm_pair_enabled(int kind, bool hint);
int gemm_set_pair_mode(int mode);
// Debug timeline of the next GEMM launches of epilogue kind `kind` (-1: off;
// 4: the MMA-rate kernel).
void gemm_set_trace(unsigned long long* buf, int stages, int tiles, int kind);
bool gemm_trace_built();  // the GEMM kernels were compiled with NVFP4_GEMM_TRACE
void gemm_get_trace(unsigned long long** buf, int* stages, int* kind);
cudaError_t gemm_status_ptr(int** ptr);
cudaError_t gemm_read_status(int* out, int reset);

}  // namespace nvfp4
