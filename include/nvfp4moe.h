/*
 * nvfp4moe.h -- C ABI of the GB300 (sm_103a) NVFP4 mixture-of-experts FFN forward.
 *
 * The method: the nvfp4-megamoe-kernel commit pages (cutedsl/bridge.py page,
 * commit 50e9b5da; vllm page, commit bde81b95; cutedsl page, commit dfd9c10a).
 * Those pages have no numbered sections; each entry point below names the
 * commit paragraph that defines its operation.
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    allocates no device memory and keeps no pointer after the call returns.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on that stream: no host synchronisation, no host<->device
 *    copy, and sizes that depend on the data stay on the device.
 *  - Return value: an nvfp4_status.  Argument errors are detected on the host
 *    before anything is launched; nothing is launched when a call fails.
 *    nvfp4_last_error() gives a one-line reason for the last failure on the
 *    calling thread.  Errors found on the device (a bounded wait that timed
 *    out) are recorded in a device status word: for the calls that take a
 *    workspace (MoE forward, calibration, shared expert) the int at byte 0 of
 *    that workspace, cleared by the call's first kernel and read with
 *    nvfp4_read_device_status(); for the others (nvfp4_grouped_gemm) one word
 *    per device inside the library, read with nvfp4_device_status().
 *  - NVFP4 tensors: E2M1 values packed two per byte along K (element 2j in the
 *    low nibble of byte j), one FP8-E4M3 scale per 16 consecutive K elements,
 *    and an FP32 global scale gs per tensor or group, multiplied into the
 *    data before encoding (decoded value = e2m1 * scale / gs).
 *  - Scale ("SF") buffers use the 128x4 tile layout of the block-scaled MMA:
 *    for a tensor with R rows (R a multiple of 128) and C = K/16 scale columns
 *    (C a multiple of 4), scale (r, c) is at byte
 *        ((r/128)*(C/4) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4,
 *    i.e. R*C bytes in 512-byte tiles.
 *  - Alignment: every pointer 16-byte aligned; K a multiple of 64.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,    /* bad pointer, size, stride or alignment        */
  NVFP4_ERR_UNSUPPORTED = 2,    /* valid request outside what is implemented     */
  NVFP4_ERR_WORKSPACE = 3,      /* workspace missing or too small                */
  NVFP4_ERR_CUDA = 4,           /* a CUDA runtime / driver call failed           */
  NVFP4_ERR_DEVICE = 5,         /* no usable sm_103a device                      */
  NVFP4_ERR_DEVICE_TIMEOUT = 6  /* a device-side bounded wait ran out            */
} nvfp4_status;

/* Library version as 10000*major + 100*minor + patch. */
int nvfp4_version(void);
/* Static description of a status code. */
const char* nvfp4_status_string(int status);
/* One-line reason of the last failing call on this thread ("" if none). */
const char* nvfp4_last_error(void);

/*
 * nvfp4_quantize -- NVFP4 activation / weight quantization
 * (bridge.py page: "Bug #3 fix", "Bug #4 fix", the 13-byte lookup-table
 * paragraph, and quantize_activation_nvfp4 with a precomputed global scale;
 * cutedsl page: the (T,G,D) -> (G,T,D) permute paragraph for strided groups).
 *
 * Quantizes `groups` groups of `rows` rows of K bf16 values each.  Row r of
 * group g is read at x + g*group_stride_x + r*ld_x (elements, K contiguous).
 * Output row g*rows_padded + r of `fp4` ([groups*rows_padded][K/2] bytes) and
 * of the swizzled scale buffer `sf` (groups*rows_padded*K/16 bytes) receives
 * it; rows rows..rows_padded-1 of every group are written as zeros.
 *   gs       device f32[groups] encode scales, or NULL: then gs = 2688/amax of
 *            the group (1 if the group is all zero) is computed on the device
 *            and written to gs_out (required in that case).
 *   gs_out   device f32[groups] or NULL (when gs != NULL it receives a copy).
 *   workspace, workspace_bytes: device scratch of at least
 *            nvfp4_quantize_workspace_size(groups) bytes when gs == NULL
 *            (ignored otherwise).
 * Requirements: K % 64 == 0, rows_padded % 128 == 0, rows <= rows_padded,
 * ld_x % 8 == 0, group_stride_x % 8 == 0, 1 <= groups <= 65535.
 */
size_t nvfp4_quantize_workspace_size(int groups);
int nvfp4_quantize(const void* x, int64_t rows, int64_t K, int64_t ld_x, int64_t group_stride_x, int groups,
                   const float* gs, float* gs_out, void* workspace, size_t workspace_bytes, void* fp4, void* sf,
                   int64_t rows_padded, void* stream);

/*
 * nvfp4_quantize_no_alloc -- nvfp4_quantize with the global scale computed
 * on the device (gs == NULL behaviour), for callers that cannot provide any
 * scratch memory.  The method's pages have no counterpart of this call; it
 * exists for hosts that own all device memory and offer no way to get a
 * temporary buffer (a server with a pre-reserved pool, a plugin interface
 * without a workspace argument), so neither they nor the library may call
 * cudaMalloc.
 *
 * Same arguments and results as nvfp4_quantize with gs == NULL (gs_out
 * receives 2688/amax per group), minus the workspace.  Instead, the partial
 * maxima of the amax reduction live in a fixed array inside the library's
 * device image (NVFP4_QUANTIZE_NO_ALLOC_MAX_GROUPS x 1024 floats = 256 KB on
 * every GPU that loads the library, held until the process exits).
 *   - groups > NVFP4_QUANTIZE_NO_ALLOC_MAX_GROUPS is rejected with
 *     NVFP4_ERR_UNSUPPORTED before anything is launched.
 *   - The first call on a device looks up that array's device address (with
 *     the device current) and caches it with the id of the CUDA context it
 *     belongs to; after cudaDeviceReset the next call finds a new context and
 *     looks the address up again.  Make the first call on a device (and the
 *     first after a reset) before any stream capture on it.
 *   - Nothing is allocated: no cudaMalloc / cudaFree, no allocating library call.
 *   - Every call on a device shares the array.  Each call rewrites every slot
 *     it reads, so no state survives from one call to the next, but calls
 *     whose kernels overlap on the GPU race on it: keep them ordered on one
 *     stream (or use nvfp4_quantize with your own workspace).
 */
#define NVFP4_QUANTIZE_NO_ALLOC_MAX_GROUPS 64
int nvfp4_quantize_no_alloc(const void* x, int64_t rows, int64_t K, int64_t ld_x, int64_t group_stride_x, int groups,
                            float* gs_out, void* fp4, void* sf, int64_t rows_padded, void* stream);

/*
 * nvfp4_assemble_scales -- place per-group linear scales into 128-row padded
 * slots in the tile layout (vllm page: "Root cause of garbage output",
 * "Bug 9" multi-chunk slots, and the wish for an assembly call that takes a
 * flat scale tensor plus offsets; cutedsl page: assemble_scales_2d_side).
 *   sf_linear       device u8 [offsets[G]][sf_cols] (row-major E4M3 codes)
 *   offsets         device i32[G+1], rows of group g are offsets[g]..offsets[g+1]-1
 *   padded_offsets  device i32[G+1], multiples of 128, with
 *                   padded_offsets[g+1]-padded_offsets[g] >= offsets[g+1]-offsets[g]
 *   rows_capacity   rows of the output buffer (multiple of 128, >= padded_offsets[G])
 *   sf_swizzled     device u8 [rows_capacity * roundup(sf_cols,4)] (tile layout);
 *                   every byte is written, pad rows and pad columns as 0.
 */
int nvfp4_assemble_scales(const void* sf_linear, int64_t sf_cols, const int32_t* offsets,
                          const int32_t* padded_offsets, int groups, int64_t rows_capacity, void* sf_swizzled,
                          void* stream);

/*
 * nvfp4_grouped_gemm -- block-scaled NVFP4 grouped GEMM with BF16 output
 * (vllm page: the GEMM reads scale_a by 128-aligned expert offsets; cutedsl
 * page: group g's rows at their own offset range, single-group linear and
 * shared-expert runners with num_groups = 1).
 *
 *   D[g][i][n] = bf16( alpha_g * sum_k A[padded_offsets[g] + i][k] * B[g][n][k] ),
 *   alpha_g = 1 / (a_gs[g] * b_gs[g]), FP32 accumulation.
 *   A    device u8 [rows_capacity][K/2], SFA tile layout over rows_capacity rows
 *   B    device u8 [G][N][K/2] (K-major),  SFB [G][roundup(N,128)*K/16] tile
 *        layout per group (a group's scale rows padded to whole 128-row tiles)
 *   a_gs, b_gs      device f32[G]
 *   padded_offsets  device i32[G+1], multiples of 128, padded_offsets[G] <= rows_capacity
 *   counts          device i32[G] rows actually stored per group (<= its padded
 *                   range), or NULL to store every padded row
 *   D    device bf16; row i of group g starts at D + g*group_stride_d + i*ldd (elements)
 * Requirements: K % 64 == 0, N % 8 == 0, ldd % 8 == 0, group_stride_d % 8 == 0,
 * rows_capacity % 128 == 0, 1 <= G <= 1024.  Tiles are 128 x 256: with N not a
 * multiple of 256 the last tile of a row block computes columns past N (from
 * the next group's B rows, or zeros past the last group's) and stores only
 * the columns below N.
 */
int nvfp4_grouped_gemm(const void* A, const void* SFA, const float* a_gs, const void* B, const void* SFB,
                       const float* b_gs, const int32_t* padded_offsets, const int32_t* counts, int groups,
                       int64_t rows_capacity, int64_t N, int64_t K, void* D, int64_t ldd, int64_t group_stride_d,
                       void* stream);

/*
 * nvfp4_debug_gemm_stall -- failure-detection check of the GEMM pipeline
 * (no counterpart on the pages; it exercises the bounded waits).
 * Launches nvfp4_grouped_gemm's kernel on the given (valid) operands with its
 * TMA producer switched off, so nothing ever fills the shared-memory ring:
 * the consumers' waits give up after timeout_ms, the kernel records
 * NVFP4_ERR_DEVICE_TIMEOUT in the device status word, frees its tensor
 * memory and returns, leaving the context usable.  D is not written.
 * Arguments as nvfp4_grouped_gemm (counts = NULL, group_stride_d = 0);
 * 1 <= timeout_ms <= 10000.  Read the result with nvfp4_device_status().
 */
int nvfp4_debug_gemm_stall(const void* A, const void* SFA, const float* a_gs, const void* B, const void* SFB,
                           const float* b_gs, const int32_t* padded_offsets, int groups, int64_t rows_capacity,
                           int64_t N, int64_t K, void* D, int64_t ldd, int timeout_ms, void* stream);

/*
 * nvfp4_debug_mma_rate -- measurement aid: the bare block-scaled FP4 MMA
 * stream, the ceiling the grouped GEMMs are compared with (no counterpart on
 * the pages).  Launches `units` CTAs (shapes 0, 3) or CTA pairs (shapes 1, 2);
 * each stages four operand sets once -- A: 128 rows x 256 FP4 from A, its B
 * rows from B, the scale tiles from SFA / SFB, bytes taken in order (any
 * quantizer output) -- and one thread issues iters x 4 back-to-back
 * tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (K = 64) into one
 * FP32 TMEM accumulator, then waits for them.  Nothing is stored.
 *   shape 0: cta_group::1, 128 x 256 per CTA       (2*128*256*256 FLOP per iter)
 *         1: cta_group::2, 256 x 256 per pair      (2*256*256*256 per iter)
 *         2: cta_group::2, 256 x 128 per pair      (2*256*128*256 per iter)
 *         3: cta_group::1, 128 x 128 per CTA       (2*128*128*256 per iter)
 * flags add, each on its own warps and for as long as the stream runs, one
 * activity of the real GEMM pipeline, to see which of them slows the tensor
 * pipe: 1 a tcgen05.commit after every 4 MMAs; 2 the scale tiles re-staged
 * into TMEM (tcgen05.st, same values); 4 the operand sets re-copied into
 * shared memory with bulk copies (same bytes); 8 the accumulator read with
 * tcgen05.ld plus FP32 work; 16 a tcgen05.fence::after_thread_sync before
 * each 4-MMA stage; 32 an mbarrier wait (already complete) before each stage;
 * 64 the MMA thread copies the stage's scale tiles into TMEM with tcgen05.cp;
 * 128 the MMA loop runs on the whole warp (warp-uniform operands) with one
 * elected lane issuing, as the GEMM does; 256 (with 128) a 4-slot ring
 * protocol between the MMA warp and a second warp; 512 (with 384) the scale
 * warps as a second hop in that ring; 1024 (with 896) tcgen05 fences around
 * their arrivals.
 * Device buffers (16-byte aligned): A >= 64 KB, B >= 128 KB, SFA >= 8 KB,
 * SFB >= 16 KB.  1 <= units <= 4096, 0 <= iters <= 2^21, 0 <= flags <= 2047.
 * Time it with events around the call.
 */
int nvfp4_debug_mma_rate(const void* A, size_t a_bytes, const void* SFA, size_t sfa_bytes, const void* B,
                         size_t b_bytes, const void* SFB, size_t sfb_bytes, int shape, int units, int iters,
                         int flags, void* stream);

/*
 * nvfp4_moe_forward -- the NVFP4 mixture-of-experts FFN forward
 * (vllm page: the MoE runner -- 128-row slots, multi-chunk slots "Bug 9",
 * sorted_token_ids gather, quantize_activation_nvfp4 with calibrated global
 * scales, scatter_add combine with zero-weight padding; bridge.py page: fused
 * SwiGLU L1 epilogue and run_nvfp4_moe_fused; cutedsl page: gate clamped
 * before SiLU).
 *
 * For each token t: experts = top_k router logits (ties -> lower expert),
 * weights = softmax renormalised over the chosen experts; for each chosen
 * expert e with weight w:
 *   G  = dq(quant(x_t, a1_gs[e])) . dq(W13[e])^T           (2I outputs)
 *   h  = bf16( silu(min(G[:I], gate_limit)) * clamp(G[I:], -up_limit, up_limit) )
 *   Y  = dq(quant(h, a2_gs[e])) . dq(W2[e])^T              (H outputs)
 *   out[t] = bf16( sum over its top_k experts, in order, of bf16(w * Y) ),
 *   FP32 sum: deterministic (no atomics).
 *   hidden         device bf16 [T][H]
 *   router_logits  device f32 [T][E]
 *   w13            device u8 [E][2I][H/2]  (rows 0..I-1 gate, I..2I-1 up)
 *   w13_sf         device u8 [E][2I*H/16]  (tile layout per expert)
 *   w2             device u8 [E][H][I/2],  w2_sf device u8 [E][H*I/16]
 *   w13_gs, w2_gs, a1_gs, a2_gs   device f32[E] global (encode) scales
 *   a2_gs may be NULL: the L2 activation scales are then taken from this
 *                  batch (vllm page: the L2 scale measured on the L1 output;
 *                  cutedsl page: a BF16 L1 output when no calibrated L2 scale
 *                  exists): a2_gs[e] = 2688 / amax(h of expert e's rows), 1
 *                  when that is 0.  L1 writes h in bf16 into the workspace's h
 *                  region with that amax, a quantize pass reads it back, and
 *                  the scales used are left in the workspace (calib region,
 *                  f32 at byte offset 4E).  Same results, bit for bit, as a
 *                  call given those scales.
 *   workspace      device scratch of nvfp4_moe_workspace_size(...) bytes, 256-aligned;
 *                  it also holds every intermediate (see nvfp4_moe_workspace_layout).
 *   out            device bf16 [T][H]
 * Requirements: H % 256 == 0, I % 128 == 0, 1 <= E <= 256, 1 <= top_k <= min(8, E),
 * T >= 0 (T == 0 launches nothing).
 */
size_t nvfp4_moe_workspace_size(int64_t T, int64_t H, int64_t I, int E, int top_k);
int nvfp4_moe_forward(const void* hidden, const float* router_logits, int64_t T, int64_t H, int64_t I, int E,
                      int top_k, const void* w13, const void* w13_sf, const float* w13_gs, const void* w2,
                      const void* w2_sf, const float* w2_gs, const float* a1_gs, const float* a2_gs,
                      float gate_limit, float up_limit, void* workspace, size_t workspace_bytes, void* out,
                      void* stream);

/*
 * nvfp4_moe_forward_l1_fp8 -- nvfp4_moe_forward with the L2 activation scales
 * taken from the batch (a2_gs NULL behaviour) and the L1 output kept as FP8
 * instead of bf16 until it is requantized (the FP8/BF16 L1-output option; the
 * pages name the option, the format is this library's reading of it): the
 * bf16 SwiGLU output h is stored as OCP E4M3 codes in blocks of 16 features
 * of a row, each block with a power-of-two scale 2^k, k the least integer
 * with max|h_block| <= 448 * 2^k (clamped to [-126, 126], 0 for a zero
 * block), code = E4M3(h / 2^k) rounded to nearest even with no negative zero;
 * h8 = dec(code) * 2^k then replaces h: a2_gs[e] = 2688 / amax(h8 of expert
 * e's rows) and h8 is quantized to NVFP4 with it.  Half the bytes of the bf16
 * round trip.  In the layout the h region holds the codes [capacity][I] and
 * then the block exponents k + 127 [capacity][I/16]; the scales land in calib
 * as with a2_gs NULL.  Arguments, requirements and errors as
 * nvfp4_moe_forward without a2_gs.
 */
int nvfp4_moe_forward_l1_fp8(const void* hidden, const float* router_logits, int64_t T, int64_t H, int64_t I,
                             int E, int top_k, const void* w13, const void* w13_sf, const float* w13_gs,
                             const void* w2, const void* w2_sf, const float* w2_gs, const float* a1_gs,
                             float gate_limit, float up_limit, void* workspace, size_t workspace_bytes, void* out,
                             void* stream);

/* The same forward with expert parallelism: routing comes from the model's
 * router as global top-k ids (vllm page, "Root cause of CUDA_ERROR_ASSERT
 * index out of bounds", fixes 1-2: experts_start_idx; global ids remapped to
 * local ids; non-local experts' weights zeroed).
 *
 *   topk_ids      device int32 [T][top_k], global expert ids (any value)
 *   topk_weights  device f32 [T][top_k], the router's weights, used as given
 *   experts_start global id of local expert 0; global id g is local expert
 *                 g - experts_start when that lies in [0, E)
 * An assignment to a non-local expert gets weight 0, no slot row and no
 * work; a token with none local gets a zero output row.  The workspace size
 * and layout are those of nvfp4_moe_forward (the topk arrays there hold the
 * local ids, -1 for non-local, and the weights actually used).  All other
 * arguments, checks and errors as nvfp4_moe_forward; router_logits is not
 * used.  Asynchronous, no allocation, no host synchronisation. */
int nvfp4_moe_forward_routed(const void* hidden, const int32_t* topk_ids, const float* topk_weights,
                             int32_t experts_start, int64_t T, int64_t H, int64_t I, int E, int top_k,
                             const void* w13, const void* w13_sf, const float* w13_gs, const void* w2,
                             const void* w2_sf, const float* w2_gs, const float* a1_gs, const float* a2_gs,
                             float gate_limit, float up_limit, void* workspace, size_t workspace_bytes, void* out,
                             void* stream);

/* Shared expert: one NVFP4 SwiGLU FFN applied to every token, no routing
 * (cutedsl page: the shared-expert runner paragraph -- a single group, no
 * scatter and no routing -- the fused L1+SiLU+L2 pipeline, rows padded to 128 for the
 * scale layout, all buffers pre-allocated).
 *
 *   out[t] = bf16( L2( requant( SwiGLU( L1( quant(hidden[t]) ) ) ) ) )
 * with the arithmetic of nvfp4_moe_forward for one expert and weight 1.
 *   hidden   bf16 [T][H];  out bf16 [T][H] (only its T rows are written)
 *   w13      [2I][H/2] nibbles (gate rows 0..I-1, up rows I..2I-1), w13_sf
 *            tile-layout scales [2I*H/16], w13_gs f32[1]; w2 [H][I/2], w2_sf,
 *            w2_gs f32[1]; a1_gs / a2_gs f32[1] activation global scales
 *   workspace device scratch of nvfp4_shared_expert_workspace_size(T, H, I)
 *            bytes, 256-byte aligned
 * H a multiple of 256, I of 128; T = 0 is a no-op.  Errors as
 * nvfp4_moe_forward.  Asynchronous, no allocation, no host synchronisation. */
size_t nvfp4_shared_expert_workspace_size(int64_t T, int64_t H, int64_t I);
int nvfp4_shared_expert_forward(const void* hidden, int64_t T, int64_t H, int64_t I, const void* w13,
                                const void* w13_sf, const float* w13_gs, const void* w2, const void* w2_sf,
                                const float* w2_gs, const float* a1_gs, const float* a2_gs, float gate_limit,
                                float up_limit, void* workspace, size_t workspace_bytes, void* out, void* stream);

/*
 * nvfp4_moe_calibrate -- per-expert activation global scales from sample data
 * (vllm page: compute_activation_global_scales -- L1 scale from the gathered
 * hidden rows, L2 scale measured on the L1 output, local expert ids, run
 * before graph capture so the forward can use fixed scales).
 *   a1_gs_out[e] = 2688 / amax(hidden rows routed to e)
 *   a2_gs_out[e] = 2688 / amax(bf16 SwiGLU output of those rows, with the L1
 *                  input quantized by a1_gs_out[e])
 * and 1 for an expert with no rows (or an all-zero amax).  Same arguments,
 * workspace and requirements as nvfp4_moe_forward (W2 is not needed).
 *   a1_gs_out, a2_gs_out   device f32[E]
 */
int nvfp4_moe_calibrate(const void* hidden, const float* router_logits, int64_t T, int64_t H, int64_t I, int E,
                        int top_k, const void* w13, const void* w13_sf, const float* w13_gs, float gate_limit,
                        float up_limit, void* workspace, size_t workspace_bytes, float* a1_gs_out, float* a2_gs_out,
                        void* stream);

/*
 * nvfp4_moe_calibrate_routed -- the same scales from the model router's
 * global top-k instead of this layer's logits (vllm page, "Root cause of
 * CUDA_ERROR_ASSERT index out of bounds": compute_activation_global_scales
 * works on local expert ids; with global ids no row matched a local expert).
 * topk_ids / topk_weights / experts_start as nvfp4_moe_forward_routed: an
 * assignment to an expert outside [experts_start, experts_start + E) takes no
 * row.  The weights are read but do not change the scales.  Other arguments,
 * outputs and errors as nvfp4_moe_calibrate.
 */
int nvfp4_moe_calibrate_routed(const void* hidden, const int32_t* topk_ids, const float* topk_weights,
                               int32_t experts_start, int64_t T, int64_t H, int64_t I, int E, int top_k,
                               const void* w13, const void* w13_sf, const float* w13_gs, float gate_limit,
                               float up_limit, void* workspace, size_t workspace_bytes, float* a1_gs_out,
                               float* a2_gs_out, void* stream);

/*
 * Byte offsets of the forward's intermediates inside the workspace, for
 * inspection by tests.  Sizes: cap = padded-row capacity
 * (roundup(T*top_k + 127*min(E, T*top_k), 128)); A = T*top_k assignments.
 *   status i32 at byte 0: the call's device status word (NVFP4_OK or
 *   NVFP4_ERR_DEVICE_TIMEOUT), cleared by the call's first kernel
 *   topk_ids i32[A], topk_w f32[A]   (token-major: index t*top_k + j)
 *   counts i32[E], offsets i32[E+1]  (padded slot starts, multiples of 128)
 *   meta i32[4] = {P (padded rows), P/128, 0, 0}
 *   tile_expert i32[cap/128], sorted_token_ids i32[cap] (-1 pad),
 *   row_weight f32[cap] (0 pad), inverse i32[A] (assignment -> row)
 *   a1 u8[cap][H/2], sfa1 u8[cap*H/16], a2 u8[cap][I/2], sfa2 u8[cap*I/16]
 *   y bf16[cap][H] (routing-weighted L2 rows in slot order),
 *   h bf16[cap][I] (with a2_gs NULL: the bf16 SwiGLU output of L1; not
 *   written otherwise),
 *   calib u32[2E] (calibration amax bits; with a2_gs NULL, E amax words of
 *   the L1 output, then the E L2 global scales as f32)
 *   tile_done i32[cap/128] (L1 n-tiles finished per m-tile: the L2 GEMM
 *   starts on an m-tile once all of its L1 output is stored)
 * Only rows < P of the row-indexed buffers are defined after a call; the
 * pad rows of a1 hold zero block scales (every value exactly 0) and
 * unspecified nibble bytes.
 */
typedef struct {
  size_t status, topk_ids, topk_w, block_counts, counts, offsets, meta, tile_expert, sorted_token_ids, row_weight,
      inverse, a1, sfa1, a2, sfa2, y, h, calib, tile_done, total;
  int64_t capacity;
  int64_t route_blocks;
} nvfp4_moe_layout;
int nvfp4_moe_workspace_layout(int64_t T, int64_t H, int64_t I, int E, int top_k, nvfp4_moe_layout* out);

/*
 * Device status word of the calls without a workspace (nvfp4_grouped_gemm,
 * nvfp4_debug_gemm_stall), one per device: NVFP4_OK or
 * NVFP4_ERR_DEVICE_TIMEOUT.  Synchronises the device.  reset != 0 clears it
 * afterwards.
 */
int nvfp4_device_status(int* status_out, int reset);

/*
 * Status of the last call that used this workspace (MoE forward, routed
 * forward, calibration or shared expert): the int at byte 0 of the
 * workspace, NVFP4_OK or NVFP4_ERR_DEVICE_TIMEOUT.  Each such call clears the
 * word in its first kernel, so it reports that call only, and calls on other
 * workspaces (other streams) never touch it.  Reads it on `stream` and waits
 * for that stream (a host synchronisation: for tests and error handling, not
 * for the hot path); reset != 0 then clears it.  workspace: 256-byte aligned
 * device pointer.
 */
int nvfp4_read_device_status(const void* workspace, void* stream, int* status_out, int reset);

/*
 * Debug timeline of the GEMM pipeline (no counterpart on the pages): every
 * following GEMM launch with epilogue `kind` (0 bf16 output, 1 SwiGLU +
 * requantization, 2 routing-weighted rows, 3 SwiGLU amax; 4: the
 * nvfp4_debug_mma_rate kernel, words 5 and 6 only) writes SM-clock stamps
 * (%clock64, cycles) of one CTA's roles (CTA 0, or kind + 256 * c for CTA c
 * of kinds 0-3) into `buffer` (device, 8-byte
 * aligned, (stages + tiles) * 8 words): 8 words per ring stage for the first
 * `stages` stages -- producer slot free, copies issued, scale warp saw the
 * data, scales staged, MMA starts waiting, MMA may issue, MMA instructions
 * issued, stage committed -- then 8 words per tile for the first `tiles`
 * tiles -- MMA waits for the accumulator, accumulator free, epilogue saw it
 * full, epilogue released it, epilogue finished.  Words not reached stay as
 * they were.  buffer NULL switches it off.  Process-wide; for performance
 * analysis only.  Kinds 0-3 need a library built with -DNVFP4_GEMM_TRACE
 * (the recording points cost the GEMM loops even when switched off, so the
 * default build leaves them out); otherwise NVFP4_ERR_UNSUPPORTED.
 */
int nvfp4_debug_gemm_trace(void* buffer, int stages, int tiles, int kind);

/*
 * Failure-detection check of the MoE forward (no counterpart on the pages).
 * timeout_ms > 0: every following nvfp4_moe_forward / _routed call launches
 * its L1 GEMM with the operand loads switched off and that wait limit, so the
 * GEMM gives up, records NVFP4_ERR_DEVICE_TIMEOUT in that call's workspace
 * status word and returns; the rest of the forward runs on whatever the L2
 * input buffer held (its output is meaningless, nothing faults).  0 switches
 * it off.  Process-wide; 0 <= timeout_ms <= 10000.
 */
int nvfp4_moe_set_debug_stall(int timeout_ms);

/*
 * nvfp4_moe_set_overlap -- measurement switch (process-wide, default 1): with
 * 1, a forward given its L2 scales lets its L2 GEMM start on the SMs the L1
 * GEMM's last partial round of tiles leaves idle, each L2 tile waiting (on
 * the device, bounded) until the L1 output of its m-tile is stored; with 0
 * the L2 GEMM waits for the whole L1 GEMM.  Results are identical either way.
 * prev (may be NULL) receives the previous setting.
 */
int nvfp4_moe_set_overlap(int enable, int* prev);

/* GEMM variant (process-wide; every GEMM above and the MoE forward).
 *
 * A "pair" GEMM runs a cluster of two CTAs on two SMs per 256 x 256 output
 * tile with the paired tensor-core instructions (tcgen05 cta_group::2); each
 * SM stages half of the B tile, so it reads fewer operand bytes per MMA, and
 * the routing-weighted L2 epilogue stores through shared-memory staging.  A
 * "single" GEMM runs one CTA per 128 x 256 tile.  Both compute every output
 * element with the same arithmetic in the same order: results are
 * bit-identical.
 *   mode 0  single CTAs for every GEMM
 *   mode 1  pairs for every GEMM with at most 256 groups
 *   mode 2  pairs for the MoE L2 GEMM when T * top_k >= 256 * E (experts
 *           average two or more 128-row tiles); single otherwise (default)
 * prev_mode (may be null) receives the previous mode.  Returns NVFP4_OK, or
 * NVFP4_ERR_INVALID_ARG (mode unchanged) for a mode outside 0..2.  Not
 * thread-safe with respect to launches issued concurrently from other host
 * threads; no device work. */
int nvfp4_gemm_set_cta_pair(int mode, int* prev_mode);

/*
 * nvfp4_moe_set_swap_l2 -- the L2 GEMM of small batches with swapped operands.
 *
 * With enable 1, a forward whose L2 GEMM runs single CTAs (T * top_k <
 * 256 * E: decode-sized batches) and whose E is at most 256 computes the L2
 * GEMM with 128-row tiles of the expert's W2 as the MMA's M operand and 64
 * of the expert's slot rows as N, over the expert's real rows only, instead
 * of 128-row slot tiles against 256 W2 rows; the routing-weighted bf16 rows
 * it stores (y) are the same, bit for bit.  enable 0 (the default): always
 * the slot-major GEMM, which measured as fast or faster (the weight stream
 * of both runs at the memory rate).  prev_enable (may be null) receives the
 * previous setting.  Returns NVFP4_OK, or NVFP4_ERR_INVALID_ARG (setting
 * unchanged) for a value other than 0 or 1.  Not thread-safe with respect
 * to launches issued concurrently from other host threads; no device work. */
int nvfp4_moe_set_swap_l2(int enable, int* prev_enable);

/*
 * Optional per-stage timing of nvfp4_moe_forward: when set, the forward
 * records events[i] (cudaEvent_t) on its stream before stage i, i = 0..6, and
 * events[7] after the last stage (stages: route, slot scan, slot scatter,
 * gather+quantize, L1 GEMM, L2 GEMM, token combine).  n_events must be 8, or 0
 * with events NULL to switch it off.  Process-wide; not thread-safe.
 */
int nvfp4_moe_set_stage_events(void* const* events, int n_events);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4MOE_H */
