// extern "C" entry points of libnvfp4moe: host-side argument checks, TMA
// tensor-map encoding (per call, so descriptors never outlive the pointers
// they describe -- the stale-descriptor lesson of the bridge.py page), and
// the launch sequence of each operation.  No device allocation, no host
// synchronisation, no host<->device copy on any of these paths.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/nvfp4moe.h"
#include "internal.h"

using namespace nvfp4;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(NVFP4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceInfo {
  int sms = 0;
  int* status = nullptr;
  bool ok = false;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Per-device properties; rejects devices other than compute capability 10.3.
int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(NVFP4_ERR_DEVICE, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ok) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
      return fail(NVFP4_ERR_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev, major, minor);
    int* st = nullptr;
    if ((e = gemm_status_ptr(&st)) != cudaSuccess) return cuda_fail(e, "status word address");
    d.sms = sms;
    d.status = st;
    d.ok = true;
  }
  *out = &d;
  return NVFP4_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// K-major packed FP4 matrix [rows][K/2] bytes; box 128 bytes x 128 rows, 128-byte swizzle.
int make_fp4_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  const cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return NVFP4_OK;
}

// bf16 matrix [rows][cols] (row stride cols elements); box 64 columns (128 bytes)
// x 32 rows, 128-byte swizzle: the staging layout of the routing-weighted L2
// epilogue's bulk stores.
int make_bf16_store_map(CUtensorMap* map, void* base, int64_t rows, int64_t cols) {
  auto fn = encode_fn();
  if (!fn) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return NVFP4_OK;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

int64_t moe_capacity(int64_t T, int E, int k) {
  const int64_t A = T * k;
  return round_up(A + 127 * (A < E ? A : (int64_t)E), 128);
}

void* g_stage_events[8] = {};
int g_n_stage_events = 0;
int g_debug_stall_ms = 0;  // > 0: MoE forwards launch their L1 GEMM with no operand loads (failure-detection test)
int g_l1_l2_overlap = 1;   // the L2 GEMM takes the L1 output per m-tile (nvfp4_moe_set_overlap)
int g_swap_l2 = 0;         // small batches: the L2 GEMM with swapped operands (nvfp4_moe_set_swap_l2)

inline void stage_mark(int i, cudaStream_t s) {
  if (g_n_stage_events == 8 && g_stage_events[i]) cudaEventRecord((cudaEvent_t)g_stage_events[i], s);
}

}  // namespace

void nvfp4::set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg ? msg : ""); }

static int grouped_gemm_impl(const void* A, const void* SFA, const float* a_gs, const void* B, const void* SFB,
                             const float* b_gs, const int32_t* padded_offsets, const int32_t* counts, int groups,
                             int64_t rows_capacity, int64_t N, int64_t K, void* D, int64_t ldd,
                             int64_t group_stride_d, void* stream, int debug_no_loads, uint64_t timeout_ns) {
  g_err[0] = 0;
  if (groups < 1 || groups > 1024) return fail(NVFP4_ERR_INVALID_ARG, "groups must be in [1, 1024]");
  if (K <= 0 || K % 64) return fail(NVFP4_ERR_INVALID_ARG, "K must be a positive multiple of 64");
  if (N <= 0 || N % 8) return fail(NVFP4_ERR_INVALID_ARG, "N must be a positive multiple of 8");
  if (rows_capacity < 0 || rows_capacity % 128) return fail(NVFP4_ERR_INVALID_ARG, "rows_capacity % 128 != 0");
  if (ldd % 8 || group_stride_d % 8 || ldd < 0 || group_stride_d < 0)
    return fail(NVFP4_ERR_INVALID_ARG, "ldd and group_stride_d must be non-negative multiples of 8");
  if (!A || !SFA || !a_gs || !B || !SFB || !b_gs || !padded_offsets || !D)
    return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(A) || !aligned16(SFA) || !aligned16(B) || !aligned16(SFB) || !aligned16(D))
    return fail(NVFP4_ERR_INVALID_ARG, "A, SFA, B, SFB and D must be 16-byte aligned");
  if ((int64_t)groups * N > INT32_MAX || rows_capacity > INT32_MAX)
    return fail(NVFP4_ERR_UNSUPPORTED, "row counts beyond 2^31");
  DeviceInfo* dev = nullptr;
  if (int rc = device_info(&dev)) return rc;
  if (rows_capacity == 0) return NVFP4_OK;
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  if (int rc = make_fp4_map(&a.tmap_a, A, rows_capacity, K)) return rc;
  if (int rc = make_fp4_map(&a.tmap_b, B, (int64_t)groups * N, K)) return rc;
  a.sfa = (const uint8_t*)SFA;
  a.sfb = (const uint8_t*)SFB;
  a.padded_offsets = padded_offsets;
  a.counts = counts;
  a.a_gs = a_gs;
  a.b_gs = b_gs;
  a.G = groups;
  a.K = (int)K;
  a.num_kb = (int)((K + 255) / 256);
  // a ragged N: ceil(N / 256) tiles per row block; the columns past N are
  // computed (from the next group's B rows, or zeros past the last group) and
  // not stored; each group's scales span whole 128-row tiles
  const int64_t n128 = round_up(N, 128);
  a.b_rows_per_group = (int)N;
  a.n_tiles = (int)((N + 255) / 256);
  a.b_second_offset = 128;
  a.b_tile_stride = 256;
  a.sfb_group_bytes = n128 * (K / 16);
  a.n_valid = N % 256 ? (int)N : 0;
  a.sfb_tiles = N % 256 ? (int)(n128 / 128) : 0;
  a.D = (uint16_t*)D;
  a.d_vec32 = (reinterpret_cast<uintptr_t>(D) & 31u) == 0 && ldd % 16 == 0 && group_stride_d % 16 == 0;
  a.ldd = ldd;
  a.gstride_d = group_stride_d;
  a.status = dev->status;
  a.timeout_ns = timeout_ns;
  a.debug_no_loads = debug_no_loads;
  const int64_t max_tiles = rows_capacity / 128 * a.n_tiles;
  // programmatic dependent launch: the prologue (barriers, tensor-map prefetch)
  // overlaps the tail of the kernel before it (typically the A quantization);
  // everything that reads inputs waits for that kernel first
  cudaError_t e = launch_gemm(kEpiBf16, a, (int)(max_tiles < INT32_MAX ? max_tiles : INT32_MAX), dev->sms,
                              (cudaStream_t)stream, true);
  return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "gemm launch");
}

extern "C" {

int nvfp4_version(void) { return 100; }

const char* nvfp4_status_string(int status) {
  switch (status) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_UNSUPPORTED: return "unsupported";
    case NVFP4_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4_ERR_CUDA: return "CUDA error";
    case NVFP4_ERR_DEVICE: return "no usable sm_103a device";
    case NVFP4_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

const char* nvfp4_last_error(void) { return g_err; }

size_t nvfp4_quantize_workspace_size(int groups) {
  return groups > 0 ? (size_t)groups * kAmaxBlocksPerGroup * sizeof(float) : 0;
}

int nvfp4_quantize(const void* x, int64_t rows, int64_t K, int64_t ld_x, int64_t group_stride_x, int groups,
                   const float* gs, float* gs_out, void* workspace, size_t workspace_bytes, void* fp4, void* sf,
                   int64_t rows_padded, void* stream) {
  g_err[0] = 0;
  if (groups < 1 || groups > 65535) return fail(NVFP4_ERR_INVALID_ARG, "groups must be in [1, 65535]");
  if (K <= 0 || K % 64) return fail(NVFP4_ERR_INVALID_ARG, "K must be a positive multiple of 64");
  if (rows < 0 || rows_padded < rows || rows_padded % 128)
    return fail(NVFP4_ERR_INVALID_ARG, "need 0 <= rows <= rows_padded and rows_padded % 128 == 0");
  if (ld_x < K || ld_x % 8 || group_stride_x < 0 || group_stride_x % 8)
    return fail(NVFP4_ERR_INVALID_ARG, "ld_x must be >= K and both strides multiples of 8 elements");
  if ((rows > 0 && !x) || (rows_padded > 0 && (!fp4 || !sf)))
    return fail(NVFP4_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(x) || !aligned16(fp4) || !aligned16(sf) || !aligned16(gs) || !aligned16(gs_out))
    return fail(NVFP4_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  if (!gs && !gs_out) return fail(NVFP4_ERR_INVALID_ARG, "gs == NULL needs gs_out");
  if (!gs && (!workspace || workspace_bytes < nvfp4_quantize_workspace_size(groups)))
    return fail(NVFP4_ERR_WORKSPACE, "workspace of %zu bytes needed", nvfp4_quantize_workspace_size(groups));
  DeviceInfo* dev = nullptr;
  if (int rc = device_info(&dev)) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  // gs == NULL: the amax kernel leaves partial maxima in the workspace and the
  // quantize kernel reduces them to gs itself (a separate gs kernel runs only
  // when there is nothing to quantize).
  const float* partial = gs ? nullptr : (const float*)workspace;
  if (!gs && (e = launch_group_amax((const uint16_t*)x, rows, K, ld_x, group_stride_x, groups, (float*)workspace,
                                    rows_padded > 0 ? nullptr : gs_out, dev->sms, s)) != cudaSuccess)
    return cuda_fail(e, "amax launch");
  if (rows_padded > 0 &&
      (e = launch_quantize((const uint16_t*)x, rows, K, ld_x, group_stride_x, groups, gs, gs_out, (uint8_t*)fp4,
                           (uint8_t*)sf, rows_padded, dev->sms, s, nullptr, partial)) != cudaSuccess)
    return cuda_fail(e, "quantize launch");
  return NVFP4_OK;
}

int nvfp4_assemble_scales(const void* sf_linear, int64_t sf_cols, const int32_t* offsets,
                          const int32_t* padded_offsets, int groups, int64_t rows_capacity, void* sf_swizzled,
                          void* stream) {
  g_err[0] = 0;
  if (groups < 1 || groups > 4096) return fail(NVFP4_ERR_INVALID_ARG, "groups must be in [1, 4096]");
  if (sf_cols <= 0) return fail(NVFP4_ERR_INVALID_ARG, "sf_cols must be positive");
  if (rows_capacity < 0 || rows_capacity % 128) return fail(NVFP4_ERR_INVALID_ARG, "rows_capacity % 128 != 0");
  if (!offsets || !padded_offsets || (rows_capacity > 0 && !sf_swizzled))
    return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(sf_swizzled)) return fail(NVFP4_ERR_INVALID_ARG, "sf_swizzled must be 16-byte aligned");
  DeviceInfo* dev = nullptr;
  if (int rc = device_info(&dev)) return rc;
  if (rows_capacity == 0) return NVFP4_OK;
  cudaError_t e = launch_assemble_scales((const uint8_t*)sf_linear, sf_cols, offsets, padded_offsets, groups,
                                         rows_capacity, (uint8_t*)sf_swizzled, dev->sms, (cudaStream_t)stream);
  return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "assemble launch");
}

int nvfp4_grouped_gemm(const void* A, const void* SFA, const float* a_gs, const void* B, const void* SFB,
                       const float* b_gs, const int32_t* padded_offsets, const int32_t* counts, int groups,
                       int64_t rows_capacity, int64_t N, int64_t K, void* D, int64_t ldd, int64_t group_stride_d,
                       void* stream) {
  return grouped_gemm_impl(A, SFA, a_gs, B, SFB, b_gs, padded_offsets, counts, groups, rows_capacity, N, K, D, ldd,
                           group_stride_d, stream, 0, 2000000000ull);
}

int nvfp4_debug_gemm_stall(const void* A, const void* SFA, const float* a_gs, const void* B, const void* SFB,
                           const float* b_gs, const int32_t* padded_offsets, int groups, int64_t rows_capacity,
                           int64_t N, int64_t K, void* D, int64_t ldd, int timeout_ms, void* stream) {
  g_err[0] = 0;
  if (timeout_ms < 1 || timeout_ms > 10000) return fail(NVFP4_ERR_INVALID_ARG, "timeout_ms must be in [1, 10000]");
  return grouped_gemm_impl(A, SFA, a_gs, B, SFB, b_gs, padded_offsets, nullptr, groups, rows_capacity, N, K, D, ldd,
                           0, stream, 1, (uint64_t)timeout_ms * 1000000ull);
}

int nvfp4_moe_workspace_layout(int64_t T, int64_t H, int64_t I, int E, int top_k, nvfp4_moe_layout* out) {
  if (!out) return fail(NVFP4_ERR_INVALID_ARG, "null layout pointer");
  if (T < 0 || H <= 0 || I <= 0 || E < 1 || E > 256 || top_k < 1 || top_k > 8 || top_k > E)
    return fail(NVFP4_ERR_INVALID_ARG, "bad MoE sizes");
  memset(out, 0, sizeof(*out));
  const int64_t A = T * top_k;
  const int64_t cap = moe_capacity(T, E, top_k);
  const int64_t nb = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  size_t off = 0;
  auto take = [&](int64_t bytes) {
    const size_t at = off;
    off = (size_t)round_up((int64_t)off + (bytes > 0 ? bytes : 0), 1024);
    return at;
  };
  out->status = take(16);  // first, at byte 0: nvfp4_read_device_status finds it from the workspace pointer
  out->topk_ids = take(A * 4);
  out->topk_w = take(A * 4);
  out->block_counts = take(nb * E * 4);
  out->counts = take((int64_t)E * 4);
  out->offsets = take((int64_t)(E + 1) * 4);
  out->meta = take(16);
  out->tile_expert = take(cap / 128 * 4);
  out->sorted_token_ids = take(cap * 4);
  out->row_weight = take(cap * 4);
  out->inverse = take(A * 4);
  out->a1 = take(cap * H / 2);
  out->sfa1 = take(cap * H / 16);
  out->a2 = take(cap * I / 2);
  out->sfa2 = take(cap * I / 16);
  out->y = take(cap * H * 2);
  out->h = take(cap * I * 2);  // bf16 L1 output when the L2 scales come from the batch
  out->calib = take((int64_t)2 * E * 4);
  out->tile_done = take(cap / 128 * 4);
  out->total = off;
  out->capacity = cap;
  out->route_blocks = nb;
  return NVFP4_OK;
}

size_t nvfp4_moe_workspace_size(int64_t T, int64_t H, int64_t I, int E, int top_k) {
  nvfp4_moe_layout L;
  if (nvfp4_moe_workspace_layout(T, H, I, E, top_k, &L) != NVFP4_OK) return 0;
  return L.total;
}

namespace {
// Routing source of a forward: the router's logits over the local experts, or
// (expert parallelism) the model router's global top-k ids and weights.
struct Routing {
  const float* logits;
  const int32_t* topk_ids;
  const float* topk_w;
  int32_t experts_start;
};

int moe_forward_impl(const void* hidden, const Routing& rt, int64_t T, int64_t H, int64_t I, int E, int top_k,
                     const void* w13, const void* w13_sf, const float* w13_gs, const void* w2, const void* w2_sf,
                     const float* w2_gs, const float* a1_gs, const float* a2_gs, float gate_limit, float up_limit,
                     void* workspace, size_t workspace_bytes, void* out, void* stream, bool l1_fp8 = false) {
  g_err[0] = 0;
  if (T < 0) return fail(NVFP4_ERR_INVALID_ARG, "T must be >= 0");
  if (l1_fp8 && a2_gs) return fail(NVFP4_ERR_INVALID_ARG, "the FP8 L1 output takes its L2 scales from the batch");
  if (H <= 0 || H % 256) return fail(NVFP4_ERR_UNSUPPORTED, "H must be a positive multiple of 256");
  if (I <= 0 || I % 128) return fail(NVFP4_ERR_UNSUPPORTED, "I must be a positive multiple of 128");
  if (E < 1 || E > 256) return fail(NVFP4_ERR_UNSUPPORTED, "E must be in [1, 256]");
  if (top_k < 1 || top_k > 8 || top_k > E) return fail(NVFP4_ERR_INVALID_ARG, "top_k must be in [1, min(8, E)]");
  if (!(gate_limit > 0.f) || !(up_limit > 0.f)) return fail(NVFP4_ERR_INVALID_ARG, "limits must be positive");
  nvfp4_moe_layout L;
  if (int rc = nvfp4_moe_workspace_layout(T, H, I, E, top_k, &L)) return rc;
  if (T == 0) return NVFP4_OK;
  if (!hidden || !w13 || !w13_sf || !w13_gs || !w2 || !w2_sf || !w2_gs || !a1_gs || !out ||
      (rt.logits ? false : (!rt.topk_ids || !rt.topk_w)))
    return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(hidden) || !aligned16(w13) || !aligned16(w13_sf) || !aligned16(w2) || !aligned16(w2_sf) ||
      !aligned16(out) || (rt.logits && !aligned16(rt.logits)))
    return fail(NVFP4_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (!workspace || workspace_bytes < L.total)
    return fail(NVFP4_ERR_WORKSPACE, "workspace of %zu bytes needed, got %zu", L.total, workspace_bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(NVFP4_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if ((int64_t)E * 2 * I > INT32_MAX || (int64_t)E * H > INT32_MAX || L.capacity > INT32_MAX)
    return fail(NVFP4_ERR_UNSUPPORTED, "row counts beyond 2^31");
  DeviceInfo* dev = nullptr;
  if (int rc = device_info(&dev)) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  int32_t* ids = (int32_t*)(ws + L.topk_ids);
  float* wts = (float*)(ws + L.topk_w);
  int32_t* bcnt = (int32_t*)(ws + L.block_counts);
  int32_t* counts = (int32_t*)(ws + L.counts);
  int32_t* offsets = (int32_t*)(ws + L.offsets);
  int32_t* meta = (int32_t*)(ws + L.meta);
  int32_t* tile_expert = (int32_t*)(ws + L.tile_expert);
  int32_t* sorted_ids = (int32_t*)(ws + L.sorted_token_ids);
  float* row_w = (float*)(ws + L.row_weight);
  int32_t* inverse = (int32_t*)(ws + L.inverse);
  uint8_t* a1 = ws + L.a1;
  uint8_t* sfa1 = ws + L.sfa1;
  uint8_t* a2 = ws + L.a2;
  uint8_t* sfa2 = ws + L.sfa2;
  uint16_t* ybuf = (uint16_t*)(ws + L.y);
  uint16_t* hbuf = (uint16_t*)(ws + L.h);
  int* status = (int*)(ws + L.status);
  const int64_t cap = L.capacity;
  // No L2 scales given: L1 stores its bf16 SwiGLU output (in the h region)
  // and per-expert amax, and a quantize pass derives the scales from them.
  const bool batch_l2_scale = a2_gs == nullptr;
  uint32_t* l2_amax = (uint32_t*)(ws + L.calib);
  float* l2_gs = (float*)(ws + L.calib) + E;

  GemmArgs g1, g2;
  memset(&g1, 0, sizeof(g1));
  memset(&g2, 0, sizeof(g2));
  if (int rc = make_fp4_map(&g1.tmap_a, a1, cap, H)) return rc;
  if (int rc = make_fp4_map(&g1.tmap_b, w13, (int64_t)E * 2 * I, H)) return rc;
  if (int rc = make_fp4_map(&g2.tmap_a, a2, cap, I)) return rc;
  if (int rc = make_fp4_map(&g2.tmap_b, w2, (int64_t)E * H, I)) return rc;
  if (int rc = make_bf16_store_map(&g2.tmap_y, ybuf, cap, H)) return rc;
  g1.sfa = sfa1;
  g1.sfb = (const uint8_t*)w13_sf;
  g1.padded_offsets = offsets;
  g1.a_gs = a1_gs;
  g1.b_gs = w13_gs;
  g1.G = E;
  g1.K = (int)H;
  g1.num_kb = (int)((H + 255) / 256);
  g1.b_rows_per_group = (int)(2 * I);
  g1.n_tiles = (int)(I / 128);
  g1.b_second_offset = (int)I;
  g1.b_tile_stride = 128;
  g1.sfb_group_bytes = 2 * I * (H / 16);
  g1.q_out = a2;
  g1.q_sf = sfa2;
  g1.q_gs = a2_gs;
  // the h region holds the bf16 h, or the FP8 codes [cap][I] followed by the
  // block exponents [cap][I/16]
  uint8_t* h8 = l1_fp8 ? (uint8_t*)hbuf : nullptr;
  uint8_t* h8_k = l1_fp8 ? (uint8_t*)hbuf + cap * I : nullptr;
  if (batch_l2_scale) {
    g1.D = l1_fp8 ? nullptr : hbuf;
    g1.ldd = I;
    g1.amax_bits = l2_amax;
    g1.h8 = h8;
    g1.h8_k = h8_k;
  }
  g1.I = (int)I;
  g1.gate_limit = gate_limit;
  g1.up_limit = up_limit;
  g1.status = status;
  g1.timeout_ns = 2000000000ull;
  if (g_debug_stall_ms > 0) {
    g1.debug_no_loads = 1;
    g1.timeout_ns = (uint64_t)g_debug_stall_ms * 1000000ull;
  }

  g2.sfa = sfa2;
  g2.sfb = (const uint8_t*)w2_sf;
  g2.padded_offsets = offsets;
  g2.a_gs = batch_l2_scale ? l2_gs : a2_gs;
  g2.b_gs = w2_gs;
  g2.G = E;
  g2.K = (int)I;
  g2.num_kb = (int)((I + 255) / 256);
  g2.b_rows_per_group = (int)H;
  g2.n_tiles = (int)(H / 256);
  g2.b_second_offset = 128;
  g2.b_tile_stride = 256;
  g2.sfb_group_bytes = H * (I / 16);
  g2.y = ybuf;
  g2.sorted_ids = sorted_ids;
  g2.row_w = row_w;
  g2.H = (int)H;
  g2.pair_hint = T * top_k >= (int64_t)256 * E;  // experts average two or more m-tiles
  g2.status = status;
  g2.timeout_ns = 2000000000ull;
  // with given L2 scales the L2 GEMM takes the L1 output m-tile by m-tile (the
  // L2 scales from the batch need the whole L1 output first)
  int* tile_done = batch_l2_scale || !g_l1_l2_overlap ? nullptr : (int*)(ws + L.tile_done);
  g1.tile_done = tile_done;
  g1.late_trigger = tile_done != nullptr;
  g2.tile_done = tile_done;
  g2.tile_done_target = tile_done ? g1.n_tiles : 0;
  if (g_debug_stall_ms > 0) g2.timeout_ns = g1.timeout_ns;  // the stalled L1 never completes its m-tiles

  const int nb = (int)L.route_blocks;
  cudaError_t e;
  stage_mark(0, s);
  if (batch_l2_scale && (e = cudaMemsetAsync(l2_amax, 0, (size_t)E * 4, s)) != cudaSuccess)
    return cuda_fail(e, "amax reset");
  if (T <= kSmallRouteTokens) {  // one block: routing, offsets and slots without launch boundaries
    if ((e = launch_route_small(rt.logits, rt.topk_ids, rt.topk_w, rt.experts_start, T, E, top_k, ids, wts, counts,
                                offsets, meta, tile_expert, sorted_ids, row_w, inverse, status, s)) != cudaSuccess)
      return cuda_fail(e, "route launch");
    stage_mark(1, s);
    stage_mark(2, s);
  } else {
    e = rt.logits ? launch_route_topk(rt.logits, T, E, top_k, ids, wts, bcnt, status, s)
                  : launch_route_external(rt.topk_ids, rt.topk_w, rt.experts_start, T, E, top_k, ids, wts, bcnt,
                                          status, s);
    if (e != cudaSuccess) return cuda_fail(e, "route launch");
    stage_mark(1, s);
    if ((e = launch_slot_scan(bcnt, nb, E, counts, offsets, meta, tile_expert, sorted_ids, row_w, nullptr, 0, s,
                              true)) != cudaSuccess)
      return cuda_fail(e, "slot scan launch");
    stage_mark(2, s);
    if ((e = launch_slot_scatter(ids, wts, T, E, top_k, bcnt, offsets, sorted_ids, row_w, inverse, s, true)) !=
        cudaSuccess)
      return cuda_fail(e, "slot scatter launch");
  }
  stage_mark(3, s);
  if ((e = launch_gather_quantize((const uint16_t*)hidden, H, T, top_k, ids, inverse, counts, offsets, E, a1_gs,
                                  cap, a1, sfa1, s, true, tile_done)) != cudaSuccess)
    return cuda_fail(e, "gather launch");
  stage_mark(4, s);
  const int64_t t1 = cap / 128 * g1.n_tiles, t2 = cap / 128 * g2.n_tiles;
  if ((e = launch_gemm(batch_l2_scale ? kEpiSwigluAmax : kEpiSwigluQuant, g1, (int)t1, dev->sms, s, true)) !=
      cudaSuccess)
    return cuda_fail(e, "L1 launch");
  if (batch_l2_scale &&
      (e = l1_fp8 ? launch_slot_quantize_fp8(h8, h8_k, I, meta, tile_expert, cap, l2_amax, E, l2_gs, a2, sfa2,
                                             dev->sms, s, true)
                  : launch_slot_quantize(hbuf, I, meta, tile_expert, cap, l2_amax, E, l2_gs, a2, sfa2, dev->sms, s,
                                         true)) != cudaSuccess)
    return cuda_fail(e, "L2 activation quantize launch");
  stage_mark(5, s);
  if (g_swap_l2 && !g2.pair_hint && E <= 256) {
    // small batches: W2 tiles as the MMA's M operand, 64 slot rows as N
    SwapArgs sw;
    memset(&sw, 0, sizeof(sw));
    sw.tmap_w = g2.tmap_b;
    if (int rc = make_fp4_map(&sw.tmap_x, a2, cap, I, 64)) return rc;
    sw.sfw = g2.sfb;
    sw.sfx = g2.sfa;
    sw.offsets = offsets;
    sw.counts = counts;
    sw.x_gs = g2.a_gs;
    sw.w_gs = g2.b_gs;
    sw.row_w = row_w;
    sw.y = ybuf;
    sw.G = E;
    sw.K = (int)I;
    sw.num_kb = g2.num_kb;
    sw.H = (int)H;
    sw.n_wtiles = (int)(H / 128);
    sw.sfw_group_bytes = g2.sfb_group_bytes;
    sw.tile_done = g2.tile_done;
    sw.tile_done_target = g2.tile_done_target;
    sw.status = status;
    sw.timeout_ns = g2.timeout_ns;
    if ((e = launch_gemm_swap(sw, dev->sms, s, true)) != cudaSuccess) return cuda_fail(e, "L2 launch");
  } else if ((e = launch_gemm(kEpiCombine, g2, (int)t2, dev->sms, s, true)) != cudaSuccess) {
    return cuda_fail(e, "L2 launch");
  }
  stage_mark(6, s);
  if ((e = launch_token_combine(ybuf, inverse, T, H, top_k, (uint16_t*)out, s, true)) != cudaSuccess)
    return cuda_fail(e, "combine launch");
  stage_mark(7, s);
  return NVFP4_OK;
}

}  // namespace

int nvfp4_moe_forward(const void* hidden, const float* router_logits, int64_t T, int64_t H, int64_t I, int E,
                      int top_k, const void* w13, const void* w13_sf, const float* w13_gs, const void* w2,
                      const void* w2_sf, const float* w2_gs, const float* a1_gs, const float* a2_gs,
                      float gate_limit, float up_limit, void* workspace, size_t workspace_bytes, void* out,
                      void* stream) {
  if (T > 0 && !router_logits) return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
  const Routing rt{router_logits, nullptr, nullptr, 0};
  return moe_forward_impl(hidden, rt, T, H, I, E, top_k, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, a1_gs, a2_gs,
                          gate_limit, up_limit, workspace, workspace_bytes, out, stream);
}

int nvfp4_moe_forward_l1_fp8(const void* hidden, const float* router_logits, int64_t T, int64_t H, int64_t I,
                             int E, int top_k, const void* w13, const void* w13_sf, const float* w13_gs,
                             const void* w2, const void* w2_sf, const float* w2_gs, const float* a1_gs,
                             float gate_limit, float up_limit, void* workspace, size_t workspace_bytes, void* out,
                             void* stream) {
  if (T > 0 && !router_logits) return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
  const Routing rt{router_logits, nullptr, nullptr, 0};
  return moe_forward_impl(hidden, rt, T, H, I, E, top_k, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, a1_gs, nullptr,
                          gate_limit, up_limit, workspace, workspace_bytes, out, stream, true);
}

int nvfp4_moe_forward_routed(const void* hidden, const int32_t* topk_ids, const float* topk_weights,
                             int32_t experts_start, int64_t T, int64_t H, int64_t I, int E, int top_k,
                             const void* w13, const void* w13_sf, const float* w13_gs, const void* w2,
                             const void* w2_sf, const float* w2_gs, const float* a1_gs, const float* a2_gs,
                             float gate_limit, float up_limit, void* workspace, size_t workspace_bytes, void* out,
                             void* stream) {
  if (T > 0 && (!topk_ids || !topk_weights)) return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
  const Routing rt{nullptr, topk_ids, topk_weights, experts_start};
  return moe_forward_impl(hidden, rt, T, H, I, E, top_k, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, a1_gs, a2_gs,
                          gate_limit, up_limit, workspace, workspace_bytes, out, stream);
}

// ------------------------------------------------------------------ shared expert
namespace {
struct SharedExpertLayout {
  size_t status, a1, sfa1, a2, sfa2, total;
  int64_t rows;  // T rounded up to 128
};
SharedExpertLayout shared_expert_layout(int64_t T, int64_t H, int64_t I) {
  SharedExpertLayout L;
  L.rows = round_up(T > 0 ? T : 1, 128);
  size_t off = 0;
  auto take = [&](int64_t bytes) {
    const size_t at = off;
    off = (size_t)round_up((int64_t)off + bytes, 1024);
    return at;
  };
  L.status = take(16);  // byte 0, as in the MoE forward's workspace
  L.a1 = take(L.rows * H / 2);
  L.sfa1 = take(L.rows * H / 16);
  L.a2 = take(L.rows * I / 2);
  L.sfa2 = take(L.rows * I / 16);
  L.total = off;
  return L;
}
}  // namespace

size_t nvfp4_shared_expert_workspace_size(int64_t T, int64_t H, int64_t I) {
  if (T < 0 || H <= 0 || I <= 0) return 0;
  return shared_expert_layout(T, H, I).total;
}

int nvfp4_shared_expert_forward(const void* hidden, int64_t T, int64_t H, int64_t I, const void* w13,
                                const void* w13_sf, const float* w13_gs, const void* w2, const void* w2_sf,
                                const float* w2_gs, const float* a1_gs, const float* a2_gs, float gate_limit,
                                float up_limit, void* workspace, size_t workspace_bytes, void* out, void* stream) {
  g_err[0] = 0;
  if (T < 0) return fail(NVFP4_ERR_INVALID_ARG, "T must be >= 0");
  if (H <= 0 || H % 256) return fail(NVFP4_ERR_UNSUPPORTED, "H must be a positive multiple of 256");
  if (I <= 0 || I % 128) return fail(NVFP4_ERR_UNSUPPORTED, "I must be a positive multiple of 128");
  if (!(gate_limit > 0.f) || !(up_limit > 0.f)) return fail(NVFP4_ERR_INVALID_ARG, "limits must be positive");
  if (T == 0) return NVFP4_OK;
  if (!hidden || !w13 || !w13_sf || !w13_gs || !w2 || !w2_sf || !w2_gs || !a1_gs || !a2_gs || !out)
    return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(hidden) || !aligned16(w13) || !aligned16(w13_sf) || !aligned16(w2) || !aligned16(w2_sf) ||
      !aligned16(out))
    return fail(NVFP4_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  const SharedExpertLayout L = shared_expert_layout(T, H, I);
  if (!workspace || workspace_bytes < L.total)
    return fail(NVFP4_ERR_WORKSPACE, "workspace of %zu bytes needed, got %zu", L.total, workspace_bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(NVFP4_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (L.rows > INT32_MAX || 2 * I > INT32_MAX) return fail(NVFP4_ERR_UNSUPPORTED, "row counts beyond 2^31");
  DeviceInfo* dev = nullptr;
  if (int rc = device_info(&dev)) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  uint8_t* a1 = ws + L.a1;
  uint8_t* sfa1 = ws + L.sfa1;
  uint8_t* a2 = ws + L.a2;
  uint8_t* sfa2 = ws + L.sfa2;
  int* status = (int*)(ws + L.status);
  GemmArgs g1, g2;
  memset(&g1, 0, sizeof(g1));
  memset(&g2, 0, sizeof(g2));
  if (int rc = make_fp4_map(&g1.tmap_a, a1, L.rows, H)) return rc;
  if (int rc = make_fp4_map(&g1.tmap_b, w13, 2 * I, H)) return rc;
  if (int rc = make_fp4_map(&g2.tmap_a, a2, L.rows, I)) return rc;
  if (int rc = make_fp4_map(&g2.tmap_b, w2, H, I)) return rc;
  // L1: one group, SwiGLU + requantization into A2 (gate rows 0..I-1, up rows I..2I-1)
  g1.sfa = sfa1;
  g1.sfb = (const uint8_t*)w13_sf;
  g1.a_gs = a1_gs;
  g1.b_gs = w13_gs;
  g1.G = 1;
  g1.host_rows = (int)L.rows;
  g1.K = (int)H;
  g1.num_kb = (int)((H + 255) / 256);
  g1.b_rows_per_group = (int)(2 * I);
  g1.n_tiles = (int)(I / 128);
  g1.b_second_offset = (int)I;
  g1.b_tile_stride = 128;
  g1.sfb_group_bytes = 2 * I * (H / 16);
  g1.q_out = a2;
  g1.q_sf = sfa2;
  g1.q_gs = a2_gs;
  g1.I = (int)I;
  g1.gate_limit = gate_limit;
  g1.up_limit = up_limit;
  g1.status = status;
  g1.timeout_ns = 2000000000ull;
  // L2: one group, bf16 rows straight into out (rows >= T not stored)
  g2.sfa = sfa2;
  g2.sfb = (const uint8_t*)w2_sf;
  g2.a_gs = a2_gs;
  g2.b_gs = w2_gs;
  g2.G = 1;
  g2.host_rows = (int)L.rows;
  g2.host_count = (int)T;
  g2.K = (int)I;
  g2.num_kb = (int)((I + 255) / 256);
  g2.b_rows_per_group = (int)H;
  g2.n_tiles = (int)(H / 256);
  g2.b_second_offset = 128;
  g2.b_tile_stride = 256;
  g2.sfb_group_bytes = H * (I / 16);
  g2.D = (uint16_t*)out;
  g2.ldd = H;
  g2.d_vec32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
  g2.status = status;
  g2.timeout_ns = 2000000000ull;
  cudaError_t e;
  if ((e = launch_quantize((const uint16_t*)hidden, T, H, H, 0, 1, a1_gs, nullptr, a1, sfa1, L.rows, dev->sms, s,
                           status)) != cudaSuccess)
    return cuda_fail(e, "quantize launch");
  const int64_t t1 = L.rows / 128 * g1.n_tiles, t2 = L.rows / 128 * g2.n_tiles;
  if ((e = launch_gemm(kEpiSwigluQuant, g1, (int)t1, dev->sms, s, true)) != cudaSuccess)
    return cuda_fail(e, "L1 launch");
  if ((e = launch_gemm(kEpiBf16, g2, (int)t2, dev->sms, s, true)) != cudaSuccess) return cuda_fail(e, "L2 launch");
  return NVFP4_OK;
}

namespace {

int calibrate_impl(const void* hidden, const Routing& rt, int64_t T, int64_t H, int64_t I, int E, int top_k,
                   const void* w13, const void* w13_sf, const float* w13_gs, float gate_limit, float up_limit,
                   void* workspace, size_t workspace_bytes, float* a1_gs_out, float* a2_gs_out, void* stream) {
  g_err[0] = 0;
  if (T < 0) return fail(NVFP4_ERR_INVALID_ARG, "T must be >= 0");
  if (H <= 0 || H % 256) return fail(NVFP4_ERR_UNSUPPORTED, "H must be a positive multiple of 256");
  if (I <= 0 || I % 128) return fail(NVFP4_ERR_UNSUPPORTED, "I must be a positive multiple of 128");
  if (E < 1 || E > 256) return fail(NVFP4_ERR_UNSUPPORTED, "E must be in [1, 256]");
  if (top_k < 1 || top_k > 8 || top_k > E) return fail(NVFP4_ERR_INVALID_ARG, "top_k must be in [1, min(8, E)]");
  if (!(gate_limit > 0.f) || !(up_limit > 0.f)) return fail(NVFP4_ERR_INVALID_ARG, "limits must be positive");
  nvfp4_moe_layout L;
  if (int rc = nvfp4_moe_workspace_layout(T, H, I, E, top_k, &L)) return rc;
  if (!a1_gs_out || !a2_gs_out) return fail(NVFP4_ERR_INVALID_ARG, "null output pointer");
  if (T > 0 && (!hidden || !w13 || !w13_sf || !w13_gs || (rt.logits ? false : (!rt.topk_ids || !rt.topk_w))))
    return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(hidden) || !aligned16(w13) || !aligned16(w13_sf) || (rt.logits && !aligned16(rt.logits)))
    return fail(NVFP4_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (!workspace || workspace_bytes < L.total)
    return fail(NVFP4_ERR_WORKSPACE, "workspace of %zu bytes needed, got %zu", L.total, workspace_bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(NVFP4_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if ((int64_t)E * 2 * I > INT32_MAX || L.capacity > INT32_MAX)
    return fail(NVFP4_ERR_UNSUPPORTED, "row counts beyond 2^31");
  DeviceInfo* dev = nullptr;
  if (int rc = device_info(&dev)) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  int32_t* ids = (int32_t*)(ws + L.topk_ids);
  float* wts = (float*)(ws + L.topk_w);
  int32_t* bcnt = (int32_t*)(ws + L.block_counts);
  int32_t* counts = (int32_t*)(ws + L.counts);
  int32_t* offsets = (int32_t*)(ws + L.offsets);
  int32_t* meta = (int32_t*)(ws + L.meta);
  int32_t* tile_expert = (int32_t*)(ws + L.tile_expert);
  int32_t* sorted_ids = (int32_t*)(ws + L.sorted_token_ids);
  float* row_w = (float*)(ws + L.row_weight);
  int32_t* inverse = (int32_t*)(ws + L.inverse);
  uint8_t* a1 = ws + L.a1;
  uint8_t* sfa1 = ws + L.sfa1;
  uint32_t* amax = (uint32_t*)(ws + L.calib);
  int* status = (int*)(ws + L.status);
  const int64_t cap = L.capacity;
  cudaError_t e;
  if (T == 0) {  // no rows: every expert gets gs 1
    if ((e = cudaMemsetAsync(status, 0, sizeof(int), s)) != cudaSuccess ||
        (e = launch_slot_scan(bcnt, 0, E, counts, offsets, meta, tile_expert, sorted_ids, row_w, amax, 2 * E, s)) !=
            cudaSuccess ||
        (e = launch_gs_from_amax(amax, E, a1_gs_out, s)) != cudaSuccess ||
        (e = launch_gs_from_amax(amax + E, E, a2_gs_out, s)) != cudaSuccess)
      return cuda_fail(e, "calibration launch");
    return NVFP4_OK;
  }
  GemmArgs g1;
  memset(&g1, 0, sizeof(g1));
  if (int rc = make_fp4_map(&g1.tmap_a, a1, cap, H)) return rc;
  if (int rc = make_fp4_map(&g1.tmap_b, w13, (int64_t)E * 2 * I, H)) return rc;
  g1.sfa = sfa1;
  g1.sfb = (const uint8_t*)w13_sf;
  g1.padded_offsets = offsets;
  g1.a_gs = a1_gs_out;
  g1.b_gs = w13_gs;
  g1.G = E;
  g1.K = (int)H;
  g1.num_kb = (int)((H + 255) / 256);
  g1.b_rows_per_group = (int)(2 * I);
  g1.n_tiles = (int)(I / 128);
  g1.b_second_offset = (int)I;
  g1.b_tile_stride = 128;
  g1.sfb_group_bytes = 2 * I * (H / 16);
  g1.I = (int)I;
  g1.gate_limit = gate_limit;
  g1.up_limit = up_limit;
  g1.amax_bits = amax + E;
  g1.status = status;
  g1.timeout_ns = 2000000000ull;
  const int nb = (int)L.route_blocks;
  if ((e = rt.logits ? launch_route_topk(rt.logits, T, E, top_k, ids, wts, bcnt, status, s)
                     : launch_route_external(rt.topk_ids, rt.topk_w, rt.experts_start, T, E, top_k, ids, wts, bcnt,
                                             status, s)) != cudaSuccess ||
      (e = launch_slot_scan(bcnt, nb, E, counts, offsets, meta, tile_expert, sorted_ids, row_w, amax, 2 * E, s)) !=
          cudaSuccess ||
      (e = launch_slot_scatter(ids, wts, T, E, top_k, bcnt, offsets, sorted_ids, row_w, inverse, s)) !=
          cudaSuccess ||
      (e = launch_gather_amax((const uint16_t*)hidden, H, sorted_ids, tile_expert, meta, cap, amax, dev->sms, s)) !=
          cudaSuccess ||
      (e = launch_gs_from_amax(amax, E, a1_gs_out, s)) != cudaSuccess ||
      (e = launch_gather_quantize((const uint16_t*)hidden, H, T, top_k, ids, inverse, counts, offsets, E,
                                  a1_gs_out, cap, a1, sfa1, s)) != cudaSuccess)
    return cuda_fail(e, "calibration launch");
  const int64_t t1 = cap / 128 * g1.n_tiles;
  if ((e = launch_gemm(kEpiSwigluAmax, g1, (int)t1, dev->sms, s)) != cudaSuccess ||
      (e = launch_gs_from_amax(amax + E, E, a2_gs_out, s)) != cudaSuccess)
    return cuda_fail(e, "calibration launch");
  return NVFP4_OK;
}

}  // namespace

int nvfp4_moe_calibrate(const void* hidden, const float* router_logits, int64_t T, int64_t H, int64_t I, int E,
                        int top_k, const void* w13, const void* w13_sf, const float* w13_gs, float gate_limit,
                        float up_limit, void* workspace, size_t workspace_bytes, float* a1_gs_out, float* a2_gs_out,
                        void* stream) {
  if (T > 0 && !router_logits) return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
  const Routing rt{router_logits, nullptr, nullptr, 0};
  return calibrate_impl(hidden, rt, T, H, I, E, top_k, w13, w13_sf, w13_gs, gate_limit, up_limit, workspace,
                        workspace_bytes, a1_gs_out, a2_gs_out, stream);
}

int nvfp4_moe_calibrate_routed(const void* hidden, const int32_t* topk_ids, const float* topk_weights,
                               int32_t experts_start, int64_t T, int64_t H, int64_t I, int E, int top_k,
                               const void* w13, const void* w13_sf, const float* w13_gs, float gate_limit,
                               float up_limit, void* workspace, size_t workspace_bytes, float* a1_gs_out,
                               float* a2_gs_out, void* stream) {
  if (T > 0 && (!topk_ids || !topk_weights)) return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
  const Routing rt{nullptr, topk_ids, topk_weights, experts_start};
  return calibrate_impl(hidden, rt, T, H, I, E, top_k, w13, w13_sf, w13_gs, gate_limit, up_limit, workspace,
                        workspace_bytes, a1_gs_out, a2_gs_out, stream);
}

int nvfp4_gemm_set_cta_pair(int mode, int* prev_mode) {
  g_err[0] = 0;
  if (mode < 0 || mode > 2) return fail(NVFP4_ERR_INVALID_ARG, "mode must be 0, 1 or 2");
  const int prev = gemm_set_pair_mode(mode);
  if (prev_mode) *prev_mode = prev;
  return NVFP4_OK;
}

int nvfp4_moe_set_swap_l2(int enable, int* prev_enable) {
  g_err[0] = 0;
  if (enable != 0 && enable != 1) return fail(NVFP4_ERR_INVALID_ARG, "enable must be 0 or 1");
  if (prev_enable) *prev_enable = g_swap_l2;
  g_swap_l2 = enable;
  return NVFP4_OK;
}

int nvfp4_device_status(int* status_out, int reset) {
  g_err[0] = 0;
  if (!status_out) return fail(NVFP4_ERR_INVALID_ARG, "null status pointer");
  DeviceInfo* dev = nullptr;
  if (int rc = device_info(&dev)) return rc;
  cudaError_t e = gemm_read_status(status_out, reset);
  return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "status read");
}

int nvfp4_read_device_status(const void* workspace, void* stream, int* status_out, int reset) {
  g_err[0] = 0;
  if (!workspace || !status_out) return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(NVFP4_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  DeviceInfo* dev = nullptr;
  if (int rc = device_info(&dev)) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && reset) {
    e = cudaMemsetAsync(const_cast<void*>(workspace), 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *status_out = v;
  return NVFP4_OK;
}

int nvfp4_debug_gemm_trace(void* buffer, int stages, int tiles, int kind) {
  g_err[0] = 0;
  if (!buffer) {
    gemm_set_trace(nullptr, 0, 0, -1);
    return NVFP4_OK;
  }
  const int k = kind & 0xFF, cta = kind >> 8;  // bits 8 and up: the CTA to record
  if (kind < 0 || k > 4 || cta > 4095 || (k == 4 && cta) || stages < 0 || tiles < 0 || (int64_t)(stages + tiles) * 8 > (int64_t)1 << 28)
    return fail(NVFP4_ERR_INVALID_ARG, "kind must be 0..4 (+ 256 * CTA) and the buffer at most 2^28 words");
  if (k < 4 && !gemm_trace_built())
    return fail(NVFP4_ERR_UNSUPPORTED, "GEMM timelines need a build with -DNVFP4_GEMM_TRACE");
  if (reinterpret_cast<uintptr_t>(buffer) & 7u) return fail(NVFP4_ERR_INVALID_ARG, "buffer must be 8-byte aligned");
  gemm_set_trace(static_cast<unsigned long long*>(buffer), stages, tiles, kind);
  return NVFP4_OK;
}

int nvfp4_moe_set_overlap(int enable, int* prev) {
  g_err[0] = 0;
  if (enable != 0 && enable != 1) return fail(NVFP4_ERR_INVALID_ARG, "enable must be 0 or 1");
  if (prev) *prev = g_l1_l2_overlap;
  g_l1_l2_overlap = enable;
  return NVFP4_OK;
}

int nvfp4_moe_set_debug_stall(int timeout_ms) {
  g_err[0] = 0;
  if (timeout_ms < 0 || timeout_ms > 10000) return fail(NVFP4_ERR_INVALID_ARG, "timeout_ms must be in [0, 10000]");
  g_debug_stall_ms = timeout_ms;
  return NVFP4_OK;
}

int nvfp4_moe_set_stage_events(void* const* events, int n_events) {
  g_err[0] = 0;
  if (n_events == 0) {
    g_n_stage_events = 0;
    memset(g_stage_events, 0, sizeof(g_stage_events));
    return NVFP4_OK;
  }
  if (n_events != 8 || !events) return fail(NVFP4_ERR_INVALID_ARG, "n_events must be 8 (or 0)");
  for (int i = 0; i < 8; ++i) g_stage_events[i] = events[i];
  g_n_stage_events = 8;
  return NVFP4_OK;
}

}  // extern "C"
