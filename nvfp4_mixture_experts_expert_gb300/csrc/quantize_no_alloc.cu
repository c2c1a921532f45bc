// nvfp4_quantize_no_alloc: nvfp4_quantize with the global scale computed on
// the device, for callers that cannot hand the library any scratch memory.
//
// Some hosts own every byte of device memory and expose no way to obtain a
// temporary buffer: an inference server that reserves its whole memory pool
// up front, or a plugin interface whose call signature has inputs and outputs
// but no workspace.  Such callers cannot call cudaMalloc themselves and
// cannot let a library call it either.  This entry point therefore keeps the
// per-group partial maxima of the amax reduction in a fixed array that lives
// in the library's own device image: it is part of the module's global
// memory on every GPU that loads the library and stays there until the
// process exits.  Limit: at most kNoAllocMaxGroups groups per call.
//
// Sharing rules.  All calls on a device use the same array.  Every call
// rewrites each slot it later reads (one partial per reduction block), so no
// slot has to start at zero and nothing carries over from one call to the
// next.  Calls whose kernels overlap on the GPU (different streams with no
// ordering between them) race on the array and give wrong scales; order them
// on one stream, or use nvfp4_quantize with a workspace of your own.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "../../include/nvfp4moe.h"
#include "internal.h"

namespace {

constexpr int kNoAllocMaxGroups = NVFP4_QUANTIZE_NO_ALLOC_MAX_GROUPS;

static __device__ __align__(256) float g_no_alloc_amax_partials[kNoAllocMaxGroups * nvfp4::kAmaxBlocksPerGroup];

constexpr int kMaxDevices = 64;
// Per device: the scratch address and the id of the CUDA context it was
// looked up in.  A context id is unique for the life of the process, so after
// cudaDeviceReset (a new primary context, the module loaded again at another
// address) the next call sees a different id and looks the address up anew.
struct ScratchEntry {
  float* addr = nullptr;
  unsigned long long ctx_id = 0;
};
ScratchEntry g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// Failures are reported through the library's nvfp4_last_error().
int fail(int code, const char* fmt, ...) {
  char msg[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, sizeof(msg), fmt, ap);
  va_end(ap);
  nvfp4::set_last_error(msg);
  return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Id of the calling thread's current CUDA context (driver entry points
// fetched through the runtime, so the library does not link libcuda).
int current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return fail(NVFP4_ERR_CUDA, "driver context entry points unavailable");
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return fail(NVFP4_ERR_CUDA, "no current CUDA context");
  if (get_id(ctx, id) != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuCtxGetId failed");
  return NVFP4_OK;
}

// Device address of the scratch array on the current device.  The symbol's
// host-side name is only a stand-in, so the address is looked up with the
// device current, once per device and context, and cached.
int scratch_on_current_device(float** out, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(NVFP4_ERR_DEVICE, "device index %d out of range", dev);
  int major = 0, minor = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return fail(NVFP4_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  if (major != 10 || minor != 3)
    return fail(NVFP4_ERR_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev, major, minor);
  // cudaSetDevice initialises the device's primary context and makes it
  // current (it already is: dev is the current device), so it has an id
  if ((e = cudaSetDevice(dev)) != cudaSuccess)
    return fail(NVFP4_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(e));
  unsigned long long ctx_id = 0;
  if (int rc = current_context_id(&ctx_id)) return rc;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchEntry& ent = g_scratch[dev];
  if (!ent.addr || ent.ctx_id != ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_no_alloc_amax_partials);
    if (e != cudaSuccess || !p)
      return fail(NVFP4_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
    ent.addr = static_cast<float*>(p);
    ent.ctx_id = ctx_id;
  }
  *out = ent.addr;
  return NVFP4_OK;
}

}  // namespace

extern "C" {

int nvfp4_quantize_no_alloc(const void* x, int64_t rows, int64_t K, int64_t ld_x, int64_t group_stride_x,
                            int groups, float* gs_out, void* fp4, void* sf, int64_t rows_padded, void* stream) {
  nvfp4::set_last_error("");
  if (groups < 1) return fail(NVFP4_ERR_INVALID_ARG, "groups must be >= 1");
  if (groups > kNoAllocMaxGroups)
    return fail(NVFP4_ERR_UNSUPPORTED, "nvfp4_quantize_no_alloc handles at most %d groups per call (got %d)",
                kNoAllocMaxGroups, groups);
  if (K <= 0 || K % 64) return fail(NVFP4_ERR_INVALID_ARG, "K must be a positive multiple of 64");
  if (rows < 0 || rows_padded < rows || rows_padded % 128)
    return fail(NVFP4_ERR_INVALID_ARG, "need 0 <= rows <= rows_padded and rows_padded % 128 == 0");
  if (ld_x < K || ld_x % 8 || group_stride_x < 0 || group_stride_x % 8)
    return fail(NVFP4_ERR_INVALID_ARG, "ld_x must be >= K and both strides multiples of 8 elements");
  if (!gs_out) return fail(NVFP4_ERR_INVALID_ARG, "gs_out is required");
  if ((rows > 0 && !x) || (rows_padded > 0 && (!fp4 || !sf))) return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(x) || !aligned16(fp4) || !aligned16(sf) || !aligned16(gs_out))
    return fail(NVFP4_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  float* scratch = nullptr;
  int sms = 0;
  if (int rc = scratch_on_current_device(&scratch, &sms)) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = nvfp4::launch_group_amax((const uint16_t*)x, rows, K, ld_x, group_stride_x, groups, scratch,
                                           rows_padded > 0 ? nullptr : gs_out, sms, s);
  if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "amax launch: %s", cudaGetErrorString(e));
  if (rows_padded > 0 &&
      (e = nvfp4::launch_quantize((const uint16_t*)x, rows, K, ld_x, group_stride_x, groups, nullptr, gs_out,
                                  (uint8_t*)fp4, (uint8_t*)sf, rows_padded, sms, s, nullptr, scratch)) != cudaSuccess)
    return fail(NVFP4_ERR_CUDA, "quantize launch: %s", cudaGetErrorString(e));
  return NVFP4_OK;
}

}  // extern "C"
