// Test-only probe: checks, on the device, the two conversion primitives the
// NVFP4 kernels rely on (it includes the library's own device header).
//  1. div_by_scale(x, d, rcp.rn(d)) == IEEE x / d for every E4M3 scale value d
//     and every fp32 mantissa of x, over several binades and both signs.
//  2. e2m1x2_code(lo, hi) == code(lo) | code(hi) << 4, where code(v) is the
//     lane-order-independent single conversion cvt(v, v) & 0xF.
//  3. e2m1x8_word(q0..q7) == sum over j of e2m1x2_code(q2j, q2j+1) << 8j.
#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_format.cuh"

using namespace nvfp4;

__global__ void div_probe_kernel(int exp_bias, unsigned long long* mismatches) {
  const uint32_t m = blockIdx.x * blockDim.x + threadIdx.x;  // fp32 mantissa bits
  if (m >= (1u << 23)) return;
  unsigned long long bad = 0;
  for (int sign = 0; sign < 2; ++sign) {
    const float x = __uint_as_float(((uint32_t)sign << 31) | ((uint32_t)(127 + exp_bias) << 23) | m);
    for (uint32_t code = 1; code < 0x7F; ++code) {
      const float d = e4m3_value(code);
      const float q = div_by_scale(x, d, __frcp_rn(d));
      const float r = __fdiv_rn(x, d);
      bad += __float_as_uint(q) != __float_as_uint(r);
    }
  }
  if (bad) atomicAdd(mismatches, bad);
}

__global__ void e2m1_pair_probe_kernel(const float* v, int n, unsigned int* mismatches) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n * n) return;
  const float lo = v[i / n], hi = v[i % n];
  const uint32_t one_lo = e2m1x2_code(lo, lo) & 0xFu, one_hi = e2m1x2_code(hi, hi) & 0xFu;
  const uint32_t pair = e2m1x2_code(lo, hi);
  if (pair != (one_lo | (one_hi << 4))) atomicAdd(mismatches, 1u);
}

__global__ void e2m1_word_probe_kernel(const float* v, int n, unsigned int* mismatches) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float q[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) q[j] = v[(i * 7 + j * 13) % n];
  uint32_t ref = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) ref |= e2m1x2_code(q[2 * j], q[2 * j + 1]) << (8 * j);
  if (e2m1x8_word(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]) != ref) atomicAdd(mismatches, 1u);
}

extern "C" int run_div_probe(int exp_bias, unsigned long long* host_mismatches) {
  unsigned long long* d = nullptr;
  if (cudaMalloc(&d, sizeof(*d)) != cudaSuccess) return 1;
  cudaMemset(d, 0, sizeof(*d));
  div_probe_kernel<<<(1 << 23) / 256, 256>>>(exp_bias, d);
  cudaError_t e = cudaMemcpy(host_mismatches, d, sizeof(*d), cudaMemcpyDeviceToHost);
  cudaFree(d);
  return e == cudaSuccess ? 0 : 2;
}

extern "C" int run_e2m1_pair_probe(const float* host_values, int n, unsigned int* host_mismatches) {
  float* dv = nullptr;
  unsigned int* dm = nullptr;
  if (cudaMalloc(&dv, n * sizeof(float)) != cudaSuccess || cudaMalloc(&dm, sizeof(unsigned int)) != cudaSuccess)
    return 1;
  cudaMemcpy(dv, host_values, n * sizeof(float), cudaMemcpyHostToDevice);
  cudaMemset(dm, 0, sizeof(unsigned int));
  e2m1_pair_probe_kernel<<<(n * n + 255) / 256, 256>>>(dv, n, dm);
  cudaError_t e = cudaMemcpy(host_mismatches, dm, sizeof(unsigned int), cudaMemcpyDeviceToHost);
  cudaFree(dv);
  cudaFree(dm);
  return e == cudaSuccess ? 0 : 2;
}

extern "C" int run_e2m1_word_probe(const float* host_values, int n, unsigned int* host_mismatches) {
  float* dv = nullptr;
  unsigned int* dm = nullptr;
  if (cudaMalloc(&dv, n * sizeof(float)) != cudaSuccess || cudaMalloc(&dm, sizeof(unsigned int)) != cudaSuccess)
    return 1;
  cudaMemcpy(dv, host_values, n * sizeof(float), cudaMemcpyHostToDevice);
  cudaMemset(dm, 0, sizeof(unsigned int));
  e2m1_word_probe_kernel<<<(n + 255) / 256, 256>>>(dv, n, dm);
  cudaError_t e = cudaMemcpy(host_mismatches, dm, sizeof(unsigned int), cudaMemcpyDeviceToHost);
  cudaFree(dv);
  cudaFree(dm);
  return e == cudaSuccess ? 0 : 2;
}
