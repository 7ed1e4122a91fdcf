// Shared device helpers for the nanochat step kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nc {

typedef __nv_bfloat16 bf16;

// Device status word codes (first failure wins; kernels never trap).
enum DevStatus : int {
  DEV_OK = 0,
  DEV_BAD_TOKEN = 1,   // a token or target id outside [0, vocab)
  DEV_TIMEOUT = 2,     // an mbarrier / pipeline wait exceeded its limit
  DEV_BAD_LAUNCH = 3,  // a kernel found a launch shape it cannot serve
};

__device__ __forceinline__ void set_status(int* st, int code) {
  if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const bf16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float v) { *p = v; }
__device__ __forceinline__ void stf(bf16* p, float v) { *p = __float2bfloat16_rn(v); }

// Value after a round trip through the storage type (identity for fp32).
__device__ __forceinline__ float rnd(float v, const float*) { return v; }
__device__ __forceinline__ float rnd(float v, const bf16*) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

constexpr float kEps = 1e-6f;     // RMSNorm epsilon, inside the square root
constexpr int kHeadDim = 128;     // fixed head width
constexpr int kHalf = 64;         // RoPE pairs dim j with dim j + 64

}  // namespace nc
