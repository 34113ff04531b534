// Shared device helpers for the BitLinear kernels (sm_103a only).
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "bitlinear.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "this library is written for sm_103a only"
#endif

namespace bl {

// ---------------------------------------------------------------------------
// Workspace header: the first 256 bytes of every workspace.
// ---------------------------------------------------------------------------
struct WsHeader {
  uint32_t status;     // 0 = ok, else a bl_status written by a device-side check
  uint32_t info;       // where the check fired (kernel-specific code)
  uint32_t pad[62];
};
static_assert(sizeof(WsHeader) == 256, "workspace header must be 256 bytes");

constexpr int kWarp = 32;
constexpr int kMaxK = 65536;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Record a device-side failure in the sticky status word (first writer wins).
__device__ inline void report_status(WsHeader* h, uint32_t status, uint32_t info) {
  if (h != nullptr && atomicCAS(&h->status, 0u, status) == 0u) atomicExch(&h->info, info);
}

// ---------------------------------------------------------------------------
// Integer dot product of 4 signed activation bytes with 4 unsigned code bytes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int dp4a_su(int a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// 128-bit streaming load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_sum(int v) { return __reduce_add_sync(0xffffffffu, v); }

// Programmatic dependent launch controls (no-ops when launched without PDL).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Dequant factor of one token: fp32(fp32(s_w * m) / 127).
__device__ __forceinline__ float dequant_factor(float s_w, float m) {
  return __fdiv_rn(__fmul_rn(s_w, m), 127.0f);
}

// Per-token quantization of one value: clamp(rint(fp32(fp32(x*127)/m)), -128, 127).
__device__ __forceinline__ int quant_one(float x, float m) {
  float r = rintf(__fdiv_rn(__fmul_rn(x, 127.0f), m));
  r = fminf(fmaxf(r, -128.0f), 127.0f);
  return __float2int_rn(r);
}

}  // namespace bl
