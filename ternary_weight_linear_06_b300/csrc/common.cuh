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

// Per-token quantization of one value, clamp(rint(fp32(fp32(x*127)/m)), -128,
// 127), for |x| <= m (m is the row's absmax or eps): returned as the integer
// code in fp32. The clamp never binds then: |fp32(x*127)| <= fp32(127 m) <=
// 127 m (1 + 2^-24), so the quotient rounds to at most 127 in magnitude.
// s127 = fp32(127 * fp32(1/m)). The product c = fp32(x * s127) carries three
// roundings of relative size 2^-24, so it lies within 127 * 3 * 2^-24 <
// 2.3e-5 of the real 127 x / m, and the defined quotient within 1.2e-5 of it
// (one rounding of x * 127, one of the division, each at most half an fp32
// step of a value below 128). Both round to the same integer unless c is
// within 3.5e-5 of a half-integer; within 1e-4 of one (about one value in
// 5000) the defined division decides.
__device__ __forceinline__ float quant_round(float x, float m, float s127) {
  const float c = __fmul_rn(x, s127);
  float r = rintf(c);
  if (fabsf(__fsub_rn(c, r)) > 0.4999f) r = rintf(__fdiv_rn(__fmul_rn(x, 127.0f), m));
  return r;
}

// Adding 1.5 * 2^23 to an integer-valued float of magnitude below 2^22 puts
// the integer, in two's complement, in the low bits of the result.
constexpr float kIntShift = 12582912.0f;

// Load 16 consecutive activations of one row (fp32, or bf16 widened exactly).
template <int DT>
__device__ __forceinline__ void load16(const void* row, int g, float (&v)[16]) {
  if constexpr (DT == BL_DTYPE_F32) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(row) + 16 * g);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 u = __ldg(p + i);
      v[4 * i + 0] = __uint_as_float(u.x);
      v[4 * i + 1] = __uint_as_float(u.y);
      v[4 * i + 2] = __uint_as_float(u.z);
      v[4 * i + 3] = __uint_as_float(u.w);
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(row) + 16 * g);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 u = __ldg(p + i);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * i + 2 * j + 0] = __uint_as_float(w[j] << 16);          // exact bf16 -> fp32
        v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d) {
  return (static_cast<uint32_t>(a) & 0xFFu) | ((static_cast<uint32_t>(b) & 0xFFu) << 8) |
         ((static_cast<uint32_t>(c) & 0xFFu) << 16) | ((static_cast<uint32_t>(d) & 0xFFu) << 24);
}

__device__ __forceinline__ uint32_t pack_h2(int lo, int hi) {
  const __half2 h = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// L2 prefetch of a byte range (16-byte aligned start and size), one thread.
__device__ __forceinline__ void prefetch_l2(const void* p, size_t bytes) {
  const char* c = static_cast<const char*>(p);
  while (bytes > 0) {
    const uint32_t n = static_cast<uint32_t>(bytes < (1u << 20) ? bytes : (1u << 20));
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c), "r"(n) : "memory");
    c += n;
    bytes -= n;
  }
}

// ---------------------------------------------------------------------------
// Shared-memory barriers and bulk copies (TMA engine), inline PTX.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Make barrier initialisation visible to the async proxy (bulk copies, MMA).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Order this thread's earlier generic shared-memory accesses before later
// async-proxy accesses (a bulk copy that overwrites a buffer just read).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Wait for a barrier phase, giving up at `deadline` (globaltimer ns).
__device__ __forceinline__ bool mbar_wait_until(uint64_t* bar, uint32_t parity, uint64_t deadline) {
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() > deadline) return false;
  }
  return true;
}
// Global -> shared bulk copy completing on `bar` (bytes and addresses 16-aligned).
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Upper bound on any device-side wait before it reports BL_ERR_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

}  // namespace bl
