// Host-side launchers of the BitLinear kernels. Each returns cudaSuccess or
// the launch error; argument checking happens in the C ABI layer.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace bl {

struct WsHeader;

// ----- weight packing ------------------------------------------------------
// Workspace bytes the pack needs past the 256-byte header.
size_t pack_scratch_bytes();
cudaError_t launch_pack(const float* W, int N, int K, float eps, uint8_t* packed, float* s_w,
                        void* workspace, cudaStream_t st);
cudaError_t launch_unpack(const uint8_t* packed, int N, int K, int8_t* t, cudaStream_t st);

// ----- activation quantization ---------------------------------------------
enum class QLayout : int {
  kRowMajorI8 = 0,   // q[m][k] int8 (public layout, read by the GEMV)
  kPairF16 = 2,      // per 16 columns: fp16 slot s holds column (s>>1) + 8*(s&1) (MMA order)
};
// X: [M][K] fp32 or bf16. m_out [M] fp32, qsum_out [M] int32 (may be null).
// absmax_in: when non-null, per-row absmax is taken from it instead of
// scanning X (the FFN requant after a fused reduction).
cudaError_t launch_quant(const void* X, int x_dtype, int M, int K, float eps, QLayout layout,
                         void* q, float* m_out, int32_t* qsum_out, const float* absmax_in,
                         bool pdl, cudaStream_t st);

// ----- decode GEMV (dp4a) ----------------------------------------------------
enum class Epi : int { kPlain = 0, kRelu2 = 1 };
// q: int8 row-major [M][K], m [M]. Writes Y [M][N] fp32 (or h = relu2(y) for kRelu2)
// and optionally acc [M][N] int32. absmax_out (kRelu2 only, may be null):
// per-row max of h, combined with atomicMax on the float bits (h >= 0).
cudaError_t launch_gemv(const uint8_t* Wp, int N, int K, const int8_t* q, const float* m,
                        const float* s_w, int M, float* Y, int32_t* acc,
                        Epi epi, float* absmax_out, bool pdl, cudaStream_t st);

}  // namespace bl
