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
// RMSNorm fused into the quantization: codes from u = fp32(x * g) (g null:
// unit gain), scale fp32(max(max|u|, eps) * r), r = 1/sqrt(mean x^2 + eps_norm).
struct RmsNorm {
  const float* g;        // [K] fp32 gain, or null
  float eps_norm;        // > 0
};
// X: [M][K] fp32 or bf16; m_out [M] fp32; norm: null for the plain quantization.
cudaError_t launch_quant(const void* X, int x_dtype, int M, int K, float eps, QLayout layout,
                         void* q, float* m_out, const RmsNorm* norm, bool pdl, cudaStream_t st);

// Row-major int8 quantization of several problems in one launch.
struct QuantProblem {
  const void* X;         // [M][K] fp32 or bf16
  int x_dtype;
  int M, K;
  int8_t* q;             // [M][K] int8 out
  float* m;              // [M] out
};
constexpr int kQuantMaxBatch = 128;
cudaError_t launch_quant_batch(const QuantProblem* ps, int count, float eps, bool pdl, cudaStream_t st);
// int8 row-major [M][K] -> fp16 [M][K] in the kPairF16 order.
cudaError_t launch_widen_pair(const int8_t* q, int M, int K, void* out, bool pdl, cudaStream_t st);

// ----- decode GEMV (dp4a) ----------------------------------------------------
enum class Epi : int { kPlain = 0, kRelu2 = 1 };
struct GemvProblem {
  const uint8_t* Wp;     // packed [N][K/4]
  const float* s_w;      // [1]
  int N, K, M;
  const int8_t* q;       // int8 activations, row-major [M][K]
  const float* m;        // their per-token scales [M]
  float* Y;              // [M][N] fp32 (h = relu2(y) for kRelu2)
  int32_t* acc;          // [M][N] or null
  Epi epi;
  const float* mul;      // [M][N] or null: y = fp32(y * mul) (the gated FFN's up projection)
  // single-problem launches only: when x is set, the GEMV quantizes the token
  // rows itself (q and m are then unused)
  const void* x;         // [M][K] fp32 or bf16, or null
  int x_dtype;
  float eps;
};
constexpr int kGemvMaxBatch = 128;
// One problem (M <= 4 per launch; more tokens take several launches).
cudaError_t launch_gemv(const GemvProblem& p, WsHeader* status, bool pdl, cudaStream_t st);
// Independent problems in one launch (count <= kGemvMaxBatch).
cudaError_t launch_gemv_batch(const GemvProblem* ps, int count, WsHeader* status, bool pdl, cudaStream_t st);

// ----- prefill / batched GEMM (tcgen05, TMEM, TMA) ---------------------------
struct GemmProblem {
  const uint8_t* Wp;     // packed [N][K/4]
  const float* s_w;      // [1]
  int M, N, K;
  const void* act;       // fp16 [M][K] in the pair order (QLayout::kPairF16)
  const float* m;        // [M] per-token scales
  float* Y;              // [M][N]
  int32_t* acc;          // [M][N] or null
  bool relu2;            // FFN up: write h = relu(y)^2
  const float* mul;      // [M][N] or null: y = fp32(y * mul) (the gated FFN's up projection)
  int32_t* acc_ws;       // [M][N] int32 scratch for a split-K run, or null (no split)
};
// How many K parts a GEMM of these sizes is cut into (1: no split). Split runs
// need an [M][N] int32 scratch (GemmProblem::acc_ws).
int gemm_splits(int M, int N, int K);
// Tokens from which the forward takes the tensor-core GEMM instead of the GEMV
// (measured on B300, each call alone with L2 flushed: at 4 tokens the GEMV is
// faster on every 2B-class shape, from 5 the GEMM, whose split-K time is flat;
// the GEMV takes at most 4 tokens per launch, so 5 tokens need two).
constexpr int kGemmMinTokens = 5;
cudaError_t launch_gemm(const GemmProblem& g, WsHeader* status, bool pdl, cudaStream_t st);

}  // namespace bl
