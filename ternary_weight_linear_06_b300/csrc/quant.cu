// Per-token absmax int8 activation quantization.
//
// "BitNet解读" (markgoyens.top), 模型架构 / 激活量化: each token's
// activations are scaled into [-Qb, Qb], symmetric, without a zero point;
// the 2B4T report (section 2) applies absmax per token. With Qb = 127:
//   m = max(max_k |x_k|, eps);  q_k = clamp(rint(fp32(fp32(x_k * 127) / m)), -128, 127).
//
// One CTA per token row: pass 1 reduces |x| to the row absmax (skipped when
// the caller supplies it), pass 2 quantizes 16 columns per thread step and
// writes them in the layout the consumer wants (row-major int8, or fp16 in
// the tensor-core operand order), plus sum_k q_k when asked (the matmul
// kernels multiply by the stored code t + 1 and subtract it).
#include "common.cuh"
#include "launchers.h"

namespace bl {
namespace {

constexpr int kThreads = 256;

template <int DT, int LAYOUT>
__global__ void __launch_bounds__(kThreads) quant_kernel(const void* __restrict__ X, int K, float eps,
                                                         void* __restrict__ qout, float* __restrict__ m_out,
                                                         int32_t* __restrict__ qsum_out,
                                                         const float* __restrict__ absmax_in) {
  __shared__ float s_red[kThreads / 32];
  __shared__ int s_sum[kThreads / 32];
  pdl_wait();
  const int row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t esize = DT == BL_DTYPE_F32 ? 4 : 2;
  const void* xr = static_cast<const char*>(X) + static_cast<size_t>(row) * K * esize;
  const int G = K >> 4;

  float amax;
  if (absmax_in != nullptr) {
    amax = absmax_in[row];
  } else {
    float a = 0.0f;
    for (int g = tid; g < G; g += kThreads) {
      float v[16];
      load16<DT>(xr, g, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) a = fmaxf(a, fabsf(v[j]));
    }
    a = warp_max(a);
    if (lane == 0) s_red[warp] = a;
    __syncthreads();
    a = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) a = fmaxf(a, s_red[w]);
    amax = a;
  }
  const float m = fmaxf(amax, eps);

  int qs = 0;
  for (int g = tid; g < G; g += kThreads) {
    float v[16];
    load16<DT>(xr, g, v);
    int q[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      q[j] = quant_one(v[j], m);
      qs += q[j];
    }
    if constexpr (LAYOUT == static_cast<int>(QLayout::kRowMajorI8)) {
      uint4 o = make_uint4(pack4(q[0], q[1], q[2], q[3]), pack4(q[4], q[5], q[6], q[7]),
                           pack4(q[8], q[9], q[10], q[11]), pack4(q[12], q[13], q[14], q[15]));
      reinterpret_cast<uint4*>(static_cast<int8_t*>(qout) + static_cast<size_t>(row) * K)[g] = o;
    } else {
      // fp16 slot s holds column (s >> 1) + 8 * (s & 1)
      uint4 o0 = make_uint4(pack_h2(q[0], q[8]), pack_h2(q[1], q[9]), pack_h2(q[2], q[10]), pack_h2(q[3], q[11]));
      uint4 o1 = make_uint4(pack_h2(q[4], q[12]), pack_h2(q[5], q[13]), pack_h2(q[6], q[14]), pack_h2(q[7], q[15]));
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(qout) + static_cast<size_t>(row) * K) + 2 * g;
      dst[0] = o0;
      dst[1] = o1;
    }
  }
  pdl_trigger();
  if (qsum_out != nullptr) {
    qs = warp_sum(qs);
    if (lane == 0) s_sum[warp] = qs;
    __syncthreads();
    if (tid == 0) {
      int t = 0;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) t += s_sum[w];
      qsum_out[row] = t;
    }
  }
  if (tid == 0 && m_out != nullptr) m_out[row] = m;
}

template <int DT, int LAYOUT>
cudaError_t launch_t(const void* X, int M, int K, float eps, void* q, float* m_out, int32_t* qsum_out,
                     const float* absmax_in, bool pdl, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(M));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, quant_kernel<DT, LAYOUT>, X, K, eps, q, m_out, qsum_out, absmax_in);
}

}  // namespace

cudaError_t launch_quant(const void* X, int x_dtype, int M, int K, float eps, QLayout layout, void* q,
                         float* m_out, int32_t* qsum_out, const float* absmax_in, bool pdl, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  const int L = static_cast<int>(layout);
  if (x_dtype == BL_DTYPE_F32) {
    if (L == 0) return launch_t<BL_DTYPE_F32, 0>(X, M, K, eps, q, m_out, qsum_out, absmax_in, pdl, st);
    return launch_t<BL_DTYPE_F32, 2>(X, M, K, eps, q, m_out, qsum_out, absmax_in, pdl, st);
  }
  if (L == 0) return launch_t<BL_DTYPE_BF16, 0>(X, M, K, eps, q, m_out, qsum_out, absmax_in, pdl, st);
  return launch_t<BL_DTYPE_BF16, 2>(X, M, K, eps, q, m_out, qsum_out, absmax_in, pdl, st);
}

}  // namespace bl
