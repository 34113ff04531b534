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
// the tensor-core operand order), plus sum_k q_k when asked. A batched
// variant quantizes the token rows of up to kQuantMaxBatch problems in one
// launch.
#include "common.cuh"
#include "launchers.h"

namespace bl {
namespace {

constexpr int kThreads = 256;

// Quantize one token row (all threads of the CTA take part).
template <int DT, int LAYOUT>
__device__ __forceinline__ void quant_row(const void* __restrict__ xr, int K, float eps, void* __restrict__ qout_row,
                                          float* __restrict__ m_out, int32_t* __restrict__ qsum_out,
                                          const float* __restrict__ absmax_in, float* s_red, int* s_sum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = K >> 4;
  float amax;
  if (absmax_in != nullptr) {
    amax = *absmax_in;
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
      reinterpret_cast<uint4*>(qout_row)[g] = o;
    } else {
      // fp16 slot s holds column (s >> 1) + 8 * (s & 1)
      uint4 o0 = make_uint4(pack_h2(q[0], q[8]), pack_h2(q[1], q[9]), pack_h2(q[2], q[10]), pack_h2(q[3], q[11]));
      uint4 o1 = make_uint4(pack_h2(q[4], q[12]), pack_h2(q[5], q[13]), pack_h2(q[6], q[14]), pack_h2(q[7], q[15]));
      uint4* dst = reinterpret_cast<uint4*>(qout_row) + 2 * g;
      dst[0] = o0;
      dst[1] = o1;
    }
  }
  if (qsum_out != nullptr) {
    qs = warp_sum(qs);
    if (lane == 0) s_sum[warp] = qs;
    __syncthreads();
    if (tid == 0) {
      int t = 0;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) t += s_sum[w];
      *qsum_out = t;
    }
  }
  if (tid == 0 && m_out != nullptr) *m_out = m;
}

template <int DT, int LAYOUT>
__global__ void __launch_bounds__(kThreads) quant_kernel(const void* __restrict__ X, int K, float eps,
                                                         void* __restrict__ qout, float* __restrict__ m_out,
                                                         int32_t* __restrict__ qsum_out,
                                                         const float* __restrict__ absmax_in) {
  __shared__ float s_red[kThreads / 32];
  __shared__ int s_sum[kThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x;
  const size_t esize = DT == BL_DTYPE_F32 ? 4 : 2;
  const size_t qsize = LAYOUT == static_cast<int>(QLayout::kRowMajorI8) ? 1 : 2;
  quant_row<DT, LAYOUT>(static_cast<const char*>(X) + static_cast<size_t>(row) * K * esize, K, eps,
                        static_cast<char*>(qout) + static_cast<size_t>(row) * K * qsize,
                        m_out != nullptr ? m_out + row : nullptr, qsum_out != nullptr ? qsum_out + row : nullptr,
                        absmax_in != nullptr ? absmax_in + row : nullptr, s_red, s_sum);
}

// Row-major int8 quantization of the token rows of several problems in one
// launch: CTA b quantizes row b of the concatenated rows.
struct QuantBatchArgs {
  QuantProblem prob[kQuantMaxBatch];
  int row_begin[kQuantMaxBatch + 1];
  int count;
  float eps;
};

__global__ void __launch_bounds__(kThreads) quant_batch_kernel(const __grid_constant__ QuantBatchArgs a) {
  __shared__ float s_red[kThreads / 32];
  __shared__ int s_sum[kThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  int lo = 0, hi = a.count - 1;             // problem p with row_begin[p] <= b < row_begin[p+1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.row_begin[mid] <= b) lo = mid;
    else hi = mid - 1;
  }
  const QuantProblem& P = a.prob[lo];
  const int row = b - a.row_begin[lo];
  const size_t esize = P.x_dtype == BL_DTYPE_F32 ? 4 : 2;
  const void* xr = static_cast<const char*>(P.X) + static_cast<size_t>(row) * P.K * esize;
  int8_t* qr = P.q + static_cast<size_t>(row) * P.K;
  if (P.x_dtype == BL_DTYPE_F32)
    quant_row<BL_DTYPE_F32, 0>(xr, P.K, a.eps, qr, P.m + row, nullptr, nullptr, s_red, s_sum);
  else
    quant_row<BL_DTYPE_BF16, 0>(xr, P.K, a.eps, qr, P.m + row, nullptr, nullptr, s_red, s_sum);
}

template <int DT, int LAYOUT>
cudaError_t launch_t(const void* X, int M, int K, float eps, void* q, float* m_out, int32_t* qsum_out,
                     const float* absmax_in, bool pdl, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cfg.gridDim = dim3(static_cast<unsigned>(M));
  return cudaLaunchKernelEx(&cfg, quant_kernel<DT, LAYOUT>, X, K, eps, q, m_out, qsum_out, absmax_in);
}

// int8 row-major -> fp16 in the tensor-core pair order (an input quantized
// elsewhere, given to the GEMM). One thread per 16-column group.
__global__ void __launch_bounds__(256) widen_pair_kernel(const int8_t* __restrict__ q, size_t groups,
                                                         uint4* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t g = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups; g += stride) {
    const uint4 v = reinterpret_cast<const uint4*>(q)[g];
    int b[16];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 16; ++i) b[i] = static_cast<int>(static_cast<int8_t>((w[i >> 2] >> (8 * (i & 3))) & 0xFFu));
    out[2 * g] = make_uint4(pack_h2(b[0], b[8]), pack_h2(b[1], b[9]), pack_h2(b[2], b[10]), pack_h2(b[3], b[11]));
    out[2 * g + 1] = make_uint4(pack_h2(b[4], b[12]), pack_h2(b[5], b[13]), pack_h2(b[6], b[14]), pack_h2(b[7], b[15]));
  }
}

}  // namespace

cudaError_t launch_widen_pair(const int8_t* q, int M, int K, void* out, bool pdl, cudaStream_t st) {
  const size_t groups = static_cast<size_t>(M) * K / 16;
  if (groups == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((groups + 255) / 256, static_cast<size_t>(8 * sms)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, widen_pair_kernel, q, groups, static_cast<uint4*>(out));
}

cudaError_t launch_quant_batch(const QuantProblem* ps, int count, float eps, bool pdl, cudaStream_t st) {
  QuantBatchArgs a;
  int rows = 0, n = 0;
  for (int i = 0; i < count; ++i) {
    if (ps[i].M <= 0) continue;
    a.prob[n] = ps[i];
    a.row_begin[n] = rows;
    rows += ps[i].M;
    ++n;
  }
  if (n == 0) return cudaSuccess;
  a.row_begin[n] = rows;
  a.count = n;
  a.eps = eps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, quant_batch_kernel, a);
}

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
