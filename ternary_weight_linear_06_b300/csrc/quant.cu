// Per-token absmax int8 activation quantization.
//
// "BitNet解读" (markgoyens.top), 模型架构 / 激活量化: each token's
// activations are scaled into [-Qb, Qb], symmetric, without a zero point;
// the 2B4T report (section 2) applies absmax per token. With Qb = 127:
//   m = max(max_k |x_k|, eps);  q_k = clamp(rint(fp32(fp32(x_k * 127) / m)), -128, 127).
//
// Pass 1 reduces |x| to the row absmax, pass 2 quantizes 16 columns per
// thread step and writes them in the layout the consumer wants (row-major
// int8, or fp16 in the tensor-core operand order). From one row per SM up, a
// team of 1-8 warps takes a row (several teams per CTA); fewer rows get one
// CTA each. Rows up to 16384 columns stay in registers between the passes. A
// batched variant quantizes the token rows of up to kQuantMaxBatch problems
// in one launch.
//
// SubLN ("BitNet b1.58 2B4T Technical Report", section 2: a sub-layer norm,
// bias-free norm layers; RMSNorm as the LLaMA-style norm in "BitNet解读",
// 模型架构 / 组件兼容性) runs in the same two passes: RMSNorm with gain g is
// n = x * g * r per token, r = 1 / sqrt(mean x^2 + eps_norm). Absmax codes
// are unchanged by the positive factor r, so pass 2 quantizes u = fp32(x * g)
// and r goes into the token's scale; pass 1 adds the sum of x^2 to the absmax
// reduction.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launchers.h"

namespace bl {
namespace {

constexpr int kThreads = 256;

// Sum of the squares of one row, carried as the unevaluated pair p + s of the
// compensated dot product Dot2 of Ogita, Rump and Oishi ("Accurate Sum and
// Dot Product", SIAM J. Sci. Comput. 26(6), 2005): each square is split
// exactly into its rounded value and the FMA remainder, each addition into its
// rounded sum and the TwoSum error. The pair holds the sum to about twice
// fp32's precision without the fp64 pipe, which is slow on B300. With
// EXACT_SQ (bf16 inputs: an 8-bit significand squares exactly in fp32) the
// FMA remainder is known to be zero and skipped.
struct F2 {
  float hi, lo;
};

__device__ __forceinline__ F2 two_sum(float a, float b) {
  const float t = __fadd_rn(a, b);
  const float z = __fsub_rn(t, a);
  return {t, __fadd_rn(__fsub_rn(a, __fsub_rn(t, z)), __fsub_rn(b, z))};
}

// (a.hi + a.lo) + (b.hi + b.lo) as a normalized pair; the terms here are all
// non-negative, so nothing cancels and the error stays near 2^-44 relative.
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  const F2 s = two_sum(a.hi, b.hi);
  const float e = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
  const float hi = __fadd_rn(s.hi, e);
  return {hi, __fsub_rn(e, __fsub_rn(hi, s.hi))};
}

template <bool EXACT_SQ>
struct SumSq {
  float p = 0.0f, s = 0.0f;
  __device__ __forceinline__ void add(float x) {
    const float h = __fmul_rn(x, x);
    const F2 t = two_sum(p, h);
    p = t.hi;
    if constexpr (EXACT_SQ) s = __fadd_rn(s, t.lo);
    else s = __fadd_rn(s, __fadd_rn(t.lo, __fmaf_rn(x, x, -h)));
  }
};

__device__ __forceinline__ F2 warp_sum_f2(F2 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const F2 w = {__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
    v = f2_add(v, w);
  }
  return v;
}

// r = 1 / sqrt(S * inv_k + eps_norm) in fp64 by Newton's iteration for the
// inverse square root, y <- y * (3/2 - a y^2 / 2), from the fp32 estimate
// rsqrtf(a): each step squares the relative error (about 2^-22 -> 2^-44 ->
// below fp64 rounding), using only multiplies and FMAs.
__device__ __forceinline__ double rms_factor(F2 S, double inv_k, float eps_norm) {
  const double s = __dadd_rn(static_cast<double>(S.hi), static_cast<double>(S.lo));
  const double a = __fma_rn(s, inv_k, static_cast<double>(eps_norm));
  double y = static_cast<double>(rsqrtf(__double2float_rn(a)));
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const double t = __dmul_rn(__dmul_rn(a, y), y);
    y = __dmul_rn(y, __fma_rn(-0.5, t, 1.5));
  }
  return y;
}

// u = fp32(x * g) for the 16 columns of group g (x stays as it is without a gain).
__device__ __forceinline__ void apply_gain(const float* __restrict__ gain, int g, float (&v)[16]) {
  if (gain == nullptr) return;
  float w[16];
  load16<BL_DTYPE_F32>(gain, g, w);
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], w[j]);
}

// Pass-1 work on one 16-column group: with NORM, the squares of x go into the
// two sum chains and v becomes u = fp32(x * g); then the running absmax.
template <int DT, bool NORM>
__device__ __forceinline__ void stat_group(float (&v)[16], int g, const float* __restrict__ gain,
                                           SumSq<DT == BL_DTYPE_BF16>& ss0, SumSq<DT == BL_DTYPE_BF16>& ss1,
                                           float& a) {
  if constexpr (NORM) {
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      ss0.add(v[j]);
      ss1.add(v[j + 1]);
    }
    apply_gain(gain, g, v);
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) a = fmaxf(a, fabsf(v[j]));
}

// Pass-2 work on one group: the codes, written in the consumer's layout
// (s127 = fp32(127 * fp32(1/m))).
template <int LAYOUT>
__device__ __forceinline__ void store_group(const float (&v)[16], int g, float m, float s127,
                                            void* __restrict__ qout_row) {
  float r[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) r[j] = quant_round(v[j], m, s127);
  if constexpr (LAYOUT == static_cast<int>(QLayout::kRowMajorI8)) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t b0 = __float_as_uint(__fadd_rn(r[4 * k + 0], kIntShift));
      const uint32_t b1 = __float_as_uint(__fadd_rn(r[4 * k + 1], kIntShift));
      const uint32_t b2 = __float_as_uint(__fadd_rn(r[4 * k + 2], kIntShift));
      const uint32_t b3 = __float_as_uint(__fadd_rn(r[4 * k + 3], kIntShift));
      w[k] = __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
    }
    reinterpret_cast<uint4*>(qout_row)[g] = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    // fp16 slot s holds column (s >> 1) + 8 * (s & 1); the codes are exact in fp16
    uint32_t h[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const __half2 p2 = __floats2half2_rn(r[j], r[j + 8]);
      h[j] = *reinterpret_cast<const uint32_t*>(&p2);
    }
    uint4* dst = reinterpret_cast<uint4*>(qout_row) + 2 * g;
    dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
    dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// Groups of 16 columns each thread keeps in registers between the passes (0:
// the row is too long, pass 2 reads it again).
constexpr int kMaxResident = 4;
inline int resident_groups(int K) {
  const int G = K >> 4;
  if (G <= kThreads) return 1;
  if (G <= 2 * kThreads) return 2;
  if (G <= kMaxResident * kThreads) return 4;
  return 0;
}

// Quantize one token row (all threads of the CTA take part). With NORM the
// row is first RMS-normalized with the gain `gain` (null: unit gain): codes
// come from u = fp32(x * g) and the scale written is
// fp32(max(max|u|, eps) * r), r = 1 / sqrt(sum x^2 / K + eps_norm); inv_k = 1/K.
// R > 0: thread t holds groups t + i * kThreads (i < R) in registers, loaded
// once; R = 0: both passes stream the row.
template <int DT, int LAYOUT, bool NORM, int R>
__device__ __forceinline__ void quant_row(const void* __restrict__ xr, int K, float eps,
                                          const float* __restrict__ gain, float eps_norm, double inv_k,
                                          void* __restrict__ qout_row, float* __restrict__ m_out, float* s_red,
                                          F2* s_ss) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = K >> 4;
  float a = 0.0f;
  SumSq<DT == BL_DTYPE_BF16> ss0, ss1;        // two chains (even, odd columns) for latency
  float v[R > 0 ? R : 1][16];
  if constexpr (R > 0) {
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (tid + i * kThreads < G) load16<DT>(xr, tid + i * kThreads, v[i]);
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (tid + i * kThreads < G) stat_group<DT, NORM>(v[i], tid + i * kThreads, gain, ss0, ss1, a);
  } else {
    for (int g = tid; g < G; g += kThreads) {
      load16<DT>(xr, g, v[0]);
      stat_group<DT, NORM>(v[0], g, gain, ss0, ss1, a);
    }
  }
  a = warp_max(a);
  if (lane == 0) s_red[warp] = a;
  if constexpr (NORM) {
    const F2 d = warp_sum_f2(f2_add({ss0.p, ss0.s}, {ss1.p, ss1.s}));
    if (lane == 0) s_ss[warp] = d;
  }
  __syncthreads();
  a = 0.0f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) a = fmaxf(a, s_red[w]);
  const float m = fmaxf(a, eps);
  const float s127 = __fmul_rn(127.0f, __frcp_rn(m));

  if constexpr (R > 0) {
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (tid + i * kThreads < G) store_group<LAYOUT>(v[i], tid + i * kThreads, m, s127, qout_row);
  } else {
    for (int g = tid; g < G; g += kThreads) {
      load16<DT>(xr, g, v[0]);
      if constexpr (NORM) apply_gain(gain, g, v[0]);
      store_group<LAYOUT>(v[0], g, m, s127, qout_row);
    }
  }
  if (tid == 0 && m_out != nullptr) {
    if constexpr (NORM) {
      F2 S = s_ss[0];
#pragma unroll
      for (int w = 1; w < kThreads / 32; ++w) S = f2_add(S, s_ss[w]);
      const double r = rms_factor(S, inv_k, eps_norm);
      *m_out = __double2float_rn(__dmul_rn(static_cast<double>(m), r));
    } else {
      *m_out = m;
    }
  }
}

template <int DT, int LAYOUT, bool NORM, int R>
__global__ void __launch_bounds__(kThreads) quant_kernel(const void* __restrict__ X, int K, float eps,
                                                         const float* __restrict__ gain, float eps_norm,
                                                         double inv_k, void* __restrict__ qout,
                                                         float* __restrict__ m_out) {
  __shared__ float s_red[kThreads / 32];
  __shared__ F2 s_ss[kThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x;
  const size_t esize = DT == BL_DTYPE_F32 ? 4 : 2;
  const size_t qsize = LAYOUT == static_cast<int>(QLayout::kRowMajorI8) ? 1 : 2;
  quant_row<DT, LAYOUT, NORM, R>(static_cast<const char*>(X) + static_cast<size_t>(row) * K * esize, K, eps, gain,
                                 eps_norm, inv_k, static_cast<char*>(qout) + static_cast<size_t>(row) * K * qsize,
                                 m_out + row, s_red, s_ss);
}

// ---------------------------------------------------------------------------
// Team kernel: a row belongs to a team of TW warps (TW = 1, 2, 4 or 8, the
// fewest for which each lane holds at most GMAX groups of 16 columns), and a
// 256-thread CTA holds 8 / TW teams. Each lane keeps the raw input words of
// its groups (t + 32 TW i) in registers from pass 1 to pass 2, and a team
// meets only on its own named barrier, so an SM works on up to 64 / TW rows
// at once rather than one per CTA.
// ---------------------------------------------------------------------------
template <int DT>
constexpr int kTeamGroups = DT == BL_DTYPE_F32 ? 2 : 4;     // GMAX: 32 registers of raw input per lane

template <int DT>
struct Raw16 {
  uint4 u[DT == BL_DTYPE_F32 ? 4 : 2];
};

template <int DT>
__device__ __forceinline__ void load_raw(const void* row, int g, Raw16<DT>& r) {
  const uint4* p = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + static_cast<size_t>(g) * sizeof(Raw16<DT>));
#pragma unroll
  for (int i = 0; i < (DT == BL_DTYPE_F32 ? 4 : 2); ++i) r.u[i] = __ldg(p + i);
}

template <int DT>
__device__ __forceinline__ void widen_raw(const Raw16<DT>& r, float (&v)[16]) {
  if constexpr (DT == BL_DTYPE_F32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[4 * i + 0] = __uint_as_float(r.u[i].x);
      v[4 * i + 1] = __uint_as_float(r.u[i].y);
      v[4 * i + 2] = __uint_as_float(r.u[i].z);
      v[4 * i + 3] = __uint_as_float(r.u[i].w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t w[4] = {r.u[i].x, r.u[i].y, r.u[i].z, r.u[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * i + 2 * j + 0] = __uint_as_float(w[j] << 16);          // exact bf16 -> fp32
        v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  }
}

// Running absmax over the raw input words of one group without widening:
// bf16 pairs go through the packed bf16x2 max of magnitudes.
template <int DT>
__device__ __forceinline__ float raw_absmax(const Raw16<DT>& r, float a) {
  if constexpr (DT == BL_DTYPE_F32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a = fmaxf(a, fabsf(__uint_as_float(r.u[i].x)));
      a = fmaxf(a, fabsf(__uint_as_float(r.u[i].y)));
      a = fmaxf(a, fabsf(__uint_as_float(r.u[i].z)));
      a = fmaxf(a, fabsf(__uint_as_float(r.u[i].w)));
    }
    return a;
  } else {
    __nv_bfloat162 m2 = __floats2bfloat162_rn(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t w[4] = {r.u[i].x, r.u[i].y, r.u[i].z, r.u[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[j])));
    }
    return fmaxf(a, fmaxf(__low2float(m2), __high2float(m2)));
  }
}

__device__ __forceinline__ void team_sync(int team, int TW) {
  if (TW == 1) {
    __syncwarp();
  } else {
    asm volatile("bar.sync %0, %1;" ::"r"(team + 1), "r"(TW * 32) : "memory");
  }
}

template <int DT, int LAYOUT, bool NORM, int TW>
__global__ void __launch_bounds__(kThreads) quant_team_kernel(const void* __restrict__ X, int M, int K, float eps,
                                                              const float* __restrict__ gain, float eps_norm,
                                                              double inv_k, void* __restrict__ qout,
                                                              float* __restrict__ m_out) {
  constexpr int kTeams = kThreads / 32 / TW;
  constexpr int GMAX = kTeamGroups<DT>;
  constexpr size_t kEs = DT == BL_DTYPE_F32 ? 4 : 2;
  constexpr size_t kQs = LAYOUT == static_cast<int>(QLayout::kRowMajorI8) ? 1 : 2;
  __shared__ float s_red[kTeams][TW];
  __shared__ F2 s_ss[kTeams][TW];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = warp / TW, wt = warp - team * TW, tt = threadIdx.x - team * TW * 32;
  const int row = blockIdx.x * kTeams + team;
  pdl_wait();
  pdl_trigger();
  if (row >= M) return;                            // whole teams leave together
  const int G = K >> 4;
  const void* xr = static_cast<const char*>(X) + static_cast<size_t>(row) * K * kEs;
  Raw16<DT> raw[GMAX];
#pragma unroll
  for (int i = 0; i < GMAX; ++i)
    if (tt + i * TW * 32 < G) load_raw<DT>(xr, tt + i * TW * 32, raw[i]);
  float a = 0.0f;
  SumSq<DT == BL_DTYPE_BF16> ss0, ss1;
#pragma unroll
  for (int i = 0; i < GMAX; ++i) {
    const int g = tt + i * TW * 32;
    if (g < G) {
      if constexpr (NORM) {
        float v[16];
        widen_raw<DT>(raw[i], v);
        stat_group<DT, NORM>(v, g, gain, ss0, ss1, a);
      } else {
        a = raw_absmax<DT>(raw[i], a);
      }
    }
  }
  a = warp_max(a);
  F2 d = {0.0f, 0.0f};
  if constexpr (NORM) d = warp_sum_f2(f2_add({ss0.p, ss0.s}, {ss1.p, ss1.s}));
  if (TW > 1) {
    if (lane == 0) {
      s_red[team][wt] = a;
      if constexpr (NORM) s_ss[team][wt] = d;
    }
    team_sync(team, TW);
#pragma unroll
    for (int w = 0; w < TW; ++w) a = fmaxf(a, s_red[team][w]);
  }
  const float m = fmaxf(a, eps);
  const float s127 = __fmul_rn(127.0f, __frcp_rn(m));
  void* qrow = static_cast<char*>(qout) + static_cast<size_t>(row) * K * kQs;
#pragma unroll
  for (int i = 0; i < GMAX; ++i) {
    const int g = tt + i * TW * 32;
    if (g < G) {
      float v[16];
      widen_raw<DT>(raw[i], v);
      if constexpr (NORM) apply_gain(gain, g, v);
      store_group<LAYOUT>(v, g, m, s127, qrow);
    }
  }
  if (tt == 0) {
    if constexpr (NORM) {
      F2 S = TW > 1 ? s_ss[team][0] : d;
#pragma unroll
      for (int w = 1; w < TW; ++w) S = f2_add(S, s_ss[team][w]);
      m_out[row] = __double2float_rn(__dmul_rn(static_cast<double>(m), rms_factor(S, inv_k, eps_norm)));
    } else {
      m_out[row] = m;
    }
  }
}

// Warps per team for rows of K columns (0: the row is too long for a team).
template <int DT>
int team_warps(int K) {
  const int G = K >> 4;
  for (int tw = 1; tw <= 8; tw *= 2)
    if (G <= tw * 32 * kTeamGroups<DT>) return tw;
  return 0;
}

// Row-major int8 quantization of the token rows of several problems in one
// launch: CTA b quantizes row b of the concatenated rows.
struct QuantBatchArgs {
  QuantProblem prob[kQuantMaxBatch];
  int row_begin[kQuantMaxBatch + 1];
  int count;
  float eps;
};

template <int R>
__global__ void __launch_bounds__(kThreads) quant_batch_kernel(const __grid_constant__ QuantBatchArgs a) {
  __shared__ float s_red[kThreads / 32];
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
    quant_row<BL_DTYPE_F32, 0, false, R>(xr, P.K, a.eps, nullptr, 0.0f, 0.0, qr, P.m + row, s_red, nullptr);
  else
    quant_row<BL_DTYPE_BF16, 0, false, R>(xr, P.K, a.eps, nullptr, 0.0f, 0.0, qr, P.m + row, s_red, nullptr);
}

template <int DT, int LAYOUT, bool NORM, int R>
cudaError_t launch_t(const void* X, int M, int K, float eps, const RmsNorm* norm, void* q, float* m_out, bool pdl,
                     cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cfg.gridDim = dim3(static_cast<unsigned>(M));
  return cudaLaunchKernelEx(&cfg, quant_kernel<DT, LAYOUT, NORM, R>, X, K, eps, NORM ? norm->g : nullptr,
                            NORM ? norm->eps_norm : 0.0f, 1.0 / static_cast<double>(K), q, m_out);
}

template <int DT, int LAYOUT, bool NORM, int TW>
cudaError_t launch_team(const void* X, int M, int K, float eps, const RmsNorm* norm, void* q, float* m_out, bool pdl,
                        cudaStream_t st) {
  constexpr int kTeams = kThreads / 32 / TW;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((M + kTeams - 1) / kTeams));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, quant_team_kernel<DT, LAYOUT, NORM, TW>, X, M, K, eps, NORM ? norm->g : nullptr,
                            NORM ? norm->eps_norm : 0.0f, 1.0 / static_cast<double>(K), q, m_out);
}

template <int DT, int LAYOUT, bool NORM>
cudaError_t launch_r(const void* X, int M, int K, float eps, const RmsNorm* norm, void* q, float* m_out, bool pdl,
                     cudaStream_t st) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // fewer rows than SMs: one CTA per row puts more threads on each row
  switch (M >= sms ? team_warps<DT>(K) : 0) {
    case 1: return launch_team<DT, LAYOUT, NORM, 1>(X, M, K, eps, norm, q, m_out, pdl, st);
    case 2: return launch_team<DT, LAYOUT, NORM, 2>(X, M, K, eps, norm, q, m_out, pdl, st);
    case 4: return launch_team<DT, LAYOUT, NORM, 4>(X, M, K, eps, norm, q, m_out, pdl, st);
    case 8: return launch_team<DT, LAYOUT, NORM, 8>(X, M, K, eps, norm, q, m_out, pdl, st);
    default: break;
  }
  switch (resident_groups(K)) {
    case 1: return launch_t<DT, LAYOUT, NORM, 1>(X, M, K, eps, norm, q, m_out, pdl, st);
    case 2: return launch_t<DT, LAYOUT, NORM, 2>(X, M, K, eps, norm, q, m_out, pdl, st);
    case 4: return launch_t<DT, LAYOUT, NORM, 4>(X, M, K, eps, norm, q, m_out, pdl, st);
    default: return launch_t<DT, LAYOUT, NORM, 0>(X, M, K, eps, norm, q, m_out, pdl, st);
  }
}

template <int DT, int LAYOUT>
cudaError_t launch_n(const void* X, int M, int K, float eps, const RmsNorm* norm, void* q, float* m_out, bool pdl,
                     cudaStream_t st) {
  if (norm != nullptr) return launch_r<DT, LAYOUT, true>(X, M, K, eps, norm, q, m_out, pdl, st);
  return launch_r<DT, LAYOUT, false>(X, M, K, eps, norm, q, m_out, pdl, st);
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
  int max_k = 0;
  for (int i = 0; i < n; ++i) max_k = std::max(max_k, a.prob[i].K);
  switch (resident_groups(max_k)) {
    case 1: return cudaLaunchKernelEx(&cfg, quant_batch_kernel<1>, a);
    case 2: return cudaLaunchKernelEx(&cfg, quant_batch_kernel<2>, a);
    case 4: return cudaLaunchKernelEx(&cfg, quant_batch_kernel<4>, a);
    default: return cudaLaunchKernelEx(&cfg, quant_batch_kernel<0>, a);
  }
}

cudaError_t launch_quant(const void* X, int x_dtype, int M, int K, float eps, QLayout layout, void* q,
                         float* m_out, const RmsNorm* norm, bool pdl, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  const bool i8 = layout == QLayout::kRowMajorI8;
  if (x_dtype == BL_DTYPE_F32) {
    if (i8) return launch_n<BL_DTYPE_F32, 0>(X, M, K, eps, norm, q, m_out, pdl, st);
    return launch_n<BL_DTYPE_F32, 2>(X, M, K, eps, norm, q, m_out, pdl, st);
  }
  if (i8) return launch_n<BL_DTYPE_BF16, 0>(X, M, K, eps, norm, q, m_out, pdl, st);
  return launch_n<BL_DTYPE_BF16, 2>(X, M, K, eps, norm, q, m_out, pdl, st);
}

}  // namespace bl
