// Decode GEMV for few tokens: packed 2-bit ternary weights x int8 activations.
//
// "BitNet b1.58 2B4T Technical Report | Summary", 5.1 GPU Inference: packed
// weights stream from HBM, are unpacked on chip and multiplied with 8-bit
// activations. "BitNet解读", 革命性的效率提升: with ternary weights the
// product is additions and subtractions of activations.
//
// Each weight row is K/4 bytes (code t+1 of column 4b+j in bits [2j,2j+1] of
// byte b). A lane streams 16-byte chunks (64 columns) with 128-bit loads; the
// four 32-bit words of a chunk each hold 16 codes, code of column 16w+4j+i at
// bit 8j+2i. The CTA stages the int8 activations (row-major) in shared memory
// in "quad" order -- word i of a 16-column group holds columns i, 4+i, 8+i,
// 12+i, a 4x4 byte transpose done with byte permutes -- so that
//   dp4a(act word i, (w >> 2i) & 0x03030303)   = sum over those 4 columns of q*c
// and, for a single token, the shift is folded into the mask:
//   dp4a(act word i, w & (0x03030303 << 2i))  = 4^i * (same sum)
// kept in four accumulators and recombined exactly at the end. The result is
// sum_k q_k * (t_k + 1); subtracting sum_k q_k (summed while staging) gives
// the exact acc = sum_k q_k * t_k. A warp owns R rows at a time and reduces
// each with one redux; the epilogue applies y = fp32(acc * fp32(fp32(s_w*m)/127)).
#include "common.cuh"
#include "launchers.h"

namespace bl {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

template <int MT, int R>
__global__ void __launch_bounds__(kThreads) gemv_kernel(
    const uint8_t* __restrict__ Wp, int N, int K, const int8_t* __restrict__ q, const float* __restrict__ mrow,
    const float* __restrict__ s_w, int M, int t0, float* __restrict__ Y,
    int32_t* __restrict__ acc_out, int epi, float* __restrict__ absmax_out) {
  extern __shared__ __align__(16) uint4 sq[];       // [MT][K/16] activation groups (quad order)
  __shared__ int s_qsum[kWarps][MT];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K16 = K >> 4;
  const int C = K >> 6;                              // 16-byte chunks per weight row
  const size_t row_bytes = static_cast<size_t>(K) >> 2;

  pdl_wait();
  int qpart[MT];
#pragma unroll
  for (int t = 0; t < MT; ++t) qpart[t] = 0;
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    const bool live = t0 + t < M;
    const uint4* src = reinterpret_cast<const uint4*>(q + static_cast<size_t>(live ? t0 + t : 0) * K);
    for (int i = tid; i < K16; i += kThreads) {
      uint4 o = make_uint4(0u, 0u, 0u, 0u);
      if (live) {
        const uint4 v = __ldg(src + i);
        const uint32_t lo01 = __byte_perm(v.x, v.y, 0x5140), lo23 = __byte_perm(v.z, v.w, 0x5140);
        const uint32_t hi01 = __byte_perm(v.x, v.y, 0x7362), hi23 = __byte_perm(v.z, v.w, 0x7362);
        o.x = __byte_perm(lo01, lo23, 0x5410);
        o.y = __byte_perm(lo01, lo23, 0x7632);
        o.z = __byte_perm(hi01, hi23, 0x5410);
        o.w = __byte_perm(hi01, hi23, 0x7632);
        int qs = qpart[t];
        qs = dp4a_su(static_cast<int>(v.x), 0x01010101u, qs);
        qs = dp4a_su(static_cast<int>(v.y), 0x01010101u, qs);
        qs = dp4a_su(static_cast<int>(v.z), 0x01010101u, qs);
        qs = dp4a_su(static_cast<int>(v.w), 0x01010101u, qs);
        qpart[t] = qs;
      }
      sq[t * K16 + i] = o;
    }
  }
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    const int v = warp_sum(qpart[t]);
    if (lane == 0) s_qsum[warp][t] = v;
  }
  __syncthreads();
  pdl_trigger();
  int qsum[MT];
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    int v = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v += s_qsum[w][t];
    qsum[t] = v;
  }

  const float sw = s_w[0];
  const int groups = (N + R - 1) / R;
  for (int g = blockIdx.x * kWarps + warp; g < groups; g += gridDim.x * kWarps) {
    const int r0 = g * R;
    int acc[R][MT][(MT == 1) ? 4 : 1];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int i = 0; i < ((MT == 1) ? 4 : 1); ++i) acc[r][t][i] = 0;

    for (int c = lane; c < C; c += 32) {
      uint4 w[R];
#pragma unroll
      for (int r = 0; r < R; ++r)
        w[r] = (r0 + r < N) ? ldg_stream(Wp + static_cast<size_t>(r0 + r) * row_bytes + 16 * static_cast<size_t>(c))
                            : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        uint4 av[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) av[t] = sq[t * K16 + 4 * c + wi];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t wv = wi == 0 ? w[r].x : wi == 1 ? w[r].y : wi == 2 ? w[r].z : w[r].w;
          if constexpr (MT == 1) {
            acc[r][0][0] = dp4a_su(static_cast<int>(av[0].x), wv & 0x03030303u, acc[r][0][0]);
            acc[r][0][1] = dp4a_su(static_cast<int>(av[0].y), wv & 0x0C0C0C0Cu, acc[r][0][1]);
            acc[r][0][2] = dp4a_su(static_cast<int>(av[0].z), wv & 0x30303030u, acc[r][0][2]);
            acc[r][0][3] = dp4a_su(static_cast<int>(av[0].w), wv & 0xC0C0C0C0u, acc[r][0][3]);
          } else {
            const uint32_t x0 = wv & 0x03030303u, x1 = (wv >> 2) & 0x03030303u;
            const uint32_t x2 = (wv >> 4) & 0x03030303u, x3 = (wv >> 6) & 0x03030303u;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
              int s = acc[r][t][0];
              s = dp4a_su(static_cast<int>(av[t].x), x0, s);
              s = dp4a_su(static_cast<int>(av[t].y), x1, s);
              s = dp4a_su(static_cast<int>(av[t].z), x2, s);
              s = dp4a_su(static_cast<int>(av[t].w), x3, s);
              acc[r][t][0] = s;
            }
          }
        }
      }
    }

#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        int part;
        if constexpr (MT == 1)
          part = acc[r][0][0] + (acc[r][0][1] >> 2) + (acc[r][0][2] >> 4) + (acc[r][0][3] >> 6);
        else
          part = acc[r][t][0];
        const int total = warp_sum(part);
        const int row = r0 + r, tok = t0 + t;
        if (lane == ((r * MT + t) & 31) && row < N && tok < M) {
          const int a = total - qsum[t];
          float y = __fmul_rn(static_cast<float>(a), dequant_factor(sw, mrow[tok]));
          if (epi == static_cast<int>(Epi::kRelu2)) {
            y = y > 0.0f ? __fmul_rn(y, y) : 0.0f;
            if (absmax_out != nullptr) atomicMax(reinterpret_cast<unsigned int*>(absmax_out + tok), __float_as_uint(y));
          }
          const size_t o = static_cast<size_t>(tok) * N + row;
          Y[o] = y;
          if (acc_out != nullptr) acc_out[o] = a;
        }
      }
    }
  }
}

struct DevInfo {
  int sms = 148;
  int max_smem = 227 * 1024;
};

DevInfo dev_info() {
  DevInfo d;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  }
  return d;
}

template <int MT, int R>
cudaError_t launch_mt(const uint8_t* Wp, int N, int K, const int8_t* q, const float* m,
                      const float* s_w, int M, int t0, float* Y, int32_t* acc, Epi epi, float* absmax_out,
                      bool pdl, cudaStream_t st) {
  const DevInfo d = dev_info();
  const size_t smem = static_cast<size_t>(MT) * K;
  auto kern = gemv_kernel<MT, R>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  int occ = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
  if (err != cudaSuccess) return err;
  if (occ < 1) occ = 1;
  const int groups = (N + R - 1) / R;
  const int need = (groups + kWarps - 1) / kWarps;
  const int grid = std::max(1, std::min(need, occ * d.sms));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, Wp, N, K, q, m, s_w, M, t0, Y, acc, static_cast<int>(epi), absmax_out);
}

template <int MT>
cudaError_t launch_rows(const uint8_t* Wp, int N, int K, const int8_t* q, const float* m,
                        const float* s_w, int M, int t0, float* Y, int32_t* acc, Epi epi, float* absmax_out,
                        bool pdl, cudaStream_t st) {
  // Most rows per warp that still gives every SM at least two CTAs.
  const int sms = dev_info().sms;
  auto ctas = [&](int R) { return ((N + R - 1) / R + kWarps - 1) / kWarps; };
  if (ctas(4) >= 2 * sms) return launch_mt<MT, 4>(Wp, N, K, q, m, s_w, M, t0, Y, acc, epi, absmax_out, pdl, st);
  if (ctas(2) >= 2 * sms) return launch_mt<MT, 2>(Wp, N, K, q, m, s_w, M, t0, Y, acc, epi, absmax_out, pdl, st);
  return launch_mt<MT, 1>(Wp, N, K, q, m, s_w, M, t0, Y, acc, epi, absmax_out, pdl, st);
}

}  // namespace

cudaError_t launch_gemv(const uint8_t* Wp, int N, int K, const int8_t* q, const float* m,
                        const float* s_w, int M, float* Y, int32_t* acc, Epi epi, float* absmax_out, bool pdl,
                        cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  // tokens per pass: up to 4, limited by the shared memory that holds MT rows of K activations
  const int smem_cap = dev_info().max_smem - 1024;
  const int mt_cap = static_cast<int>(K) * 4 <= smem_cap ? 4 : (static_cast<int>(K) * 2 <= smem_cap ? 2 : 1);
  if (M == 1 || mt_cap == 1) {
    for (int t0 = 0; t0 < M; ++t0) {
      const cudaError_t err = launch_rows<1>(Wp, N, K, q, m, s_w, M, t0, Y, acc, epi, absmax_out, pdl, st);
      if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
  }
  if (M == 2 || mt_cap == 2) {
    for (int t0 = 0; t0 < M; t0 += 2) {
      const cudaError_t err = launch_rows<2>(Wp, N, K, q, m, s_w, M, t0, Y, acc, epi, absmax_out, pdl, st);
      if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
  }
  for (int t0 = 0; t0 < M; t0 += 4) {
    const cudaError_t err = launch_rows<4>(Wp, N, K, q, m, s_w, M, t0, Y, acc, epi, absmax_out, pdl, st);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace bl
