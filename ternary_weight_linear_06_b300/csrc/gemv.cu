// Decode GEMV for a few tokens: packed 2-bit ternary weights x int8 activations,
// per-token quantization fused in, over a table of independent problems.
//
// "BitNet b1.58 2B4T Technical Report | Summary", 5.1 GPU Inference: packed
// weights are loaded from HBM into shared memory, unpacked on chip and
// multiplied with 8-bit activations. "BitNet解读", 革命性的效率提升: with
// ternary weights the product is additions and subtractions of activations;
// 激活量化: each token is scaled to [-127, 127] by its absmax.
//
// Work split: the row quads (4 rows) of all problems of a launch form one
// sequence; CTA c owns a contiguous run of it, balanced by bytes. It walks its
// run in pieces (up to one stage of whole quads of one problem) that the TMA
// engine copies into a ring of shared-memory stages with cp.async.bulk.
//   1. thread 0 issues the first `stages` copies before the programmatic-
//      dependency wait (weights are only read), so they stream while the
//      preceding kernel finishes;
//   2. after the wait, the CTA quantizes the token rows of every problem it
//      touches into shared memory (redundantly per CTA: K values per token);
//   3. per piece, warps take (quad, K-part) units; the 32 lanes form 32/LPR
//      groups of LPR lanes, each group owning LPR/8 rows of the quad and
//      striding over its 16-byte chunks, so one shared-memory read of a
//      chunk's activations serves all groups; partial sums meet in shared
//      memory, then the epilogue writes y for every row of the piece.
//
// Packed rows are K/4 bytes (code t+1 of column 4b+j in bits [2j,2j+1] of byte
// b): in a 32-bit word the code of column 16w+4j+i sits at bit 8j+2i. The
// activations are kept in "quad" order (word i of a 16-column group holds
// columns i, 4+i, 8+i, 12+i), so
//   dp4a(act word i, (w >> 2i) & 0x03030303)  = sum over those 4 columns of q*c
// and, for one token, the shift is folded into the mask:
//   dp4a(act word i, w & (0x03030303 << 2i)) = 4^i * (same sum),
// kept in four accumulators and recombined exactly. The result is
// sum_k q_k * (t_k + 1); subtracting sum_k q_k gives acc = sum_k q_k * t_k,
// and y = fp32(acc * fp32(fp32(s_w * m) / 127)).
#include "common.cuh"
#include "launchers.h"

namespace bl {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxCtas = 160;     // one CTA per SM; >= the 148 SMs of a B300
constexpr int kMaxStages = 4;
constexpr int kMaxSpan = 8;       // problems one CTA may touch
constexpr int kRowsCap = 256;     // rows per piece (partial-sum slots)
constexpr int kUnroll = 2;

struct DevProb {
  const uint8_t* Wp;
  const void* X;          // unquantized input, or null
  const int8_t* q;        // already-quantized input (row-major int8), or null
  const float* m_in;
  const float* s_w;
  float* Y;
  int32_t* acc;
  float* absmax_out;
  float eps;
  int N, K, M;
  int x_dtype;
  int epi;
  int quad_begin;         // index of the problem's first quad in the launch sequence
};

template <int CAP>
struct BatchArgs {
  DevProb prob[CAP];
  int cta_quad[kMaxCtas + 1];   // CTA c owns quads [cta_quad[c], cta_quad[c+1])
  int count;
  int t0;                       // tokens t0 .. t0+MT-1 of every problem
  int stage_bytes;
  int stages;
  int act_cap;                  // bytes of the activation area
  int trigger;                  // trigger dependents at kernel start
  WsHeader* status;
};

__host__ __device__ __forceinline__ int quads_of(const DevProb& p) { return (p.N + 3) >> 2; }

// Next piece of a CTA's run: quads [qa, qb) of problem p, with q advanced.
template <int CAP>
__device__ __forceinline__ bool next_piece(const BatchArgs<CAP>& a, int& p, int& q, int q_end, int& qa, int& qb) {
  if (q >= q_end) return false;
  while (a.prob[p].quad_begin + quads_of(a.prob[p]) <= q) ++p;
  const DevProb& P = a.prob[p];
  const int qbytes = P.K;                                   // 4 rows of K/4 bytes
  const int by_bytes = max(1, a.stage_bytes / qbytes);
  const int by_rows = kRowsCap / 4;
  qa = q;
  qb = min(min(q + min(by_bytes, by_rows), P.quad_begin + quads_of(P)), q_end);
  q = qb;
  return true;
}

template <int CAP>
__device__ __forceinline__ void issue_piece(const BatchArgs<CAP>& a, int p, int qa, int qb, uint8_t* dst,
                                            uint64_t* bar) {
  const DevProb& P = a.prob[p];
  const size_t rb = static_cast<size_t>(P.K) >> 2;
  const int r0 = 4 * (qa - P.quad_begin);
  const int r1 = min(P.N, 4 * (qb - P.quad_begin));
  const uint32_t bytes = static_cast<uint32_t>((r1 - r0) * rb);
  mbar_arrive_expect_tx(bar, bytes);
  bulk_copy_g2s(dst, P.Wp + static_cast<size_t>(r0) * rb, bytes, bar);
}

__device__ __forceinline__ uint32_t quad_word(int a, int b, int c, int d) {
  return (static_cast<uint32_t>(a) & 0xFFu) | ((static_cast<uint32_t>(b) & 0xFFu) << 8) |
         ((static_cast<uint32_t>(c) & 0xFFu) << 16) | ((static_cast<uint32_t>(d) & 0xFFu) << 24);
}

// 4x4 byte transpose of a 16-column group: row-major bytes -> quad order.
__device__ __forceinline__ uint4 to_quad(uint4 v) {
  const uint32_t lo01 = __byte_perm(v.x, v.y, 0x5140), lo23 = __byte_perm(v.z, v.w, 0x5140);
  const uint32_t hi01 = __byte_perm(v.x, v.y, 0x7362), hi23 = __byte_perm(v.z, v.w, 0x7362);
  return make_uint4(__byte_perm(lo01, lo23, 0x5410), __byte_perm(lo01, lo23, 0x7632),
                    __byte_perm(hi01, hi23, 0x5410), __byte_perm(hi01, hi23, 0x7632));
}

// Quantize (or copy) tokens t0..t0+MT-1 of one problem into `sq` in quad
// order; scale -> s_m[t], sum of codes -> s_qs[t]. All threads take part.
template <int MT, int DT>
__device__ void stage_tokens(const DevProb& P, int t0, uint4* sq, float* s_m, int* s_qs, float (*s_red)[MT],
                             int (*s_ired)[MT]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K16 = P.K >> 4;
  const bool fused = P.X != nullptr;
  constexpr size_t esize = DT == BL_DTYPE_F32 ? 4 : 2;
  float m_t[MT];
  if (fused) {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      float amax = 0.0f;
      if (t0 + t < P.M) {
        const void* xr = static_cast<const char*>(P.X) + static_cast<size_t>(t0 + t) * P.K * esize;
        for (int g = tid; g < K16; g += kThreads) {
          float v[16];
          load16<DT>(xr, g, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
        }
      }
      amax = warp_max(amax);
      if (lane == 0) s_red[warp][t] = amax;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v = fmaxf(v, s_red[w][t]);
      m_t[t] = fmaxf(v, P.eps);
    }
  }
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    int qpart = 0;
    const bool live = t0 + t < P.M;
    const int row = live ? t0 + t : 0;
    if (fused) {
      const void* xr = static_cast<const char*>(P.X) + static_cast<size_t>(row) * P.K * esize;
      for (int g = tid; g < K16; g += kThreads) {
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (live) {
          float v[16];
          load16<DT>(xr, g, v);
          int qv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            qv[j] = quant_one(v[j], m_t[t]);
            qpart += qv[j];
          }
          o = make_uint4(quad_word(qv[0], qv[4], qv[8], qv[12]), quad_word(qv[1], qv[5], qv[9], qv[13]),
                         quad_word(qv[2], qv[6], qv[10], qv[14]), quad_word(qv[3], qv[7], qv[11], qv[15]));
        }
        sq[t * K16 + g] = o;
      }
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(P.q + static_cast<size_t>(row) * P.K);
      for (int g = tid; g < K16; g += kThreads) {
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (live) {
          const uint4 v = __ldg(src + g);
          o = to_quad(v);
          qpart = dp4a_su(static_cast<int>(v.x), 0x01010101u, qpart);
          qpart = dp4a_su(static_cast<int>(v.y), 0x01010101u, qpart);
          qpart = dp4a_su(static_cast<int>(v.z), 0x01010101u, qpart);
          qpart = dp4a_su(static_cast<int>(v.w), 0x01010101u, qpart);
        }
        sq[t * K16 + g] = o;
      }
    }
    qpart = warp_sum(qpart);
    if (lane == 0) s_ired[warp][t] = qpart;
  }
  __syncthreads();
  if (tid < MT) {
    int v = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v += s_ired[w][tid];
    s_qs[tid] = v;
    float mv = 1.0f;
    if (fused) {
#pragma unroll
      for (int t = 0; t < MT; ++t)
        if (t == tid) mv = m_t[t];
    } else if (t0 + tid < P.M) {
      mv = P.m_in[t0 + tid];
    }
    s_m[tid] = mv;
  }
  __syncthreads();
}

// One (quad, K-part) unit: rows 4*jq .. 4*jq+3 of the piece in `wbuf`,
// chunks [c_begin, c_end). Adds the partial sums of sum_k q*(t+1) into s_acc.
template <int MT, int LPR>
__device__ __forceinline__ void run_unit(const uint8_t* wbuf, int rows, int rb, const uint4* sq, int K16, int jq,
                                         int c_begin, int c_end, int* s_acc) {
  constexpr int RL = LPR / 8;
  const int lane = threadIdx.x & 31;
  const int grp = lane / LPR, sub = lane % LPR;
  const int rbase = 4 * jq + grp * RL;
  int acc[RL][MT][(MT == 1) ? 4 : 1];
#pragma unroll
  for (int r = 0; r < RL; ++r)
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int i = 0; i < ((MT == 1) ? 4 : 1); ++i) acc[r][t][i] = 0;
  bool rvalid[RL];
  const uint8_t* wrow[RL];
#pragma unroll
  for (int r = 0; r < RL; ++r) {
    rvalid[r] = rbase + r < rows;
    wrow[r] = wbuf + static_cast<size_t>(rvalid[r] ? rbase + r : 0) * rb;
  }
  for (int c0 = c_begin + sub; c0 < c_end; c0 += kUnroll * LPR) {
    uint4 w[kUnroll][RL];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = c0 + u * LPR;
#pragma unroll
      for (int r = 0; r < RL; ++r)
        w[u][r] = (c < c_end && rvalid[r]) ? *reinterpret_cast<const uint4*>(wrow[r] + 16 * c)
                                           : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = c0 + u * LPR;
      if (c >= c_end) break;
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        uint4 av[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) av[t] = sq[t * K16 + 4 * c + wi];
#pragma unroll
        for (int r = 0; r < RL; ++r) {
          const uint32_t wv = wi == 0 ? w[u][r].x : wi == 1 ? w[u][r].y : wi == 2 ? w[u][r].z : w[u][r].w;
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
  }
#pragma unroll
  for (int r = 0; r < RL; ++r) {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      int v;
      if constexpr (MT == 1)
        v = acc[r][0][0] + (acc[r][0][1] >> 2) + (acc[r][0][2] >> 4) + (acc[r][0][3] >> 6);
      else
        v = acc[r][t][0];
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (sub == ((r * MT + t) % LPR) && rvalid[r]) atomicAdd(&s_acc[(rbase + r) * MT + t], v);
    }
  }
}

// Lanes per row for a run of C chunks: the choice that wastes the fewest
// lane-chunk slots, more lanes on ties.
__host__ __device__ inline int lpr_for_chunks(int C) {
  int best = 8, best_num = -1, best_den = 1;
  for (int lpr = 8; lpr <= 32; lpr *= 2) {
    const int den = lpr * ((C + lpr - 1) / lpr);
    if (static_cast<long long>(C) * best_den >= static_cast<long long>(best_num) * den) {
      best_num = C;
      best_den = den;
      best = lpr;
    }
  }
  return best;
}

template <int MT, int CAP>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const __grid_constant__ BatchArgs<CAP> a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[kMaxStages];
  __shared__ float s_m[kMaxSpan][MT];
  __shared__ int s_qs[kMaxSpan][MT];
  __shared__ float s_sw[kMaxSpan];
  __shared__ int s_act_off[kMaxSpan];
  __shared__ float s_red[kWarps][MT];
  __shared__ int s_ired[kWarps][MT];

  const int tid = threadIdx.x, warp = tid >> 5;
  const int q_begin = a.cta_quad[blockIdx.x], q_end = a.cta_quad[blockIdx.x + 1];
  uint8_t* ring = smem;
  uint8_t* act = smem + static_cast<size_t>(a.stages) * a.stage_bytes;
  int* s_acc = reinterpret_cast<int*>(act + a.act_cap);

  // 1. start the weight stream (weights are never written by the kernels
  //    that precede this one in a programmatic-dependency chain)
  int pp = 0, pq = q_begin;   // producer cursor (thread 0)
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
    for (int s = 0; s < a.stages; ++s) {
      int qa, qb;
      if (!next_piece(a, pp, pq, q_end, qa, qb)) break;
      issue_piece(a, pp, qa, qb, ring + static_cast<size_t>(s) * a.stage_bytes, &full[s]);
    }
  }
  for (int i = tid; i < kRowsCap * MT; i += kThreads) s_acc[i] = 0;
  __syncthreads();
  if (a.trigger) pdl_trigger();
  pdl_wait();

  // 2. activations of every problem this CTA touches
  int p_first = 0, nspan = 0;
  if (q_begin < q_end) {
    while (a.prob[p_first].quad_begin + quads_of(a.prob[p_first]) <= q_begin) ++p_first;
    int p_last = p_first;
    while (a.prob[p_last].quad_begin + quads_of(a.prob[p_last]) < q_end) ++p_last;
    nspan = p_last - p_first + 1;
  }
  {
    int off = 0;
    for (int j = 0; j < nspan; ++j) {
      const DevProb& P = a.prob[p_first + j];
      if (tid == 0) {
        s_act_off[j] = off;
        s_sw[j] = P.s_w[0];
      }
      uint4* sq = reinterpret_cast<uint4*>(act + off);
      if (P.X != nullptr && P.x_dtype == BL_DTYPE_BF16)
        stage_tokens<MT, BL_DTYPE_BF16>(P, a.t0, sq, s_m[j], s_qs[j], s_red, s_ired);
      else
        stage_tokens<MT, BL_DTYPE_F32>(P, a.t0, sq, s_m[j], s_qs[j], s_red, s_ired);
      off += MT * P.K;
    }
  }
  __syncthreads();

  // 3. pieces
  const uint64_t deadline = global_ns() + kWaitLimitNs;
  int cp = 0, cq = q_begin;   // consumer cursor (all threads)
  int i_abort = -1;
  for (int i = 0;; ++i) {
    int qa, qb;
    if (!next_piece(a, cp, cq, q_end, qa, qb)) break;
    const int s = i % a.stages;
    const bool ok = mbar_wait_until(&full[s], static_cast<uint32_t>((i / a.stages) & 1), deadline);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) report_status(a.status, BL_ERR_TIMEOUT, 0x100u + blockIdx.x);
      i_abort = i;
      break;
    }
    const DevProb& P = a.prob[cp];
    const int j = cp - p_first;
    const int rb = P.K >> 2;
    const int rows = min(P.N, 4 * (qb - P.quad_begin)) - 4 * (qa - P.quad_begin);
    const int nq = qb - qa;
    const int C = P.K >> 6;
    int kp = 1;
    while (kp < 8 && nq * kp < kWarps && C / (2 * kp) >= 8) kp *= 2;
    const uint8_t* wbuf = ring + static_cast<size_t>(s) * a.stage_bytes;
    const uint4* sq = reinterpret_cast<const uint4*>(act + s_act_off[j]);
    const int lpr = lpr_for_chunks(C / kp);
    for (int u = warp; u < nq * kp; u += kWarps) {
      const int jq = u / kp, part = u % kp;
      const int cb = static_cast<int>(static_cast<long long>(C) * part / kp);
      const int ce = static_cast<int>(static_cast<long long>(C) * (part + 1) / kp);
      if (lpr == 8) run_unit<MT, 8>(wbuf, rows, rb, sq, P.K >> 4, jq, cb, ce, s_acc);
      else if (lpr == 16) run_unit<MT, 16>(wbuf, rows, rb, sq, P.K >> 4, jq, cb, ce, s_acc);
      else run_unit<MT, 32>(wbuf, rows, rb, sq, P.K >> 4, jq, cb, ce, s_acc);
    }
    __syncthreads();
    // epilogue for the piece's rows
    const int row0 = 4 * (qa - P.quad_begin);
    const float sw = s_sw[j];
    for (int idx = tid; idx < rows * MT; idx += kThreads) {
      const int r = idx / MT, t = idx % MT;
      const int tok = a.t0 + t;
      const int v = s_acc[idx];
      s_acc[idx] = 0;
      if (tok < P.M) {
        const int accv = v - s_qs[j][t];
        float y = __fmul_rn(static_cast<float>(accv), dequant_factor(sw, s_m[j][t]));
        if (P.epi == static_cast<int>(Epi::kRelu2)) {
          y = y > 0.0f ? __fmul_rn(y, y) : 0.0f;
          if (P.absmax_out != nullptr)
            atomicMax(reinterpret_cast<unsigned int*>(P.absmax_out + tok), __float_as_uint(y));
        }
        const size_t o = static_cast<size_t>(tok) * P.N + row0 + r;
        P.Y[o] = y;
        if (P.acc != nullptr) P.acc[o] = accv;
      }
    }
    __syncthreads();
    // refill the stage just consumed
    if (tid == 0) {
      int qa2, qb2;
      if (next_piece(a, pp, pq, q_end, qa2, qb2)) {
        fence_proxy_async_smem();
        issue_piece(a, pp, qa2, qb2, ring + static_cast<size_t>(s) * a.stage_bytes, &full[s]);
      }
    }
  }
  if (i_abort >= 0 && tid == 0) {
    // let the copies still in flight (pieces i_abort .. i_abort+stages-1 at
    // most) land before the CTA's shared memory is released
    const uint64_t d2 = global_ns() + kWaitLimitNs / 4;
    for (int k = i_abort; k < i_abort + a.stages; ++k)
      (void)mbar_wait_until(&full[k % a.stages], static_cast<uint32_t>((k / a.stages) & 1), d2);
  }
}

struct DevInfo {
  int sms = 148;
  int max_smem = 227 * 1024;
};

DevInfo dev_info() {
  static thread_local int cached_dev = -1;
  static thread_local DevInfo cached;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cached;
  if (dev != cached_dev) {
    DevInfo d;
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cached = d;
    cached_dev = dev;
  }
  return cached;
}

// Host-side plan for one launch: CTA runs balanced by bytes, stage size,
// activation area. Returns false if the problems cannot share one launch.
template <int CAP>
bool plan(BatchArgs<CAP>& a, int mt, int sms, int smem_limit, bool single) {
  long long total = 0;
  int quads = 0;
  int maxK = 0;
  for (int i = 0; i < a.count; ++i) {
    DevProb& P = a.prob[i];
    P.quad_begin = quads;
    quads += quads_of(P);
    total += static_cast<long long>(P.N) * (P.K / 4);
    maxK = std::max(maxK, P.K);
  }
  if (quads == 0) return false;
  const int grid = std::max(1, std::min(std::min(sms, kMaxCtas), quads));
  // boundaries: first quad whose cumulative byte count reaches c/grid of the total
  int c = 1, p = 0;
  long long cum = 0;
  a.cta_quad[0] = 0;
  for (int g = 0; g < quads && c < grid; ++g) {
    while (a.prob[p].quad_begin + quads_of(a.prob[p]) <= g) ++p;
    const DevProb& P = a.prob[p];
    const int lq = g - P.quad_begin;
    const int rows = std::min(4, P.N - 4 * lq);
    cum += static_cast<long long>(rows) * (P.K / 4);
    while (c < grid && cum * grid >= total * c) a.cta_quad[c++] = g + 1;
  }
  while (c <= grid) a.cta_quad[c++] = quads;
  for (int i = grid + 1; i <= kMaxCtas; ++i) a.cta_quad[i] = quads;
  // activation area: the most any CTA needs; at most kMaxSpan problems per CTA
  int act = 0;
  for (int b = 0; b < grid; ++b) {
    const int qa = a.cta_quad[b], qb = a.cta_quad[b + 1];
    if (qa >= qb) continue;
    int p0 = 0;
    while (a.prob[p0].quad_begin + quads_of(a.prob[p0]) <= qa) ++p0;
    int p1 = p0;
    while (a.prob[p1].quad_begin + quads_of(a.prob[p1]) < qb) ++p1;
    if (p1 - p0 + 1 > kMaxSpan) return false;
    int need = 0;
    for (int q = p0; q <= p1; ++q) need += mt * a.prob[q].K;
    act = std::max(act, need);
  }
  a.act_cap = static_cast<int>(align_up(static_cast<size_t>(act), 128));
  a.stage_bytes = static_cast<int>(align_up(static_cast<size_t>(std::max(single ? 16384 : 32768, maxK)), 128));
  const int acc_bytes = kRowsCap * mt * 4;
  const int room = smem_limit - a.act_cap - acc_bytes - 1024;
  a.stages = std::min(kMaxStages, room / a.stage_bytes);
  return a.stages >= 2;
}

template <int MT, int CAP>
cudaError_t launch_batch(BatchArgs<CAP>& a, bool pdl, cudaStream_t st, bool* planned) {
  const DevInfo d = dev_info();
  *planned = plan(a, MT, d.sms, d.max_smem, CAP == 1);
  if (!*planned) return cudaSuccess;
  int grid = 0;
  while (grid < kMaxCtas && a.cta_quad[grid] < a.cta_quad[kMaxCtas]) ++grid;
  grid = std::max(grid, 1);
  const size_t smem = static_cast<size_t>(a.stages) * a.stage_bytes + a.act_cap + kRowsCap * MT * 4;
  auto kern = gemv_kernel<MT, CAP>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
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
  return cudaLaunchKernelEx(&cfg, kern, a);
}

DevProb to_dev(const GemvProblem& p) {
  DevProb d = {};
  d.Wp = p.Wp;
  d.X = p.X;
  d.q = p.q;
  d.m_in = p.m;
  d.s_w = p.s_w;
  d.Y = p.Y;
  d.acc = p.acc;
  d.absmax_out = p.absmax_out;
  d.eps = p.eps;
  d.N = p.N;
  d.K = p.K;
  d.M = p.M;
  d.x_dtype = p.x_dtype;
  d.epi = static_cast<int>(p.epi);
  return d;
}

template <int MT, int CAP>
cudaError_t run_tokens(const GemvProblem* ps, int count, int t0, WsHeader* status, bool pdl, cudaStream_t st,
                       bool* planned) {
  BatchArgs<CAP> a;
  int n = 0;
  for (int i = 0; i < count; ++i)
    if (ps[i].N > 0 && ps[i].M > t0) a.prob[n++] = to_dev(ps[i]);
  *planned = true;
  if (n == 0) return cudaSuccess;
  a.count = n;
  a.t0 = t0;
  a.trigger = 1;
  a.status = status;
  return launch_batch<MT, CAP>(a, pdl, st, planned);
}

template <int CAP>
cudaError_t run_all(const GemvProblem* ps, int count, WsHeader* status, bool pdl, cudaStream_t st) {
  int maxM = 0, maxK = 0;
  for (int i = 0; i < count; ++i) {
    maxM = std::max(maxM, ps[i].M);
    maxK = std::max(maxK, ps[i].K);
  }
  // tokens per launch: up to 4, fewer when MT rows of the longest K do not
  // leave room for two weight stages
  const int limit = dev_info().max_smem - 2 * std::max(32768, maxK) - 8192;
  const int mt_cap = 4 * maxK <= limit ? 4 : (2 * maxK <= limit ? 2 : 1);
  const int mt = std::min(mt_cap, maxM <= 1 ? 1 : (maxM == 2 ? 2 : 4));
  for (int t0 = 0; t0 < maxM; t0 += mt) {
    bool planned = true;
    cudaError_t err;
    if (mt == 1) err = run_tokens<1, CAP>(ps, count, t0, status, pdl, st, &planned);
    else if (mt == 2) err = run_tokens<2, CAP>(ps, count, t0, status, pdl, st, &planned);
    else err = run_tokens<4, CAP>(ps, count, t0, status, pdl, st, &planned);
    if (err != cudaSuccess) return err;
    if (!planned) {
      if (count == 1) return cudaErrorInvalidConfiguration;
      // split the batch in halves (each half plans its own CTA runs)
      const int h = count / 2;
      err = run_all<CAP>(ps, h, status, pdl, st);
      if (err != cudaSuccess) return err;
      return run_all<CAP>(ps + h, count - h, status, pdl, st);
    }
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemv(const GemvProblem& p, WsHeader* status, bool pdl, cudaStream_t st) {
  if (p.M == 0 || p.N == 0) return cudaSuccess;
  return run_all<1>(&p, 1, status, pdl, st);
}

cudaError_t launch_gemv_batch(const GemvProblem* ps, int count, WsHeader* status, bool pdl, cudaStream_t st) {
  if (count <= 0) return cudaSuccess;
  if (count == 1) return launch_gemv(ps[0], status, pdl, st);
  return run_all<kGemvMaxBatch>(ps, count, status, pdl, st);
}

}  // namespace bl
