// Decode GEMV for a few tokens: packed 2-bit ternary weights x int8 activations
// over a table of independent problems.
//
// "BitNet b1.58 2B4T Technical Report | Summary", 5.1 GPU Inference: packed
// weights are loaded from HBM, unpacked on chip and multiplied with 8-bit
// activations. "BitNet解读", 革命性的效率提升: with ternary weights the product
// is additions and subtractions of activations.
//
// The activations arrive quantized (int8, row-major, with their per-token
// scale m) from the quantization kernel that precedes this one, or, for a
// single problem of a few short rows, raw (fp32/bf16): the CTAs then quantize
// them while staging, with the quantization kernel's code rule.
//
// Work split. The rows of all problems of a launch form one sequence; CTA c
// owns a contiguous run of it, balanced by packed bytes (two CTAs of 16 warps
// per SM: 32 warps with 128-bit loads in flight are what it takes to stream
// HBM).
//   1. thread 0 asks L2 to prefetch the start of the CTA's weight run, then
//      the CTA waits for the preceding kernel (programmatic dependent launch)
//      and copies the token rows of every problem its run touches into shared
//      memory, transposed into the order below, with each token's sum of
//      codes and dequant factor;
//   2. the run is cut into items of G = 32/LPR rows of one problem; warps
//      take items round-robin. In an item the 32 lanes form G groups of LPR
//      lanes, one group per row; lane `sub` of a group reads the row's 16-byte
//      chunks sub, sub + LPR, ... straight from HBM with 128-bit loads into
//      registers, in batches of kUnroll chunks. Every lane group reads the
//      same activation chunk at the same time (a shared-memory broadcast);
//   3. the LPR partial sums of a row meet by warp shuffles and one lane per
//      token writes y.
// LPR is picked per problem by a cost model (a warp's item costs about its
// chunks per lane plus one): 4 lanes for every 2B- and 70B-class row; a
// launch with too few rows to give every warp two items widens the groups.
//
// Packed rows are K/4 bytes (code t+1 of column 4b+j in bits [2j,2j+1] of byte
// b): in a 32-bit word the code of column 16w+4j+i sits at bit 8j+2i. The
// activations of a 16-column group g are kept as four "quad" words (word i
// holds columns 16g+i, 16g+4+i, 16g+8+i, 16g+12+i), so
//   dp4a(quad word i, (w >> 2i) & 0x03030303)  = sum over those 4 columns of q*c
// and, for one token, the shift is folded into the mask:
//   dp4a(quad word i, w & (0x03030303 << 2i)) = 4^i * (same sum),
// kept in four accumulators and recombined exactly. The result is
// sum_k q_k * (t_k + 1); subtracting sum_k q_k gives acc = sum_k q_k * t_k,
// and y = fp32(acc * fp32(fp32(s_w * m) / 127)).
// In shared memory the 16 bytes of group g = 4c + j (chunk c, word j) sit at
// uint4 index j * C + c (C = K / 64 chunks per row), so the LPR lanes of a
// group, reading consecutive chunks, hit consecutive 16-byte slots.
#include "common.cuh"
#include "launchers.h"

namespace bl {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kCtasPerSm = 2;              // 32 warps per SM
constexpr int kMaxCtas = 320;              // >= 2 x the 148 SMs of a B300
constexpr int kMaxSpan = 8;                // problems one CTA may touch
constexpr int kActBudget = 100 * 1024;     // shared memory for staged activations (two CTAs per SM)
// 16-byte weight loads per lane per batch (fewer when several tokens need
// registers for their accumulators and activations)
template <int MT>
constexpr int kUnroll = MT == 1 ? 8 : 4;

struct DevProb {
  const uint8_t* Wp;
  const int8_t* q;        // quantized activations, row-major [M][K]
  const float* m_in;      // their per-token scales [M]
  const float* s_w;
  float* Y;
  int32_t* acc;
  const float* mul;       // [M][N] or null: y = fp32(y * mul)
  const void* x;          // raw activations [M][K] when the launch quantizes them itself
  int x_dtype;
  float eps;
  int N, K, M;
  int epi;
  int lpr;                // lanes per row
  int row_begin;          // first row of the problem in the launch's row sequence
};

template <int CAP>
struct BatchArgs {
  DevProb prob[CAP];
  int cta_row[kMaxCtas + 1];        // CTA c owns rows [cta_row[c], cta_row[c+1])
  unsigned char cta_p0[kMaxCtas];   // the problem holding row cta_row[c]
  int count;
  int t0;                           // tokens t0 .. t0+MT-1 of every problem
  int from_x;                       // quantize the token rows from DevProb::x while staging
};

// What one CTA knows about a problem its run touches.
template <int MT>
struct Span {
  int p;             // problem index
  int r0, r1;        // rows [r0, r1) of the problem in this CTA's run
  int item0;         // index of the span's first item among the CTA's items
  int act;           // uint4 offset of the staged activations
  float c[MT];       // dequant factor fp32(fp32(s_w * m) / 127) of each token
  int qs[MT];        // sum of the token's codes
};

// 4x4 byte transpose of a 16-column group: row-major bytes -> quad order.
__device__ __forceinline__ uint4 to_quad(uint4 v) {
  const uint32_t lo01 = __byte_perm(v.x, v.y, 0x5140), lo23 = __byte_perm(v.z, v.w, 0x5140);
  const uint32_t hi01 = __byte_perm(v.x, v.y, 0x7362), hi23 = __byte_perm(v.z, v.w, 0x7362);
  return make_uint4(__byte_perm(lo01, lo23, 0x5410), __byte_perm(lo01, lo23, 0x7632),
                    __byte_perm(hi01, hi23, 0x5410), __byte_perm(hi01, hi23, 0x7632));
}

// Copy the token rows of every span into shared memory in one pass: the
// spans' rows lie end to end in the activation area (span j from uint4 offset
// spans[j].act, MT rows of K/16 groups each), and thread tid takes the
// 16-column groups tid, tid + kThreads, ... of that area, transposing each
// into the order above. The sums of codes meet in shared memory by atomics;
// then each token's dequant factor is computed once.
template <int MT, int CAP>
__device__ void stage_all(const BatchArgs<CAP>& a, Span<MT>* spans, int nspan, uint4* s_act, int* s_qs,
                          unsigned* s_amax) {
  const int tid = threadIdx.x;
  const int total = spans[nspan - 1].act + MT * (a.prob[spans[nspan - 1].p].K >> 4);
  if (a.from_x) {
    // per-token absmax of the raw rows first (non-negative floats order like
    // their bit patterns, so an integer max reduces them exactly)
    int j = 0;
    for (int g = tid; g < total; g += kThreads) {
      while (j + 1 < nspan && spans[j + 1].act <= g) ++j;
      const DevProb& P = a.prob[spans[j].p];
      const int K16 = P.K >> 4;
      const int local = g - spans[j].act;
      const int t = local / K16, gg = local - t * K16;
      if (a.t0 + t < P.M) {
        float v[16];
        const size_t off = static_cast<size_t>(a.t0 + t) * P.K;
        if (P.x_dtype == BL_DTYPE_F32) load16<BL_DTYPE_F32>(static_cast<const float*>(P.x) + off, gg, v);
        else load16<BL_DTYPE_BF16>(static_cast<const uint16_t*>(P.x) + off, gg, v);
        float mx = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(v[i]));
        atomicMax(&s_amax[j * MT + t], __float_as_uint(mx));
      }
    }
    __syncthreads();
  }
  int j = 0;
  for (int g = tid; g < total; g += kThreads) {
    while (j + 1 < nspan && spans[j + 1].act <= g) ++j;
    const DevProb& P = a.prob[spans[j].p];
    const int K16 = P.K >> 4, C = P.K >> 6;
    const int local = g - spans[j].act;
    const int t = local / K16, gg = local - t * K16;
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (a.t0 + t < P.M) {
      uint4 v;
      if (a.from_x) {
        // the same codes as the quantization kernel: m = max(absmax, eps)
        const float m = fmaxf(__uint_as_float(s_amax[j * MT + t]), P.eps);
        const float s127 = __fmul_rn(127.0f, __frcp_rn(m));
        float f[16];
        const size_t off = static_cast<size_t>(a.t0 + t) * P.K;
        if (P.x_dtype == BL_DTYPE_F32) load16<BL_DTYPE_F32>(static_cast<const float*>(P.x) + off, gg, f);
        else load16<BL_DTYPE_BF16>(static_cast<const uint16_t*>(P.x) + off, gg, f);
        int c[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) c[i] = static_cast<int>(quant_round(f[i], m, s127));
        v = make_uint4(pack4(c[0], c[1], c[2], c[3]), pack4(c[4], c[5], c[6], c[7]), pack4(c[8], c[9], c[10], c[11]),
                       pack4(c[12], c[13], c[14], c[15]));
      } else {
        v = __ldg(reinterpret_cast<const uint4*>(P.q + static_cast<size_t>(a.t0 + t) * P.K) + gg);
      }
      o = to_quad(v);
      int qpart = dp4a_su(static_cast<int>(v.x), 0x01010101u, 0);
      qpart = dp4a_su(static_cast<int>(v.y), 0x01010101u, qpart);
      qpart = dp4a_su(static_cast<int>(v.z), 0x01010101u, qpart);
      qpart = dp4a_su(static_cast<int>(v.w), 0x01010101u, qpart);
      atomicAdd(&s_qs[j * MT + t], qpart);
    }
    s_act[spans[j].act + t * K16 + (gg & 3) * C + (gg >> 2)] = o;
  }
  __syncthreads();
  if (tid < nspan * MT) {
    const int jj = tid / MT, t = tid - jj * MT;
    const DevProb& P = a.prob[spans[jj].p];
    spans[jj].qs[t] = s_qs[tid];
    float m = 0.0f;
    if (a.t0 + t < P.M) m = a.from_x ? fmaxf(__uint_as_float(s_amax[tid]), P.eps) : P.m_in[a.t0 + t];
    spans[jj].c[t] = a.t0 + t < P.M ? dequant_factor(P.s_w[0], m) : 0.0f;
  }
  __syncthreads();
}

// One batch of up to U chunks of a lane's row: loads issued together, then
// consumed. FULL: all U chunks exist (no per-chunk checks).
template <int MT, int LPR, int U, bool FULL>
__device__ __forceinline__ void gemv_batch(const uint4* wrow, int c0, int lim, bool valid, const uint4* a0, int C,
                                           int (&acc)[MT][MT == 1 ? 4 : 1]) {
  uint4 w[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if constexpr (FULL) w[u] = __ldg(wrow + c0 + u * LPR);
    else w[u] = (valid && u * LPR < lim) ? __ldg(wrow + c0 + u * LPR) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (!FULL && u * LPR >= lim) break;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t wv = j == 0 ? w[u].x : j == 1 ? w[u].y : j == 2 ? w[u].z : w[u].w;
      if constexpr (MT == 1) {
        const uint4 av = a0[j * C + u * LPR];
        acc[0][0] = dp4a_su(static_cast<int>(av.x), wv & 0x03030303u, acc[0][0]);
        acc[0][1] = dp4a_su(static_cast<int>(av.y), wv & 0x0C0C0C0Cu, acc[0][1]);
        acc[0][2] = dp4a_su(static_cast<int>(av.z), wv & 0x30303030u, acc[0][2]);
        acc[0][3] = dp4a_su(static_cast<int>(av.w), wv & 0xC0C0C0C0u, acc[0][3]);
      } else {
        const uint32_t x0 = wv & 0x03030303u, x1 = (wv >> 2) & 0x03030303u;
        const uint32_t x2 = (wv >> 4) & 0x03030303u, x3 = (wv >> 6) & 0x03030303u;
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const uint4 av = a0[(t * 4 + j) * C + u * LPR];
          int s = acc[t][0];
          s = dp4a_su(static_cast<int>(av.x), x0, s);
          s = dp4a_su(static_cast<int>(av.y), x1, s);
          s = dp4a_su(static_cast<int>(av.z), x2, s);
          s = dp4a_su(static_cast<int>(av.w), x3, s);
          acc[t][0] = s;
        }
      }
    }
  }
}

// One warp's share of a span: items (32/LPR rows each, one row per lane
// group) it = it0, it0 + kWarps, ... A row's C chunks are read in batches of
// up to U chunks per lane; the U loads of a batch are issued together, then
// consumed. Latency is hidden by the 32 warps each SM runs (two CTAs).
template <int MT, int LPR, int U>
__device__ __forceinline__ void run_span(const DevProb& P, const Span<MT>& S, const uint4* act, int it0, int t0) {
  constexpr int G = 32 / LPR;
  constexpr int NA = (MT == 1) ? 4 : 1;
  const int lane = threadIdx.x & 31;
  const int grp = lane / LPR, sub = lane % LPR;
  const int C = P.K >> 6;
  const int n_per = (C + LPR - 1) / LPR;               // chunks per lane per row
  const int nb = (n_per + U - 1) / U;                  // batches per row
  // full batches first (measured: more loads in flight beats an even split);
  // a lane whose batch is complete skips the per-chunk checks
  const int r0 = S.r0, r1 = S.r1;
  const int n_items = (r1 - r0 + G - 1) / G;
  const size_t rb = static_cast<size_t>(P.K) >> 2;
  for (int item = it0; item < n_items; item += kWarps) {
    const int row = r0 + item * G + grp;
    const bool valid = row < r1;
    const uint4* wrow = reinterpret_cast<const uint4*>(P.Wp + static_cast<size_t>(valid ? row : r0) * rb);
    int acc[MT][NA];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int i = 0; i < NA; ++i) acc[t][i] = 0;
    for (int b = 0; b < nb; ++b) {
      const int c0 = b * (LPR * U) + sub;
      const int lim = C - c0;                 // chunk u exists when u * LPR < lim
      if (valid && lim > (U - 1) * LPR) gemv_batch<MT, LPR, U, true>(wrow, c0, lim, valid, act + c0, C, acc);
      else gemv_batch<MT, LPR, U, false>(wrow, c0, lim, valid, act + c0, C, acc);
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      int v;
      if constexpr (MT == 1)
        v = acc[0][0] + (acc[0][1] >> 2) + (acc[0][2] >> 4) + (acc[0][3] >> 6);
      else
        v = acc[t][0];
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      const int tok = t0 + t;
      if (sub == t && valid && tok < P.M) {
        const int accv = v - S.qs[t];
        float y = __fmul_rn(static_cast<float>(accv), S.c[t]);
        if (P.epi == static_cast<int>(Epi::kRelu2)) y = y > 0.0f ? __fmul_rn(y, y) : 0.0f;
        const size_t o = static_cast<size_t>(tok) * P.N + row;
        if (P.mul != nullptr) y = __fmul_rn(y, P.mul[o]);
        P.Y[o] = y;
        if (P.acc != nullptr) P.acc[o] = accv;
      }
    }
  }
}

template <int MT, int CAP>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) gemv_kernel(const __grid_constant__ BatchArgs<CAP> a) {
  extern __shared__ __align__(128) uint4 s_act[];
  __shared__ Span<MT> s_span[kMaxSpan];
  __shared__ int s_nspan;
  __shared__ int s_qs[kMaxSpan * MT];
  __shared__ unsigned s_amax[kMaxSpan * MT];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int r_begin = a.cta_row[blockIdx.x], r_end = a.cta_row[blockIdx.x + 1];
  if (tid < kMaxSpan * MT) {
    s_qs[tid] = 0;
    s_amax[tid] = 0u;
  }
  if (tid == 0) {
    int nspan = 0, items = 0, act = 0;
    if (r_begin < r_end) {
      for (int p = a.cta_p0[blockIdx.x]; p < a.count && a.prob[p].row_begin < r_end && nspan < kMaxSpan; ++p) {
        const DevProb& P = a.prob[p];
        Span<MT>& S = s_span[nspan++];
        S.p = p;
        S.r0 = max(r_begin, P.row_begin) - P.row_begin;
        S.r1 = min(r_end, P.row_begin + P.N) - P.row_begin;
        S.item0 = items;
        items += (S.r1 - S.r0 + (32 / P.lpr) - 1) / (32 / P.lpr);
        S.act = act;
        act += MT * (P.K >> 4);
      }
      // weights never depend on the preceding kernel: start pulling the
      // first ones of the run into L2 before waiting for it
      const DevProb& P0 = a.prob[s_span[0].p];
      const size_t rb = static_cast<size_t>(P0.K) >> 2;
      const size_t bytes = static_cast<size_t>(s_span[0].r1 - s_span[0].r0) * rb;
      prefetch_l2(P0.Wp + static_cast<size_t>(s_span[0].r0) * rb, bytes < (256u << 10) ? bytes : (256u << 10));
    }
    s_nspan = nspan;
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();
  const int nspan = s_nspan;
  if (nspan == 0) return;
  stage_all<MT, CAP>(a, s_span, nspan, s_act, s_qs, s_amax);
  // items are dealt round-robin over the warps across all spans (item i of
  // the CTA goes to warp i % kWarps); the rows of a span are contiguous in
  // HBM, so the CTA streams one region at a time
  for (int j = 0; j < nspan; ++j) {
    const Span<MT>& S = s_span[j];
    const DevProb& P = a.prob[S.p];
    const uint4* act = s_act + S.act;
    const int it0 = (warp - S.item0 % kWarps + kWarps) % kWarps;
    switch (P.lpr) {
      case 4: run_span<MT, 4, kUnroll<MT>>(P, S, act, it0, a.t0); break;
      case 8: run_span<MT, 8, kUnroll<MT>>(P, S, act, it0, a.t0); break;
      case 16: run_span<MT, 16, kUnroll<MT>>(P, S, act, it0, a.t0); break;
      default: run_span<MT, 32, kUnroll<MT>>(P, S, act, it0, a.t0); break;
    }
  }
}

// Lanes per row for a row of C 16-byte chunks, from a cost model measured on
// B300: a warp's item (32/LPR rows) costs about its chunks per lane plus one
// (the reduction and the stores), so the cost per row is
// (ceil(C/LPR) + 1) * LPR / 32. At least 4 lanes, so that one lane per token
// can write the result; ties go to fewer lanes.
int row_cost_x32(int C, int lpr) { return ((C + lpr - 1) / lpr + 1) * lpr; }

int lpr_for_chunks(int C) {
  int best = 4;
  for (int lpr = 8; lpr <= 32; lpr *= 2)
    if (row_cost_x32(C, lpr) < row_cost_x32(C, best)) best = lpr;
  return best;
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

// Host-side plan for one launch: CTA runs balanced by the row cost model and the shared
// memory the staged activations need. Returns 0 when the problems cannot
// share one launch, else the dynamic shared-memory size.
template <int CAP>
size_t plan(BatchArgs<CAP>& a, int mt, int sms, int* grid_out) {
  long long total = 0;
  int rows = 0;
  for (int i = 0; i < a.count; ++i) {
    DevProb& P = a.prob[i];
    P.row_begin = rows;
    P.lpr = lpr_for_chunks(P.K >> 6);
    rows += P.N;
    total += static_cast<long long>(P.N) * row_cost_x32(P.K >> 6, P.lpr);
  }
  if (rows == 0) return 0;
  const int grid = std::max(1, std::min(std::min(kCtasPerSm * sms, kMaxCtas), rows));
  // few long rows (one large matrix): widen the lane groups until every warp
  // has items (rows / (32 / LPR)) to stream, at least two on average
  for (;;) {
    long long items = 0;
    for (int i = 0; i < a.count; ++i) items += (a.prob[i].N + 32 / a.prob[i].lpr - 1) / (32 / a.prob[i].lpr);
    if (items >= 2ll * grid * kWarps) break;
    bool widened = false;
    for (int i = 0; i < a.count; ++i)
      if (a.prob[i].lpr < 32) {
        a.prob[i].lpr *= 2;
        widened = true;
      }
    if (!widened) break;
  }
  total = 0;
  for (int i = 0; i < a.count; ++i)
    total += static_cast<long long>(a.prob[i].N) * row_cost_x32(a.prob[i].K >> 6, a.prob[i].lpr);
  // boundaries: first row whose cumulative byte count reaches c/grid of the total
  int c = 1, p = 0;
  long long cum = 0;
  a.cta_row[0] = 0;
  for (int r = 0; r < rows && c < grid; ++r) {
    while (a.prob[p].row_begin + a.prob[p].N <= r) ++p;
    cum += row_cost_x32(a.prob[p].K >> 6, a.prob[p].lpr);
    while (c < grid && cum * grid >= total * c) a.cta_row[c++] = r + 1;
  }
  while (c <= grid) a.cta_row[c++] = rows;
  for (int i = grid + 1; i <= kMaxCtas; ++i) a.cta_row[i] = rows;
  for (int b = 0, q = 0; b < grid; ++b) {
    while (q + 1 < a.count && a.prob[q].row_begin + a.prob[q].N <= a.cta_row[b]) ++q;
    a.cta_p0[b] = static_cast<unsigned char>(q);
  }
  // activation area: the most any CTA needs; at most kMaxSpan problems per CTA
  size_t act = 0;
  for (int b = 0; b < grid; ++b) {
    const int r0 = a.cta_row[b], r1 = a.cta_row[b + 1];
    if (r0 >= r1) continue;
    int p0 = 0;
    while (a.prob[p0].row_begin + a.prob[p0].N <= r0) ++p0;
    int p1 = p0;
    while (a.prob[p1].row_begin + a.prob[p1].N < r1) ++p1;
    if (p1 - p0 + 1 > kMaxSpan) return 0;
    size_t need = 0;
    for (int q = p0; q <= p1; ++q) need += static_cast<size_t>(mt) * a.prob[q].K;
    act = std::max(act, need);
  }
  if (act > static_cast<size_t>(kActBudget)) return 0;
  *grid_out = grid;
  return std::max<size_t>(act, 16);
}

template <int MT, int CAP>
cudaError_t launch_batch(BatchArgs<CAP>& a, bool pdl, cudaStream_t st, bool* planned) {
  const DevInfo d = dev_info();
  int grid = 0;
  const size_t smem = plan(a, MT, d.sms, &grid);
  *planned = smem != 0;
  if (!*planned) return cudaSuccess;
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
  d.q = p.q;
  d.m_in = p.m;
  d.s_w = p.s_w;
  d.Y = p.Y;
  d.acc = p.acc;
  d.mul = p.mul;
  d.x = p.x;
  d.x_dtype = p.x_dtype;
  d.eps = p.eps;
  d.N = p.N;
  d.K = p.K;
  d.M = p.M;
  d.epi = static_cast<int>(p.epi);
  return d;
}

template <int MT, int CAP>
cudaError_t run_tokens(const GemvProblem* ps, int count, int t0, WsHeader* status, bool pdl, cudaStream_t st,
                       bool* planned) {
  (void)status;   // the GEMV has no device-side waits to report
  BatchArgs<CAP> a;
  int n = 0;
  for (int i = 0; i < count; ++i)
    if (ps[i].N > 0 && ps[i].M > t0) a.prob[n++] = to_dev(ps[i]);
  *planned = true;
  if (n == 0) return cudaSuccess;
  a.count = n;
  a.t0 = t0;
  a.from_x = (n == 1 && a.prob[0].x != nullptr) ? 1 : 0;
  return launch_batch<MT, CAP>(a, pdl, st, planned);
}

template <int CAP>
cudaError_t run_mt(int mt, const GemvProblem* ps, int count, int t0, WsHeader* status, bool pdl, cudaStream_t st,
                   bool* planned) {
  if (mt == 1) return run_tokens<1, CAP>(ps, count, t0, status, pdl, st, planned);
  if (mt == 2) return run_tokens<2, CAP>(ps, count, t0, status, pdl, st, planned);
  return run_tokens<4, CAP>(ps, count, t0, status, pdl, st, planned);
}

template <int CAP>
cudaError_t run_all(const GemvProblem* ps, int count, WsHeader* status, bool pdl, cudaStream_t st) {
  int maxM = 0;
  for (int i = 0; i < count; ++i) maxM = std::max(maxM, ps[i].M);
  // tokens per launch: up to 4; fewer when the staged activations of a run
  // would not fit in shared memory
  int mt = maxM <= 1 ? 1 : (maxM == 2 ? 2 : 4);
  for (int t0 = 0; t0 < maxM;) {
    bool planned = true;
    cudaError_t err = run_mt<CAP>(mt, ps, count, t0, status, pdl, st, &planned);
    if (err != cudaSuccess) return err;
    if (planned) {
      t0 += mt;
      continue;
    }
    if (mt > 1) {
      mt >>= 1;
      continue;
    }
    if (count == 1) return cudaErrorInvalidConfiguration;
    // one token per launch still does not fit: split the batch in halves,
    // each planning its own CTA runs (tokens already written are simply
    // written again with the same values)
    const int h = count / 2;
    err = run_all<CAP>(ps, h, status, pdl, st);
    if (err != cudaSuccess) return err;
    return run_all<CAP>(ps + h, count - h, status, pdl, st);
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
