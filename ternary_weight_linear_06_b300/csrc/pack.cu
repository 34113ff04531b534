// Weight packing: absmean scale, ternarization and 2-bit codes.
//
// "BitNet解读" (markgoyens.top), 模型架构 / 权重量化函数, eqs. (1)-(3):
//   gamma = (1/nm) sum |W_ij|,  W~ = RoundClip(W / (gamma + eps), -1, 1).
// "BitNet b1.58 2B4T Technical Report | Summary", 5.1 GPU Inference: four
// ternary values per 8-bit value.
//
// gamma is computed exactly (order-independent) and rounded once to fp32:
//   1. abs_sum_kernel: every |w| = mant * 2^(e-150) (e = biased exponent,
//      e >= 1; subnormals use e = 1). For e in [86, 158] the thread adds
//      mant << (e - 86) to a 128-bit fixed-point accumulator (unit 2^-64);
//      the bound N*K < 2^31 keeps the grand total below 2^127. The rare
//      values outside that window go to 64-bit per-exponent buckets.
//   2. finalize_kernel: the CTA adds the block partials in 128 bits, then
//      one thread adds that sum and the buckets into a 352-bit integer (unit
//      2^-149), divides by N*K with long division and rounds to nearest-even
//      fp32, then s_w = fp32(gamma + eps).
//   3. codes_kernel: one float4 -> one byte. rint(fp32(w / s)) clipped to
//      [-1, 1] is 0 exactly when 2|w| <= s (for finite w and s > 0: the
//      quotient rounds to at most 0.5 iff |w|/s <= 0.5 + 2^-25, and no fp32
//      value lies in (s, s * (1 + 2^-24)]), else sign(w); so the kernel needs
//      no division and makes the same decision as the formula.
#include "common.cuh"
#include "launchers.h"

namespace bl {
namespace {

constexpr int kSumThreads = 256;
constexpr int kMaxSumBlocks = 1184;   // 8 per SM on a 148-SM part
constexpr uint32_t kWinLo = 86, kWinHi = 158;
constexpr int kLimbs = 11;            // 352-bit big integer

struct PackScratch {
  unsigned long long bucket[256];                  // out-of-window mantissa sums
  unsigned long long partial[kMaxSumBlocks][2];    // per-block 128-bit window sums
  unsigned int nonfinite;
  unsigned int pad0;
  float gamma;
  float pad;
};

__device__ __forceinline__ void add_abs(uint32_t bits, unsigned __int128& acc, PackScratch* sc) {
  const uint32_t e = (bits >> 23) & 0xFFu;
  const uint32_t f = bits & 0x7FFFFFu;
  if (e - kWinLo <= kWinHi - kWinLo) {
    acc += static_cast<unsigned __int128>(f | 0x800000u) << (e - kWinLo);
  } else if (e == 0xFFu) {
    atomicOr(&sc->nonfinite, 1u);
  } else if ((e | f) != 0u) {
    atomicAdd(&sc->bucket[e ? e : 1u], static_cast<unsigned long long>(e ? (f | 0x800000u) : f));
  }
}

__global__ void __launch_bounds__(kSumThreads) abs_sum_kernel(const uint4* __restrict__ W4, size_t n4,
                                                              PackScratch* __restrict__ sc) {
  unsigned __int128 acc = 0;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const uint4 v = ldg_stream(W4 + i);
    add_abs(v.x, acc, sc);
    add_abs(v.y, acc, sc);
    add_abs(v.z, acc, sc);
    add_abs(v.w, acc, sc);
  }
  __shared__ unsigned __int128 red[kSumThreads];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = kSumThreads / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    sc->partial[blockIdx.x][0] = static_cast<unsigned long long>(red[0]);
    sc->partial[blockIdx.x][1] = static_cast<unsigned long long>(red[0] >> 64);
  }
}

// Add a 64-bit value, shifted left by `shift` bits, into carry-save limbs
// (32-bit digits held in 64-bit slots; normalized later).
__device__ void big_add(unsigned long long* limb, unsigned long long v, int shift) {
  const int j = shift >> 5, r = shift & 31;
  const unsigned long long lo = v & 0xFFFFFFFFull, hi = v >> 32;
  const unsigned long long a = lo << r, b = hi << r;      // each < 2^64
  limb[j] += a & 0xFFFFFFFFull;
  limb[j + 1] += (a >> 32) + (b & 0xFFFFFFFFull);
  limb[j + 2] += b >> 32;
}

__device__ uint32_t bits_at(const uint32_t* Q, int pos, int len) {
  const int li = pos >> 5, off = pos & 31;
  const unsigned long long w =
      Q[li] | (static_cast<unsigned long long>(li + 1 < kLimbs ? Q[li + 1] : 0u) << 32);
  return static_cast<uint32_t>((w >> off) & ((1ull << len) - 1ull));
}

__device__ bool any_below(const uint32_t* Q, int pos) {
  for (int i = 0; i < kLimbs && 32 * i < pos; ++i) {
    const int n = min(32, pos - 32 * i);
    const uint32_t mask = n == 32 ? 0xFFFFFFFFu : ((1u << n) - 1u);
    if (Q[i] & mask) return true;
  }
  return false;
}

__global__ void __launch_bounds__(kSumThreads) finalize_kernel(PackScratch* __restrict__ sc, uint32_t nblocks,
                                                                uint32_t n, float eps, float* __restrict__ s_w) {
  // The window partials add up to less than 2^127 (N*K < 2^31), so any subset
  // of them sums exactly in 128 bits: the CTA adds them in parallel, and the
  // buckets are read into shared memory at the same time.
  __shared__ unsigned __int128 red[kSumThreads];
  __shared__ unsigned long long s_bucket[256];
  const int tid = threadIdx.x;
  unsigned __int128 part = 0;
  for (uint32_t b = tid; b < nblocks; b += kSumThreads)
    part += (static_cast<unsigned __int128>(sc->partial[b][1]) << 64) | sc->partial[b][0];
  red[tid] = part;
  for (int e = tid; e < 256; e += kSumThreads) s_bucket[e] = sc->bucket[e];
  __syncthreads();
  for (int st = kSumThreads / 2; st > 0; st >>= 1) {
    if (tid < st) red[tid] += red[tid + st];
    __syncthreads();
  }
  if (tid != 0) return;
  unsigned long long limb[kLimbs + 2];
  for (int i = 0; i < kLimbs + 2; ++i) limb[i] = 0;
  // window sum: value = P * 2^-64 = P * 2^85 in units of 2^-149
  big_add(limb, static_cast<unsigned long long>(red[0]), 85);
  big_add(limb, static_cast<unsigned long long>(red[0] >> 64), 85 + 64);
  // buckets: value = S * 2^(e-150) = S * 2^(e-1) in units of 2^-149
  for (int e = 1; e < 255; ++e)
    if (s_bucket[e]) big_add(limb, s_bucket[e], e - 1);
  uint32_t S[kLimbs];
  unsigned long long carry = 0;
  for (int i = 0; i < kLimbs; ++i) {
    const unsigned long long v = limb[i] + carry;
    S[i] = static_cast<uint32_t>(v);
    carry = v >> 32;
  }
  // Q = floor(S / n), rem = S mod n
  uint32_t Q[kLimbs];
  unsigned long long rem = 0;
  for (int i = kLimbs - 1; i >= 0; --i) {
    const unsigned long long cur = (rem << 32) | S[i];
    Q[i] = static_cast<uint32_t>(cur / n);
    rem = cur % n;
  }
  int h = 0;
  for (int i = kLimbs - 1; i >= 0; --i)
    if (Q[i]) { h = 32 * i + (32 - __clz(Q[i])); break; }
  int shift;
  uint32_t mant;
  bool up;
  if (h > 24) {
    shift = h - 24;
    mant = bits_at(Q, shift, 24);
    const bool guard = bits_at(Q, shift - 1, 1) != 0u;
    const bool sticky = any_below(Q, shift - 1) || rem != 0;
    up = guard && (sticky || (mant & 1u));
  } else {
    shift = 0;
    mant = Q[0];
    const unsigned long long twice = rem * 2ull;
    up = twice > n || (twice == n && (mant & 1u));
  }
  mant += up ? 1u : 0u;
  if (mant == (1u << 24)) { mant >>= 1; ++shift; }
  uint32_t bits;
  if (mant < (1u << 23)) {
    bits = mant;                                   // subnormal (shift == 0)
  } else {
    const int be = shift + 1;                      // biased exponent
    bits = be >= 255 ? 0x7F800000u : ((static_cast<uint32_t>(be) << 23) | (mant & 0x7FFFFFu));
  }
  const float gamma = __uint_as_float(bits);
  sc->gamma = gamma;
  s_w[0] = sc->nonfinite ? __uint_as_float(0x7FC00000u) : __fadd_rn(gamma, eps);
}

__device__ __forceinline__ uint32_t code_of(float w, float s) {
  const float a = fabsf(w);
  return (__fadd_rn(a, a) <= s) ? 1u : (w > 0.0f ? 2u : 0u);
}

__global__ void __launch_bounds__(256) codes_kernel(const float4* __restrict__ W4, size_t n4,
                                                    const float* __restrict__ s_w, uint8_t* __restrict__ out) {
  const float s = s_w[0];
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const uint4 u = ldg_stream(W4 + i);
    const uint32_t c = code_of(__uint_as_float(u.x), s) | (code_of(__uint_as_float(u.y), s) << 2) |
                       (code_of(__uint_as_float(u.z), s) << 4) | (code_of(__uint_as_float(u.w), s) << 6);
    out[i] = static_cast<uint8_t>(c);
  }
}

__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t* __restrict__ packed, size_t nbytes,
                                                     uint32_t* __restrict__ t) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nbytes; i += stride) {
    const uint32_t b = packed[i];
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) w |= ((((b >> (2 * j)) & 3u) - 1u) & 0xFFu) << (8 * j);
    t[i] = w;
  }
}

int sm_count() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

}  // namespace

size_t pack_scratch_bytes() { return align_up(sizeof(PackScratch), 256); }

cudaError_t launch_pack(const float* W, int N, int K, float eps, uint8_t* packed, float* s_w,
                        void* workspace, cudaStream_t st) {
  auto* sc = reinterpret_cast<PackScratch*>(static_cast<char*>(workspace) + sizeof(WsHeader));
  const size_t n4 = static_cast<size_t>(N) * K / 4;
  const int nsm = sm_count();
  int blocks = static_cast<int>(std::min<size_t>((n4 + kSumThreads - 1) / kSumThreads,
                                                 static_cast<size_t>(std::min(kMaxSumBlocks, 8 * nsm))));
  if (blocks < 1) blocks = 1;
  cudaError_t err = cudaMemsetAsync(sc, 0, sizeof(PackScratch), st);
  if (err != cudaSuccess) return err;
  abs_sum_kernel<<<blocks, kSumThreads, 0, st>>>(reinterpret_cast<const uint4*>(W), n4, sc);
  finalize_kernel<<<1, kSumThreads, 0, st>>>(sc, static_cast<uint32_t>(blocks),
                                             static_cast<uint32_t>(static_cast<size_t>(N) * K), eps, s_w);
  const int cblocks = static_cast<int>(std::min<size_t>((n4 + 255) / 256, static_cast<size_t>(16 * nsm)));
  codes_kernel<<<cblocks, 256, 0, st>>>(reinterpret_cast<const float4*>(W), n4, s_w, packed);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* packed, int N, int K, int8_t* t, cudaStream_t st) {
  const size_t nbytes = static_cast<size_t>(N) * K / 4;
  const int blocks = static_cast<int>(std::min<size_t>((nbytes + 255) / 256, static_cast<size_t>(16 * sm_count())));
  unpack_kernel<<<blocks, 256, 0, st>>>(packed, nbytes, reinterpret_cast<uint32_t*>(t));
  return cudaGetLastError();
}

}  // namespace bl
