// Prefill / batched GEMM on the 5th-generation tensor cores (tcgen05, TMEM,
// TMA): Y[m][n] = dequant(sum_k q[m][k] * t[n][k]) for many tokens m.
//
// "BitNet b1.58 2B4T Technical Report | Summary", 5.1 GPU Inference: packed
// ternary weights are loaded from HBM into on-chip memory, unpacked there and
// multiplied with 8-bit activations. "BitNet解读", 革命性的效率提升: the
// products are additions and subtractions of activations, so the sum is an
// exact integer.
//
// sm_103a has no integer tcgen05 MMA (ptxas rejects kind::i8 for it), so the
// contraction runs as kind::f16 on integer-valued fp16 operands: t in {-1,0,1}
// and q in [-128, 127] are exact in fp16, every product is exact, and every
// partial sum is an integer of magnitude <= 128 * K <= 2^23 (K <= 65536), so
// the fp32 accumulation in TMEM is exact and acc = float(sum) holds the
// integer result.
//
// Tile: 128 weight rows (the MMA's M) x 128, 192 or 256 tokens (its N; the
// host picks the width from the tile count, wider instructions run closer to
// the tensor-core peak), K in steps of 64.
//   * A (weights) lives in TMEM: converter warps read the 2-bit codes of their
//     row (16 bytes per K step, staged by TMA), turn them into fp16 t values
//     in registers and write them with tcgen05.st, so the expanded weights
//     never take shared-memory bandwidth;
//   * B (activations) is fp16 in shared memory, staged by TMA with the
//     128-byte swizzle the MMA descriptor names;
//   * D is fp32 in TMEM: two accumulators for 128- and 192-token tiles, so the
//     epilogue of one tile overlaps the MMAs of the next; one for 256-token
//     tiles (TMEM has 512 columns, and the weight stages need some).
// Warp roles (one CTA per SM, persistent over tiles):
//   warp 0      TMA producer (one lane): activation tile + packed code tile per stage
//   warp 1      MMA issuer (one lane); the warp owns the TMEM allocation
//   warps 2-9   converters: packed codes -> fp16 t in TMEM; warp w owns TMEM lanes
//               32*(w%4).. and every other K step (two warps per lane quarter)
//   warps 10-17 epilogue: TMEM -> registers, y = fp32(acc * fp32(fp32(s_w*m)/127)), stores;
//               warp w owns TMEM lanes 32*(w%4).. and every other 32-token chunk
// Every mbarrier wait is bounded: on a timeout the thread records
// BL_ERR_TIMEOUT, raises the CTA's abort flag (which ends every other role's
// waits), and the CTA drains its copies and MMAs (bounded) before it frees
// TMEM and exits.
//
// K order. The activations are written by the quantization kernel with fp16
// slot s of every 16-column group holding column (s >> 1) + 8 * (s & 1), so
// the 32-bit word c of a group holds columns (c, c + 8). The packed code of
// column 4j + i of a group sits at bit 8j + 2i of its 32-bit word, so columns
// c and c + 8 sit 16 bits apart: masking a word with 0x00030003 << b leaves
// both codes in place, one per half, and OR-ing in 0x6400 per half makes the
// fp16 values 1024 + code * 2^b; one HFMA2 (x * 2^-b - (1024 * 2^-b + 1))
// gives the exact t = code - 1 in both halves.
#include <cuda.h>

#include "common.cuh"
#include "launchers.h"

namespace bl {
namespace {

constexpr int kTileN = 128;           // weight rows per tile (MMA M)
constexpr int kTileK = 64;            // K per stage: one 128-byte swizzle row of fp16
constexpr int kConvWarps = 8;         // two per TMEM lane quarter, alternating K steps
constexpr int kEpiWarp0 = 2 + kConvWarps;
constexpr int kEpiWarps = 8;          // two per TMEM lane quarter, alternating 32-token chunks
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;   // 18 warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPBytes = kTileN * kTileK / 4;   // 2 KB of codes per stage
// at least this much dynamic shared memory, so that one CTA fits per SM and
// no second CTA waits on the first one's TMEM
constexpr size_t kMinSmem = 120 * 1024;

// Tile shapes: TM tokens per tile (the MMA's N; one instruction covers all
// of them, and wider instructions run closer to the tensor-core peak),
// ST pipeline stages, NB accumulator buffers in TMEM (two let the epilogue of
// one tile overlap the MMAs of the next). TMEM columns: NB * TM for the
// accumulators, then ST * 32 for the weight stages.
template <int TM, int ST, int NB>
struct Cfg {
  static constexpr int kTileM = TM;
  static constexpr int kStages = ST;
  static constexpr int kAccBufs = NB;
  static constexpr uint32_t kAccCol = 0;
  static constexpr uint32_t kACol = static_cast<uint32_t>(TM * NB);
  static constexpr uint32_t kBBytes = TM * kTileK * 2;
  static_assert(TM % 16 == 0 && TM >= 16 && TM <= 256, "MMA N must be a multiple of 16 in [16, 256]");
  static_assert(kACol + ST * 32 <= kTmemCols, "accumulators and weight stages exceed TMEM");
  static_assert(ST % 2 == 0, "converter parity split assumes an even stage count");
  // Instruction descriptor: D fp32, A fp16, B fp16, both K-major, N = TM, M = kTileN.
  static constexpr uint32_t kIdesc =
      (1u << 4) | (static_cast<uint32_t>(TM >> 3) << 17) | (static_cast<uint32_t>(kTileN >> 4) << 24);
  static size_t smem_bytes() {
    const size_t need = 1024 + ST * (kBBytes + kPBytes) + 256;
    return need > kMinSmem ? need : kMinSmem;
  }
};
using CfgWide = Cfg<256, 6, 1>;     // 256 tokens, one accumulator
using CfgMid = Cfg<192, 4, 2>;      // 192 tokens, two accumulators
using CfgNarrow = Cfg<128, 8, 2>;   // 128 tokens (few tokens), two accumulators

struct GemmParams {
  int M, N, K;
  int splits;            // K is cut into this many parts, one work unit each
  int32_t* acc_ws;       // splits > 1: [M][N] int32 partial-sum target (zeroed)
  const float* mul;      // [M][N] or null: y = fp32(y * mul)
  const float* m;        // [M] per-token scales
  const float* s_w;      // [1]
  float* Y;              // [M][N]
  int32_t* acc;          // [M][N] or null
  WsHeader* status;
};

template <int ST>
struct SmemCtl {
  uint64_t full[ST];           // TMA bytes of a stage landed
  uint64_t aready[ST];         // converters wrote the stage's A into TMEM
  uint64_t empty[ST];          // MMAs that read the stage are done
  uint64_t accfull[2];         // accumulator b holds a finished tile
  uint64_t accempty[2];        // epilogue drained accumulator b
  uint64_t done;               // final commit of the MMA thread
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory operand descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (the layout a 128-byte-swizzled TMA box of 64 fp16 per row
// leaves behind).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

template <uint32_t IDESC>
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(bdesc), "n"(IDESC), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Bounded wait that also ends when another role has raised the abort flag.
// Returns false on timeout or abort.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t deadline,
                                              volatile int* abort_flag) {
  for (int n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15) == 0) {
      if (*abort_flag) return false;
      if (global_ns() > deadline) return false;
    }
  }
}

// Warp-wide wait: lane 0 polls (with a short sleep between polls when
// `sleepy`, for waits that are long by design), then every lane confirms the
// completed phase once, which gives each of them the barrier's acquire
// ordering. Returns the same verdict in every lane.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t deadline, volatile int* abort_flag,
                                          bool sleepy) {
  const int lane = threadIdx.x & 31;
  bool ok = true;
  if (lane == 0) {
    for (int n = 1;; ++n) {
      if (mbar_try_wait(bar, parity)) break;
      if (sleepy) __nanosleep(64);
      if ((n & 15) == 0 && (*abort_flag || global_ns() > deadline)) {
        ok = false;
        break;
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (ok) ok = mbar_wait_until(bar, parity, deadline);
  return __all_sync(0xffffffffu, ok);
}

template <typename Ctl>
__device__ __forceinline__ void raise_abort(Ctl* ctl, WsHeader* status, uint32_t where) {
  if (atomicExch(&ctl->abort, 1) == 0) report_status(status, BL_ERR_TIMEOUT, where);
}

// fp16 pair word (column c, column c + 8) of a 16-column group from its code
// word w: t = code - 1 in both halves.
template <int C>
__device__ __forceinline__ uint32_t pair_word(uint32_t w_lo, uint32_t w_hi) {
  constexpr int b = 2 * (C & 3);
  const uint32_t src = (C < 4) ? w_lo : w_hi;      // columns 0-3 / 4-7 sit in bytes 0,2 / 1,3
  const uint32_t x = (src & (0x00030003u << b)) | 0x64006400u;
  const __half2 scale = __float2half2_rn(1.0f / static_cast<float>(1 << b));
  const __half2 bias = __float2half2_rn(-(1024.0f / static_cast<float>(1 << b) + 1.0f));
  const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&x), scale, bias);
  return *reinterpret_cast<const uint32_t*>(&r);
}

template <class C, bool RELU2, bool ACC, bool SPLIT, bool MUL>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_codes,
                   const GemmParams p) {
  constexpr int kTileM = C::kTileM;
  constexpr int kStages = C::kStages;
  constexpr uint32_t kBBytes = C::kBBytes;
  constexpr uint32_t kAccCol = C::kAccCol;
  constexpr uint32_t kACol = C::kACol;
  using Ctl = SmemCtl<kStages>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled stages
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem;                                           // [kStages][kBBytes]
  uint8_t* sP = smem + kStages * kBBytes;                       // [kStages][kPBytes]
  Ctl* ctl = reinterpret_cast<Ctl*>(sP + kStages * kPBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_n = (p.N + kTileN - 1) / kTileN;
  const int tiles_m = (p.M + kTileM - 1) / kTileM;
  const int tiles = tiles_n * tiles_m;
  const int ktiles = p.K / kTileK;
  // work units: (tile, K part); a tile's parts are consecutive units, so they
  // run on different CTAs at the same time
  const int splits = SPLIT ? p.splits : 1;
  const int units = tiles * splits;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->aready[s], 4);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->accfull[b], 1);
      mbar_init(&ctl->accempty[b], kEpiWarps);
    }
    mbar_init(&ctl->done, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&ctl->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort;

  // the activations (and scales) come from the preceding kernel
  pdl_wait();
  const uint64_t deadline = global_ns() + kWaitLimitNs;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    int issued = 0;
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const int tile = u / splits, kp = u - tile * splits;
        const int tn = tile / tiles_m, tm = tile % tiles_m;
        const int kb = kp * ktiles / splits, ke = (kp + 1) * ktiles / splits;
        for (int kt = kb; kt < ke; ++kt) {
          if (!wait_or_abort(&ctl->empty[s], ph ^ 1u, deadline, abort_flag)) {
            raise_abort(ctl, p.status, 0x300u + blockIdx.x);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&ctl->full[s], kBBytes + kPBytes);
          tma_load_2d(sB + s * kBBytes, &tm_act, kt * kTileK, tm * kTileM, &ctl->full[s]);
          tma_load_2d(sP + s * kPBytes, &tm_codes, kt * (kTileK / 4), tn * kTileN, &ctl->full[s]);
          ++issued;
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // no copy may still be landing when the CTA exits: wait (bounded) for
      // the last use of every stage
      const uint64_t d2 = global_ns() + kWaitLimitNs / 4;
      for (int u = max(0, issued - kStages); u < issued; ++u)
        (void)mbar_wait_until(&ctl->full[u % kStages], static_cast<uint32_t>((u / kStages) & 1), d2);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      int local = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++local) {
        const int kp = u % splits;
        const int kb = kp * ktiles / splits, ke = (kp + 1) * ktiles / splits;
        const int b = C::kAccBufs == 2 ? (local & 1) : 0;
        const uint32_t use = static_cast<uint32_t>(C::kAccBufs == 2 ? (local >> 1) : local);
        if (!wait_or_abort(&ctl->accempty[b], (use & 1u) ^ 1u, deadline, abort_flag)) {
          raise_abort(ctl, p.status, 0x400u + blockIdx.x);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + kAccCol + b * kTileM;
        for (int kt = kb; kt < ke; ++kt) {
          // the converters waited for the stage's TMA bytes before they
          // arrived on aready, so this one wait orders both operands
          if (!wait_or_abort(&ctl->aready[s], ph, deadline, abort_flag)) {
            raise_abort(ctl, p.status, 0x500u + blockIdx.x);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = tmem + kACol + s * 32;
          const uint64_t bdesc = sw128_desc(smem_u32(sB + s * kBBytes));
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk)
            mma_f16_tmem_a<C::kIdesc>(d, a + kk * 8, bdesc + static_cast<uint64_t>(kk * 2), (kt != kb || kk != 0) ? 1u : 0u);
          mma_commit(&ctl->empty[s]);
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) mma_commit(&ctl->accfull[b]);
      }
      // every MMA issued by this thread is complete once `done` fires
      mma_commit(&ctl->done);
      (void)mbar_wait_until(&ctl->done, 0, global_ns() + kWaitLimitNs / 4);
    }
  } else if (warp < kEpiWarp0) {
    // ---------------- converters: codes -> fp16 t in TMEM ----------------
    const int quarter = warp & 3;
    const int parity = (warp - 2) >> 2;                  // this warp's K steps: step % 2 == parity
    const int row = quarter * 32 + lane;                 // row of the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    int step = 0;                                        // K steps of all tiles, in order
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const int kp = u % splits;
      const int kb = kp * ktiles / splits, ke = (kp + 1) * ktiles / splits;
      for (int kt = kb; kt < ke; ++kt, ++step) {
        if ((step & 1) != parity) {
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
          continue;
        }
        const bool got = wait_or_abort(&ctl->full[s], ph, deadline, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) raise_abort(ctl, p.status, 0x600u + blockIdx.x);
          ok = false;
          break;
        }
        const uint4 cw = *reinterpret_cast<const uint4*>(sP + s * kPBytes + row * 16);
        uint32_t r[32];
        const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint32_t lo = words[g], hi = words[g] >> 8;
          r[g * 8 + 0] = pair_word<0>(lo, hi);
          r[g * 8 + 1] = pair_word<1>(lo, hi);
          r[g * 8 + 2] = pair_word<2>(lo, hi);
          r[g * 8 + 3] = pair_word<3>(lo, hi);
          r[g * 8 + 4] = pair_word<4>(lo, hi);
          r[g * 8 + 5] = pair_word<5>(lo, hi);
          r[g * 8 + 6] = pair_word<6>(lo, hi);
          r[g * 8 + 7] = pair_word<7>(lo, hi);
        }
        tmem_st32(tmem + lane_base + kACol + s * 32, r);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->aready[s]);
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else {
    // ---------------- epilogue (warps kEpiWarp0 .. kEpiWarp0 + kEpiWarps - 1) ----------------
    const int quarter = warp & 3;
    const int half = (warp - kEpiWarp0) >> 2;            // this warp's chunks: c % 2 == half
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float sw = p.s_w[0];
    int local = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++local) {
      const int tile = u / splits;
      const int tn = tile / tiles_m, tm = tile % tiles_m;
      const int b = C::kAccBufs == 2 ? (local & 1) : 0;
      const uint32_t use = static_cast<uint32_t>(C::kAccBufs == 2 ? (local >> 1) : local);
      if (!warp_wait(&ctl->accfull[b], use & 1u, deadline, abort_flag, true)) {
        if (lane == 0) raise_abort(ctl, p.status, 0x700u + blockIdx.x);
        break;
      }
      tc_fence_after();
      const int n = tn * kTileN + quarter * 32 + lane;
      const bool n_ok = n < p.N;
#pragma unroll 1
      for (int c = half; c < kTileM / 32; c += 2) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kAccCol + b * kTileM + c * 32, v);
        const int tok0 = tm * kTileM + c * 32;
        // lane j holds the dequant factor of token tok0 + j
        const float my_c = tok0 + lane < p.M ? dequant_factor(sw, p.m[tok0 + lane]) : 0.0f;
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (tok0 >= p.M) continue;
        if constexpr (SPLIT) {
          // exact integer partial sums, added in any order
          int32_t* wp = p.acc_ws + static_cast<size_t>(tok0) * p.N + n;
          const int jmax = min(32, p.M - tok0);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j < jmax && n_ok) atomicAdd(wp, __float2int_rn(__uint_as_float(v[j])));
            wp += p.N;
          }
          continue;
        }
        float* yp = p.Y + static_cast<size_t>(tok0) * p.N + n;
        int32_t* ap = ACC ? p.acc + static_cast<size_t>(tok0) * p.N + n : nullptr;
        const int jmax = min(32, p.M - tok0);
        // the factors of the product, all loaded before the first store (the
        // stores to Y could otherwise alias them and serialize the loads)
        float mv[MUL ? 32 : 1];
        if constexpr (MUL) {
          const float* mp = p.mul + static_cast<size_t>(tok0) * p.N + n;
#pragma unroll
          for (int j = 0; j < 32; ++j) mv[j] = (j < jmax && n_ok) ? __ldg(mp + static_cast<size_t>(j) * p.N) : 0.0f;
        }
        if (jmax == 32 && n_ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float accf = __uint_as_float(v[j]);
            float y = __fmul_rn(accf, __shfl_sync(0xffffffffu, my_c, j));
            if constexpr (RELU2) y = y > 0.0f ? __fmul_rn(y, y) : 0.0f;
            if constexpr (MUL) y = __fmul_rn(y, mv[j]);
            *yp = y;
            yp += p.N;
            if constexpr (ACC) {
              *ap = __float2int_rn(accf);
              ap += p.N;
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float accf = __uint_as_float(v[j]);
            float y = __fmul_rn(accf, __shfl_sync(0xffffffffu, my_c, j));
            if constexpr (RELU2) y = y > 0.0f ? __fmul_rn(y, y) : 0.0f;
            if (j < jmax && n_ok) {
              if constexpr (MUL) y = __fmul_rn(y, mv[j]);
              *yp = y;
              if constexpr (ACC) *ap = __float2int_rn(accf);
            }
            yp += p.N;
            if constexpr (ACC) ap += p.N;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->accempty[b]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// After a split-K GEMM: y = fp32(acc * fp32(fp32(s_w * m) / 127)) (then ReLU^2
// for the FFN up projection) from the summed integer accumulators. One CTA
// row per token (blockIdx.y), threads over the outputs.
__global__ void __launch_bounds__(256) split_finalize_kernel(const int32_t* __restrict__ acc_ws, int M, int N,
                                                             const float* __restrict__ m,
                                                             const float* __restrict__ s_w, float* __restrict__ Y,
                                                             int32_t* __restrict__ acc, int relu2,
                                                             const float* __restrict__ mul) {
  pdl_wait();
  pdl_trigger();
  const int tok = blockIdx.y;
  const float c = dequant_factor(s_w[0], m[tok]);
  for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < N; n += gridDim.x * blockDim.x) {
    const size_t o = static_cast<size_t>(tok) * N + n;
    const int v = acc_ws[o];
    float y = __fmul_rn(static_cast<float>(v), c);
    if (relu2) y = y > 0.0f ? __fmul_rn(y, y) : 0.0f;
    if (mul != nullptr) y = __fmul_rn(y, mul[o]);
    Y[o] = y;
    if (acc != nullptr) acc[o] = v;
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps (driver entry point looked up once) and the launch.
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}


template <class C>
cudaError_t launch_cfg(const GemmProblem& g, WsHeader* status, bool pdl, cudaStream_t st, int splits) {
  CUtensorMap tm_act, tm_codes;
  // activations: fp16 [M][K] (pair order within 16-column groups)
  if (!make_map_2d(&tm_act, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, g.act, static_cast<uint64_t>(g.K),
                   static_cast<uint64_t>(g.M), static_cast<uint64_t>(g.K) * 2, kTileK, C::kTileM,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // packed codes: uint8 [N][K/4]
  if (!make_map_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.Wp, static_cast<uint64_t>(g.K) / 4,
                   static_cast<uint64_t>(g.N), static_cast<uint64_t>(g.K) / 4, kTileK / 4, kTileN,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  GemmParams p;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.splits = std::max(1, splits);
  p.acc_ws = g.acc_ws;
  p.mul = g.mul;
  p.m = g.m;
  p.s_w = g.s_w;
  p.Y = g.Y;
  p.acc = g.acc;
  p.status = status;
  const int tiles = ((g.N + kTileN - 1) / kTileN) * ((g.M + C::kTileM - 1) / C::kTileM);
  const int grid = std::max(1, std::min(tiles * p.splits, sm_count()));
  const size_t smem = C::smem_bytes();
  // epilogue variants in use: plain, ReLU^2 (FFN up), times a second operand
  // (gated FFN up), each with or without the integer accumulators; split-K
  // runs apply the epilogue in split_finalize_kernel
  auto kern = p.splits > 1 ? gemm_tc_kernel<C, false, false, true, false>
               : g.mul != nullptr ? gemm_tc_kernel<C, false, false, false, true>
               : g.relu2 ? (g.acc != nullptr ? gemm_tc_kernel<C, true, true, false, false>
                                              : gemm_tc_kernel<C, true, false, false, false>)
                         : (g.acc != nullptr ? gemm_tc_kernel<C, false, true, false, false>
                                              : gemm_tc_kernel<C, false, false, false, false>);
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
  return cudaLaunchKernelEx(&cfg, kern, tm_act, tm_codes, p);
}

// Estimated cost of a tile shape: rounds of persistent tiles over the SMs
// times the tile's token count plus a fixed per-tile cost, with a small
// penalty for a single accumulator (the epilogue then stalls the MMAs).
double tile_cost(int M, int N, int tile_m, bool single_acc, int sms) {
  const long long tiles = static_cast<long long>((N + kTileN - 1) / kTileN) * ((M + tile_m - 1) / tile_m);
  const long long rounds = (tiles + sms - 1) / sms;
  return static_cast<double>(rounds) * (tile_m + 32) * (single_acc ? 1.05 : 1.0);
}

}  // namespace

int gemm_splits(int M, int N, int K) {
  if (M < 1 || M > CfgNarrow::kTileM) return 1;
  const int sms = sm_count();
  const int tiles = (N + kTileN - 1) / kTileN;      // one 128-token tile column
  const int ktiles = K / kTileK;
  if (2 * tiles > sms || ktiles < 8) return 1;
  // enough parts to fill the SMs, each of at least four K steps
  return std::max(1, std::min(sms / tiles, ktiles / 4));
}

cudaError_t launch_gemm(const GemmProblem& g, WsHeader* status, bool pdl, cudaStream_t st) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  const int sms = sm_count();
  if (g.M <= CfgNarrow::kTileM) {
    const int splits = gemm_splits(g.M, g.N, g.K);
    if (splits > 1 && g.acc_ws != nullptr) {
      cudaError_t err = cudaMemsetAsync(g.acc_ws, 0, static_cast<size_t>(g.M) * g.N * 4, st);
      if (err == cudaSuccess) err = launch_cfg<CfgNarrow>(g, status, false, st, splits);
      if (err != cudaSuccess) return err;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(std::min((g.N + 255) / 256, 64)), static_cast<unsigned>(g.M));
      cfg.blockDim = dim3(256);
      cfg.stream = st;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      return cudaLaunchKernelEx(&cfg, split_finalize_kernel, static_cast<const int32_t*>(g.acc_ws), g.M, g.N, g.m,
                                g.s_w, g.Y, g.acc, g.relu2 ? 1 : 0, g.mul);
    }
    return launch_cfg<CfgNarrow>(g, status, pdl, st, 1);
  }
  const double wide = tile_cost(g.M, g.N, CfgWide::kTileM, true, sms);
  const double mid = tile_cost(g.M, g.N, CfgMid::kTileM, false, sms);
  const double narrow = tile_cost(g.M, g.N, CfgNarrow::kTileM, false, sms);
  if (wide <= mid && wide <= narrow) return launch_cfg<CfgWide>(g, status, pdl, st, 1);
  if (mid <= narrow) return launch_cfg<CfgMid>(g, status, pdl, st, 1);
  return launch_cfg<CfgNarrow>(g, status, pdl, st, 1);
}

}  // namespace bl
