// C ABI of the BitLinear library: argument checks, workspace layout and the
// launch sequence of each call. The kernels live in pack.cu, quant.cu,
// gemv.cu (decode, fewer than kGemmMinTokens tokens) and gemm_tc.cu (more).
#include <atomic>
#include <cmath>

#include "common.cuh"
#include "launchers.h"

namespace bl {
namespace {

constexpr int kAbiVersion = 102;

// Per-device capability cache: 0 unknown, 1 compute capability 10.3, -1 other.
std::atomic<int> g_dev_ok[64];

bl_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BL_ERR_CUDA;
  if (dev < 0 || dev >= 64) return BL_ERR_UNSUPPORTED;
  int v = g_dev_ok[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return BL_ERR_CUDA;
    v = (major == 10 && minor == 3) ? 1 : -1;
    g_dev_ok[dev].store(v, std::memory_order_relaxed);
  }
  return v == 1 ? BL_OK : BL_ERR_UNSUPPORTED;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_k(int K) { return K > 0 && K % 64 == 0 && K <= kMaxK; }

bool valid_nk(int N, int K) { return N >= 0 && valid_k(K) && static_cast<long long>(N) * K < (1ll << 31); }

bool valid_eps(float eps) { return std::isfinite(eps) && eps > 0.0f; }

bool valid_dtype(int d) { return d == BL_DTYPE_F32 || d == BL_DTYPE_BF16; }

bl_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BL_OK : BL_ERR_CUDA; }

// A GEMM with its K cut into parts needs an [M][N] int32 scratch for the
// partial sums (the forward takes the GEMM from kGemmMinTokens tokens;
// bitlinear_forward_tc for any count).
bool uses_split(int M, int N, int K) { return gemm_splits(M, N, K) > 1; }

// A single GEMV launch (up to 4 tokens) quantizes its raw rows in-kernel when
// they hold at most this many values; measured on B300, the staging of 4 rows
// of 8192 fp32 values in every CTA cost more than the launch it saves.
constexpr int kGemvInKernelQuantTokens = 4;
constexpr int kGemvInKernelQuantElems = 16384;

// Forward workspace: header | q (M*K fp16 or int8) | m [M] | split-K sums [M*N] int32
// Batch workspace: header | q of every problem (M_p * K_p int8 each) | m of every problem
struct FwdLayout {
  size_t q, m, accw, total;
};
FwdLayout fwd_layout(int M, int N, int K) {
  FwdLayout L;
  L.q = sizeof(WsHeader);
  L.m = align_up(L.q + static_cast<size_t>(M) * K * 2, 256);
  L.accw = align_up(L.m + 4 * static_cast<size_t>(M), 256);
  L.total = uses_split(M, N, K) ? align_up(L.accw + 4 * static_cast<size_t>(M) * N, 256) : L.accw;
  return L;
}

// FFN workspace: header | qx | mx | h [M*F] fp32 | qh | mh | split-K sums
// (gated: then ReLU^2(gate) [M*F] after the split-K sums)
struct FfnLayout {
  size_t qx, mx, h, qh, mh, accw, g, total;
};
FfnLayout ffn_layout(int M, int D, int F, bool gated = false) {
  FfnLayout L;
  const size_t m4 = 4 * static_cast<size_t>(M);
  L.qx = sizeof(WsHeader);
  L.mx = align_up(L.qx + static_cast<size_t>(M) * D * 2, 256);
  L.h = align_up(L.mx + m4, 256);
  L.qh = align_up(L.h + static_cast<size_t>(M) * F * 4, 256);
  L.mh = align_up(L.qh + static_cast<size_t>(M) * F * 2, 256);
  L.accw = align_up(L.mh + m4, 256);
  const bool split = uses_split(M, F, D) || uses_split(M, D, F);
  L.g = split ? align_up(L.accw + 4 * static_cast<size_t>(M) * std::max(D, F), 256) : L.accw;
  L.total = gated ? align_up(L.g + 4 * static_cast<size_t>(M) * F, 256) : L.g;
  return L;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

GemvProblem make_problem(int M, int K, const uint8_t* packed, const float* s_w, int N, float* Y, int32_t* acc) {
  GemvProblem p = {};
  p.Wp = packed;
  p.s_w = s_w;
  p.N = N;
  p.K = K;
  p.M = M;
  p.Y = Y;
  p.acc = acc;
  p.epi = Epi::kPlain;
  return p;
}

GemmProblem make_gemm(int M, int K, const uint8_t* packed, const float* s_w, int N, const void* act, const float* m,
                      float* Y, int32_t* acc, bool relu2, int32_t* acc_ws) {
  GemmProblem g = {};
  g.Wp = packed;
  g.s_w = s_w;
  g.M = M;
  g.N = N;
  g.K = K;
  g.act = act;
  g.m = m;
  g.Y = Y;
  g.acc = acc;
  g.relu2 = relu2;
  g.acc_ws = uses_split(M, N, K) ? acc_ws : nullptr;
  return g;
}

bl_status check_linear_args(int M, int K, const uint8_t* packed, const float* s_w, int N, const float* Y,
                            const int32_t* acc, void* workspace, size_t workspace_bytes) {
  if (M < 0 || !valid_nk(N, K)) return BL_ERR_SHAPE;
  if (M == 0 || N == 0) return BL_OK;
  if (!packed || !s_w || !Y || !workspace) return BL_ERR_ARG;
  if (!aligned16(packed) || !aligned16(Y) || !aligned16(workspace) || (acc && !aligned16(acc)) ||
      (reinterpret_cast<uintptr_t>(s_w) & 3u))
    return BL_ERR_ALIGN;
  if (workspace_bytes < bitlinear_workspace_bytes(BL_OP_FORWARD, M, N, K)) return BL_ERR_WORKSPACE;
  return check_device();
}

// The BitLinear forward, with the RMSNorm fused into its quantization when
// `norm` is given.
bl_status run_forward(const void* X, int x_dtype, int M, int K, const RmsNorm* norm, const uint8_t* packed,
                      const float* s_w, int N, float eps, float* Y, int32_t* acc, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!valid_dtype(x_dtype) || !valid_eps(eps)) return BL_ERR_ARG;
  if (M < 0 || !valid_nk(N, K)) return BL_ERR_SHAPE;
  if (M == 0 || N == 0) return BL_OK;
  if (!X) return BL_ERR_ARG;
  if (!aligned16(X)) return BL_ERR_ALIGN;
  if (bl_status s = check_linear_args(M, K, packed, s_w, N, Y, acc, workspace, workspace_bytes); s != BL_OK)
    return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const FwdLayout L = fwd_layout(M, N, K);
  float* m = at<float>(workspace, L.m);
  if (M >= kGemmMinTokens) {
    // prefill: fp16 activations in the tensor-core order, then the tcgen05 GEMM
    void* act = at<void>(workspace, L.q);
    if (launch_quant(X, x_dtype, M, K, eps, QLayout::kPairF16, act, m, norm, true, st) != cudaSuccess)
      return BL_ERR_CUDA;
    return from_cuda(launch_gemm(make_gemm(M, K, packed, s_w, N, act, m, Y, acc, false, at<int32_t>(workspace, L.accw)),
                                 static_cast<WsHeader*>(workspace), true, st));
  }
  GemvProblem p = make_problem(M, K, packed, s_w, N, Y, acc);
  if (norm == nullptr && M <= kGemvInKernelQuantTokens && M * K <= kGemvInKernelQuantElems) {
    // decode without a norm, few short rows: the GEMV quantizes them while
    // staging (one launch instead of two in a chain of dependent calls);
    // every CTA reads the raw rows twice, so longer or more rows go through
    // the quantization kernel once
    p.x = X;
    p.x_dtype = x_dtype;
    p.eps = eps;
    return from_cuda(launch_gemv(p, static_cast<WsHeader*>(workspace), true, st));
  }
  int8_t* q = at<int8_t>(workspace, L.q);
  if (launch_quant(X, x_dtype, M, K, eps, QLayout::kRowMajorI8, q, m, norm, true, st) != cudaSuccess)
    return BL_ERR_CUDA;
  p.q = q;
  p.m = m;
  return from_cuda(launch_gemv(p, static_cast<WsHeader*>(workspace), true, st));
}

}  // namespace
}  // namespace bl

using namespace bl;

extern "C" {

int bitlinear_version(void) { return kAbiVersion; }

const char* bitlinear_status_str(int status) {
  switch (status) {
    case BL_OK: return "BL_OK";
    case BL_ERR_ARG: return "BL_ERR_ARG: invalid argument";
    case BL_ERR_SHAPE: return "BL_ERR_SHAPE: unsupported shape";
    case BL_ERR_ALIGN: return "BL_ERR_ALIGN: pointer not 16-byte aligned";
    case BL_ERR_CUDA: return "BL_ERR_CUDA: CUDA call or launch failed";
    case BL_ERR_TIMEOUT: return "BL_ERR_TIMEOUT: device-side wait gave up";
    case BL_ERR_UNSUPPORTED: return "BL_ERR_UNSUPPORTED: device is not compute capability 10.3";
    case BL_ERR_WORKSPACE: return "BL_ERR_WORKSPACE: workspace too small";
    default: return "unknown bl_status";
  }
}

size_t bitlinear_workspace_bytes(int op, int M, int N, int K) {
  switch (op) {
    case BL_OP_PACK:
      if (!valid_nk(N, K) || N == 0) return 0;
      return sizeof(WsHeader) + pack_scratch_bytes();
    case BL_OP_FORWARD:
      if (M < 0 || !valid_nk(N, K)) return 0;
      return fwd_layout(M, N, K).total;
    case BL_OP_FORWARD_BATCH:     // M = total tokens of the batch, K = the largest K
      if (M < 0 || (M > 0 && !valid_k(K))) return 0;
      return sizeof(WsHeader) + align_up(static_cast<size_t>(M) * (M > 0 ? K : 0), 256) +
             align_up(4 * static_cast<size_t>(M), 256);
    case BL_OP_FFN:
    case BL_OP_FFN_GATED:
      if (M < 0 || !valid_nk(N, K) || !valid_k(N) || N == 0) return 0;
      return ffn_layout(M, K, N, op == BL_OP_FFN_GATED).total;
    default: return 0;
  }
}

bl_status bitlinear_pack(const float* W, int N, int K, float eps, uint8_t* packed, float* s_w, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (!W || !packed || !s_w || !workspace) return BL_ERR_ARG;
  if (!valid_eps(eps)) return BL_ERR_ARG;
  if (!valid_nk(N, K) || N == 0) return BL_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(packed) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(s_w) & 3u))
    return BL_ERR_ALIGN;
  if (workspace_bytes < bitlinear_workspace_bytes(BL_OP_PACK, 0, N, K)) return BL_ERR_WORKSPACE;
  if (bl_status s = check_device(); s != BL_OK) return s;
  return from_cuda(launch_pack(W, N, K, eps, packed, s_w, workspace, static_cast<cudaStream_t>(stream)));
}

bl_status bitlinear_quant_act(const void* X, int x_dtype, int M, int K, float eps, int8_t* q, float* m,
                              void* stream) {
  if (!valid_dtype(x_dtype) || !valid_eps(eps)) return BL_ERR_ARG;
  if (M < 0 || !valid_k(K)) return BL_ERR_SHAPE;
  if (M == 0) return BL_OK;
  if (!X || !q || !m) return BL_ERR_ARG;
  if (!aligned16(X) || !aligned16(q) || !aligned16(m)) return BL_ERR_ALIGN;
  if (bl_status s = check_device(); s != BL_OK) return s;
  return from_cuda(launch_quant(X, x_dtype, M, K, eps, QLayout::kRowMajorI8, q, m, nullptr, false,
                                static_cast<cudaStream_t>(stream)));
}

bl_status bitlinear_forward(const void* X, int x_dtype, int M, int K, const uint8_t* packed, const float* s_w, int N,
                            float eps, float* Y, int32_t* acc, void* workspace, size_t workspace_bytes,
                            void* stream) {
  return run_forward(X, x_dtype, M, K, nullptr, packed, s_w, N, eps, Y, acc, workspace, workspace_bytes, stream);
}

bl_status bitlinear_rmsnorm_quant(const void* X, int x_dtype, int M, int K, const float* g, float eps_norm, float eps,
                                  int8_t* q, float* m, void* stream) {
  if (!valid_dtype(x_dtype) || !valid_eps(eps) || !valid_eps(eps_norm)) return BL_ERR_ARG;
  if (M < 0 || !valid_k(K)) return BL_ERR_SHAPE;
  if (M == 0) return BL_OK;
  if (!X || !q || !m) return BL_ERR_ARG;
  if (!aligned16(X) || !aligned16(q) || !aligned16(m) || (g && !aligned16(g))) return BL_ERR_ALIGN;
  if (bl_status s = check_device(); s != BL_OK) return s;
  const RmsNorm norm{g, eps_norm};
  return from_cuda(launch_quant(X, x_dtype, M, K, eps, QLayout::kRowMajorI8, q, m, &norm, false,
                                static_cast<cudaStream_t>(stream)));
}

bl_status bitlinear_forward_rmsnorm(const void* X, int x_dtype, int M, int K, const float* g, float eps_norm,
                                    const uint8_t* packed, const float* s_w, int N, float eps, float* Y,
                                    int32_t* acc, void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_eps(eps_norm)) return BL_ERR_ARG;
  if (g && !aligned16(g)) return BL_ERR_ALIGN;
  const RmsNorm norm{g, eps_norm};
  return run_forward(X, x_dtype, M, K, &norm, packed, s_w, N, eps, Y, acc, workspace, workspace_bytes, stream);
}

bl_status bitlinear_forward_batch(const bl_forward_desc* descs, int count, float eps, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (count < 0 || count > BL_MAX_BATCH || !valid_eps(eps)) return BL_ERR_ARG;
  if (count == 0) return BL_OK;
  if (!descs || !workspace) return BL_ERR_ARG;
  if (!aligned16(workspace)) return BL_ERR_ALIGN;
  if (workspace_bytes < sizeof(WsHeader)) return BL_ERR_WORKSPACE;
  GemvProblem ps[BL_MAX_BATCH];
  QuantProblem qs[BL_MAX_BATCH];
  int qidx[BL_MAX_BATCH];
  int n = 0, nq = 0;
  size_t q_bytes = 0, tokens = 0;
  for (int i = 0; i < count; ++i) {
    const bl_forward_desc& d = descs[i];
    const bool pre = d.x_dtype == BL_DTYPE_I8;
    if (!valid_dtype(d.x_dtype) && !pre) return BL_ERR_ARG;
    if (pre && d.M > 0 && d.N > 0 && !d.m) return BL_ERR_ARG;
    if (d.M < 0 || !valid_nk(d.N, d.K)) return BL_ERR_SHAPE;
    if (d.M == 0 || d.N == 0) continue;
    if (!d.X || !d.packed || !d.s_w || !d.Y) return BL_ERR_ARG;
    if (!aligned16(d.X) || !aligned16(d.packed) || !aligned16(d.Y) || (d.acc && !aligned16(d.acc)) ||
        (reinterpret_cast<uintptr_t>(d.s_w) & 3u))
      return BL_ERR_ALIGN;
    if (pre && (reinterpret_cast<uintptr_t>(d.m) & 3u)) return BL_ERR_ALIGN;
    ps[n] = make_problem(d.M, d.K, d.packed, d.s_w, d.N, d.Y, d.acc);
    if (pre) {
      ps[n].q = static_cast<const int8_t*>(d.X);
      ps[n].m = d.m;
    } else {
      qs[nq] = QuantProblem{d.X, d.x_dtype, d.M, d.K, nullptr, nullptr};
      qidx[nq++] = n;
      q_bytes += static_cast<size_t>(d.M) * d.K;
      tokens += static_cast<size_t>(d.M);
    }
    ++n;
  }
  if (n == 0) return BL_OK;
  // layout: header | q of problem 0, 1, ... | m of problem 0, 1, ...
  const size_t m_off = sizeof(WsHeader) + align_up(q_bytes, 256);
  if (workspace_bytes < m_off + align_up(4 * tokens, 256)) return BL_ERR_WORKSPACE;
  if (bl_status s = check_device(); s != BL_OK) return s;
  size_t qo = sizeof(WsHeader), mo = m_off;
  for (int i = 0; i < nq; ++i) {
    qs[i].q = at<int8_t>(workspace, qo);
    qs[i].m = at<float>(workspace, mo);
    ps[qidx[i]].q = qs[i].q;
    ps[qidx[i]].m = qs[i].m;
    qo += static_cast<size_t>(qs[i].M) * qs[i].K;
    mo += 4 * static_cast<size_t>(qs[i].M);
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (nq > 0 && launch_quant_batch(qs, nq, eps, true, st) != cudaSuccess) return BL_ERR_CUDA;
  return from_cuda(launch_gemv_batch(ps, n, static_cast<WsHeader*>(workspace), true, st));
}

bl_status bitlinear_forward_q8(const int8_t* q, const float* m, int M, int K, const uint8_t* packed, const float* s_w,
                               int N, float* Y, int32_t* acc, void* workspace, size_t workspace_bytes,
                               void* stream) {
  if (M < 0 || !valid_nk(N, K)) return BL_ERR_SHAPE;
  if (M == 0 || N == 0) return BL_OK;
  if (!q || !m) return BL_ERR_ARG;
  if (!aligned16(q) || (reinterpret_cast<uintptr_t>(m) & 3u)) return BL_ERR_ALIGN;
  if (bl_status s = check_linear_args(M, K, packed, s_w, N, Y, acc, workspace, workspace_bytes); s != BL_OK)
    return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (M >= kGemmMinTokens) {
    const FwdLayout L = fwd_layout(M, N, K);
    void* act = at<void>(workspace, L.q);
    if (launch_widen_pair(q, M, K, act, true, st) != cudaSuccess) return BL_ERR_CUDA;
    return from_cuda(launch_gemm(make_gemm(M, K, packed, s_w, N, act, m, Y, acc, false, at<int32_t>(workspace, L.accw)),
                                 static_cast<WsHeader*>(workspace), true, st));
  }
  GemvProblem p = make_problem(M, K, packed, s_w, N, Y, acc);
  p.q = q;
  p.m = m;
  return from_cuda(launch_gemv(p, static_cast<WsHeader*>(workspace), true, st));
}

bl_status bitlinear_quant_act_tc(const void* X, int x_dtype, int M, int K, float eps, void* act, float* m,
                                 void* stream) {
  if (!valid_dtype(x_dtype) || !valid_eps(eps)) return BL_ERR_ARG;
  if (M < 0 || !valid_k(K)) return BL_ERR_SHAPE;
  if (M == 0) return BL_OK;
  if (!X || !act || !m) return BL_ERR_ARG;
  if (!aligned16(X) || !aligned16(act) || (reinterpret_cast<uintptr_t>(m) & 3u)) return BL_ERR_ALIGN;
  if (bl_status s = check_device(); s != BL_OK) return s;
  return from_cuda(launch_quant(X, x_dtype, M, K, eps, QLayout::kPairF16, act, m, nullptr, false,
                                static_cast<cudaStream_t>(stream)));
}

bl_status bitlinear_forward_tc(const void* act, const float* m, int M, int K, const uint8_t* packed,
                               const float* s_w, int N, float* Y, int32_t* acc, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (M < 0 || !valid_nk(N, K)) return BL_ERR_SHAPE;
  if (M == 0 || N == 0) return BL_OK;
  if (!act || !m || !packed || !s_w || !Y || !workspace) return BL_ERR_ARG;
  if (!aligned16(act) || !aligned16(packed) || !aligned16(Y) || !aligned16(workspace) || (acc && !aligned16(acc)) ||
      (reinterpret_cast<uintptr_t>(m) & 3u) || (reinterpret_cast<uintptr_t>(s_w) & 3u))
    return BL_ERR_ALIGN;
  if (workspace_bytes < sizeof(WsHeader)) return BL_ERR_WORKSPACE;
  if (bl_status s = check_device(); s != BL_OK) return s;
  // with room for the [M][N] partial sums right after the header, few tokens
  // may cut K across more SMs
  const size_t accw = sizeof(WsHeader);
  int32_t* acc_ws = workspace_bytes >= accw + 4 * static_cast<size_t>(M) * N ? at<int32_t>(workspace, accw) : nullptr;
  return from_cuda(launch_gemm(make_gemm(M, K, packed, s_w, N, act, m, Y, acc, false, acc_ws),
                               static_cast<WsHeader*>(workspace), true, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// The FFN block: up (and gate) on one quantization of X, ReLU^2 (times the up
// projection when gated), requantization, down. gate == nullptr: ungated.
// With n_in / n_sub the RMSNorms of SubLN are fused into the quantization of
// X and of h.
bl_status run_ffn(const void* X, int x_dtype, int M, int D, const uint8_t* up, const float* s_up,
                  const uint8_t* gate, const float* s_gate, const uint8_t* down, const float* s_down, int F,
                  float eps, float* Y, void* workspace, size_t workspace_bytes, void* stream,
                  const RmsNorm* n_in = nullptr, const RmsNorm* n_sub = nullptr) {
  const bool gated = gate != nullptr || s_gate != nullptr;
  if (!valid_dtype(x_dtype) || !valid_eps(eps)) return BL_ERR_ARG;
  if (M < 0 || !valid_nk(F, D) || !valid_nk(D, F) || F == 0) return BL_ERR_SHAPE;
  if (M == 0) return BL_OK;
  if (!X || !up || !s_up || !down || !s_down || !Y || !workspace || (gated && (!gate || !s_gate)))
    return BL_ERR_ARG;
  if (!aligned16(X) || !aligned16(up) || !aligned16(down) || !aligned16(Y) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(s_up) & 3u) || (reinterpret_cast<uintptr_t>(s_down) & 3u) ||
      (gated && (!aligned16(gate) || (reinterpret_cast<uintptr_t>(s_gate) & 3u))))
    return BL_ERR_ALIGN;
  if (workspace_bytes < bitlinear_workspace_bytes(gated ? BL_OP_FFN_GATED : BL_OP_FFN, M, F, D))
    return BL_ERR_WORKSPACE;
  if (bl_status s = check_device(); s != BL_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const FfnLayout L = ffn_layout(M, D, F, gated);
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  float* mx = at<float>(workspace, L.mx);
  float* h = at<float>(workspace, L.h);
  float* mh = at<float>(workspace, L.mh);
  float* g = gated ? at<float>(workspace, L.g) : nullptr;
  if (M >= kGemmMinTokens) {
    void* ax = at<void>(workspace, L.qx);
    void* ah = at<void>(workspace, L.qh);
    int32_t* accw = at<int32_t>(workspace, L.accw);
    if (launch_quant(X, x_dtype, M, D, eps, QLayout::kPairF16, ax, mx, n_in, true, st) != cudaSuccess)
      return BL_ERR_CUDA;
    if (gated) {
      if (launch_gemm(make_gemm(M, D, gate, s_gate, F, ax, mx, g, nullptr, true, accw), hdr, true, st) !=
          cudaSuccess)
        return BL_ERR_CUDA;
      GemmProblem gu = make_gemm(M, D, up, s_up, F, ax, mx, h, nullptr, false, accw);
      gu.mul = g;
      if (launch_gemm(gu, hdr, true, st) != cudaSuccess) return BL_ERR_CUDA;
    } else if (launch_gemm(make_gemm(M, D, up, s_up, F, ax, mx, h, nullptr, true, accw), hdr, true, st) !=
               cudaSuccess) {
      return BL_ERR_CUDA;
    }
    if (launch_quant(h, BL_DTYPE_F32, M, F, eps, QLayout::kPairF16, ah, mh, n_sub, true, st) !=
        cudaSuccess)
      return BL_ERR_CUDA;
    return from_cuda(launch_gemm(make_gemm(M, F, down, s_down, D, ah, mh, Y, nullptr, false, accw), hdr, true, st));
  }
  int8_t* qx = at<int8_t>(workspace, L.qx);
  int8_t* qh = at<int8_t>(workspace, L.qh);
  if (launch_quant(X, x_dtype, M, D, eps, QLayout::kRowMajorI8, qx, mx, n_in, true, st) != cudaSuccess)
    return BL_ERR_CUDA;
  if (gated) {
    GemvProblem pg = make_problem(M, D, gate, s_gate, F, g, nullptr);
    pg.q = qx;
    pg.m = mx;
    pg.epi = Epi::kRelu2;
    if (launch_gemv(pg, hdr, true, st) != cudaSuccess) return BL_ERR_CUDA;
  }
  GemvProblem pu = make_problem(M, D, up, s_up, F, h, nullptr);
  pu.q = qx;
  pu.m = mx;
  if (gated) pu.mul = g;
  else pu.epi = Epi::kRelu2;
  if (launch_gemv(pu, hdr, true, st) != cudaSuccess) return BL_ERR_CUDA;
  if (launch_quant(h, BL_DTYPE_F32, M, F, eps, QLayout::kRowMajorI8, qh, mh, n_sub, true, st) !=
      cudaSuccess)
    return BL_ERR_CUDA;
  GemvProblem pd = make_problem(M, F, down, s_down, D, Y, nullptr);
  pd.q = qh;
  pd.m = mh;
  return from_cuda(launch_gemv(pd, hdr, true, st));
}

}  // namespace

extern "C" {

bl_status bitlinear_ffn(const void* X, int x_dtype, int M, int D, const uint8_t* up, const float* s_up,
                        const uint8_t* down, const float* s_down, int F, float eps, float* Y, void* workspace,
                        size_t workspace_bytes, void* stream) {
  return run_ffn(X, x_dtype, M, D, up, s_up, nullptr, nullptr, down, s_down, F, eps, Y, workspace, workspace_bytes,
                 stream);
}

bl_status bitlinear_ffn_gated(const void* X, int x_dtype, int M, int D, const uint8_t* up, const float* s_up,
                              const uint8_t* gate, const float* s_gate, const uint8_t* down, const float* s_down,
                              int F, float eps, float* Y, void* workspace, size_t workspace_bytes, void* stream) {
  if (!gate || !s_gate) return BL_ERR_ARG;
  return run_ffn(X, x_dtype, M, D, up, s_up, gate, s_gate, down, s_down, F, eps, Y, workspace, workspace_bytes,
                 stream);
}

bl_status bitlinear_ffn_subln(const void* X, int x_dtype, int M, int D, const float* g_in, const uint8_t* up,
                              const float* s_up, const uint8_t* gate, const float* s_gate, const float* g_sub,
                              const uint8_t* down, const float* s_down, int F, float eps_norm, float eps, float* Y,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_eps(eps_norm) || (gate == nullptr) != (s_gate == nullptr)) return BL_ERR_ARG;
  if ((g_in && !aligned16(g_in)) || (g_sub && !aligned16(g_sub))) return BL_ERR_ALIGN;
  const RmsNorm n_in{g_in, eps_norm}, n_sub{g_sub, eps_norm};
  return run_ffn(X, x_dtype, M, D, up, s_up, gate, s_gate, down, s_down, F, eps, Y, workspace, workspace_bytes,
                 stream, &n_in, &n_sub);
}

bl_status bitlinear_unpack(const uint8_t* packed, int N, int K, int8_t* t, void* stream) {
  if (!valid_nk(N, K)) return BL_ERR_SHAPE;
  if (N == 0) return BL_OK;
  if (!packed || !t) return BL_ERR_ARG;
  if (!aligned16(packed) || !aligned16(t)) return BL_ERR_ALIGN;
  if (bl_status s = check_device(); s != BL_OK) return s;
  return from_cuda(launch_unpack(packed, N, K, t, static_cast<cudaStream_t>(stream)));
}

bl_status bitlinear_workspace_status(void* workspace, void* stream) {
  if (!workspace) return BL_ERR_ARG;
  if (!aligned16(workspace)) return BL_ERR_ALIGN;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader h;
  if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return BL_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return BL_ERR_CUDA;
  if (h.status == 0) return BL_OK;
  if (cudaMemsetAsync(workspace, 0, sizeof(WsHeader), st) != cudaSuccess) return BL_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return BL_ERR_CUDA;
  return static_cast<bl_status>(h.status);
}

}  // extern "C"
