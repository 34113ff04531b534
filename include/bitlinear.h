/*
 * bitlinear.h - C ABI of the BitLinear forward of BitNet b1.58 on B300 (sm_103a).
 *
 * What the calls compute (sources are the pages' titles and sections):
 *   - "BitNet解读" (markgoyens.top), 模型架构 / 权重量化函数, eqs. (1)-(3):
 *       gamma = (1/nm) sum |W_ij|;  W~ = RoundClip(W / (gamma + eps), -1, 1).
 *     Same section, 激活量化: activations scaled per token into [-Qb, Qb],
 *     symmetric, no zero point (Qb = 127 here).
 *   - "BitNet b1.58 2B4T Technical Report | Summary", 5.1 GPU Inference (and
 *     the Chinese translation of the report, 5.1 GPU推理): four ternary values
 *     are packed into one 8-bit value in HBM, loaded, unpacked on chip and
 *     multiplied with 8-bit activations.
 *   - "BitNet解读", 革命性的效率提升: the matmul is integer additions and
 *     subtractions (+1 adds, -1 subtracts, 0 skips).
 *   - bitnet.cpp intro (gitcode.csdn.net), 1.1: the result is scaled back
 *     with the scale factors; the report's section 2 (架构): BitLinear replaces
 *     torch.nn.Linear, no bias terms, the FFN uses squared ReLU.
 *
 * Exact definitions used by every call (fp32 is IEEE round-to-nearest-even):
 *   gamma  = exact mean of |W| rounded once to fp32;  s_w = fp32(gamma + eps)
 *   t_nk   = clamp(rint(fp32(W_nk / s_w)), -1, 1)            (int, {-1,0,1})
 *   packed = byte (n, b) holds t+1 of column k = 4b+j in bits [2j, 2j+1]
 *   m_i    = max(max_k |x_ik|, eps)
 *   q_ik   = clamp(rint(fp32(fp32(x_ik * 127) / m_i)), -128, 127)
 *   acc_in = sum_k q_ik * t_nk                                 (exact int32)
 *   y_in   = fp32(float(acc_in) * fp32(fp32(s_w * m_i) / 127))
 *   FFN    : h = y_up > 0 ? fp32(y_up * y_up) : 0, requantized as above,
 *            then the down projection (no gate, no norm in between).
 *   RMSNorm: (the *_rmsnorm / *_subln calls) with gain g [K] (null: 1) and
 *            r_i = 1 / sqrt(S_i / K + eps_norm), S_i = sum_k x_ik^2, in fp64:
 *            codes from u_ik = fp32(x_ik * g_k) as above (absmax codes do not
 *            change under the positive factor r_i), m_i = fp32(max(max_k
 *            |u_ik|, eps) * r_i). S_i is summed with compensated fp32
 *            arithmetic, far below an fp32 step from exact, so m_i matches
 *            the exact-sum value except within that distance of an fp32
 *            rounding boundary (then it is one step off).
 *
 * Conventions for every call:
 *   - All tensors are row-major, on the current CUDA device, allocated and
 *     owned by the caller; the library allocates nothing and keeps no state
 *     besides per-device attributes it queries once.
 *   - Every device pointer must be 16-byte aligned (BL_ERR_ALIGN otherwise).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). All work is
 *     enqueued on it asynchronously; a call returns once the work is queued.
 *     Scales stay on the device, so no call synchronizes the host.
 *   - Shapes: M >= 0 and N >= 0 (zero is a valid no-op); K > 0, K % 64 == 0,
 *     K <= 65536, N * K < 2^31 (BL_ERR_SHAPE otherwise). The K bound keeps
 *     every partial sum of the contraction an integer below 2^24.
 *   - Arguments are checked on the host before any launch; nothing is
 *     launched when a check fails. A failed launch returns BL_ERR_CUDA.
 *   - `workspace` is scratch device memory of at least
 *     bitlinear_workspace_bytes(op, ...) bytes. Its first 256 bytes hold a
 *     sticky device status word: zero them once when the workspace is
 *     allocated; bitlinear_workspace_status() reads and clears it. Calls that
 *     share one workspace must be ordered on one stream.
 *   - Non-finite inputs are outside the contract: results are unspecified
 *     (bitlinear_pack writes s_w = NaN when W holds Inf or NaN).
 */
#ifndef BITLINEAR_H
#define BITLINEAR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BL_API __attribute__((visibility("default")))
#else
#define BL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BL_OK = 0,
  BL_ERR_ARG = 1,          /* null pointer, unknown dtype/op, eps not finite and > 0   */
  BL_ERR_SHAPE = 2,        /* shape outside the supported range (see above)          */
  BL_ERR_ALIGN = 3,        /* a pointer is not 16-byte aligned                       */
  BL_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed            */
  BL_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up (see workspace_status) */
  BL_ERR_UNSUPPORTED = 6,  /* current device is not compute capability 10.3          */
  BL_ERR_WORKSPACE = 7     /* workspace smaller than bitlinear_workspace_bytes()     */
} bl_status;

typedef enum {
  BL_DTYPE_F32 = 0,
  BL_DTYPE_BF16 = 1,
  BL_DTYPE_I8 = 2      /* already quantized (int8 + per-token scale); bl_forward_desc only */
} bl_dtype;

typedef enum {
  BL_OP_PACK = 0,          /* bitlinear_pack(N, K)                          */
  BL_OP_FORWARD = 1,       /* bitlinear_forward(M, N, K)                    */
  BL_OP_FFN = 2,           /* bitlinear_ffn(M, N = F (hidden), K = D (model)) */
  BL_OP_FORWARD_BATCH = 3, /* bitlinear_forward_batch(M = total tokens of all
                              problems, K = their largest K, N ignored)      */
  BL_OP_FFN_GATED = 4      /* bitlinear_ffn_gated(M, N = F (hidden), K = D)  */
} bl_op;

/* Version of this ABI (major * 100 + minor). */
BL_API int bitlinear_version(void);

/* Human-readable name of a bl_status value. Never NULL. */
BL_API const char* bitlinear_status_str(int status);

/* Bytes of workspace the call `op` needs for these sizes (0 if the sizes are
 * invalid). For BL_OP_PACK pass M = 0. */
BL_API size_t bitlinear_workspace_bytes(int op, int M, int N, int K);

/*
 * Absmean ternary quantization and 2-bit packing of one weight matrix
 * ("BitNet解读", 权重量化函数, eqs. (1)-(3); packing per the report's 5.1).
 *   W        [N, K] fp32, device.
 *   eps      > 0 (1e-5 in the reference configuration).
 *   packed   [N, K/4] uint8, device, output (the layout documented above).
 *   s_w      [1] fp32, device, output: fp32(gamma + eps).
 *   workspace >= bitlinear_workspace_bytes(BL_OP_PACK, 0, N, K) bytes.
 * gamma is exact (order-independent), so packed and s_w are bit-exact
 * functions of W.
 */
BL_API bl_status bitlinear_pack(const float* W, int N, int K, float eps,
                         uint8_t* packed, float* s_w,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * Per-token absmax int8 quantization ("BitNet解读", 激活量化).
 *   X        [M, K] fp32 (x_dtype = BL_DTYPE_F32) or bf16 bits (BL_DTYPE_BF16,
 *            widened exactly to fp32 first), device.
 *   q        [M, K] int8, device, output.
 *   m        [M] fp32, device, output: max(max_k |x_ik|, eps).
 */
BL_API bl_status bitlinear_quant_act(const void* X, int x_dtype, int M, int K, float eps,
                              int8_t* q, float* m, void* stream);

/*
 * BitLinear forward Y = dequant(quant(X) . T^T) (no bias).
 *   X        [M, K] fp32 or bf16, device.
 *   packed   [N, K/4] uint8 from bitlinear_pack; s_w [1] fp32, device.
 *   Y        [M, N] fp32, device, output.
 *   acc      [M, N] int32, device, output, or NULL: the exact integer
 *            accumulators (for checking).
 *   workspace >= bitlinear_workspace_bytes(BL_OP_FORWARD, M, N, K) bytes.
 */
BL_API bl_status bitlinear_forward(const void* X, int x_dtype, int M, int K,
                            const uint8_t* packed, const float* s_w, int N, float eps,
                            float* Y, int32_t* acc,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * One problem of bitlinear_forward_batch: the arguments of one
 * bitlinear_forward call (all pointers on the device).
 */
typedef struct {
  const void* X;            /* [M, K] fp32, bf16, or int8 (BL_DTYPE_I8)  */
  int x_dtype;              /* BL_DTYPE_F32, BL_DTYPE_BF16 or BL_DTYPE_I8 */
  int M;                    /* tokens (>= 0)                             */
  int K;                    /* input features                            */
  int N;                    /* output features (>= 0)                    */
  const uint8_t* packed;    /* [N, K/4] from bitlinear_pack              */
  const float* s_w;         /* [1]                                       */
  float* Y;                 /* [M, N] output                             */
  int32_t* acc;             /* [M, N] int32 output, or NULL              */
  const float* m;           /* BL_DTYPE_I8 only: [M] per-token scales as
                               written by bitlinear_quant_act; else NULL */
} bl_forward_desc;

#define BL_MAX_BATCH 128

/*
 * `count` independent BitLinear forwards in one launch sequence (e.g. the
 * q, k and v projections of a layer, or the projections of several
 * independent sequences): each result equals that of bitlinear_forward on
 * the same arguments (or of bitlinear_forward_q8 for BL_DTYPE_I8 inputs).
 * No problem may read another's outputs. One kernel quantizes the inputs of
 * all problems, then the packed weights of all problems stream through one
 * grid, so small matrices do not each pay a launch and a pipeline ramp.
 *   descs     host array of `count` descriptors (0 <= count <= BL_MAX_BATCH),
 *             read during the call only.
 *   workspace >= bitlinear_workspace_bytes(BL_OP_FORWARD_BATCH, sum of M, 0,
 *             largest K) bytes (the quantized activations of every problem;
 *             problems given as BL_DTYPE_I8 need none).
 * Each descriptor is checked like bitlinear_forward's arguments; the first
 * failing check is returned and nothing is launched.
 */
BL_API bl_status bitlinear_forward_batch(const bl_forward_desc* descs, int count, float eps,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * BitLinear forward on an input that is already quantized: q [M, K] int8 and
 * m [M] fp32 as written by bitlinear_quant_act (e.g. one quantization shared
 * by the q, k and v projections, which read the same activations; each
 * BitLinear quantizes its input the same way, so the result is identical to
 * bitlinear_forward on the unquantized X). Other arguments as above.
 */
BL_API bl_status bitlinear_forward_q8(const int8_t* q, const float* m, int M, int K,
                               const uint8_t* packed, const float* s_w, int N,
                               float* Y, int32_t* acc,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * Per-token absmax quantization ("BitNet解读", 激活量化) into the operand form
 * of the tensor-core contraction: the same int8 values q as
 * bitlinear_quant_act, stored as fp16 [M, K] (exact: |q| <= 128), with the
 * columns of every 16-column group in the order 0, 8, 1, 9, ..., 7, 15.
 *   act      [M, K] fp16 (2 bytes per element), device, output, 16-byte aligned.
 *   m        [M] fp32, device, output.
 * Use it to quantize once and run several bitlinear_forward_tc calls.
 */
BL_API bl_status bitlinear_quant_act_tc(const void* X, int x_dtype, int M, int K, float eps, void* act, float* m,
                                 void* stream);

/*
 * BitLinear forward on an input already in the tensor-core operand form
 * (bitlinear_quant_act_tc): the tcgen05 contraction and the dequant epilogue
 * only ("BitNet b1.58 2B4T Technical Report | Summary", 5.1: packed weights
 * unpacked on chip and multiplied with 8-bit activations). Any M >= 0; the
 * result equals bitlinear_forward on the unquantized input.
 *   workspace >= 256 bytes (its status word; see bitlinear_workspace_status).
 *             With 256 + 4 * M * N bytes, few tokens (M <= 128) may cut K into
 *             parts run on more SMs, their exact integer partial sums added
 *             in the workspace.
 */
BL_API bl_status bitlinear_forward_tc(const void* act, const float* m, int M, int K,
                               const uint8_t* packed, const float* s_w, int N,
                               float* Y, int32_t* acc,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * Size of the fixed device scratch array behind bitlinear_forward_noalloc.
 */
#define BL_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * bitlinear_forward without a workspace argument. The pages have no
 * counterpart to this call; it exists for callers that cannot allocate
 * device memory when they run the forward (a runtime that fixes its memory
 * plan at start-up, a plugin whose host framework owns all device memory).
 * It computes exactly what bitlinear_forward computes, with the same launch
 * sequence, and calls no cudaMalloc, cudaFree or other allocating routine.
 *   Scratch: a library-owned array of BL_STATIC_SCRATCH_BYTES (8 MiB) in device
 *     global memory, present on every GPU that loads the library until the
 *     process exits. Sizes whose bitlinear_workspace_bytes(BL_OP_FORWARD, M, N,
 *     K) exceeds it return BL_ERR_WORKSPACE before any launch (e.g. M * K up to
 *     about 4 million activations).
 *   The first call on each device looks up the array's device address with
 *     cudaGetSymbolAddress (set-up); make that first call before any stream
 *     capture.
 *   All calls on a device share the one array, and it keeps the last call's
 *     contents (nothing in it has to start at zero: each call writes its
 *     scratch before reading it). Calls that overlap on the GPU (e.g. on two
 *     streams without ordering) race on it: order them.
 *   Other arguments, checks and error codes as for bitlinear_forward.
 */
BL_API bl_status bitlinear_forward_noalloc(const void* X, int x_dtype, int M, int K,
                                    const uint8_t* packed, const float* s_w, int N, float eps,
                                    float* Y, int32_t* acc, void* stream);

/*
 * FFN block of the 2B4T architecture (report section 2: squared ReLU):
 *   Y = BitLinear_down(ReLU^2(BitLinear_up(X))), ungated, each BitLinear
 *   quantizing its own input per token.
 *   X        [M, D] fp32 or bf16; up [F, D/4] uint8 + s_up [1]; down [D, F/4]
 *            uint8 + s_down [1]; Y [M, D] fp32 output. D and F obey the K rules.
 *   workspace >= bitlinear_workspace_bytes(BL_OP_FFN, M, F, D) bytes.
 */
BL_API bl_status bitlinear_ffn(const void* X, int x_dtype, int M, int D,
                        const uint8_t* up, const float* s_up,
                        const uint8_t* down, const float* s_down, int F, float eps,
                        float* Y, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Gated FFN block: Y = BitLinear_down(ReLU^2(BitLinear_gate(X)) * BitLinear_up(X)),
 *   the squared ReLU of the report's section 2 (架构) in place of SwiGLU's SiLU
 *   in a gated unit; gate and up quantize the same input once; the product h
 *   = fp32(fp32(ReLU(y_gate)^2) * y_up) is requantized per token before down.
 *   up, gate [F, D/4] uint8 + s_up, s_gate [1]; other arguments as bitlinear_ffn.
 *   workspace >= bitlinear_workspace_bytes(BL_OP_FFN_GATED, M, F, D) bytes.
 */
BL_API bl_status bitlinear_ffn_gated(const void* X, int x_dtype, int M, int D,
                              const uint8_t* up, const float* s_up,
                              const uint8_t* gate, const float* s_gate,
                              const uint8_t* down, const float* s_down, int F, float eps,
                              float* Y, void* workspace, size_t workspace_bytes, void* stream);

/*
 * SubLN's RMSNorm fused into the per-token absmax quantization ("BitNet b1.58
 * 2B4T Technical Report", section 2 (架构): a sub-layer norm, norm layers
 * without bias; "BitNet解读", 模型架构 / 组件兼容性: RMSNorm as the norm).
 *   X        [M, K] fp32 or bf16, device.  g [K] fp32 gain, device, or NULL
 *            (unit gain). eps_norm > 0 and finite (1e-5 in the reference
 *            configuration); eps as bitlinear_quant_act.
 *   q        [M, K] int8, device, output: the codes of fp32(x * g).
 *   m        [M] fp32, device, output: the token scales with the norm factor
 *            folded in (the RMSNorm definition at the top of this file), ready
 *            for bitlinear_forward_q8 or a BL_DTYPE_I8 batch problem.
 * S_i must be finite in fp32 (|x| below about 1e19).
 */
BL_API bl_status bitlinear_rmsnorm_quant(const void* X, int x_dtype, int M, int K, const float* g, float eps_norm,
                                  float eps, int8_t* q, float* m, void* stream);

/*
 * BitLinear forward on RMSNorm(X): Y = dequant(quant(RMSNorm_g(X)) . T^T).
 * Arguments as bitlinear_forward plus g and eps_norm as
 * bitlinear_rmsnorm_quant; the workspace is sized with BL_OP_FORWARD.
 */
BL_API bl_status bitlinear_forward_rmsnorm(const void* X, int x_dtype, int M, int K, const float* g,
                                    float eps_norm, const uint8_t* packed, const float* s_w, int N,
                                    float eps, float* Y, int32_t* acc,
                                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * FFN block with SubLN: the input X is RMS-normalized (gain g_in) and
 * quantized once for up (and gate); h = ReLU^2(y_up), or fp32(ReLU^2(y_gate)
 * * y_up) when gate is given, is RMS-normalized (gain g_sub) and quantized
 * for down. gate and s_gate are both NULL (ungated) or both set; g_in, g_sub
 * NULL mean unit gains. Other arguments as bitlinear_ffn_gated; the workspace
 * is sized with BL_OP_FFN_GATED when gated, BL_OP_FFN otherwise.
 */
BL_API bl_status bitlinear_ffn_subln(const void* X, int x_dtype, int M, int D, const float* g_in,
                              const uint8_t* up, const float* s_up,
                              const uint8_t* gate, const float* s_gate, const float* g_sub,
                              const uint8_t* down, const float* s_down, int F, float eps_norm, float eps,
                              float* Y, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Decode packed codes back to ternary values (the inverse of the packing of
 * the report's 5.1): t [N, K] int8 in {-1, 0, 1} (code 3, never written by
 * bitlinear_pack, decodes to 2).
 */
BL_API bl_status bitlinear_unpack(const uint8_t* packed, int N, int K, int8_t* t, void* stream);

/*
 * Synchronizes `stream`, reads the sticky status word of `workspace`
 * (BL_OK or BL_ERR_TIMEOUT), and clears it.
 */
BL_API bl_status bitlinear_workspace_status(void* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BITLINEAR_H */
