// bitlinear_forward_noalloc: the BitLinear forward for callers that cannot
// hand the library a workspace.
//
// Some callers have no way to obtain device scratch memory at call time: an
// inference runtime that fixes its whole device-memory plan at start-up and
// forbids allocation afterwards, a plugin whose host framework owns every
// device allocation and exposes no allocator, or code that must not call
// into an allocator on its hot path. For them this entry point takes only the
// inputs and outputs and runs the same launch sequence as bitlinear_forward,
// with its scratch in a fixed-size array in device global memory that the
// library defines (every GPU that loads the library holds it until the
// process exits). It calls no cudaMalloc, cudaFree or other allocating routine.
#include <atomic>

#include "common.cuh"

namespace {

constexpr size_t kStaticScratchBytes = BL_STATIC_SCRATCH_BYTES;

// Shared by every call on a device; the first 256 bytes are the status header.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch per device, looked up once. In host
// code the array's name is only a host-side stand-in, so the kernels must be
// given this address, never &g_static_scratch.
std::atomic<void*> g_scratch_addr[64];

bl_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BL_ERR_CUDA;
  if (dev < 0 || dev >= 64) return BL_ERR_UNSUPPORTED;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return BL_ERR_CUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return BL_OK;
}

}  // namespace

extern "C" bl_status bitlinear_forward_noalloc(const void* X, int x_dtype, int M, int K, const uint8_t* packed,
                                               const float* s_w, int N, float eps, float* Y, int32_t* acc,
                                               void* stream) {
  if (M < 0 || N < 0 || K <= 0) return BL_ERR_SHAPE;
  if (M == 0 || N == 0) return BL_OK;
  const size_t need = bitlinear_workspace_bytes(BL_OP_FORWARD, M, N, K);
  if (need == 0) return BL_ERR_SHAPE;
  if (need > kStaticScratchBytes) return BL_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (bl_status s = scratch_address(&scratch); s != BL_OK) return s;
  return bitlinear_forward(X, x_dtype, M, K, packed, s_w, N, eps, Y, acc, scratch, kStaticScratchBytes, stream);
}
