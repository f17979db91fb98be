// wqmm_noalloc.cu -- fp8_weight_matmul_w8a8_noalloc: the W8A8 matmul for
// more than 8 rows (activation quantize-dequantize into an [M, K] scratch,
// then the FP8 weight-only GEMM on it) with the scratch taken from a fixed
// array that the library itself owns, for callers that are not allowed to
// allocate device memory.  Everything else is fp8_weight_matmul_w8a8_ws.
//
// The scratch is a module-scope __device__ array: the CUDA runtime reserves
// it on every GPU where this library's code is loaded and keeps it there
// until the process exits.  Its device address is looked up once per device,
// on the first call made with that device current.
//
// Nothing in the scratch has to start at zero: each call first writes the
// 2 * M * K bytes of A_deq and only then runs the GEMM that reads them, both
// on the caller's stream.  All calls on one device share the one array, so
// calls that may run at the same time (different streams without an order
// between them, or several host threads) race on it.
#include <mutex>

#include "../../include/wqmm.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[WQMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch[kMaxDevices];
int g_scratch_status[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

// Runs once per device, with that device current.
void lookup_scratch(int dev) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e == cudaSuccess && p != nullptr) {
    g_scratch[dev] = p;
    g_scratch_status[dev] = WQMM_OK;
  } else {
    cudaGetLastError();
    g_scratch_status[dev] = WQMM_ERR_CUDA;
  }
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

}  // namespace

extern "C" int fp8_weight_matmul_w8a8_noalloc(const void* A, const float* a_scale,
                                              const uint8_t* B, const float* b_scale,
                                              const void* bias, void* Y, int64_t M, int64_t N,
                                              int64_t K, int block_size, int dtype,
                                              void* stream) {
  if (dtype != WQMM_FP16 && dtype != WQMM_BF16) return WQMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || block_size < 1) return WQMM_ERR_INVALID_ARG;
  // Up to 8 rows, an empty output or K == 0 need no scratch.
  if (M <= 8 || N == 0 || K == 0)
    return fp8_weight_matmul_w8a8(A, a_scale, B, b_scale, bias, Y, M, N, K, block_size, dtype,
                                  stream);
  // The host-side checks come before the first CUDA call, as everywhere in
  // the library; the size limit is this entry point's own.
  const int64_t need = fp8_w8a8_workspace_bytes(M, K);
  if (need <= 0 || need > (int64_t)WQMM_NOALLOC_SCRATCH_BYTES) return WQMM_ERR_UNSUPPORTED;
  if (block_size % 16 != 0) return WQMM_ERR_UNSUPPORTED;
  if (!Y || !A || !B || !b_scale || !a_scale) return WQMM_ERR_INVALID_ARG;
  if (!aligned(Y, 16) || !aligned(A, 16) || !aligned(B, 16) || !aligned(b_scale, 16) ||
      !aligned(a_scale, 4) || (bias && !aligned(bias, 2)))
    return WQMM_ERR_MISALIGNED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WQMM_ERR_CUDA;
  std::call_once(g_scratch_once[dev], lookup_scratch, dev);
  if (g_scratch_status[dev] != WQMM_OK) return g_scratch_status[dev];
  return fp8_weight_matmul_w8a8_ws(A, a_scale, B, b_scale, bias, Y, M, N, K, block_size, dtype,
                                   g_scratch[dev], (int64_t)WQMM_NOALLOC_SCRATCH_BYTES, stream);
}
