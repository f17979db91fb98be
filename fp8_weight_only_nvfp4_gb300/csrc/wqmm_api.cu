// wqmm_api.cu -- the C-ABI (include/wqmm.h): argument checks, path
// selection and per-device setup.  Every check happens on the host before any
// CUDA call, so a bad argument never reaches the GPU.
//
// Path selection ("MatMulBlockQuantizedFp4Weight - CUDA Operator
// Documentation" §3, "MatMulBlockQuantizedFp8Weight - ..." §3, restated for
// sm_103a; the pages' SM120 branch and the dequantize -> scratch -> cuBLAS
// fallback are replaced):
//   empty output          -> return, no launch
//   K == 0                -> Y = bias (or 0)
//   M <= 8                -> decode GEMV
//   M <= 32, NVFP4 bs 16, K % 256 == 0 -> decode GEMV (up to four 8-row tiles;
//                            25..32 rows of a many-tile weight take the GEMM)
//   M > 8, GEMM-eligible  -> fused tcgen05 GEMM (weight decoded in the main loop;
//                            token tile 32 / 64 / 128 / 256 by M)
//   otherwise             -> decode GEMV, one launch per 8-row group
#include <mutex>
#include <cstring>

#include "../../include/wqmm.h"
#include "wqmm_device.cuh"
#include "wqmm_internal.h"

namespace wqmm {

namespace {

__device__ int g_error_word;

constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
int* g_err_ptr[kMaxDevices];
std::once_flag g_once[kMaxDevices];

void init_device(int dev) {
  DeviceInfo& d = g_info[dev];
  d.device = dev;
  cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev);
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) g_err_ptr[dev] = static_cast<int*>(p);
  cudaGetLastError();
}

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev < 0 || dev >= kMaxDevices) return -1;
  std::call_once(g_once[dev], init_device, dev);
  return dev;
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<EncodeFn>(fn);
  cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_n(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

constexpr int64_t kMaxDim = int64_t(1) << 31;

}  // namespace

const DeviceInfo& device_info() {
  const int dev = current_device();
  static DeviceInfo none;
  return dev < 0 ? none : g_info[dev];
}

int* device_error_word() {
  const int dev = current_device();
  return dev < 0 ? nullptr : g_err_ptr[dev];
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t inner_elems, uint64_t rows, uint64_t row_stride_bytes,
                    uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle,
                    CUtensorMapL2promotion promo) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return false;
  std::memset(map, 0, sizeof(*map));
  const cuuint64_t dims[2] = {inner_elems, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace wqmm

using namespace wqmm;

namespace {

int check_common(int64_t M, int64_t N, int64_t K, int bs, int dtype) {
  if (dtype != WQMM_FP16 && dtype != WQMM_BF16) return WQMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return WQMM_ERR_INVALID_ARG;
  if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return WQMM_ERR_UNSUPPORTED;
  if (bs < 1) return WQMM_ERR_INVALID_ARG;
  return WQMM_OK;
}

int matmul_common(GemvArgs& a, cudaStream_t st) {
  if (a.K == 0) return launch_fill_bias(a.bias, a.Y, a.M, a.N, a.dtype, st);
  if (a.M <= 8) return launch_gemv(a, st);
  // Up to 32 rows the decode GEMV shares each decoded weight across all of
  // them and stays bound by the weight stream.  With four 8-row activation
  // tiles (25..32 rows) and a weight of many row tiles the GEMM's two light
  // CTAs per SM are faster (N = 17408: 27.7 against 30.6 us; N = 5120: the
  // GEMV, 14.0 against 16.4 us).
  if (a.M <= 32 && gemv_tma_supports(a) &&
      !(a.M > 24 && gemm_supports(a) && gemm_prefers_light(a)))
    return launch_gemv(a, st);
  if (gemm_supports(a)) return launch_gemm(a, st);
  // Decode GEMV per group of rows (blockIdx.z covers up to 65535 groups).
  const int64_t rows_per_launch = int64_t(8) * 65535;
  const size_t esz = 2;
  for (int64_t m0 = 0; m0 < a.M; m0 += rows_per_launch) {
    GemvArgs b = a;
    b.M = std::min<int64_t>(rows_per_launch, a.M - m0);
    b.A = static_cast<const char*>(a.A) + m0 * a.K * esz;
    b.Y = static_cast<char*>(a.Y) + m0 * a.N * esz;
    const int r = launch_gemv(b, st);
    if (r != WQMM_OK) return r;
  }
  return WQMM_OK;
}

}  // namespace

extern "C" {

int fp4_weight_matmul(const void* A, const uint8_t* B_packed, const uint8_t* weight_scale,
                      const float* weight_scale_2, const void* bias, void* Y, int64_t M,
                      int64_t N, int64_t K, int block_size, int dtype, void* stream) {
  int r = check_common(M, N, K, block_size, dtype);
  if (r != WQMM_OK) return r;
  if (K % 2 != 0) return WQMM_ERR_INVALID_ARG;
  if (block_size % 16 != 0) return WQMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return WQMM_OK;
  if (!Y) return WQMM_ERR_INVALID_ARG;
  if (K > 0 && (!A || !B_packed || !weight_scale || !weight_scale_2)) return WQMM_ERR_INVALID_ARG;
  if (!aligned16(Y) || (A && !aligned16(A)) || (B_packed && !aligned16(B_packed)) ||
      (weight_scale && !aligned16(weight_scale)) ||
      (weight_scale_2 && !aligned_n(weight_scale_2, 4)) || (bias && !aligned_n(bias, 2)))
    return WQMM_ERR_MISALIGNED;
  if (current_device() < 0) return WQMM_ERR_CUDA;
  GemvArgs a{};
  a.kind = 0;
  a.A = A;
  a.B = B_packed;
  a.ws = weight_scale;
  a.gscale = weight_scale_2;
  a.fscale = nullptr;
  a.bias = bias;
  a.Y = Y;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bs = block_size;
  a.dtype = dtype;
  return matmul_common(a, static_cast<cudaStream_t>(stream));
}

int fp8_weight_matmul(const void* A, const uint8_t* B, const float* b_scale, const void* bias,
                      void* Y, int64_t M, int64_t N, int64_t K, int block_size, int dtype,
                      void* stream) {
  int r = check_common(M, N, K, block_size, dtype);
  if (r != WQMM_OK) return r;
  if (block_size % 16 != 0) return WQMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return WQMM_OK;
  if (!Y) return WQMM_ERR_INVALID_ARG;
  if (K > 0 && (!A || !B || !b_scale)) return WQMM_ERR_INVALID_ARG;
  if (!aligned16(Y) || (A && !aligned16(A)) || (B && !aligned16(B)) ||
      (b_scale && !aligned16(b_scale)) || (bias && !aligned_n(bias, 2)))
    return WQMM_ERR_MISALIGNED;
  if (current_device() < 0) return WQMM_ERR_CUDA;
  GemvArgs a{};
  a.kind = 1;
  a.A = A;
  a.B = B;
  a.ws = nullptr;
  a.gscale = nullptr;
  a.fscale = b_scale;
  a.bias = bias;
  a.Y = Y;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bs = block_size;
  a.dtype = dtype;
  return matmul_common(a, static_cast<cudaStream_t>(stream));
}

int fp8_weight_matmul_w8a8(const void* A, const float* a_scale, const uint8_t* B,
                           const float* b_scale, const void* bias, void* Y, int64_t M,
                           int64_t N, int64_t K, int block_size, int dtype, void* stream) {
  int r = check_common(M, N, K, block_size, dtype);
  if (r != WQMM_OK) return r;
  if (block_size % 16 != 0) return WQMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return WQMM_OK;
  if (!Y) return WQMM_ERR_INVALID_ARG;
  if (K > 0 && (!A || !B || !b_scale || !a_scale)) return WQMM_ERR_INVALID_ARG;
  if (!aligned16(Y) || (A && !aligned16(A)) || (B && !aligned16(B)) ||
      (b_scale && !aligned16(b_scale)) || (a_scale && !aligned_n(a_scale, 4)) ||
      (bias && !aligned_n(bias, 2)))
    return WQMM_ERR_MISALIGNED;
  if (current_device() < 0) return WQMM_ERR_CUDA;
  GemvArgs a{};
  a.kind = 1;
  a.A = A;
  a.B = B;
  a.fscale = b_scale;
  a.ascale = a_scale;
  a.bias = bias;
  a.Y = Y;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bs = block_size;
  a.dtype = dtype;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) return launch_fill_bias(bias, Y, M, N, dtype, st);
  // The activation is rounded where the GEMV stages it; the GEMM has no such
  // step, so every M runs the GEMV (per group of 8 rows above that).
  for (int64_t m0 = 0; m0 < M; m0 += 8) {
    GemvArgs b = a;
    b.M = std::min<int64_t>(8, M - m0);
    b.A = static_cast<const char*>(A) + m0 * K * 2;
    b.Y = static_cast<char*>(Y) + m0 * N * 2;
    const int rr = launch_gemv(b, st);
    if (rr != WQMM_OK) return rr;
  }
  return WQMM_OK;
}

int64_t fp8_w8a8_workspace_bytes(int64_t M, int64_t K) {
  if (M <= 8 || K <= 0 || M >= kMaxDim || K >= kMaxDim) return 0;
  return M * K * 2;
}

int fp8_weight_matmul_w8a8_ws(const void* A, const float* a_scale, const uint8_t* B,
                              const float* b_scale, const void* bias, void* Y, int64_t M,
                              int64_t N, int64_t K, int block_size, int dtype, void* workspace,
                              int64_t workspace_bytes, void* stream) {
  // Up to 8 rows the activation is rounded inside the decode GEMV's loads:
  // no workspace is used.
  if (M <= 8 || N == 0 || K == 0)
    return fp8_weight_matmul_w8a8(A, a_scale, B, b_scale, bias, Y, M, N, K, block_size, dtype,
                                  stream);
  int r = check_common(M, N, K, block_size, dtype);
  if (r != WQMM_OK) return r;
  if (block_size % 16 != 0) return WQMM_ERR_UNSUPPORTED;
  if (!Y || !A || !B || !b_scale || !a_scale) return WQMM_ERR_INVALID_ARG;
  const int64_t need = fp8_w8a8_workspace_bytes(M, K);
  if (!workspace || workspace_bytes < need) return WQMM_ERR_INVALID_ARG;
  // The workspace receives A_deq while A is read and before Y is written:
  // it may overlap neither.
  const uintptr_t w0 = reinterpret_cast<uintptr_t>(workspace), w1 = w0 + (uintptr_t)need;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(A), a1 = a0 + (uintptr_t)(M * K * 2);
  const uintptr_t y0 = reinterpret_cast<uintptr_t>(Y), y1 = y0 + (uintptr_t)(M * N * 2);
  if ((w0 < a1 && a0 < w1) || (w0 < y1 && y0 < w1)) return WQMM_ERR_INVALID_ARG;
  if (!aligned16(workspace) || !aligned16(Y) || !aligned16(A) || !aligned16(B) ||
      !aligned16(b_scale) || !aligned_n(a_scale, 4) || (bias && !aligned_n(bias, 2)))
    return WQMM_ERR_MISALIGNED;
  if (current_device() < 0) return WQMM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  r = launch_fp8_qdq_activation(A, a_scale, workspace, M * K, dtype, st);
  if (r != WQMM_OK) return r;
  GemvArgs a{};
  a.kind = 1;
  a.A = workspace;
  a.B = B;
  a.fscale = b_scale;
  a.bias = bias;
  a.Y = Y;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bs = block_size;
  a.dtype = dtype;
  return matmul_common(a, st);
}

int fp8_quantize_dequantize_activation(const void* A, const float* a_scale, void* out,
                                       int64_t count, int dtype, void* stream) {
  if (dtype != WQMM_FP16 && dtype != WQMM_BF16) return WQMM_ERR_INVALID_ARG;
  if (count < 0) return WQMM_ERR_INVALID_ARG;
  if (count == 0) return WQMM_OK;
  if (!A || !a_scale || !out) return WQMM_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(out) || !aligned_n(a_scale, 4)) return WQMM_ERR_MISALIGNED;
  if (current_device() < 0) return WQMM_ERR_CUDA;
  return launch_fp8_qdq_activation(A, a_scale, out, count, dtype,
                                   static_cast<cudaStream_t>(stream));
}

int fp4_quantize_activation(const void* A, uint8_t* A_packed, uint8_t* A_scale, int64_t M,
                            int64_t K, int dtype, void* stream) {
  if (dtype != WQMM_FP16 && dtype != WQMM_BF16) return WQMM_ERR_INVALID_ARG;
  if (M < 0 || K < 0 || K % 2 != 0) return WQMM_ERR_INVALID_ARG;
  if (M >= kMaxDim || K >= kMaxDim) return WQMM_ERR_UNSUPPORTED;
  if (M == 0 || K == 0) return WQMM_OK;
  if (!A || !A_packed || !A_scale) return WQMM_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(A_packed) || !aligned16(A_scale)) return WQMM_ERR_MISALIGNED;
  if (current_device() < 0) return WQMM_ERR_CUDA;
  return launch_nvfp4_quantize_activation(A, A_packed, A_scale, M, K, dtype,
                                          static_cast<cudaStream_t>(stream));
}

int fp4_quantize_dequantize_activation(const void* A, void* out, int64_t M, int64_t K, int dtype,
                                       void* stream) {
  if (dtype != WQMM_FP16 && dtype != WQMM_BF16) return WQMM_ERR_INVALID_ARG;
  if (M < 0 || K < 0 || K % 2 != 0) return WQMM_ERR_INVALID_ARG;
  if (M >= kMaxDim || K >= kMaxDim) return WQMM_ERR_UNSUPPORTED;
  if (M == 0 || K == 0) return WQMM_OK;
  if (!A || !out) return WQMM_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(out)) return WQMM_ERR_MISALIGNED;
  if (current_device() < 0) return WQMM_ERR_CUDA;
  return launch_nvfp4_qdq_activation(A, out, M, K, dtype, static_cast<cudaStream_t>(stream));
}

int fp4_fp4_matmul(const uint8_t* A_packed, const uint8_t* A_scale, const uint8_t* B_packed,
                   const uint8_t* weight_scale, const float* weight_scale_2, const void* bias,
                   void* Y, int64_t M, int64_t N, int64_t K, int dtype, void* stream) {
  int r = check_common(M, N, K, 16, dtype);
  if (r != WQMM_OK) return r;
  if (K % 2 != 0) return WQMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return WQMM_OK;
  if (!Y) return WQMM_ERR_INVALID_ARG;
  if (K > 0 && (!A_packed || !A_scale || !B_packed || !weight_scale || !weight_scale_2))
    return WQMM_ERR_INVALID_ARG;
  // Packed code rows (K / 2 bytes) that the tensor copies can address: K a
  // multiple of 32.
  if (K % 32 != 0) return WQMM_ERR_UNSUPPORTED;
  if (!aligned16(Y) || (K > 0 && (!aligned16(A_packed) || !aligned16(A_scale) ||
                                  !aligned16(B_packed) || !aligned16(weight_scale) ||
                                  !aligned_n(weight_scale_2, 4))) ||
      (bias && !aligned_n(bias, 2)))
    return WQMM_ERR_MISALIGNED;
  if (current_device() < 0) return WQMM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) return launch_fill_bias(bias, Y, M, N, dtype, st);
  F4F4Args a{};
  a.A = A_packed;
  a.A_scale = A_scale;
  a.B = B_packed;
  a.ws = weight_scale;
  a.gscale = weight_scale_2;
  a.bias = bias;
  a.Y = Y;
  a.M = M;
  a.N = N;
  a.K = K;
  a.dtype = dtype;
  return launch_gemm_f4f4(a, st);
}

int fp4_dequantize(const uint8_t* B_packed, const uint8_t* weight_scale,
                   const float* weight_scale_2, void* out, int64_t N, int64_t K, int block_size,
                   int dtype, void* stream) {
  int r = check_common(0, N, K, block_size, dtype);
  if (r != WQMM_OK) return r;
  if (K % 2 != 0) return WQMM_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return WQMM_OK;
  if (!B_packed || !weight_scale || !weight_scale_2 || !out) return WQMM_ERR_INVALID_ARG;
  if (!aligned16(B_packed) || !aligned16(weight_scale) || !aligned16(out) ||
      !aligned_n(weight_scale_2, 4))
    return WQMM_ERR_MISALIGNED;
  if (current_device() < 0) return WQMM_ERR_CUDA;
  return launch_fp4_dequant(B_packed, weight_scale, weight_scale_2, out, N, K, block_size, dtype,
                            static_cast<cudaStream_t>(stream));
}

int fp8_dequantize(const uint8_t* B, const float* b_scale, void* out, int64_t N, int64_t K,
                   int block_size, int dtype, void* stream) {
  int r = check_common(0, N, K, block_size, dtype);
  if (r != WQMM_OK) return r;
  if (N == 0 || K == 0) return WQMM_OK;
  if (!B || !b_scale || !out) return WQMM_ERR_INVALID_ARG;
  if (!aligned16(B) || !aligned16(b_scale) || !aligned16(out)) return WQMM_ERR_MISALIGNED;
  if (current_device() < 0) return WQMM_ERR_CUDA;
  return launch_fp8_dequant(B, b_scale, out, N, K, block_size, dtype,
                            static_cast<cudaStream_t>(stream));
}

const char* wqmm_status_string(int status) {
  switch (status) {
    case WQMM_OK: return "WQMM_OK";
    case WQMM_ERR_INVALID_ARG: return "WQMM_ERR_INVALID_ARG";
    case WQMM_ERR_UNSUPPORTED: return "WQMM_ERR_UNSUPPORTED";
    case WQMM_ERR_MISALIGNED: return "WQMM_ERR_MISALIGNED";
    case WQMM_ERR_CUDA: return "WQMM_ERR_CUDA";
    case WQMM_ERR_TIMEOUT: return "WQMM_ERR_TIMEOUT";
    default: return "WQMM_ERR_UNKNOWN";
  }
}

int wqmm_device_status(void* stream) {
  const int dev = current_device();
  if (dev < 0) return WQMM_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return WQMM_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return WQMM_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
  }
  return v;
}

// One warp waits, through the same bounded-wait helper the kernels use, on an
// mbarrier that nothing arrives on: after the wait limit it records
// WQMM_ERR_TIMEOUT in the error word and returns.
__global__ void selftest_wait_kernel(int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  mbar_wait(&bar, 0, err);  // phase 0 never completes
}

int wqmm_selftest_wait_timeout(void* stream) {
  if (current_device() < 0) return WQMM_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(device_error_word());
  return cudaGetLastError() == cudaSuccess ? WQMM_OK : WQMM_ERR_CUDA;
}

int wqmm_version(void) { return 100; }

}  // extern "C"
