// wqmm_internal.h -- host-side declarations shared by the library's
// translation units (launchers called by the C-ABI in wqmm_api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace wqmm {

enum Status : int {
  kOk = 0,
  kInvalidArg = 1,
  kUnsupported = 2,
  kMisaligned = 3,
  kCuda = 4,
  kTimeout = 5,
};

// Per-device facts, queried once per device.
struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0;
  int cc_minor = 0;
  int max_smem_optin = 0;
  int l2_bytes = 0;
};

// Returns the info for the current device (cached per device).
const DeviceInfo& device_info();

// Device address of the error word of the current device (see
// wqmm_device_status in wqmm.h).  Kernels with bounded waits receive it.
int* device_error_word();

// cuTensorMapEncodeTiled through the runtime's driver entry point.
// Returns false if the entry point is unavailable or the encode fails.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t inner_elems, uint64_t rows, uint64_t row_stride_bytes,
                    uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle,
                    CUtensorMapL2promotion promo);

// ---- dequantize (wqmm_dequant.cu) ----
int launch_fp4_dequant(const uint8_t* Bp, const uint8_t* ws, const float* ws2, void* out,
                       int64_t N, int64_t K, int bs, int dtype, cudaStream_t st);
int launch_fp8_dequant(const uint8_t* B, const float* bsc, void* out, int64_t N, int64_t K,
                       int bs, int dtype, cudaStream_t st);
// Y[m, n] = bias[n] (or 0) for every m: the K == 0 case of the matmul.
int launch_fill_bias(const void* bias, void* Y, int64_t M, int64_t N, int dtype,
                     cudaStream_t st);

// ---- decode GEMV, M rows in groups of 8 (wqmm_gemv.cu) ----
// kind: 0 = NVFP4 weight (ws = E4M3 block scales, gscale = weight_scale_2),
//       1 = FP8 weight (fscale = float block scales).
struct GemvArgs {
  int kind;
  const void* A;
  const uint8_t* B;       // packed NVFP4 [N, K/2] or FP8 [N, K]
  const uint8_t* ws;      // NVFP4 block scales [N, S]
  const float* gscale;    // NVFP4 weight_scale_2 (device)
  const float* fscale;    // FP8 block scales [N, S]
  const float* ascale;    // FP8 W8A8: activation scale (device), or nullptr
  const void* bias;
  void* Y;
  int64_t M, N, K;
  int bs;
  int dtype;
};
int launch_gemv(const GemvArgs& a, cudaStream_t st);
// The TMA decode GEMV also takes 8 < M <= 32 (NVFP4, bs 16, K % 256 == 0).
bool gemv_tma_supports(const GemvArgs& a);

// W8A8 activation quantize-dequantize over n elements (wqmm_gemv.cu).
int launch_fp8_qdq_activation(const void* A, const float* a_scale, void* out, int64_t n,
                              int dtype, cudaStream_t st);

// ---- NVFP4 activation quantization (wqmm_actq.cu) ----
// codes [M, K/2] (two per byte, even k low), scales [M, ceil(K/16)] E4M3.
int launch_nvfp4_quantize_activation(const void* A, uint8_t* codes, uint8_t* scales, int64_t M,
                                     int64_t K, int dtype, cudaStream_t st);
// out [M, K] = e2m1(code) * e4m3(scale) in the activation type (exact).
int launch_nvfp4_qdq_activation(const void* A, void* out, int64_t M, int64_t K, int dtype,
                                cudaStream_t st);

// ---- fused tcgen05 GEMM for large M (wqmm_gemm.cu) ----
// Returns kUnsupported if the shape cannot take this path.
int launch_gemm(const GemvArgs& a, cudaStream_t st);
bool gemm_supports(const GemvArgs& a);
// The GEMM would run its narrow tile as two light CTAs per SM (the tiles fill
// at least half of the SMs).
bool gemm_prefers_light(const GemvArgs& a);

// ---- NVFP4 x NVFP4 block-scaled tcgen05 GEMM (wqmm_gemm_f4f4.cu) ----
struct F4F4Args {
  const uint8_t* A;        // activation codes [M, K/2]
  const uint8_t* A_scale;  // activation block scales [M, K/16], E4M3
  const uint8_t* B;        // weight codes [N, K/2]
  const uint8_t* ws;       // weight block scales [N, K/16], E4M3
  const float* gscale;     // weight_scale_2 (device)
  const void* bias;
  void* Y;
  int64_t M, N, K;
  int dtype;
};
// Returns kUnsupported if the device or the shape cannot take this path
// (K % 32 != 0).
int launch_gemm_f4f4(const F4F4Args& a, cudaStream_t st);
bool gemm_f4f4_supports(const F4F4Args& a);

}  // namespace wqmm
