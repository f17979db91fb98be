/*
 * wqmm.h -- block-quantized weight-only matrix multiplication for NVIDIA
 * GB300 (sm_103a): NVFP4 and FP8 (E4M3) weights, FP16/BF16 activations.
 *
 *     Y[M, N] = A[M, K] * dequant(B)[N, K]^T (+ bias[N])
 *
 * Sources (web pages, by title and section):
 *   [FP4]  "MatMulBlockQuantizedFp4Weight - CUDA Operator Documentation"
 *   [FP8]  "MatMulBlockQuantizedFp8Weight - CUDA Operator Documentation"
 *   [BLOG] "ONNX Runtime #32128 -- Why Dequantizing 4-Bit Weights Became the
 *          Most Expensive Kernel in H200 Prefill"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer (global memory of the current
 *    device), row-major and contiguous.  The caller owns every buffer.  The
 *    library allocates no device memory and keeps no per-call state (its
 *    only device data are an error word and the fixed scratch array of
 *    fp8_weight_matmul_w8a8_noalloc, both reserved when its code loads).
 *  - `dtype` selects the activation type used for A, bias, Y and dequantized
 *    outputs: WQMM_FP16 (IEEE binary16) or WQMM_BF16 (bfloat16).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call is asynchronous on that stream; the return value
 *    reports argument checks and launch errors only.
 *  - Base pointers must be 16-byte aligned (WQMM_ERR_MISALIGNED otherwise).
 *  - Empty outputs (M == 0 or N == 0) return WQMM_OK without launching
 *    ([FP4] §3 and [FP8] §3: the dispatch chain returns on empty output).
 *  - K == 0 with a non-empty output writes Y = bias (or zeros).
 *  - No entry point traps or aborts.  Waits inside the kernels are bounded;
 *    a wait that runs out records WQMM_ERR_TIMEOUT in a device word that
 *    wqmm_device_status() reports.  That call then leaves Y untouched,
 *    except on the persistent paths (the prefill GEMM over enough 256-token
 *    tiles to fill the GPU, and fp4_fp4_matmul), which store each output
 *    tile as soon as it is complete: there the tiles finished before the
 *    wait ran out hold their results and the rest of Y is left untouched.
 *  - Weights are parameters.  The decode GEMVs (M <= 32) start reading the
 *    weight -- B_packed / B, weight_scale / b_scale and weight_scale_2 --
 *    before the kernel launched just before them on `stream` has finished
 *    (programmatic dependent launch), so the weight must not be written by
 *    that immediately preceding kernel.  Every other input (A, bias,
 *    a_scale) is read only after all earlier work on the stream has
 *    completed; a bias may be the previous call's output.
 *  - Thread safety: calls may be issued from several host threads at once.
 *    Per-device setup (kernel attributes, driver entry points) runs once.
 */
#ifndef WQMM_H_
#define WQMM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WQMM_FP16 = 0,
  WQMM_BF16 = 1
} wqmm_dtype;

typedef enum {
  WQMM_OK = 0,
  WQMM_ERR_INVALID_ARG = 1,  /* null pointer, negative size, odd K (FP4), block_size < 1 */
  WQMM_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement */
  WQMM_ERR_MISALIGNED = 3,   /* a base pointer is not 16-byte aligned */
  WQMM_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  WQMM_ERR_TIMEOUT = 5       /* a bounded device-side wait ran out */
} wqmm_status;

/*
 * fp4_weight_matmul -- Y = A * dequant(B)^T (+ bias) with an NVFP4 weight.
 * [FP4] §1 Operator Schema, §2 Weight Format:
 *     B_dequant[n, k] = e2m1(B[n, k]) * e4m3(weight_scale[n, k / block_size])
 *                       * weight_scale_2
 *
 *   A              [M, K] activations (dtype).
 *   B_packed       [N, K/2] uint8: two E2M1 codes per byte, the LOW nibble
 *                  holds the even k, the HIGH nibble the odd k.
 *   weight_scale   [N, S] uint8 raw E4M3FN bytes, S = ceil(K / block_size);
 *                  element k uses column floor(k / block_size).
 *   weight_scale_2 one float32 global scale, read on the device.
 *   bias           [N] (dtype) or NULL.
 *   Y              [M, N] output (dtype), written with one round-to-nearest-
 *                  even from the float32 value  acc * weight_scale_2 + bias.
 *   M, N, K        sizes; M is the product of A's leading dimensions.
 *   block_size     K elements per scale; must be a positive multiple of 16.
 *
 * Paths: M <= 8 runs the decode GEMV (each weight byte read once, the decode
 * shared by all M rows), and so does M <= 32 when block_size == 16 and
 * K % 256 == 0 (up to four 8-row activation tiles per decoded weight
 * fragment), except 25..32 rows of a weight with many 128-row tiles; larger M
 * with K % 32 == 0 runs the fused tcgen05 GEMM (the weight is dequantized
 * inside the main loop, no [N, K] scratch; a 32/64/128/256-token tile by M);
 * other shapes run the GEMV once per 8-row group of A.  All paths meet the
 * accuracy bound below; which one runs changes only the summation order.
 * Errors: odd K or block_size < 1 -> INVALID_ARG; block_size % 16 != 0 ->
 * UNSUPPORTED; any size < 0 -> INVALID_ARG.
 * Accuracy: |Y - Y_exact| <= 8e-3 * sum_k |A * B_dq| + 1e-3 (BF16) and
 * <= 2e-3 * sum_k |A * B_dq| + 1e-4 (FP16), Y_exact in exact arithmetic.
 */
int fp4_weight_matmul(const void* A, const uint8_t* B_packed,
                      const uint8_t* weight_scale, const float* weight_scale_2,
                      const void* bias, void* Y, int64_t M, int64_t N, int64_t K,
                      int block_size, int dtype, void* stream);

/*
 * fp8_weight_matmul -- Y = A * dequant(B)^T (+ bias) with an FP8 E4M3 weight.
 * [FP8] §2 Tensor and Scale Format:
 *     B_dequant[n, k] = fp8_e4m3(B[n, k]) * b_scale[n, k / block_size]
 *
 *   A        [M, K] activations (dtype).
 *   B        [N, K] uint8 E4M3FN bytes.
 *   b_scale  [N, S] float32, S = ceil(K / block_size); a partial final block
 *            uses the last column.
 *   bias     [N] (dtype) or NULL.
 *   Y        [M, N] (dtype).
 *   block_size must be a positive multiple of 16.
 * Paths as for fp4_weight_matmul (the GEMM needs K % 16 == 0).
 * Accuracy bound as for fp4_weight_matmul, for any finite b_scale: with FP16
 * activations no path rounds e4m3 * b_scale into an FP16 operand, which
 * would overflow above |b_scale| ~ 146 (the GEMM divides each weight row's
 * block scales by a power of two and multiplies it back in FP32; the GEMV
 * applies blocks of 128 k or more in FP32 after the MMAs and takes TF32
 * operands for smaller blocks).
 */
int fp8_weight_matmul(const void* A, const uint8_t* B, const float* b_scale,
                      const void* bias, void* Y, int64_t M, int64_t N, int64_t K,
                      int block_size, int dtype, void* stream);

/*
 * fp8_weight_matmul_w8a8 -- the optional W8A8 activation path of the FP8
 * operator: Y = A_deq * dequant(B)^T (+ bias) with
 * [FP8] §6 Optional W8A8 Activation Path:
 *     A_deq = fp8_e4m3(A / a_scale) * a_scale
 * computed inside the GEMV's activation loads (no [M, K] scratch).
 *
 *   a_scale  device pointer to one float32 (the static activation scale).
 *   Other arguments, layouts and errors as for fp8_weight_matmul; a NULL
 *   a_scale (with a non-empty output) is INVALID_ARG.
 * Per element: one float32 division (IEEE), E4M3FN by round-to-nearest-even
 * saturating at +-448 (NaN stays NaN), one float32 multiplication by a_scale,
 * one RNE to dtype; exactly fp8_quantize_dequantize_activation.
 * Paths: the decode GEMV for every M (per 8-row group above 8 rows, each
 * group streaming the whole weight); for prefill-sized M the cheaper route
 * is fp8_weight_matmul_w8a8_ws below (a caller-owned [M, K] workspace),
 * which gives the same A_deq bit for bit.
 * Accuracy: the bound of fp8_weight_matmul with A_deq in place of A.
 */
int fp8_weight_matmul_w8a8(const void* A, const float* a_scale, const uint8_t* B,
                           const float* b_scale, const void* bias, void* Y, int64_t M,
                           int64_t N, int64_t K, int block_size, int dtype, void* stream);

/*
 * fp8_weight_matmul_w8a8_ws -- the W8A8 path of fp8_weight_matmul_w8a8 for
 * prefill-sized M, with a caller-owned workspace:
 * [FP8] §6 Optional W8A8 Activation Path (A_deq = fp8_e4m3(A / a_scale) *
 * a_scale, then the FP8 weight-only product on A_deq).
 * For M <= 8 (or an empty output, or K == 0) it is fp8_weight_matmul_w8a8
 * itself and the workspace is not used.  Above 8 rows it writes A_deq once
 * into `workspace` ([M, K] in dtype, as fp8_quantize_dequantize_activation)
 * and runs fp8_weight_matmul on it (the fused tcgen05 GEMM where its
 * alignment holds), so each weight byte is read once per 256-token tile
 * instead of once per 8 rows; the result is bit-identical to those two calls.
 *   workspace        device pointer, 16-byte aligned, at least
 *                    fp8_w8a8_workspace_bytes(M, K) bytes, owned by the
 *                    caller; it may overlap neither A nor Y and is
 *                    overwritten (contents undefined afterwards).
 *   workspace_bytes  its size in bytes.
 * Other arguments, layouts and errors as for fp8_weight_matmul_w8a8; a NULL
 * or too small workspace (M > 8) or one overlapping A or Y -> INVALID_ARG;
 * a workspace not 16-byte aligned -> MISALIGNED.  Checks run on the host
 * before any launch; the two launches are asynchronous on `stream`.
 */
int fp8_weight_matmul_w8a8_ws(const void* A, const float* a_scale, const uint8_t* B,
                              const float* b_scale, const void* bias, void* Y, int64_t M,
                              int64_t N, int64_t K, int block_size, int dtype, void* workspace,
                              int64_t workspace_bytes, void* stream);

/*
 * fp8_w8a8_workspace_bytes -- workspace size fp8_weight_matmul_w8a8_ws needs
 * for an [M, K] activation: 2 * M * K bytes when M > 8, else 0 (also 0 for
 * K <= 0 or sizes beyond the library's 2^31 limit).  Host-only, no CUDA call.
 */
int64_t fp8_w8a8_workspace_bytes(int64_t M, int64_t K);

/* Size of the scratch array that fp8_weight_matmul_w8a8_noalloc draws on. */
#define WQMM_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * fp8_weight_matmul_w8a8_noalloc -- fp8_weight_matmul_w8a8_ws for callers
 * that may not allocate device memory.  The source pages have no counterpart
 * to this entry point; it computes exactly what fp8_weight_matmul_w8a8_ws
 * computes ([FP8] §6 Optional W8A8 Activation Path), bit for bit.
 *
 * Who needs it: code that runs where a device allocation is not allowed or
 * not affordable -- inference hosts that hand out all device memory through
 * their own pool and forbid any other allocation, serving loops that must not
 * call cudaMalloc after start-up because it can stall the device and every
 * other stream on it, plugins whose host process owns the memory budget.
 * Such a caller cannot provide (or cannot allocate) the [M, K] workspace of
 * fp8_weight_matmul_w8a8_ws.  This call allocates nothing: the workspace is a
 * fixed array of WQMM_NOALLOC_SCRATCH_BYTES (16 MiB) inside the library,
 * which the CUDA runtime reserves on every GPU where the library's code is
 * loaded and which stays reserved until the process exits.
 *
 * Arguments, layouts and errors as for fp8_weight_matmul_w8a8_ws without
 * `workspace` / `workspace_bytes`.  Limit: 2 * M * K <= 16 MiB for M > 8
 * (e.g. M <= 1638 at K = 5120); a larger problem -> WQMM_ERR_UNSUPPORTED,
 * detected on the host before any CUDA call.  M <= 8 (or an empty output,
 * or K == 0) uses no scratch and has no such limit.
 *
 * Set-up: the first call on a device with M > 8 looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; a failure there
 * -> WQMM_ERR_CUDA.  Make that first call before any stream capture begins.
 * Nothing in the array needs to start at zero: each call writes the values
 * it reads.  Concurrency: one array per device is shared by all calls, so
 * calls that may overlap in time on the same device (unordered streams, or
 * several host threads) race on it and give undefined results; order them
 * on one stream or with events.
 */
int fp8_weight_matmul_w8a8_noalloc(const void* A, const float* a_scale, const uint8_t* B,
                                   const float* b_scale, const void* bias, void* Y, int64_t M,
                                   int64_t N, int64_t K, int block_size, int dtype, void* stream);

/*
 * fp8_quantize_dequantize_activation -- out = A_deq as defined above, for
 * `count` activation elements (any shape, contiguous).  Bit-exact contract.
 *   A, out   count values of dtype (16-byte aligned, may not overlap partly).
 *   a_scale  device pointer to one float32.
 * Errors: count < 0 or a NULL pointer with count > 0 -> INVALID_ARG.
 */
int fp8_quantize_dequantize_activation(const void* A, const float* a_scale, void* out,
                                       int64_t count, int dtype, void* stream);

/*
 * fp4_quantize_activation -- NVFP4 quantization of an activation, the first
 * step of the native FP4 x FP4 path of [FP4] §6: the activation takes the
 * weight's format (two E2M1 codes per byte, one E4M3 scale per 16
 * elements).  The page gives no formula; per 16-element block of each row
 * of A:
 *     scale = E4M3(fp32(amax / 6))          RNE, saturating at 448
 *     code  = E2M1(fp32(a / e4m3(scale)))   RNE, ties to the even code,
 *                                           saturating at 6, sign of a kept;
 *                                           a zero scale gives +-0
 * (no activation global scale: the page names none).  Bit-exact contract.
 *   A         [M, K] dtype, row-major (16-byte aligned); finite values.
 *   A_packed  [M, K/2] uint8: two codes per byte, the even k in the low
 *             nibble (the weight layout of [FP4] §2).
 *   A_scale   [M, ceil(K/16)] uint8 E4M3FN; a partial last block (K % 16 != 0)
 *             takes its amax over the elements it has.
 * Errors: K odd, M or K < 0, or a NULL pointer with M*K > 0 -> INVALID_ARG;
 * a base pointer not 16-byte aligned -> MISALIGNED; M*K == 0 -> OK, no launch.
 */
int fp4_quantize_activation(const void* A, uint8_t* A_packed, uint8_t* A_scale, int64_t M,
                            int64_t K, int dtype, void* stream);

/*
 * fp4_quantize_dequantize_activation -- out = e2m1(code) * e4m3(scale) of
 * fp4_quantize_activation, element by element in dtype ([M, K], 16-byte
 * aligned).  The value has at most 6 significant bits in [2^-10, 2688] (or
 * is zero), so it is exact in FP16 and BF16, and
 *     fp4_weight_matmul(fp4_quantize_dequantize_activation(A), B, ...)
 * computes the activation-and-weight FP4 product of [FP4] §6 (exact
 * products, FP32 accumulation) with the weight-only kernels.  Errors as for
 * fp4_quantize_activation.
 */
int fp4_quantize_dequantize_activation(const void* A, void* out, int64_t M, int64_t K, int dtype,
                                       void* stream);

/*
 * fp4_fp4_matmul -- Y = A_q * B_q^T (+ bias) with BOTH operands in NVFP4,
 * steps 2-3 of the native FP4 x FP4 path of [FP4] §6 (step 1 is
 * fp4_quantize_activation):
 *     Y[m, n] = weight_scale_2 * sum_k e2m1(A_packed[m, k]) e4m3(A_scale[m, k/16])
 *                                    * e2m1(B_packed[n, k]) e4m3(weight_scale[n, k/16])
 *               (+ bias[n]), one RNE to dtype.
 * Runs on the block-scaled tensor-core MMA (tcgen05.mma.kind::mxf4nvf4):
 * products are exact, sums are FP32.
 *   A_packed      [M, K/2] uint8, two E2M1 codes per byte (even k low), as
 *                 written by fp4_quantize_activation.
 *   A_scale       [M, K/16] uint8 E4M3 block scales of A.
 *   B_packed, weight_scale, weight_scale_2, bias   the NVFP4 weight of
 *                 fp4_weight_matmul with block_size 16.
 *   Y             [M, N] dtype (dtype selects only the output and bias type).
 * Block scales are read as unsigned E4M3 (the tensor core's scale type): the
 * sign bit must be clear and 0x7F (NaN) is not allowed; the quantizer's
 * scales always qualify.  K must be a multiple of 32 (WQMM_ERR_UNSUPPORTED
 * otherwise; a multiple of 256 takes the fastest path); K == 0 writes
 * Y = bias (or 0).
 * Errors: odd K, a size < 0 or a NULL pointer -> INVALID_ARG; a pointer not
 * 16-byte aligned (weight_scale_2 4, bias 2) -> MISALIGNED.
 * Accuracy: the bound of fp4_weight_matmul with sum_k |A_q * B_dq| in place
 * of sum_k |A * B_dq| (A_q = e2m1 * e4m3 of the codes).
 */
int fp4_fp4_matmul(const uint8_t* A_packed, const uint8_t* A_scale, const uint8_t* B_packed,
                   const uint8_t* weight_scale, const float* weight_scale_2, const void* bias,
                   void* Y, int64_t M, int64_t N, int64_t K, int dtype, void* stream);

/*
 * fp4_dequantize -- expand an NVFP4 weight to the activation type.
 * [FP4] §2 formula, §5 step 1; [BLOG] vectorised dequant.
 *   out[n, k] = RNE_dtype( fp32( fp32(e2m1 * e4m3) * weight_scale_2 ) )
 * The first product is exact in fp32; the multiply by weight_scale_2 rounds
 * once (fp32, nearest even); the conversion to dtype rounds once more.  The
 * result is bit-exact to that definition.
 *   out  [N, K] (dtype).  Any block_size >= 1 (odd included) and any even K.
 */
int fp4_dequantize(const uint8_t* B_packed, const uint8_t* weight_scale,
                   const float* weight_scale_2, void* out, int64_t N, int64_t K,
                   int block_size, int dtype, void* stream);

/*
 * fp8_dequantize -- expand an FP8 weight to the activation type.
 * [FP8] §2 formula, §5 step 1.
 *   out[n, k] = RNE_dtype( fp32(e4m3(B[n, k]) * b_scale[n, k / block_size]) )
 * Bit-exact to that definition.  Any K >= 0 and block_size >= 1.
 */
int fp8_dequantize(const uint8_t* B, const float* b_scale, void* out,
                   int64_t N, int64_t K, int block_size, int dtype, void* stream);

/* Human-readable name of a wqmm_status value (static string). */
const char* wqmm_status_string(int status);

/*
 * wqmm_device_status -- synchronise `stream`, then return and clear the
 * device-side error word (WQMM_OK if no bounded wait ran out since the last
 * call), or WQMM_ERR_CUDA if the synchronisation itself failed.
 */
int wqmm_device_status(void* stream);

/*
 * wqmm_selftest_wait_timeout -- diagnostic for the bounded waits: launches one
 * warp on `stream` that waits, through the same bounded-wait helper as the
 * kernels, on a barrier that nothing completes.  After the wait limit (2 s)
 * it records WQMM_ERR_TIMEOUT in the device error word and returns; the CUDA
 * context stays usable.  Returns WQMM_OK once launched (WQMM_ERR_CUDA if the
 * launch fails); read the outcome with wqmm_device_status.
 */
int wqmm_selftest_wait_timeout(void* stream);

/* Version of this interface (major * 100 + minor). */
int wqmm_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* WQMM_H_ */
