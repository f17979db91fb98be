// wqmm_dequant.cu -- standalone dequantization of NVFP4 and FP8 weights to
// FP16/BF16, and the bias fill used when K == 0.
//
// Definition ("MatMulBlockQuantizedFp4Weight - CUDA Operator Documentation"
// §2 and §5 step 1):
//   out[n, k] = RNE_act( fp32( fp32(e2m1 * e4m3(ws[n, k / bs])) * ws2 ) )
// FP8 ("MatMulBlockQuantizedFp8Weight - CUDA Operator Documentation" §2, §5):
//   out[n, k] = RNE_act( fp32(e4m3(B[n, k]) * b_scale[n, k / bs]) )
//
// Design for an HBM-bound stream (the vectorised dequant of "ONNX Runtime
// #32128 ...", sections on the Vec8 kernel, restated for sm_103a):
//  * When block_size is a multiple of 8 and divides K, [N, K] is one flat
//    array of 8-code units whose scale index is unit / (bs / 8) (a shift for
//    power-of-two block sizes): no row/column division at all.
//  * Each thread handles U units; unit j of lane l sits at warp_base + 32 j + l,
//    so every load instruction reads 128 contiguous bytes per warp (NVFP4) and
//    every store instruction writes 512 contiguous bytes per warp.
//  * All U loads are issued before any conversion (memory-level parallelism).
//  * The output is written with streaming (evict-first) stores: it is written
//    once and, for the weights the pages dequantize, larger than L2.
//  * weight_scale_2 is read once per thread into a register.
//  * E2M1 and E4M3 decode with the hardware cvt instructions (exact); the two
//    multiplies use __fmul_rn so that no FMA contraction changes the rounding.
//  * Other shapes (odd block sizes, block sizes that do not divide K) take a
//    row kernel with per-element scale tracking and masked tails.
#include "wqmm_device.cuh"

namespace wqmm {

namespace {

constexpr int kThreads = 256;

template <int DT, int U>
__global__ void __launch_bounds__(kThreads)
    fp4_dequant_flat(const uint32_t* __restrict__ Bw, const uint8_t* __restrict__ ws,
                     const float* __restrict__ ws2p, uint4* __restrict__ out, int64_t units,
                     int upb_shift, int64_t upb) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t base = ((int64_t)blockIdx.x * (kThreads / 32) + warp) * (32 * U);
  const float ws2 = __ldg(ws2p);

  uint32_t w[U];
  uint32_t sb[U];
#pragma unroll
  for (int j = 0; j < U; ++j) {
    const int64_t u = base + 32 * j + lane;
    w[j] = 0;
    sb[j] = 0;
    if (u < units) {
      w[j] = ldg_stream_u32(Bw + u);
      const int64_t s = upb_shift >= 0 ? (u >> upb_shift) : (u / upb);
      sb[j] = __ldg(ws + s);
    }
  }
#pragma unroll
  for (int j = 0; j < U; ++j) {
    const int64_t u = base + 32 * j + lane;
    if (u < units) {
      const float sc = e4m3_to_f32(sb[j]);
      uint32_t h[4];
      e2m1x8_to_f16x8(w[j], h);
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 c = f16x2_to_f32x2(h[i]);
        const float t0 = __fmul_rn(__fmul_rn(c.x, sc), ws2);
        const float t1 = __fmul_rn(__fmul_rn(c.y, sc), ws2);
        o[i] = pack2_rn<DT>(t0, t1);
      }
      stg_v4_stream(out + u, make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
}

// Row kernel for any even K and any block_size >= 1: blockIdx.y strides over
// rows, each thread converts 8 consecutive codes of one row with byte loads
// and 16-bit stores, tracking the scale block incrementally.
template <int DT>
__global__ void __launch_bounds__(kThreads)
    fp4_dequant_rows(const uint8_t* __restrict__ Bp, const uint8_t* __restrict__ ws,
                     const float* __restrict__ ws2p, uint16_t* __restrict__ out, int64_t N,
                     int64_t K, int bs) {
  const int64_t S = (K + bs - 1) / bs;
  const int64_t k0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) * 8;
  if (k0 >= K) return;
  const float ws2 = __ldg(ws2p);
  const int64_t kend = min(k0 + 8, K);
  for (int64_t n = blockIdx.y; n < N; n += gridDim.y) {
    const uint8_t* row = Bp + n * (K / 2);
    const uint8_t* srow = ws + n * S;
    int64_t blk = k0 / bs;
    int left = bs - (int)(k0 - blk * bs);  // codes left in the current block
    float sc = e4m3_to_f32(__ldg(srow + blk));
    for (int64_t k = k0; k < kend; k += 2) {
      const uint32_t byte = __ldg(row + k / 2);
      uint32_t h[4];
      e2m1x8_to_f16x8(byte, h);
      const float2 c = f16x2_to_f32x2(h[0]);
      const float t0 = __fmul_rn(__fmul_rn(c.x, sc), ws2);
      if (--left == 0) {
        ++blk;
        left = bs;
        if (blk < S) sc = e4m3_to_f32(__ldg(srow + blk));
      }
      const float t1 = __fmul_rn(__fmul_rn(c.y, sc), ws2);
      if (--left == 0) {
        ++blk;
        left = bs;
        if (blk < S) sc = e4m3_to_f32(__ldg(srow + blk));
      }
      out[n * K + k] = to_act_rn<DT>(t0);
      out[n * K + k + 1] = to_act_rn<DT>(t1);
    }
  }
}

// FP8 flat kernel: unit = 8 codes (one 8-byte load, one 16-byte store).
template <int DT, int U>
__global__ void __launch_bounds__(kThreads)
    fp8_dequant_flat(const uint2* __restrict__ B8, const float* __restrict__ bsc,
                     uint4* __restrict__ out, int64_t units, int upb_shift, int64_t upb) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t base = ((int64_t)blockIdx.x * (kThreads / 32) + warp) * (32 * U);
  uint2 w[U];
  float sc[U];
#pragma unroll
  for (int j = 0; j < U; ++j) {
    const int64_t u = base + 32 * j + lane;
    w[j] = make_uint2(0, 0);
    sc[j] = 0.f;
    if (u < units) {
      w[j] = __ldg(B8 + u);
      sc[j] = __ldg(bsc + (upb_shift >= 0 ? (u >> upb_shift) : (u / upb)));
    }
  }
#pragma unroll
  for (int j = 0; j < U; ++j) {
    const int64_t u = base + 32 * j + lane;
    if (u < units) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t two = ((i < 2 ? w[j].x : w[j].y) >> (16 * (i & 1))) & 0xFFFFu;
        const float2 c = f16x2_to_f32x2(e4m3x2_to_f16x2(two));
        o[i] = pack2_rn<DT>(__fmul_rn(c.x, sc[j]), __fmul_rn(c.y, sc[j]));
      }
      stg_v4_stream(out + u, make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
    fp8_dequant_rows(const uint8_t* __restrict__ B, const float* __restrict__ bsc,
                     uint16_t* __restrict__ out, int64_t N, int64_t K, int bs) {
  const int64_t S = (K + bs - 1) / bs;
  const int64_t k0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) * 8;
  if (k0 >= K) return;
  const int64_t kend = min(k0 + 8, K);
  for (int64_t n = blockIdx.y; n < N; n += gridDim.y) {
    for (int64_t k = k0; k < kend; ++k) {
      const float w = e4m3_to_f32(__ldg(B + n * K + k));
      out[n * K + k] = to_act_rn<DT>(__fmul_rn(w, __ldg(bsc + n * S + k / bs)));
    }
  }
}

template <int DT>
__global__ void fill_bias_kernel(const uint16_t* __restrict__ bias, uint16_t* __restrict__ Y,
                                 int64_t M, int64_t N) {
  const int64_t total = M * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    Y[i] = bias ? bias[i % N] : (uint16_t)0;
  }
}

int log2_exact(int64_t v) {
  if (v <= 0 || (v & (v - 1))) return -1;
  int s = 0;
  while ((int64_t(1) << s) < v) ++s;
  return s;
}

int check_launch() {
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}

}  // namespace

int launch_fp4_dequant(const uint8_t* Bp, const uint8_t* ws, const float* ws2, void* out,
                       int64_t N, int64_t K, int bs, int dtype, cudaStream_t st) {
  if (bs % 8 == 0 && K % bs == 0) {
    constexpr int U = 4;
    const int64_t units = N * K / 8;
    const int64_t per_block = (int64_t)kThreads * U;
    const int64_t blocks = (units + per_block - 1) / per_block;
    const int64_t upb = bs / 8;
    const int sh = log2_exact(upb);
    const uint32_t* Bw = reinterpret_cast<const uint32_t*>(Bp);
    uint4* o = reinterpret_cast<uint4*>(out);
    if (dtype == 1)
      fp4_dequant_flat<1, U><<<(unsigned)blocks, kThreads, 0, st>>>(Bw, ws, ws2, o, units, sh, upb);
    else
      fp4_dequant_flat<0, U><<<(unsigned)blocks, kThreads, 0, st>>>(Bw, ws, ws2, o, units, sh, upb);
    return check_launch();
  }
  const int64_t chunks = (K + 7) / 8;
  dim3 grid((unsigned)((chunks + kThreads - 1) / kThreads),
            (unsigned)(N < 65535 ? N : 65535));
  uint16_t* o = reinterpret_cast<uint16_t*>(out);
  if (dtype == 1) fp4_dequant_rows<1><<<grid, kThreads, 0, st>>>(Bp, ws, ws2, o, N, K, bs);
  else fp4_dequant_rows<0><<<grid, kThreads, 0, st>>>(Bp, ws, ws2, o, N, K, bs);
  return check_launch();
}

int launch_fp8_dequant(const uint8_t* B, const float* bsc, void* out, int64_t N, int64_t K,
                       int bs, int dtype, cudaStream_t st) {
  if (bs % 8 == 0 && K % bs == 0) {
    constexpr int U = 4;
    const int64_t units = N * K / 8;
    const int64_t per_block = (int64_t)kThreads * U;
    const int64_t blocks = (units + per_block - 1) / per_block;
    const int64_t upb = bs / 8;
    const int sh = log2_exact(upb);
    const uint2* B8 = reinterpret_cast<const uint2*>(B);
    uint4* o = reinterpret_cast<uint4*>(out);
    if (dtype == 1)
      fp8_dequant_flat<1, U><<<(unsigned)blocks, kThreads, 0, st>>>(B8, bsc, o, units, sh, upb);
    else
      fp8_dequant_flat<0, U><<<(unsigned)blocks, kThreads, 0, st>>>(B8, bsc, o, units, sh, upb);
    return check_launch();
  }
  const int64_t chunks = (K + 7) / 8;
  dim3 grid((unsigned)((chunks + kThreads - 1) / kThreads),
            (unsigned)(N < 65535 ? N : 65535));
  uint16_t* o = reinterpret_cast<uint16_t*>(out);
  if (dtype == 1) fp8_dequant_rows<1><<<grid, kThreads, 0, st>>>(B, bsc, o, N, K, bs);
  else fp8_dequant_rows<0><<<grid, kThreads, 0, st>>>(B, bsc, o, N, K, bs);
  return check_launch();
}

int launch_fill_bias(const void* bias, void* Y, int64_t M, int64_t N, int dtype,
                     cudaStream_t st) {
  const int64_t total = M * N;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 65535);
  const uint16_t* b = reinterpret_cast<const uint16_t*>(bias);
  uint16_t* y = reinterpret_cast<uint16_t*>(Y);
  if (dtype == 1) fill_bias_kernel<1><<<(unsigned)blocks, 256, 0, st>>>(b, y, M, N);
  else fill_bias_kernel<0><<<(unsigned)blocks, 256, 0, st>>>(b, y, M, N);
  return check_launch();
}

}  // namespace wqmm
