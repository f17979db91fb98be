// wqmm_gemv.cu -- decode GEMV for small M (M <= 8 per launch row group).
//
// Computes Y[m, n] = gscale * sum_k A[m, k] * w[n, k] (+ bias[n]) where
//   NVFP4: w = e2m1(B[n, k]) * e4m3(ws[n, k / bs]), gscale = weight_scale_2
//          ("MatMulBlockQuantizedFp4Weight - CUDA Operator Documentation" §4:
//          the block scale is folded into the decoded weight before the
//          tensor-core product -- exact, <= 6 significant bits -- and the
//          global scale is applied once after the reduction);
//   FP8:   w = e4m3(B[n, k]) * b_scale[n, k / bs], gscale = 1
//          ("MatMulBlockQuantizedFp8Weight - CUDA Operator Documentation" §4).
//
// Mapping (FP4 page §4, tensor-core sub-path, restated): the weight is the
// MMA "A" operand (16 output columns n per warp), the activation the MMA "B"
// operand (MMA-N = 8 rows of A, rows >= M are zero).  K is permuted so that
// each lane's operands come from one contiguous 16-byte (NVFP4) or 32-byte
// (FP8) run of its weight row: lane (g, t) = (lane >> 2, lane & 3) owns
// k in [win*128 + 32t, win*128 + 32t + 32) of weight rows g and g + 8 and of
// activation row g.  MMA j of a window takes k = 32t + 2j into k-slot t and
// k = 32t + 2j + 1 into k-slot t + 4.  The permutation is the same on both
// operands, so the reduction is unchanged.
//
// The tensor-core instruction is mma.m16n8k8 with TF32 operands and FP32
// accumulation.  TF32 holds every folded NVFP4 weight and every BF16/FP16
// activation exactly, so each product is exact; decoding into 32-bit
// operands costs one conversion per code pair plus one fused multiply per
// code (the scale fold), cheaper than producing packed BF16 pairs.
//
// Per-row results do not depend on M: a row's products and their summation
// order are fixed by (n, k) alone.
#include "wqmm_device.cuh"

namespace wqmm {

namespace {

constexpr int kGemvWarps = 4;

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// f16x2 E2M1 pair times an f16 scale, exactly, into two fp32 values.
__device__ __forceinline__ void fold_pair_f16(uint32_t h2, uint32_t sc16, float& lo, float& hi) {
  asm("{ .reg .b16 l, h, s; .reg .f32 z;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.u16.u32 s, %3;\n\t"
      "mov.f32 z, 0f00000000;\n\t"
      "fma.rn.f32.f16 %0, l, s, z;\n\t"
      "fma.rn.f32.f16 %1, h, s, z; }"
      : "=f"(lo), "=f"(hi)
      : "r"(h2), "r"(sc16));
}

__device__ __forceinline__ uint32_t f32_to_tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// Activation word (two 16-bit values) -> two fp32 bit patterns.
template <int DT>
__device__ __forceinline__ void act_pair_to_f32(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (DT == 1) {
    lo = w << 16;
    hi = w & 0xFFFF0000u;
  } else {
    const float2 f = f16x2_to_f32x2(w);
    lo = __float_as_uint(f.x);
    hi = __float_as_uint(f.y);
  }
}

// Loads the lane's 32 activation values (row m, k in [k0, k0 + 32)) as 16
// words, zero outside [0, K) and for rows m >= M.
template <bool ALIGNED>
__device__ __forceinline__ void load_act(const uint16_t* __restrict__ A, int64_t M, int64_t K,
                                         int64_t m, int64_t k0, uint32_t (&x)[16]) {
  if (m < M && ALIGNED && k0 + 32 <= K) {
    const uint4* p = reinterpret_cast<const uint4*>(A + m * K + k0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(p + i);
      x[4 * i + 0] = v.x;
      x[4 * i + 1] = v.y;
      x[4 * i + 2] = v.z;
      x[4 * i + 3] = v.w;
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    uint32_t lo = 0, hi = 0;
    const int64_t k = k0 + 2 * i;
    if (m < M && k < K) lo = __ldg(A + m * K + k);
    if (m < M && k + 1 < K) hi = __ldg(A + m * K + k + 1);
    x[i] = lo | (hi << 16);
  }
}

// NVFP4: 16 packed bytes of row n covering k in [k0, k0 + 32) (k0 even).
template <bool ALIGNED>
__device__ __forceinline__ uint4 load_fp4_row(const uint8_t* __restrict__ B, int64_t N, int64_t K,
                                              int64_t n, int64_t k0) {
  if (n >= N || k0 >= K) return make_uint4(0, 0, 0, 0);
  const uint8_t* row = B + n * (K / 2);
  if (ALIGNED && k0 + 32 <= K) return ldg_stream_v4(row + k0 / 2);
  uint32_t w[4] = {0, 0, 0, 0};
  for (int i = 0; i < 16; ++i) {
    if (k0 + 2 * i < K) w[i >> 2] |= (uint32_t)__ldg(row + k0 / 2 + i) << (8 * (i & 3));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// FP8: 32 bytes of row n covering k in [k0, k0 + 32).
template <bool ALIGNED>
__device__ __forceinline__ void load_fp8_row(const uint8_t* __restrict__ B, int64_t N, int64_t K,
                                             int64_t n, int64_t k0, uint4& lo, uint4& hi) {
  lo = hi = make_uint4(0, 0, 0, 0);
  if (n >= N || k0 >= K) return;
  const uint8_t* row = B + n * K;
  if (ALIGNED && k0 + 32 <= K) {
    lo = ldg_stream_v4(row + k0);
    hi = ldg_stream_v4(row + k0 + 16);
    return;
  }
  uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int i = 0; i < 32; ++i) {
    if (k0 + i < K) w[i >> 2] |= (uint32_t)__ldg(row + k0 + i) << (8 * (i & 3));
  }
  lo = make_uint4(w[0], w[1], w[2], w[3]);
  hi = make_uint4(w[4], w[5], w[6], w[7]);
}

// One 128-k window for one lane: weight rows r0, r1, activation words x.
// KIND 0: NVFP4 (packed bytes pb0/pb1, f16 scale bits s0[2]/s1[2]);
// KIND 1: FP8 (bytes in q0/q1, float scales f0[2]/f1[2]).
template <int DT>
__device__ __forceinline__ void window_fp4(float (&acc)[4], const uint4& pb0, const uint4& pb1,
                                           const uint32_t (&s0)[2], const uint32_t (&s1)[2],
                                           const uint32_t (&x)[16]) {
  const uint32_t w0[4] = {pb0.x, pb0.y, pb0.z, pb0.w};
  const uint32_t w1[4] = {pb1.x, pb1.y, pb1.z, pb1.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h0[4], h1[4];
    e2m1x8_to_f16x8(w0[q], h0);
    e2m1x8_to_f16x8(w1[q], h1);
    const uint32_t sc0 = s0[q >> 1], sc1 = s1[q >> 1];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = 4 * q + i;  // byte index 0..15 == MMA index
      float a0, a2, a1, a3;
      fold_pair_f16(h0[i], sc0, a0, a2);
      fold_pair_f16(h1[i], sc1, a1, a3);
      uint32_t b0, b1;
      act_pair_to_f32<DT>(x[j], b0, b1);
      const uint32_t a[4] = {__float_as_uint(a0), __float_as_uint(a1), __float_as_uint(a2),
                             __float_as_uint(a3)};
      mma_tf32(acc, a, b0, b1);
    }
  }
}

template <int DT>
__device__ __forceinline__ void window_fp8(float (&acc)[4], const uint4 (&q0)[2],
                                           const uint4 (&q1)[2], const float (&f0)[2],
                                           const float (&f1)[2], const uint32_t (&x)[16]) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t w0[4] = {q0[half].x, q0[half].y, q0[half].z, q0[half].w};
    const uint32_t w1[4] = {q1[half].x, q1[half].y, q1[half].z, q1[half].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = 8 * half + i;  // MMA index: bytes 2j, 2j+1 of the 32-byte run
      const uint32_t two0 = (w0[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
      const uint32_t two1 = (w1[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
      const float2 e0 = f16x2_to_f32x2(e4m3x2_to_f16x2(two0));
      const float2 e1 = f16x2_to_f32x2(e4m3x2_to_f16x2(two1));
      const uint32_t a[4] = {f32_to_tf32_rna(e0.x * f0[half]), f32_to_tf32_rna(e1.x * f1[half]),
                             f32_to_tf32_rna(e0.y * f0[half]), f32_to_tf32_rna(e1.y * f1[half])};
      uint32_t b0, b1;
      act_pair_to_f32<DT>(x[j], b0, b1);
      mma_tf32(acc, a, b0, b1);
    }
  }
}

// General GEMV: one CTA = 16 weight rows (one MMA tile) x all of K, four
// warps splitting the 128-k windows round-robin, blockIdx.z = group of 8
// activation rows.  Handles every shape (masked tails, unaligned rows).
template <int DT, int KIND, bool ALIGNED>
__global__ void __launch_bounds__(kGemvWarps * 32)
    gemv_general(const uint16_t* __restrict__ A, const uint8_t* __restrict__ B,
                 const uint8_t* __restrict__ ws, const float* __restrict__ gscale,
                 const float* __restrict__ fscale, const uint16_t* __restrict__ bias,
                 uint16_t* __restrict__ Y, int64_t M, int64_t N, int64_t K, int bs) {
  __shared__ float red[kGemvWarps][4][32];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t n0 = (int64_t)blockIdx.x * 16;
  const int64_t m0 = (int64_t)blockIdx.z * 8;
  const int64_t r0 = n0 + g, r1 = n0 + g + 8;
  const int64_t m = m0 + g;
  const int64_t S = (K + bs - 1) / bs;
  const int64_t nwin = (K + 127) / 128;

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int64_t win = warp; win < nwin; win += kGemvWarps) {
    const int64_t k0 = win * 128 + 32 * t;
    uint32_t x[16];
    load_act<ALIGNED>(A, M, K, m, k0, x);
    if constexpr (KIND == 0) {
      const uint4 pb0 = load_fp4_row<ALIGNED>(B, N, K, r0, k0);
      const uint4 pb1 = load_fp4_row<ALIGNED>(B, N, K, r1, k0);
      uint32_t s0[2] = {0, 0}, s1[2] = {0, 0};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int64_t kc = k0 + 16 * c;
        if (kc < K) {
          if (r0 < N) s0[c] = e4m3x2_to_f16x2(__ldg(ws + r0 * S + kc / bs)) & 0xFFFFu;
          if (r1 < N) s1[c] = e4m3x2_to_f16x2(__ldg(ws + r1 * S + kc / bs)) & 0xFFFFu;
        }
      }
      window_fp4<DT>(acc, pb0, pb1, s0, s1, x);
    } else {
      uint4 q0[2], q1[2];
      load_fp8_row<ALIGNED>(B, N, K, r0, k0, q0[0], q0[1]);
      load_fp8_row<ALIGNED>(B, N, K, r1, k0, q1[0], q1[1]);
      float f0[2] = {0.f, 0.f}, f1[2] = {0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int64_t kc = k0 + 16 * c;
        if (kc < K) {
          if (r0 < N) f0[c] = __ldg(fscale + r0 * S + kc / bs);
          if (r1 < N) f1[c] = __ldg(fscale + r1 * S + kc / bs);
        }
      }
      window_fp8<DT>(acc, q0, q1, f0, f1, x);
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) red[warp][i][lane] = acc[i];
  __syncthreads();
  if (warp != 0) return;
  float sum[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float s = red[0][i][lane];
#pragma unroll
    for (int w = 1; w < kGemvWarps; ++w) s += red[w][i][lane];
    sum[i] = s;
  }
  const float gs = (KIND == 0) ? __ldg(gscale) : 1.0f;
  // c0: (n = r0, m = 2t), c1: (r0, 2t + 1), c2: (r1, 2t), c3: (r1, 2t + 1)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t n = (i < 2) ? r0 : r1;
    const int64_t mm = m0 + 2 * t + (i & 1);
    if (n < N && mm < M) {
      float y = sum[i] * gs;
      if (bias) y += act_to_f32<DT>(__ldg(bias + n));
      Y[mm * N + n] = to_act_rn<DT>(y);
    }
  }
}

template <int DT, int KIND>
int launch_general_t(const GemvArgs& a, cudaStream_t st) {
  dim3 grid((unsigned)((a.N + 15) / 16), 1, (unsigned)((a.M + 7) / 8));
  const bool aligned = (KIND == 0) ? (a.K % 32 == 0) : (a.K % 16 == 0);
  const uint16_t* A = reinterpret_cast<const uint16_t*>(a.A);
  const uint16_t* bias = reinterpret_cast<const uint16_t*>(a.bias);
  uint16_t* Y = reinterpret_cast<uint16_t*>(a.Y);
  if (aligned)
    gemv_general<DT, KIND, true><<<grid, kGemvWarps * 32, 0, st>>>(
        A, a.B, a.ws, a.gscale, a.fscale, bias, Y, a.M, a.N, a.K, a.bs);
  else
    gemv_general<DT, KIND, false><<<grid, kGemvWarps * 32, 0, st>>>(
        A, a.B, a.ws, a.gscale, a.fscale, bias, Y, a.M, a.N, a.K, a.bs);
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}

}  // namespace

int launch_gemv(const GemvArgs& a, cudaStream_t st) {
  if (a.kind == 0) {
    return a.dtype == 1 ? launch_general_t<1, 0>(a, st) : launch_general_t<0, 0>(a, st);
  }
  return a.dtype == 1 ? launch_general_t<1, 1>(a, st) : launch_general_t<0, 1>(a, st);
}

}  // namespace wqmm
