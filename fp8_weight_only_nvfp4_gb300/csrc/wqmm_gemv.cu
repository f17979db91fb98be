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
#include <algorithm>
#include <mutex>

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
                 const float* __restrict__ fscale, const float* __restrict__ ascale,
                 const uint16_t* __restrict__ bias, uint16_t* __restrict__ Y, int64_t M,
                 int64_t N, int64_t K, int bs) {
  __shared__ float red[kGemvWarps][4][32];
  const float a_s = ascale != nullptr ? __ldg(ascale) : 1.f;
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
    if (ascale != nullptr) {
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = qdq_fp8_act_pair<DT>(x[i], a_s);
    }
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
        A, a.B, a.ws, a.gscale, a.fscale, a.ascale, bias, Y, a.M, a.N, a.K, a.bs);
  else
    gemv_general<DT, KIND, false><<<grid, kGemvWarps * 32, 0, st>>>(
        A, a.B, a.ws, a.gscale, a.fscale, a.ascale, bias, Y, a.M, a.N, a.K, a.bs);
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}


// ===========================================================================
// Fast decode GEMV (the path for M <= 8 with K % 32 == 0, block_size a power
// of two >= 16, NVFP4 or FP8 weight).
//
// * CTA = 8 warps = 128 weight rows (warp w owns rows 16w .. 16w + 15), all M
//   activation rows.  A thread-block cluster of C CTAs along gridDim.y splits
//   K: rank r takes 128-k windows [r * wpc, (r + 1) * wpc).  Partial sums go
//   to rank 0 through distributed shared memory and are added there in rank
//   order (deterministic; no global scratch).
// * Every lane issues the weight loads of a whole chunk of WPC windows before
//   decoding anything (16 B per row per window, two rows per lane), and the
//   next chunk's loads are in flight while the current one is decoded: with
//   two CTAs per SM that is 64 KB of weight in flight per SM.
// * The CTA's K-range of the activation is staged once in shared memory (row
//   pitch an odd multiple of 16 bytes, so the fragment reads of the active
//   lanes hit distinct banks).
// * mma.m16n8k16 (FP16 or BF16 operands, FP32 accumulate), weight as the A
//   operand.  Lane (g, t) owns k in [w*128 + 32t, w*128 + 32t + 32) of rows
//   g, g + 8 and activation row g; MMA j of a window takes k = 32t + 4j .. +1
//   into k-slots 2t, 2t + 1 and k = 32t + 4j + 2 .. +3 into 2t + 8, 2t + 9.
// * Decode per packed byte: cvt.rn.f16x2.e2m1x2, then for FP16 activations one
//   f16x2 multiply by the block scale (exact), for BF16 two mixed
//   f16 x f16 -> f32 multiplies (exact) and one pack to bf16x2 (exact).
// * Programmatic dependent launch: before griddepcontrol.wait the kernel
//   prefetches its weight rows into L2 and loads its first chunk of weight
//   codes and block scales into registers (weights are parameters, not
//   written by the kernel launched just before), so it overlaps the previous
//   kernel's tail; the activation is read after the wait.
// ===========================================================================

constexpr int kFastWarps = 8;
constexpr int kFastRows = kFastWarps * 16;
// 128-k windows per register chunk: 4 for NVFP4 (16 B per row per window),
// 2 for FP8 (32 B per row per window): 128 B of weight per lane either way.
template <int KIND>
constexpr int wpc_of() { return KIND == 0 ? 4 : 2; }

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1, int dt) {
  if (dt == 1)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E4M3 bytes (low 16 bits) -> the same values as an operand pair, exact
// (4 significant bits): FP16 straight from the convert, BF16 through two
// exact FP32 widenings and a pack.
template <int DT>
__device__ __forceinline__ uint32_t e4m3x2_exact(uint32_t two) {
  const uint32_t h = e4m3x2_to_f16x2(two);
  if constexpr (DT == 0) {
    return h;
  } else {
    float lo, hi;
    asm("{ .reg .b16 l, u; mov.b32 {l, u}, %2;\n\t"
        "cvt.f32.f16 %0, l; cvt.f32.f16 %1, u; }"
        : "=f"(lo), "=f"(hi) : "r"(h));
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  }
}

// FP8: two E4M3 bytes (low 16 bits) times a float scale -> operand pair,
// rounded once to the activation type.
template <int DT>
__device__ __forceinline__ uint32_t fp8_pair(uint32_t two, float sc) {
  const float2 e = f16x2_to_f32x2(e4m3x2_to_f16x2(two));
  return pack2_rn<DT>(e.x * sc, e.y * sc);
}

struct FastParams {
  const uint16_t* A;
  const uint8_t* B;
  const uint8_t* ws;      // NVFP4 scales
  const float* gscale;
  const float* fscale;    // FP8 scales
  const float* ascale;    // FP8 W8A8 activation scale, or nullptr
  const uint16_t* bias;
  uint16_t* Y;
  int M, N, K;
  int bs_shift;           // log2(block_size)
  int wpc;                // 128-k windows per cluster rank
  int act_pitch;          // activation smem row pitch, bytes
  int* err;
};

template <int DT, int KIND>
struct Chunk {
  // NVFP4: 16 B per row per window; FP8: 32 B per row per window.
  static constexpr int kV = (KIND == 0) ? 1 : 2;
  static constexpr int kWpc = wpc_of<KIND>();
  uint4 w0[kWpc][kV], w1[kWpc][kV];  // rows g and g + 8
  uint32_t s0[kWpc], s1[kWpc];         // NVFP4: the two E4M3 scale bytes of the 32-k run
  float f0[kWpc][2], f1[kWpc][2];      // FP8: the two float scales of the 32-k run
};

template <int DT, int KIND>
__device__ __forceinline__ void chunk_load(Chunk<DT, KIND>& c, const FastParams& p, int row0,
                                           int row1, int win_begin, int win_end, int t) {
  constexpr int kWpc = wpc_of<KIND>();
  const int S = (p.K + (1 << p.bs_shift) - 1) >> p.bs_shift;
#pragma unroll
  for (int i = 0; i < kWpc; ++i) {
    const int w = win_begin + i;
    const int k0 = w * 128 + 32 * t;
    const bool kin = (w < win_end) && (k0 < p.K);
    const bool v0 = kin && row0 < p.N, v1 = kin && row1 < p.N;
#pragma unroll
    for (int v = 0; v < Chunk<DT, KIND>::kV; ++v) {
      c.w0[i][v] = make_uint4(0, 0, 0, 0);
      c.w1[i][v] = make_uint4(0, 0, 0, 0);
    }
    c.s0[i] = c.s1[i] = 0;
    c.f0[i][0] = c.f0[i][1] = c.f1[i][0] = c.f1[i][1] = 0.f;
    const int sa = k0 >> p.bs_shift, sb = (k0 + 16) >> p.bs_shift;
    if constexpr (KIND == 0) {
      if (v0) {
        c.w0[i][0] = ldg_stream_v4(p.B + (int64_t)row0 * (p.K / 2) + k0 / 2);
        const uint8_t* sr = p.ws + (int64_t)row0 * S;
        c.s0[i] = (uint32_t)__ldg(sr + sa) | ((uint32_t)__ldg(sr + sb) << 8);
      }
      if (v1) {
        c.w1[i][0] = ldg_stream_v4(p.B + (int64_t)row1 * (p.K / 2) + k0 / 2);
        const uint8_t* sr = p.ws + (int64_t)row1 * S;
        c.s1[i] = (uint32_t)__ldg(sr + sa) | ((uint32_t)__ldg(sr + sb) << 8);
      }
    } else {
      if (v0) {
        const uint8_t* r = p.B + (int64_t)row0 * p.K + k0;
        c.w0[i][0] = ldg_stream_v4(r);
        c.w0[i][1] = ldg_stream_v4(r + 16);
      }
      if (v1) {
        const uint8_t* r = p.B + (int64_t)row1 * p.K + k0;
        c.w1[i][0] = ldg_stream_v4(r);
        c.w1[i][1] = ldg_stream_v4(r + 16);
      }
      if (p.bs_shift >= 7) {
        // One block per window: its scale, whatever part of the window this
        // lane's 32-k run covers (the MMA mixes the four lanes' runs).
        const int sw = (w * 128) >> p.bs_shift;
        if (w < win_end && row0 < p.N) c.f0[i][0] = __ldg(p.fscale + (int64_t)row0 * S + sw);
        if (w < win_end && row1 < p.N) c.f1[i][0] = __ldg(p.fscale + (int64_t)row1 * S + sw);
      } else {
        if (v0) {
          c.f0[i][0] = __ldg(p.fscale + (int64_t)row0 * S + sa);
          c.f0[i][1] = __ldg(p.fscale + (int64_t)row0 * S + sb);
        }
        if (v1) {
          c.f1[i][0] = __ldg(p.fscale + (int64_t)row1 * S + sa);
          c.f1[i][1] = __ldg(p.fscale + (int64_t)row1 * S + sb);
        }
      }
    }
  }
}

template <int DT, int KIND>
__device__ __forceinline__ void chunk_compute(float (&acc)[4], const Chunk<DT, KIND>& c,
                                              const uint8_t* act_row, bool act_on, int k_lo,
                                              int win_begin, int win_end, int t,
                                              bool block_is_window) {
  constexpr int kWpc = wpc_of<KIND>();
#pragma unroll
  for (int i = 0; i < kWpc; ++i) {
    const int w = win_begin + i;
    if (w >= win_end) break;
    uint32_t x[16];
    if (act_on) {
      const uint4* ap = reinterpret_cast<const uint4*>(act_row + (w * 128 + 32 * t - k_lo) * 2);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = ap[q];
        x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 16; ++q) x[q] = 0;
    }
    if constexpr (KIND == 0) {
      // f16 scale pairs {s, s} for the two 16-k chunks of each row.
      const uint32_t h0 = e4m3x2_to_f16x2(c.s0[i]);
      const uint32_t h1 = e4m3x2_to_f16x2(c.s1[i]);
      const uint32_t sc0[2] = {__byte_perm(h0, 0, 0x1010), __byte_perm(h0, 0, 0x3232)};
      const uint32_t sc1[2] = {__byte_perm(h1, 0, 0x1010), __byte_perm(h1, 0, 0x3232)};
      const uint32_t p0[4] = {c.w0[i][0].x, c.w0[i][0].y, c.w0[i][0].z, c.w0[i][0].w};
      const uint32_t p1[4] = {c.w1[i][0].x, c.w1[i][0].y, c.w1[i][0].z, c.w1[i][0].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // word q = bytes 4q .. 4q + 3 = MMAs 2q (bytes 4q, 4q+1) and 2q + 1.
        uint32_t h0[4], h1[4];
        e2m1x8_to_f16x8(p0[q], h0);
        e2m1x8_to_f16x8(p1[q], h1);
        const uint32_t s0 = sc0[q >> 1], s1 = sc1[q >> 1];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int j = 2 * q + u;
          mma_16816(acc, fold_f16x2<DT>(h0[2 * u], s0), fold_f16x2<DT>(h1[2 * u], s1),
                    fold_f16x2<DT>(h0[2 * u + 1], s0), fold_f16x2<DT>(h1[2 * u + 1], s1),
                    x[2 * j], x[2 * j + 1], DT);
        }
      }
    } else if (block_is_window) {
      // One scale block per row and window (bs >= 128): the window's MMAs
      // take the E4M3 values themselves (exact in FP16 and BF16) into a fresh
      // accumulator, which is then scaled by the rows' block scales in FP32:
      // one convert per weight pair for FP16 activations, and the weight is
      // never rounded after scaling.
      float w4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 q0 = c.w0[i][j >> 2], q1 = c.w1[i][j >> 2];
        const uint32_t wv0 = ((const uint32_t*)&q0)[j & 3];
        const uint32_t wv1 = ((const uint32_t*)&q1)[j & 3];
        const uint32_t a0 = e4m3x2_exact<DT>(wv0 & 0xFFFF), a2 = e4m3x2_exact<DT>(wv0 >> 16);
        const uint32_t a1 = e4m3x2_exact<DT>(wv1 & 0xFFFF), a3 = e4m3x2_exact<DT>(wv1 >> 16);
        mma_16816(w4, a0, a1, a2, a3, x[2 * j], x[2 * j + 1], DT);
      }
      acc[0] = fmaf(w4[0], c.f0[i][0], acc[0]);
      acc[1] = fmaf(w4[1], c.f0[i][0], acc[1]);
      acc[2] = fmaf(w4[2], c.f1[i][0], acc[2]);
      acc[3] = fmaf(w4[3], c.f1[i][0], acc[3]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        // bytes 4j .. 4j + 3 of the 32-byte run; chunk j / 4 of 16 k.
        const uint4 q0 = c.w0[i][j >> 2], q1 = c.w1[i][j >> 2];
        const uint32_t wv0 = ((const uint32_t*)&q0)[j & 3];
        const uint32_t wv1 = ((const uint32_t*)&q1)[j & 3];
        const float sa = c.f0[i][j >> 2], sb = c.f1[i][j >> 2];
        const uint32_t a0 = fp8_pair<DT>(wv0 & 0xFFFF, sa);
        const uint32_t a2 = fp8_pair<DT>(wv0 >> 16, sa);
        const uint32_t a1 = fp8_pair<DT>(wv1 & 0xFFFF, sb);
        const uint32_t a3 = fp8_pair<DT>(wv1 >> 16, sb);
        mma_16816(acc, a0, a1, a2, a3, x[2 * j], x[2 * j + 1], DT);
      }
    }
  }
}

template <int DT, int KIND>
__global__ void __launch_bounds__(kFastWarps * 32, 2) gemv_fast(const FastParams p) {
  extern __shared__ __align__(16) uint8_t gsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int C = gridDim.y;
  const int rank = blockIdx.y;
  const int nwin = (p.K + 127) / 128;
  const int win_lo = rank * p.wpc;
  const int win_hi = min(win_lo + p.wpc, nwin);
  const int k_lo = win_lo * 128;
  const int k_hi = min(win_hi * 128, p.K);
  const int row0 = blockIdx.x * kFastRows + warp * 16 + g;
  const int row1 = row0 + 8;
  uint8_t* act = gsm;
  float4* red = reinterpret_cast<float4*>(gsm + p.M * p.act_pitch);

  // Cluster peers must be running before any distributed shared-memory store.
  if (C > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  // L2 prefetch of this lane pair's weight rows (before the dependency wait).
  if (t == 0 && win_hi > win_lo) {
    const int wbytes = (KIND == 0) ? (k_hi - k_lo) / 2 : (k_hi - k_lo);
    const int64_t pitch = (KIND == 0) ? p.K / 2 : p.K;
    const int64_t off = (KIND == 0) ? k_lo / 2 : k_lo;
    if (row0 < p.N)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.B + row0 * pitch + off),
                   "r"(wbytes) : "memory");
    if (row1 < p.N)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.B + row1 * pitch + off),
                   "r"(wbytes) : "memory");
  }
  // The first chunk of weight codes and block scales (parameters) before the
  // dependency wait: 2-4 % per layer in the FP8 chain.
  Chunk<DT, KIND> c0, c1;
  chunk_load<DT, KIND>(c0, p, row0, row1, win_lo, win_hi, t);
  pdl_wait();

  // Stage A[:, win_lo*128 .. win_hi*128) in shared memory (zero beyond K).
  {
    const int kr = (win_hi - win_lo) * 128;
    const int vec_per_row = kr / 8;
    for (int v = threadIdx.x; v < p.M * vec_per_row; v += blockDim.x) {
      const int m = v / vec_per_row, cv = v - m * vec_per_row;
      const int k = k_lo + cv * 8;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (k < p.K) val = __ldg(reinterpret_cast<const uint4*>(p.A + (int64_t)m * p.K + k));
      if (p.ascale != nullptr) {
        // W8A8: the activation is quantized and dequantized as it is staged.
        const float a_s = __ldg(p.ascale);
        val = make_uint4(qdq_fp8_act_pair<DT>(val.x, a_s), qdq_fp8_act_pair<DT>(val.y, a_s),
                         qdq_fp8_act_pair<DT>(val.z, a_s), qdq_fp8_act_pair<DT>(val.w, a_s));
      }
      *reinterpret_cast<uint4*>(act + m * p.act_pitch + cv * 16) = val;
    }
  }
  __syncthreads();
  pdl_launch_dependents();

  constexpr int kWpc = wpc_of<KIND>();
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const bool block_is_window = KIND == 1 && p.bs_shift >= 7;
  const bool act_on = g < p.M;
  const uint8_t* act_row = act + (act_on ? g : 0) * p.act_pitch;
  for (int wb = win_lo; wb < win_hi; wb += 2 * kWpc) {
    if (wb + kWpc < win_hi) chunk_load<DT, KIND>(c1, p, row0, row1, wb + kWpc, win_hi, t);
    chunk_compute<DT, KIND>(acc, c0, act_row, act_on, k_lo, wb, win_hi, t, block_is_window);
    if (wb + 2 * kWpc < win_hi) chunk_load<DT, KIND>(c0, p, row0, row1, wb + 2 * kWpc, win_hi, t);
    if (wb + kWpc < win_hi)
      chunk_compute<DT, KIND>(acc, c1, act_row, act_on, k_lo, wb + kWpc, win_hi, t, block_is_window);
  }

  if (C > 1) {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    const uint32_t local = smem_u32(red + (rank * kFastWarps + warp) * 32 + lane);
    st_cluster_f32x4(mapa_shared(local, 0), acc[0], acc[1], acc[2], acc[3]);
    cluster_sync();
    if (rank != 0) return;
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = 0.f;
    for (int r = 0; r < C; ++r) {
      const float4 v = red[(r * kFastWarps + warp) * 32 + lane];
      acc[0] += v.x; acc[1] += v.y; acc[2] += v.z; acc[3] += v.w;
    }
  }
  const float gs = (KIND == 0) ? __ldg(p.gscale) : 1.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = (i < 2) ? row0 : row1;
    const int m = 2 * t + (i & 1);
    if (n < p.N && m < p.M) {
      float y = acc[i] * gs;
      if (p.bias) y += act_to_f32<DT>(__ldg(p.bias + n));
      p.Y[(int64_t)m * p.N + n] = to_act_rn<DT>(y);
    }
  }
}

int ilog2(int v) {
  int s = 0;
  while ((1 << s) < v) ++s;
  return (1 << s) == v ? s : -1;
}

struct FastPlan {
  int C = 1, wpc = 1, act_pitch = 0;
  size_t smem = 0;
};

constexpr size_t kFastSmemLimit = 200 * 1024;

// Cluster size and K split: two CTAs per SM where the column count allows
// it, the rest of the parallelism from splitting K across up to 8 CTAs, and
// the activation slice small enough for shared memory.
bool plan_fast(const GemvArgs& a, FastPlan& pl) {
  if (a.M < 1 || a.M > 8 || a.K % 32 != 0 || ilog2(a.bs) < 4) return false;
  // FP8 weights with FP16 activations and blocks under 128 k would fold
  // e4m3 * b_scale into an FP16 operand, which overflows for b_scale above
  // about 146; the general kernel's TF32 operands have the FP32 range.
  // (With blocks of 128 k or more the scale is applied in FP32 after the
  // MMAs on exact E4M3 operands.)
  if (a.kind == 1 && a.dtype == 0 && a.bs < 128) return false;
  if (a.N >= (int64_t(1) << 31) || a.K >= (int64_t(1) << 30)) return false;
  const DeviceInfo& d = device_info();
  const int64_t groups = (a.N + kFastRows - 1) / kFastRows;
  const int nwin = (int)((a.K + 127) / 128);
  // Two CTAs per SM are resident.  Rounding the split up oversubscribes them
  // a little, which measured best at N = 5120 (320 CTAs: 12.1 us against
  // 12.7 rounded down); by more than a quarter it runs a second wave, and
  // rounding down is faster (N = 17408, K = 5120: 408 CTAs 34.0 us, 272 CTAs
  // 26.0 us).
  int C = (int)((2 * d.sm_count + groups - 1) / groups);
  if (groups * C * 4 > 2 * (int64_t)d.sm_count * 5) C = (int)((2 * d.sm_count) / groups);
  C = std::max(1, std::min(C, std::min(8, nwin)));
  for (;; ++C) {
    if (C > std::min(8, nwin)) return false;
    const int wpc = (nwin + C - 1) / C;
    const int Ce = (nwin + wpc - 1) / wpc;  // no empty ranks
    const int pitch = wpc * 256 + 16;
    const size_t smem = (size_t)a.M * pitch + (Ce > 1 ? (size_t)Ce * kFastWarps * 32 * 16 : 0);
    if (smem <= kFastSmemLimit) {
      pl.C = Ce;
      pl.wpc = wpc;
      pl.act_pitch = pitch;
      pl.smem = smem;
      return true;
    }
  }
}

template <int DT, int KIND>
int launch_fast_t(const GemvArgs& a, const FastPlan& pl, cudaStream_t st) {
  const int groups = (int)((a.N + kFastRows - 1) / kFastRows);
  FastParams p;
  p.A = reinterpret_cast<const uint16_t*>(a.A);
  p.B = a.B;
  p.ws = a.ws;
  p.gscale = a.gscale;
  p.fscale = a.fscale;
  p.ascale = a.ascale;
  p.bias = reinterpret_cast<const uint16_t*>(a.bias);
  p.Y = reinterpret_cast<uint16_t*>(a.Y);
  p.M = (int)a.M;
  p.N = (int)a.N;
  p.K = (int)a.K;
  p.bs_shift = ilog2(a.bs);
  p.wpc = pl.wpc;
  p.act_pitch = pl.act_pitch;
  p.err = device_error_word();
  // The shared-memory opt-in is a per-device function attribute.
  static std::once_flag once[64];
  const int dev = device_info().device;
  if (dev < 0 || dev >= 64) return kCuda;
  std::call_once(once[dev], [] {
    cudaFuncSetAttribute(gemv_fast<DT, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)kFastSmemLimit);
  });
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)groups, (unsigned)pl.C, 1);
  cfg.blockDim = dim3(kFastWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)pl.C;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_fast<DT, KIND>, p);
  return e == cudaSuccess ? kOk : kCuda;
}


// ===========================================================================
// TMA-fed decode GEMV for NVFP4 with block_size 16 and K % 256 == 0,
// M <= 32 (NT = ceil(M / 8) activation tiles of the MMA's 8 columns).
//
// Same MMA mapping as gemv_fast, with the bytes in flight held in shared
// memory instead of registers.  A producer warp streams, per 256-k step,
// three 2-D tensor copies into a stage ring:
//   packed weight  [64 rows x 128 B]   8 KB, 128-byte swizzle
//   activation     [M rows x 256 k]    four 64-k boxes, 128-byte swizzle
//   block scales   [64 rows x 16 B]    1 KB
// Four consumer warps, one 16-row MMA tile each, decode and multiply whole
// steps (both 128-k windows), alternating two accumulator chains per
// activation tile: each decoded weight fragment feeds the MMAs of all NT
// activation tiles.  A stage goes back to the producer after the step's
// last MMA.  Waits block with a suspend-time hint instead of spinning.  A
// thread-block cluster of C CTAs along gridDim.y splits K; after a cluster
// barrier every rank writes its partial sums into rank 0's (now idle) stage
// memory and rank 0 adds them in rank order: deterministic, no global
// scratch.
// ===========================================================================

constexpr int kTTiles = 4;                  // 16-row tiles (= consumer warps) per CTA
constexpr int kTRows = 16 * kTTiles;        // 64 weight rows per CTA
constexpr int kTCons = kTTiles;             // consumer warps
constexpr int kTStepW = kTRows * 128;       // packed bytes per step
constexpr int kTStepS = kTRows * 16;        // scale bytes per step
constexpr int kTMaxStages = 8;
constexpr int kTThreads = (kTCons + 1) * 32;
constexpr int kTMaxM = 32;

// Per activation-tile count NT: each 64-k activation box (M <= 8 NT rows of
// 128 bytes) sits in its own 1024-aligned slot of NT KB.
template <int NT>
struct TStage {
  static constexpr int slot = 1024 * NT;
  static constexpr int stepA = 4 * slot;
  static constexpr int bytes = kTStepW + stepA + kTStepS;
};

struct TmaGemvParams {
  const float* gscale;
  const uint16_t* bias;
  uint16_t* Y;
  int M, N, K;
  int spc;        // 256-k steps per cluster rank
  int nstages;    // ring depth
  int* err;
};

struct TmaGemvSmem {
  int stages, bars, total;
  __host__ __device__ TmaGemvSmem(int nstages, int stage_bytes) {
    stages = 0;
    bars = stages + nstages * stage_bytes;
    total = bars + 2 * kTMaxStages * 8 + 16;
  }
};

// Blocking, bounded wait: try_wait with a suspend-time hint parks the warp
// until the phase completes (or the hint expires) instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool wait_abortable(uint64_t* bar, uint32_t parity, int* err,
                                               volatile int* abort_flag) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_sleep(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(a, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) break;
  }
  record_error(err, kTimeout);
  *abort_flag = 1;
  return false;
}

template <int DT, int NT>
__global__ void __launch_bounds__(kTThreads, NT == 1 ? 4 : (NT == 2 ? 3 : 2)) gemv_tma(const __grid_constant__ CUtensorMap tmW,
                                                      const __grid_constant__ CUtensorMap tmS,
                                                      const __grid_constant__ CUtensorMap tmA,
                                                      const TmaGemvParams p) {
  extern __shared__ uint8_t gsm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int C = gridDim.y;
  const int rank = blockIdx.y;
  constexpr int kTStage = TStage<NT>::bytes, kTStepA = TStage<NT>::stepA, kSlot = TStage<NT>::slot;
  const TmaGemvSmem L(p.nstages, kTStage);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + kTMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kTMaxStages);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int nsteps = p.K / 256;
  const int s_lo = rank * p.spc;
  const int s_hi = min(s_lo + p.spc, nsteps);
  const int nst = s_hi - s_lo;
  const int row_base = blockIdx.x * kTRows;
  const int NS = p.nstages;
  const uint32_t a_bytes = (uint32_t)p.M * 512u;  // activation bytes per step

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kTCons);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (C > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  __syncthreads();

  float acc[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;

  // Epilogue constants.  The global scale is part of the weight (a
  // parameter, like the packed codes and block scales copied before the
  // dependency wait): read now, by rank 0's consumers.  The bias is read
  // right after their first stage has landed: that stage holds activation
  // bytes copied after the producer's dependency wait, so the read is ordered
  // after the previous kernel's writes (the bias may be that kernel's output)
  // and its latency is hidden behind the main loop.  (Reading the global
  // scale there too cost 0.34 us per layer in the M = 4 chain.)
  const int ep_row0 = row_base + (warp < kTCons ? warp : 0) * 16 + g;
  float ep_gs = 0.f, ep_b0 = 0.f, ep_b1 = 0.f;
  if (warp < kTCons && rank == 0) ep_gs = __ldg(p.gscale);

  if (warp == kTCons) {
    // ---------------- producer ----------------
    if (lane == 0) {
      // The weight and its scales do not depend on the previous kernel: the
      // first ring's worth of them is copied into shared memory before the
      // dependency wait, and the next two steps are pulled into L2.  Only
      // the activation copies wait.
      const int npre = min(nst, NS);
      for (int i = 0; i < npre; ++i) {
        uint8_t* base = sm + L.stages + i * kTStage;
        mbar_arrive_expect_tx(&full[i], kTStepW + kTStepS + a_bytes);
        tma_load_2d(base, &tmW, (s_lo + i) * 128, row_base, &full[i]);
        tma_load_2d(base + kTStepW + kTStepA, &tmS, (s_lo + i) * 16, row_base, &full[i]);
      }
      for (int i = npre; i < min(nst, NS + 2); ++i) {
        tma_prefetch_2d(&tmW, (s_lo + i) * 128, row_base);
        tma_prefetch_2d(&tmS, (s_lo + i) * 16, row_base);
      }
      prefetch_tmap(&tmA);
      pdl_wait();
      for (int i = 0; i < npre; ++i) {
        uint8_t* base = sm + L.stages + i * kTStage;
#pragma unroll
        for (int b = 0; b < 4; ++b)
          tma_load_2d(base + kTStepW + b * kSlot, &tmA, (s_lo + i) * 256 + 64 * b, 0, &full[i]);
      }
      int issued = npre, st = npre % NS;
      uint32_t ph = npre == NS ? 1u : 0u;
      for (int i = npre; i < nst; ++i) {
        if (i >= NS && !wait_abortable(&empty[st], ph ^ 1u, p.err, abort_flag)) break;
        uint8_t* base = sm + L.stages + st * kTStage;
        mbar_arrive_expect_tx(&full[st], kTStepW + kTStepS + a_bytes);
        tma_load_2d(base, &tmW, (s_lo + i) * 128, row_base, &full[st]);
#pragma unroll
        for (int b = 0; b < 4; ++b)
          tma_load_2d(base + kTStepW + b * kSlot, &tmA, (s_lo + i) * 256 + 64 * b, 0, &full[st]);
        tma_load_2d(base + kTStepW + kTStepA, &tmS, (s_lo + i) * 16, row_base, &full[st]);
        ++issued;
        if (++st == NS) { st = 0; ph ^= 1u; }
      }
      // No copy may still be landing when the CTA moves on or exits.
      for (int i = (issued > NS ? issued - NS : 0); i < issued; ++i) {
        const uint32_t a = smem_u32(&full[i % NS]);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait_sleep(a, (i / NS) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else {
    // ---------------- consumers ----------------
    // Lanes g >= M read activation row (g mod M): those MMA columns feed only
    // outputs m >= M, which are never stored.
    const int tile = warp;
    const int r0 = tile * 16 + g, r1 = r0 + 8;  // rows within the CTA
    // Activation row of tile j for this lane: 8 j + g, or a valid row when
    // that is past M (its MMA column only feeds outputs that are not stored).
    uint32_t a_row[NT], a_sw[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int r = 8 * j + g < p.M ? 8 * j + g : (8 * j + g) % p.M;
      a_row[j] = (uint32_t)r * 128u;
      a_sw[j] = (uint32_t)(r & 7);
    }
    uint32_t w_off[2][2], s_off[2][2], a_off[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      w_off[h][0] = (r0 * 128 + 64 * h + 16 * t) ^ ((r0 & 7) << 4);
      w_off[h][1] = (r1 * 128 + 64 * h + 16 * t) ^ ((r1 & 7) << 4);
      s_off[h][0] = kTStepW + kTStepA + r0 * 16 + 8 * h + 2 * t;
      s_off[h][1] = kTStepW + kTStepA + r1 * 16 + 8 * h + 2 * t;
      a_off[h] = kTStepW + (2 * h + (t >> 1)) * kSlot;
    }
    const uint32_t a_c0 = 4 * (t & 1);
    float acc2[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc2[j][i] = 0.f;
    int st = 0;
    uint32_t ph = 0;
    for (int i = 0; i < nst; ++i) {
      if (!wait_abortable(&full[st], ph, p.err, abort_flag)) break;
      const uint8_t* stage = sm + L.stages + st * kTStage;
      uint4 pw[2][2];
      uint32_t sb[2][2];
      uint32_t x[2][16];   // activation tile 0 (NT == 1: all of it)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        pw[h][0] = *reinterpret_cast<const uint4*>(stage + w_off[h][0]);
        pw[h][1] = *reinterpret_cast<const uint4*>(stage + w_off[h][1]);
        sb[h][0] = *reinterpret_cast<const uint16_t*>(stage + s_off[h][0]);
        sb[h][1] = *reinterpret_cast<const uint16_t*>(stage + s_off[h][1]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = *reinterpret_cast<const uint4*>(stage + a_off[h] + a_row[0] +
                                                          (((a_c0 + q) ^ a_sw[0]) << 4));
          x[h][4 * q] = v.x; x[h][4 * q + 1] = v.y; x[h][4 * q + 2] = v.z; x[h][4 * q + 3] = v.w;
        }
      }
      const int st_used = st;
      if (++st == NS) { st = 0; ph ^= 1u; }
      if (i == 0) {
        pdl_launch_dependents();
        if (rank == 0) {
          if (p.bias != nullptr) {
            if (ep_row0 < p.N) ep_b0 = act_to_f32<DT>(ld_global_u16(p.bias + ep_row0));
            if (ep_row0 + 8 < p.N) ep_b1 = act_to_f32<DT>(ld_global_u16(p.bias + ep_row0 + 8));
          }
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t h0 = e4m3x2_to_f16x2(sb[h][0]);
        const uint32_t h1 = e4m3x2_to_f16x2(sb[h][1]);
        const uint32_t sc0[2] = {__byte_perm(h0, 0, 0x1010), __byte_perm(h0, 0, 0x3232)};
        const uint32_t sc1[2] = {__byte_perm(h1, 0, 0x1010), __byte_perm(h1, 0, 0x3232)};
        const uint32_t p0[4] = {pw[h][0].x, pw[h][0].y, pw[h][0].z, pw[h][0].w};
        const uint32_t p1[4] = {pw[h][1].x, pw[h][1].y, pw[h][1].z, pw[h][1].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t e0[4], e1[4];
          e2m1x8_to_f16x8(p0[q], e0);
          e2m1x8_to_f16x8(p1[q], e1);
          const uint32_t s0 = sc0[q >> 1], s1 = sc1[q >> 1];
          const int j0 = 2 * q, j1 = 2 * q + 1;
          const uint32_t fa0 = fold_f16x2<DT>(e0[0], s0), fa1 = fold_f16x2<DT>(e1[0], s1);
          const uint32_t fa2 = fold_f16x2<DT>(e0[1], s0), fa3 = fold_f16x2<DT>(e1[1], s1);
          const uint32_t fb0 = fold_f16x2<DT>(e0[2], s0), fb1 = fold_f16x2<DT>(e1[2], s1);
          const uint32_t fb2 = fold_f16x2<DT>(e0[3], s0), fb3 = fold_f16x2<DT>(e1[3], s1);
          mma_16816(acc[0], fa0, fa1, fa2, fa3, x[h][2 * j0], x[h][2 * j0 + 1], DT);
          mma_16816(acc2[0], fb0, fb1, fb2, fb3, x[h][2 * j1], x[h][2 * j1 + 1], DT);
#pragma unroll
          for (int j = 1; j < NT; ++j) {
            // The same decoded fragment against activation tile j.
            const uint4 v = *reinterpret_cast<const uint4*>(stage + a_off[h] + a_row[j] +
                                                            (((a_c0 + q) ^ a_sw[j]) << 4));
            mma_16816(acc[j], fa0, fa1, fa2, fa3, v.x, v.y, DT);
            mma_16816(acc2[j], fb0, fb1, fb2, fb3, v.z, v.w, DT);
          }
        }
      }
      // Release the stage only once every operand loaded from it has been
      // consumed: issuing the shared loads and arriving right away let the
      // next tensor copy overwrite the stage under loads still in flight.
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st_used]);
    }
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[j][i] += acc2[j][i];
  }

  // Cross-CTA reduction (rank order) into rank 0's idle stage memory.
  __syncwarp();  // the producer warp reconverges before the .aligned cluster barriers
  const bool owner = warp < kTCons;
  if (C > 1) {
    float4* red = reinterpret_cast<float4*>(sm + L.stages);
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // peers are running
    cluster_sync();                                              // every ring is drained
    if (owner) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const uint32_t local = smem_u32(red + ((rank * kTCons + warp) * NT + j) * 32 + lane);
        st_cluster_f32x4(mapa_shared(local, 0), acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
      }
      // A rank whose wait ran out tells rank 0, which then stores nothing.
      if (rank != 0 && lane == 0 && *abort_flag)
        st_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), 0), 1u);
    }
    cluster_sync();
    if (rank != 0 || !owner) return;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
      for (int r = 0; r < C; ++r) {
        const float4 v = red[((r * kTCons + warp) * NT + j) * 32 + lane];
        acc[j][0] += v.x; acc[j][1] += v.y; acc[j][2] += v.z; acc[j][3] += v.w;
      }
    }
  } else if (!owner) {
    return;
  }
  // After a wait that ran out (WQMM_ERR_TIMEOUT) Y is left untouched.
  if (*abort_flag) return;
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = (i < 2) ? ep_row0 : ep_row0 + 8;
      const int m = 8 * j + 2 * t + (i & 1);
      if (n < p.N && m < p.M)
        p.Y[(int64_t)m * p.N + n] = to_act_rn<DT>(acc[j][i] * ep_gs + ((i < 2) ? ep_b0 : ep_b1));
    }
}

struct TmaPlan {
  int nt = 1, C = 1, spc = 1, nstages = 1;
  size_t smem = 0;
};

static int tma_stage_bytes(int nt) {
  switch (nt) {
    case 1: return TStage<1>::bytes;
    case 2: return TStage<2>::bytes;
    case 3: return TStage<3>::bytes;
    default: return TStage<4>::bytes;
  }
}

// Cluster size: the largest K split (at least two steps per rank) whose CTA
// count stays within two per SM, so that every CTA is resident at once and
// the next launch's CTAs still find room to start early (programmatic
// dependent launch); with many column groups that is one rank per group.
// The ranks' partial sums must also fit in rank 0's ring.
// Measured on GB300 for N = K = 5120, M = 4: C = 3 beats 1, 2, 4, 5 and 7.
// With two activation tiles (9..16 rows) a CTA does twice the MMA work per
// step and three of them are resident per SM: up to three per SM (C = 5)
// took 9.5 instead of 11.8 us per layer in the chain; with three or four
// tiles only two are resident, and the same rule ran in two waves (15.9 /
// 18.6 instead of 11.4 / 13.3 us).
bool plan_tma(const GemvArgs& a, TmaPlan& pl) {
  if (a.kind != 0 || a.bs != 16 || a.K % 256 != 0 || a.M < 1 || a.M > kTMaxM) return false;
  if (a.N >= (int64_t(1) << 31) || a.K >= (int64_t(1) << 30)) return false;
  const DeviceInfo& d = device_info();
  const int nt = (int)((a.M + 7) / 8);
  const int stage = tma_stage_bytes(nt);
  const int64_t groups = (a.N + kTRows - 1) / kTRows;
  const int nsteps = (int)(a.K / 256);
  int C = 1;
  for (int c = 2; c <= 8 && c <= nsteps; ++c) {
    const int spc = (nsteps + c - 1) / c;
    if (spc < 2) break;
    const int ce = (nsteps + spc - 1) / spc;
    if (groups * ce > (nt == 2 ? 3 : 2) * (int64_t)d.sm_count) break;
    if (ce * kTCons * nt * 512 > std::min(spc, 4) * stage) break;
    C = ce;
  }
  const int spc = (nsteps + C - 1) / C;
  C = (nsteps + spc - 1) / spc;
  const int ns = std::min(spc, 4);
  const TmaGemvSmem L(ns, stage);
  pl.nt = nt;
  pl.C = C;
  pl.spc = spc;
  pl.nstages = ns;
  pl.smem = (size_t)L.total + 1024;
  return pl.smem <= kFastSmemLimit;
}

template <int DT, int NT>
int launch_tma_t(const GemvArgs& a, const TmaPlan& pl, cudaStream_t st) {
  CUtensorMap tmW, tmS, tmA;
  const uint64_t S = (uint64_t)a.K / 16;
  const CUtensorMapDataType adt =
      DT == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (!encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, (uint64_t)a.K / 2, (uint64_t)a.N,
                      (uint64_t)a.K / 2, 128, kTRows, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !encode_tmap_2d(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.ws, S, (uint64_t)a.N, S, 16, kTRows,
                      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !encode_tmap_2d(&tmA, adt, a.A, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.K * 2, 64,
                      (uint32_t)a.M, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return kCuda;
  TmaGemvParams p;
  p.gscale = a.gscale;
  p.bias = reinterpret_cast<const uint16_t*>(a.bias);
  p.Y = reinterpret_cast<uint16_t*>(a.Y);
  p.M = (int)a.M;
  p.N = (int)a.N;
  p.K = (int)a.K;
  p.spc = pl.spc;
  p.nstages = pl.nstages;
  p.err = device_error_word();
  // The shared-memory opt-in is a per-device function attribute.
  static std::once_flag once[64];
  const int dev = device_info().device;
  if (dev < 0 || dev >= 64) return kCuda;
  std::call_once(once[dev], [] {
    cudaFuncSetAttribute(gemv_tma<DT, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)kFastSmemLimit);
  });
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((a.N + kTRows - 1) / kTRows), (unsigned)pl.C, 1);
  cfg.blockDim = dim3(kTThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)pl.C;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_tma<DT, NT>, tmW, tmS, tmA, p);
  return e == cudaSuccess ? kOk : kCuda;
}

template <int DT>
int launch_tma_dt(const GemvArgs& a, const TmaPlan& pl, cudaStream_t st) {
  switch (pl.nt) {
    case 1: return launch_tma_t<DT, 1>(a, pl, st);
    case 2: return launch_tma_t<DT, 2>(a, pl, st);
    case 3: return launch_tma_t<DT, 3>(a, pl, st);
    default: return launch_tma_t<DT, 4>(a, pl, st);
  }
}

}  // namespace

// Standalone W8A8 activation quantize-dequantize: eight elements per thread
// (16-byte loads and stores), the tail element by element.
template <int DT>
__global__ void fp8_qdq_act_kernel(const uint16_t* __restrict__ A, const float* __restrict__ ascale,
                                   uint16_t* __restrict__ out, int64_t n) {
  const float a_s = __ldg(ascale);
  const int64_t n8 = n / 8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(A) + i);
    reinterpret_cast<uint4*>(out)[i] =
        make_uint4(qdq_fp8_act_pair<DT>(v.x, a_s), qdq_fp8_act_pair<DT>(v.y, a_s),
                   qdq_fp8_act_pair<DT>(v.z, a_s), qdq_fp8_act_pair<DT>(v.w, a_s));
  }
  const int64_t tail = n8 * 8 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tail < n) out[tail] = (uint16_t)(qdq_fp8_act_pair<DT>(A[tail], a_s) & 0xFFFFu);
}

int launch_fp8_qdq_activation(const void* A, const float* a_scale, void* out, int64_t n,
                              int dtype, cudaStream_t st) {
  if (n == 0) return kOk;
  const DeviceInfo& d = device_info();
  const int64_t blocks = std::min<int64_t>(std::max<int64_t>((n / 8 + 255) / 256, 1),
                                           (int64_t)d.sm_count * 8);
  auto a = reinterpret_cast<const uint16_t*>(A);
  auto o = reinterpret_cast<uint16_t*>(out);
  if (dtype == 1)
    fp8_qdq_act_kernel<1><<<(unsigned)blocks, 256, 0, st>>>(a, a_scale, o, n);
  else
    fp8_qdq_act_kernel<0><<<(unsigned)blocks, 256, 0, st>>>(a, a_scale, o, n);
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}

bool gemv_tma_supports(const GemvArgs& a) {
  TmaPlan tp;
  return plan_tma(a, tp);
}

int launch_gemv(const GemvArgs& a, cudaStream_t st) {
  TmaPlan tp;
  if (plan_tma(a, tp))
    return a.dtype == 1 ? launch_tma_dt<1>(a, tp, st) : launch_tma_dt<0>(a, tp, st);
  FastPlan pl;
  if (plan_fast(a, pl)) {
    if (a.kind == 0)
      return a.dtype == 1 ? launch_fast_t<1, 0>(a, pl, st) : launch_fast_t<0, 0>(a, pl, st);
    return a.dtype == 1 ? launch_fast_t<1, 1>(a, pl, st) : launch_fast_t<0, 1>(a, pl, st);
  }
  if (a.kind == 0) {
    return a.dtype == 1 ? launch_general_t<1, 0>(a, st) : launch_general_t<0, 0>(a, st);
  }
  return a.dtype == 1 ? launch_general_t<1, 1>(a, st) : launch_general_t<0, 1>(a, st);
}

}  // namespace wqmm
