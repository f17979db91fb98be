// wqmm_actq.cu -- NVFP4 activation quantization: step 1 of the native FP4 x
// FP4 path of "MatMulBlockQuantizedFp4Weight - CUDA Operator Documentation"
// §6, which brings the activation into the weight's format (two E2M1 codes
// per byte, one E4M3 scale per 16 elements).  The page gives no formula; per
// 16-element block of a row:
//
//   amax  = max |a|                      (a exact in float32)
//   scale = E4M3(fp32(amax / 6))         RNE, saturating at 448
//   q     = E2M1(fp32(a / e4m3(scale)))  RNE (ties to even), saturating at 6,
//                                        sign of a kept; a zero scale gives +-0
//
// Codes are packed two per byte with the even k in the low nibble (the weight
// layout of the page's §2), scales are one byte per block; a partial last
// block (K % 16 != 0) takes its amax over the elements it has.  The
// quantize-dequantize form writes e2m1(q) * e4m3(scale) in the activation
// type: at most 6 significant bits in [2^-10, 2688] (or zero), exact, so a
// weight-only matmul of it has the numerics of the FP4 x FP4 product.
//
// One thread per block: two 16-byte loads, amax on packed 16-bit pairs, two
// float32 divisions per block (the scale and its reciprocal), a fused
// multiply-add and an add per element (an exact stand-in for the division,
// see below), the E2M1 and E4M3 conversions in hardware, the sign bits
// gathered with byte permutes, one 8-byte code store and one scale byte (or
// two 16-byte stores for the quantize-dequantize form).  Bound by HBM
// (2 bytes read per element) and, before that, by the ALU work per element.
#include "wqmm_device.cuh"

namespace wqmm {

namespace {

constexpr int kAqThreads = 256;

// E4M3 byte of a non-negative float32 (RNE, saturating).
__device__ __forceinline__ uint32_t e4m3_of(float s) {
  uint32_t r;
  asm("{ .reg .b16 c; cvt.rn.satfinite.e4m3x2.f32 c, %2, %1; cvt.u32.u16 %0, c; }"
      : "=r"(r)
      : "f"(s), "f"(0.0f));
  return r & 0xFFu;
}

// Eight E2M1 magnitude codes (RNE, saturating, in hardware) from eight
// non-negative float32 values, packed four bytes to a word: byte j holds
// elements 2j (low nibble) and 2j + 1.
__device__ __forceinline__ uint32_t e2m1x8(const float (&m)[8]) {
  uint32_t r;
  asm("{ .reg .b8 c0, c1, c2, c3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c3, %8, %7;\n\t"
      "mov.b32 %0, {c0, c1, c2, c3}; }"
      : "=r"(r)
      : "f"(m[0]), "f"(m[1]), "f"(m[2]), "f"(m[3]), "f"(m[4]), "f"(m[5]), "f"(m[6]), "f"(m[7]));
  return r;
}

// Sign bits of the eight activation values in words w0..w3 (two 16-bit
// values per word, the even element low) placed where e2m1x8 puts the codes:
// bit 3 of byte j for element 2j, bit 7 for element 2j + 1.  So -0.0 and
// negatives that round to zero give code 0x8.
__device__ __forceinline__ uint32_t e2m1x8_signs(uint32_t w0, uint32_t w1, uint32_t w2,
                                                 uint32_t w3) {
  const uint32_t t = __byte_perm(w0, w1, 0x7531);   // high bytes: elements 0..3
  const uint32_t u = __byte_perm(w2, w3, 0x7531);   // elements 4..7
  const uint32_t ev = __byte_perm(t, u, 0x6420);    // elements 0, 2, 4, 6
  const uint32_t od = __byte_perm(t, u, 0x7531);    // elements 1, 3, 5, 7
  return ((ev >> 4) & 0x08080808u) | (od & 0x80808080u);
}

// Largest of the two 16-bit halves of non-negative activation words (their
// float order is their unsigned order), as a float32.
template <int DT>
__device__ __forceinline__ float act_pair_max(uint32_t v) {
  const float lo = act_bits_to_f32<DT>(v & 0xFFFFu), hi = act_bits_to_f32<DT>(v >> 16);
  return fmaxf(lo, hi);
}

template <int DT>
__device__ __forceinline__ uint32_t max2_act(uint32_t a, uint32_t b) {
  uint32_t r;
  if constexpr (DT == 1)
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  else
    asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

template <int DT, bool QDQ>
__global__ void __launch_bounds__(kAqThreads)
    nvfp4_act_kernel(const uint16_t* __restrict__ A, int64_t M, int64_t K, int64_t S,
                     uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                     uint16_t* __restrict__ out) {
  const int64_t blk = (int64_t)blockIdx.x * kAqThreads + threadIdx.x;
  if (blk >= M * S) return;
  const int64_t m = blk / S, b = blk - m * S;
  const int64_t k0 = 16 * b;
  const int n = K - k0 < 16 ? (int)(K - k0) : 16;
  const uint16_t* a = A + m * K + k0;
  uint32_t w[8];  // 16 activation values, two per word (low half = even k)
  if (n == 16 && (reinterpret_cast<uintptr_t>(a) & 15u) == 0) {
    const uint4 v0 = *reinterpret_cast<const uint4*>(a);
    const uint4 v1 = *reinterpret_cast<const uint4*>(a + 8);
    w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
    w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = (2 * i < n) ? a[2 * i] : 0u;
      const uint32_t hi = (2 * i + 1 < n) ? a[2 * i + 1] : 0u;
      w[i] = lo | (hi << 16);
    }
  }
  // amax on the packed magnitudes: sign bits cleared, pairwise max.
  uint32_t aw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) aw[i] = w[i] & 0x7FFF7FFFu;
  const uint32_t m01 = max2_act<DT>(aw[0], aw[1]), m23 = max2_act<DT>(aw[2], aw[3]);
  const uint32_t m45 = max2_act<DT>(aw[4], aw[5]), m67 = max2_act<DT>(aw[6], aw[7]);
  const float amax =
      act_pair_max<DT>(max2_act<DT>(max2_act<DT>(m01, m23), max2_act<DT>(m45, m67)));
  const uint32_t sc = e4m3_of(__fdiv_rn(amax, 6.0f));
  const float sd = e4m3_to_f32(sc);
  // The E2M1 code of fp32(a / sd) without a division per element: |a| *
  // RN(1 / sd) is within 2^-24 (relative) of |a| / sd, and a quotient that is
  // not one of the E2M1 rounding midpoints (0.25, 0.75, ..., 5) lies at least
  // 2^-11 (relative) away from all of them (a has at most 11 significant
  // bits, sd 4).  Snapping the product to a grid of 2^-15 with one fused
  // multiply-add (RN(|a| * inv + 384) - 384, exact subtraction; valid below
  // 8, larger values saturate either way) moves every exact midpoint onto
  // the midpoint and keeps every other value on its side, so the hardware
  // round-to-nearest-even conversion gives the code of the division.
  // A zero scale gives inv = 0 and codes +-0.
  const float inv = sd == 0.0f ? 0.0f : __fdiv_rn(1.0f, sd);
  float mag[2][8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float v = act_bits_to_f32<DT>(h ? (aw[i] >> 16) : (aw[i] & 0xFFFFu));
      mag[i >> 2][2 * (i & 3) + h] = __fadd_rn(__fmaf_rn(v, inv, 384.0f), -384.0f);
    }
  }
  const uint32_t lo4 = e2m1x8(mag[0]) | e2m1x8_signs(w[0], w[1], w[2], w[3]);
  const uint32_t hi4 = e2m1x8(mag[1]) | e2m1x8_signs(w[4], w[5], w[6], w[7]);
  if constexpr (!QDQ) {
    uint8_t* c = codes + m * (K / 2) + k0 / 2;
    if (n == 16 && (reinterpret_cast<uintptr_t>(c) & 7u) == 0) {
      *reinterpret_cast<uint2*>(c) = make_uint2(lo4, hi4);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (2 * i < n) c[i] = (uint8_t)((i < 4 ? lo4 : hi4) >> (8 * (i & 3)));
    }
    scales[blk] = (uint8_t)sc;
  } else {
    uint32_t o[8];
    uint32_t h[8];
    e2m1x8_to_f16x8(lo4, *reinterpret_cast<uint32_t(*)[4]>(&h[0]));
    e2m1x8_to_f16x8(hi4, *reinterpret_cast<uint32_t(*)[4]>(&h[4]));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 e = f16x2_to_f32x2(h[i]);
      o[i] = pack2_rn<DT>(e.x * sd, e.y * sd);  // exact products
    }
    uint16_t* y = out + m * K + k0;
    if (n == 16 && (reinterpret_cast<uintptr_t>(y) & 15u) == 0) {
      *reinterpret_cast<uint4*>(y) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(y + 8) = make_uint4(o[4], o[5], o[6], o[7]);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i < n) y[i] = (uint16_t)(o[i >> 1] >> (16 * (i & 1)));
    }
  }
}

template <bool QDQ>
int launch_actq(const void* A, uint8_t* codes, uint8_t* scales, void* out, int64_t M, int64_t K,
                int dtype, cudaStream_t st) {
  const int64_t S = (K + 15) / 16;
  const int64_t blocks = (M * S + kAqThreads - 1) / kAqThreads;
  if (blocks > 0x7FFFFFFF) return kUnsupported;
  const uint16_t* a = static_cast<const uint16_t*>(A);
  uint16_t* o = static_cast<uint16_t*>(out);
  if (dtype == 1)
    nvfp4_act_kernel<1, QDQ><<<(unsigned)blocks, kAqThreads, 0, st>>>(a, M, K, S, codes, scales, o);
  else
    nvfp4_act_kernel<0, QDQ><<<(unsigned)blocks, kAqThreads, 0, st>>>(a, M, K, S, codes, scales, o);
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}

}  // namespace

int launch_nvfp4_quantize_activation(const void* A, uint8_t* codes, uint8_t* scales, int64_t M,
                                     int64_t K, int dtype, cudaStream_t st) {
  return launch_actq<false>(A, codes, scales, nullptr, M, K, dtype, st);
}

int launch_nvfp4_qdq_activation(const void* A, void* out, int64_t M, int64_t K, int dtype,
                                cudaStream_t st) {
  return launch_actq<true>(A, nullptr, nullptr, out, M, K, dtype, st);
}

}  // namespace wqmm
