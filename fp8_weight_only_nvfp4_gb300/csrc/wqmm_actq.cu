// wqmm_actq.cu -- NVFP4 activation quantization: step 1 of the native FP4 x
// FP4 path of "MatMulBlockQuantizedFp4Weight - CUDA Operator Documentation"
// §6 ("quantize activation A to packed NVFP4 E2M1 with per-16-block E4M3
// scales").  The page gives no formula; per 16-element block of a row:
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
// One thread per block: two 16-byte loads, two float32 divisions per block
// (the scale and its reciprocal), a multiply and two adds per element (an
// exact stand-in for the division, see below), the E2M1 and E4M3
// conversions in hardware, one
// 8-byte code store and one scale byte (or two 16-byte stores for the
// quantize-dequantize form).  HBM-bound: 2 bytes read per element.
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

// E2M1 code pair (low nibble = lo) from two non-negative magnitudes (RNE,
// saturating, in hardware) and the signs of two values (xlo, xhi): -0.0 and
// negatives that round to zero give code 0x8.
__device__ __forceinline__ uint32_t e2m1_pair(float xlo, float xhi, float mlo, float mhi) {
  uint32_t r;
  asm("{ .reg .b8 c; .reg .b32 w; cvt.rn.satfinite.e2m1x2.f32 c, %2, %1;\n\t"
      "mov.b32 w, {c, c, c, c}; and.b32 %0, w, 0xFF; }"
      : "=r"(r)
      : "f"(mlo), "f"(mhi));
  r |= (__float_as_uint(xlo) >> 31) << 3;
  r |= (__float_as_uint(xhi) >> 31) << 7;
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
  float x[16];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = act_bits_to_f32<DT>(w[i] & 0xFFFFu);
    x[2 * i + 1] = act_bits_to_f32<DT>(w[i] >> 16);
    amax = fmaxf(amax, fmaxf(fabsf(x[2 * i]), fabsf(x[2 * i + 1])));
  }
  const uint32_t sc = e4m3_of(__fdiv_rn(amax, 6.0f));
  const float sd = e4m3_to_f32(sc);
  // The E2M1 code of fp32(a / sd) without a division per element: p = a *
  // RN(1 / sd) is within 2^-23 (relative) of a / sd, and a quotient that is
  // not one of the E2M1 rounding midpoints (0.25, 0.75, ..., 5) lies at least
  // 2^-11 (relative) away from all of them (a has at most 11 significant
  // bits, sd 4).  Snapping p to a grid of 2^-15 ((p + 384) - 384, valid
  // below 8; larger values saturate either way) moves every exact midpoint
  // onto the midpoint and keeps every other value on its side, so the
  // hardware round-to-nearest-even conversion gives the code of the division.
  // A zero scale gives inv = 0 and codes +-0.
  const float inv = sd == 0.0f ? 0.0f : __fdiv_rn(1.0f, sd);
  auto snap = [&](float v) {
    return __fadd_rn(__fadd_rn(fabsf(v) * inv, 384.0f), -384.0f);
  };
  uint32_t q[8];  // one code pair (byte) per word
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = e2m1_pair(x[2 * i], x[2 * i + 1], snap(x[2 * i]),
                                              snap(x[2 * i + 1]));
  if constexpr (!QDQ) {
    uint8_t* c = codes + m * (K / 2) + k0 / 2;
    const uint32_t lo4 = q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24);
    const uint32_t hi4 = q[4] | (q[5] << 8) | (q[6] << 16) | (q[7] << 24);
    if (n == 16 && (reinterpret_cast<uintptr_t>(c) & 7u) == 0) {
      *reinterpret_cast<uint2*>(c) = make_uint2(lo4, hi4);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (2 * i < n) c[i] = (uint8_t)q[i];
    }
    scales[blk] = (uint8_t)sc;
  } else {
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t h;
      asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1;\n\t"
          "cvt.rn.f16x2.e2m1x2 %0, b0; }"
          : "=r"(h)
          : "r"(q[i]));
      const float2 e = f16x2_to_f32x2(h);
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
