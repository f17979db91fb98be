// wqmm_oracle.cpp -- CPU oracle for block-quantized weight-only matmul.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
// reference that the CUDA library is checked against.  Only the test suite,
// the smoke check and the benchmark's CPU-baseline leg may load it.  It shares
// no code, header, table or helper with the CUDA path under
// fp8_weight_only_nvfp4_gb300/csrc, and it includes nothing from there.
//
// Every quantity is decoded from the format definitions and accumulated in
// float64.  Sources (web pages, by title and section):
//   [FP4] "MatMulBlockQuantizedFp4Weight - CUDA Operator Documentation"
//         §2 Weight Format, §4 Decode Path (scale-fold exactness and range).
//   [FP8] "MatMulBlockQuantizedFp8Weight - CUDA Operator Documentation"
//         §1 Operator Schema (float8e4m3fn), §2 Tensor and Scale Format.
//   [BLOG] "ONNX Runtime #32128 -- Why Dequantizing 4-Bit Weights Became the
//         Most Expensive Kernel in H200 Prefill", section "Bitwise equivalence
//         was checked at three levels" (-0.0 from code 0x8).
//
// Readings taken where the pages are silent:
//   * dequant order: (e2m1 * e4m3) in fp32 (exact), then * weight_scale_2 in
//     fp32 (one RNE rounding), then RNE to the activation type;
//   * E4M3 scale bytes are the "fn" variant (no infinities, 0x7F/0xFF = NaN);
//   * scale columns S = ceil(K / block_size), indexed by floor(k / block_size);
//   * FP8 dequant: fp32(e4m3 * b_scale) with one RNE, then RNE to act;
//   * matmul reference: exact decode in float64, float64 sums, bias added in
//     float64; the tolerance is applied by the caller.
//
//   * NVFP4 activation quantization ([FP4] §6, step 1 of the native path):
//     per 16-element block, scale = E4M3(fp32(amax / 6)), codes =
//     E2M1(fp32(a / scale)) (RNE, ties to even, saturating, sign kept), no
//     activation global scale (the page names none).
//   * W8A8 activation quantization ([FP8] §6, "Optional W8A8 Activation
//     Path": A_deq = fp8_e4m3(A / a_scale) * a_scale): A / a_scale as one
//     float32 division (IEEE, correctly rounded), E4M3FN by round-to-nearest-
//     even with saturation to +-448 (NaN stays NaN), the product with a_scale
//     as one float32 multiplication, then RNE to the activation type.
//
// Parity pins for every function here live in tests/test_oracle_pins.py.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

// ---------------------------------------------------------------------------
// E2M1 (4-bit: sign, 2 exponent bits, 1 mantissa bit).  [FP4] §2 lists the
// magnitudes implicitly through the range argument of §4 (max 6); the value
// set {0, 0.5, 1, 1.5, 2, 3, 4, 6} is the E2M1 definition: exponent bias 1,
// exponent 0 is subnormal (m * 0.5).  Codes 8..15 are the negatives, and code
// 0x8 is negative zero ([BLOG], bitwise checks).
// Written as an explicit 16-entry table.
const double kE2M1[16] = {
    +0.0, +0.5, +1.0, +1.5, +2.0, +3.0, +4.0, +6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
};

// E4M3FN (8-bit: sign, 4 exponent bits with bias 7, 3 mantissa bits; no
// infinities; exponent 15 with mantissa 7 is NaN).  [FP8] §1 names the type
// float8e4m3fn; [FP4] §4 gives its extremes (448 and 2^-9).
// The 256-entry table is filled once from the field definition.
double g_e4m3[256];
bool g_e4m3_ready = false;

void build_e4m3_table() {
  if (g_e4m3_ready) return;
  for (int b = 0; b < 256; ++b) {
    const int s = (b >> 7) & 1;
    const int e = (b >> 3) & 0xF;
    const int m = b & 0x7;
    double v;
    if (e == 0xF && m == 0x7) {
      v = std::nan("");
    } else if (e == 0) {
      v = (m / 8.0) * std::ldexp(1.0, -6);          // subnormal: 0.m * 2^(1-7)
    } else {
      v = (1.0 + m / 8.0) * std::ldexp(1.0, e - 7);  // normal: 1.m * 2^(e-7)
    }
    g_e4m3[b] = s ? -v : v;
  }
  g_e4m3_ready = true;
}

// float32 <-> bits
inline uint32_t f32_bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }
inline float bits_f32(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }

// Round a float32 (given as bits) to bfloat16 bits, round-to-nearest-even.
// bfloat16 keeps the float32 exponent field and the top 7 mantissa bits, so
// the rounding looks only at the 16 discarded low bits.  NaN maps to the
// canonical quiet NaN with the input's sign.  A carry out of the mantissa
// moves into the exponent, which turns the largest finite values into inf,
// as RNE requires.
uint16_t rne_f32_to_bf16(uint32_t x) {
  if ((x & 0x7F800000u) == 0x7F800000u && (x & 0x007FFFFFu) != 0)
    return (uint16_t)(((x >> 16) & 0x8000u) | 0x7FC0u);
  uint32_t keep = x >> 16;
  const uint32_t rem = x & 0xFFFFu;
  if (rem > 0x8000u || (rem == 0x8000u && (keep & 1u))) keep += 1;
  return (uint16_t)keep;
}

// Round a float32 (given as bits) to IEEE binary16 bits, round-to-nearest-even,
// with gradual underflow (subnormals down to 2^-24) and overflow to inf.
uint16_t rne_f32_to_f16(uint32_t x) {
  const uint32_t sign = (x >> 16) & 0x8000u;
  const uint32_t ax = x & 0x7FFFFFFFu;
  if (ax > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);   // NaN
  if (ax == 0x7F800000u) return (uint16_t)(sign | 0x7C00u);  // inf
  const int e = (int)(ax >> 23);
  if (e == 0) return (uint16_t)sign;  // |x| < 2^-126: far below 2^-25, rounds to 0
  const int ue = e - 127;                                   // unbiased exponent
  const uint32_t sig = (ax & 0x007FFFFFu) | 0x00800000u;   // 24-bit significand
  if (ue > 15) return (uint16_t)(sign | 0x7C00u);          // >= 2^16: inf
  // binary16 normal numbers keep 11 significant bits (drop 13); below 2^-14
  // the grid is fixed at 2^-24, so more bits are dropped.
  const int shift = (ue >= -14) ? 13 : 13 + (-14 - ue);
  if (shift > 24) return (uint16_t)sign;                    // < 2^-25: rounds to 0
  uint32_t q = sig >> shift;
  const uint32_t rem = sig & ((1u << shift) - 1u);
  const uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (q & 1u))) q += 1;
  if (ue >= -14) {
    // q in [2^10, 2^11]; q == 2^11 carries into the exponent.
    const uint32_t bits = ((uint32_t)(ue + 15) << 10) + (q - 0x400u);
    if (bits >= 0x7C00u) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | bits);
  }
  return (uint16_t)(sign | q);  // subnormal (q == 2^10 becomes the smallest normal)
}

inline uint16_t rne_to_act(uint32_t f32bits, int dtype) {
  return dtype == 1 ? rne_f32_to_bf16(f32bits) : rne_f32_to_f16(f32bits);
}

// Activation bits -> double.  bfloat16 is the top half of a float32.
double bf16_to_double(uint16_t h) { return (double)bits_f32((uint32_t)h << 16); }

double f16_to_double(uint16_t h) {
  const int s = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1F;
  const int m = h & 0x3FF;
  double v;
  if (e == 0x1F) v = m ? std::nan("") : INFINITY;
  else if (e == 0) v = std::ldexp((double)m, -24);                 // 0.m * 2^-14
  else v = std::ldexp(1.0 + m / 1024.0, e - 15);
  return s ? -v : v;
}

inline double act_to_double(uint16_t h, int dtype) {
  return dtype == 1 ? bf16_to_double(h) : f16_to_double(h);
}

// The E2M1 code of logical element (n, k) in the packed [N, K/2] matrix:
// the low nibble holds the even k, the high nibble the odd k ([FP4] §2).
inline int fp4_code(const uint8_t* Bp, int64_t K, int64_t n, int64_t k) {
  const uint8_t byte = Bp[n * (K / 2) + k / 2];
  return (k & 1) ? (byte >> 4) : (byte & 0xF);
}

// Number of scale columns: ceil(K / block_size).
inline int64_t scale_cols(int64_t K, int bs) { return (K + bs - 1) / bs; }

// Dequantized FP4 weight in float64 (exact: at most 6 + 24 significant bits).
//   B_dequant[n, k] = e2m1(B[n, k]) * e4m3(weight_scale[n, k / bs]) * ws2
void fp4_decode_row(const uint8_t* Bp, const uint8_t* ws, float ws2, int64_t K,
                    int bs, int64_t n, double* row) {
  const int64_t S = scale_cols(K, bs);
  for (int64_t k = 0; k < K; ++k) {
    const double q = kE2M1[fp4_code(Bp, K, n, k)];
    const double s = g_e4m3[ws[n * S + k / bs]];
    row[k] = q * s * (double)ws2;
  }
}

// Dequantized FP8 weight in float64 (exact: 4 + 24 significant bits).
//   B_dequant[n, k] = e4m3(B[n, k]) * b_scale[n, k / bs]   ([FP8] §2)
// A partial final block uses the last scale column: floor(k / bs) reaches it.
void fp8_decode_row(const uint8_t* B, const float* bsc, int64_t K, int bs,
                    int64_t n, double* row) {
  const int64_t S = scale_cols(K, bs);
  for (int64_t k = 0; k < K; ++k)
    row[k] = g_e4m3[B[n * K + k]] * (double)bsc[n * S + k / bs];
}

template <class F>
void parallel_for(int64_t count, int threads, F&& body) {
  if (threads < 1) threads = 1;
  if (count < threads) threads = (int)std::max<int64_t>(count, 1);
  if (threads == 1) { for (int64_t i = 0; i < count; ++i) body(i); return; }
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t) {
    pool.emplace_back([&, t]() {
      for (int64_t i = t; i < count; i += threads) body(i);
    });
  }
  for (auto& th : pool) th.join();
}

// Y_ref[m, n] = sum_k A[m, k] * Bdq[n, k] + bias[n];  Sabs[m, n] = sum_k |A * Bdq|
// over rows n, given a per-row decoder.
template <class Decode>
void matmul_full(const uint16_t* A, const uint16_t* bias, int64_t M, int64_t N,
                 int64_t K, int dtype, double* Y, double* Sabs, int threads,
                 Decode&& decode) {
  // Decode A once (rows are shared by every n).
  std::vector<double> Ad((size_t)(M * K));
  for (int64_t i = 0; i < M * K; ++i) Ad[i] = act_to_double(A[i], dtype);
  parallel_for(N, threads, [&](int64_t n) {
    std::vector<double> row((size_t)K);
    decode(n, row.data());
    const double b = bias ? act_to_double(bias[n], dtype) : 0.0;
    for (int64_t m = 0; m < M; ++m) {
      const double* a = Ad.data() + m * K;
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double p = a[k] * row[k];
        acc += p;
        mag += std::fabs(p);
      }
      Y[m * N + n] = acc + b;
      Sabs[m * N + n] = mag;
    }
  });
}

// Same quantities for a list of (m, n) output positions only.
template <class Decode>
void matmul_sampled(const uint16_t* A, const uint16_t* bias, int64_t K,
                    int dtype, const int64_t* ms, const int64_t* ns,
                    int64_t count, double* Y, double* Sabs, int threads,
                    Decode&& decode) {
  parallel_for(count, threads, [&](int64_t i) {
    std::vector<double> row((size_t)K);
    decode(ns[i], row.data());
    const uint16_t* a = A + ms[i] * K;
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double p = act_to_double(a[k], dtype) * row[k];
      acc += p;
      mag += std::fabs(p);
    }
    Y[i] = acc + (bias ? act_to_double(bias[ns[i]], dtype) : 0.0);
    Sabs[i] = mag;
  });
}

}  // namespace

// E4M3FN code of a float32 value: round to nearest, ties to the even
// mantissa, saturating to the largest finite magnitude 448; NaN -> 0x7F with
// the input's sign.  Plain table search over the 127 non-negative finite
// codes (0x00 .. 0x7E ascend in value).
uint8_t e4m3_rne_satfinite(float f) {
  build_e4m3_table();
  const uint8_t sign = std::signbit(f) ? 0x80 : 0x00;
  if (std::isnan(f)) return (uint8_t)(sign | 0x7F);
  const double a = std::fabs((double)f);
  if (a >= g_e4m3[0x7E]) return (uint8_t)(sign | 0x7E);
  int lo = 0;
  while (lo + 1 <= 0x7E && g_e4m3[lo + 1] <= a) ++lo;  // g[lo] <= a < g[lo + 1]
  if (g_e4m3[lo] == a) return (uint8_t)(sign | lo);
  const double dlo = a - g_e4m3[lo], dhi = g_e4m3[lo + 1] - a;
  int c;
  if (dlo < dhi) c = lo;
  else if (dhi < dlo) c = lo + 1;
  else c = (lo % 2 == 0) ? lo : lo + 1;  // tie: even mantissa (code parity = mantissa parity)
  return (uint8_t)(sign | c);
}

// E2M1 code of a float32 value: round to nearest, ties to the even mantissa
// (code parity = mantissa parity), saturating to the largest magnitude 6.
// The sign of the input is kept, so -0.0 and negative values that round to
// zero give code 0x8 (negative zero).  Plain search over the 8 magnitudes
// (codes 0..7 ascend in value).  Finite inputs only.
uint8_t e2m1_rne_satfinite(float f) {
  const uint8_t sign = std::signbit(f) ? 0x8 : 0x0;
  const double a = std::fabs((double)f);
  if (a >= kE2M1[7]) return (uint8_t)(sign | 7);
  int lo = 0;
  while (lo + 1 <= 7 && kE2M1[lo + 1] <= a) ++lo;  // kE2M1[lo] <= a < kE2M1[lo + 1]
  if (kE2M1[lo] == a) return (uint8_t)(sign | lo);
  const double dlo = a - kE2M1[lo], dhi = kE2M1[lo + 1] - a;
  int c;
  if (dlo < dhi) c = lo;
  else if (dhi < dlo) c = lo + 1;
  else c = (lo % 2 == 0) ? lo : lo + 1;
  return (uint8_t)(sign | c);
}

// NVFP4 activation quantization, one 16-element block of one row ([FP4] §6,
// the native SM120 FP4 x FP4 path, step 1, which turns the activation into
// the weight's own format: two E2M1 codes per byte and one E4M3 scale per 16
// elements).  The page gives no formula;
// the reading taken (plainest, no activation global scale since the page
// names none):
//   amax  = max |a| over the block (a exact in float32)
//   scale = E4M3(fp32(amax / 6))              RNE, saturating at 448
//   q_i   = E2M1(fp32(a_i / e4m3(scale)))     RNE, saturating at 6, sign kept;
//           a scale that decodes to 0 gives q_i = +-0 (sign of a_i).
// Writes n codes (n <= 16) and returns the scale byte.
uint8_t nvfp4_quantize_block(const uint16_t* a, int n, int dtype, uint8_t* codes) {
  build_e4m3_table();
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    const float v = (float)std::fabs(act_to_double(a[i], dtype));  // exact
    if (v > amax) amax = v;
  }
  const uint8_t sc = e4m3_rne_satfinite(amax / 6.0f);  // one float32 division
  const float sd = (float)g_e4m3[sc];
  for (int i = 0; i < n; ++i) {
    const float x = (float)act_to_double(a[i], dtype);
    if (sd == 0.0f) codes[i] = std::signbit(x) ? 0x8 : 0x0;
    else codes[i] = e2m1_rne_satfinite(x / sd);          // one float32 division
  }
  return sc;
}

// One activation element of the W8A8 path: RNE_act(fp32(e4m3(fp32(a / s)) * s)).
uint16_t fp8_qdq_one(uint16_t a_bits, float a_scale, int dtype) {
  const float a = (float)act_to_double(a_bits, dtype);     // exact
  const float q = a / a_scale;                               // one float32 division
  const uint8_t code = e4m3_rne_satfinite(q);
  const float v = (float)g_e4m3[code] * a_scale;             // one float32 multiplication
  return rne_to_act(f32_bits(v), dtype);
}

extern "C" {

int orc_hardware_threads(void) {
  const unsigned n = std::thread::hardware_concurrency();
  return n ? (int)n : 1;
}

double orc_e2m1_value(int code) { return kE2M1[code & 0xF]; }

double orc_e4m3_value(int byte) { build_e4m3_table(); return g_e4m3[byte & 0xFF]; }

uint16_t orc_rne_f32_to_bf16(uint32_t bits) { return rne_f32_to_bf16(bits); }
uint16_t orc_rne_f32_to_f16(uint32_t bits) { return rne_f32_to_f16(bits); }

void orc_rne_f32_to_act_array(const uint32_t* in, uint16_t* out, int64_t n, int dtype) {
  for (int64_t i = 0; i < n; ++i) out[i] = rne_to_act(in[i], dtype);
}

double orc_act_to_double(uint16_t bits, int dtype) { return act_to_double(bits, dtype); }

int orc_e4m3_from_f32(float f) { return e4m3_rne_satfinite(f); }

// W8A8 activation quantize-dequantize ([FP8] §6), element by element.
void orc_fp8_qdq_activation(const uint16_t* A, float a_scale, uint16_t* out, int64_t n,
                            int dtype) {
  build_e4m3_table();
  for (int64_t i = 0; i < n; ++i) out[i] = fp8_qdq_one(A[i], a_scale, dtype);
}

int orc_e2m1_from_f32(float f) { return e2m1_rne_satfinite(f); }

// NVFP4 activation quantization of A [M, K] (K even): codes packed two per
// byte, the even k in the low nibble (the weight layout of [FP4] §2), into
// codes [M, K / 2]; E4M3 block scales into scales [M, ceil(K / 16)].  A
// partial last block (K % 16 != 0) takes its amax over the elements it has.
void orc_nvfp4_quantize_act(const uint16_t* A, int64_t M, int64_t K, int dtype, uint8_t* codes,
                            uint8_t* scales) {
  const int64_t S = (K + 15) / 16;
  for (int64_t m = 0; m < M; ++m) {
    std::memset(codes + m * (K / 2), 0, (size_t)(K / 2));
    for (int64_t b = 0; b < S; ++b) {
      const int n = (int)std::min<int64_t>(16, K - 16 * b);
      uint8_t q[16];
      scales[m * S + b] = nvfp4_quantize_block(A + m * K + 16 * b, n, dtype, q);
      for (int i = 0; i < n; ++i) {
        const int64_t k = 16 * b + i;
        uint8_t& byte = codes[m * (K / 2) + k / 2];
        byte = (uint8_t)(byte | ((k % 2 == 0) ? q[i] : (q[i] << 4)));
      }
    }
  }
}

// NVFP4 activation quantize-dequantize: out = RNE_act(e2m1(q) * e4m3(scale))
// per element.  The product has at most 6 significant bits and lies in
// [2^-10, 2688] (or is zero), so it is exact in float32 and in both
// activation types: the rounding to the activation type is exact.
void orc_nvfp4_qdq_act(const uint16_t* A, int64_t M, int64_t K, int dtype, uint16_t* out) {
  build_e4m3_table();
  const int64_t S = (K + 15) / 16;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t b = 0; b < S; ++b) {
      const int n = (int)std::min<int64_t>(16, K - 16 * b);
      uint8_t q[16];
      const uint8_t sc = nvfp4_quantize_block(A + m * K + 16 * b, n, dtype, q);
      const float sd = (float)g_e4m3[sc];
      for (int i = 0; i < n; ++i) {
        const float v = (float)kE2M1[q[i]] * sd;  // exact
        out[m * K + 16 * b + i] = rne_to_act(f32_bits(v), dtype);
      }
    }
  }
}

// Standalone FP4 dequantize (bit-exact contract):
//   t = fp32(e2m1 * e4m3)        -- exact
//   t = fp32(t * weight_scale_2) -- one RNE rounding
//   out = RNE_act(t)
// The fp32 rounding is taken from the exact float64 product (which is the
// correctly rounded fp32 product by definition of IEEE multiplication).
void orc_fp4_dequantize(const uint8_t* Bp, const uint8_t* ws, float ws2,
                        uint16_t* out, int64_t N, int64_t K, int bs, int dtype,
                        int threads) {
  build_e4m3_table();
  const int64_t S = scale_cols(K, bs);
  parallel_for(N, threads, [&](int64_t n) {
    for (int64_t k = 0; k < K; ++k) {
      const double q = kE2M1[fp4_code(Bp, K, n, k)];
      const double s = g_e4m3[ws[n * S + k / bs]];
      const float t = (float)(q * s);                 // exact
      const float r = (float)((double)t * (double)ws2);  // one RNE rounding
      out[n * K + k] = rne_to_act(f32_bits(r), dtype);
    }
  });
}

// Standalone FP8 dequantize: out = RNE_act(fp32(e4m3(B) * b_scale)).
void orc_fp8_dequantize(const uint8_t* B, const float* bsc, uint16_t* out,
                        int64_t N, int64_t K, int bs, int dtype, int threads) {
  build_e4m3_table();
  const int64_t S = scale_cols(K, bs);
  parallel_for(N, threads, [&](int64_t n) {
    for (int64_t k = 0; k < K; ++k) {
      const double w = g_e4m3[B[n * K + k]];
      const float r = (float)(w * (double)bsc[n * S + k / bs]);  // one RNE rounding
      out[n * K + k] = rne_to_act(f32_bits(r), dtype);
    }
  });
}

// Float64 dequantized FP4 weight rows [N, K] (for library cross-checks).
void orc_fp4_dequantize_f64(const uint8_t* Bp, const uint8_t* ws, float ws2,
                            double* out, int64_t N, int64_t K, int bs, int threads) {
  build_e4m3_table();
  parallel_for(N, threads, [&](int64_t n) { fp4_decode_row(Bp, ws, ws2, K, bs, n, out + n * K); });
}

void orc_fp8_dequantize_f64(const uint8_t* B, const float* bsc, double* out,
                            int64_t N, int64_t K, int bs, int threads) {
  build_e4m3_table();
  parallel_for(N, threads, [&](int64_t n) { fp8_decode_row(B, bsc, K, bs, n, out + n * K); });
}

// Y_ref = A * dequant(B)^T + bias in float64, and Sabs = sum |A * Bdq|.
void orc_fp4_matmul(const uint16_t* A, const uint8_t* Bp, const uint8_t* ws,
                    float ws2, const uint16_t* bias, int64_t M, int64_t N,
                    int64_t K, int bs, int dtype, double* Y, double* Sabs,
                    int threads) {
  build_e4m3_table();
  matmul_full(A, bias, M, N, K, dtype, Y, Sabs, threads,
              [&](int64_t n, double* row) { fp4_decode_row(Bp, ws, ws2, K, bs, n, row); });
}

void orc_fp8_matmul(const uint16_t* A, const uint8_t* B, const float* bsc,
                    const uint16_t* bias, int64_t M, int64_t N, int64_t K,
                    int bs, int dtype, double* Y, double* Sabs, int threads) {
  build_e4m3_table();
  matmul_full(A, bias, M, N, K, dtype, Y, Sabs, threads,
              [&](int64_t n, double* row) { fp8_decode_row(B, bsc, K, bs, n, row); });
}

void orc_fp4_matmul_sampled(const uint16_t* A, const uint8_t* Bp,
                            const uint8_t* ws, float ws2, const uint16_t* bias,
                            int64_t K, int bs, int dtype, const int64_t* ms,
                            const int64_t* ns, int64_t count, double* Y,
                            double* Sabs, int threads) {
  build_e4m3_table();
  matmul_sampled(A, bias, K, dtype, ms, ns, count, Y, Sabs, threads,
                 [&](int64_t n, double* row) { fp4_decode_row(Bp, ws, ws2, K, bs, n, row); });
}

void orc_fp8_matmul_sampled(const uint16_t* A, const uint8_t* B,
                            const float* bsc, const uint16_t* bias, int64_t K,
                            int bs, int dtype, const int64_t* ms,
                            const int64_t* ns, int64_t count, double* Y,
                            double* Sabs, int threads) {
  build_e4m3_table();
  matmul_sampled(A, bias, K, dtype, ms, ns, count, Y, Sabs, threads,
                 [&](int64_t n, double* row) { fp8_decode_row(B, bsc, K, bs, n, row); });
}

}  // extern "C"
