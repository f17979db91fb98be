// wqmm_device.cuh -- device-side building blocks shared by the kernels:
// bounded mbarrier waits, bulk/tensor copies (TMA), cluster shared memory,
// tcgen05 (TMEM allocation, MMA, loads/stores) and the format decoders.
//
// Formats ("MatMulBlockQuantizedFp4Weight - CUDA Operator Documentation" §2;
// "MatMulBlockQuantizedFp8Weight - CUDA Operator Documentation" §2):
//   NVFP4 byte = two E2M1 codes, low nibble = even k, high nibble = odd k;
//   block scales are raw E4M3FN bytes; FP8 weights are raw E4M3FN bytes.
// Decoding uses the sm_100-family conversion instructions
// cvt.rn.f16x2.e2m1x2 and cvt.rn.f16x2.e4m3x2, which are exact: every E2M1
// and E4M3 value is representable in binary16.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "wqmm_internal.h"

namespace wqmm {

// Records the first error code in the device-side error word `err` (owned by
// the C-ABI translation unit, reported by wqmm_device_status()).
__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Every spin-wait in this library gives up after this much wall time.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// Address helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns
// false (and records WQMM_ERR_TIMEOUT in *err) if the limit runs out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 63u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) break;
  }
  record_error(err, 5 /* WQMM_ERR_TIMEOUT */);
  return false;
}

// ---------------------------------------------------------------------------
// Bulk copies (TMA)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled tensor load into this CTA's shared memory; completes on `bar`.
// x is the innermost coordinate (elements), y the row.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* m, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint (createpolicy result).
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* m, int x,
                                                 int y, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// L2 prefetch of a 2-D tile (no shared-memory write, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* m, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Cluster helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Map a local shared-memory address to the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_f32x4(uint32_t addr, float a, float b, float c,
                                                 float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// ---------------------------------------------------------------------------
// Global loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Streaming loads: read-only path, no L1 allocation (each byte is used once).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// 32-byte load (sm_100 family), evict-first in L2.
__device__ __forceinline__ void ldg_stream_v8(const void* p, uint32_t (&r)[8]) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "l"(p));
}

// Coherent (L2) loads for data another kernel may have just written: no
// read-only or L1 caching.
__device__ __forceinline__ float ld_global_f32(const float* p) {
  float r;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint16_t ld_global_u16(const uint16_t* p) {
  uint16_t r;
  asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ void stg_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// 16-byte streaming store (evict-first): for outputs written once and larger
// than L2.
__device__ __forceinline__ void stg_v4_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------------------
// Format decoders
// ---------------------------------------------------------------------------
// Four packed bytes (eight E2M1 codes) -> four f16x2 words; word j holds the
// codes of byte j, the low nibble in the low half.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Two E4M3 bytes (low byte -> low half) -> f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("{ .reg .b16 h; cvt.u16.u32 h, %1; cvt.rn.f16x2.e4m3x2 %0, h; }" : "=r"(r) : "r"(two_bytes));
  return r;
}

// W8A8 activation path ("MatMulBlockQuantizedFp8Weight - CUDA Operator
// Documentation" §6): A_deq = fp8_e4m3(A / a_scale) * a_scale, for a pair of
// activation values (low half = first).  The division is IEEE float32
// (correctly rounded), the E4M3 conversion rounds to nearest even and
// saturates at +-448 (NaN stays NaN), the product is one float32 rounding,
// then one RNE to the activation type.
template <int DT>
__device__ __forceinline__ float act_bits_to_f32(uint32_t bits16) {
  if constexpr (DT == 1) return __uint_as_float(bits16 << 16);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

template <int DT>
__device__ __forceinline__ uint32_t qdq_fp8_act_pair(uint32_t two, float a_scale) {
  const float lo = __fdiv_rn(act_bits_to_f32<DT>(two & 0xFFFFu), a_scale);
  const float hi = __fdiv_rn(act_bits_to_f32<DT>(two >> 16), a_scale);
  uint32_t q;
  asm("{ .reg .b16 c; cvt.rn.satfinite.e4m3x2.f32 c, %2, %1; cvt.u32.u16 %0, c; }"
      : "=r"(q) : "f"(lo), "f"(hi));
  uint32_t h;
  asm("{ .reg .b16 c; cvt.u16.u32 c, %1; cvt.rn.f16x2.e4m3x2 %0, c; }" : "=r"(h) : "r"(q));
  const float dlo = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
  const float dhi = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
  uint32_t r;
  if constexpr (DT == 1) {
    __nv_bfloat162 v = __floats2bfloat162_rn(__fmul_rn(dlo, a_scale), __fmul_rn(dhi, a_scale));
    r = *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(__fmul_rn(dlo, a_scale), __fmul_rn(dhi, a_scale));
    r = *reinterpret_cast<uint32_t*>(&v);
  }
  return r;
}

// One E4M3 byte -> float (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  const uint32_t h2 = e4m3x2_to_f16x2(byte & 0xFFu);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// f16x2 word -> two floats (exact).
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// float -> f16/bf16 bits, round to nearest even.
template <int DT>
__device__ __forceinline__ uint32_t pack2_rn(float lo, float hi) {
  if constexpr (DT == 1) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <int DT>
__device__ __forceinline__ uint16_t to_act_rn(float x) {
  if constexpr (DT == 1) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return __half_as_ushort(__float2half_rn(x));
}

template <int DT>
__device__ __forceinline__ float act_to_f32(uint16_t bits) {
  if constexpr (DT == 1) return __uint_as_float(static_cast<uint32_t>(bits) << 16);
  else return __half2float(__ushort_as_half(bits));
}

// A decoded f16x2 E2M1 pair times an f16 scale -> 16-bit operand pair (DT).
// Exact: the products have at most 6 significant bits.
template <int DT>
__device__ __forceinline__ uint32_t fold_f16x2(uint32_t h, uint32_t sc16x2) {
  if constexpr (DT == 1) {
    float lo, hi;
    asm("{ .reg .b16 l, u, s, s2; mov.b32 {l, u}, %2; mov.b32 {s, s2}, %3;\n\t"
        "fma.rn.f32.f16 %0, l, s, 0f80000000; fma.rn.f32.f16 %1, u, s, 0f80000000; }"
        : "=f"(lo), "=f"(hi) : "r"(h), "r"(sc16x2));
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  } else {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(sc16x2));  // exact
    return r;
  }
}

}  // namespace wqmm
