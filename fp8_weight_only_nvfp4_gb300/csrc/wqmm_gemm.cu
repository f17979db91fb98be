// wqmm_gemm.cu -- fused dequantize + tcgen05 GEMM for large M (prefill).
//
//   Y[m, n] = gscale * sum_k A[m, k] * w[n, k] (+ bias[n])
//   NVFP4: w = e2m1(B[n, k]) * e4m3(ws[n, k / bs]), gscale = weight_scale_2
//   FP8:   w = e4m3(B[n, k]) * b_scale[n, k / bs], gscale = 1
//
// The pages' prefill path ("MatMulBlockQuantizedFp4Weight - CUDA Operator
// Documentation" §5; "ONNX Runtime #32128 ...") expands B into an [N, K]
// FP16/BF16 scratch tensor and then runs a library GEMM; the blog's closing
// questions ask whether that scratch must exist at all.  Here it does not:
// the packed weight is decoded inside the GEMM main loop, straight into
// tensor memory, and never written back to global memory.
//
// Tile: 128 weight rows (MMA M) x BN tokens (MMA N) per CTA, K in stages of
// 64; BN = 256 for prefill, 128 / 64 / 32 when M fits a narrower tile.
// Roles (one CTA = 2 + 4 PH warps, PH = decoder phases, see Shape below):
//   warp 0     TMA producer: activation tile [BN tokens x 64 k] (128-byte
//              swizzle, K-major) and packed weight tile [128 rows x 64 k]
//              into a shared-memory ring (6 stages for NVFP4 and 5 for FP8
//              at BN = 256, up to 12 for narrower tiles; always a multiple
//              of PH);
//   warp 1     TMEM owner and MMA issuer (one elected thread):
//              tcgen05.mma.kind::f16, A = decoded weight from TMEM,
//              B = activation tile from shared memory, D = FP32 in TMEM;
//   warps 2..  decoders: warp w serves TMEM lane quarter (w % 4) and decodes
//              every PH-th stage in full; thread i of the quarter owns
//              weight row i (TMEM lane i).  It reads its packed bytes from
//              shared memory, folds the E4M3 block scales (exact for NVFP4:
//              <= 6 significant bits, FP4 page §4), writes the 16-bit
//              operands to TMEM with one tcgen05.st, and after the main loop
//              runs the epilogue for its share of the BN token columns: TMEM
//              -> registers, * gscale, + bias, one RNE, then Y (through a
//              shared-memory transpose and one tensor store when the row
//              pitch allows, else direct stores with lanes = consecutive n).
//   split-K    when the tiles fill less than half of the GPU (mid-range M
//              with few weight-row tiles), a cluster of C = 2..4 CTAs along
//              gridDim.z splits K; the FP32 partial tiles are reduce-
//              scattered through distributed shared memory (rank b owns
//              token-column block b and adds the partials in rank order).
//              Measured: without the tensor-memory stores the kernel runs at
//              the speed of the plain MMA pipeline; the stores complete late
//              while the MMA streams, so the PH warps of a quarter keep PH
//              stages in flight instead of splitting one stage's k.
//
// The weight being the MMA A operand is the FP4 page §4 idea (weight in the
// A slot, activation in the B slot) carried to tcgen05: the decoded weight
// never touches shared memory, which keeps shared-memory traffic per MMA to
// the activation tile alone.
//
// Every mbarrier wait is bounded; a wait that runs out raises a CTA-wide
// abort flag, records WQMM_ERR_TIMEOUT, and all roles drain to the TMEM
// release at the end.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "wqmm_tcgen05.cuh"

namespace wqmm {

namespace {

constexpr int kBM = 128;       // weight rows per tile (MMA M)
constexpr int kBK = 64;        // k per stage
constexpr int kAccCol = 0;     // accumulator: columns [0, BN)

// PH = decoder warps per TMEM lane quarter, each taking every PH-th stage (PH
// stages in flight per quarter).  Two shapes of CTA:
//   PH >= 3 one CTA per SM with all 512 tensor-memory columns (prefill tiles,
//           and narrow tiles when the tiles are few);
//   PH = 2  two CTAs per SM, 256 columns and about 100 KB of shared memory
//           each, for the narrow token tiles: there the pace of one CTA's
//           stage loop, not the SM's MMA or decode throughput, bounds the
//           time, and a second resident CTA (with a K split) runs another
//           stage loop beside it.  Four quarter-size CTAs per SM (one decoder
//           warp per lane quarter, 128 columns) were measured no faster than
//           two: from the second one on, the CTAs' common share of the SM
//           sets the pace.
template <int PH>
struct Shape {
  static constexpr int ctas_per_sm = PH == 2 ? 2 : 1;
  static constexpr int dec_warps = 4 * PH;
  static constexpr int threads = (2 + dec_warps) * 32;
  static constexpr int tmem_cols = 512 / ctas_per_sm;
  static constexpr int smem_budget = ctas_per_sm == 1 ? 216 * 1024 : 100 * 1024;
};

// Layout per weight format (KIND 0 = NVFP4, 1 = FP8) and token-tile width BN
// (the MMA N: 256 for prefill, 128 / 64 / 32 for mid-range M, where a
// 256-token tile would spend most of its MMA work on padding rows).  The
// ring holds as many stages as shared memory and tensor memory allow (it has
// to cover the tensor-copy latency): a stage is the activation tile [BN x 64
// k] plus the packed weight tile (4 KB NVFP4, 8 KB FP8) in shared memory and
// 32 tensor-memory columns of decoded operand.
template <int KIND, int BN, int PH>
struct GemmCfg {
  static_assert(BN == 32 || BN == 64 || BN == 128 || BN == 256, "token tile");
  using SH = Shape<PH>;
  static constexpr int act_stage = BN * kBK * 2;
  static constexpr int wstage = KIND == 0 ? kBM * kBK / 2 : kBM * kBK;
  static constexpr int a_col = BN;                         // A stages after the accumulator
  static constexpr int tmem_stages = (SH::tmem_cols - a_col) / (kBK / 2);
  static constexpr int smem_stages = SH::smem_budget / (act_stage + wstage);
  static constexpr int stages0 = tmem_stages < smem_stages ? tmem_stages : smem_stages;
  static constexpr int stages1 = stages0 > 12 ? 12 : stages0;
  // A whole number of turns: a decoder warp waits on a stage's barrier by
  // parity, which is only safe if that barrier's previous phase (the slot's
  // previous fill) has completed.  With stages % PH == 0 the slot's previous
  // fill is this same warp's previous stage, whose wait it has passed; with
  // any other depth it belongs to another warp, and a copy landing out of
  // order would let the wait match the phase two fills back.
  static constexpr int stages = stages1 / PH * PH;
  static constexpr int act = 0;
  static constexpr int w = act + stages * act_stage;
  static constexpr int bars = w + stages * wstage;
  static constexpr int full = bars;
  static constexpr int empty = full + 8 * stages;
  static constexpr int afull = empty + 8 * stages;
  static constexpr int accfull = afull + 8 * stages;
  static constexpr int accempty = accfull + 8;   // persistent kernel only
  static constexpr int tmem_slot = accempty + 8;
  static constexpr int abort_flag = tmem_slot + 4;
  static constexpr int total = abort_flag + 4;
  static constexpr int smem_bytes = total + 1024;  // + alignment slack
  static_assert(stages >= PH && stages % PH == 0, "ring depth");
  static_assert(a_col + stages * (kBK / 2) <= SH::tmem_cols, "TMEM columns");
  static_assert(smem_bytes * SH::ctas_per_sm <= 227 * 1024, "shared memory");
  // The Y staging tile [BN x 128] and the split-K receive slots (at most 3 x
  // BN/4 columns x 128 rows of FP32, rounded up to 8 columns) fit in the
  // activation ring.
  static_assert(BN * kBM * 2 <= stages * act_stage, "Y staging");
  static_assert(3 * ((BN / 4 + 7) / 8 * 8) * kBM * 4 <= stages * act_stage, "split-K slots");
};

// ---------------------------------------------------------------------------
// kind::f16 MMA (the other tcgen05 wrappers are in wqmm_tcgen05.cuh)
// ---------------------------------------------------------------------------
// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16, single CTA, for one 64-k
// stage: four K=16 MMAs into D, A stepping 8 tensor-memory columns
// and B 32 bytes (2 descriptor units) per MMA; the first accumulates only if
// `accumulate`, the others always.
__device__ __forceinline__ void mma_ts_stage(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p, t; .reg .b32 a1, a2, a3; .reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 p, %4, 0; setp.eq.b32 t, %3, %3;\n\t"
      "add.u32 a1, %1, 8; add.u32 a2, %1, 16; add.u32 a3, %1, 24;\n\t"
      "add.u64 b1, %2, 2; add.u64 b2, %2, 4; add.u64 b3, %2, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, t; }" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Instruction descriptor, kind::f16: D = F32, A/B = F16 (0) or BF16 (1),
// both K-major, N = BN, M = 128.
template <int BN>
__host__ __device__ constexpr uint32_t make_idesc(int ab_fmt) {
  return (1u << 4) | ((uint32_t)ab_fmt << 7) | ((uint32_t)ab_fmt << 10) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

// Reads 16 bytes at logical offset `off` of a shared-memory tile written by
// TMA with a 32/64-byte swizzle (16-byte chunk index XOR address bits 7..).
template <int SWZ_MASK>
__device__ __forceinline__ uint4 lds_swz(const uint8_t* tile, uint32_t off) {
  const uint32_t phys = off ^ (((off >> 7) & SWZ_MASK) << 4);
  return *reinterpret_cast<const uint4*>(tile + phys);
}

// Decode one packed NVFP4 word (4 bytes, 8 codes) with one block scale
// (f16 bits, low half) -> 4 words of 16-bit operands (DT) holding
// e2m1 * scale exactly (at most 6 significant bits).
template <int DT>
__device__ __forceinline__ void decode_fp4_word(uint32_t w, uint32_t sc16, uint32_t* out) {
  uint32_t h[4];
  e2m1x8_to_f16x8(w, h);
  const uint32_t sc2 = __byte_perm(sc16, 0, 0x1010);
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = fold_f16x2<DT>(h[i], sc2);
}

// One decoder thread's weight row n over the K range [k_lo, k_lo + num_k)
// stages: its block scales, fetched a turn ahead of use, and the decode of
// one 64-k stage of its packed codes (from the stage's shared-memory weight
// tile) into 32 words of 16-bit MMA operands.
template <int DT, int KIND>
struct RowDecoder {
  const uint8_t* ws_row;
  const float* fs_row;
  int n, N, K, bs, bs_shift, k_lo, num_k;
  // With 16-element blocks and a scale row length that is a multiple of 4,
  // a stage's four scale bytes are one aligned word, all of it in range.
  bool scale_word;
  // FP8 with blocks of 64 or more k: one scale for the whole stage.
  bool scale_one;
  // FP8 weights with FP16 activations: the folded operand e4m3 * b_scale has
  // to stay inside the FP16 range whatever b_scale is (448 * 147 already
  // overflows it).  A decoder thread owns one weight row over its K range, so
  // it divides that row's block scales by the power of two 2^E that brings
  // their largest magnitude into [1, 2) -- exact -- and its accumulator is
  // multiplied by row_pow2 = 2^E afterwards, also exact: every operand then
  // lies within 448 * 2.  1 otherwise.
  float scale_norm, row_pow2;

  __device__ __forceinline__ void init(const uint8_t* ws, const float* fscale, int n_, int N_,
                                       int K_, int bs_, int k_lo_, int num_k_) {
    n = n_;
    N = N_;
    K = K_;
    bs = bs_;
    k_lo = k_lo_;
    num_k = num_k_;
    const int S = (K + bs - 1) / bs;
    bs_shift = ((bs & (bs - 1)) == 0) ? __ffs(bs) - 1 : -1;
    ws_row = ws + (int64_t)n * S;
    fs_row = fscale + (int64_t)n * S;
    scale_word = KIND == 0 && bs == 16 && (S & 3) == 0;
    scale_one = KIND == 1 && (bs & 63) == 0;
    scale_norm = 1.0f;
    row_pow2 = 1.0f;
    if constexpr (KIND == 1 && DT == 0) {
      float rmax = 0.f;
      if (n < N) {
        const int k_begin = k_lo * kBK, k_end = min(K, (k_lo + num_k) * kBK);
        const int c0 = bs_shift >= 0 ? k_begin >> bs_shift : k_begin / bs;
        const int c1 = bs_shift >= 0 ? (k_end - 1) >> bs_shift : (k_end - 1) / bs;
        for (int c = c0; c <= c1; ++c) rmax = fmaxf(rmax, fabsf(__ldg(fs_row + c)));
      }
      // floor(log2(rmax)) for a normal rmax; zero, subnormal, inf and NaN
      // maxima keep E = 0.
      const int e = (int)((__float_as_uint(rmax) >> 23) & 0xFFu) - 127;
      const int ec = (e >= -126 && e <= 126) ? e : 0;
      scale_norm = __uint_as_float((uint32_t)(127 - ec) << 23);
      row_pow2 = __uint_as_float((uint32_t)(127 + ec) << 23);
    }
  }

  // Raw scales of the four 16-k chunks of stage `it` (bs is a multiple of 16);
  // zeros past the range.
  __device__ __forceinline__ void fetch(int it, uint32_t (&r)[4]) const {
    if (scale_one) {
      const int k0 = (k_lo + it) * kBK;
      uint32_t v = 0u;
      if (n < N && it < num_k && k0 < K) {
        const int col = bs_shift >= 0 ? k0 >> bs_shift : k0 / bs;
        v = __float_as_uint(__ldg(fs_row + col));
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) r[c] = v;
      return;
    }
    if (scale_word) {
      const int k0 = (k_lo + it) * kBK;
      uint32_t w = 0u;
      if (n < N && it < num_k && k0 < K)
        w = __ldg(reinterpret_cast<const uint32_t*>(ws_row + (k0 >> 4)));
#pragma unroll
      for (int c = 0; c < 4; ++c) r[c] = (w >> (8 * c)) & 0xFFu;
      return;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int k1 = (k_lo + it) * kBK + 16 * c;
      r[c] = 0u;
      if (n < N && it < num_k && k1 < K) {
        const int col = bs_shift >= 0 ? k1 >> bs_shift : k1 / bs;
        if constexpr (KIND == 0)
          r[c] = __ldg(ws_row + col);
        else
          r[c] = __float_as_uint(__ldg(fs_row + col));
      }
    }
  }

  // Decodes this thread's weight row `row` of the stage tile `wt` with the
  // stage's scales `sc`.
  __device__ __forceinline__ void decode(const uint8_t* wt, int row, const uint32_t (&sc)[4],
                                         uint32_t (&v)[32]) const {
    if constexpr (KIND == 0) {
      // The row's 32-byte stage run (64 k), 32-byte swizzle.
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t off = row * 32 + 16 * h;
        const uint32_t phys = off ^ (((off >> 7) & 1u) << 4);
        const uint4 pw = *reinterpret_cast<const uint4*>(wt + phys);
        const uint32_t sa = e4m3x2_to_f16x2(sc[2 * h]) & 0xFFFFu;
        const uint32_t sb = e4m3x2_to_f16x2(sc[2 * h + 1]) & 0xFFFFu;
        decode_fp4_word<DT>(pw.x, sa, &v[16 * h + 0]);
        decode_fp4_word<DT>(pw.y, sa, &v[16 * h + 4]);
        decode_fp4_word<DT>(pw.z, sb, &v[16 * h + 8]);
        decode_fp4_word<DT>(pw.w, sb, &v[16 * h + 12]);
      }
    } else {
      // The row's 64-byte stage run (64 k), 64-byte swizzle.
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 p = lds_swz<3>(wt, row * 64 + 16 * c);
        const uint32_t w4[4] = {p.x, p.y, p.z, p.w};
        float scf = __uint_as_float(sc[c]);
        if constexpr (DT == 0) scf *= scale_norm;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float2 e = f16x2_to_f32x2(e4m3x2_to_f16x2((w4[i] >> (16 * h)) & 0xFFFFu));
            v[8 * c + 2 * i + h] = pack2_rn<DT>(e.x * scf, e.y * scf);
          }
        }
      }
    }
  }
};

// KIND 0 = NVFP4 weight, 1 = FP8 weight.  DT 0 = FP16, 1 = BF16.  BN =
// tokens per tile (MMA N).
template <int DT, int KIND, int BN, int PH>
__global__ void __launch_bounds__(Shape<PH>::threads, Shape<PH>::ctas_per_sm)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmY, int y_tma,
                   const uint8_t* __restrict__ ws, const float* __restrict__ gscale,
                   const float* __restrict__ fscale, const uint16_t* __restrict__ bias,
                   uint16_t* __restrict__ Y, int M, int N, int K, int bs, int* err) {
  using L = GemmCfg<KIND, BN, PH>;
  constexpr int kStages = L::stages;
  constexpr int kPh = PH;
  constexpr int kTmemCols = Shape<PH>::tmem_cols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L::empty);
  uint64_t* afull = reinterpret_cast<uint64_t*>(smem + L::afull);
  uint64_t* accfull = reinterpret_cast<uint64_t*>(smem + L::accfull);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::tmem_slot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::abort_flag);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBM;
  const int m0 = blockIdx.y * BN;
  const int num_k_all = (K + kBK - 1) / kBK;
  // Split-K across a cluster of C CTAs along gridDim.z: rank r takes stages
  // [k_lo, k_lo + num_k) (the host sizes ranks so that every one has some).
  const int C = gridDim.z;
  const int rank = blockIdx.z;
  const int spc = (num_k_all + C - 1) / C;
  const int k_lo = rank * spc;
  const int num_k = min(num_k_all, k_lo + spc) - k_lo;
  constexpr int kWBytes = (KIND == 0) ? kBK / 2 : kBK;  // packed bytes per row per stage

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&afull[s], 4);  // one decoder warp per lane quarter
    }
    mbar_init(accfull, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool have = false;  // decoder warps: this CTA's accumulator is complete
  // FP8 weights with FP16 activations: 2^E of this decoder thread's weight
  // row, by which its accumulator is multiplied back (1 otherwise).
  float row_pow2 = 1.0f;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint32_t bytes = L::act_stage + kBM * kWBytes;
      int issued = 0;
      for (int it = 0; it < num_k; ++it) {
        const int s = it % kStages;
        if (it >= kStages && !wait_bar(&empty[s], ((it / kStages) + 1) & 1, err, abort_flag)) break;
        mbar_arrive_expect_tx(&full[s], bytes);
        tma_load_2d(smem + L::act + s * L::act_stage, &tmA, (k_lo + it) * kBK, m0, &full[s]);
        tma_load_2d(smem + L::w + s * L::wstage, &tmW, (k_lo + it) * kWBytes, n0, &full[s]);
        ++issued;
      }
      // No copy may still be landing in shared memory when the CTA exits:
      // wait (bounded) for the last use of every stage.  On the normal path
      // these phases completed long ago.
      for (int it = (issued > kStages ? issued - kStages : 0); it < issued; ++it)
        drain_wait(&full[it % kStages], (it / kStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc<BN>(DT == 1 ? 1 : 0);
      bool ok = true;
      int committed = -1;
      // Stage, parity, operand descriptor and tensor-memory address advance
      // by counters: this thread's turn sets the pipeline's pace, so it does
      // as little as possible.
      const uint64_t bdesc0 = desc_kmajor_sw128(smem_u32(smem + L::act));
      const uint32_t afull0 = smem_u32(afull);
      uint64_t bdesc = bdesc0;
      uint32_t a_tmem = tmem + L::a_col;
      int s = 0;
      uint32_t par = 0;
      for (int it = 0; it < num_k; ++it) {
        // afull[s] implies full[s]: every lane quarter's decoder arrives on it
        // only after its own wait on full[s] (the activation and weight
        // copies share that barrier), so the activation tile has landed.
        // One barrier per turn (without the second wait, 1,492 / 1,566 ->
        // 1,590 / 1,667 TFLOP/s at M = 8192).
        if (!mbar_try_wait(afull0 + 8u * (uint32_t)s, par) &&
            !wait_bar(&afull[s], par, err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        static_assert(kBK == 64, "four MMAs of K = 16 per stage");
        mma_ts_stage(tmem + kAccCol, a_tmem, bdesc, idesc, it > 0 ? 1u : 0u);
        mma_commit(&empty[s]);
        committed = it;
        if (++s == kStages) {
          s = 0;
          par ^= 1u;
          bdesc = bdesc0;
          a_tmem = tmem + L::a_col;
        } else {
          bdesc += (uint64_t)(L::act_stage >> 4);
          a_tmem += kBK / 2;
        }
      }
      if (ok) {
        mma_commit(accfull);
      } else if (committed >= 0) {
        // MMAs still reading TMEM must finish before the release below.
        drain_wait(&empty[committed % kStages], (committed / kStages) & 1);
      }
    }
  } else {
    // ---------------- decoders, then epilogue ----------------
    // Warp w serves TMEM lane quarter q = w % 4 and decodes every PH-th
    // stage (phase j = (w - 2) / 4) in full: the PH warps of a quarter have
    // PH stages in flight, so the latency of one warp's stage (shared load,
    // decode, tensor-memory store, which completes late while the MMA
    // streams) is spread over PH stages.  The ring depth is a multiple of
    // PH, so a warp's parity wait on a slot always follows its own wait on
    // the slot's previous fill.
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int j4 = (warp - 2) >> 2;         // stage phase of this warp
    const int row = q * 32 + lane;          // weight row within the tile
    const int n = n0 + row;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    RowDecoder<DT, KIND> rd;
    rd.init(ws, fscale, n, N, K, bs, k_lo, num_k);
    row_pow2 = rd.row_pow2;
    uint32_t scn[4];
    rd.fetch(j4, scn);  // (j4 = this warp's stage phase, 0 .. kPh - 1)
    bool ok = true;
    for (int it = j4; it < num_k; it += kPh) {
      const int s = it % kStages;
      uint32_t sc[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) sc[c] = scn[c];
      rd.fetch(it + kPh, scn);
      if (!wait_bar(&full[s], (it / kStages) & 1, err, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[32];
      rd.decode(smem + L::w + s * L::wstage, row, sc, v);
      tmem_st32(lane_base + L::a_col + s * (kBK / 2), v);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[s]);  // one arrival per lane quarter
    }
    // Epilogue: this warp's lane quarter, token-column chunks j4, j4 + kPh, ...
    // With a tensor map for Y the tile is staged transposed, [BN tokens x
    // 128 n], in the (now idle) activation ring and written by one tensor
    // store; otherwise each column is stored directly (lanes = consecutive n).
    have = ok && wait_bar(accfull, 0, err, abort_flag) && !*abort_flag;
    if (have && C == 1) {
      tc_fence_after();
      const float gs = (KIND == 0) ? __ldg(gscale) : row_pow2;
      const float b = (bias != nullptr && n < N) ? act_to_f32<DT>(__ldg(bias + n)) : 0.0f;
      uint16_t* stage_y = reinterpret_cast<uint16_t*>(smem + L::act);
      constexpr int kCh = BN / 4 < 32 ? BN / 4 : 32;  // columns per tensor-memory load
#pragma unroll 1
      for (int c0 = kCh * j4; c0 < BN; c0 += kCh * kPh) {
        uint32_t r[kCh];
        tmem_ld_cols<kCh>(lane_base + kAccCol + c0, r);
        if (y_tma) {
#pragma unroll
          for (int j = 0; j < kCh; ++j)
            stage_y[(c0 + j) * kBM + row] = to_act_rn<DT>(__uint_as_float(r[j]) * gs + b);
        } else if (n < N) {
#pragma unroll
          for (int j = 0; j < kCh; ++j) {
            const int m = m0 + c0 + j;
            if (m < M) Y[(int64_t)m * N + n] = to_act_rn<DT>(__uint_as_float(r[j]) * gs + b);
          }
        }
      }
    }
    if (y_tma && C == 1) {
      // Make the staged tile visible to the tensor-copy engine, then one
      // elected thread stores it (out-of-range rows and columns are clipped).
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("bar.sync 1, %0;" ::"n"(Shape<PH>::dec_warps * 32) : "memory");
      if (have && warp == 2 && lane == 0 && !*abort_flag) {
        asm volatile(
            "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                reinterpret_cast<uint64_t>(&tmY)),
            "r"(n0), "r"(m0), "r"(smem_u32(smem + L::act))
            : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      }
    }
  }

  // Split-K: reduce-scatter of the FP32 partial tiles through distributed
  // shared memory.  Token columns are cut into C blocks (multiples of 8);
  // rank b owns block b: every other rank writes its partial of that block
  // into rank b's (now idle) activation ring, then rank b adds them in rank
  // order to its own and runs the epilogue for the block.  Deterministic, no
  // global scratch.
  if (C > 1) {
    __syncwarp();
    cluster_sync();  // every rank's MMAs are complete and its rings are idle
    const int wmax = (BN / C + 7) / 8 * 8;
    auto block_lo = [&](int bb) { return min(BN, bb * wmax); };
    // [C-1 slots][wmax columns][128 rows]: lanes (consecutive rows) write and
    // read consecutive words, one 128-byte line per warp access.
    float* recv = reinterpret_cast<float*>(smem + L::act);
    if (warp >= 2 && have) {
      const int q = warp & 3, j4 = (warp - 2) >> 2;
      const int row = q * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
      tc_fence_after();
      for (int bb = 0; bb < C; ++bb) {
        if (bb == rank) continue;
        const int c_lo = block_lo(bb), w = block_lo(bb + 1) - c_lo;
        const int slot = rank < bb ? rank : rank - 1;
        // This warp: the block's 8-column chunks j4, j4 + kPh, ...
        for (int c8 = 8 * j4; c8 < w; c8 += 8 * kPh) {
          uint32_t r[8];
          tmem_ld8(lane_base + kAccCol + c_lo + c8, r);
          const uint32_t remote =
              mapa_shared(smem_u32(recv + ((size_t)slot * wmax + c8) * kBM + row), (uint32_t)bb);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_cluster_f32(remote + 4u * kBM * j, __uint_as_float(r[j]) * row_pow2);
        }
      }
    }
    // A rank whose wait ran out tells every other rank: then no rank stores
    // (Y is left untouched after WQMM_ERR_TIMEOUT).
    if (threadIdx.x == 0 && *abort_flag) {
      for (int bb = 0; bb < C; ++bb)
        if (bb != rank)
          st_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), (uint32_t)bb), 1u);
    }
    cluster_sync();  // every partial has arrived
    if (warp >= 2 && have && !*abort_flag) {
      const int q = warp & 3, j4 = (warp - 2) >> 2;
      const int row = q * 32 + lane;
      const int n = n0 + row;
      const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
      tc_fence_after();
      const float gs = (KIND == 0) ? __ldg(gscale) : 1.0f;
      const float bv = (bias != nullptr && n < N) ? act_to_f32<DT>(__ldg(bias + n)) : 0.0f;
      const int c_lo = block_lo(rank), w = block_lo(rank + 1) - c_lo;
      for (int c8 = 8 * j4; c8 < w; c8 += 8 * kPh) {
        uint32_t r[8];
        tmem_ld8(lane_base + kAccCol + c_lo + c8, r);
        // Rank order: partials of ranks 0 .. C-1, this rank's own in place.
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
        for (int src = 0; src < C; ++src) {
          if (src == rank) {
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += __uint_as_float(r[j]) * row_pow2;
          } else {
            const int slot = src < rank ? src : src - 1;
            const float* pv = recv + ((size_t)slot * wmax + c8) * kBM + row;
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = pv[j * kBM];  // independent loads
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += v[j];
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int m = m0 + c_lo + c8 + j;
          if (n < N && m < M) Y[(int64_t)m * N + n] = to_act_rn<DT>(acc[j] * gs + bv);
        }
      }
    }
  }

  // Teardown: every tcgen05 access of this CTA is complete before the release.
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Persistent form of gemm_tc_kernel for the 256-token prefill tile without a
// K split: one CTA per SM walks the tiles blockIdx.x, blockIdx.x + gridDim.x,
// ... (NVFP4: weight-row tiles fastest; FP8: bands of token tiles, see the
// walk below).  Producer, decoders and MMA run on across
// tile boundaries -- the producer keeps filling the ring with the next tile's
// stages while the current one finishes -- and the decoders run each tile's
// epilogue as soon as their own last stage of it is done: they read their
// accumulator columns, hand the accumulator back to the MMA thread (the first
// MMA of the next tile waits for that), store Y directly (lanes = consecutive
// weight rows, 64 bytes per warp store) and go on decoding.  A CTA per tile
// paid about 6 us per tile outside its main loop (start-up, pipeline fill and
// an epilogue that overlapped nothing; a K sweep at M = 8192, N = 17408).
template <int DT, int KIND, int PH>
__global__ void __launch_bounds__(Shape<PH>::threads, 1)
    gemm_tc_persist(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                    const uint8_t* __restrict__ ws, const float* __restrict__ gscale,
                    const float* __restrict__ fscale, const uint16_t* __restrict__ bias,
                    uint16_t* __restrict__ Y, int M, int N, int K, int bs, int tiles_n, int tiles,
                    int* err) {
  constexpr int BN = 256;
  using L = GemmCfg<KIND, BN, PH>;
  constexpr int kStages = L::stages;
  constexpr int kPh = PH;
  constexpr int kTmemCols = Shape<PH>::tmem_cols;
  constexpr int kDec = Shape<PH>::dec_warps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L::empty);
  uint64_t* afull = reinterpret_cast<uint64_t*>(smem + L::afull);
  uint64_t* accfull = reinterpret_cast<uint64_t*>(smem + L::accfull);
  uint64_t* accempty = reinterpret_cast<uint64_t*>(smem + L::accempty);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::tmem_slot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::abort_flag);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_k = (K + kBK - 1) / kBK;
  const int my_tiles = (int)blockIdx.x < tiles
                           ? (tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                           : 0;
  // Tile t of the walk.  An NVFP4 weight (about 50 MB at 17408 x 5120 with
  // its scales) stays in L2 while the token tiles pass over it, so weight
  // tiles run fastest.  An FP8 weight has twice the bytes and did not: at
  // M = 2048 the kernel read 572 MB from DRAM for 113 MB of operands, the
  // whole weight once per token tile.  FP8 therefore walks bands of kBand
  // token tiles with the token tiles fastest, so the CTAs in flight share
  // each weight tile through L2 (W8A8 at M = 8192, N = 17408, K = 5120:
  // 1,067 -> 1,012 us; the same walk for NVFP4: 873 -> 883 us).
  constexpr int kBand = KIND == 1 ? 8 : 0;
  const int tiles_m = tiles / tiles_n;
  auto tile_nm = [&](int i, int& nt, int& mt) {
    const int t = (int)blockIdx.x + i * (int)gridDim.x;
    if constexpr (kBand == 0) {
      nt = t % tiles_n;
      mt = t / tiles_n;
    } else {
      const int band = t / (tiles_n * kBand);
      const int r = t - band * tiles_n * kBand;
      const int gm = min(kBand, tiles_m - band * kBand);
      nt = r / gm;
      mt = band * kBand + r % gm;
    }
  };
  auto tile_n0 = [&](int i) { int nt, mt; tile_nm(i, nt, mt); return nt * kBM; };
  auto tile_m0 = [&](int i) { int nt, mt; tile_nm(i, nt, mt); return mt * BN; };
  constexpr int kWBytes = (KIND == 0) ? kBK / 2 : kBK;  // packed bytes per row per stage

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&afull[s], 4);  // one decoder warp per lane quarter
    }
    mbar_init(accfull, 1);
    mbar_init(accempty, kDec);  // every decoder warp has read its columns
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint32_t bytes = L::act_stage + kBM * kWBytes;
      int g = 0;  // stages issued (ring slot g % kStages, fill g / kStages)
      bool ok = true;
      for (int i = 0; i < my_tiles && ok; ++i) {
        const int n0 = tile_n0(i), m0 = tile_m0(i);
        for (int it = 0; it < num_k; ++it, ++g) {
          const int s = g % kStages;
          if (g >= kStages && !wait_bar(&empty[s], ((g / kStages) + 1) & 1, err, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], bytes);
          tma_load_2d(smem + L::act + s * L::act_stage, &tmA, it * kBK, m0, &full[s]);
          tma_load_2d(smem + L::w + s * L::wstage, &tmW, it * kWBytes, n0, &full[s]);
        }
      }
      for (int it = (g > kStages ? g - kStages : 0); it < g; ++it)
        drain_wait(&full[it % kStages], (it / kStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc<BN>(DT == 1 ? 1 : 0);
      bool ok = true;
      int committed = -1;
      const uint64_t bdesc0 = desc_kmajor_sw128(smem_u32(smem + L::act));
      const uint32_t afull0 = smem_u32(afull);
      uint64_t bdesc = bdesc0;
      uint32_t a_tmem = tmem + L::a_col;
      int s = 0, g = 0;
      uint32_t par = 0;
      for (int i = 0; i < my_tiles && ok; ++i) {
        // The accumulator is free once the decoders have read tile i - 1.
        if (i > 0 && !wait_bar(accempty, (i - 1) & 1, err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int it = 0; it < num_k; ++it, ++g) {
          if (!mbar_try_wait(afull0 + 8u * (uint32_t)s, par) &&
              !wait_bar(&afull[s], par, err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_ts_stage(tmem + kAccCol, a_tmem, bdesc, idesc, it > 0 ? 1u : 0u);
          mma_commit(&empty[s]);
          committed = g;
          if (++s == kStages) {
            s = 0;
            par ^= 1u;
            bdesc = bdesc0;
            a_tmem = tmem + L::a_col;
          } else {
            bdesc += (uint64_t)(L::act_stage >> 4);
            a_tmem += kBK / 2;
          }
        }
        if (ok) mma_commit(accfull);  // tile i's accumulator is complete
      }
      if (!ok && committed >= 0)
        drain_wait(&empty[committed % kStages], (committed / kStages) & 1);
    }
  } else {
    // ---------------- decoders, each tile's epilogue ----------------
    // A warp that has finished its stages of tile i first decodes its first
    // stage of tile i + 1 (those stages depend only on tile i's MMAs, never
    // on its epilogue), then runs tile i's epilogue: when the accumulator is
    // handed back, the MMA finds the next tile's first stages ready.
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int j4 = (warp - 2) >> 2;         // stage phase of this warp
    const int row = q * 32 + lane;          // weight row within the tile
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const int total = my_tiles * num_k;
    // Epilogue of tile e.
    auto epilogue = [&](int e) -> bool {
      if (!wait_bar(accfull, e & 1, err, abort_flag)) return false;
      tc_fence_after();
      const int n = tile_n0(e) + row, m0 = tile_m0(e);
      float gs = 1.0f;
      if constexpr (KIND == 0) {
        gs = __ldg(gscale);
      } else if constexpr (DT == 0) {
        // The power of two this row's FP8 block scales were divided by.
        RowDecoder<DT, KIND> t;
        t.init(ws, fscale, n, N, K, bs, 0, num_k);
        gs = t.row_pow2;
      }
      const float b = (bias != nullptr && n < N) ? act_to_f32<DT>(__ldg(bias + n)) : 0.0f;
#pragma unroll 1
      for (int c0 = 32 * j4; c0 < BN; c0 += 32 * kPh) {
        uint32_t r[32];
        tmem_ld32(lane_base + kAccCol + c0, r);
        if (c0 + 32 * kPh >= BN) {
          // This warp's last read of the accumulator: hand it back.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(accempty);
        }
        if (n < N) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int m = m0 + c0 + j;
            if (m < M) Y[(int64_t)m * N + n] = to_act_rn<DT>(__uint_as_float(r[j]) * gs + b);
          }
        }
      }
      return true;
    };
    RowDecoder<DT, KIND> rd;
    int cur = -1;   // tile rd is set up for
    int owed = 0;   // next tile whose epilogue this warp has not run
    uint32_t scn[4];
    bool ok = true;
    for (int g = j4; g < total && ok; g += kPh) {
      const int i = g / num_k, it = g - i * num_k;
      if (i != cur) {
        rd.init(ws, fscale, tile_n0(i) + row, N, K, bs, 0, num_k);
        cur = i;
        rd.fetch(it, scn);
      }
      const int s = g % kStages;
      uint32_t sc[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) sc[c] = scn[c];
      rd.fetch(it + kPh, scn);
      if (!wait_bar(&full[s], (g / kStages) & 1, err, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[32];
      rd.decode(smem + L::w + s * L::wstage, row, sc, v);
      tmem_st32(lane_base + L::a_col + s * (kBK / 2), v);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[s]);  // one arrival per lane quarter
      // Epilogues owed for the tiles before this stage's tile (more than one
      // when a warp has no stage in some tile, num_k < kPh).
      while (ok && owed < i) ok = epilogue(owed++);
    }
    while (ok && owed < my_tiles) ok = epilogue(owed++);
  }

  // Teardown: every tcgen05 access of this CTA is complete before the release.
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int DT, int KIND, int PH>
int launch_persist(const GemvArgs& a, cudaStream_t st) {
  constexpr int BN = 256;
  const int wbytes_per_stage = (KIND == 0) ? kBK / 2 : kBK;
  CUtensorMap tmA, tmW;
  const CUtensorMapDataType adt =
      DT == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (!encode_tmap_2d(&tmA, adt, a.A, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.K * 2, kBK, BN,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return kCuda;
  const uint64_t wrow = (KIND == 0) ? (uint64_t)a.K / 2 : (uint64_t)a.K;
  if (!encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, wrow, (uint64_t)a.N, wrow,
                      wbytes_per_stage, kBM,
                      KIND == 0 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return kCuda;
  using L = GemmCfg<KIND, BN, PH>;
  using SH = Shape<PH>;
  static std::once_flag once[64];
  const int dev = device_info().device;
  if (dev < 0 || dev >= 64) return kCuda;
  std::call_once(once[dev], [] {
    cudaFuncSetAttribute(gemm_tc_persist<DT, KIND, PH>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::smem_bytes);
  });
  const int64_t tiles_n = (a.N + kBM - 1) / kBM;
  const int64_t tiles = tiles_n * ((a.M + BN - 1) / BN);
  const int grid = (int)std::min<int64_t>(tiles, device_info().sm_count);
  gemm_tc_persist<DT, KIND, PH><<<grid, SH::threads, L::smem_bytes, st>>>(
      tmA, tmW, a.ws, a.gscale, a.fscale, reinterpret_cast<const uint16_t*>(a.bias),
      reinterpret_cast<uint16_t*>(a.Y), (int)a.M, (int)a.N, (int)a.K, a.bs, (int)tiles_n,
      (int)tiles, device_error_word());
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}

template <int DT, int KIND, int BN, int PH>
int launch_t(const GemvArgs& a, cudaStream_t st) {
  const int wbytes_per_stage = (KIND == 0) ? kBK / 2 : kBK;
  CUtensorMap tmA, tmW;
  const CUtensorMapDataType adt =
      DT == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (!encode_tmap_2d(&tmA, adt, a.A, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.K * 2, kBK, BN,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return kCuda;
  const uint64_t wrow = (KIND == 0) ? (uint64_t)a.K / 2 : (uint64_t)a.K;
  if (!encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, wrow, (uint64_t)a.N, wrow,
                      wbytes_per_stage, kBM,
                      KIND == 0 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return kCuda;
  // Y through a tensor store when its rows are 16-byte multiples.
  CUtensorMap tmY;
  int y_tma = 0;
  std::memset(&tmY, 0, sizeof(tmY));
  if (a.N % 8 == 0)
    y_tma = encode_tmap_2d(&tmY, adt, a.Y, (uint64_t)a.N, (uint64_t)a.M, (uint64_t)a.N * 2, kBM,
                           BN, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE)
                ? 1
                : 0;
  using L = GemmCfg<KIND, BN, PH>;
  using SH = Shape<PH>;
  // The shared-memory opt-in is a per-device function attribute.
  static std::once_flag once[64];
  const int dev = device_info().device;
  if (dev < 0 || dev >= 64) return kCuda;
  std::call_once(once[dev], [] {
    cudaFuncSetAttribute(gemm_tc_kernel<DT, KIND, BN, PH>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::smem_bytes);
  });
  const int64_t tiles_n = (a.N + kBM - 1) / kBM, tiles_m = (a.M + BN - 1) / BN;
  const int64_t tiles = tiles_n * tiles_m;
  const int num_k = (int)((a.K + kBK - 1) / kBK);
  const int sms = device_info().sm_count;
  // Split-K (cluster of C CTAs along z) when the tiles fill less than half
  // of the resident CTA slots.
  const int64_t slots = (int64_t)sms * SH::ctas_per_sm;
  int C = 1;
  if (tiles * 2 <= slots) {
    for (int c = 4; c >= 2; --c) {
      if (tiles * c <= slots && num_k >= 8 * c) {
        C = c;
        break;
      }
    }
    if (C > 1) {
      const int spc = (num_k + C - 1) / C;
      C = (num_k + spc - 1) / spc;
    }
    // The receive slots of the reduce-scatter live in the activation ring.
    while (C > 1 && (C - 1) * ((BN / C + 7) / 8 * 8) * kBM * 4 > L::stages * L::act_stage) --C;
  }
  const dim3 grid((unsigned)tiles_n, (unsigned)tiles_m, (unsigned)C);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(SH::threads, 1, 1);
  cfg.dynamicSmemBytes = L::smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)C;
  cfg.attrs = attr;
  cfg.numAttrs = C > 1 ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, gemm_tc_kernel<DT, KIND, BN, PH>, tmA, tmW, tmY, y_tma, a.ws, a.gscale, a.fscale,
      reinterpret_cast<const uint16_t*>(a.bias), reinterpret_cast<uint16_t*>(a.Y), (int)a.M,
      (int)a.N, (int)a.K, a.bs, device_error_word());
  return e == cudaSuccess ? kOk : kCuda;
}

// Token-tile width by M: the narrowest MMA N that covers M in one tile up to
// 128 tokens (a wider tile multiplies padding rows), 256 above that (one
// decode of the weight tile feeds the most tokens).
int pick_bn(int64_t M) {
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

// Decoder phases of the full CTA at the 256-token tile, per weight format:
// the ring depth is the largest multiple of the phase count that fits, so
// the counts that divide the deepest rings (6 stages NVFP4, 5 FP8) keep them.
// Measured at M = 8192 (TFLOP/s gate/up / down, FP8): 3 phases x 6 stages
// 1,606 / 1,666; 6 x 6 1,598 / 1,673; 4 x 4 1,549 / 1,472; FP8 5 x 5 1,380,
// 4 x 4 1,135.
constexpr int kFullPh256[2] = {3, 5};

// CTA shape for a narrow token tile: when the tiles alone fill at least half
// of the SMs, two light CTAs per SM (each with a K split of its own); with
// fewer tiles, one full CTA per SM and a wider K split.  Measured (µs, M = 64
// / 128): N = 17408 (136 tiles) 36.0 / 36.2 full, 27.9 / 30.5 light; N = 5120
// (40 tiles) 16.6 / 17.7 full, 16.7 / 19.1 light.
template <int DT, int KIND, int BN>
int launch_narrow(const GemvArgs& a, cudaStream_t st) {
  const int64_t tiles = ((a.N + kBM - 1) / kBM) * ((a.M + BN - 1) / BN);
  if (tiles * 2 > device_info().sm_count) return launch_t<DT, KIND, BN, 2>(a, st);
  return launch_t<DT, KIND, BN, 4>(a, st);
}

template <int DT, int KIND>
int launch_bn(const GemvArgs& a, cudaStream_t st) {
  switch (pick_bn(a.M)) {
    case 32: return launch_narrow<DT, KIND, 32>(a, st);
    case 64: return launch_narrow<DT, KIND, 64>(a, st);
    case 128: return launch_narrow<DT, KIND, 128>(a, st);
    default: {
      // Enough 256-token tiles to fill the GPU without a K split: the
      // persistent kernel; fewer: one CTA per tile with a cluster K split.
      const int64_t tiles = ((a.N + kBM - 1) / kBM) * ((a.M + 255) / 256);
      if (tiles * 2 > device_info().sm_count)
        return launch_persist<DT, KIND, kFullPh256[KIND]>(a, st);
      return launch_t<DT, KIND, 256, kFullPh256[KIND]>(a, st);
    }
  }
}

}  // namespace

bool gemm_prefers_light(const GemvArgs& a) {
  const int bn = pick_bn(a.M);
  if (bn > 128) return false;
  const int64_t tiles = ((a.N + kBM - 1) / kBM) * ((a.M + bn - 1) / bn);
  return tiles * 2 > device_info().sm_count;
}

bool gemm_supports(const GemvArgs& a) {
  const DeviceInfo& d = device_info();
  if (d.cc_major != 10) return false;
  constexpr int kMaxSmem = GemmCfg<1, 256, 4>::smem_bytes;
  if (d.max_smem_optin < kMaxSmem) return false;
  if (a.M <= 8 || a.M >= (int64_t(1) << 31) || a.N >= (int64_t(1) << 31)) return false;
  if (a.bs % 16 != 0) return false;
  if (a.kind == 0) return a.K % 32 == 0;   // packed row stride must be a multiple of 16 bytes
  return a.K % 16 == 0;                    // FP8 row stride must be a multiple of 16 bytes
}

int launch_gemm(const GemvArgs& a, cudaStream_t st) {
  if (!gemm_supports(a)) return kUnsupported;
  if (a.kind == 0)
    return a.dtype == 1 ? launch_bn<1, 0>(a, st) : launch_bn<0, 0>(a, st);
  return a.dtype == 1 ? launch_bn<1, 1>(a, st) : launch_bn<0, 1>(a, st);
}

}  // namespace wqmm
