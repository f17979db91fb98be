// wqmm_gemm_f4f4.cu -- NVFP4 x NVFP4 block-scaled tensor-core GEMM.
//
//   Y[m, n] = weight_scale_2 * sum_k e2m1(Aq[m, k]) e4m3(As[m, k / 16])
//                                  * e2m1(B[n, k])  e4m3(ws[n, k / 16])   (+ bias[n])
//
// Steps 2 and 3 of the native FP4 x FP4 path of "MatMulBlockQuantizedFp4Weight
// - CUDA Operator Documentation" §6 (step 1, quantizing the activation to
// NVFP4, is wqmm_actq.cu): both operands stay packed E2M1 from global memory
// to the tensor core, and the block-scaled MMA of the sm_100 family
// (tcgen05.mma.kind::mxf4nvf4, 16-element blocks, unsigned E4M3 scales)
// applies both operands' block scales itself; products are exact and
// accumulate in FP32.  The page runs a CUTLASS kernel on SM120 and prepacks
// the weight scales into that kernel's layout; here the scales keep the plain
// [rows, K/16] layout of the weight format and are rearranged on chip (a
// prepacked variant whose MMA thread copied them to tensor memory with
// tcgen05.cp gave the same result but took 429 instead of 318 us at
// M = 8192: those copies share the in-order tensor pipe with the MMAs).
//
// Tile: 128 weight rows (MMA M) x 256 tokens (MMA N); K in stages of 256
// (one 128-byte swizzled row of packed codes per operand row), four MMAs of
// K = 64 per stage.  Persistent: one CTA per SM walks the tiles t = blockIdx.x,
// blockIdx.x + gridDim.x, ... (weight-row tiles fastest), and its stage ring,
// scale writers and MMA run on without a break from one tile to the next; only
// the first MMA of a tile waits until the epilogue warps have read the
// previous tile's accumulator out of tensor memory.  (Measured at M = 8192,
// N = 17408: one CTA per tile paid about 6 us per tile outside the main loop
// -- start-up, pipeline fill, epilogue -- 42 % of the time at K = 5120.  A
// cluster of 2 or 4 CTAs sharing the token tile through multicast copies, which
// cuts the L2 traffic per SM by a third or a half, was 13 % / 18 % slower.)
// Roles (14 warps):
//   warp 0      TMA producer: per stage the packed weight tile [128 x 128 B]
//               and activation tile [256 x 128 B] (K-major, 128-byte swizzle)
//               and their scale tiles [128 x 16 B] and [256 x 16 B];
//   warp 1      TMEM owner and MMA issuer (one elected thread);
//   warps 2-5   scale writers: warp w serves TMEM lane quarter w % 4 and moves
//               every stage's scale bytes from shared memory to tensor memory
//               in the layout the block-scaled MMA reads (below) with
//               tcgen05.st (one or two writer warps per quarter measured the
//               same);
//   warps 6-13  epilogue: warp w serves lane quarter w % 4 and half of the 256
//               token columns: TMEM -> registers, * weight_scale_2, + bias, one
//               RNE into packed pairs; it hands the accumulator back after its
//               last tensor-memory load and only then stores to Y (lanes =
//               consecutive weight rows n, 64 bytes per warp store).  Handing
//               it back before the stores: 349 -> 324 us at M = 8192.
//
// Scale factors in tensor memory (scale_vec::4X): one 32-bit cell per operand
// row and 64-k chunk, byte i holding the scale of the chunk's i-th 16-element
// block.  The cells of operand row r sit in lane r % 32 and column r / 32 of
// the chunk's column group (4 columns for the 128 weight rows, 8 for the 256
// tokens: rows 128..255 in the upper 4), and every lane quarter holds the same
// copy.
//
// Every mbarrier wait is bounded; a wait that runs out raises a CTA-wide
// abort flag, records WQMM_ERR_TIMEOUT and all roles drain to the TMEM
// release at the end.
#include <algorithm>
#include <mutex>

#include "wqmm_tcgen05.cuh"

namespace wqmm {

namespace {

constexpr int kBM = 128;              // weight rows per tile (MMA M)
constexpr int kBN = 256;              // tokens per tile (MMA N)
constexpr int kBK = 256;              // k per stage
constexpr int kRowBytes = kBK / 2;    // packed bytes per operand row per stage
constexpr int kScBytes = kBK / 16;    // scale bytes per operand row per stage
constexpr int kStages = 4;
constexpr int kPh = 1;                // scale-writer warps per TMEM lane quarter
constexpr int kWriters = 4 * kPh;
constexpr int kEpi = 8;               // epilogue warps: 4 lane quarters x 2 column halves
constexpr int kWarpEpi0 = 2 + kWriters;
constexpr int kThreads = (2 + kWriters + kEpi) * 32;
constexpr int kTmemCols = 512;

// Shared memory (offsets from a 1024-byte aligned base).
constexpr int kActTile = kBN * kRowBytes;   // 32 KB
constexpr int kWTile = kBM * kRowBytes;     // 16 KB
constexpr int kActSc = kBN * kScBytes;      // 4 KB
constexpr int kWSc = kBM * kScBytes;        // 2 KB
constexpr int kOffAct = 0;
constexpr int kOffW = kOffAct + kStages * kActTile;
constexpr int kOffActSc = kOffW + kStages * kWTile;
constexpr int kOffWSc = kOffActSc + kStages * kActSc;
constexpr int kOffFull = kOffWSc + kStages * kWSc;
constexpr int kOffEmpty = kOffFull + 8 * kStages;
constexpr int kOffReady = kOffEmpty + 8 * kStages;
constexpr int kOffAcc = kOffReady + 8 * kStages;
constexpr int kOffAccEmpty = kOffAcc + 8;
constexpr int kOffSlot = kOffAccEmpty + 8;
constexpr int kOffAbort = kOffSlot + 4;
constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack
constexpr uint32_t kStageBytes = kActTile + kWTile + kActSc + kWSc;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(kStages % kPh == 0, "a writer's parity wait follows its own previous wait");

// Tensor memory: accumulator [0, 256); per stage the token scales (8 columns
// per 64-k chunk, 32 per stage) and the weight scales (4 per chunk, 16 per
// stage).
constexpr int kColAcc = 0;
constexpr int kColSfb = kBN;
constexpr int kColSfa = kColSfb + kStages * 32;
static_assert(kColSfa + kStages * 16 <= kTmemCols, "TMEM columns");

// Instruction descriptor, kind::mxf4nvf4: A (weight) and B (tokens) E2M1
// (format code 1), both K-major, unsigned-E4M3 scale factors (scale type 0),
// scale-factor ids 0, N = 256, M = 128, D = FP32.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

// One stage: four block-scaled MMAs of K = 64, A and B stepping 32 bytes (2
// descriptor units) along their swizzled rows, the weight scales 4 columns and
// the token scales 8 columns per MMA; the first MMA accumulates only if
// `accumulate`.
__device__ __forceinline__ void mma_f4_stage(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p, t; .reg .b64 a1, a2, a3, b1, b2, b3; .reg .b32 sa1, sa2, sa3, sb1, sb2, sb3;\n\t"
      "setp.ne.b32 p, %5, 0; setp.eq.b32 t, %5, %5;\n\t"
      "add.u64 a1, %1, 2; add.u64 a2, %1, 4; add.u64 a3, %1, 6;\n\t"
      "add.u64 b1, %2, 2; add.u64 b2, %2, 4; add.u64 b3, %2, 6;\n\t"
      "add.u32 sa1, %3, 4; add.u32 sa2, %3, 8; add.u32 sa3, %3, 12;\n\t"
      "add.u32 sb1, %4, 8; add.u32 sb2, %4, 16; add.u32 sb3, %4, 24;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %6, [%3], [%4], p;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %6, [sa1], [sb1], t;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a2, b2, %6, [sa2], [sb2], t;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a3, b3, %6, [sa3], [sb3], t; }"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(sfa), "r"(sfb), "r"(accumulate), "r"(kIdesc)
      : "memory");
}

// GSC: scales from global memory (K % 256 != 0), a separate instantiation so
// that the tensor-copy path keeps its code unchanged.
template <int DT, bool GSC>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_f4f4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmAS, const __grid_constant__ CUtensorMap tmWS,
                     const uint8_t* __restrict__ as_g, const uint8_t* __restrict__ ws_g,
                     const float* __restrict__ gscale, const uint16_t* __restrict__ bias,
                     uint16_t* __restrict__ Y, int M, int N, int K, int tiles_n, int tiles,
                     int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffFull);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + kOffEmpty);
  uint64_t* ready = reinterpret_cast<uint64_t*>(smem + kOffReady);
  uint64_t* accfull = reinterpret_cast<uint64_t*>(smem + kOffAcc);
  uint64_t* accempty = reinterpret_cast<uint64_t*>(smem + kOffAccEmpty);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_k = (K + kBK - 1) / kBK;  // a partial last stage reads zero codes past K
  const int S = K / 16;                      // scale columns (K % 32 == 0)
  // This CTA's tiles: blockIdx.x + i * gridDim.x for i < my_tiles.
  const int my_tiles = (int)blockIdx.x < tiles
                           ? (tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                           : 0;
  const int total = my_tiles * num_k;  // stages this CTA runs
  auto tile_n0 = [&](int i) { return ((int)blockIdx.x + i * (int)gridDim.x) % tiles_n * kBM; };
  auto tile_m0 = [&](int i) { return ((int)blockIdx.x + i * (int)gridDim.x) / tiles_n * kBN; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&ready[s], 4);   // one writer warp per lane quarter
    }
    mbar_init(accfull, 1);
    mbar_init(accempty, kEpi);   // every epilogue warp has read its columns
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmW);
    if constexpr (!GSC) {
      prefetch_tmap(&tmAS);
      prefetch_tmap(&tmWS);
    }
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int g = 0;  // stages issued so far (ring slot g % kStages, fill g / kStages)
      bool ok = true;
      for (int i = 0; i < my_tiles && ok; ++i) {
        const int n0 = tile_n0(i), m0 = tile_m0(i);
        for (int k = 0; k < num_k; ++k, ++g) {
          const int s = g % kStages;
          if (g >= kStages && !wait_bar(&empty[s], ((g / kStages) + 1) & 1, err, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], GSC ? (uint32_t)(kActTile + kWTile) : kStageBytes);
          tma_load_2d(smem + kOffAct + s * kActTile, &tmA, k * kRowBytes, m0, &full[s]);
          tma_load_2d(smem + kOffW + s * kWTile, &tmW, k * kRowBytes, n0, &full[s]);
          if constexpr (!GSC) {
            tma_load_2d(smem + kOffActSc + s * kActSc, &tmAS, k * kScBytes, m0, &full[s]);
            tma_load_2d(smem + kOffWSc + s * kWSc, &tmWS, k * kScBytes, n0, &full[s]);
          }
        }
      }
      // No copy may still be landing in shared memory when the CTA exits.
      for (int it = (g > kStages ? g - kStages : 0); it < g; ++it)
        drain_wait(&full[it % kStages], (it / kStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      int committed = -1;
      const uint64_t adesc0 = desc_kmajor_sw128(smem_u32(smem + kOffW));
      const uint64_t bdesc0 = desc_kmajor_sw128(smem_u32(smem + kOffAct));
      int g = 0;
      for (int i = 0; i < my_tiles && ok; ++i) {
        // The accumulator is free once the epilogue has read tile i - 1.
        if (i > 0 && !wait_bar(accempty, (i - 1) & 1, err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int k = 0; k < num_k; ++k, ++g) {
          const int s = g % kStages;
          // ready[s] implies full[s]: each writer warp arrives only after its
          // own wait on full[s], which covers all four copies of the stage.
          if (!wait_bar(&ready[s], (g / kStages) & 1, err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_f4_stage(tmem + kColAcc, adesc0 + (uint64_t)((s * kWTile) >> 4),
                       bdesc0 + (uint64_t)((s * kActTile) >> 4), tmem + kColSfa + 16 * s,
                       tmem + kColSfb + 32 * s, k > 0 ? 1u : 0u);
          mma_commit(&empty[s]);
          committed = g;
        }
        if (ok) mma_commit(accfull);  // tile i's accumulator is complete
      }
      if (!ok && committed >= 0) {
        // MMAs still reading tensor memory must finish before the release.
        drain_wait(&empty[committed % kStages], (committed / kStages) & 1);
      }
    }
  } else if (warp < kWarpEpi0) {
    // ---------------- scale writers ----------------
    const int q = warp & 3;               // TMEM lane quarter
    const int ph = (warp - 2) >> 2;       // stage phase of this warp
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    for (int g = ph; g < total; g += kPh) {
      const int s = g % kStages;
      if (!wait_bar(&full[s], (g / kStages) & 1, err, abort_flag)) break;
      // Register j of the weight-scale store goes to column j: chunk j / 4,
      // row group j % 4 (rows 32 (j % 4) + lane); the token-scale store has 8
      // columns per chunk, row group (j % 8) of 32 tokens.
      const uint8_t* wsc = smem + kOffWSc + s * kWSc;
      const uint8_t* asc = smem + kOffActSc + s * kActSc;
      // With K not a multiple of 256 the scale rows cannot be tensor-copied
      // (row pitch K/16 bytes): this stage's 16 scale bytes of each row come
      // straight from global memory, zero past the last row or column.
      const int gi = g / num_k, gk = g - gi * num_k;
      auto scales16 = [&](const uint8_t* base, int row, int rows) -> uint4 {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (row < rows) {
          const int64_t off = (int64_t)row * S + 16 * gk;
          if ((S & 3) == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (16 * gk + 4 * j < S) w[j] = __ldg(reinterpret_cast<const uint32_t*>(base + off) + j);
          } else {
#pragma unroll
            for (int b = 0; b < 16; ++b)
              if (16 * gk + b < S) w[b >> 2] |= (uint32_t)__ldg(base + off + b) << (8 * (b & 3));
          }
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
      };
      uint32_t va[16], vb[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 r;
        if constexpr (GSC)
          r = scales16(ws_g, tile_n0(gi) + 32 * c + lane, N);
        else
          r = *reinterpret_cast<const uint4*>(wsc + (32 * c + lane) * kScBytes);
        va[c] = r.x;
        va[4 + c] = r.y;
        va[8 + c] = r.z;
        va[12 + c] = r.w;
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 r;
        if constexpr (GSC)
          r = scales16(as_g, tile_m0(gi) + 32 * c + lane, M);
        else
          r = *reinterpret_cast<const uint4*>(asc + (32 * c + lane) * kScBytes);
        vb[c] = r.x;
        vb[8 + c] = r.y;
        vb[16 + c] = r.z;
        vb[24 + c] = r.w;
      }
      tmem_st16(lane_base + kColSfa + 16 * s, va);
      tmem_st32(lane_base + kColSfb + 32 * s, vb);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ready[s]);
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;                   // TMEM lane quarter
    const int h = (warp - kWarpEpi0) >> 2;    // token-column half
    const int row = q * 32 + lane;            // weight row within the tile
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const float gs = __ldg(gscale);
    for (int i = 0; i < my_tiles; ++i) {
      if (!wait_bar(accfull, i & 1, err, abort_flag)) break;
      tc_fence_after();
      const int n = tile_n0(i) + row, m0 = tile_m0(i);
      const float b = (bias != nullptr && n < N) ? act_to_f32<DT>(__ldg(bias + n)) : 0.0f;
      // The warp's 128 columns leave tensor memory 16 at a time and stay in
      // registers as packed output pairs, so the accumulator is handed back
      // before any store is issued.
      uint32_t pk[kBN / 64][16];
#pragma unroll
      for (int c = 0; c < kBN / 64; ++c) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r[16];
          tmem_ld16(lane_base + kColAcc + 64 * c + 32 * h + 16 * half, r);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            pk[c][8 * half + j] = pack2_rn<DT>(__uint_as_float(r[2 * j]) * gs + b,
                                               __uint_as_float(r[2 * j + 1]) * gs + b);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accempty);
      if (n < N) {
        // Token rows m0 + 64 c + 32 h + t, t < 32, in order, one running pointer.
        uint16_t* yp = Y + (int64_t)(m0 + 32 * h) * N + n;
        int m = m0 + 32 * h;
#pragma unroll
        for (int c = 0; c < kBN / 64; ++c) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (m < M) *yp = (uint16_t)(pk[c][j] & 0xFFFFu);
            yp += N;
            if (m + 1 < M) *yp = (uint16_t)(pk[c][j] >> 16);
            yp += N;
            m += 2;
          }
          yp += (int64_t)32 * N;  // the other half's 32 tokens
          m += 32;
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

template <int DT, bool GSC>
int launch_t(const F4F4Args& a, cudaStream_t st) {
  const uint64_t rowb = (uint64_t)a.K / 2, scb = (uint64_t)a.K / 16;
  constexpr bool gsc = GSC;  // scale rows not tensor-copyable: read them from global memory
  CUtensorMap tmA, tmW, tmAS, tmWS;
  if (!encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, rowb, (uint64_t)a.M, rowb,
                      kRowBytes, kBN, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, rowb, (uint64_t)a.N, rowb,
                      kRowBytes, kBM, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      (!gsc && (!encode_tmap_2d(&tmAS, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A_scale, scb,
                                (uint64_t)a.M, scb, kScBytes, kBN, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_NONE) ||
                !encode_tmap_2d(&tmWS, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.ws, scb, (uint64_t)a.N,
                                scb, kScBytes, kBM, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_NONE))))
    return kCuda;
  if (gsc) {  // unused by the kernel
    tmAS = tmA;
    tmWS = tmW;
  }
  static std::once_flag once[64];
  const int dev = device_info().device;
  if (dev < 0 || dev >= 64) return kCuda;
  std::call_once(once[dev], [] {
    cudaFuncSetAttribute(gemm_f4f4_kernel<DT, GSC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kSmemBytes);
  });
  const int64_t tiles_n = (a.N + kBM - 1) / kBM;
  const int64_t tiles = tiles_n * ((a.M + kBN - 1) / kBN);
  const int grid = (int)std::min<int64_t>(tiles, device_info().sm_count);
  gemm_f4f4_kernel<DT, GSC><<<grid, kThreads, kSmemBytes, st>>>(
      tmA, tmW, tmAS, tmWS, a.A_scale, a.ws, a.gscale,
      reinterpret_cast<const uint16_t*>(a.bias),
      reinterpret_cast<uint16_t*>(a.Y), (int)a.M, (int)a.N, (int)a.K, (int)tiles_n, (int)tiles,
      device_error_word());
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}

}  // namespace

bool gemm_f4f4_supports(const F4F4Args& a) {
  const DeviceInfo& d = device_info();
  if (d.cc_major != 10 || d.max_smem_optin < kSmemBytes) return false;
  if (a.K % 32 != 0) return false;   // packed code rows of 16-byte multiples
  // Tile indices are int.
  const int64_t tiles = ((a.N + kBM - 1) / kBM) * ((a.M + kBN - 1) / kBN);
  return tiles < (int64_t(1) << 31) && a.N < (int64_t(1) << 31);
}

int launch_gemm_f4f4(const F4F4Args& a, cudaStream_t st) {
  if (!gemm_f4f4_supports(a)) return kUnsupported;
  if (a.K % kBK != 0) return a.dtype == 1 ? launch_t<1, true>(a, st) : launch_t<0, true>(a, st);
  return a.dtype == 1 ? launch_t<1, false>(a, st) : launch_t<0, false>(a, st);
}

}  // namespace wqmm
