// Block-scaled GEMM on the 5th-generation tensor cores (tcgen05), for MXFP8
// (kind::mxf8f6f4, E4M3 x E4M3, UE8M0 scale per 32 along K) and NVFP4
// (kind::mxf4nvf4, packed E2M1 x E2M1, UE4M3 scale per 16 along K), plain and
// grouped (MoE routed experts).
//
// "Miles Blackwell RL Cambia la Uniformidad BF16 por MXFP8 y NVFP4 Nativos",
// section "La Compatibilidad...": MXFP8 serves the forward, weight-gradient
// and data-gradient GEMMs; NVFP4 serves the routed-expert weights and
// activations of MoE layers, with a per-token FP32 scale.  Section "Un
// Cuantizador Compartido...": the tensor cores expect the microscaling blocks
// along the reduction dimension.  "NVIDIA presenta una metodologia de
// preentrenamiento de 4 bits utilizando NVFP4", section "Que es realmente
// NVFP4": the block scales are applied by the tensor core, the FP32 scale
// outside it -- here in the epilogue.
//
//   C[m, n] (+)= A32[m] * B32[n or group] * sum_k A^[m, k] B^[n, k]
//
// Structure (one CTA per SM, persistent over 128x128 output tiles):
//   warp 0      : TMA producer -- A and B tiles (128 rows x 128 bytes of K,
//                 128-byte swizzle) and the matching 512-byte scale tiles,
//                 into a ring of shared-memory stages guarded by mbarriers;
//   warp 1      : allocates tensor memory; one thread copies each stage's
//                 scale tiles into tensor memory (tcgen05.cp) and issues the
//                 block-scaled MMAs, accumulating in one of two 128-column
//                 FP32 accumulators, then commits the stage back to the
//                 producer and the finished accumulator to the epilogue;
//   warps 2..5  : epilogue -- tcgen05.ld of their 32-lane quarter, FP32
//                 scales, convert, store; the accumulator is released as soon
//                 as it has been read, so the next tile's MMAs overlap.
// Every mbarrier wait is bounded (about a second) and reports through the
// workspace error word.
#include <cuda_bf16.h>

#include "device.cuh"
#include "groups.cuh"
#include "kernels.h"

namespace mx8q {

namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kKBytes = 128;               // bytes of K per stage and row (one swizzle atom)
constexpr int kThreads = 192;
constexpr int kTileBytes = BM * kKBytes;   // 16 KB for A (and for B, since BN == BM)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = BN;          // f32 accumulator: one column per output column

template <int kFmt>
struct Cfg;
template <>
struct Cfg<0> {                 // MXFP8: K = 128 elements per stage, 32 per MMA
  static constexpr int kElemsPerStage = 128;
  static constexpr int kElemsPerMma = 32;
  static constexpr int kSfTiles = 1;     // 128x4 scale tiles per operand per stage
  static constexpr int kBlock = 32;
};
template <>
struct Cfg<1> {                 // NVFP4: K = 256 elements per stage, 64 per MMA
  static constexpr int kElemsPerStage = 256;
  static constexpr int kElemsPerMma = 64;
  static constexpr int kSfTiles = 4;
  static constexpr int kBlock = 16;
};

template <int kFmt, bool kGrouped>
struct Layout {
  static constexpr int kStages = (kFmt == 1 && kGrouped) ? 5 : 6;
  static constexpr int kSfBytes = Cfg<kFmt>::kSfTiles * 512;
  static constexpr uint32_t kSfCols = 4 * Cfg<kFmt>::kSfTiles;   // tmem columns per operand
};

template <int kFmt, bool kGrouped>
struct __align__(1024) GemmSmem {
  using L = Layout<kFmt, kGrouped>;
  uint8_t a[L::kStages][kTileBytes];
  uint8_t b[L::kStages][kTileBytes];
  uint8_t sfa[L::kStages][L::kSfBytes];
  uint8_t sfb[L::kStages][L::kSfBytes];
  uint64_t full[L::kStages];
  uint64_t empty[L::kStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Instruction descriptor of the block-scaled MMA (M = 128, N = BN, both
// operands K-major): B scale id bits 4-5, A/B element type bits 7-9 / 10-12,
// N >> 3 bits 17-22, scale type bit 23 (1 = UE8M0, 0 = UE4M3), M >> 4 bits
// 24-28, A scale id bits 29-30.
__device__ __forceinline__ uint32_t make_idesc(int fmt, uint32_t sf_id) {
  const uint32_t etype = fmt == 0 ? 0u /* E4M3 */ : 1u /* E2M1 */;
  uint32_t d = 0;
  d |= (sf_id & 3u) << 4;
  d |= etype << 7;
  d |= etype << 10;
  d |= static_cast<uint32_t>(BN >> 3) << 17;
  d |= (fmt == 0 ? 1u : 0u) << 23;
  d |= static_cast<uint32_t>(BM >> 4) << 24;
  d |= (sf_id & 3u) << 29;
  return d;
}

// Output tile -> (group, first row of A, rows valid, scale-tile row of A, n0).
struct TileCoord {
  int g;
  int64_t a_row0;     // first row of A / C
  int64_t rows;       // valid rows in this tile
  int64_t sfa_tile;   // 128-row scale tile index of A
  int64_t n0;
};

template <bool kGrouped>
__device__ __forceinline__ TileCoord decode_tile(int64_t t, int64_t tiles_n, int64_t M,
                                                 const GroupSmem* gs, int G) {
  TileCoord c;
  if (!kGrouped) {
    const int64_t tm = (M + BM - 1) / BM;
    const int64_t mt = t % tm, nt = t / tm;
    c.g = 0;
    c.a_row0 = mt * BM;
    c.rows = M - c.a_row0 < BM ? M - c.a_row0 : BM;
    c.sfa_tile = mt;
    c.n0 = nt * BN;
    return c;
  }
  const int64_t gmt = t / tiles_n;                   // global m-tile band
  const int g = upper_group(gs->pref, G, gmt * BM);
  const int64_t mt0 = gs->pref[g] / BM;
  const int64_t mtiles = gs->pref[g + 1] / BM - mt0;
  const int64_t local = t - mt0 * tiles_n;
  const int64_t mt = local % mtiles, nt = local / mtiles;
  const int64_t ng = gs->offs[g + 1] - gs->offs[g];
  c.g = g;
  c.a_row0 = gs->offs[g] + mt * BM;
  c.rows = ng - mt * BM < BM ? ng - mt * BM : BM;
  c.sfa_tile = mt0 + mt;
  c.n0 = nt * BN;
  return c;
}

template <int kFmt, bool kGrouped>
__global__ void __launch_bounds__(kThreads, 1)
    bs_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, const GemmArgs args) {
  using L = Layout<kFmt, kGrouped>;
  using F = Cfg<kFmt>;
  using Smem = GemmSmem<kFmt, kGrouped>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  Smem& sm = *reinterpret_cast<Smem*>(base);
  GroupSmem* gs = reinterpret_cast<GroupSmem*>(base + sizeof(Smem));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* err = args.err;

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.acc_full[i]), 1);
      mbar_init(smem_u32(&sm.acc_empty[i]), 128);
    }
    mbar_init(smem_u32(&sm.drain), 1);
    sm.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (kGrouped) load_group_prefix(*gs, args.offs, args.G);   // contains __syncthreads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  const int64_t M = args.M, N = args.N, K = args.K;
  const int64_t tiles_n = (N + BN - 1) / BN;
  const int64_t tiles_m = kGrouped ? gs->pref[args.G] / BM : (M + BM - 1) / BM;
  const int64_t ntiles = tiles_m * tiles_n;
  const int64_t kbytes = kFmt == 0 ? K : K / 2;
  const int ktiles = static_cast<int>((kbytes + kKBytes - 1) / kKBytes);
  const int64_t sf_kt = (K / F::kBlock + 3) / 4;          // scale tiles along K
  const int G = args.G;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
        const TileCoord tc = decode_tile<kGrouped>(t, tiles_n, M, gs, G);
        const int64_t nt = tc.n0 / BN;
        const uint8_t* sfa_src = args.SA + tc.sfa_tile * sf_kt * 512;
        const uint8_t* sfb_src =
            args.SB + ((kGrouped ? static_cast<int64_t>(tc.g) * tiles_n : 0) + nt) * sf_kt * 512;
        for (int kt = 0; kt < ktiles; ++kt, ++it) {
          const int s = it % L::kStages;
          const uint32_t ph = (it / L::kStages) & 1;
          if (!mbar_wait(smem_u32(&sm.empty[s]), ph ^ 1, err, kErrWaitProducer, &sm.abort)) {
            ok = false;
            break;
          }
          const int64_t sf0 = static_cast<int64_t>(kt) * F::kSfTiles;
          const int nsf = static_cast<int>(sf_kt - sf0 < F::kSfTiles ? sf_kt - sf0 : F::kSfTiles);
          const uint32_t full = smem_u32(&sm.full[s]);
          mbar_arrive_expect_tx(full, 2 * kTileBytes + 2 * nsf * 512);
          tma_load_2d(smem_u32(sm.a[s]), &tmap_a, kt * kKBytes, static_cast<int32_t>(tc.a_row0), full);
          if (kGrouped)
            tma_load_3d(smem_u32(sm.b[s]), &tmap_b, kt * kKBytes, static_cast<int32_t>(tc.n0), tc.g, full);
          else
            tma_load_2d(smem_u32(sm.b[s]), &tmap_b, kt * kKBytes, static_cast<int32_t>(tc.n0), full);
          bulk_load(smem_u32(sm.sfa[s]), sfa_src + sf0 * 512, nsf * 512, full);
          bulk_load(smem_u32(sm.sfb[s]), sfb_src + sf0 * 512, nsf * 512, full);
        }
      }
      if (!ok) {
        // let the copies already issued land before the block exits
        for (int j = (it > L::kStages ? it - L::kStages : 0); j < it; ++j)
          mbar_wait(smem_u32(&sm.full[j % L::kStages]), (j / L::kStages) & 1, err, kErrWaitTeardown,
                    nullptr, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0, tcount = 0;
      bool ok = true;
      const uint32_t sf_base = tmem + 2 * kAccCols;
      for (int64_t t = blockIdx.x; ok && t < ntiles; t += gridDim.x, ++tcount) {
        const int as = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1;
        if (!mbar_wait(smem_u32(&sm.acc_empty[as]), aph ^ 1, err, kErrWaitAccum, &sm.abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + as * kAccCols;
        for (int kt = 0; kt < ktiles; ++kt, ++it) {
          const int s = it % L::kStages;
          const uint32_t ph = (it / L::kStages) & 1;
          if (!mbar_wait(smem_u32(&sm.full[s]), ph, err, kErrWaitConsumer, &sm.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int64_t sf0 = static_cast<int64_t>(kt) * F::kSfTiles;
          const int nsf = static_cast<int>(sf_kt - sf0 < F::kSfTiles ? sf_kt - sf0 : F::kSfTiles);
          const uint32_t tsfa = sf_base + s * 2 * L::kSfCols;
          const uint32_t tsfb = tsfa + L::kSfCols;
          for (int j = 0; j < nsf; ++j) {
            tc_cp_32x128b_x4(tsfa + 4 * j, smem_desc(smem_u32(sm.sfa[s]) + 512 * j, 128, 128, kSwizzleNone));
            tc_cp_32x128b_x4(tsfb + 4 * j, smem_desc(smem_u32(sm.sfb[s]) + 512 * j, 128, 128, kSwizzleNone));
          }
          const int64_t krem = K - static_cast<int64_t>(kt) * F::kElemsPerStage;
          const int nmma = static_cast<int>(krem >= F::kElemsPerStage
                                                ? F::kElemsPerStage / F::kElemsPerMma
                                                : (krem + F::kElemsPerMma - 1) / F::kElemsPerMma);
          const uint32_t a0 = smem_u32(sm.a[s]), b0 = smem_u32(sm.b[s]);
          for (int kk = 0; kk < nmma; ++kk) {
            const uint64_t ad = smem_desc(a0 + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(b0 + kk * 32, 16, 1024, kSwizzle128B);
            const uint32_t acc = (kt > 0 || kk > 0) ? 1u : 0u;
            if (kFmt == 0)
              tc_mma_mxf8(d_tmem, ad, bd, make_idesc(0, kk), tsfa, tsfb, acc);
            else
              tc_mma_nvf4(d_tmem, ad, bd, make_idesc(1, 0), tsfa + 4 * kk, tsfb + 4 * kk, acc);
          }
          tc_commit(smem_u32(&sm.empty[s]));   // stage free once these MMAs finish
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm.acc_full[as]));  // accumulator ready for the epilogue
      }
      // no MMA may be in flight when tensor memory is released
      tc_commit(smem_u32(&sm.drain));
      mbar_wait(smem_u32(&sm.drain), 0, err, kErrWaitTeardown, nullptr, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;              // tcgen05.ld lane quarter of this warp
    const int r_in_tile = quarter * 32 + lane;
    int tcount = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++tcount) {
      const int as = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      const bool ok = mbar_wait(smem_u32(&sm.acc_full[as]), aph, err, kErrWaitEpilogue, &sm.abort);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const TileCoord tc = decode_tile<kGrouped>(t, tiles_n, M, gs, G);
      const bool row_ok = r_in_tile < tc.rows;
      const int64_t m = tc.a_row0 + r_in_tile;
      float sa = 1.f;
      if (row_ok) {
        if (args.a32_mode == 1) sa = args.A32[m];
        else if (args.a32_mode == 2) sa = args.A32[0];
      }
      float sg = 1.f;
      if (kGrouped && args.B32 != nullptr) sg = args.B32[tc.g];
      else if (!kGrouped && args.b32_mode == 2) sg = args.B32[0];
      const bool b_row = !kGrouped && args.b32_mode == 1;
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + as * kAccCols + ch * 32, r);
        tmem_wait_ld();
        if (ch == BN / 32 - 1) {
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.acc_empty[as]));
        }
        const int64_t n0 = tc.n0 + ch * 32;
        if (!row_ok || n0 >= N) continue;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float y = __fmul_rn(__uint_as_float(r[j]), sa);
          float sbn = sg;
          if (b_row) sbn = (n0 + j < N) ? args.B32[n0 + j] : 0.f;
          v[j] = __fmul_rn(y, sbn);
        }
        const bool full_chunk = n0 + 32 <= N;
        if (args.out_bf16) {
          uint16_t* crow = static_cast<uint16_t*>(args.C) + m * args.ldc + n0;
          if (full_chunk) {
            uint32_t p[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              p[j] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * j]))) |
                     (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * j + 1]))) << 16);
            uint4* d = reinterpret_cast<uint4*>(crow);
#pragma unroll
            for (int j = 0; j < 4; ++j) d[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
          } else {
            for (int j = 0; j < 32 && n0 + j < N; ++j) crow[j] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
          }
        } else {
          float* crow = static_cast<float*>(args.C) + m * args.ldc + n0;
          if (full_chunk) {
            float4* d = reinterpret_cast<float4*>(crow);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float4 o = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
              if (args.accumulate) {
                const float4 c = d[j];
                o.x += c.x; o.y += c.y; o.z += c.z; o.w += c.w;
              }
              d[j] = o;
            }
          } else {
            for (int j = 0; j < 32 && n0 + j < N; ++j) crow[j] = args.accumulate ? crow[j] + v[j] : v[j];
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int kFmt, bool kGrouped>
size_t smem_bytes_for() {
  return sizeof(GemmSmem<kFmt, kGrouped>) + (kGrouped ? sizeof(GroupSmem) : 0) + 1024;
}

}  // namespace

size_t gemm_smem_bytes(int fmt) {
  return fmt == 0 ? smem_bytes_for<0, true>() : smem_bytes_for<1, true>();
}

cudaError_t launch_bs_gemm(const GemmArgs& a, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                           int sm_count, cudaStream_t stream) {
  const int64_t tiles_n = (a.N + BN - 1) / BN;
  int64_t tiles_m = (a.M + BM - 1) / BM;
  if (a.grouped) tiles_m = (a.M + BM - 1) / BM + a.G;   // upper bound: every group pads a tile
  const int64_t ntiles = tiles_m * tiles_n;
  const unsigned grid = static_cast<unsigned>(ntiles < sm_count ? ntiles : sm_count);
  if (grid == 0) return cudaSuccess;
#define MX8Q_GEMM_LAUNCH(F, GRP)                                                               \
  do {                                                                                          \
    auto k = bs_gemm_kernel<F, GRP>;                                                           \
    const size_t smem = smem_bytes_for<F, GRP>();                                              \
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,       \
                                         static_cast<int>(smem));                             \
    if (e != cudaSuccess) return e;                                                             \
    k<<<grid, kThreads, smem, stream>>>(tmap_a, tmap_b, a);                                    \
  } while (0)
  if (a.fmt == 0) {
    if (a.grouped) MX8Q_GEMM_LAUNCH(0, true); else MX8Q_GEMM_LAUNCH(0, false);
  } else {
    if (a.grouped) MX8Q_GEMM_LAUNCH(1, true); else MX8Q_GEMM_LAUNCH(1, false);
  }
#undef MX8Q_GEMM_LAUNCH
  return cudaGetLastError();
}

}  // namespace mx8q
