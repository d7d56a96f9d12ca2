// Block-scaled GEMM on the 5th-generation tensor cores (tcgen05), for MXFP8
// (kind::mxf8f6f4, E4M3 x E4M3, UE8M0 scale per 32 along K), NVFP4
// (kind::mxf4nvf4, packed E2M1 x E2M1, UE4M3 scale per 16 along K) and MXFP4
// (kind::mxf4nvf4, packed E2M1 x E2M1, UE8M0 scale per 32 along K), plain and
// grouped (MoE routed experts); and the plain BF16 GEMM (kind::f16, no block
// scales) of the dequantized-backward mode, on the same pipeline.
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
// Structure (one CTA per SM, persistent over 128 x BN output tiles):
//   producers   : TMA loads of A (128 rows) and B (BN rows) tiles of 128
//                 bytes of K with the 128-byte swizzle, plus the matching
//                 512-byte scale tiles, into a ring of shared-memory stages
//                 guarded by mbarriers.  One thread of warp 0 issues A and its
//                 scale tiles, one thread in each of BN/128 further warps one
//                 128-row box of B and its scale tiles: a single issuing
//                 thread moves at most
//                 about 50 GB/s per SM on this GPU, several in separate warps
//                 move several times that, so the operand stream of a stage
//                 is split over 1 + BN/128 issuers;
//   warp 1      : allocates tensor memory; one thread issues the block-scaled
//                 MMAs (M = 128, N = BN) into an FP32 accumulator in tensor
//                 memory once a stage's operands have landed and its scales
//                 are in tensor memory, commits each stage back to the
//                 producers and each finished accumulator to the epilogue;
//   epilogue    : BN/32 warps, two per 32-lane quarter of tensor memory when
//                 BN = 256.  When the accumulator is full each warp pulls its
//                 32 rows x 128 columns into registers, releases it at once
//                 (so the next tile's MMAs start), then applies the FP32
//                 scales, converts and stores.
// Scales into tensor memory, two ways:
//   - single GEMM: while an accumulator fills, the epilogue warps move each
//     landed stage's scale tiles from shared into tensor memory (ld.shared +
//     tcgen05.st into their own lane quarter, A's tiles by one warp of the
//     quarter, B's by the other), also between the pieces of their stores,
//     so the tensor pipe runs MMAs only.  A tcgen05.cp of a 512-byte scale
//     tile costs the in-order tensor pipe about 45 ns; NVFP4 copies 12 per
//     stage, which was 40% of the Fprop GEMM (39 -> 31 us on 2048x2048->8192);
//   - grouped GEMM (BN = 256): the three producer warps, each right after
//     issuing its loads, and one more warp (epilogue warp 5 in the SwiGLU
//     GEMM, between its own work; the MMA warp in the others) move one lane
//     quarter each.  The MoE GEMMs have short K per tile (3 stages for the
//     768-wide down projection) and, for gate|up, a SwiGLU epilogue: the
//     epilogue warps alone could not keep the MMAs fed (gate|up 154-214 us
//     against 115 us with tcgen05.cp in the MMA thread); with the producers
//     staging, the DeepSeek-V3-shaped gate|up runs in 2139 us against 3019;
//   - grouped GEMM with gathered A: the MMA thread copies them with
//     tcgen05.cp right before the stage's MMAs.
// BN = 128 keeps two accumulators (epilogue fully overlapped); BN = 256 moves
// half the operand bytes per FLOP of BN = 128 and keeps one accumulator (the
// 512 tensor-memory columns hold 256 accumulator columns plus the scales).
// Every mbarrier wait is bounded (about a second) and reports through the
// workspace error word.
#include <cuda_bf16.h>

#include "device.cuh"
#include "groups.cuh"
#include "kernels.h"

#ifndef MX8Q_GEMM_BN
#define MX8Q_GEMM_BN 256
#endif

namespace mx8q {

namespace {

constexpr int BM = 128;
constexpr int kKBytes = kGemmKBytes;       // bytes of K per stage and row (one swizzle atom)
static_assert(kKBytes == 64 || kKBytes == 128, "one 64- or 128-byte swizzle atom per stage row");
constexpr uint32_t kSwizzle = kKBytes == 128 ? kSwizzle128B : kSwizzle64B;
constexpr uint32_t kAtomSbo = 8 * kKBytes;  // bytes between 8-row groups of a swizzled operand
constexpr int kBoxBytes = 128 * kKBytes;   // one 128-row TMA box
constexpr int kTileABytes = BM * kKBytes;
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemBudget = 227 * 1024 - 1024;

template <int kFmt>
struct Cfg;
// A 512-byte scale tile holds 4 scales for each of 128 rows: 128 K elements
// for MXFP8 and MXFP4, 64 for NVFP4.  A stage covers kElemsPerStage elements of K and
// needs kSfTiles tiles, from tile (first element of the stage) / kElemsPerTile;
// an MXFP8 stage of 64 bytes uses half a tile, and selects its scales with
// the MMA's scale id.
template <>
struct Cfg<0> {                 // MXFP8: 1 byte per element, 32 elements per MMA
  static constexpr int kElemsPerStage = kKBytes;
  static constexpr int kElemsPerMma = 32;
  static constexpr int kBlock = 32;
  static constexpr int kElemsPerTile = 128;
  static constexpr int kSfTiles = 1;
};
template <>
struct Cfg<1> {                 // NVFP4: 2 elements per byte, 64 elements per MMA
  static constexpr int kElemsPerStage = 2 * kKBytes;
  static constexpr int kElemsPerMma = 64;
  static constexpr int kBlock = 16;
  static constexpr int kElemsPerTile = 64;
  static constexpr int kSfTiles = kElemsPerStage / kElemsPerTile;
};
template <>
struct Cfg<3> {                 // BF16: 2 bytes per element, 16 elements per MMA, no scales
  static constexpr int kElemsPerStage = kKBytes / 2;
  static constexpr int kElemsPerMma = 16;
  static constexpr int kBlock = 32;            // unused
  static constexpr int kElemsPerTile = 128;    // unused
  static constexpr int kSfTiles = 0;
};
template <>
struct Cfg<2> {                 // MXFP4: 2 elements per byte, 64 elements (2 scales) per MMA
  static constexpr int kElemsPerStage = 2 * kKBytes;
  static constexpr int kElemsPerMma = 64;
  static constexpr int kBlock = 32;
  static constexpr int kElemsPerTile = 128;
  static constexpr int kSfTiles = kElemsPerStage / kElemsPerTile;
};

// Fused MoE modes of the grouped GEMM (bit flags):
//   kModeGather : A is the token-major quantized matrix; the producer gathers
//                 the rows of each tile (and their scales) through a row ->
//                 token map, so tokens are quantized once, before dispatch;
//   kModeSwiGLU : B holds gate rows [0, F) and up rows [F, 2F) per expert; a
//                 tile pairs gate rows n0.. and up rows F + n0.. (128 each),
//                 and the epilogue writes h = silu(g) * u for 128 columns;
//   kModeQuantH : (with kModeSwiGLU) the epilogue also quantizes h per token
//                 to NVFP4.  The F / 128 tiles of a 128-row band are computed
//                 at the same time by the CTAs of one thread-block cluster
//                 (CTA rank = h tile); each CTA sends the row maxima of its
//                 128 h columns to every CTA of the cluster (distributed
//                 shared memory), so every CTA knows each row's amax, and
//                 encodes its own columns from registers: codes, block scales
//                 and S_dec of h, with no bf16 h round trip through memory.
constexpr int kModeGather = 1, kModeSwiGLU = 2, kModeQuantH = 4;
constexpr int kMaxClusterTiles = 8;          // h tiles of a band = CTAs of a cluster (portable maximum)

template <int kFmt, bool kGrouped, int kBN, int kMode>
struct Layout {
  static constexpr int kBRow128 = kBN / 128;                         // 128-row blocks of B
  static constexpr int kTileBBytes = kBN * kKBytes;
  // (16 bytes of unused placeholder when the format has no block scales)
  static constexpr int kSfaBytes = Cfg<kFmt>::kSfTiles > 0 ? Cfg<kFmt>::kSfTiles * 512 : 16;
  static constexpr int kSfbBytes = Cfg<kFmt>::kSfTiles > 0 ? Cfg<kFmt>::kSfTiles * 512 * kBRow128 : 16;
  static constexpr int kStageBytes = kTileABytes + kTileBBytes + kSfaBytes + kSfbBytes;
  // 32 rows x 64 B per epilogue warp for the bulk stores (the SwiGLU
  // epilogue stores h directly; with h quantization the area holds the row
  // maxima)
  static constexpr int kEpiStageBytes = (kMode & kModeSwiGLU) && !(kMode & kModeQuantH) ? 16 : 2048;
  static constexpr int kFixed = 256 + (kBN / 32) * kEpiStageBytes + ((kMode & kModeQuantH) ? 1024 + 32 : 0) +
                                ((kMode & kModeGather) ? 4 * BM : 0) +
                                (kGrouped ? static_cast<int>(sizeof(GroupTiles)) : 0);
  static constexpr int kStagesFit = (kSmemBudget - kFixed) / kStageBytes;
  static constexpr int kStages = kStagesFit > 10 ? 10 : kStagesFit;
  static constexpr int kAccBufs = kBN == 128 ? 2 : 1;
  static constexpr uint32_t kSfaCols = 4 * Cfg<kFmt>::kSfTiles;      // tensor-memory columns
  static constexpr uint32_t kSfbCols = 4 * Cfg<kFmt>::kSfTiles * kBRow128;
  static constexpr uint32_t kSfColsPerStage = kSfaCols + kSfbCols;
  static constexpr uint32_t kAccCols = kAccBufs * kBN;
  static constexpr int kEpiWarps = kBN / 32;                         // 128 columns per warp
  // warp 0 + one warp per B box (+ the 32 lanes of warp 0 that gather A rows,
  // each arriving when its copies have landed)
  static constexpr int kProducers = 1 + kBRow128 + ((kMode & kModeGather) ? 32 : 0);
  // warp 0 producer, warp 1 MMA, warps 2 .. 1 + kEpiWarps epilogue, then the B producers
  static constexpr int kThreads = 64 + 32 * kEpiWarps + 32 * kBRow128;
  static_assert(kStages >= 3, "pipeline too shallow");
  static_assert(!(kMode & kModeSwiGLU) || kBN == 256, "the SwiGLU epilogue pairs two 128-row boxes");
  static_assert(!(kMode & kModeQuantH) || ((kMode & kModeSwiGLU) && !(kMode & kModeGather)),
                "h is quantized in the SwiGLU epilogue of dispatched rows");
  // h quantization: the row maxima of a band, [2 buffers][2 halves x tiles][128 rows] floats,
  // live in the epilogue staging area (the SwiGLU epilogue stores h directly)
  static_assert(!(kMode & kModeQuantH) || kEpiWarps * kEpiStageBytes >= 2 * 2 * kMaxClusterTiles * 128 * 4,
                "row-maximum exchange does not fit the staging area");
  static_assert(kAccCols + kStages * kSfColsPerStage <= kTmemCols, "tensor memory overflow");
};

template <int kFmt, bool kGrouped, int kBN, int kMode>
struct __align__(1024) GemmSmem {
  using L = Layout<kFmt, kGrouped, kBN, kMode>;
  uint8_t a[L::kStages][kTileABytes];
  uint8_t b[L::kStages][L::kTileBBytes];
  uint8_t sfa[L::kStages][L::kSfaBytes];
  uint8_t sfb[L::kStages][L::kSfbBytes];
  uint8_t cstage[L::kEpiWarps][L::kEpiStageBytes];   // epilogue staging for bulk stores
  uint64_t full[L::kStages];
  uint64_t empty[L::kStages];
  uint64_t sf_full[L::kStages];                       // a stage's scale tiles have landed
  uint64_t sf_ready[L::kStages];                      // a stage's scales are in tensor memory
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int32_t gtok[(kMode & kModeGather) ? BM : 1];       // gathered mode: source rows of the tile
  uint64_t hmax_full[2];                              // h quantization: a band's row maxima are all in
  float2 tab[(kMode & kModeQuantH) ? 128 : 1];        // h quantization: {E4M3 value, RN(1/value)}
};

// Instruction descriptor of the block-scaled MMA (M = 128, both operands
// K-major): B scale id bits 4-5, A/B element type bits 7-9 / 10-12, N >> 3
// bits 17-22, scale type bit 23 (1 = UE8M0, 0 = UE4M3), M >> 4 bits 24-28,
// A scale id bits 29-30.
__device__ __forceinline__ uint32_t make_idesc(int fmt, int n, uint32_t sf_id) {
  const uint32_t etype = fmt == 0 ? 0u /* E4M3 */ : 1u /* E2M1 */;
  uint32_t d = 0;
  d |= (sf_id & 3u) << 4;
  d |= etype << 7;
  d |= etype << 10;
  d |= static_cast<uint32_t>(n >> 3) << 17;
  d |= (fmt == 1 ? 0u : 1u) << 23;
  d |= static_cast<uint32_t>(BM >> 4) << 24;
  d |= (sf_id & 3u) << 29;
  return d;
}

// Instruction descriptor of the dense BF16 MMA (kind::f16; M = 128, both
// operands K-major): D format F32 bits 4-5, A/B format BF16 bits 7-9 / 10-12,
// N >> 3 bits 17-22, M >> 4 bits 24-28.
__device__ __forceinline__ uint32_t make_idesc_bf16(int n) {
  uint32_t d = 0;
  d |= 1u << 4;    // F32 accumulator
  d |= 1u << 7;    // A: BF16
  d |= 1u << 10;   // B: BF16
  d |= static_cast<uint32_t>(n >> 3) << 17;
  d |= static_cast<uint32_t>(BM >> 4) << 24;
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

template <bool kGrouped, int kNT>
__device__ __forceinline__ TileCoord decode_tile(int64_t t, int64_t tiles_n, int64_t M,
                                                 const GroupTiles* gs, int G) {
  TileCoord c;
  if (!kGrouped) {
    const int64_t tm = (M + BM - 1) / BM;
    const int64_t mt = t % tm, nt = t / tm;
    c.g = 0;
    c.a_row0 = mt * BM;
    c.rows = M - c.a_row0 < BM ? M - c.a_row0 : BM;
    c.sfa_tile = mt;
    c.n0 = nt * kNT;
    return c;
  }
  const int64_t gmt = t / tiles_n;                   // global m-tile band
  const int g = upper_group(gs->tpref, G, gmt);
  const int64_t mt0 = gs->tpref[g];
  const int64_t mtiles = gs->tpref[g + 1] - mt0;
  const int64_t local = t - mt0 * tiles_n;
  const int64_t mt = local % mtiles, nt = local / mtiles;
  const int64_t ng = gs->offs[g + 1] - gs->offs[g];
  c.g = g;
  c.a_row0 = gs->offs[g] + mt * BM;
  c.rows = ng - mt * BM < BM ? ng - mt * BM : BM;
  c.sfa_tile = mt0 + mt;
  c.n0 = nt * kNT;
  return c;
}

// Grouped band gmt (a 128-row tile of the padded grouped layout) and h tile
// nt of the cluster mode.
__device__ __forceinline__ TileCoord decode_band(int64_t gmt, int nt, const GroupTiles* gs, int G) {
  TileCoord c;
  const int g = upper_group(gs->tpref, G, gmt);
  const int64_t mt = gmt - gs->tpref[g];
  const int64_t ng = gs->offs[g + 1] - gs->offs[g];
  c.g = g;
  c.a_row0 = gs->offs[g] + mt * BM;
  c.rows = ng - mt * BM < BM ? ng - mt * BM : BM;
  c.sfa_tile = gmt;
  c.n0 = static_cast<int64_t>(nt) * 128;
  return c;
}

template <int kFmt, bool kGrouped, int kBN, int kMode>
__global__ void __launch_bounds__(Layout<kFmt, kGrouped, kBN, kMode>::kThreads, 1)
    bs_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_c, const GemmArgs args) {
  using L = Layout<kFmt, kGrouped, kBN, kMode>;
  using F = Cfg<kFmt>;
  using Smem = GemmSmem<kFmt, kGrouped, kBN, kMode>;
  constexpr bool kGather = (kMode & kModeGather) != 0;
  constexpr bool kSwiGLU = (kMode & kModeSwiGLU) != 0;
  constexpr bool kQuantH = (kMode & kModeQuantH) != 0;
  // scales moved into tensor memory by the epilogue warps (single GEMMs), by
  // the three producer warps and one more warp per lane quarter (grouped
  // GEMMs with BN = 256: see kEpiStager), else by the MMA thread with
  // tcgen05.cp (gathered A)
  constexpr bool kWarpScales = F::kSfTiles > 0 && !kGrouped;
  constexpr bool kProdScales = F::kSfTiles > 0 && kGrouped && !kGather && kBN == 256;
  constexpr bool kSepScales = kWarpScales || kProdScales;   // scale tiles land on their own barrier
  // Lane quarter 1 of the producer staging: epilogue warp 5 in the SwiGLU
  // GEMM (it stages while it waits for an accumulator and half-way through
  // each tile's SwiGLU); the MMA warp in the other modes, whose epilogues
  // stage badly (long bulk stores, cluster exchanges).  A tcgen05.st /
  // wait::st in the warp that issues the MMAs waits for its MMAs in flight
  // and so serialises them with the staging.
  // (Measured: gate|up 2569 -> 2139 us on the DeepSeek-V3 shape; warp 5
  // staging in the down projection made it 71.6 -> 79.8 us on Qwen3.)
  constexpr bool kEpiStager = kProdScales && kSwiGLU && !kQuantH;
  constexpr bool kMmaStages = kProdScales && !kEpiStager;
  static_assert(kGather <= kGrouped && kSwiGLU <= kGrouped, "fused modes are grouped only");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  Smem& sm = *reinterpret_cast<Smem*>(base);
  GroupTiles* gs = reinterpret_cast<GroupTiles*>(base + sizeof(Smem));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* err = args.err;
  constexpr int kEpiThreads = 32 * L::kEpiWarps;

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    prefetch_tmap(&tmap_c);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), L::kProducers);
      mbar_init(smem_u32(&sm.empty[s]), 1);
      mbar_init(smem_u32(&sm.sf_full[s]), 1 + L::kBRow128);
      mbar_init(smem_u32(&sm.sf_ready[s]), kProdScales ? 4 : L::kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.acc_full[i]), 1);
      mbar_init(smem_u32(&sm.acc_empty[i]), kEpiThreads);
    }
    mbar_init(smem_u32(&sm.drain), 1);
    if (kQuantH) {
      // every epilogue warp of every CTA of the cluster arrives once per band
      uint32_t nct;
      asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(nct));
      for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&sm.hmax_full[i]), L::kEpiWarps * nct);
    }
    sm.abort = 0;
    fence_barrier_init();
  }
  if (kQuantH) nvfp4_init_scale_table(sm.tab);
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (kGrouped) load_group_tiles(*gs, args.offs, args.G);   // contains __syncthreads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // the other CTAs of the cluster send row maxima to this CTA's barriers:
  // they must be initialised everywhere first
  if (kQuantH) cluster_sync_all();

  const int64_t M = args.M, N = args.N, K = args.K;
  // output columns per tile: BN, or 128 h columns (from 128 gate + 128 up rows of B)
  constexpr int kNT = kSwiGLU ? 128 : kBN;
  const int64_t F_ = args.ffn;                            // SwiGLU: B rows of the up half start at F
  const int64_t n_out = kSwiGLU ? F_ : N;
  const int64_t tiles_n = (n_out + kNT - 1) / kNT;
  const int64_t n_rt = (N + 127) / 128;                   // 128-row scale tiles of B (per group)
  const int64_t tiles_m = kGrouped ? gs->tpref[args.G] : (M + BM - 1) / BM;
  // output tiles strided over the CTAs; with h quantization, 128-row bands
  // strided over the clusters, CTA rank r of a cluster taking h tile r
  const int64_t nunits = kQuantH ? tiles_m : tiles_m * tiles_n;
  const int64_t unit0 = kQuantH ? cluster_id_x() : blockIdx.x;
  const int64_t ustep = kQuantH ? cluster_count_x() : gridDim.x;
  const int ctile = kQuantH ? static_cast<int>(cluster_ctarank()) : 0;
  auto tile_of = [&](int64_t u) {
    return kQuantH ? decode_band(u, ctile, gs, args.G) : decode_tile<kGrouped, kNT>(u, tiles_n, M, gs, args.G);
  };
  // first B row (within the group) of 128-row box h of a tile
  auto b_row0 = [&](const TileCoord& tc, int h) -> int64_t {
    return kSwiGLU ? tc.n0 + h * F_ : tc.n0 + h * 128;
  };
  const int64_t kbytes = kFmt == 0 ? K : (kFmt == 3 ? 2 * K : K / 2);
  const int ktiles = static_cast<int>((kbytes + kKBytes - 1) / kKBytes);
  const int64_t sf_kt = (K / F::kBlock + 3) / 4;          // scale tiles along K

  // producer index: 0 = warp 0 (A and the scale tiles), 1 + h = B box h
  const int prod = warp == 0 ? 0 : (warp >= 2 + L::kEpiWarps ? warp - 1 - L::kEpiWarps : -1);
  // B scale tiles of a tile's 128-row boxes
  auto b_scale_srcs = [&](const TileCoord& tc, const uint8_t* (&src)[L::kBRow128]) {
    const int64_t gbase = kGrouped ? static_cast<int64_t>(tc.g) * n_rt : 0;
#pragma unroll
    for (int h = 0; h < L::kBRow128; ++h) {
      // a 128-row block of B past N has zero data; reuse a valid scale tile for it
      const int64_t rt = b_row0(tc, h) / 128 < n_rt ? gbase + b_row0(tc, h) / 128 : gbase + tc.n0 / 128;
      src[h] = args.SB + rt * sf_kt * 512;
    }
  };
  auto scale_tiles_of_stage = [&](int kt, int64_t& sf0) -> int {
    sf0 = static_cast<int64_t>(kt) * F::kElemsPerStage / F::kElemsPerTile;
    return F::kSfTiles == 0 ? 0 : static_cast<int>(sf_kt - sf0 < F::kSfTiles ? sf_kt - sf0 : F::kSfTiles);
  };

  // Scale staging (kSepScales).  Each 512-byte scale tile is 32 rows of 16
  // bytes; every lane quarter of tensor memory gets the same 32 x 16 bytes,
  // row i in lane i of the quarter, over the tile's 4 columns (the layout the
  // block-scaled MMA reads).  A staging warp moves its quarter of every stage,
  // in order, as soon as the stage's scale tiles have landed, then arrives on
  // the stage's "scales ready" barrier.  Single GEMMs: the epilogue warps
  // (A's tiles by the first four, B's by the last four).  Grouped GEMMs with
  // BN = 256: the A producer and the two B producers (warps 0, 10, 11) and,
  // for lane quarter 1, epilogue warp 5 or the MMA warp (kEpiStager), A's and
  // B's tiles each, between their own waits.  A stage can only be refilled after its MMAs, which wait for its
  // scales, so a stage's barriers are never more than one phase ahead and its
  // shared-memory tiles and tensor-memory columns are never overwritten while
  // in use.
  const int cta_units = unit0 < nunits ? static_cast<int>((nunits - 1 - unit0) / ustep + 1) : 0;
  const int stage_total = kSepScales ? cta_units * ktiles : 0;
  const int squarter = warp & 3;
  const bool epi_warp = warp >= 2 && warp < 2 + L::kEpiWarps;
  // (grouped: warps 0, 10, 11 and 5 or 1, see kEpiStager)
  const bool stager = kWarpScales ? epi_warp
                                  : (kProdScales && (warp == 0 || warp >= 2 + L::kEpiWarps || warp == (kEpiStager ? 5 : 1)));
  const bool stage_a = kProdScales || (warp - 2) / 4 == 0;
  const bool stage_b = kProdScales || (warp - 2) / 4 == L::kBRow128 - 1;
  int staged = 0;
  auto stage_scales = [&](int j) {
    const int ss = j % L::kStages;
    const uint32_t tq = tmem + (static_cast<uint32_t>(squarter * 32) << 16) + L::kAccCols +
                        static_cast<uint32_t>(ss) * L::kSfColsPerStage;
    if (stage_a) {
#pragma unroll
      for (int jj = 0; jj < F::kSfTiles; ++jj)
        tmem_st_32x32b_x4(tq + 4 * jj, *reinterpret_cast<const uint4*>(sm.sfa[ss] + 512 * jj + 16 * lane));
    }
    if (stage_b) {
#pragma unroll
      for (int jj = 0; jj < F::kSfTiles; ++jj)
#pragma unroll
        for (int h = 0; h < L::kBRow128; ++h)
          tmem_st_32x32b_x4(tq + L::kSfaCols + (jj * L::kBRow128 + h) * 4,
                            *reinterpret_cast<const uint4*>(sm.sfb[ss] + (h * F::kSfTiles + jj) * 512 + 16 * lane));
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.sf_ready[ss]));
  };
  // Stages every landed stage below `limit` (warp-uniform, never blocks).
  auto stage_landed = [&](int limit) -> bool {
    bool any = false;
    if (kSepScales && stager) {
      const int lim = limit < stage_total ? limit : stage_total;
      while (staged < lim && __all_sync(0xffffffffu, mbar_test_wait(smem_u32(&sm.sf_full[staged % L::kStages]),
                                                                    (staged / L::kStages) & 1))) {
        stage_scales(staged++);
        any = true;
      }
    }
    return any;
  };
  // Warp-uniform bounded wait for the phase `parity` of barrier `bar`, staging
  // landed scales below `limit` meanwhile.  The producer and MMA warps sleep
  // in mbarrier.try_wait (first on the oldest stage they still have to move:
  // its scales land before the operands and before the stage is released, so
  // it is the next event; then on `bar`); the epilogue warps of single GEMMs
  // poll, as they have their own work between the tests.
  auto wait_staging = [&](uint32_t bar, uint32_t parity, int limit, int code) -> bool {
    const int lim = limit < stage_total ? limit : stage_total;
    uint64_t t0 = 0;
    while (true) {
      if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;
      if (stager && staged < lim) {
        const uint32_t sb = smem_u32(&sm.sf_full[staged % L::kStages]);
        const uint32_t sp = (staged / L::kStages) & 1;
        if (__all_sync(0xffffffffu, kProdScales ? mbar_try_wait(sb, sp) : mbar_test_wait(sb, sp))) {
          stage_scales(staged++);
          t0 = 0;
          continue;
        }
      } else if (kProdScales) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
      }
      if (__any_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&sm.abort) != 0)) return false;
      const uint64_t now = __shfl_sync(0xffffffffu, globaltimer(), 0);
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kWaitLimitNs) {
        if (lane == 0) {
          atomicCAS(err, 0, code);
          sm.abort = 1;
        }
        return false;
      }
    }
  };

  if (prod >= 0) {
    // ------------------------------------------------------------ producers
    if (kGather && prod == 0) {
      // Gathered A (dispatch fused into the GEMM): the 32 lanes copy each
      // tile's 128 rows from the token-major codes with 16-byte cp.async, 8
      // lanes per 128-byte row segment (4 rows per instruction), into the
      // swizzled K-major layout the MMA reads: the 16-byte chunk at offset o
      // of the tile goes to o ^ (((o >> 7) % atom rows) << 4).  Each lane
      // arrives on the stage's barrier once its copies have landed (the MMA
      // thread fences them for the tensor core's reads).  Lane 0 also loads
      // A's scale tiles (the dispatched rows' scales are laid out by the
      // quantizer, grouped, so they arrive as whole tiles); the B producers
      // load B's.
      constexpr uint32_t kAtomMask = kKBytes == 128 ? 7u : 3u;
      const uint32_t sub = static_cast<uint32_t>(lane & 7);   // 16-byte chunk of the row segment
      const int rq = lane >> 3;                                // row within a group of 4
      int it = 0;
      bool ok = true;
      for (int64_t u = unit0; ok && u < nunits; u += ustep) {
        const TileCoord tc = tile_of(u);
        __syncwarp();                          // the previous tile's row list is no longer read
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = lane + 32 * i;
          const int64_t t = args.a_rows[tc.a_row0 + (r < tc.rows ? r : 0)];
          sm.gtok[r] = static_cast<int32_t>(t < 0 ? 0 : (t >= args.a_src_rows ? args.a_src_rows - 1 : t));
        }
        __syncwarp();
        const uint8_t* sfa_src = args.SA + tc.sfa_tile * sf_kt * 512;
        for (int kt = 0; kt < ktiles; ++kt, ++it) {
          const int s = it % L::kStages;
          const uint32_t ph = (it / L::kStages) & 1;
          bool w = true;
          if (lane == 0) w = mbar_wait(smem_u32(&sm.empty[s]), ph ^ 1, err, kErrWaitProducer, &sm.abort);
          if (!__shfl_sync(0xffffffffu, w, 0)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&sm.full[s]);
          if (lane == 0) {
            int64_t sf0;
            const int nsf = scale_tiles_of_stage(kt, sf0);
            mbar_arrive_expect_tx(full, nsf * 512);   // the gathered rows arrive below, lane by lane
            bulk_load(smem_u32(sm.sfa[s]), sfa_src + sf0 * 512, nsf * 512, full);
          }
          const uint32_t a_s = smem_u32(sm.a[s]);
          const int64_t kb = static_cast<int64_t>(kt) * kKBytes + 16 * sub;
          const int64_t rem = kbytes - kb;
          const uint32_t nb = rem >= 16 ? 16u : (rem > 0 ? static_cast<uint32_t>(rem) : 0u);
#pragma unroll 8
          for (int i = 0; i < BM / 4; ++i) {
            const uint32_t r = static_cast<uint32_t>(4 * i + rq);
            const uint8_t* src = nb ? args.A + static_cast<int64_t>(sm.gtok[r]) * kbytes + kb : args.A;
            const uint32_t o = r * kKBytes + 16u * sub;
            cp_async_16(a_s + (o ^ (((o >> 7) & kAtomMask) << 4)), src, nb);
          }
          cp_async_arrive_noinc(full);
        }
      }
      cp_async_wait_all();                     // no copy may land after the block exits
      if (lane == 0 && !ok) {
        // let the scale copies already issued land before the block exits
        for (int j = (it > L::kStages ? it - L::kStages : 0); j < it; ++j)
          mbar_wait(smem_u32(&sm.full[j % L::kStages]), (j / L::kStages) & 1, err, kErrWaitTeardown,
                    nullptr, 100000000ull);
      }
    } else if (kProdScales || lane == 0) {
      // (with producer staging the whole warp runs the loop; lane 0 issues)
      int it = 0;
      bool ok = true;
      for (int64_t u = unit0; ok && u < nunits; u += ustep) {
        const TileCoord tc = tile_of(u);
        const uint8_t* sfa_src = args.SA + tc.sfa_tile * sf_kt * 512;
        const uint8_t* sfb_src[L::kBRow128];
        b_scale_srcs(tc, sfb_src);
        for (int kt = 0; kt < ktiles; ++kt, ++it) {
          const int s = it % L::kStages;
          const uint32_t ph = (it / L::kStages) & 1;
          if constexpr (kProdScales) {
            const uint32_t eb = smem_u32(&sm.empty[s]);
            if (!wait_staging(eb, ph ^ 1, it, kErrWaitProducer)) {
              ok = false;
              break;
            }
            if (lane != 0) continue;
          } else if (!mbar_wait(smem_u32(&sm.empty[s]), ph ^ 1, err, kErrWaitProducer, &sm.abort)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&sm.full[s]);
          // Each issuer also loads its scale tiles (A's, or its B box's).  When
          // the epilogue warps move them into tensor memory they land on the
          // stage's scale barrier: small, they arrive well before the operand
          // tiles and are moved while the operands are still in flight.
          // Otherwise they land with the operands.
          const uint32_t op_bytes = prod == 0 ? static_cast<uint32_t>(kTileABytes) : static_cast<uint32_t>(kBoxBytes);
          if constexpr (F::kSfTiles > 0) {
            int64_t sf0;
            const int nsf = scale_tiles_of_stage(kt, sf0);
            const uint32_t sbar = kSepScales ? smem_u32(&sm.sf_full[s]) : full;
            if (kSepScales) {
              mbar_arrive_expect_tx(sbar, nsf * 512);
              mbar_arrive_expect_tx(full, op_bytes);
            } else {
              mbar_arrive_expect_tx(full, op_bytes + nsf * 512);
            }
            if (prod == 0)
              bulk_load(smem_u32(sm.sfa[s]), sfa_src + sf0 * 512, nsf * 512, sbar);
            else
              bulk_load(smem_u32(sm.sfb[s]) + (prod - 1) * F::kSfTiles * 512, sfb_src[prod - 1] + sf0 * 512,
                        nsf * 512, sbar);
          } else {
            mbar_arrive_expect_tx(full, op_bytes);
          }
          if (prod == 0) {
            tma_load_2d(smem_u32(sm.a[s]), &tmap_a, kt * kKBytes, static_cast<int32_t>(tc.a_row0), full);
          } else {
            // B in 128-row boxes (a 128-row box is 16 KB; boxes stack in shared
            // memory), one issuer each, so every issuer moves about the same
            // bytes per stage
            const int h = prod - 1;
            if (kGrouped)
              tma_load_3d(smem_u32(sm.b[s]) + h * kBoxBytes, &tmap_b, kt * kKBytes,
                          static_cast<int32_t>(b_row0(tc, h)), tc.g, full);
            else
              tma_load_2d(smem_u32(sm.b[s]) + h * kBoxBytes, &tmap_b, kt * kKBytes,
                          static_cast<int32_t>(b_row0(tc, h)), full);
          }
        }
      }
      if constexpr (kProdScales) {
        // the stages this warp has not moved yet (the MMAs wait for them)
        if (ok) {
          const int last = stage_total;
          while (ok && staged < last) {
            const uint32_t fb = smem_u32(&sm.sf_full[staged % L::kStages]);
            const uint32_t fp = (staged / L::kStages) & 1;
            ok = wait_staging(fb, fp, staged, kErrWaitScales);
            if (ok) stage_scales(staged++);
          }
        }
      }
      if (!ok && lane == 0) {
        // let the copies already issued land before the block exits
        for (int j = (it > L::kStages ? it - L::kStages : 0); j < it; ++j) {
          mbar_wait(smem_u32(&sm.full[j % L::kStages]), (j / L::kStages) & 1, err, kErrWaitTeardown,
                    nullptr, 100000000ull);
          if (kSepScales)
            mbar_wait(smem_u32(&sm.sf_full[j % L::kStages]), (j / L::kStages) & 1, err, kErrWaitTeardown,
                      nullptr, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (when it stages a lane quarter the whole warp runs the loop; lane 0
    // issues)
    if (kMmaStages || lane == 0) {
      int it = 0, tcount = 0;
      bool ok = true;
      const uint32_t sf_base = tmem + L::kAccCols;
      for (int64_t u = unit0; ok && u < nunits; u += ustep, ++tcount) {
        const int as = tcount % L::kAccBufs;
        const uint32_t aph = (tcount / L::kAccBufs) & 1;
        if constexpr (kMmaStages) {
          if (!wait_staging(smem_u32(&sm.acc_empty[as]), aph ^ 1, it + 1, kErrWaitAccum)) {
            ok = false;
            break;
          }
        } else if (!mbar_wait(smem_u32(&sm.acc_empty[as]), aph ^ 1, err, kErrWaitAccum, &sm.abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + as * kBN;
        for (int kt = 0; kt < ktiles; ++kt, ++it) {
          const int s = it % L::kStages;
          const uint32_t ph = (it / L::kStages) & 1;
          if constexpr (kMmaStages) {
            // this warp's own quarter first (the scales land before the operands)
            if (!wait_staging(smem_u32(&sm.full[s]), ph, it + 1, kErrWaitConsumer) ||
                !wait_staging(smem_u32(&sm.sf_ready[s]), ph, it + 1, kErrWaitScales)) {
              ok = false;
              break;
            }
            if (lane != 0) continue;
          } else {
            if (!mbar_wait(smem_u32(&sm.full[s]), ph, err, kErrWaitConsumer, &sm.abort)) {
              ok = false;
              break;
            }
            if constexpr (kSepScales) {
              if (!mbar_wait(smem_u32(&sm.sf_ready[s]), ph, err, kErrWaitScales, &sm.abort)) {
                ok = false;
                break;
              }
            }
          }
          tc_fence_after();
          if (kGather) fence_proxy_async_smem();   // the gathered rows were written by cp.async
          // tensor-memory scale layout per stage: A -> 4 columns per K
          // sub-tile; B -> (4 columns x kBRow128) per K sub-tile, the 128-row
          // blocks adjacent
          const uint32_t tsfa = sf_base + s * L::kSfColsPerStage;
          const uint32_t tsfb = tsfa + L::kSfaCols;
          if constexpr (F::kSfTiles > 0 && !kSepScales) {
            int64_t sf0;
            const int nsf = scale_tiles_of_stage(kt, sf0);
            for (int j = 0; j < nsf; ++j) {
              tc_cp_32x128b_x4(tsfa + 4 * j, smem_desc(smem_u32(sm.sfa[s]) + 512 * j, 128, 128, kSwizzleNone));
#pragma unroll
              for (int h = 0; h < L::kBRow128; ++h)
                tc_cp_32x128b_x4(tsfb + (j * L::kBRow128 + h) * 4,
                                 smem_desc(smem_u32(sm.sfb[s]) + (h * F::kSfTiles + j) * 512, 128, 128,
                                           kSwizzleNone));
            }
          }
          const int64_t krem = K - static_cast<int64_t>(kt) * F::kElemsPerStage;
          const int nmma = static_cast<int>(krem >= F::kElemsPerStage
                                                ? F::kElemsPerStage / F::kElemsPerMma
                                                : (krem + F::kElemsPerMma - 1) / F::kElemsPerMma);
          const uint32_t a0 = smem_u32(sm.a[s]), b0 = smem_u32(sm.b[s]);
          // MXFP8: scale id of the stage's first MMA within its 4-scale tile;
          // MXFP4: MMA kk takes scales 2(kk%2), 2(kk%2)+1 of tile kk/2
          const uint32_t sf_id0 = static_cast<uint32_t>((static_cast<int64_t>(kt) * F::kElemsPerStage / 32) & 3);
          for (int kk = 0; kk < nmma; ++kk) {
            const uint64_t ad = smem_desc(a0 + kk * 32, 16, kAtomSbo, kSwizzle);
            const uint64_t bd = smem_desc(b0 + kk * 32, 16, kAtomSbo, kSwizzle);
            const uint32_t acc = (kt > 0 || kk > 0) ? 1u : 0u;
            if (kFmt == 3)
              tc_mma_bf16(d_tmem, ad, bd, make_idesc_bf16(kBN), acc);
            else if (kFmt == 0)
              tc_mma_mxf8(d_tmem, ad, bd, make_idesc(0, kBN, sf_id0 + kk), tsfa, tsfb, acc);
            else if (kFmt == 2)
              tc_mma_mxf4(d_tmem, ad, bd, make_idesc(2, kBN, 2u * (kk & 1)), tsfa + 4 * (kk >> 1),
                          tsfb + 4 * L::kBRow128 * (kk >> 1), acc);
            else
              tc_mma_nvf4(d_tmem, ad, bd, make_idesc(1, kBN, 0), tsfa + 4 * kk,
                          tsfb + 4 * L::kBRow128 * kk, acc);
          }
          tc_commit(smem_u32(&sm.empty[s]));   // stage free once these MMAs finish
        }
        if (!ok) break;
        if (lane == 0) tc_commit(smem_u32(&sm.acc_full[as]));  // accumulator ready for the epilogue
      }
      // no MMA may be in flight when tensor memory is released
      if (lane == 0) {
        tc_commit(smem_u32(&sm.drain));
        mbar_wait(smem_u32(&sm.drain), 0, err, kErrWaitTeardown, nullptr, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2 .. 1 + kEpiWarps)
    const int ew = warp - 2;
    const int quarter = warp & 3;              // tcgen05.ld lane quarter of this warp
    const int col0 = (ew / 4) * 128;           // this warp's 128 accumulator columns
    const int r_in_tile = quarter * 32 + lane;
    // Waits (warp-uniformly, bounded) for accumulator `as` to fill, staging
    // (single GEMMs; warp 5 of the SwiGLU GEMM) every stage that lands
    // meanwhile.
    auto wait_accumulator = [&](int as, uint32_t aph) -> bool {
      const uint32_t fb = smem_u32(&sm.acc_full[as]);
      if constexpr (kWarpScales || kEpiStager) {
        if (stager)
          return wait_staging(fb, aph, stage_total, staged < stage_total ? kErrWaitScales : kErrWaitEpilogue);
      }
      return __all_sync(0xffffffffu, mbar_wait(fb, aph, err, kErrWaitEpilogue, &sm.abort));
    };
    int tcount = 0;
    for (int64_t u = unit0; u < nunits; u += ustep, ++tcount) {
      const int as = tcount % L::kAccBufs;
      const uint32_t aph = (tcount / L::kAccBufs) & 1;
      // Grouped GEMMs read the tile's FP32 decode scales before the wait, so
      // the loads complete while the accumulator fills (not with h
      // quantization, nor in single GEMMs: their epilogues have no registers
      // to spare; measured slower).
      constexpr bool kEarlyScales = kGrouped && !kQuantH;
      TileCoord tc;
      bool row_ok = false;
      int64_t m = 0;
      auto load_coords = [&]() {
        tc = tile_of(u);
        row_ok = r_in_tile < tc.rows;
        m = tc.a_row0 + r_in_tile;
      };
      auto load_sa = [&]() -> float {
        float v = 1.f;
        if (row_ok) {
          if (args.a32_mode == 1) {
            int64_t src = m;
            if (kGather) {
              src = args.a_rows[m];
              src = src < 0 ? 0 : (src >= args.a_src_rows ? args.a_src_rows - 1 : src);
            }
            v = args.A32[src];
          } else if (args.a32_mode == 2) {
            v = args.A32[0];
          }
        }
        return v;
      };
      auto load_sg = [&]() -> float {
        if (kGrouped && args.B32 != nullptr) return args.B32[tc.g];
        if (!kGrouped && args.b32_mode == 2) return args.B32[0];
        return 1.f;
      };
      float sa = 1.f, sg = 1.f;
      if constexpr (kEarlyScales) {
        load_coords();
        sa = load_sa();
        sg = load_sg();
      }
      const bool b_row = !kGrouped && args.b32_mode == 1;
      if (!wait_accumulator(as, aph)) break;
      tc_fence_after();
      uint32_t r[4][32];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + as * kBN;
      // SwiGLU: this warp's 64 h columns need gate columns 64*half.. (chunks 0,
      // 1) and the matching up columns 128 + 64*half.. (chunks 2, 3)
      const int half = ew / 4;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        tmem_ld_32x32b_x32(taddr + (kSwiGLU ? (ch < 2 ? 64 * half + 32 * ch : 128 + 64 * half + 32 * (ch - 2))
                                            : col0 + ch * 32),
                           r[ch]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.acc_empty[as]));   // accumulator drained into registers
      if constexpr (kWarpScales || kEpiStager) stage_landed(stage_total);
      if constexpr (!kEarlyScales) {
        load_coords();
        sa = load_sa();
        sg = load_sg();
      }
      // the two FP32 decode scales are combined first: acc * A32 alone can
      // overflow for tokens whose amax is near the bf16 maximum
      const float s_ab = __fmul_rn(sa, sg);
      if constexpr (kSwiGLU && !kQuantH) {
        // g and u rounded to bf16 exactly as the unfused gate|up output would
        // be, then h = RN_bf16(silu(g) * u): 64 columns, 128 contiguous bytes.
        // Every lane runs the loop (rows past the tile's end store nothing),
        // so the warp can stage scales half-way through.
        uint4* hrow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.C) + m * args.ldc + tc.n0 + 64 * half);
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          if (kEpiStager && q8 == 4) stage_landed(stage_total);   // (warp-uniform here)
          uint32_t p[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float hv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = q8 * 8 + j * 2 + e;
              const float g = bf16_round(__fmul_rn(__uint_as_float(r[c >> 5][c & 31]), s_ab));
              const float uu = bf16_round(__fmul_rn(__uint_as_float(r[2 + (c >> 5)][c & 31]), s_ab));
              hv[e] = silu_mul(g, uu);
            }
            p[j] = pack_bf16x2(hv[0], hv[1]);
          }
          if (row_ok) hrow[q8] = make_uint4(p[0], p[1], p[2], p[3]);
        }
        continue;
      }
      if constexpr (kQuantH) {
        // as above, the 64 columns kept as bf16 pairs (column 2j in the low
        // half of hp[j]; the bf16 h also stored when C is given), then
        // quantized
        uint32_t hp[32];
        uint4* hrow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.C) + m * args.ldc + tc.n0 + 64 * half);
        const bool store_h = row_ok && args.C != nullptr;
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float hv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = q8 * 8 + j * 2 + e;
              const float g = bf16_round(__fmul_rn(__uint_as_float(r[c >> 5][c & 31]), s_ab));
              const float uu = bf16_round(__fmul_rn(__uint_as_float(r[2 + (c >> 5)][c & 31]), s_ab));
              hv[e] = silu_mul(g, uu);
            }
            hp[4 * q8 + j] = pack_bf16x2(hv[0], hv[1]);
          }
          if (store_h) hrow[q8] = make_uint4(hp[4 * q8], hp[4 * q8 + 1], hp[4 * q8 + 2], hp[4 * q8 + 3]);
        }
        {
          // Per-token NVFP4 of h.  This thread's row maximum over its 64
          // columns goes to slot (tile, half) of every CTA of the cluster;
          // once all 2 x tiles maxima of the band's rows are in (barrier of
          // this band's buffer), each row's amax gives S_enc and the thread
          // encodes its 4 blocks of 16.  Two buffers alternate between
          // bands: a CTA can only send band b + 2's maxima after receiving
          // everyone's band b + 1 maxima, which each sends after it has read
          // band b's buffer.
          uint32_t mx2 = 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) mx2 = amax2(mx2, hp[j]);
          const float hmax = abs_halves_max(mx2);
          const int buf = tcount & 1;
          const int ntile = static_cast<int>(F_ / 128);
          float* red = reinterpret_cast<float*>(&sm.cstage[0][0]) + buf * (2 * kMaxClusterTiles * 128);
          const uint32_t slot = smem_u32(red + (2 * ctile + half) * 128 + r_in_tile);
#pragma unroll 1
          for (int p = 0; p < ntile; ++p) st_cluster_u32(mapa_shared(slot, static_cast<uint32_t>(p)), __float_as_uint(hmax));
          __syncwarp();
          const uint32_t bar = smem_u32(&sm.hmax_full[buf]);
          if (lane == 0) {
#pragma unroll 1
            for (int p = 0; p < ntile; ++p) mbar_arrive_cluster(mapa_shared(bar, static_cast<uint32_t>(p)));
          }
          if (!__all_sync(0xffffffffu, mbar_wait_cluster(bar, (tcount >> 1) & 1, err, kErrWaitCluster, &sm.abort)))
            break;
          float amax = 0.f;
#pragma unroll 1
          for (int sl = 0; sl < 2 * ntile; ++sl) amax = fmaxf(amax, red[sl * 128 + r_in_tile]);
          float senc, sdec;
          nvfp4_scales(amax, senc, sdec);
          uint2 cw[4];
          uint32_t sw = 0;
#pragma unroll
          for (int bk = 0; bk < 4; ++bk) {
            const uint4 a = make_uint4(hp[8 * bk], hp[8 * bk + 1], hp[8 * bk + 2], hp[8 * bk + 3]);
            const uint4 b = make_uint4(hp[8 * bk + 4], hp[8 * bk + 5], hp[8 * bk + 6], hp[8 * bk + 7]);
            sw |= nvfp4_encode_block(a, b, senc, sm.tab, cw[bk]) << (8 * bk);
          }
          // scale word of h's 4-block group (tc.n0 + 64 half) / 64 in scale row
          // (band, row): zero for the padding rows of a group's last band
          const int64_t srow = tc.sfa_tile * BM + r_in_tile;
          const int64_t k4 = (tc.n0 + 64 * half) / 64;
          *reinterpret_cast<uint32_t*>(args.qh_scales + sf_row_base(srow, F_ / 64) + k4 * 512) = row_ok ? sw : 0u;
          if (row_ok) {
            uint4* qrow = reinterpret_cast<uint4*>(args.qh + m * (F_ / 2) + (tc.n0 + 64 * half) / 2);
            qrow[0] = make_uint4(cw[0].x, cw[0].y, cw[1].x, cw[1].y);
            qrow[1] = make_uint4(cw[2].x, cw[2].y, cw[3].x, cw[3].y);
            if (ctile == 0 && half == 0) args.qh_s32[m] = sdec;
          }
        }
        continue;
      }
      // Whole 32-row slabs leave through shared memory and bulk tensor stores
      // (full lines, asynchronous); a slab that crosses the end of its group
      // or that accumulates into C is stored directly, row by row.
      if (quarter * 32 + 32 <= tc.rows && !args.accumulate) {
        const uint32_t stage = smem_u32(sm.cstage[ew]);
        const int32_t y = static_cast<int32_t>(tc.a_row0 + quarter * 32);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          if ((kWarpScales || kEpiStager) && ch > 0) stage_landed(stage_total);
          const int64_t n0 = tc.n0 + col0 + ch * 32;
          if (n0 >= N) break;
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float sc = s_ab;
            if (b_row) sc = (n0 + j < N) ? __fmul_rn(sa, args.B32[n0 + j]) : 0.f;
            v[j] = __fmul_rn(__uint_as_float(r[ch][j]), sc);
          }
#pragma unroll
          for (int half = 0; half < (args.out_bf16 ? 1 : 2); ++half) {
            if (lane == 0) bulk_wait_read_all();      // staging buffer free again
            __syncwarp();
            uint4* dst = reinterpret_cast<uint4*>(sm.cstage[ew] + lane * 64);
            if (args.out_bf16) {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t p[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  p[j] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[8 * q4 + 2 * j]))) |
                         (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[8 * q4 + 2 * j + 1]))) << 16);
                dst[q4] = make_uint4(p[0], p[1], p[2], p[3]);
              }
            } else {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                dst[q4] = make_uint4(__float_as_uint(v[16 * half + 4 * q4]), __float_as_uint(v[16 * half + 4 * q4 + 1]),
                                     __float_as_uint(v[16 * half + 4 * q4 + 2]), __float_as_uint(v[16 * half + 4 * q4 + 3]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmap_c, static_cast<int32_t>(n0 + 16 * half), y, stage);
              bulk_commit_group();
            }
          }
        }
        continue;
      }
      if (!row_ok) continue;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int64_t n0 = tc.n0 + col0 + ch * 32;
        if (n0 >= N) break;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float sc = s_ab;
          if (b_row) sc = (n0 + j < N) ? __fmul_rn(sa, args.B32[n0 + j]) : 0.f;
          v[j] = __fmul_rn(__uint_as_float(r[ch][j]), sc);
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

  if (warp >= 2 && lane == 0) bulk_wait_all();   // every bulk store has landed
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // no CTA of a cluster leaves while another may still write to its shared memory
  if (kQuantH) cluster_sync_all();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int kFmt, bool kGrouped, int kBN, int kMode = 0>
cudaError_t launch_variant(const GemmArgs& a, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                           const CUtensorMap& tmap_c, int sm_count, cudaStream_t stream) {
  using L = Layout<kFmt, kGrouped, kBN, kMode>;
  const int64_t tiles_n = (kMode & kModeSwiGLU) ? (a.ffn + 127) / 128 : (a.N + kBN - 1) / kBN;
  int64_t tiles_m = (a.M + BM - 1) / BM;
  if (a.grouped) tiles_m += a.G;                  // upper bound: every group pads a tile
  const int64_t ntiles = tiles_m * tiles_n;
  const unsigned grid = static_cast<unsigned>(ntiles < sm_count ? ntiles : sm_count);
  if (grid == 0) return cudaSuccess;
  auto k = bs_gemm_kernel<kFmt, kGrouped, kBN, kMode>;
  constexpr size_t smem = sizeof(GemmSmem<kFmt, kGrouped, kBN, kMode>) + (kGrouped ? sizeof(GroupTiles) : 0) + 1024;
  static_assert(smem <= 227 * 1024, "shared memory over the per-block limit");
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k<<<grid, L::kThreads, smem, stream>>>(tmap_a, tmap_b, tmap_c, a);
  return cudaGetLastError();
}

// The SwiGLU grouped GEMM with h quantized: clusters of F / 128 CTAs (one per
// h tile of a band), as many clusters as can be resident at once (each
// persistent over the bands).
cudaError_t launch_quant_h(const GemmArgs& a, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                           const CUtensorMap& tmap_c, cudaStream_t stream) {
  constexpr int kMode = kModeSwiGLU | kModeQuantH;
  using L = Layout<1, true, 256, kMode>;
  const int cs = static_cast<int>(a.ffn / 128);
  if (cs < 1 || cs > kMaxClusterTiles || a.ffn % 128 != 0) return cudaErrorInvalidValue;
  auto k = bs_gemm_kernel<1, true, 256, kMode>;
  constexpr size_t smem = sizeof(GemmSmem<1, true, 256, kMode>) + sizeof(GroupTiles) + 1024;
  static_assert(smem <= 227 * 1024, "shared memory over the per-block limit");
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(L::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // clusters that fit on the GPU at once (cached per device and cluster size)
  static int cache[64][kMaxClusterTiles + 1] = {};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (cache[dev][cs] == 0) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>((sms / cs) * cs), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    cache[dev][cs] = n;
  }
  const int64_t bands = (a.M + BM - 1) / BM + a.G;     // upper bound: every group pads a band
  const int64_t ncl = bands < cache[dev][cs] ? bands : cache[dev][cs];
  if (ncl == 0) return cudaSuccess;
  cfg.gridDim = dim3(static_cast<unsigned>(ncl * cs), 1, 1);
  e = cudaLaunchKernelEx(&cfg, k, tmap_a, tmap_b, tmap_c, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bs_gemm(const GemmArgs& a, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                           const CUtensorMap& tmap_c, int sm_count, cudaStream_t stream) {
  constexpr int BN = MX8Q_GEMM_BN;
  const int mode = (a.a_rows != nullptr ? kModeGather : 0) | (a.ffn > 0 ? kModeSwiGLU : 0);
  if (a.qh != nullptr) {
    if (mode != kModeSwiGLU || a.fmt != 1 || !a.grouped || BN != 256) return cudaErrorInvalidValue;
    return launch_quant_h(a, tmap_a, tmap_b, tmap_c, stream);
  }
  if (mode != 0) {
    // fused MoE modes: NVFP4 grouped only
    if (a.fmt != 1 || !a.grouped || BN != 256) return cudaErrorInvalidValue;
    if (mode == kModeGather) return launch_variant<1, true, 256, kModeGather>(a, tmap_a, tmap_b, tmap_c, sm_count, stream);
    if (mode == kModeSwiGLU) return launch_variant<1, true, 256, kModeSwiGLU>(a, tmap_a, tmap_b, tmap_c, sm_count, stream);
    return launch_variant<1, true, 256, kModeGather | kModeSwiGLU>(a, tmap_a, tmap_b, tmap_c, sm_count, stream);
  }
  if (a.fmt == 0) {
    return a.grouped ? launch_variant<0, true, BN>(a, tmap_a, tmap_b, tmap_c, sm_count, stream)
                     : launch_variant<0, false, BN>(a, tmap_a, tmap_b, tmap_c, sm_count, stream);
  }
  if (a.fmt == 3) {
    return a.grouped ? cudaErrorInvalidValue
                     : launch_variant<3, false, BN>(a, tmap_a, tmap_b, tmap_c, sm_count, stream);
  }
  if (a.fmt == 2) {
    return a.grouped ? launch_variant<2, true, BN>(a, tmap_a, tmap_b, tmap_c, sm_count, stream)
                     : launch_variant<2, false, BN>(a, tmap_a, tmap_b, tmap_c, sm_count, stream);
  }
  return a.grouped ? launch_variant<1, true, BN>(a, tmap_a, tmap_b, tmap_c, sm_count, stream)
                   : launch_variant<1, false, BN>(a, tmap_a, tmap_b, tmap_c, sm_count, stream);
}

}  // namespace mx8q
