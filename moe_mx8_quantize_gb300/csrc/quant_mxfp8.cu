// MXFP8 quantization: 1x32 E4M3 blocks with one E8M0 (power-of-two) scale,
// rowwise and columnwise copies from ONE read of the bf16 input.  The same
// kernel makes MXFP4 (kFP4): 1x32 E2M1 blocks under one E8M0 scale, packed
// two codes per byte ("NVIDIA presenta una metodologia de preentrenamiento
// de 4 bits utilizando NVFP4", section "Que es realmente NVFP4").
//
// "Miles Blackwell RL Cambia la Uniformidad BF16 por MXFP8 y NVFP4 Nativos",
// section "La Compatibilidad de Miles Blackwell Ahora Abarca Todo el Ciclo de
// RL": 32 consecutive E4M3 values share one E8M0 scale.  Section "Un
// Cuantizador Compartido Es el Mecanismo Real": scale blocks must follow the
// GEMM reduction axis, forward and backward reduce along different axes, so
// a rowwise and a columnwise copy are both made from the high-precision input
// (not by requantizing one copy).
//
// Design: a persistent grid; each CTA streams 128x128 bf16 tiles through a
// TMA -> shared-memory ring (2 stages, 32 KB each).  One launch may cover up
// to kQuantBatchMax tensors (the X, W and dY of a linear layer): their tiles
// form one list, so a small tensor's latency hides behind the others' tiles.  From the same staged
// tile the CTA emits
//   rowwise : 16 threads per row, 8 elements each (one 16-byte smem read),
//             4-thread shuffle for the 1x32 block amax, 8-byte stores;
//   colwise : one thread per (column pair, 32-row block), 32 u32 smem reads
//             down the column pair, 32-byte stores into the transposed copy;
// and both 128x4 scale tiles (exactly one 512-byte tensor-core tile each),
// staged in shared memory and written with 16-byte stores.  |x| maxima are
// taken two bf16 values per instruction and the products x * 2^-e two per
// instruction.
#include "device.cuh"
#include "kernels.h"

namespace mx8q {

namespace {

constexpr int kTile = 128;            // rows and columns of a staged tile
constexpr int kStages = 2;
constexpr int kThreads = 256;
constexpr int kTileBytes = kTile * kTile * 2;

struct __align__(16) QuantSmem {
  uint8_t tile[kStages][kTileBytes];
  uint8_t srow[2][512];               // double-buffered scale staging
  uint8_t scol[2][512];
  uint64_t full[kStages];
  int abort;
};

// Shared exponent of a block from its amax (an f32 holding a bf16 value):
// the smallest e with amax <= emax * 2^e, clamped to [-127, 127], for the
// element maximum emax = 448 = 1.75 * 2^8 (E4M3) or 6 = 1.5 * 2^2 (E2M1).
// amax = (1 + f) * 2^k  ->  E4M3: e = k - 8 if (1 + f) <= 1.75 else k - 7;
//                           E2M1: e = k - 2 if (1 + f) <= 1.5  else k - 1.
template <bool kFP4>
__device__ __forceinline__ int mx_block_exp(float amax) {
  const uint32_t u = __float_as_uint(amax);
  const int ef = static_cast<int>((u >> 23) & 0xFF);
  if (ef == 0) return -127;                      // zero or subnormal: k <= -127
  const int k = ef - 127;
  const uint32_t frac = u & 0x7FFFFFu;
  int e = kFP4 ? ((frac <= 0x400000u) ? k - 2 : k - 1)    // 0x400000 / 2^23 = 0.5
               : ((frac <= 0x600000u) ? k - 8 : k - 7);   // 0x600000 / 2^23 = 0.75
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as an f32 (e in [-127, 127]); exact.
__device__ __forceinline__ float exp2_neg(int e) {
  const int b = 127 - e;                         // biased exponent of 2^-e
  if (b >= 1) return __uint_as_float(static_cast<uint32_t>(b) << 23);
  return __uint_as_float(0x00400000u >> (-b));   // 2^-127 and below: subnormal
}

__device__ __forceinline__ int swz(int r, int k) {  // offset inside a 128x4 tile
  return (r & 31) * 16 + ((r >> 5) & 3) * 4 + (k & 3);
}

template <bool kRow, bool kCol, bool kFP4>
__global__ void __launch_bounds__(kThreads) mxfp8_quant_kernel(const __grid_constant__ QuantBatch b, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  QuantSmem& sm = *reinterpret_cast<QuantSmem*>(
      smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023));
  const int tid = threadIdx.x;
  const int64_t ntiles = b.ntiles;

  if (tid == 0) {
    for (int i = 0; i < b.n; ++i) prefetch_tmap(&b.maps[i]);
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
    sm.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // tile t of the batch -> tensor i and the tile's row / column of it
  auto locate = [&](int64_t t, int& i, int64_t& tr, int64_t& tc) {
    i = 0;
#pragma unroll
    for (int j = 1; j < kQuantBatchMax; ++j)
      if (j < b.n && t >= b.t[j].tile0) i = j;
    const int64_t local = t - b.t[i].tile0;
    const int64_t tiles_c = (b.t[i].C + kTile - 1) / kTile;
    tr = local / tiles_c;
    tc = local % tiles_c;
  };

  auto issue = [&](int64_t t, int stage) {
    int i;
    int64_t tr, tc;
    locate(t, i, tr, tc);
    const uint32_t bar = smem_u32(&sm.full[stage]);
    mbar_arrive_expect_tx(bar, kTileBytes);
    tma_load_2d(smem_u32(sm.tile[stage]), &b.maps[i], static_cast<int32_t>(tc * kTile),
                static_cast<int32_t>(tr * kTile), bar);
  };

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      const int64_t t = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
      if (t < ntiles) issue(t, s);
    }
  }

  int it = 0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
    const int stage = it % kStages;
    const uint32_t parity = (it / kStages) & 1;
    const bool ok = mbar_wait(smem_u32(&sm.full[stage]), parity, err, kErrWaitConsumer, &sm.abort);
    if (!__syncthreads_and(ok)) break;  // every thread leaves together

    int ti;
    int64_t tr, tc;
    locate(t, ti, tr, tc);
    const QuantTensor& qt = b.t[ti];
    const int64_t R = qt.R, C = qt.C;
    uint8_t* __restrict__ q_row = qt.q_row;
    uint8_t* __restrict__ s_row = qt.s_row;
    uint8_t* __restrict__ q_col = qt.q_col;
    uint8_t* __restrict__ s_col = qt.s_col;
    const int64_t tiles_c = (C + kTile - 1) / kTile;
    const int64_t tiles_r = (R + kTile - 1) / kTile;
    const int64_t r0 = tr * kTile, c0 = tc * kTile;
    const uint8_t* tile = sm.tile[stage];
    uint8_t* srow = sm.srow[it & 1];
    uint8_t* scol = sm.scol[it & 1];

    if (kRow) {
      // 16 threads per row, 8 elements per thread, 16 rows per pass.
      const int cchunk = tid & 15;         // 8-element chunk within the row
      const int blk = cchunk >> 2;         // 32-element block (0..3)
#pragma unroll 2
      for (int pass = 0; pass < kTile / 16; ++pass) {
        const int lr = pass * 16 + (tid >> 4);
        const uint4 w = *reinterpret_cast<const uint4*>(tile + lr * (kTile * 2) + cchunk * 16);
        // |x| maxima two bf16 values per instruction, then the 4-thread block maximum
        float amax = abs_halves_max(amax2(amax2(w.x, w.y), amax2(w.z, w.w)));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int e = mx_block_exp<kFP4>(amax);
        const uint64_t sc = f32x2_splat(exp2_neg(e));
        float v[8];                                  // x * 2^-e, two products per instruction
        mul_bf16x2(w.x, sc, v[0], v[1]);
        mul_bf16x2(w.y, sc, v[2], v[3]);
        mul_bf16x2(w.z, sc, v[4], v[5]);
        mul_bf16x2(w.w, sc, v[6], v[7]);
        const int64_t gr = r0 + lr, gc = c0 + cchunk * 8;
        if (kFP4) {
          const uint32_t p = cvt_e2m1x8(v);        // 8 codes, element 0 in the low nibble
          if (gr < R && gc < C) *reinterpret_cast<uint32_t*>(q_row + gr * (C / 2) + gc / 2) = p;
        } else {
          const uint32_t p0 = cvt_e4m3x2(v[0], v[1]) | (static_cast<uint32_t>(cvt_e4m3x2(v[2], v[3])) << 16);
          const uint32_t p1 = cvt_e4m3x2(v[4], v[5]) | (static_cast<uint32_t>(cvt_e4m3x2(v[6], v[7])) << 16);
          if (gr < R && gc < C) *reinterpret_cast<uint2*>(q_row + gr * C + gc) = make_uint2(p0, p1);
        }
        if ((tid & 3) == 0) srow[swz(lr, blk)] = static_cast<uint8_t>(e + 127);
      }
    }

    if (kCol) {
      // thread -> (column pair cp, 32-row block rb)
      const int cp = tid & 63, rb = tid >> 6;
      uint32_t w[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        w[i] = *reinterpret_cast<const uint32_t*>(tile + (rb * 32 + i) * (kTile * 2) + cp * 4);
      // both columns' |x| maxima at once: low halves column 2cp, high halves 2cp + 1
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) m = amax2(m, w[i]);
      const float a0 = __uint_as_float((m << 16) & 0x7FFFFFFFu), a1 = __uint_as_float(m & 0x7FFF0000u);
      const int e0 = mx_block_exp<kFP4>(a0), e1 = mx_block_exp<kFP4>(a1);
      const uint64_t s0 = f32x2_splat(exp2_neg(e0)), s1 = f32x2_splat(exp2_neg(e1));
      const int64_t gc0 = c0 + 2 * cp, gr = r0 + rb * 32;
      if (kFP4) {
        // 32 codes per column: four 8-code words each
        uint32_t o0[4], o1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float p0[8], p1[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t xa = w[8 * j + 2 * i], xb = w[8 * j + 2 * i + 1];
            mul_f32x2(bf16_lo(xa), bf16_lo(xb), s0, p0[2 * i], p0[2 * i + 1]);
            mul_f32x2(bf16_hi(xa), bf16_hi(xb), s1, p1[2 * i], p1[2 * i + 1]);
          }
          o0[j] = cvt_e2m1x8(p0);
          o1[j] = cvt_e2m1x8(p1);
        }
        if (gr < R) {
          if (gc0 < C) *reinterpret_cast<uint4*>(q_col + gc0 * (R / 2) + gr / 2) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
          if (gc0 + 1 < C)
            *reinterpret_cast<uint4*>(q_col + (gc0 + 1) * (R / 2) + gr / 2) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
        }
      } else {
        uint32_t o0[8], o1[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t x0 = w[4 * j], x1 = w[4 * j + 1], x2 = w[4 * j + 2], x3 = w[4 * j + 3];
          float p[8];
          mul_f32x2(bf16_lo(x0), bf16_lo(x1), s0, p[0], p[1]);
          mul_f32x2(bf16_lo(x2), bf16_lo(x3), s0, p[2], p[3]);
          mul_f32x2(bf16_hi(x0), bf16_hi(x1), s1, p[4], p[5]);
          mul_f32x2(bf16_hi(x2), bf16_hi(x3), s1, p[6], p[7]);
          o0[j] = cvt_e4m3x2(p[0], p[1]) | (static_cast<uint32_t>(cvt_e4m3x2(p[2], p[3])) << 16);
          o1[j] = cvt_e4m3x2(p[4], p[5]) | (static_cast<uint32_t>(cvt_e4m3x2(p[6], p[7])) << 16);
        }
        if (gr < R) {
          if (gc0 < C) {
            uint4* dst = reinterpret_cast<uint4*>(q_col + gc0 * R + gr);
            dst[0] = make_uint4(o0[0], o0[1], o0[2], o0[3]);
            dst[1] = make_uint4(o0[4], o0[5], o0[6], o0[7]);
          }
          if (gc0 + 1 < C) {
            uint4* dst = reinterpret_cast<uint4*>(q_col + (gc0 + 1) * R + gr);
            dst[0] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
            dst[1] = make_uint4(o1[4], o1[5], o1[6], o1[7]);
          }
        }
      }
      scol[swz(2 * cp, rb)] = static_cast<uint8_t>(e0 + 127);
      scol[swz(2 * cp + 1, rb)] = static_cast<uint8_t>(e1 + 127);
    }

    __syncthreads();  // tile fully read; scale staging complete

    // One 512-byte tensor-core scale tile per copy.
    if (kRow && tid < 32) {
      uint8_t* dst = s_row + (tr * tiles_c + tc) * 512;
      reinterpret_cast<uint4*>(dst)[tid] = reinterpret_cast<const uint4*>(srow)[tid];
    }
    if (kCol && tid >= 32 && tid < 64) {
      uint8_t* dst = s_col + (tc * tiles_r + tr) * 512;
      reinterpret_cast<uint4*>(dst)[tid - 32] = reinterpret_cast<const uint4*>(scol)[tid - 32];
    }
    if (tid == 0) {
      const int64_t nt = t + static_cast<int64_t>(kStages) * gridDim.x;
      if (nt < ntiles) issue(nt, stage);
    }
  }

  // Teardown after an aborted wait: let issued copies land before exit.
  if (sm.abort && tid == 0) {
    int j = it;
    for (int64_t t = blockIdx.x + static_cast<int64_t>(it) * gridDim.x; t < ntiles && j < it + kStages;
         t += gridDim.x, ++j)
      mbar_wait(smem_u32(&sm.full[j % kStages]), (j / kStages) & 1, err, kErrWaitTeardown, nullptr);
  }
}

}  // namespace

size_t mxfp8_quant_smem_bytes() { return sizeof(QuantSmem) + 1024; }

cudaError_t launch_mxfp8_quant(const QuantBatch& batch, bool row, bool col, bool fp4, int* err, int sm_count,
                               cudaStream_t stream) {
  const int64_t ntiles = batch.ntiles;
  if (ntiles == 0) return cudaSuccess;
  const size_t smem = mxfp8_quant_smem_bytes();
  auto kern = fp4 ? (row ? (col ? mxfp8_quant_kernel<true, true, true> : mxfp8_quant_kernel<true, false, true>)
                         : mxfp8_quant_kernel<false, true, true>)
                  : (row ? (col ? mxfp8_quant_kernel<true, true, false> : mxfp8_quant_kernel<true, false, false>)
                         : mxfp8_quant_kernel<false, true, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t grid = ntiles < static_cast<int64_t>(sm_count) * per_sm ? ntiles
                                                                        : static_cast<int64_t>(sm_count) * per_sm;
  kern<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(batch, err);
  return cudaGetLastError();
}

}  // namespace mx8q
