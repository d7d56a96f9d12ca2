// Two-level NVFP4 quantization with the FP32 scale computed online per
// token (or per group / per tensor), fused into one kernel that emits the
// packed E2M1 values, the E4M3 block scales (tensor-core tile layout) and the
// FP32 decode scale.
//
// "Miles Blackwell RL Cambia la Uniformidad BF16 por MXFP8 y NVFP4 Nativos",
// section "La Compatibilidad...": NVFP4 = E2M1 values with an E4M3 scale per
// 16-value block plus a second FP32 scale, computed per token so a token's
// representation does not depend on the batch.  Section "Un Cuantizador
// Compartido Es el Mecanismo Real": the per-token FP32 scale is computed
// online inside the activation quantizer, which emits packed FP4, block
// scales and token scales in one operation; the FP4 quantizer runs without
// approximate math.  Section "Las Curvas de Recompensa...": running the
// per-token scale as a separate framework op is what slowed NVFP4 training.
// "NVIDIA presenta una metodologia de preentrenamiento de 4 bits utilizando
// NVFP4", section "Que es realmente NVFP4": E4M3 block scales under an FP32
// scale that keeps them in range; section "La metodologia...": 1x16 blocks,
// round-to-nearest-even.
//
// Arithmetic (all FP32, one IEEE round-to-nearest step each):
//   S_enc = min(2688 / A, FLT_MAX), S_dec = A / 2688      (A = scope amax)
//   sb    = RNE_E4M3_sat((amax_b / 6) * S_enc)
//   r     = sb ? min(S_enc / sb, FLT_MAX) : 0,   code = RNE_E2M1_sat(x * r)
//
// Design: one warp per scale row, 8 elements (16 bytes) per lane per step so
// loads and stores are fully coalesced; a 16-element block is a lane pair, a
// 4-block scale group (one aligned 32-bit word of the tensor-core tile) is 8
// lanes.  Per-token scope reads the row twice (amax, then encode); the second
// read is served from L1/L2, so HBM sees one read.  Rows of the padded scale
// tile that hold no token are written as zero by the same warps.
#include <float.h>

#include "device.cuh"
#include "groups.cuh"
#include "kernels.h"

namespace mx8q {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ void nvfp4_scales(float amax, float& senc, float& sdec) {
  float e = __fdiv_rn(2688.0f, amax);          // 2688 = 6 (E2M1 max) * 448 (E4M3 max)
  if (!(e <= FLT_MAX)) e = FLT_MAX;
  senc = e;
  sdec = __fdiv_rn(amax, 2688.0f);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

__device__ __forceinline__ float row_amax(const uint16_t* __restrict__ xr, int64_t C, int lane) {
  float a = 0.f;
  for (int64_t c = lane * 8; c < C; c += 256) {
    const uint4 w = *reinterpret_cast<const uint4*>(xr + c);
    a = fmaxf(a, fmaxf(fmaxf(fabsf(bf16_lo(w.x)), fabsf(bf16_hi(w.x))),
                       fmaxf(fabsf(bf16_lo(w.y)), fabsf(bf16_hi(w.y)))));
    a = fmaxf(a, fmaxf(fmaxf(fabsf(bf16_lo(w.z)), fabsf(bf16_hi(w.z))),
                       fmaxf(fabsf(bf16_lo(w.w)), fabsf(bf16_hi(w.w)))));
  }
  return warp_max(a);
}

// Scale-tile byte offset of the 4-scale word (row sr, scale columns k4*4..+3).
__device__ __forceinline__ int64_t sf_word(int64_t sr, int64_t k4, int64_t kt) {
  return ((sr >> 7) * kt + k4) * 512 + (sr & 31) * 16 + ((sr >> 5) & 3) * 4;
}

// scope: 0 token, 1 group, 2 tensor.  grouped: scale layout padded per group.
template <int kScope, bool kGrouped>
__global__ void __launch_bounds__(kThreads) nvfp4_quant_kernel(
    const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ld,
    const int64_t* __restrict__ offs, int G, int64_t tp_bound, uint8_t* __restrict__ q,
    uint8_t* __restrict__ sblk, float* __restrict__ s32, const float* __restrict__ amax_ws) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GroupSmem& gs = *reinterpret_cast<GroupSmem*>(smem_raw);
  int64_t TP;
  if (kGrouped) {
    load_group_prefix(gs, offs, G);
    TP = gs.pref[G];
  } else {
    TP = (R + 127) / 128 * 128;
  }
  (void)tp_bound;
  if (kScope != 0 && blockIdx.x == 0) {
    const int ng = (kScope == 1) ? G : 1;
    for (int g = threadIdx.x; g < ng; g += blockDim.x) s32[g] = __fdiv_rn(amax_ws[g], 2688.0f);
  }

  const int lane = threadIdx.x & 31;
  const int64_t kt = (C / 16 + 3) / 4;           // scale-tile columns (4 scales each)
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;

  for (int64_t sr = warp0; sr < TP; sr += nwarps) {
    int64_t row;
    int g = 0;
    if (kGrouped) {
      g = upper_group(gs.pref, G, sr);
      const int64_t local = sr - gs.pref[g];
      row = (local < gs.offs[g + 1] - gs.offs[g]) ? gs.offs[g] + local : -1;
    } else {
      row = sr < R ? sr : -1;
    }
    if (row < 0) {  // padding row of the scale tile
      for (int64_t k4 = lane; k4 < kt; k4 += 32)
        *reinterpret_cast<uint32_t*>(sblk + sf_word(sr, k4, kt)) = 0u;
      continue;
    }
    const uint16_t* xr = x + row * ld;
    float amax;
    if (kScope == 0) amax = row_amax(xr, C, lane);
    else amax = amax_ws[kScope == 1 ? g : 0];
    float senc, sdec;
    nvfp4_scales(amax, senc, sdec);
    if (kScope == 0 && lane == 0) s32[row] = sdec;

    uint8_t* qr = q + row * (C / 2);
    for (int64_t base = 0; base < C; base += 256) {
      const int64_t c = base + lane * 8;
      const bool valid = c < C;
      uint4 w = make_uint4(0, 0, 0, 0);
      if (valid) w = *reinterpret_cast<const uint4*>(xr + c);
      float v[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                    bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
      float bmax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
      bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 1));   // lane pair = block
      const float t = __fmul_rn(__fdiv_rn(bmax, 6.0f), senc);
      const uint32_t sb = cvt_e4m3x2(t, 0.0f) & 0xFFu;
      float r = 0.f;
      if (sb != 0) r = fminf(__fdiv_rn(senc, e4m3_to_f32(sb)), FLT_MAX);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], r);
      const uint32_t packed = cvt_e2m1x8(v);
      if (valid) *reinterpret_cast<uint32_t*>(qr + c / 2) = packed;

      // gather the 4 block scales of this lane's 8-lane group
      const int l0 = lane & ~7;
      const uint32_t s0 = __shfl_sync(0xffffffffu, sb, l0);
      const uint32_t s1 = __shfl_sync(0xffffffffu, sb, l0 + 2);
      const uint32_t s2 = __shfl_sync(0xffffffffu, sb, l0 + 4);
      const uint32_t s3 = __shfl_sync(0xffffffffu, sb, l0 + 6);
      const int64_t k4 = (base >> 6) + (lane >> 3);
      if ((lane & 7) == 0 && k4 < kt)
        *reinterpret_cast<uint32_t*>(sblk + sf_word(sr, k4, kt)) = s0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
    }
  }
}

// Per-row amax folded into the scope amax (group or tensor) with atomicMax on
// the bit pattern (non-negative floats order like their bits).
template <bool kGroupScope>
__global__ void __launch_bounds__(kThreads) nvfp4_amax_kernel(
    const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ld,
    const int64_t* __restrict__ offs, int G, float* __restrict__ amax_ws) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t row = warp0; row < R; row += nwarps) {
    const float a = row_amax(x + row * ld, C, lane);
    if (lane == 0) {
      int g = 0;
      if (kGroupScope) {
        g = upper_group(offs, G, row);        // group with offs[g] <= row < offs[g+1]
      }
      atomicMax(reinterpret_cast<unsigned int*>(amax_ws + g), __float_as_uint(a));
    }
  }
}

}  // namespace

cudaError_t launch_nvfp4_quant(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int scope,
                               const int64_t* offs, int G, uint8_t* q, uint8_t* sblk, float* s32,
                               float* amax_ws, int sm_count, cudaStream_t stream) {
  const bool grouped = offs != nullptr;
  if (scope != 0) {
    cudaError_t e = cudaMemsetAsync(amax_ws, 0, sizeof(float) * (scope == 1 ? G : 1), stream);
    if (e != cudaSuccess) return e;
    if (R > 0) {
      const int64_t want = (R + kWarps - 1) / kWarps;
      const int64_t cap = static_cast<int64_t>(sm_count) * 8;
      const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
      if (scope == 1) nvfp4_amax_kernel<true><<<grid, kThreads, 0, stream>>>(x, R, C, ld, offs, G, amax_ws);
      else nvfp4_amax_kernel<false><<<grid, kThreads, 0, stream>>>(x, R, C, ld, offs, G, amax_ws);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  const int64_t tp_bound = grouped ? (R + 127 * static_cast<int64_t>(G) + 127) / 128 * 128
                                   : (R + 127) / 128 * 128;
  const int64_t want = (tp_bound + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (grid == 0) grid = 1;
  const size_t smem = grouped ? sizeof(GroupSmem) : 0;
#define MX8Q_NV_LAUNCH(S, GRP)                                                                 \
  do {                                                                                          \
    auto k = nvfp4_quant_kernel<S, GRP>;                                                       \
    if (smem > 0) {                                                                             \
      cudaError_t ea = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                                            static_cast<int>(smem));                          \
      if (ea != cudaSuccess) return ea;                                                         \
    }                                                                                           \
    k<<<grid, kThreads, smem, stream>>>(x, R, C, ld, offs, G, tp_bound, q, sblk, s32, amax_ws); \
  } while (0)
  if (grouped) {
    if (scope == 0) MX8Q_NV_LAUNCH(0, true);
    else if (scope == 1) MX8Q_NV_LAUNCH(1, true);
    else MX8Q_NV_LAUNCH(2, true);
  } else {
    if (scope == 0) MX8Q_NV_LAUNCH(0, false);
    else MX8Q_NV_LAUNCH(2, false);
  }
#undef MX8Q_NV_LAUNCH
  return cudaGetLastError();
}

}  // namespace mx8q
