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
// Design: one warp per scale row.  Lane l owns elements [256*i + 8*l, +8) of
// the row for every 256-element chunk i, so loads and stores are fully
// coalesced; a 16-element block is a lane pair and a 4-block scale group (one
// aligned 32-bit word of the tensor-core tile) is 8 lanes.  Rows of up to
// 256*kCh elements are loaded into registers with all loads issued up front
// (many bytes in flight per warp, one HBM read per element); longer rows are
// streamed twice (the second read comes from L1/L2).  Rows of the padded
// scale tile that hold no token are written as zero by the same warps.
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

__device__ __forceinline__ float amax8(const uint4& w) {
  return fmaxf(fmaxf(fmaxf(fabsf(bf16_lo(w.x)), fabsf(bf16_hi(w.x))),
                     fmaxf(fabsf(bf16_lo(w.y)), fabsf(bf16_hi(w.y)))),
               fmaxf(fmaxf(fabsf(bf16_lo(w.z)), fabsf(bf16_hi(w.z))),
                     fmaxf(fabsf(bf16_lo(w.w)), fabsf(bf16_hi(w.w)))));
}

__device__ __forceinline__ uint4 ld_nc(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// Streaming row amax, 8 chunks of 256 elements in flight per lane.
__device__ __forceinline__ float row_amax_stream(const uint16_t* __restrict__ xr, int64_t C, int lane) {
  float a = 0.f;
  for (int64_t base = 0; base < C; base += 256 * 8) {
    uint4 w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t c = base + i * 256 + lane * 8;
      w[i] = c < C ? ld_nc(xr + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, amax8(w[i]));
  }
  return warp_max(a);
}

// Scale-tile byte offset of the 4-scale word (row sr, scale columns k4*4..+3).
__device__ __forceinline__ int64_t sf_word(int64_t sr, int64_t k4, int64_t kt) {
  return ((sr >> 7) * kt + k4) * 512 + (sr & 31) * 16 + ((sr >> 5) & 3) * 4;
}

// Encodes one 256-element chunk (8 elements per lane) starting at column
// `base`: packed nibbles to qr, the chunk's 16 block scales to the tile.
__device__ __forceinline__ void encode_chunk(const uint4& w, int64_t base, int64_t C, int lane, float senc,
                                             uint8_t* __restrict__ qr, uint8_t* __restrict__ sblk,
                                             int64_t sr, int64_t kt) {
  const int64_t c = base + lane * 8;
  const bool valid = c < C;
  float v[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
  float bmax = amax8(w);
  bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 1));   // lane pair = one 16-block
  const float t = __fmul_rn(__fdiv_rn(bmax, 6.0f), senc);
  const uint32_t sb = cvt_e4m3x2(t, 0.0f) & 0xFFu;
  float r = 0.f;
  if (sb != 0) r = fminf(__fdiv_rn(senc, e4m3_to_f32(sb)), FLT_MAX);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], r);
  const uint32_t packed = cvt_e2m1x8(v);
  if (valid) *reinterpret_cast<uint32_t*>(qr + c / 2) = packed;
  const int l0 = lane & ~7;                    // gather the 8-lane group's 4 scales
  const uint32_t s0 = __shfl_sync(0xffffffffu, sb, l0);
  const uint32_t s1 = __shfl_sync(0xffffffffu, sb, l0 + 2);
  const uint32_t s2 = __shfl_sync(0xffffffffu, sb, l0 + 4);
  const uint32_t s3 = __shfl_sync(0xffffffffu, sb, l0 + 6);
  const int64_t k4 = (base >> 6) + (lane >> 3);
  if ((lane & 7) == 0 && k4 < kt)
    *reinterpret_cast<uint32_t*>(sblk + sf_word(sr, k4, kt)) = s0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
}

// scope: 0 token, 1 group, 2 tensor.  kCh: 256-element chunks held in
// registers (0 = stream the row twice).
template <int kCh>
__global__ void __launch_bounds__(kThreads) nvfp4_quant_kernel(
    const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ld, int scope,
    const int64_t* __restrict__ offs, int G, uint8_t* __restrict__ q, uint8_t* __restrict__ sblk,
    float* __restrict__ s32, const float* __restrict__ amax_ws) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GroupSmem& gs = *reinterpret_cast<GroupSmem*>(smem_raw);
  const bool grouped = offs != nullptr;
  int64_t TP;
  if (grouped) {
    load_group_prefix(gs, offs, G);
    TP = gs.pref[G];
  } else {
    TP = (R + 127) / 128 * 128;
  }
  if (scope != 0 && blockIdx.x == 0) {
    const int ng = (scope == 1) ? G : 1;
    for (int g = threadIdx.x; g < ng; g += blockDim.x) s32[g] = __fdiv_rn(amax_ws[g], 2688.0f);
  }

  const int lane = threadIdx.x & 31;
  const int64_t kt = (C / 16 + 3) / 4;           // scale-tile columns (4 scales each)
  const int nch = static_cast<int>((C + 255) / 256);
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;

  for (int64_t sr = warp0; sr < TP; sr += nwarps) {
    int64_t row;
    int g = 0;
    if (grouped) {
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
    uint8_t* qr = q + row * (C / 2);
    if (kCh > 0) {
      uint4 w[kCh > 0 ? kCh : 1];
#pragma unroll
      for (int i = 0; i < kCh; ++i) {
        const int64_t c = static_cast<int64_t>(i) * 256 + lane * 8;
        w[i] = (i < nch && c < C) ? ld_nc(xr + c) : make_uint4(0, 0, 0, 0);
      }
      float amax;
      if (scope == 0) {
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < kCh; ++i) a = fmaxf(a, amax8(w[i]));
        amax = warp_max(a);
      } else {
        amax = amax_ws[scope == 1 ? g : 0];
      }
      float senc, sdec;
      nvfp4_scales(amax, senc, sdec);
      if (scope == 0 && lane == 0) s32[row] = sdec;
#pragma unroll
      for (int i = 0; i < kCh; ++i)
        if (i < nch) encode_chunk(w[i], static_cast<int64_t>(i) * 256, C, lane, senc, qr, sblk, sr, kt);
    } else {
      const float amax = scope == 0 ? row_amax_stream(xr, C, lane) : amax_ws[scope == 1 ? g : 0];
      float senc, sdec;
      nvfp4_scales(amax, senc, sdec);
      if (scope == 0 && lane == 0) s32[row] = sdec;
      for (int64_t base = 0; base < C; base += 256) {
        const int64_t c = base + lane * 8;
        const uint4 w = c < C ? ld_nc(xr + c) : make_uint4(0, 0, 0, 0);
        encode_chunk(w, base, C, lane, senc, qr, sblk, sr, kt);
      }
    }
  }
}

// Scope amax (group or tensor): each warp owns a contiguous range of rows,
// keeps a running maximum while the group stays the same and folds it into
// the group's word with one atomicMax on the bit pattern (non-negative floats
// order like their bits) when the group changes or the range ends -- a few
// atomics per warp instead of one per row on a handful of addresses.
__global__ void __launch_bounds__(kThreads) nvfp4_amax_kernel(
    const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ld,
    const int64_t* __restrict__ offs, int G, bool group_scope, float* __restrict__ amax_ws) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  const int64_t per = (R + nwarps - 1) / nwarps;
  const int64_t r0 = warp0 * per;
  const int64_t r1 = r0 + per < R ? r0 + per : R;
  if (r0 >= r1) return;
  int g = group_scope ? upper_group(offs, G, r0) : 0;      // offs[g] <= r0 < offs[g+1]
  int64_t gend = group_scope ? offs[g + 1] : R;
  float run = 0.f;
  for (int64_t row = r0; row < r1; ++row) {
    if (row >= gend) {                                      // entering the next group
      if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(amax_ws + g), __float_as_uint(run));
      run = 0.f;
      g = upper_group(offs, G, row);
      gend = offs[g + 1];
    }
    run = fmaxf(run, row_amax_stream(x + row * ld, C, lane));
  }
  if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(amax_ws + g), __float_as_uint(run));
}

template <int kCh>
cudaError_t launch_quant(unsigned grid, size_t smem, cudaStream_t stream, const uint16_t* x, int64_t R,
                         int64_t C, int64_t ld, int scope, const int64_t* offs, int G, uint8_t* q,
                         uint8_t* sblk, float* s32, const float* amax_ws) {
  auto k = nvfp4_quant_kernel<kCh>;
  if (smem > 0) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  k<<<grid, kThreads, smem, stream>>>(x, R, C, ld, scope, offs, G, q, sblk, s32, amax_ws);
  return cudaGetLastError();
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
      nvfp4_amax_kernel<<<grid, kThreads, 0, stream>>>(x, R, C, ld, offs, G, scope == 1, amax_ws);
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
  if (C <= 1024) return launch_quant<4>(grid, smem, stream, x, R, C, ld, scope, offs, G, q, sblk, s32, amax_ws);
  if (C <= 2048) return launch_quant<8>(grid, smem, stream, x, R, C, ld, scope, offs, G, q, sblk, s32, amax_ws);
  if (C <= 4096) return launch_quant<16>(grid, smem, stream, x, R, C, ld, scope, offs, G, q, sblk, s32, amax_ws);
  if (C <= 8192) return launch_quant<32>(grid, smem, stream, x, R, C, ld, scope, offs, G, q, sblk, s32, amax_ws);
  return launch_quant<0>(grid, smem, stream, x, R, C, ld, scope, offs, G, q, sblk, s32, amax_ws);
}

}  // namespace mx8q
