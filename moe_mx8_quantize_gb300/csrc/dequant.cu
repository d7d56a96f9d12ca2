// Dequantization of MXFP8 / NVFP4 / MXFP4 matrices back to f32 or bf16: the
// "dequantized backward" mode of "Miles Blackwell RL Cambia la Uniformidad
// BF16 por MXFP8 y NVFP4 Nativos" (section "La Compatibilidad...") rebuilds
// high-precision operands from the exact low-precision values of the forward
// pass.
//   MXFP8: out = e4m3 * 2^(s - 127)          (exact in f32 unless it overflows)
//   NVFP4: out = RN((e2m1 * sb) * S_dec)     (the inner product is exact)
//   MXFP4: out = e2m1 * 2^(s - 127)          (exact in f32 unless it overflows)
// bf16 output is the round-to-nearest-even of the f32 value.
//
// Elementwise and bandwidth-bound: each thread turns 16 elements (one NVFP4
// block or half an MXFP8 / MXFP4 block) into 64 bytes of f32 or 32 bytes of bf16 with
// 16-byte stores; the block scale is read from the tensor-core tile layout.
#include <cuda_bf16.h>

#include "device.cuh"
#include "groups.cuh"
#include "kernels.h"

namespace mx8q {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float e8m0_to_f32(uint32_t c) {
  if (c == 255u) return __uint_as_float(0x7FC00000u);
  if (c == 0u) return __uint_as_float(0x00400000u);   // 2^-127
  return __uint_as_float(c << 23);
}

// E2M1 nibble: exponent field e (2 bits), mantissa m (1 bit), sign bit 3.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const uint32_t mag = (e == 0u) ? (m ? 0x3F000000u : 0u) : (((e + 126u) << 23) | (m << 22));
  return __uint_as_float(mag | ((c & 8u) << 28));
}

__device__ __forceinline__ void e4m3x2_to_f32(uint32_t two, float& lo, float& hi) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(two & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  __half_raw a, b;
  a.x = static_cast<unsigned short>(h2 & 0xFFFFu);
  b.x = static_cast<unsigned short>(h2 >> 16);
  lo = __half2float(__half(a));
  hi = __half2float(__half(b));
}

__device__ __forceinline__ int64_t sf_byte(int64_t sr, int64_t k, int64_t kt) {
  return ((sr >> 7) * kt + (k >> 2)) * 512 + (sr & 31) * 16 + ((sr >> 5) & 3) * 4 + (k & 3);
}

template <int kFmt, bool kGrouped>
__global__ void __launch_bounds__(kThreads) dequant_kernel(
    const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, const float* __restrict__ s32,
    int s32_mode, const int64_t* __restrict__ offs, int G, int64_t R, int64_t C, int out_bf16,
    void* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GroupSmem& gs = *reinterpret_cast<GroupSmem*>(smem_raw);
  if (kGrouped || s32_mode == MX8Q_S32_GROUP_MODE) load_group_prefix(gs, offs, G);

  const int64_t bs = (kFmt == 1) ? 16 : 32;
  const int64_t kt = (C / bs + 3) / 4;
  const int64_t chunks = C / 16;
  const int64_t total = R * chunks;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t r = i / chunks, c = (i % chunks) * 16;
    int64_t sr = r;
    int g = 0;
    if (kGrouped || s32_mode == MX8Q_S32_GROUP_MODE) {
      g = upper_group(gs.offs, G, r);
      if (kGrouped) sr = gs.pref[g] + (r - gs.offs[g]);
    }
    const float sc = (kFmt == 1) ? e4m3_to_f32(s[sf_byte(sr, c / 16, kt)])
                                 : e8m0_to_f32(s[sf_byte(sr, c / 32, kt)]);
    float v[16];
    if (kFmt == 0) {
      const uint4 w = *reinterpret_cast<const uint4*>(q + r * C + c);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        e4m3x2_to_f32(ws[j] & 0xFFFFu, v[4 * j], v[4 * j + 1]);
        e4m3x2_to_f32(ws[j] >> 16, v[4 * j + 2], v[4 * j + 3]);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], sc);
    } else if (kFmt == 2) {
      const uint2 w = *reinterpret_cast<const uint2*>(q + r * (C / 2) + c / 2);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t byte = ((j < 4 ? w.x : w.y) >> (8 * (j & 3))) & 0xFFu;
        v[2 * j] = __fmul_rn(e2m1_to_f32(byte & 15u), sc);
        v[2 * j + 1] = __fmul_rn(e2m1_to_f32(byte >> 4), sc);
      }
    } else {
      const uint2 w = *reinterpret_cast<const uint2*>(q + r * (C / 2) + c / 2);
      float sd = 1.f;
      if (s32_mode == 1) sd = s32[r];
      else if (s32_mode == 2) sd = s32[0];
      else if (s32_mode == 3) sd = s32[g];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t byte = ((j < 4 ? w.x : w.y) >> (8 * (j & 3))) & 0xFFu;
        v[2 * j] = __fmul_rn(__fmul_rn(e2m1_to_f32(byte & 15u), sc), sd);
        v[2 * j + 1] = __fmul_rn(__fmul_rn(e2m1_to_f32(byte >> 4), sc), sd);
      }
    }
    if (out_bf16) {
      uint32_t p[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const __nv_bfloat16 a = __float2bfloat16_rn(v[2 * j]);
        const __nv_bfloat16 b = __float2bfloat16_rn(v[2 * j + 1]);
        p[j] = static_cast<uint32_t>(__bfloat16_as_ushort(a)) |
               (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + r * C + c);
      dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
      dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
    } else {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + r * C + c);
#pragma unroll
      for (int j = 0; j < 4; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
  }
}

}  // namespace

cudaError_t launch_dequant(int fmt, const uint8_t* q, const uint8_t* s, const float* s32,
                           int s32_mode, const int64_t* offs, int G, int64_t R, int64_t C,
                           int out_bf16, void* out, int sm_count, cudaStream_t stream) {
  const int64_t total = R * (C / 16);
  if (total == 0) return cudaSuccess;
  const bool grouped = offs != nullptr;
  const bool need_groups = grouped || s32_mode == MX8Q_S32_GROUP_MODE;
  const size_t smem = need_groups ? sizeof(GroupSmem) : 0;
  const int64_t want = (total + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
#define MX8Q_DQ_LAUNCH(F, GRP)                                                                  \
  do {                                                                                           \
    auto k = dequant_kernel<F, GRP>;                                                            \
    if (smem > 0) {                                                                              \
      cudaError_t ea = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,     \
                                            static_cast<int>(smem));                           \
      if (ea != cudaSuccess) return ea;                                                          \
    }                                                                                            \
    k<<<grid, kThreads, smem, stream>>>(q, s, s32, s32_mode, offs, G, R, C, out_bf16, out);     \
  } while (0)
  if (fmt == 0) {
    if (grouped) MX8Q_DQ_LAUNCH(0, true); else MX8Q_DQ_LAUNCH(0, false);
  } else if (fmt == 2) {
    if (grouped) MX8Q_DQ_LAUNCH(2, true); else MX8Q_DQ_LAUNCH(2, false);
  } else {
    if (grouped) MX8Q_DQ_LAUNCH(1, true); else MX8Q_DQ_LAUNCH(1, false);
  }
#undef MX8Q_DQ_LAUNCH
  return cudaGetLastError();
}

// SwiGLU between the gate|up and down GEMMs of a MoE expert: gate and up are
// the two halves of one fused GEMM output ("Un Cuantizador Compartido Es el
// Mecanismo Real": SwiGLU experts compute gate and up in one fused GEMM).
//   h[r, j] = RN_bf16( silu(g) * u ),  silu(g) = g / (1 + exp(-g)),
//   g = gu[r, j], u = gu[r, F + j]; f32 arithmetic (silu_mul: e^-|g| from
//   ex2.approx with a split argument, the reciprocal refined by Newton),
//   evaluated as g*e^-|g|/(1+e^-|g|) for negative g so nothing overflows.
namespace {
__global__ void __launch_bounds__(kThreads) swiglu_kernel(const uint16_t* __restrict__ gu, int64_t R,
                                                          int64_t F, int64_t ld_gu,
                                                          uint16_t* __restrict__ h, int64_t ld_h) {
  const int64_t chunks = F / 8;
  const int64_t total = R * chunks;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t r = i / chunks, c = (i % chunks) * 8;
    const uint4 g = *reinterpret_cast<const uint4*>(gu + r * ld_gu + c);
    const uint4 u = *reinterpret_cast<const uint4*>(gu + r * ld_gu + F + c);
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float v[2];
      const float gv[2] = {bf16_lo(gw[j]), bf16_hi(gw[j])};
      const float uv[2] = {bf16_lo(uw[j]), bf16_hi(uw[j])};
#pragma unroll
      for (int k = 0; k < 2; ++k) v[k] = silu_mul(gv[k], uv[k]);
      o[j] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[0]))) |
             (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[1]))) << 16);
    }
    *reinterpret_cast<uint4*>(h + r * ld_h + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}
}  // namespace

// MoE combine: out[t] = sum_j w[t][j] * y[rows[t][j]] in binary32, j in
// order (acc = RN(acc + RN(w * y))), so the result is deterministic and
// equal to a serial evaluation; each thread owns 8 columns of one token and
// reads the k rows' 16-byte pieces (coalesced along the row).
namespace {
template <bool kBf16Out>
__global__ void __launch_bounds__(kThreads) combine_kernel(const uint16_t* __restrict__ y, int64_t ldy, int64_t R,
                                                          const int64_t* __restrict__ rows,
                                                          const float* __restrict__ w, int64_t T, int64_t H, int k,
                                                          void* __restrict__ out, int64_t ldo) {
  const int64_t chunks = H / 8;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < T * chunks;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t t = i / chunks, c = (i % chunks) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < k; j0 += 8) {
      // the (up to) 8 rows' loads are issued together, then summed in order
      uint4 v[8];
      float wj[8];
      bool ok[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int j = j0 + jj;
        const int64_t r = j < k ? rows[t * k + j] : -1;
        ok[jj] = r >= 0 && r < R;
        wj[jj] = ok[jj] ? w[t * k + j] : 0.f;
        v[jj] = ok[jj] ? __ldg(reinterpret_cast<const uint4*>(y + r * ldy + c)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        if (!ok[jj]) continue;             // a missing row contributes nothing (not +0)
        const uint32_t ws[4] = {v[jj].x, v[jj].y, v[jj].z, v[jj].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[2 * e] = __fadd_rn(acc[2 * e], __fmul_rn(wj[jj], bf16_lo(ws[e])));
          acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], __fmul_rn(wj[jj], bf16_hi(ws[e])));
        }
      }
    }
    if (kBf16Out) {
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + t * ldo + c) =
          make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                     pack_bf16x2(acc[6], acc[7]));
    } else {
      float4* d = reinterpret_cast<float4*>(static_cast<float*>(out) + t * ldo + c);
      d[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      d[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
}
}  // namespace

cudaError_t launch_combine(const uint16_t* y, int64_t ldy, int64_t R, const int64_t* rows, const float* w, int64_t T,
                           int64_t H, int k, bool bf16_out, void* out, int64_t ldo, int sm_count, cudaStream_t stream) {
  const int64_t total = T * (H / 8);
  if (total == 0) return cudaSuccess;
  const int64_t want = (total + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (bf16_out)
    combine_kernel<true><<<grid, kThreads, 0, stream>>>(y, ldy, R, rows, w, T, H, k, out, ldo);
  else
    combine_kernel<false><<<grid, kThreads, 0, stream>>>(y, ldy, R, rows, w, T, H, k, out, ldo);
  return cudaGetLastError();
}

cudaError_t launch_swiglu(const uint16_t* gu, int64_t R, int64_t F, int64_t ld_gu, uint16_t* h,
                          int64_t ld_h, int sm_count, cudaStream_t stream) {
  const int64_t total = R * (F / 8);
  if (total == 0) return cudaSuccess;
  const int64_t want = (total + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  swiglu_kernel<<<static_cast<unsigned>(want < cap ? want : cap), kThreads, 0, stream>>>(gu, R, F, ld_gu,
                                                                                        h, ld_h);
  return cudaGetLastError();
}

}  // namespace mx8q
