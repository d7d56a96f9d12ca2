// Columnwise NVFP4 of a Wgrad input with the 16x16 random Hadamard transform
// ("NVIDIA presenta una metodologia de preentrenamiento de 4 bits utilizando
// NVFP4", section "La metodologia de formacion de cuatro partes"): the
// inputs of the weight-gradient GEMM are multiplied, in 16-element tiles
// along the reduction dimension, by a 16x16 Hadamard matrix combined with one
// random +-1 sign vector shared by all linear layers, which spreads outliers
// and cancels inside the Wgrad product (the transform is orthogonal).
//   y = (1/4) H16 diag(s) x  per 16 rows of a column, in binary32 as the
//       natural-order fast Walsh-Hadamard butterfly (v_i = s_i x_i; for
//       h = 1, 2, 4, 8: (v_i, v_i+h) <- (v_i + v_i+h, v_i - v_i+h); y = v / 4)
//   then NVFP4 of y with one FP32 scale from the amax of y (two launches:
//   amax pass, encode pass) and per 16-block E4M3 scales; the output is the
//   transposed copy qT [C, R/2] that the Wgrad GEMM reads with K = R.
// A block of 256 threads stages a 128 x 128 bf16 tile; thread t transforms
// column t % 128 for chunks t / 128, +2, +4, +6 (conflict-free column reads),
// and in the encode pass stages its codes and scales so that the transposed
// rows and the 512-byte scale tiles leave with 16-byte stores.
//
// Gradients (same section: round-to-nearest-even biases gradients; stochastic
// rounding, gradients only) take stochastically rounded codes: the block
// scales stay round-to-nearest, and element e of the output (its index in the
// quantized matrix) rounds with the 32 bits of Philox4x64-10 block e / 8 under
// the caller's seed.  nvfp4_sr_token_kernel is the per-token quantizer of a
// gradient (the Dgrad operand) with stochastic codes: one warp per row, the
// row read once for its amax and once more (from L2) for the encode.
#include "device.cuh"
#include "kernels.h"

namespace mx8q {

namespace {

constexpr int kTile = 128;
constexpr int kWThreads = 256;

__device__ __forceinline__ void rht16(float (&v)[16], uint32_t mask) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if ((mask >> i) & 1u) v[i] = -v[i];
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], 0.25f);
}

__device__ __forceinline__ int tile_byte(int row, int k) {
  return (row & 31) * 16 + ((row >> 5) & 3) * 4 + (k & 3);
}

// kEncode = false: atomicMax of max |y| into amax_bits; true: encode (kSR:
// stochastically rounded codes).
template <bool kEncode, bool kSR>
__global__ void __launch_bounds__(kWThreads) rht_colwise_kernel(
    const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ld, uint32_t mask, uint64_t seed,
    uint32_t* __restrict__ amax_bits, uint8_t* __restrict__ qT, uint8_t* __restrict__ sT,
    float* __restrict__ s32) {
  __shared__ __align__(16) uint16_t tile[kTile][kTile];   // 32 KB of bf16 (rows = reduction dim)
  __shared__ __align__(16) uint8_t codes[kTile][64];      // transposed codes: 128 columns x 128 rows / 2
  __shared__ __align__(16) uint8_t stile[2][512];         // transposed scale tiles
  __shared__ float red[kWThreads / 32];
  const int t = threadIdx.x;
  float senc = 0.f;
  if (kEncode) {
    float sdec;
    nvfp4_scales(__uint_as_float(*amax_bits), senc, sdec);
    if (blockIdx.x == 0 && t == 0) s32[0] = sdec;
  }
  const int64_t tiles_c = (C + kTile - 1) / kTile, tiles_r = (R + kTile - 1) / kTile;
  const int64_t kt = (R / 16 + 3) / 4;                    // scale tiles per 128 transposed rows
  float tmax = 0.f;
  for (int64_t tl = blockIdx.x; tl < tiles_r * tiles_c; tl += gridDim.x) {
    const int64_t r0 = (tl / tiles_c) * kTile, c0 = (tl % tiles_c) * kTile;
    __syncthreads();                                      // the previous tile is no longer read
    // stage the tile: 128 rows x 16 chunks of 16 bytes, zeros outside
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int idx = t + j * kWThreads;
      const int rr = idx >> 4, ch = idx & 15;
      const int64_t gr = r0 + rr, gc = c0 + ch * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (gr < R && gc < C) v = __ldg(reinterpret_cast<const uint4*>(x + gr * ld + gc));
      *reinterpret_cast<uint4*>(&tile[rr][ch * 8]) = v;
    }
    __syncthreads();
    const int c = t & 127;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = (t >> 7) + 2 * j;                     // 16-row chunk of the tile
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(static_cast<uint32_t>(tile[16 * k + i][c]) << 16);
      rht16(v, mask);
      float bmax = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
      if (!kEncode) {
        tmax = fmaxf(tmax, bmax);
        continue;
      }
      const uint32_t sb = cvt_e4m3x2(__fmul_rn(__fdiv_rn(bmax, 6.0f), senc), 0.0f) & 0xFFu;
      const float r = sb ? fminf(__fdiv_rn(senc, e4m3_to_f32(sb)), FLT_MAX) : 0.f;
      float a[8], b[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        a[i] = __fmul_rn(v[i], r);
        b[i] = __fmul_rn(v[8 + i], r);
      }
      uint2 packed;
      if (kSR) {
        // element index in the transposed copy: row c0 + c, column r0 + 16 k
        const uint64_t e0 = static_cast<uint64_t>(c0 + c) * static_cast<uint64_t>(R) + static_cast<uint64_t>(r0 + 16 * k);
        uint32_t ba[8], bb[8];
        sr_bits8(seed, e0, ba);
        sr_bits8(seed, e0 + 8, bb);
        packed = make_uint2(e2m1x8_sr(a, ba), e2m1x8_sr(b, bb));
      } else {
        packed = make_uint2(cvt_e2m1x8(a), cvt_e2m1x8(b));
      }
      *reinterpret_cast<uint2*>(&codes[c][8 * k]) = packed;
      stile[k >> 2][tile_byte(c, k)] = static_cast<uint8_t>(sb);
    }
    if (!kEncode) continue;
    __syncthreads();
    // transposed rows c0 + c: 64 code bytes each (4 x 16 bytes)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int idx = t + j * kWThreads;
      const int rc = idx >> 2, part = idx & 3;
      const int64_t gc = c0 + rc, gb = r0 / 2 + part * 16;
      if (gc < C && gb < R / 2)
        *reinterpret_cast<uint4*>(qT + gc * (R / 2) + gb) = *reinterpret_cast<const uint4*>(&codes[rc][part * 16]);
    }
    if (t < 64) {
      const int j = t >> 5;
      const int64_t kg = r0 / 64 + j;
      if (kg < kt)
        reinterpret_cast<uint4*>(sT + ((c0 / kTile) * kt + kg) * 512)[t & 31] =
            reinterpret_cast<const uint4*>(stile[j])[t & 31];
    }
  }
  if (!kEncode) {
    tmax = warp_max(tmax);
    if ((t & 31) == 0) red[t >> 5] = tmax;
    __syncthreads();
    if (t == 0) {
      for (int i = 1; i < kWThreads / 32; ++i) tmax = fmaxf(tmax, red[i]);
      atomicMax(amax_bits, __float_as_uint(tmax));
    }
  }
}

// Per-token NVFP4 of a gradient with stochastically rounded codes (block
// scales and S_dec as the round-to-nearest quantizer); scale rows past R
// (padding of the last 128-row tile) are written as zero.
__global__ void __launch_bounds__(kWThreads) nvfp4_sr_token_kernel(
    const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ld, uint64_t seed, uint8_t* __restrict__ q,
    uint8_t* __restrict__ sblk, float* __restrict__ s32) {
  const int lane = threadIdx.x & 31;
  const int64_t kt = (C / 16 + 3) / 4;
  const int64_t RP = (R + 127) / 128 * 128;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * (kWThreads / 32);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (kWThreads / 32) + (threadIdx.x >> 5); row < RP; row += nw) {
    uint8_t* srow = sblk + (row >> 7) * kt * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
    if (row >= R) {                                        // padding scale row
      for (int64_t b = lane; b < kt * 4; b += 32) srow[(b >> 2) * 512 + (b & 3)] = 0;
      continue;
    }
    const uint16_t* xr = x + row * ld;
    uint32_t m = 0;
    for (int64_t c = 8 * lane; c < C; c += 256) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(xr + c));
      m = amax2(m, amax2(amax2(w.x, w.y), amax2(w.z, w.w)));
    }
    float senc, sdec;
    nvfp4_scales(warp_max(abs_halves_max(m)), senc, sdec);
    if (lane == 0) s32[row] = sdec;
    for (int64_t b = lane; b < C / 16; b += 32) {          // 16-element block b of the row
      const uint4 w0 = __ldg(reinterpret_cast<const uint4*>(xr + 16 * b));
      const uint4 w1 = __ldg(reinterpret_cast<const uint4*>(xr + 16 * b + 8));
      const float bmax = abs_halves_max(absmax16(w0, w1));
      const uint32_t sb = cvt_e4m3x2(__fmul_rn(__fdiv_rn(bmax, 6.0f), senc), 0.0f) & 0xFFu;
      const float r = sb ? fminf(__fdiv_rn(senc, e4m3_to_f32(sb)), FLT_MAX) : 0.f;
      const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      float a[8], bv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[2 * i] = __fmul_rn(bf16_lo(ws[i]), r);
        a[2 * i + 1] = __fmul_rn(bf16_hi(ws[i]), r);
        bv[2 * i] = __fmul_rn(bf16_lo(ws[4 + i]), r);
        bv[2 * i + 1] = __fmul_rn(bf16_hi(ws[4 + i]), r);
      }
      const uint64_t e0 = static_cast<uint64_t>(row) * static_cast<uint64_t>(C) + static_cast<uint64_t>(16 * b);
      uint32_t ba[8], bb[8];
      sr_bits8(seed, e0, ba);
      sr_bits8(seed, e0 + 8, bb);
      *reinterpret_cast<uint2*>(q + row * (C / 2) + 8 * b) = make_uint2(e2m1x8_sr(a, ba), e2m1x8_sr(bv, bb));
      srow[(b >> 2) * 512 + (b & 3)] = static_cast<uint8_t>(sb);
    }
    // padding scale columns of the row's last 4-block group are zero
    for (int64_t b = C / 16 + lane; b < kt * 4; b += 32) srow[(b >> 2) * 512 + (b & 3)] = 0;
  }
}

}  // namespace

cudaError_t launch_nvfp4_sr_token(const uint16_t* x, int64_t R, int64_t C, int64_t ld, uint64_t seed, uint8_t* q,
                                  uint8_t* sblk, float* s32, int sm_count, cudaStream_t stream) {
  const int64_t rows = (R + 127) / 128 * 128;
  const int64_t want = (rows + kWThreads / 32 - 1) / (kWThreads / 32);
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  nvfp4_sr_token_kernel<<<static_cast<unsigned>(want < cap ? want : cap), kWThreads, 0, stream>>>(x, R, C, ld, seed,
                                                                                                 q, sblk, s32);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_rht_colwise(const uint16_t* x, int64_t R, int64_t C, int64_t ld, uint32_t mask, bool sr,
                                     uint64_t seed, uint8_t* qT, uint8_t* sT, float* s32, uint32_t* amax_bits,
                                     int sm_count, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  const int64_t tiles = ((R + kTile - 1) / kTile) * ((C + kTile - 1) / kTile);
  const int64_t cap = static_cast<int64_t>(sm_count) * 4;
  const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
  rht_colwise_kernel<false, false><<<grid, kWThreads, 0, stream>>>(x, R, C, ld, mask, seed, amax_bits, qT, sT, s32);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (sr)
    rht_colwise_kernel<true, true><<<grid, kWThreads, 0, stream>>>(x, R, C, ld, mask, seed, amax_bits, qT, sT, s32);
  else
    rht_colwise_kernel<true, false><<<grid, kWThreads, 0, stream>>>(x, R, C, ld, mask, seed, amax_bits, qT, sT, s32);
  return cudaGetLastError();
}

}  // namespace mx8q
