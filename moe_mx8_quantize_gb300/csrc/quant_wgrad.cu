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
// quantized matrix) rounds with word e % 4 of Philox4x32-10 block e / 4 under
// the caller's seed.  nvfp4_sr_token_kernel is the per-token quantizer of a
// gradient (the Dgrad operand) with stochastic codes: a team of up to 256
// threads per row, which holds rows of up to 16384 values in registers (one
// HBM read) and reduces the row's amax over the team.
#include "device.cuh"
#include "kernels.h"

namespace mx8q {

namespace {

constexpr int kTile = 128;
constexpr int kWThreads = 256;

// ---------------------------------------------------------------- stochastic rounding
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011) on four counters at once: ten rounds of two
// 32x32->64-bit products with the round constants M0, M1, and the Weyl key
// increments W0, W1 between rounds; the four blocks share the key schedule
// and give the scheduler four independent chains.
__device__ __forceinline__ void philox4x32_10_x4(uint32_t (&c)[4][4], uint32_t k0, uint32_t k1) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += W0;
      k1 += W1;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint64_t p0 = static_cast<uint64_t>(M0) * c[j][0];
      const uint64_t p1 = static_cast<uint64_t>(M1) * c[j][2];
      const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c[j][1] ^ k0;
      const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c[j][3] ^ k1;
      c[j][0] = n0;
      c[j][1] = static_cast<uint32_t>(p1);
      c[j][2] = n2;
      c[j][3] = static_cast<uint32_t>(p0);
    }
  }
}

// The 32 random bits of elements e0 .. e0 + 15 (e0 % 4 == 0) under seed:
// element e takes word e % 4 of the block with counter (e / 4 split into two
// 32-bit words, 0, 0) and key (seed split into two 32-bit words).
__device__ __forceinline__ void sr_bits16(uint64_t seed, uint64_t e0, uint32_t (&bits)[16]) {
  uint32_t c[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t n = (e0 >> 2) + static_cast<uint64_t>(j);
    c[j][0] = static_cast<uint32_t>(n);
    c[j][1] = static_cast<uint32_t>(n >> 32);
    c[j][2] = 0;
    c[j][3] = 0;
  }
  philox4x32_10_x4(c, static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
#pragma unroll
  for (int i = 0; i < 16; ++i) bits[i] = c[i >> 2][i & 3];
}

// E2M1 code of v by stochastic rounding with 32 random bits b: |v| >= 6
// gives 6; otherwise |v| lies in [lo, hi) of the grid {0, .5, 1, 1.5, 2, 3,
// 4, 6} and rounds up to hi when (b >> 8) < p * 2^24, p = (|v| - lo) / (hi -
// lo); the sign is kept and NaN gives a zero code.  Read off the binary32
// fields of a = |v| (s = its exponent and top mantissa bit): for a >= 0.5
// the code of lo is max(s, 253) - 252 (from 1 for [0.5, 1) to 6 for [4, 6),
// 7 and up from 6 on, capped at 7), and p * 2^24 is 4 times the 22 mantissa
// bits below the top one (a >= 1) or 2 times the 23 mantissa bits ([0.5,
// 1)), so the test is b < (a << 10) or b < (a << 9) as 32-bit integers (the
// exponent bits shift out).  For a < 0.5, lo = 0 and p * 2^24 = a * 2^25,
// exact in binary32, compared with the 24 bits as a float.
__device__ __forceinline__ uint32_t e2m1_sr(float v, uint32_t bits) {
  const uint32_t ub = __float_as_uint(v);
  const uint32_t ab = ub & 0x7FFFFFFFu;
  const uint32_t t = ab >= 0x3F800000u ? ab << 10 : ab << 9;
  uint32_t code = min(max(ab >> 22, 253u) - 252u + (bits < t ? 1u : 0u), 7u);
  if (ab < 0x3F000000u) code = __uint2float_rn(bits >> 8) < __fmul_rn(__uint_as_float(ab), 33554432.0f) ? 1u : 0u;
  if (ab > 0x7F800000u) code = 0u;
  return code | ((ub >> 28) & 8u);
}

// Sixteen values -> sixteen stochastically rounded E2M1 nibbles (element 0
// in the low nibble of codes.x).
__device__ __forceinline__ uint2 e2m1x16_sr(const float (&v)[16], const uint32_t (&bits)[16]) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    lo |= e2m1_sr(v[i], bits[i]) << (4 * i);
    hi |= e2m1_sr(v[8 + i], bits[8 + i]) << (4 * i);
  }
  return make_uint2(lo, hi);
}

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
__global__ void __launch_bounds__(kWThreads, 4) rht_colwise_kernel(
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
      uint2 packed;
      if (kSR) {
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(v[i], r);
        // element index in the transposed copy: row c0 + c, column r0 + 16 k
        const uint64_t e0 = static_cast<uint64_t>(c0 + c) * static_cast<uint64_t>(R) + static_cast<uint64_t>(r0 + 16 * k);
        uint32_t bits[16];
        sr_bits16(seed, e0, bits);
        packed = e2m1x16_sr(y, bits);
      } else {
        float a[8], b[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          a[i] = __fmul_rn(v[i], r);
          b[i] = __fmul_rn(v[8 + i], r);
        }
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
// (padding of the last 128-row tile) are written as zero.  A team of kTeam
// threads (a power of two, 32 .. 256) quantizes one row: thread t of the team
// takes the row's 16-element blocks t, t + kTeam, ..., holds them in
// registers (kNB of them; kNB = 0 for longer rows, which are read twice, the
// second time from L2), and the team reduces the row's amax with shuffles
// and, across its warps, through shared memory (two buffers, one barrier a
// row).
template <int kTeam, int kNB>
__global__ void __launch_bounds__(kWThreads) nvfp4_sr_token_kernel(
    const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ld, uint64_t seed, uint8_t* __restrict__ q,
    uint8_t* __restrict__ sblk, float* __restrict__ s32) {
  constexpr int kRowsPerCta = kWThreads / kTeam;
  constexpr int kTeamWarps = kTeam / 32;
  __shared__ float2 tab[128];
  __shared__ float red[2][kWThreads / 32];
  nvfp4_init_scale_table(tab);
  __syncthreads();
  const int tt = threadIdx.x % kTeam;
  const int team = threadIdx.x / kTeam;
  const int64_t nb = C / 16;
  const int64_t kt = (nb + 3) / 4;
  const int64_t RP = (R + 127) / 128 * 128;
  const int64_t groups = (RP + kRowsPerCta - 1) / kRowsPerCta;
  int par = 0;
  for (int64_t g = blockIdx.x; g < groups; g += gridDim.x, par ^= 1) {
    const int64_t row = g * kRowsPerCta + team;
    const bool live = row < R;
    const uint16_t* xr = x + (live ? row : 0) * ld;
    uint4 w[kNB > 0 ? kNB : 1][2];
    uint32_t m = 0;
    if (live) {
      if constexpr (kNB > 0) {
#pragma unroll
        for (int j = 0; j < kNB; ++j) {
          const int64_t b = tt + static_cast<int64_t>(j) * kTeam;
          if (b < nb) {
            w[j][0] = __ldg(reinterpret_cast<const uint4*>(xr + 16 * b));
            w[j][1] = __ldg(reinterpret_cast<const uint4*>(xr + 16 * b + 8));
            m = amax2(m, absmax16(w[j][0], w[j][1]));
          }
        }
      } else {
        for (int64_t b = tt; b < nb; b += kTeam)
          m = amax2(m, absmax16(__ldg(reinterpret_cast<const uint4*>(xr + 16 * b)),
                                __ldg(reinterpret_cast<const uint4*>(xr + 16 * b + 8))));
      }
    }
    float amax = warp_max(abs_halves_max(m));
    if constexpr (kTeamWarps > 1) {
      if ((threadIdx.x & 31) == 0) red[par][threadIdx.x >> 5] = amax;
      __syncthreads();
#pragma unroll
      for (int i = 0; i < kTeamWarps; ++i) amax = fmaxf(amax, red[par][team * kTeamWarps + i]);
    }
    if (row >= RP) continue;
    uint8_t* srow = sblk + sf_row_base(row, kt);
    if (!live) {                                           // padding scale row
      for (int64_t b = tt; b < kt * 4; b += kTeam) srow[(b >> 2) * 512 + (b & 3)] = 0;
      continue;
    }
    float senc, sdec;
    nvfp4_scales(amax, senc, sdec);
    if (tt == 0) s32[row] = sdec;
    auto encode = [&](const uint4& w0, const uint4& w1, int64_t b) {
      float r;
      const uint32_t sb = nvfp4_block_scale(abs_halves_max(absmax16(w0, w1)), senc, tab, r);
      const uint64_t rr = f32x2_splat(r);
      const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) mul_bf16x2(ws[i], rr, v[2 * i], v[2 * i + 1]);
      uint32_t bits[16];
      sr_bits16(seed, static_cast<uint64_t>(row) * static_cast<uint64_t>(C) + static_cast<uint64_t>(16 * b), bits);
      *reinterpret_cast<uint2*>(q + row * (C / 2) + 8 * b) = e2m1x16_sr(v, bits);
      srow[(b >> 2) * 512 + (b & 3)] = static_cast<uint8_t>(sb);
    };
    if constexpr (kNB > 0) {
#pragma unroll
      for (int j = 0; j < kNB; ++j) {
        const int64_t b = tt + static_cast<int64_t>(j) * kTeam;
        if (b < nb) encode(w[j][0], w[j][1], b);
      }
    } else {
      for (int64_t b = tt; b < nb; b += kTeam)
        encode(__ldg(reinterpret_cast<const uint4*>(xr + 16 * b)), __ldg(reinterpret_cast<const uint4*>(xr + 16 * b + 8)),
               b);
    }
    // padding scale columns of the row's last 4-block group are zero
    for (int64_t b = nb + tt; b < kt * 4; b += kTeam) srow[(b >> 2) * 512 + (b & 3)] = 0;
  }
}

template <int kTeam, int kNB>
void launch_sr_token(const uint16_t* x, int64_t R, int64_t C, int64_t ld, uint64_t seed, uint8_t* q, uint8_t* sblk,
                     float* s32, int sm_count, cudaStream_t stream) {
  const int64_t groups = ((R + 127) / 128 * 128 + kWThreads / kTeam - 1) / (kWThreads / kTeam);
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  nvfp4_sr_token_kernel<kTeam, kNB><<<static_cast<unsigned>(groups < cap ? groups : cap), kWThreads, 0, stream>>>(
      x, R, C, ld, seed, q, sblk, s32);
}

}  // namespace

cudaError_t launch_nvfp4_sr_token(const uint16_t* x, int64_t R, int64_t C, int64_t ld, uint64_t seed, uint8_t* q,
                                  uint8_t* sblk, float* s32, int sm_count, cudaStream_t stream) {
  // the smallest team that covers the row's 16-element blocks once (32 ..
  // 256 threads); wider rows take 2 or 4 blocks a thread, past 16384 values
  // the two-read path
  const int64_t nb = C / 16;
  if (nb <= 32)
    launch_sr_token<32, 1>(x, R, C, ld, seed, q, sblk, s32, sm_count, stream);
  else if (nb <= 64)
    launch_sr_token<64, 1>(x, R, C, ld, seed, q, sblk, s32, sm_count, stream);
  else if (nb <= 128)
    launch_sr_token<128, 1>(x, R, C, ld, seed, q, sblk, s32, sm_count, stream);
  else if (nb <= 256)
    launch_sr_token<256, 1>(x, R, C, ld, seed, q, sblk, s32, sm_count, stream);
  else if (nb <= 512)
    launch_sr_token<256, 2>(x, R, C, ld, seed, q, sblk, s32, sm_count, stream);
  else if (nb <= 1024)
    launch_sr_token<256, 4>(x, R, C, ld, seed, q, sblk, s32, sm_count, stream);
  else
    launch_sr_token<256, 0>(x, R, C, ld, seed, q, sblk, s32, sm_count, stream);
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
