// NVFP4 weights with 2-D 16x16 block scaling ("NVIDIA presenta una
// metodologia de preentrenamiento de 4 bits utilizando NVFP4", section "La
// metodologia de formacion de cuatro partes"): the backward pass multiplies
// by the transposed weight, and 1x16 blocks along K would quantize it
// differently from the forward weight; one scale per 16x16 block gives both
// passes the same quantized values.  One FP32 scale for the tensor:
//   S_enc = min(RN(2688 / A), FLT_MAX), S_dec = RN(A / 2688)   (A = tensor amax)
//   per 16x16 block: sb = RNE_E4M3_sat(RN(RN(amax_b / 6) * S_enc)),
//                    r  = sb ? min(RN(S_enc / sb), FLT_MAX) : 0,
//                    code = RNE_E2M1_sat(RN(x * r))
// Outputs: the rowwise copy (q_row [R, C/2], every row of a block carrying
// the block's scale in the tensor-core tile layout) and the columnwise copy
// (q_col [C, R/2]): the transposes of each other, codes and scales alike.
//
// Two launches: a tensor abs-max (atomicMax of the f32 bits, which order
// like the values for x >= 0), then the encode over 128 x 128 tiles: thread
// t owns rows 4(t%4)..+3 of 16x16 block t/4 (8 x 8 blocks per tile), takes
// the block maximum with two shuffles, writes its rows' codes, parks the
// bf16 tile in shared memory and reads its 4 columns of the block back for
// the transposed codes.  Scale bytes are staged per 128-row group as whole
// 512-byte tensor-core tiles and written with 16-byte stores.
#include "device.cuh"
#include "kernels.h"

namespace mx8q {

namespace {

constexpr int kTile = 128;
constexpr int k2dThreads = 256;

__global__ void __launch_bounds__(k2dThreads) absmax_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                           int64_t ld, uint32_t* __restrict__ amax_bits) {
  const int64_t chunks = C / 8;                  // 16-byte chunks per row
  uint32_t m = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * k2dThreads + threadIdx.x; i < R * chunks;
       i += static_cast<int64_t>(gridDim.x) * k2dThreads) {
    const int64_t r = i / chunks, c = (i % chunks) * 8;
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(x + r * ld + c));
    m = amax2(m, amax2(amax2(w.x, w.y), amax2(w.z, w.w)));
  }
  float v = warp_max(abs_halves_max(m));
  __shared__ float red[k2dThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < k2dThreads / 32; ++i) v = fmaxf(v, red[i]);
    atomicMax(amax_bits, __float_as_uint(v));
  }
}

__device__ __forceinline__ int tile_byte(int row, int k) {   // offset in a 128 x 4 scale tile
  return (row & 31) * 16 + ((row >> 5) & 3) * 4 + (k & 3);
}

template <bool kRow, bool kCol>
__global__ void __launch_bounds__(k2dThreads) nvfp4_2d_kernel(
    const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ld, const uint32_t* __restrict__ amax_bits,
    uint8_t* __restrict__ q_row, uint8_t* __restrict__ s_row, uint8_t* __restrict__ q_col,
    uint8_t* __restrict__ s_col, float* __restrict__ s32) {
  __shared__ __align__(16) uint16_t tile[kTile][kTile];        // 32 KB
  __shared__ __align__(16) uint8_t srow[2][512];
  __shared__ __align__(16) uint8_t scol[2][512];
  const int t = threadIdx.x;
  const int b = t >> 2, p = t & 3;            // block of the tile, part of the block
  const int bi = b >> 3, bj = b & 7;          // block row / column in the tile
  float senc, sdec;
  nvfp4_scales(__uint_as_float(*amax_bits), senc, sdec);
  if (blockIdx.x == 0 && t == 0) s32[0] = sdec;

  const int64_t tiles_c = (C + kTile - 1) / kTile, tiles_r = (R + kTile - 1) / kTile;
  const int64_t kt_row = (C / 16 + 3) / 4, kt_col = (R / 16 + 3) / 4;   // scale tiles per 128-row group
  for (int64_t tl = blockIdx.x; tl < tiles_r * tiles_c; tl += gridDim.x) {
    const int64_t r0 = (tl / tiles_c) * kTile, c0 = (tl % tiles_c) * kTile;
    const int64_t br = r0 + 16 * bi + 4 * p;   // first of this thread's 4 rows
    const int64_t bc = c0 + 16 * bj;           // first column of the block
    const bool in = br < R && bc < C;          // R, C are multiples of 16: blocks are whole
    uint4 w[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t* src = x + (br + i) * ld + bc;
      w[2 * i] = in ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0, 0, 0, 0);
      w[2 * i + 1] = in ? __ldg(reinterpret_cast<const uint4*>(src + 8)) : make_uint4(0, 0, 0, 0);
    }
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = amax2(m, absmax16(w[2 * i], w[2 * i + 1]));
    float bmax = abs_halves_max(m);
    bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 1));
    bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 2));
    const uint32_t sb = cvt_e4m3x2(__fmul_rn(__fdiv_rn(bmax, 6.0f), senc), 0.0f) & 0xFFu;
    const float r = sb ? fminf(__fdiv_rn(senc, e4m3_to_f32(sb)), FLT_MAX) : 0.f;
    const uint64_t rr = f32x2_splat(r);

    __syncthreads();                           // the previous tile's staging has been read
    if (kRow) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t ws[8] = {w[2 * i].x, w[2 * i].y, w[2 * i].z, w[2 * i].w,
                                w[2 * i + 1].x, w[2 * i + 1].y, w[2 * i + 1].z, w[2 * i + 1].w};
        float v0[8], v1[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          mul_bf16x2(ws[j], rr, v0[2 * j], v0[2 * j + 1]);
          mul_bf16x2(ws[4 + j], rr, v1[2 * j], v1[2 * j + 1]);
        }
        if (in) *reinterpret_cast<uint2*>(q_row + (br + i) * (C / 2) + bc / 2) = make_uint2(cvt_e2m1x8(v0), cvt_e2m1x8(v1));
        srow[bj >> 2][tile_byte(16 * bi + 4 * p + i, bj)] = static_cast<uint8_t>(sb);
      }
    }
    if (kCol) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        *reinterpret_cast<uint4*>(&tile[16 * bi + 4 * p + i][16 * bj]) = w[2 * i];
        *reinterpret_cast<uint4*>(&tile[16 * bi + 4 * p + i][16 * bj + 8]) = w[2 * i + 1];
      }
    }
    __syncthreads();
    if (kCol) {
      // columns 16 bj + 4p .. +3 of the block, 16 rows each: the transposed copy
      uint32_t col[2][16];                     // bf16 pairs (columns 4p+2h, 4p+2h+1) per row
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint2 v = *reinterpret_cast<const uint2*>(&tile[16 * bi + i][16 * bj + 4 * p]);
        col[0][i] = v.x;
        col[1][i] = v.y;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {          // column 4p + 2h + e
          float v0[8], v1[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t a = col[h][i], c = col[h][8 + i];
            v0[i] = __fmul_rn(e ? bf16_hi(a) : bf16_lo(a), r);
            v1[i] = __fmul_rn(e ? bf16_hi(c) : bf16_lo(c), r);
          }
          const int64_t k = bc + 4 * p + 2 * h + e;
          if (in) *reinterpret_cast<uint2*>(q_col + k * (R / 2) + (r0 + 16 * bi) / 2) = make_uint2(cvt_e2m1x8(v0), cvt_e2m1x8(v1));
          scol[bi >> 2][tile_byte(16 * bj + 4 * p + 2 * h + e, bi)] = static_cast<uint8_t>(sb);
        }
      }
    }
    if (kCol) __syncthreads();                 // the transposed scales are staged
    // whole 512-byte scale tiles: rows r0.. (k4 groups c0/64, +1) and
    // transposed rows c0.. (k4 groups r0/64, +1)
    if (kRow && t < 64) {
      const int j = t >> 5;
      const int64_t kg = c0 / 64 + j;
      if (kg < kt_row)
        reinterpret_cast<uint4*>(s_row + ((r0 / kTile) * kt_row + kg) * 512)[t & 31] =
            reinterpret_cast<const uint4*>(srow[j])[t & 31];
    }
    if (kCol && t >= 64 && t < 128) {
      const int j = (t - 64) >> 5;
      const int64_t kg = r0 / 64 + j;
      if (kg < kt_col)
        reinterpret_cast<uint4*>(s_col + ((c0 / kTile) * kt_col + kg) * 512)[t & 31] =
            reinterpret_cast<const uint4*>(scol[j])[t & 31];
    }
  }
}

}  // namespace

cudaError_t launch_absmax(const uint16_t* x, int64_t R, int64_t C, int64_t ld, uint32_t* amax_bits, int sm_count,
                          cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  const int64_t work = R * (C / 8);
  const int64_t ga = (work + k2dThreads - 1) / k2dThreads;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  absmax_kernel<<<static_cast<unsigned>(ga < cap ? ga : cap), k2dThreads, 0, stream>>>(x, R, C, ld, amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_2d(const uint16_t* x, int64_t R, int64_t C, int64_t ld, bool row, bool col,
                            uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, float* s32,
                            uint32_t* amax_bits, int sm_count, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  const int64_t work = R * (C / 8);
  const int64_t ga = (work + k2dThreads - 1) / k2dThreads;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  absmax_kernel<<<static_cast<unsigned>(ga < cap ? ga : cap), k2dThreads, 0, stream>>>(x, R, C, ld, amax_bits);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t tiles = ((R + kTile - 1) / kTile) * ((C + kTile - 1) / kTile);
  const int64_t cap2 = static_cast<int64_t>(sm_count) * 4;
  const unsigned grid = static_cast<unsigned>(tiles < cap2 ? tiles : cap2);
  auto k = row ? (col ? nvfp4_2d_kernel<true, true> : nvfp4_2d_kernel<true, false>) : nvfp4_2d_kernel<false, true>;
  k<<<grid, k2dThreads, 0, stream>>>(x, R, C, ld, amax_bits, q_row, s_row, q_col, s_col, s32);
  return cudaGetLastError();
}

}  // namespace mx8q
