// Host-side launch interface of the CUDA kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mx8q {

// Bytes of K per GEMM pipeline stage and operand row: one swizzle atom, 128
// (SWIZZLE_128B boxes and descriptors) or 64 (SWIZZLE_64B).  64-byte stages
// double the stage count in the same shared memory but measured slower on
// GB300 (MXFP8 Fprop 2048x8192x2048: 78 us against 51 us): each stage's
// barrier, scale copies and commit cost about the same fixed time.
constexpr int kGemmKBytes = 128;

constexpr int kMaxGroups = 1024;   // groups (experts) per grouped call
#define MX8Q_S32_GROUP_MODE 3          // FP32 scale per group (same value as MX8_S32_GROUP)

// Tensors of one MXFP8 / MXFP4 quantization launch: their 128x128 tiles are
// numbered one after the other (tensor i's tiles start at t[i].tile0).
constexpr int kQuantBatchMax = 4;
struct QuantTensor {
  int64_t R, C;
  uint8_t* q_row;
  uint8_t* s_row;
  uint8_t* q_col;
  uint8_t* s_col;
  int64_t tile0;
};
struct __align__(64) QuantBatch {
  CUtensorMap maps[kQuantBatchMax];   // bf16 [R, C] with 128x128 boxes
  QuantTensor t[kQuantBatchMax];
  int n;
  int64_t ntiles;
};

size_t mxfp8_quant_smem_bytes();
// fp4: MXFP4 (packed E2M1 data) instead of MXFP8 (E4M3 data)
cudaError_t launch_mxfp8_quant(const QuantBatch& batch, bool row, bool col, bool fp4, int* err, int sm_count,
                               cudaStream_t stream);

// Scratch bytes of the group / tensor scope path (amax, done counts, ticket).
size_t nvfp4_scratch_bytes(int groups);
// scratch: nvfp4_scratch_bytes(groups) bytes, 16-byte aligned (zeroed here on
// the stream); err: the error word a timed-out wait writes.
cudaError_t launch_nvfp4_quant(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int scope,
                               const int64_t* offs, int G, uint8_t* q, uint8_t* sblk, float* s32,
                               void* scratch, int* err, int sm_count, cudaStream_t stream);

// Per-token NVFP4 of T tokens before dispatch: scale words to the grouped
// scale rows of each token's topk dispatched copies (dest [T * topk], offs
// [G + 1]); codes and S_dec to the copies' rows (disp_codes) or token-major.
constexpr int kMaxTopk = 16;
cudaError_t launch_nvfp4_dispatch(const uint16_t* x, int64_t T, int64_t C, int64_t ld, const int64_t* dest,
                                  int topk, const int64_t* offs, int G, int disp_codes, uint8_t* q, uint8_t* sblk,
                                  float* s32, int sm_count, cudaStream_t stream);

// Tensor abs-max of a bf16 matrix (C % 8 == 0) as f32 bits in *amax_bits
// (zeroed here on the stream).
cudaError_t launch_absmax(const uint16_t* x, int64_t R, int64_t C, int64_t ld, uint32_t* amax_bits, int sm_count,
                          cudaStream_t stream);

// NVFP4 with 16x16 block scales and one FP32 tensor scale (rowwise and/or
// the transposed copy); amax_bits: 4 bytes of device scratch.
cudaError_t launch_nvfp4_2d(const uint16_t* x, int64_t R, int64_t C, int64_t ld, bool row, bool col,
                            uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, float* s32,
                            uint32_t* amax_bits, int sm_count, cudaStream_t stream);

// Transposed NVFP4 copy of a Wgrad input with the 16x16 random Hadamard
// transform along its rows (tensor-scope scale from the transformed amax).
cudaError_t launch_nvfp4_rht_colwise(const uint16_t* x, int64_t R, int64_t C, int64_t ld, uint32_t mask, bool sr,
                                     uint64_t seed, uint8_t* qT, uint8_t* sT, float* s32, uint32_t* amax_bits,
                                     int sm_count, cudaStream_t stream);
// Per-token NVFP4 of a gradient with stochastically rounded codes.
cudaError_t launch_nvfp4_sr_token(const uint16_t* x, int64_t R, int64_t C, int64_t ld, uint64_t seed, uint8_t* q,
                                  uint8_t* sblk, float* s32, int sm_count, cudaStream_t stream);

cudaError_t launch_dequant(int fmt, const uint8_t* q, const uint8_t* s, const float* s32,
                           int s32_mode, const int64_t* offs, int G, int64_t R, int64_t C,
                           int out_bf16, void* out, int sm_count, cudaStream_t stream);

// out[t] = sum_j w[t][j] * y[rows[t][j]], binary32 in j order (rows outside
// [0, R) skipped); H % 8 == 0.
cudaError_t launch_combine(const uint16_t* y, int64_t ldy, int64_t R, const int64_t* rows, const float* w, int64_t T,
                           int64_t H, int k, bool bf16_out, void* out, int64_t ldo, int sm_count, cudaStream_t stream);

cudaError_t launch_swiglu(const uint16_t* gu, int64_t R, int64_t F, int64_t ld_gu, uint16_t* h,
                          int64_t ld_h, int sm_count, cudaStream_t stream);

struct GemmArgs {
  int fmt;                 // 0 MXFP8, 1 NVFP4, 2 MXFP4, 3 BF16 (no block scales)
  int64_t M, N, K;         // K in elements
  const uint8_t* SA;       // tensor-core scale tiles of A
  const uint8_t* SB;
  const float* A32;        // per-row (or per-tensor) FP32 decode scales
  int a32_mode;
  const float* B32;
  int b32_mode;            // grouped: per group
  void* C;
  int64_t ldc;
  int out_bf16;
  int accumulate;
  // grouped GEMM
  int grouped;
  int G;
  const int64_t* offs;
  // fused MoE modes (grouped only)
  const uint8_t* A;        // gathered mode: token-major A data [a_src_rows, K bytes]
  const int64_t* a_rows;   // gathered mode: token of each dispatched row [M]
  int64_t a_src_rows;      // gathered mode: rows of the token-major A
  int64_t ffn;             // SwiGLU mode: F (up rows of B start at F; output has F columns)
  // SwiGLU mode with h quantized per token to NVFP4 (C, the bf16 h, optional)
  uint8_t* qh;             // [M, F/2] packed E2M1 codes of h
  uint8_t* qh_scales;      // E4M3 block scales of h, grouped tile layout
  float* qh_s32;           // [M] S_dec of h
  int* err;
};

// tmap_c: the output [rows, N] as a 2-D map with a box of 64 bytes x 32 rows
// (element type of the output), used for the epilogue's bulk stores.
// (qh set: the SwiGLU grouped GEMM with h quantized, launched as clusters of
// F / 128 CTAs; F / 128 must be 1 .. 8)
cudaError_t launch_bs_gemm(const GemmArgs& a, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                           const CUtensorMap& tmap_c, int sm_count, cudaStream_t stream);

cudaError_t launch_selftest_wait(int* err, uint64_t limit_ns, cudaStream_t stream);

}  // namespace mx8q
