// C-ABI entry points: argument validation, TMA descriptor encoding and kernel
// launches on the caller's stream.  The library never allocates device
// memory; all buffers, including the workspace, belong to the caller.
#include <cudaTypedefs.h>
#include <stdio.h>

#include <mutex>

#include "mx8q.h"
#include "device.cuh"
#include "kernels.h"

using namespace mx8q;

namespace {

constexpr size_t kErrWordBytes = 256;   // error word + padding; scratch starts here

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------- device info
int sm_count_current() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// ------------------------------------------------------------- TMA encode
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D or 3-D tiled map; dims/strides innermost first, strides in bytes for
// dimensions 1.. (dimension 0 is contiguous).
bool encode_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  uint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dt, rank, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int* err_word(void* ws) { return static_cast<int*>(ws); }

mx8_status check_ws(void* ws, size_t bytes, int groups) {
  if (ws == nullptr || !aligned16(ws)) return MX8_ERR_WORKSPACE;
  if (bytes < mx8_workspace_bytes(groups)) return MX8_ERR_WORKSPACE;
  return MX8_OK;
}

mx8_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MX8_OK : MX8_ERR_CUDA; }

}  // namespace

// ===================================================================== sizes
extern "C" size_t mx8_scale_bytes(int fmt, int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0) return 0;
  const int64_t bs = fmt == MX8_FMT_NVFP4 ? 16 : 32;
  return static_cast<size_t>(cdiv(rows, 128) * 128 * cdiv(cols / bs, 4) * 4);
}

extern "C" size_t mx8_scale_bytes_grouped(int fmt, int64_t total_rows, int num_groups, int64_t cols) {
  if (total_rows < 0 || cols < 0 || num_groups < 0) return 0;
  const int64_t bs = fmt == MX8_FMT_NVFP4 ? 16 : 32;
  const int64_t tiles = cdiv(total_rows, 128) + num_groups;
  return static_cast<size_t>(tiles * 128 * cdiv(cols / bs, 4) * 4);
}

extern "C" size_t mx8_workspace_bytes(int num_groups) {
  const int64_t g = num_groups > 1 ? num_groups : 1;
  return kErrWordBytes + static_cast<size_t>(cdiv(static_cast<int64_t>(nvfp4_scratch_bytes(static_cast<int>(g))), 256) * 256);
}

extern "C" int mx8_device_sm_count(void) { return sm_count_current(); }

extern "C" const char* mx8_status_string(mx8_status s) {
  switch (s) {
    case MX8_OK: return "ok";
    case MX8_ERR_INVALID_ARG: return "invalid argument";
    case MX8_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case MX8_ERR_UNSUPPORTED: return "unsupported request";
    case MX8_ERR_CUDA: return "CUDA error";
    case MX8_ERR_TIMEOUT: return "a bounded device wait ran out";
    case MX8_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

// ===================================================================== MXFP8 / MXFP4
namespace {
// Checks one quantization input (same rules for mx8_quantize / mxfp4_quantize
// and their batch form); *empty is set when there is nothing to do.
mx8_status check_quant_item(bool row, bool col, const void* x, int64_t rows, int64_t cols, int64_t ld,
                            const uint8_t* q_row, const uint8_t* s_row, const uint8_t* q_col, const uint8_t* s_col,
                            bool* empty) {
  *empty = true;
  if (rows < 0 || cols < 0 || ld < cols || cols % 32 != 0) return MX8_ERR_INVALID_ARG;
  if (col && rows % 32 != 0) return MX8_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MX8_OK;
  if (x == nullptr || (row && (q_row == nullptr || s_row == nullptr)) ||
      (col && (q_col == nullptr || s_col == nullptr)))
    return MX8_ERR_INVALID_ARG;
  if (!aligned16(x) || ld % 8 != 0 || (row && (!aligned16(q_row) || !aligned16(s_row))) ||
      (col && (!aligned16(q_col) || !aligned16(s_col))))
    return MX8_ERR_ALIGNMENT;
  if (rows > INT32_MAX || cols > INT32_MAX) return MX8_ERR_UNSUPPORTED;
  *empty = false;
  return MX8_OK;
}

// Adds a checked, non-empty input to the batch: its tensor map and tile range.
bool add_quant_item(QuantBatch& b, const void* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q_row,
                    uint8_t* s_row, uint8_t* q_col, uint8_t* s_col) {
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(ld) * 2};
  const uint32_t box[2] = {128, 128};
  const int i = b.n;
  if (!encode_map(&b.maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
    return false;
  b.t[i] = QuantTensor{rows, cols, q_row, s_row, q_col, s_col, b.ntiles};
  b.ntiles += cdiv(rows, 128) * cdiv(cols, 128);
  b.n = i + 1;
  return true;
}

mx8_status mx_quantize(bool fp4, const void* x, int64_t rows, int64_t cols, int64_t ld, int flags,
                       uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                       void* workspace, size_t workspace_bytes, mx8_stream_t stream) {
  const bool row = flags & MX8_ROWWISE, col = flags & MX8_COLWISE;
  if ((flags & ~(MX8_ROWWISE | MX8_COLWISE)) || !(row || col)) return MX8_ERR_INVALID_ARG;
  bool empty = true;
  mx8_status st = check_quant_item(row, col, x, rows, cols, ld, q_row, s_row, q_col, s_col, &empty);
  if (st != MX8_OK || empty) return st;
  st = check_ws(workspace, workspace_bytes, 1);
  if (st != MX8_OK) return st;
  QuantBatch b{};
  if (!add_quant_item(b, x, rows, cols, ld, q_row, s_row, q_col, s_col)) return MX8_ERR_CUDA;
  return from_cuda(launch_mxfp8_quant(b, row, col, fp4, err_word(workspace), sm_count_current(),
                                      reinterpret_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" mx8_status mx8_quantize_batch(int fmt, const mx8_quantize_item* items, int n, int flags,
                                         void* workspace, size_t workspace_bytes, mx8_stream_t stream) {
  if (fmt != MX8_FMT_MXFP8 && fmt != MX8_FMT_MXFP4) return MX8_ERR_INVALID_ARG;
  if (n < 1 || n > MX8_BATCH_MAX || items == nullptr) return MX8_ERR_INVALID_ARG;
  static_assert(MX8_BATCH_MAX <= kQuantBatchMax, "batch larger than the kernel's tensor list");
  const bool row = flags & MX8_ROWWISE, col = flags & MX8_COLWISE;
  if ((flags & ~(MX8_ROWWISE | MX8_COLWISE)) || !(row || col)) return MX8_ERR_INVALID_ARG;
  bool any = false;
  for (int i = 0; i < n; ++i) {
    const mx8_quantize_item& it = items[i];
    bool empty = true;
    mx8_status st = check_quant_item(row, col, it.x, it.rows, it.cols, it.ld, it.q_row, it.s_row, it.q_col,
                                     it.s_col, &empty);
    if (st != MX8_OK) return st;
    any = any || !empty;
  }
  if (!any) return MX8_OK;
  mx8_status st = check_ws(workspace, workspace_bytes, 1);
  if (st != MX8_OK) return st;
  QuantBatch b{};
  for (int i = 0; i < n; ++i) {
    const mx8_quantize_item& it = items[i];
    if (it.rows == 0 || it.cols == 0) continue;
    if (!add_quant_item(b, it.x, it.rows, it.cols, it.ld, it.q_row, it.s_row, it.q_col, it.s_col))
      return MX8_ERR_CUDA;
  }
  return from_cuda(launch_mxfp8_quant(b, row, col, fmt == MX8_FMT_MXFP4, err_word(workspace), sm_count_current(),
                                      reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" mx8_status mx8_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int flags,
                                   uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                   void* workspace, size_t workspace_bytes, mx8_stream_t stream) {
  return mx_quantize(false, x, rows, cols, ld, flags, q_row, s_row, q_col, s_col, workspace,
                     workspace_bytes, stream);
}

extern "C" mx8_status mxfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int flags,
                                     uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                     void* workspace, size_t workspace_bytes, mx8_stream_t stream) {
  return mx_quantize(true, x, rows, cols, ld, flags, q_row, s_row, q_col, s_col, workspace,
                     workspace_bytes, stream);
}

// ===================================================================== NVFP4
extern "C" mx8_status nvfp4_quantize_per_token(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                               int scope, const int64_t* group_offsets,
                                               int num_groups, uint8_t* q, uint8_t* s_blk,
                                               float* s32, void* workspace, size_t workspace_bytes,
                                               mx8_stream_t stream) {
  if (scope < NVFP4_SCOPE_TOKEN || scope > NVFP4_SCOPE_TENSOR) return MX8_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || ld < cols || cols % 16 != 0) return MX8_ERR_INVALID_ARG;
  if (cols > (int64_t{1} << 30)) return MX8_ERR_UNSUPPORTED;   // columns are 32-bit in the kernels
  if (scope == NVFP4_SCOPE_GROUP && group_offsets == nullptr) return MX8_ERR_INVALID_ARG;
  if (group_offsets != nullptr && (num_groups < 1 || num_groups > kMaxGroups)) return MX8_ERR_INVALID_ARG;
  const int G = group_offsets ? num_groups : 1;
  if (cols == 0) return MX8_OK;
  if (rows > 0 && (x == nullptr || q == nullptr)) return MX8_ERR_INVALID_ARG;
  if (s_blk == nullptr || s32 == nullptr) return MX8_ERR_INVALID_ARG;
  if ((rows > 0 && (!aligned16(x) || !aligned16(q))) || !aligned16(s_blk) || ld % 8 != 0)
    return MX8_ERR_ALIGNMENT;
  mx8_status st = check_ws(workspace, workspace_bytes, G);
  if (st != MX8_OK) return st;
  void* scratch = static_cast<uint8_t*>(workspace) + kErrWordBytes;
  return from_cuda(launch_nvfp4_quant(static_cast<const uint16_t*>(x), rows, cols, ld, scope,
                                      group_offsets, G, q, s_blk, s32, scratch, err_word(workspace),
                                      sm_count_current(), reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" mx8_status nvfp4_quantize_dispatch(const void* x, int64_t tokens, int64_t cols, int64_t ld,
                                              const int64_t* dest_rows, int topk, const int64_t* group_offsets,
                                              int num_groups, int layout, uint8_t* q, uint8_t* s_blk, float* s32,
                                              void* workspace, size_t workspace_bytes, mx8_stream_t stream) {
  if (tokens < 0 || cols < 0 || ld < cols || cols % 16 != 0) return MX8_ERR_INVALID_ARG;
  if (layout != MX8_DISPATCH_TOKENS && layout != MX8_DISPATCH_ROWS) return MX8_ERR_INVALID_ARG;
  if (topk < 1 || topk > kMaxTopk) return MX8_ERR_INVALID_ARG;
  if (group_offsets == nullptr || num_groups < 1 || num_groups > kMaxGroups) return MX8_ERR_INVALID_ARG;
  if (cols > (int64_t{1} << 30)) return MX8_ERR_UNSUPPORTED;
  if (tokens == 0 || cols == 0) return MX8_OK;
  if (x == nullptr || q == nullptr || s_blk == nullptr || s32 == nullptr || dest_rows == nullptr)
    return MX8_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(s_blk) || ld % 8 != 0) return MX8_ERR_ALIGNMENT;
  mx8_status st = check_ws(workspace, workspace_bytes, num_groups);
  if (st != MX8_OK) return st;
  return from_cuda(launch_nvfp4_dispatch(static_cast<const uint16_t*>(x), tokens, cols, ld, dest_rows, topk,
                                         group_offsets, num_groups, layout == MX8_DISPATCH_ROWS, q, s_blk, s32,
                                         sm_count_current(),
                                         reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" mx8_status nvfp4_quantize_2d(const void* x, int64_t rows, int64_t cols, int64_t ld, int flags,
                                        uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                        float* s32, void* workspace, size_t workspace_bytes,
                                        mx8_stream_t stream) {
  const bool row = flags & MX8_ROWWISE, col = flags & MX8_COLWISE;
  if ((flags & ~(MX8_ROWWISE | MX8_COLWISE)) || !(row || col)) return MX8_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || ld < cols || rows % 32 != 0 || cols % 32 != 0) return MX8_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MX8_OK;
  if (x == nullptr || s32 == nullptr || (row && (q_row == nullptr || s_row == nullptr)) ||
      (col && (q_col == nullptr || s_col == nullptr)))
    return MX8_ERR_INVALID_ARG;
  if (!aligned16(x) || ld % 8 != 0 || (row && (!aligned16(q_row) || !aligned16(s_row))) ||
      (col && (!aligned16(q_col) || !aligned16(s_col))))
    return MX8_ERR_ALIGNMENT;
  if (rows > INT32_MAX || cols > INT32_MAX) return MX8_ERR_UNSUPPORTED;
  mx8_status st = check_ws(workspace, workspace_bytes, 1);
  if (st != MX8_OK) return st;
  uint32_t* amax_bits = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + kErrWordBytes);
  return from_cuda(launch_nvfp4_2d(static_cast<const uint16_t*>(x), rows, cols, ld, row, col, q_row, s_row,
                                   q_col, s_col, s32, amax_bits, sm_count_current(),
                                   reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" mx8_status nvfp4_quantize_rht_colwise(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                                 uint32_t sign_mask, int stochastic, uint64_t seed, uint8_t* q_col,
                                                 uint8_t* s_col, float* s32, void* workspace,
                                                 size_t workspace_bytes, mx8_stream_t stream) {
  if (rows < 0 || cols < 0 || ld < cols || rows % 32 != 0 || cols % 8 != 0 || sign_mask > 0xFFFFu)
    return MX8_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MX8_OK;
  if (x == nullptr || q_col == nullptr || s_col == nullptr || s32 == nullptr) return MX8_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q_col) || !aligned16(s_col) || ld % 8 != 0) return MX8_ERR_ALIGNMENT;
  if (rows > INT32_MAX || cols > INT32_MAX) return MX8_ERR_UNSUPPORTED;
  mx8_status st = check_ws(workspace, workspace_bytes, 1);
  if (st != MX8_OK) return st;
  uint32_t* amax_bits = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + kErrWordBytes);
  return from_cuda(launch_nvfp4_rht_colwise(static_cast<const uint16_t*>(x), rows, cols, ld, sign_mask,
                                            stochastic != 0, seed, q_col, s_col, s32, amax_bits,
                                            sm_count_current(), reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" mx8_status nvfp4_quantize_per_token_sr(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                                  uint64_t seed, uint8_t* q, uint8_t* s_blk, float* s32,
                                                  mx8_stream_t stream) {
  if (rows < 0 || cols < 0 || ld < cols || cols % 16 != 0) return MX8_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MX8_OK;
  if (x == nullptr || q == nullptr || s_blk == nullptr || s32 == nullptr) return MX8_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(s_blk) || ld % 8 != 0) return MX8_ERR_ALIGNMENT;
  return from_cuda(launch_nvfp4_sr_token(static_cast<const uint16_t*>(x), rows, cols, ld, seed, q, s_blk, s32,
                                         sm_count_current(), reinterpret_cast<cudaStream_t>(stream)));
}

// ===================================================================== dequantize
extern "C" mx8_status dequantize(int fmt, const uint8_t* q, const uint8_t* s, const float* s32,
                                 int s32_mode, const int64_t* group_offsets, int num_groups,
                                 int64_t rows, int64_t cols, int out_dtype, void* out,
                                 mx8_stream_t stream) {
  if (fmt != MX8_FMT_MXFP8 && fmt != MX8_FMT_NVFP4 && fmt != MX8_FMT_MXFP4) return MX8_ERR_INVALID_ARG;
  if (out_dtype != MX8_OUT_F32 && out_dtype != MX8_OUT_BF16) return MX8_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || cols % (fmt == MX8_FMT_NVFP4 ? 16 : 32) != 0) return MX8_ERR_INVALID_ARG;
  if (s32_mode < MX8_S32_NONE || s32_mode > MX8_S32_GROUP) return MX8_ERR_INVALID_ARG;
  if (fmt != MX8_FMT_NVFP4 && s32_mode != MX8_S32_NONE) return MX8_ERR_INVALID_ARG;
  if (s32_mode != MX8_S32_NONE && s32 == nullptr) return MX8_ERR_INVALID_ARG;
  if ((s32_mode == MX8_S32_GROUP || group_offsets != nullptr) &&
      (group_offsets == nullptr || num_groups < 1 || num_groups > kMaxGroups))
    return MX8_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MX8_OK;
  if (q == nullptr || s == nullptr || out == nullptr) return MX8_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return MX8_ERR_ALIGNMENT;
  return from_cuda(launch_dequant(fmt, q, s, s32, s32_mode, group_offsets, num_groups, rows, cols,
                                  out_dtype == MX8_OUT_BF16, out, sm_count_current(),
                                  reinterpret_cast<cudaStream_t>(stream)));
}

// ===================================================================== SwiGLU
extern "C" mx8_status mx8_swiglu(const void* gate_up, int64_t rows, int64_t ffn, int64_t ld_gate_up,
                                 void* h, int64_t ld_h, mx8_stream_t stream) {
  if (rows < 0 || ffn < 0 || ffn % 8 != 0 || ld_gate_up < 2 * ffn || ld_h < ffn) return MX8_ERR_INVALID_ARG;
  if (rows == 0 || ffn == 0) return MX8_OK;
  if (gate_up == nullptr || h == nullptr) return MX8_ERR_INVALID_ARG;
  if (!aligned16(gate_up) || !aligned16(h) || ld_gate_up % 8 != 0 || ld_h % 8 != 0) return MX8_ERR_ALIGNMENT;
  return from_cuda(launch_swiglu(static_cast<const uint16_t*>(gate_up), rows, ffn, ld_gate_up,
                                 static_cast<uint16_t*>(h), ld_h, sm_count_current(),
                                 reinterpret_cast<cudaStream_t>(stream)));
}

// ===================================================================== MoE combine
extern "C" mx8_status mx8_moe_combine(const void* y, int64_t rows_y, int64_t ld_y, const int64_t* rows_of_slot,
                                      const float* weights, int64_t tokens, int64_t hidden, int topk,
                                      int out_dtype, void* out, int64_t ld_out, mx8_stream_t stream) {
  if (rows_y < 0 || tokens < 0 || hidden < 0 || hidden % 8 != 0 || ld_y < hidden || ld_out < hidden)
    return MX8_ERR_INVALID_ARG;
  if (topk < 1 || topk > kMaxTopk) return MX8_ERR_INVALID_ARG;
  if (out_dtype != MX8_OUT_F32 && out_dtype != MX8_OUT_BF16) return MX8_ERR_INVALID_ARG;
  if (tokens == 0 || hidden == 0) return MX8_OK;
  if (y == nullptr || rows_of_slot == nullptr || weights == nullptr || out == nullptr) return MX8_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out) || ld_y % 8 != 0 || ld_out % 8 != 0) return MX8_ERR_ALIGNMENT;
  return from_cuda(launch_combine(static_cast<const uint16_t*>(y), ld_y, rows_y, rows_of_slot, weights, tokens,
                                  hidden, topk, out_dtype == MX8_OUT_BF16, out, ld_out, sm_count_current(),
                                  reinterpret_cast<cudaStream_t>(stream)));
}

// ===================================================================== GEMM
namespace {

mx8_status gemm_common_checks(int fmt, int64_t N, int64_t K, const uint8_t* A, const uint8_t* SA,
                              const uint8_t* B, const uint8_t* SB, int out_dtype, void* C,
                              int64_t ldc) {
  if (fmt != MX8_FMT_MXFP8 && fmt != MX8_FMT_NVFP4 && fmt != MX8_FMT_MXFP4) return MX8_ERR_INVALID_ARG;
  if (out_dtype != MX8_OUT_F32 && out_dtype != MX8_OUT_BF16) return MX8_ERR_INVALID_ARG;
  if (N < 0 || K < 0 || K % 32 != 0 || ldc < N) return MX8_ERR_INVALID_ARG;
  if (A == nullptr || SA == nullptr || B == nullptr || SB == nullptr || C == nullptr)
    return MX8_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(SA) || !aligned16(B) || !aligned16(SB) || !aligned16(C) ||
      ldc % 8 != 0)
    return MX8_ERR_ALIGNMENT;
  return MX8_OK;
}

// TMA swizzle of the GEMM operand boxes: one swizzle atom of kGemmKBytes.
CUtensorMapSwizzle gemm_swizzle() {
  return kGemmKBytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
}

// Output map for the GEMM epilogue's bulk stores: [rows, N] with row stride
// ldc, box 64 bytes x 32 rows.
bool encode_output_map(CUtensorMap* map, void* C, int64_t rows, int64_t N, int64_t ldc, int out_dtype) {
  const bool bf = out_dtype == MX8_OUT_BF16;
  const uint64_t es = bf ? 2 : 4;
  const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(ldc) * es};
  const uint32_t box[2] = {static_cast<uint32_t>(64 / es), 32};
  return encode_map(map, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims,
                    strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

cudaError_t zero_output(void* C, int64_t ldc, int64_t rows, int64_t N, int out_dtype, cudaStream_t s) {
  const size_t es = out_dtype == MX8_OUT_BF16 ? 2 : 4;
  return cudaMemset2DAsync(C, ldc * es, 0, N * es, rows, s);
}

}  // namespace

extern "C" mx8_status bs_gemm(int fmt, int64_t M, int64_t N, int64_t K, const uint8_t* A,
                              const uint8_t* SA, const float* A32, int a32_mode, const uint8_t* B,
                              const uint8_t* SB, const float* B32, int b32_mode, int out_dtype,
                              void* C, int64_t ldc, int accumulate, void* workspace,
                              size_t workspace_bytes, mx8_stream_t stream) {
  if (M < 0) return MX8_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MX8_OK;
  mx8_status st = gemm_common_checks(fmt, N, K, A, SA, B, SB, out_dtype, C, ldc);
  if (st != MX8_OK) return st;
  if (a32_mode < 0 || a32_mode > MX8_S32_TENSOR || b32_mode < 0 || b32_mode > MX8_S32_TENSOR)
    return MX8_ERR_INVALID_ARG;
  if ((a32_mode != MX8_S32_NONE && A32 == nullptr) || (b32_mode != MX8_S32_NONE && B32 == nullptr))
    return MX8_ERR_INVALID_ARG;
  if (accumulate && out_dtype != MX8_OUT_F32) return MX8_ERR_UNSUPPORTED;
  if (M > INT32_MAX || N > INT32_MAX) return MX8_ERR_UNSUPPORTED;
  st = check_ws(workspace, workspace_bytes, 1);
  if (st != MX8_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return accumulate ? MX8_OK : from_cuda(zero_output(C, ldc, M, N, out_dtype, s));

  const uint64_t kbytes = fmt == MX8_FMT_MXFP8 ? K : K / 2;
  CUtensorMap ma, mb;
  // one swizzle atom of K per row, 128 rows per box (B is loaded in 128-row boxes)
  const uint32_t box[2] = {kGemmKBytes, 128};
  const uint32_t box_b[2] = {kGemmKBytes, 128};
  const uint64_t da[2] = {kbytes, static_cast<uint64_t>(M)}, sa[1] = {kbytes};
  const uint64_t db[2] = {kbytes, static_cast<uint64_t>(N)}, sb[1] = {kbytes};
  if (!encode_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, A, da, sa, box, gemm_swizzle()) ||
      !encode_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, B, db, sb, box_b, gemm_swizzle()))
    return MX8_ERR_CUDA;
  CUtensorMap mc;
  if (!encode_output_map(&mc, C, M, N, ldc, out_dtype)) return MX8_ERR_CUDA;
  GemmArgs a{};
  a.fmt = fmt; a.M = M; a.N = N; a.K = K;
  a.SA = SA; a.SB = SB; a.A32 = A32; a.a32_mode = a32_mode; a.B32 = B32; a.b32_mode = b32_mode;
  a.C = C; a.ldc = ldc; a.out_bf16 = out_dtype == MX8_OUT_BF16; a.accumulate = accumulate;
  a.grouped = 0; a.G = 1; a.offs = nullptr; a.err = err_word(workspace);
  return from_cuda(launch_bs_gemm(a, ma, mb, mc, sm_count_current(), s));
}

extern "C" mx8_status bs_grouped_gemm(int fmt, int num_groups, const int64_t* group_offsets,
                                      int64_t total_rows, int64_t N, int64_t K, const uint8_t* A,
                                      const uint8_t* SA, const float* A32, const uint8_t* B,
                                      const uint8_t* SB, const float* B32, int out_dtype, void* C,
                                      int64_t ldc, void* workspace, size_t workspace_bytes,
                                      mx8_stream_t stream) {
  if (num_groups < 1 || num_groups > kMaxGroups || group_offsets == nullptr || total_rows < 0)
    return MX8_ERR_INVALID_ARG;
  if (total_rows == 0 || N == 0) return MX8_OK;
  mx8_status st = gemm_common_checks(fmt, N, K, A, SA, B, SB, out_dtype, C, ldc);
  if (st != MX8_OK) return st;
  if (total_rows > INT32_MAX || N > INT32_MAX) return MX8_ERR_UNSUPPORTED;
  st = check_ws(workspace, workspace_bytes, num_groups);
  if (st != MX8_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return from_cuda(zero_output(C, ldc, total_rows, N, out_dtype, s));

  const uint64_t kbytes = fmt == MX8_FMT_MXFP8 ? K : K / 2;
  CUtensorMap ma, mb;
  const uint32_t box2[2] = {kGemmKBytes, 128};
  const uint64_t da[2] = {kbytes, static_cast<uint64_t>(total_rows)}, sa[1] = {kbytes};
  const uint32_t box3[3] = {kGemmKBytes, 128, 1};
  const uint64_t db[3] = {kbytes, static_cast<uint64_t>(N), static_cast<uint64_t>(num_groups)};
  const uint64_t sb[2] = {kbytes, kbytes * static_cast<uint64_t>(N)};
  if (!encode_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, A, da, sa, box2, gemm_swizzle()) ||
      !encode_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, B, db, sb, box3, gemm_swizzle()))
    return MX8_ERR_CUDA;
  CUtensorMap mc;
  if (!encode_output_map(&mc, C, total_rows, N, ldc, out_dtype)) return MX8_ERR_CUDA;
  GemmArgs a{};
  a.fmt = fmt; a.M = total_rows; a.N = N; a.K = K;
  a.SA = SA; a.SB = SB; a.A32 = A32; a.a32_mode = A32 ? MX8_S32_ROW : MX8_S32_NONE;
  a.B32 = B32; a.b32_mode = B32 ? MX8_S32_GROUP : MX8_S32_NONE;
  a.C = C; a.ldc = ldc; a.out_bf16 = out_dtype == MX8_OUT_BF16; a.accumulate = 0;
  a.grouped = 1; a.G = num_groups; a.offs = group_offsets; a.err = err_word(workspace);
  return from_cuda(launch_bs_gemm(a, ma, mb, mc, sm_count_current(), s));
}

// ===================================================================== fused MoE GEMM
extern "C" mx8_status bs_grouped_gemm_fused(int fmt, int num_groups, const int64_t* group_offsets,
                                            int64_t total_rows, int64_t N, int64_t K, const uint8_t* A,
                                            const uint8_t* SA, const float* A32, const int64_t* a_rows,
                                            int64_t a_src_rows, const uint8_t* B, const uint8_t* SB,
                                            const float* B32, int epilogue, int out_dtype, void* C,
                                            int64_t ldc, void* workspace, size_t workspace_bytes,
                                            mx8_stream_t stream) {
  if (num_groups < 1 || num_groups > kMaxGroups || group_offsets == nullptr || total_rows < 0)
    return MX8_ERR_INVALID_ARG;
  if (epilogue != MX8_EPI_NONE && epilogue != MX8_EPI_SWIGLU) return MX8_ERR_INVALID_ARG;
  const bool swiglu = epilogue == MX8_EPI_SWIGLU;
  if (swiglu && (N % 256 != 0 || out_dtype != MX8_OUT_BF16)) return MX8_ERR_INVALID_ARG;
  const int64_t n_out = swiglu ? N / 2 : N;
  if (a_rows != nullptr && (a_src_rows < 1 || a_src_rows > INT32_MAX)) return MX8_ERR_INVALID_ARG;
  if (total_rows == 0 || N == 0) return MX8_OK;
  mx8_status st = gemm_common_checks(fmt, n_out, K, A, SA, B, SB, out_dtype, C, ldc);
  if (st != MX8_OK) return st;
  if (fmt != MX8_FMT_NVFP4) return MX8_ERR_UNSUPPORTED;
  if (total_rows > INT32_MAX || N > INT32_MAX) return MX8_ERR_UNSUPPORTED;
  st = check_ws(workspace, workspace_bytes, num_groups);
  if (st != MX8_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return from_cuda(zero_output(C, ldc, total_rows, n_out, out_dtype, s));

  const uint64_t kbytes = K / 2;
  const uint64_t a_rows_map = a_rows != nullptr ? static_cast<uint64_t>(a_src_rows) : static_cast<uint64_t>(total_rows);
  CUtensorMap ma, mb, mc;
  const uint32_t box2[2] = {kGemmKBytes, 128};
  const uint64_t da[2] = {kbytes, a_rows_map}, sa[1] = {kbytes};
  const uint32_t box3[3] = {kGemmKBytes, 128, 1};
  const uint64_t db[3] = {kbytes, static_cast<uint64_t>(N), static_cast<uint64_t>(num_groups)};
  const uint64_t sb[2] = {kbytes, kbytes * static_cast<uint64_t>(N)};
  if (!encode_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, A, da, sa, box2, gemm_swizzle()) ||
      !encode_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, B, db, sb, box3, gemm_swizzle()) ||
      !encode_output_map(&mc, C, total_rows, n_out, ldc, out_dtype))
    return MX8_ERR_CUDA;
  GemmArgs a{};
  a.fmt = fmt; a.M = total_rows; a.N = N; a.K = K;
  a.SA = SA; a.SB = SB; a.A32 = A32; a.a32_mode = A32 ? MX8_S32_ROW : MX8_S32_NONE;
  a.B32 = B32; a.b32_mode = B32 ? MX8_S32_GROUP : MX8_S32_NONE;
  a.C = C; a.ldc = ldc; a.out_bf16 = out_dtype == MX8_OUT_BF16; a.accumulate = 0;
  a.grouped = 1; a.G = num_groups; a.offs = group_offsets; a.err = err_word(workspace);
  a.A = A; a.a_rows = a_rows; a.a_src_rows = a_rows ? a_src_rows : 0; a.ffn = swiglu ? N / 2 : 0;
  return from_cuda(launch_bs_gemm(a, ma, mb, mc, sm_count_current(), s));
}

// ===================================================================== gate|up + SwiGLU + NVFP4 of h
extern "C" mx8_status bs_grouped_gemm_swiglu_nvfp4(int num_groups, const int64_t* group_offsets, int64_t total_rows,
                                                   int64_t N, int64_t K, const uint8_t* A, const uint8_t* SA,
                                                   const float* A32, const uint8_t* B, const uint8_t* SB,
                                                   const float* B32, uint8_t* q_h, uint8_t* s_h, float* s32_h,
                                                   void* h, int64_t ld_h, void* workspace, size_t workspace_bytes,
                                                   mx8_stream_t stream) {
  if (num_groups < 1 || num_groups > kMaxGroups || group_offsets == nullptr || total_rows < 0)
    return MX8_ERR_INVALID_ARG;
  if (N < 0 || N % 256 != 0) return MX8_ERR_INVALID_ARG;
  const int64_t F = N / 2;
  if (F / 128 > 8) return MX8_ERR_UNSUPPORTED;          // h tiles of a band = CTAs of one cluster
  if (h != nullptr && ld_h < F) return MX8_ERR_INVALID_ARG;
  if (total_rows == 0 || N == 0) return MX8_OK;
  if (K <= 0 || K % 32 != 0) return MX8_ERR_INVALID_ARG;
  if (A == nullptr || SA == nullptr || B == nullptr || SB == nullptr || q_h == nullptr || s_h == nullptr ||
      s32_h == nullptr)
    return MX8_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(SA) || !aligned16(B) || !aligned16(SB) || !aligned16(q_h) || !aligned16(s_h) ||
      (reinterpret_cast<uintptr_t>(s32_h) & 3u) != 0 || (h != nullptr && (!aligned16(h) || ld_h % 8 != 0)))
    return MX8_ERR_ALIGNMENT;
  if (total_rows > INT32_MAX || N > INT32_MAX) return MX8_ERR_UNSUPPORTED;
  mx8_status st = check_ws(workspace, workspace_bytes, num_groups);
  if (st != MX8_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint64_t kbytes = K / 2;
  CUtensorMap ma, mb, mc;
  const uint32_t box2[2] = {kGemmKBytes, 128};
  const uint64_t da[2] = {kbytes, static_cast<uint64_t>(total_rows)}, sa[1] = {kbytes};
  const uint32_t box3[3] = {kGemmKBytes, 128, 1};
  const uint64_t db[3] = {kbytes, static_cast<uint64_t>(N), static_cast<uint64_t>(num_groups)};
  const uint64_t sb[2] = {kbytes, kbytes * static_cast<uint64_t>(N)};
  // the output map is not used by this epilogue (h leaves with plain stores);
  // it is encoded over h, or over the codes of h, so the kernel's tensor-map
  // prefetch sees a valid map
  const bool map_ok = h != nullptr ? encode_output_map(&mc, h, total_rows, F, ld_h, MX8_OUT_BF16)
                                   : encode_output_map(&mc, q_h, total_rows, F / 4, F / 4, MX8_OUT_BF16);
  if (!encode_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, A, da, sa, box2, gemm_swizzle()) ||
      !encode_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, B, db, sb, box3, gemm_swizzle()) || !map_ok)
    return MX8_ERR_CUDA;
  GemmArgs a{};
  a.fmt = MX8_FMT_NVFP4; a.M = total_rows; a.N = N; a.K = K;
  a.SA = SA; a.SB = SB; a.A32 = A32; a.a32_mode = A32 ? MX8_S32_ROW : MX8_S32_NONE;
  a.B32 = B32; a.b32_mode = B32 ? MX8_S32_GROUP : MX8_S32_NONE;
  a.C = h; a.ldc = h != nullptr ? ld_h : F; a.out_bf16 = 1; a.accumulate = 0;
  a.grouped = 1; a.G = num_groups; a.offs = group_offsets; a.err = err_word(workspace);
  a.A = A; a.a_rows = nullptr; a.a_src_rows = 0; a.ffn = F;
  a.qh = q_h; a.qh_scales = s_h; a.qh_s32 = s32_h;
  return from_cuda(launch_bs_gemm(a, ma, mb, mc, sm_count_current(), s));
}

// ===================================================================== BF16 GEMM
extern "C" mx8_status bf16_gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                const void* B, int64_t ldb, int out_dtype, void* C, int64_t ldc,
                                int accumulate, void* workspace, size_t workspace_bytes,
                                mx8_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return MX8_ERR_INVALID_ARG;
  if (out_dtype != MX8_OUT_F32 && out_dtype != MX8_OUT_BF16) return MX8_ERR_INVALID_ARG;
  if (K % 8 != 0 || lda < K || ldb < K || ldc < N) return MX8_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MX8_OK;
  if (A == nullptr || B == nullptr || C == nullptr) return MX8_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || lda % 8 != 0 || ldb % 8 != 0 || ldc % 8 != 0)
    return MX8_ERR_ALIGNMENT;
  if (accumulate && out_dtype != MX8_OUT_F32) return MX8_ERR_UNSUPPORTED;
  if (M > INT32_MAX || N > INT32_MAX) return MX8_ERR_UNSUPPORTED;
  mx8_status st = check_ws(workspace, workspace_bytes, 1);
  if (st != MX8_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return accumulate ? MX8_OK : from_cuda(zero_output(C, ldc, M, N, out_dtype, s));

  // the bf16 rows are moved as bytes: one swizzle atom (64 elements) of K per
  // row and stage, 128 rows per box
  CUtensorMap ma, mb, mc;
  const uint32_t box[2] = {kGemmKBytes, 128};
  const uint64_t da[2] = {static_cast<uint64_t>(2 * K), static_cast<uint64_t>(M)};
  const uint64_t sa[1] = {static_cast<uint64_t>(2 * lda)};
  const uint64_t db[2] = {static_cast<uint64_t>(2 * K), static_cast<uint64_t>(N)};
  const uint64_t sb[1] = {static_cast<uint64_t>(2 * ldb)};
  if (!encode_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, A, da, sa, box, gemm_swizzle()) ||
      !encode_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, B, db, sb, box, gemm_swizzle()) ||
      !encode_output_map(&mc, C, M, N, ldc, out_dtype))
    return MX8_ERR_CUDA;
  GemmArgs a{};
  a.fmt = 3; a.M = M; a.N = N; a.K = K;
  a.a32_mode = MX8_S32_NONE; a.b32_mode = MX8_S32_NONE;
  a.C = C; a.ldc = ldc; a.out_bf16 = out_dtype == MX8_OUT_BF16; a.accumulate = accumulate;
  a.grouped = 0; a.G = 1; a.offs = nullptr; a.err = err_word(workspace);
  return from_cuda(launch_bs_gemm(a, ma, mb, mc, sm_count_current(), s));
}

// ===================================================================== errors
extern "C" mx8_status mx8_check_device_error(void* workspace, mx8_stream_t stream) {
  if (workspace == nullptr) return MX8_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MX8_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MX8_ERR_CUDA;
  if (word == 0) return MX8_OK;
  if (cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return MX8_ERR_CUDA;
  return MX8_ERR_TIMEOUT;
}

namespace mx8q {
namespace {
// One block waits on a barrier that no thread will ever complete.
__global__ void selftest_wait_kernel(int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, err, kErrWaitSelftest, &abort, limit_ns);
}
}  // namespace

cudaError_t launch_selftest_wait(int* err, uint64_t limit_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}
}  // namespace mx8q

extern "C" mx8_status mx8_selftest_bounded_wait(void* workspace, uint64_t limit_ns, mx8_stream_t stream) {
  if (workspace == nullptr || !aligned16(workspace)) return MX8_ERR_WORKSPACE;
  if (limit_ns == 0 || limit_ns > 2000000000ull) return MX8_ERR_INVALID_ARG;
  return from_cuda(launch_selftest_wait(err_word(workspace), limit_ns,
                                        reinterpret_cast<cudaStream_t>(stream)));
}
