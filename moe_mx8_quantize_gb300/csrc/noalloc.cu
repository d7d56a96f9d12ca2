// Allocation-free variant of the NVFP4 quantizer entry point.
//
// Some callers cannot allocate device memory at all: code that runs inside a
// host that owns every allocation (a plugin or a serving runtime with its own
// arena), or code called where an allocation would be unsafe or forbidden.
// They cannot pass the workspace that nvfp4_quantize_per_token() needs for the
// per-group / per-tensor amax of its first pass.  This entry point instead
// keeps that scratch in a fixed array inside the library itself.
//
// The array lives in device memory for as long as the library is loaded, on
// every GPU that loads it: two words per group for up to kNoAllocMaxGroups
// groups plus a counter and an error word (about 8 KB).  Its device
// address is looked up once per device, on the first call made with that
// device current; make that first call before capturing any stream.  The
// address is kept for the life of the process, so neither entry point may be
// used on a device after cudaDeviceReset() (the module, and with it the
// array, is loaded again at a new address).  Every call shares the one
// array: its scratch words are cleared at the start of each call, and calls
// that overlap on the GPU (different streams, or different host threads
// without ordering) race on it and must be serialised.
//
// A bounded device wait that runs out (see the workspace entry points)
// records its code in the array's error word; calls do not clear that word,
// so nvfp4_noalloc_check_error() reports a timeout of any call made since it
// was last called, and clears it.
#include <mutex>

#include "mx8q.h"
#include "kernels.h"

namespace {

constexpr int kNoAllocMaxGroups = 1024;   // groups the library's scratch can serve
constexpr int kNoAllocWords = 2 * kNoAllocMaxGroups + 8;   // amax, counts, ticket, error word

static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocWords];

std::mutex g_lock;
uint32_t* g_scratch_addr[64] = {nullptr};   // device address of the array, per device

// Device address of the array on the current device (looked up once).
cudaError_t scratch_address(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> guard(g_lock);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

extern "C" mx8_status nvfp4_quantize_per_token_noalloc(const void* x, int64_t rows, int64_t cols,
                                                       int64_t ld, int scope,
                                                       const int64_t* group_offsets, int num_groups,
                                                       uint8_t* q, uint8_t* s_blk, float* s32,
                                                       mx8_stream_t stream) {
  if (scope < NVFP4_SCOPE_TOKEN || scope > NVFP4_SCOPE_TENSOR) return MX8_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || ld < cols || cols % 16 != 0) return MX8_ERR_INVALID_ARG;
  if (cols > (int64_t{1} << 30)) return MX8_ERR_UNSUPPORTED;   // columns are 32-bit in the kernels
  if (scope == NVFP4_SCOPE_GROUP && group_offsets == nullptr) return MX8_ERR_INVALID_ARG;
  // the library's scratch holds kNoAllocMaxGroups amax words: more groups are refused
  if (group_offsets != nullptr && (num_groups < 1 || num_groups > kNoAllocMaxGroups))
    return MX8_ERR_INVALID_ARG;
  const int G = group_offsets ? num_groups : 1;
  if (cols == 0) return MX8_OK;
  if (rows > 0 && (x == nullptr || q == nullptr)) return MX8_ERR_INVALID_ARG;
  if (s_blk == nullptr || s32 == nullptr) return MX8_ERR_INVALID_ARG;
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if ((rows > 0 && (misaligned(x) || misaligned(q))) || misaligned(s_blk) || ld % 8 != 0)
    return MX8_ERR_ALIGNMENT;
  uint32_t* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MX8_ERR_CUDA;
  // words 0 .. 2*groups+1 are the quantizer scratch; the error word sits after them
  static_assert(kNoAllocWords - 4 >= 2 * kNoAllocMaxGroups + 2, "scratch too small");
  int* err = reinterpret_cast<int*>(scratch + kNoAllocWords - 4);
  const cudaError_t e = mx8q::launch_nvfp4_quant(static_cast<const uint16_t*>(x), rows, cols, ld, scope,
                                                 group_offsets, G, q, s_blk, s32, scratch, err, sm_count(),
                                                 reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MX8_OK : MX8_ERR_CUDA;
}

extern "C" mx8_status nvfp4_noalloc_check_error(mx8_stream_t stream) {
  uint32_t* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MX8_ERR_CUDA;
  int* err = reinterpret_cast<int*>(scratch + kNoAllocWords - 4);
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MX8_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MX8_ERR_CUDA;
  if (word == 0) return MX8_OK;
  if (cudaMemset(err, 0, sizeof(int)) != cudaSuccess) return MX8_ERR_CUDA;
  return MX8_ERR_TIMEOUT;
}
