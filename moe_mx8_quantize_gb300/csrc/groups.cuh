// Device-side view of MoE group offsets: each group's rows start a fresh run
// of 128-row scale tiles, so its scale rows begin at the padded prefix
// P_g = sum_{h<g} ceil(n_h / 128) * 128.
#pragma once

#include <stdint.h>

#include "kernels.h"

namespace mx8q {

struct GroupSmem {
  int64_t offs[kMaxGroups + 1];   // group row offsets (copied from the caller)
  int64_t pref[kMaxGroups + 1];   // padded scale-row prefix P_g
};

// Fills gs from the device offsets: all threads copy, warp 0 scans.
__device__ inline void load_group_prefix(GroupSmem& gs, const int64_t* __restrict__ offs, int G) {
  for (int i = threadIdx.x; i <= G; i += blockDim.x) gs.offs[i] = offs[i];
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (G + 31) / 32;
    const int g0 = lane * per;
    int64_t local = 0;
    for (int g = g0; g < g0 + per && g < G; ++g) local += (gs.offs[g + 1] - gs.offs[g] + 127) / 128 * 128;
    int64_t incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int64_t run = incl - local;
    for (int g = g0; g < g0 + per && g < G; ++g) {
      gs.pref[g] = run;
      run += (gs.offs[g + 1] - gs.offs[g] + 127) / 128 * 128;
    }
    if (lane == 31) gs.pref[G] = incl;
  }
  __syncthreads();
}

// Compact table of the GEMMs (int32: their row counts are below 2^31):
// group row offsets and the 128-row tiles before each group, P_g / 128.
struct GroupTiles {
  int32_t offs[kMaxGroups + 1];
  int32_t tpref[kMaxGroups + 1];
};

__device__ inline void load_group_tiles(GroupTiles& gt, const int64_t* __restrict__ offs, int G) {
  for (int i = threadIdx.x; i <= G; i += blockDim.x) gt.offs[i] = static_cast<int32_t>(offs[i]);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (G + 31) / 32;
    const int g0 = lane * per;
    int32_t local = 0;
    for (int g = g0; g < g0 + per && g < G; ++g) local += (gt.offs[g + 1] - gt.offs[g] + 127) / 128;
    int32_t incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int32_t run = incl - local;
    for (int g = g0; g < g0 + per && g < G; ++g) {
      gt.tpref[g] = run;
      run += (gt.offs[g + 1] - gt.offs[g] + 127) / 128;
    }
    if (lane == 31) gt.tpref[G] = incl;
  }
  __syncthreads();
}

// The last g in [0, G) with a[g] <= v (a non-decreasing, a[0] <= v).
template <typename T>
__device__ __forceinline__ int upper_group(const T* a, int G, int64_t v) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= v) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace mx8q
