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
// approximate math; gate and up weights share one FP32 scale.  Section "Las
// Curvas de Recompensa...": running the per-token scale as a separate
// framework op is what slowed NVFP4 training.  "NVIDIA presenta una
// metodologia de preentrenamiento de 4 bits utilizando NVFP4", section "Que es
// realmente NVFP4": E4M3 block scales under an FP32 scale that keeps them in
// range; section "La metodologia...": 1x16 blocks, round-to-nearest-even.
//
// Arithmetic (all FP32, one IEEE round-to-nearest step each):
//   S_enc = min(2688 / A, FLT_MAX), S_dec = A / 2688      (A = scope amax)
//   sb    = RNE_E4M3_sat((amax_b / 6) * S_enc)
//   r     = sb ? min(S_enc / sb, FLT_MAX) : 0,   code = RNE_E2M1_sat(x * r)
//
// Layout of the work: one warp per row; lane l owns the 16-element block
// [512*i + 16*l, +16) of every 512-element chunk i, so each lane computes its
// block's scale once, loads are 32 contiguous bytes per lane and the 8-byte
// code stores of a warp are contiguous.  |x| maxima are taken two bf16 values
// per instruction (max of magnitudes), the products x * r two per instruction
// (packed binary32 multiply).  Four lanes hold one 4-scale group of the
// tensor-core tile and write it as one 32-bit word.
//
// The two divisions of a block, amax_b / 6 and S_enc / sb, are computed as
// Markstein's FMA-corrected quotients (P. Markstein, "IA-64 and Elementary
// Functions", 2000; J.-M. Muller et al., "Handbook of Floating-Point
// Arithmetic", the theorem on correcting a quotient with one FMA): with
// y = RN(1/b) and q = RN(a y), the remainder a - b q is exact in one FMA and
// RN(q + (a - b q) y) = RN(a / b).  Both dividends come from bf16 maxima
// (amax_b, and S_enc = min(2688 / A, FLT_MAX) for a bf16 A), so the result
// was checked bit for bit against IEEE division over every finite bf16 value
// and every positive E4M3 divisor, the overflow cases included (they
// saturate to FLT_MAX through the min).  1/sb comes from a 128-entry table of
// {E4M3 value, RN(1/value)} per block.
//
// Token scope: rows of up to 512*kCh elements (4096) are held in registers,
// all loads issued up front, so the amax and the encode read HBM once.
// Longer rows (the 7168-wide DeepSeek-V3 activations) are read twice, four
// 512-value chunks in flight at a time, the second read served by L1/L2: at 4
// blocks per SM instead of 1 that measured faster (dispatch of 16384 x 7168
// tokens to 8 experts each: 407 -> 253 us).
//
// Group / tensor scope (one FP32 scale per expert weight or per tensor) needs
// the scope amax before any element is encoded.  A single kernel takes work
// items from an ordered ticket counter: "amax" items (16 rows; 32 for paired
// rows, 8 for rows over 2048 values: fold their
// maximum into the group's word, then count themselves done) and "encode"
// items (16 scale rows of the group: wait until all of the group's amax items
// are done, then encode).  Tickets hand out a lead of amax items first (about
// 32 MB of input, and at least the largest group), then encode and amax
// items alternately, so the DRAM reads of the amax items and the L2 reads
// of the encode items overlap throughout, and the second read of a group,
// about one lead later, is served from L2.  An encode item only waits on
// items with smaller tickets, which are already held by running blocks that
// never wait, so the order cannot deadlock; the wait is bounded anyway.
#include <float.h>

#include "device.cuh"
#include "groups.cuh"
#include "kernels.h"

namespace mx8q {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
// Rows (or scale rows) per work item of the scoped kernel: two per data warp
// (two pairs for the paired-row shapes; one for rows over 2048 values).
// Smaller items keep the data that the blocks hold between an amax item and
// its encode item -- about two items per block -- well inside L2 (measured:
// 16-row items read less from DRAM than 32-row ones; 8-row items cost more in
// ticket traffic.  For the 7168-wide DeepSeek-V3 gate|up expert weights, 8-row
// items (115 KB) read 1.72x the input from DRAM against 1.94x for 16 rows,
// 4958 -> 4286 us; 4-row items read 1.50x but cost more in tickets).
template <int kCh>
struct ScopedItem {
  static constexpr int kRows = kCh < 0 ? 32 : (kCh == 0 ? 8 : 16);
};
constexpr int64_t kL2LeadBytes = 32ll << 20;  // input bytes between a group's amax and encode items


__device__ __forceinline__ uint4 ld_nc(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// L2 eviction-priority policies: a first read whose data is read again soon
// keeps its lines (evict_last); the last read of data marks them evict_first.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_hint(const uint16_t* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

template <bool kHint>
__device__ __forceinline__ uint4 ld_row16(const uint16_t* p, uint64_t pol) {
  return kHint ? ld_hint(p, pol) : ld_nc(p);
}

// This lane's packed |x| maximum over its blocks of a row (sign bits not
// meaningful).  kCh > 0: the row has at most kCh 512-value chunks, all loads
// issued at once; kCh = 0: any length, 4 chunks in flight.  With kHint the
// loads carry the L2 policy `pol`.
template <int kCh, bool kHint = false>
__device__ __forceinline__ uint32_t row_absmax_lane(const uint16_t* __restrict__ xr, int C, int lane,
                                                    uint64_t pol = 0) {
  constexpr int kN = kCh > 0 ? kCh : 4;
  uint32_t m = 0;
  for (int base = 0; base < C; base += 512 * kN) {
    uint4 w[2 * kN];
#pragma unroll
    for (int i = 0; i < kN; ++i) {
      const int c = base + i * 512 + lane * 16;
      const bool ok = c < C;
      w[2 * i] = ok ? ld_row16<kHint>(xr + c, pol) : make_uint4(0, 0, 0, 0);
      w[2 * i + 1] = ok ? ld_row16<kHint>(xr + c + 8, pol) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kN; ++i) m = amax2(m, absmax16(w[2 * i], w[2 * i + 1]));
    if (kCh > 0) break;
  }
  return m;
}

// Where an encoded row goes: out.codes(byte offset, 8 bytes of codes),
// out.scale(4-block group k4, 32-bit scale word in the tensor-core tile
// layout) and out.sdec(S_dec) (lane 0).  RowOut writes one row; the
// before-dispatch quantizer writes a token to its dispatched copies.
struct RowOut {
  uint8_t* qr;        // the row's codes
  uint8_t* swr;       // its first scale word
  float* s32;         // its S_dec
  __device__ __forceinline__ void codes(int off, uint2 v) const { *reinterpret_cast<uint2*>(qr + off) = v; }
  __device__ __forceinline__ void scale(int k4, uint32_t w) const { *reinterpret_cast<uint32_t*>(swr + k4 * 512) = w; }
  __device__ __forceinline__ void sdec(float v) const { *s32 = v; }
};

// Encodes 512-element chunk j of a row: lane l encodes the 16-element block
// [512 j + 16 l, +16) held in (a, b); the 4 scales of a 4-block group are
// gathered by shuffles into one 32-bit word.
template <typename Out>
__device__ __forceinline__ void encode_chunk(const uint4& a, const uint4& b, int j, int C, int lane, float senc,
                                             const float2* __restrict__ tab, const Out& out, int kt) {
  const int c = j * 512 + lane * 16;
  uint2 cw;
  const uint32_t sb = nvfp4_encode_block(a, b, senc, tab, cw);
  if (c < C) out.codes(c >> 1, cw);
  const uint32_t s1 = __shfl_down_sync(0xffffffffu, sb, 1);
  const uint32_t s2 = __shfl_down_sync(0xffffffffu, sb, 2);
  const uint32_t s3 = __shfl_down_sync(0xffffffffu, sb, 3);
  const int k4 = j * 8 + (lane >> 2);
  if ((lane & 3) == 0 && k4 < kt) out.scale(k4, sb | (s1 << 8) | (s2 << 16) | (s3 << 24));
}

// Encodes data row `row` with scale S_enc (for scope_token the amax and
// S_dec come from the row itself) into out.
template <int kCh, bool kHint, typename Out>
__device__ __forceinline__ void encode_row(const uint16_t* __restrict__ x, int64_t row, int C, int64_t ld,
                                           bool scope_token, float senc_given, const float2* __restrict__ tab,
                                           const Out& out, int kt, int lane, uint64_t pol) {
  const uint16_t* xr = x + row * ld;
  if (kCh > 0) {
    const int nch = (C + 511) / 512;
    uint4 w[2 * (kCh > 0 ? kCh : 1)];
#pragma unroll
    for (int i = 0; i < kCh; ++i) {
      const int c = i * 512 + lane * 16;
      const bool ok = i < nch && c < C;
      w[2 * i] = ok ? ld_row16<kHint>(xr + c, pol) : make_uint4(0, 0, 0, 0);
      w[2 * i + 1] = ok ? ld_row16<kHint>(xr + c + 8, pol) : make_uint4(0, 0, 0, 0);
    }
    float senc = senc_given;
    if (scope_token) {
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < kCh; ++i) m = amax2(m, absmax16(w[2 * i], w[2 * i + 1]));
      float sdec;
      nvfp4_scales(warp_max(abs_halves_max(m)), senc, sdec);
      if (lane == 0) out.sdec(sdec);
    }
#pragma unroll
    for (int i = 0; i < kCh; ++i)
      if (i < nch) encode_chunk(w[2 * i], w[2 * i + 1], i, C, lane, senc, tab, out, kt);
  } else {
    float senc = senc_given;
    if (scope_token) {
      float sdec;
      nvfp4_scales(warp_max(abs_halves_max(row_absmax_lane<0, kHint>(xr, C, lane, pol))), senc, sdec);
      if (lane == 0) out.sdec(sdec);
    }
    // four chunks' loads in flight, then their encoding
    for (int j0 = 0; j0 * 512 < C; j0 += 4) {
      uint4 w[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = (j0 + i) * 512 + lane * 16;
        const bool ok = c < C;
        w[2 * i] = ok ? ld_row16<kHint>(xr + c, pol) : make_uint4(0, 0, 0, 0);
        w[2 * i + 1] = ok ? ld_row16<kHint>(xr + c + 8, pol) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if ((j0 + i) * 512 < C) encode_chunk(w[2 * i], w[2 * i + 1], j0 + i, C, lane, senc, tab, out, kt);
    }
  }
}

// Encodes data row `row` (or zeros scale row sr when row < 0) into scale row sr.
template <int kCh, bool kHint = false>
__device__ __forceinline__ void process_row(const uint16_t* __restrict__ x, int64_t row, int C, int64_t ld,
                                            bool scope_token, float senc_given, const float2* __restrict__ tab,
                                            uint8_t* __restrict__ q, uint8_t* __restrict__ sblk,
                                            float* __restrict__ s32, int64_t sr, int kt, int lane,
                                            uint64_t pol = 0) {
  uint8_t* swr = sblk + sf_row_base(sr, kt);
  if (row < 0) {  // padding row of the scale tile
    for (int k4 = lane; k4 < kt; k4 += 32) *reinterpret_cast<uint32_t*>(swr + k4 * 512) = 0u;
    return;
  }
  const RowOut out{q + row * (C / 2), swr, s32 + row};
  encode_row<kCh, kHint>(x, row, C, ld, scope_token, senc_given, tab, out, kt, lane, pol);
}

// ------------------------------------------------------------------ paired rows
// Rows of C = 256 or 768 elements fill 512-element chunks only partly (for
// 768, half the lanes of the second chunk would idle), so a warp takes two
// rows ra, rb as one virtual row of 2C = 512 kP elements: virtual block v is
// block v of ra for v < C/16, else block v - C/16 of rb.  A 4-block scale
// group never straddles the two rows (C/16 is a multiple of 4).  rb = -1 (or
// ra = -1) is a missing row: zeros in, codes not written, scale words zero.
struct PairOut {
  uint8_t* qa;        // codes of ra (nullptr: none)
  uint8_t* qb;
  uint8_t* swa;       // first scale word of ra's / rb's scale row
  uint8_t* swb;
  int half;           // code bytes per row, C / 2
  int g4;             // 4-block groups per row, C / 64
  __device__ __forceinline__ void codes(int off, uint2 v) const {
    if (off < half) {
      if (qa) *reinterpret_cast<uint2*>(qa + off) = v;
    } else if (qb) {
      *reinterpret_cast<uint2*>(qb + off - half) = v;
    }
  }
  __device__ __forceinline__ void scale(int k4, uint32_t w) const {
    if (k4 < g4) *reinterpret_cast<uint32_t*>(swa + k4 * 512) = w;
    else *reinterpret_cast<uint32_t*>(swb + (k4 - g4) * 512) = w;
  }
};

template <int kP, bool kHint>
__device__ __forceinline__ void load_pair(const uint16_t* __restrict__ x, int64_t ra, int64_t rb, int C, int64_t ld,
                                          int lane, uint64_t pol, uint4 (&w)[2 * kP]) {
#pragma unroll
  for (int i = 0; i < kP; ++i) {
    const int cv = i * 512 + lane * 16;
    const int64_t row = cv < C ? ra : rb;
    const int c = cv < C ? cv : cv - C;
    const uint16_t* p = x + row * ld + c;
    w[2 * i] = row >= 0 ? ld_row16<kHint>(p, pol) : make_uint4(0, 0, 0, 0);
    w[2 * i + 1] = row >= 0 ? ld_row16<kHint>(p + 8, pol) : make_uint4(0, 0, 0, 0);
  }
}

// This lane's packed |x| maximum over its blocks of the two rows together.
template <int kP, bool kHint>
__device__ __forceinline__ uint32_t pair_absmax_lane(const uint16_t* __restrict__ x, int64_t ra, int64_t rb, int C,
                                                     int64_t ld, int lane, uint64_t pol) {
  uint4 w[2 * kP];
  load_pair<kP, kHint>(x, ra, rb, C, ld, lane, pol, w);
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < kP; ++i) m = amax2(m, absmax16(w[2 * i], w[2 * i + 1]));
  return m;
}

// Encodes rows ra, rb (scale rows sra, srb); scope_token: each row's own amax
// gives its S_enc and S_dec, else both use senc_given.
template <int kP, bool kHint>
__device__ __forceinline__ void encode_pair(const uint16_t* __restrict__ x, int64_t ra, int64_t rb, int C, int64_t ld,
                                            bool scope_token, float senc_given, const float2* __restrict__ tab,
                                            uint8_t* __restrict__ q, uint8_t* __restrict__ sblk,
                                            float* __restrict__ s32, int64_t sra, int64_t srb, int kt, int lane,
                                            uint64_t pol) {
  uint4 w[2 * kP];
  load_pair<kP, kHint>(x, ra, rb, C, ld, lane, pol, w);
  float senc_a = senc_given, senc_b = senc_given;
  if (scope_token) {
    uint32_t ma = 0, mb = 0;
#pragma unroll
    for (int i = 0; i < kP; ++i) {
      const uint32_t m = absmax16(w[2 * i], w[2 * i + 1]);
      if (i * 512 + lane * 16 < C) ma = amax2(ma, m); else mb = amax2(mb, m);
    }
    float sdec_a, sdec_b;
    nvfp4_scales(warp_max(abs_halves_max(ma)), senc_a, sdec_a);
    nvfp4_scales(warp_max(abs_halves_max(mb)), senc_b, sdec_b);
    if (lane == 0) {
      if (ra >= 0) s32[ra] = sdec_a;
      if (rb >= 0) s32[rb] = sdec_b;
    }
  }
  const PairOut out{ra >= 0 ? q + ra * (C / 2) : nullptr, rb >= 0 ? q + rb * (C / 2) : nullptr,
                    sblk + sf_row_base(sra, kt), sblk + sf_row_base(srb, kt), C / 2, C / 64};
#pragma unroll
  for (int i = 0; i < kP; ++i)
    encode_chunk(w[2 * i], w[2 * i + 1], i, 2 * C, lane, i * 512 + lane * 16 < C ? senc_a : senc_b, tab, out, C / 32);
}

// Data row behind scale row sr (-1 for padding).
__device__ __forceinline__ int64_t data_row(const GroupSmem& gs, bool grouped, int G, int64_t R, int64_t sr) {
  if (!grouped) return sr < R ? sr : -1;
  const int g = upper_group(gs.pref, G, sr);
  const int64_t local = sr - gs.pref[g];
  return local < gs.offs[g + 1] - gs.offs[g] ? gs.offs[g] + local : -1;
}

// ------------------------------------------------------------------ token scope
template <int kCh>
__global__ void __launch_bounds__(kThreads, kCh >= 8 ? 1 : 4) nvfp4_token_kernel(
    const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ld, const int64_t* __restrict__ offs, int G,
    uint8_t* __restrict__ q, uint8_t* __restrict__ sblk, float* __restrict__ s32,
    const uint32_t* __restrict__ tensor_amax) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GroupSmem& gs = *reinterpret_cast<GroupSmem*>(smem_raw);
  __shared__ float2 tab[128];
  nvfp4_init_scale_table(tab);
  __syncthreads();
  const bool grouped = offs != nullptr;
  int64_t TP;
  if (grouped) {
    load_group_prefix(gs, offs, G);
    TP = gs.pref[G];
  } else {
    TP = (R + 127) / 128 * 128;
  }
  const int lane = threadIdx.x & 31;
  const int C32 = static_cast<int>(C);
  const int kt = (C32 / 16 + 3) / 4;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  // tensor scope: the amax of the whole tensor comes from the amax launch
  const bool per_token = tensor_amax == nullptr;
  float senc = 0.f;
  if (!per_token) {
    float sdec;
    nvfp4_scales(__uint_as_float(*tensor_amax), senc, sdec);
    if (blockIdx.x == 0 && threadIdx.x == 0) s32[0] = sdec;
  }
  if constexpr (kCh < 0) {           // pairs of scale rows (TP is a multiple of 128)
    for (int64_t sp = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); 2 * sp < TP; sp += nwarps)
      encode_pair<-kCh, false>(x, data_row(gs, grouped, G, R, 2 * sp), data_row(gs, grouped, G, R, 2 * sp + 1), C32,
                               ld, per_token, senc, tab, q, sblk, s32, 2 * sp, 2 * sp + 1, kt, lane, 0);
  } else {
    for (int64_t sr = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); sr < TP; sr += nwarps)
      process_row<kCh>(x, data_row(gs, grouped, G, R, sr), C32, ld, per_token, senc, tab, q, sblk, s32, sr, kt,
                       lane);
  }
}

// ------------------------------------------------------------------ token scope, before dispatch
// Each token is encoded once; its copies are the dispatched rows
// dest[t * topk + j] (grouped by the dispatch offsets).  The scale words go
// to the copies' scale rows in the grouped layout; the codes and S_dec go to
// the copies' rows too (disp_codes: a plain grouped GEMM reads them) or stay
// token-major (q [T, C/2], s32 [T]: the GEMM gathers the rows).  Per-token
// scaling makes this byte-identical to quantizing the dispatched rows.
struct DispatchOut {
  const int64_t* srow;   // [topk] scale rows of the copies (-1: skipped)
  const int64_t* drow;   // [topk] dispatched rows of the copies (-1: skipped)
  int n;
  bool disp_codes;
  int64_t token;
  int64_t c2;            // code bytes per row
  int kt;
  uint8_t* q;
  uint8_t* sblk;
  float* s32;
  __device__ __forceinline__ void codes(int off, uint2 v) const {
    if (!disp_codes) {
      *reinterpret_cast<uint2*>(q + token * c2 + off) = v;
      return;
    }
    for (int j = 0; j < n; ++j)
      if (drow[j] >= 0) *reinterpret_cast<uint2*>(q + drow[j] * c2 + off) = v;
  }
  __device__ __forceinline__ void scale(int k4, uint32_t w) const {
    for (int j = 0; j < n; ++j)
      if (srow[j] >= 0) *reinterpret_cast<uint32_t*>(sblk + sf_row_base(srow[j], kt) + k4 * 512) = w;
  }
  __device__ __forceinline__ void sdec(float v) const {
    if (!disp_codes) {
      s32[token] = v;
      return;
    }
    for (int j = 0; j < n; ++j)
      if (drow[j] >= 0) s32[drow[j]] = v;
  }
};

// Warps first take the T tokens, then the scale rows, zeroing the padding
// rows of each group's last tile.
template <int kCh>
__global__ void __launch_bounds__(kThreads, kCh >= 8 ? 1 : 4) nvfp4_dispatch_kernel(
    const uint16_t* __restrict__ x, int64_t T, int64_t C, int64_t ld, const int64_t* __restrict__ dest,
    int topk, const int64_t* __restrict__ offs, int G, int disp_codes, uint8_t* __restrict__ q,
    uint8_t* __restrict__ sblk, float* __restrict__ s32) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GroupSmem& gs = *reinterpret_cast<GroupSmem*>(smem_raw);
  __shared__ float2 tab[128];
  __shared__ int64_t dsr[kWarps][kMaxTopk];          // copies' scale rows ...
  __shared__ int64_t ddr[kWarps][kMaxTopk];          // ... and dispatched rows, for a warp's token
  nvfp4_init_scale_table(tab);
  __syncthreads();
  load_group_prefix(gs, offs, G);
  const int64_t R = gs.offs[G], TP = gs.pref[G];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int C32 = static_cast<int>(C);
  const int kt = (C32 / 16 + 3) / 4;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * kWarps + wl; u < T + TP; u += nwarps) {
    if (u < T) {
      if (lane < topk) {
        int64_t dr = dest[u * topk + lane];
        int64_t sr = -1;                              // rows outside [0, R) are skipped
        if (dr >= 0 && dr < R) {
          const int g = upper_group(gs.offs, G, dr);
          sr = gs.pref[g] + (dr - gs.offs[g]);
        } else {
          dr = -1;
        }
        dsr[wl][lane] = sr;
        ddr[wl][lane] = dr;
      }
      __syncwarp();
      const DispatchOut out{dsr[wl], ddr[wl], topk, disp_codes != 0, u, C / 2, kt, q, sblk, s32};
      encode_row<kCh, false>(x, u, C32, ld, true, 0.f, tab, out, kt, lane, 0);
      __syncwarp();
    } else {
      const int64_t sr = u - T;
      if (data_row(gs, true, G, R, sr) < 0) process_row<kCh>(x, -1, C32, ld, true, 0.f, tab, q, sblk, s32, sr, kt, lane);
    }
  }
}

// ------------------------------------------------------------------ group / tensor scope
// Scratch words (zeroed before launch): amax bits [Gp], done counts [Gp],
// then a 64-bit ticket counter; Gp = scope groups rounded up to even.
__host__ __device__ __forceinline__ int scratch_gp(int groups) { return (groups + 1) / 2 * 2; }

// Block of the scoped kernel: warp 0 is the control warp (tickets, the amax
// hand-off between blocks, dependency checks), warps 1..kDataWarps move data.
// The control warp's latencies (the ticket atomic, the release of an amax
// item's maximum, the check that a group's amax is complete) overlap the
// data warps' work on the current item instead of stalling the block.
constexpr int kDataWarps = 8;
constexpr int kScopedThreads = 32 * (kDataWarps + 1);

struct ScopedSmem {
  GroupSmem gs;                       // scale-layout groups (or one group)
  int64_t toffs[2];                   // tensor scope: data rows [0, R) ...
  int64_t tpref[2];                   // ... and scale rows [0, TP)
  int32_t ca[kMaxGroups + 1];         // amax items of the scope groups before group g
  int32_t ce[kMaxGroups + 1];         // encode items of the scope groups before group g
  int32_t lead;                       // amax items handed out before the first encode item
  float2 tab[128];
  // Two ticket slots, used by alternate work items: the control warp fills
  // the next item's slot while the data warps run the current one.
  int64_t tk[2];
  int64_t titem[2];                   // item index within its scope group
  int32_t tg[2];                      // scope group
  int32_t tenc[2];                    // 1 = encode item
  int32_t tready[2];                  // encode item whose group amax is known
  float tsenc[2];                     // ... and its S_enc
  float red[2][kDataWarps];           // amax items: per-warp maxima
  uint64_t filled[2];                 // slot holds a new item (control lane arrives)
  uint64_t consumed[2];               // every data warp finished the slot's item
};

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Ordering of the work items and the deadlock argument.  Tickets are taken in
// order from one counter.  The amax items of a group all precede the group's
// encode items in ticket order.  A data warp waits only for its own control
// lane to fill the next slot.  The control lane releases a slot's amax item
// as soon as the data warps have finished it.  It only blocks on other blocks
// in the rare case of an encode item whose group amax was not complete when
// its ticket was taken, and before that it releases the one amax item the
// block may still hold.  So every amax item taken is released once its block
// finishes it, whatever the other blocks wait for.  Every wait is bounded
// anyway (error word on timeout).
// (Row pairs, kCh < 0: 3 blocks per SM leave the compiler registers to keep
// a pair's loads in flight; measured 133 -> 127 us on the 128 x 2048 x 768
// Qwen3 down-projection weights.  With whole rows, 4 blocks measured faster.)
template <int kCh>
__global__ void __launch_bounds__(kScopedThreads, kCh >= 8 ? 1 : (kCh < 0 ? 3 : 4)) nvfp4_scoped_kernel(
    const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ld, int scope,
    const int64_t* __restrict__ offs, int G, uint8_t* __restrict__ q, uint8_t* __restrict__ sblk,
    float* __restrict__ s32, uint32_t* __restrict__ scratch, int* err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ScopedSmem& sm = *reinterpret_cast<ScopedSmem*>(smem_raw);
  constexpr int kItemRows = ScopedItem<kCh>::kRows;
  const bool grouped = offs != nullptr;
  const int Gs = scope == 1 ? G : 1;                       // scope groups
  uint32_t* amax_bits = scratch;
  uint32_t* done = scratch + scratch_gp(Gs);
  unsigned long long* ticket = reinterpret_cast<unsigned long long*>(scratch + 2 * scratch_gp(Gs));

  nvfp4_init_scale_table(sm.tab);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.filled[i]), 1);
      mbar_init(smem_u32(&sm.consumed[i]), kDataWarps);
    }
    fence_barrier_init();
  }
  if (grouped) load_group_prefix(sm.gs, offs, G);
  __syncthreads();
  const int64_t TP = grouped ? sm.gs.pref[G] : (R + 127) / 128 * 128;
  // scope groups: data rows and padded scale rows
  const int64_t* aoffs = scope == 1 ? sm.gs.offs : sm.toffs;
  const int64_t* apref = scope == 1 ? sm.gs.pref : sm.tpref;
  if (threadIdx.x == 0) {
    sm.toffs[0] = 0; sm.toffs[1] = R; sm.tpref[0] = 0; sm.tpref[1] = TP;
  }
  __syncthreads();
  // Item counts per scope group -- amax items: ceil(rows / 32); encode items:
  // padded scale rows / 32 -- as exclusive prefix sums (warp 0), and the lead.
  if (threadIdx.x < 32) {
    const int lane0 = threadIdx.x;
    const int per = (Gs + 31) / 32, g0 = lane0 * per;
    int32_t la = 0, le = 0, mx = 0;
    for (int g = g0; g < g0 + per && g < Gs; ++g) {
      const int32_t a = static_cast<int32_t>((aoffs[g + 1] - aoffs[g] + kItemRows - 1) / kItemRows);
      la += a;
      le += static_cast<int32_t>((apref[g + 1] - apref[g]) / kItemRows);
      mx = a > mx ? a : mx;
    }
    int32_t ia = la, ie = le;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t oa = __shfl_up_sync(0xffffffffu, ia, d), oe = __shfl_up_sync(0xffffffffu, ie, d);
      if (lane0 >= d) {
        ia += oa;
        ie += oe;
      }
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    }
    int32_t ra = ia - la, re = ie - le;
    for (int g = g0; g < g0 + per && g < Gs; ++g) {
      sm.ca[g] = ra;
      sm.ce[g] = re;
      ra += static_cast<int32_t>((aoffs[g + 1] - aoffs[g] + kItemRows - 1) / kItemRows);
      re += static_cast<int32_t>((apref[g + 1] - apref[g]) / kItemRows);
    }
    if (lane0 == 31) {
      sm.ca[Gs] = ia;
      sm.ce[Gs] = ie;
      // about kL2LeadBytes of input between an amax item and the encode item
      // that reads the same rows again, and never less than the largest
      // group plus a quarter (no encode item waits for an amax item handed out
      // after it, and the last amax items of a group have some time to
      // finish before its first encode items are taken; measured on groups
      // larger than the lead, the quarter lowers the waits more than it
      // costs in L2 hits)
      const int64_t item_bytes = static_cast<int64_t>(kItemRows) * C * 2;
      int64_t lead = item_bytes > 0 ? (kL2LeadBytes + item_bytes - 1) / item_bytes : 0;
      if (lead < mx + mx / 4) lead = mx + mx / 4;
      if (lead > ia) lead = ia;
      sm.lead = static_cast<int32_t>(lead);
    }
  }
  __syncthreads();
  const int64_t NA = sm.ca[Gs], NE = sm.ce[Gs], LEAD = sm.lead;
  const int64_t total = NA + NE;
  // groups with no rows still get their (zero) decode scale
  if (blockIdx.x == 0)
    for (int g = threadIdx.x; g < Gs; g += blockDim.x)
      if (aoffs[g + 1] == aoffs[g]) s32[g] = 0.f;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C32 = static_cast<int>(C);
  const int kt = (C32 / 16 + 3) / 4;

  // ---- control-lane helpers (thread 0 only)
  auto amax_items = [&](int g) {
    return static_cast<uint32_t>((aoffs[g + 1] - aoffs[g] + kItemRows - 1) / kItemRows);
  };
  auto publish = [&](int slot, int g, int64_t item, float amax) {
    float senc, sdec;
    nvfp4_scales(amax, senc, sdec);
    sm.tsenc[slot] = senc;
    if (item == 0) s32[g] = sdec;
  };
  // Takes the next ticket into `slot`; for an encode item whose group amax is
  // already complete, also its S_enc (no waiting here).
  auto take = [&](int slot) {
    const int64_t t = static_cast<int64_t>(atomicAdd(ticket, 1ull));
    sm.tk[slot] = t;
    if (t >= total) return;
    // Ticket order: amax items 0 .. LEAD-1, then encode item j and amax item
    // LEAD + j alternately, then the encode items left.  Encode item j of
    // group g follows every amax item of g: the last has index < LEAD + j
    // (LEAD >= any group's amax items, and g's encode items start at or after
    // its amax items), so it was handed out before ticket LEAD + 2j.
    const int64_t P = NA - LEAD;
    int enc;
    int64_t k;
    if (t < LEAD) {
      enc = 0;
      k = t;
    } else if (t - LEAD < 2 * P) {
      const int64_t u = t - LEAD;
      enc = (u & 1) == 0;
      k = enc ? (u >> 1) : LEAD + (u >> 1);
    } else {
      enc = 1;
      k = P + (t - LEAD - 2 * P);
    }
    const int32_t* cum = enc ? sm.ce : sm.ca;
    int lo = 0, hi = Gs - 1;                   // the last group with cum[g] <= k
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cum[mid] <= k) lo = mid; else hi = mid - 1;
    }
    const int g = lo;
    // A group's encode items run in the reverse order of its amax items: the
    // rows read last for the amax are read again first, while still in L2
    // (a group larger than L2 -- 58.7 MB for a DeepSeek-V3 gate|up expert --
    // otherwise misses L2 on every row of its second read).
    const int64_t item = enc ? (cum[g + 1] - cum[g]) - 1 - (k - cum[g]) : k - cum[g];
    sm.tg[slot] = g;
    sm.tenc[slot] = enc;
    sm.titem[slot] = item;
    sm.tready[slot] = 0;
    if (enc && ld_acquire_u32(done + g) >= amax_items(g)) {
      publish(slot, g, item, __uint_as_float(ld_relaxed_u32(amax_bits + g)));
      sm.tready[slot] = 1;
    }
  };
  // Folds a finished amax item's maximum into its group, then counts it done
  // (the fence orders the two for the encode side's acquire load).
  auto release = [&](int g, int rslot) {
    float m = sm.red[rslot][0];
#pragma unroll
    for (int i = 1; i < kDataWarps; ++i) m = fmaxf(m, sm.red[rslot][i]);
    atomicMax(amax_bits + g, __float_as_uint(m));
    __threadfence();
    atomicAdd(done + g, 1u);
  };

  const uint64_t keep = policy_evict_last();    // first read: to be read again
  const uint64_t drop = policy_evict_first();   // second read: last use

  // Items alternate between two slots.  The control lane fills a slot
  // (filled[slot]); the data warps each take their share and report
  // (consumed[slot]); the control lane then releases the slot's amax item, if
  // it was one, and refills the slot two items ahead.  No block-wide barrier:
  // a data warp moves on to the next item as soon as its own share is done.
  if (warp == 0) {
    if (lane == 0) {
      bool rel[2] = {false, false};   // slot's amax item already released
      // For an encode item whose group amax was not complete when its ticket
      // was taken: release the other slot's amax item first (it is being worked
      // on, and the data warps never wait on other blocks), then wait.
      auto resolve = [&](int slot, int other_it) {
        const int other = slot ^ 1;
        if (other_it >= 0 && sm.tk[other] < total && !sm.tenc[other] && !rel[other]) {
          mbar_wait(smem_u32(&sm.consumed[other]), (other_it >> 1) & 1, err, kErrWaitConsumer, nullptr);
          release(sm.tg[other], other);
          rel[other] = true;
        }
        const int g = sm.tg[slot];
        const uint32_t need = amax_items(g);
        if (ld_acquire_u32(done + g) < need) {
          const uint64_t t0 = globaltimer();
          while (ld_acquire_u32(done + g) < need) {
            if (globaltimer() - t0 > kWaitLimitNs) {
              atomicCAS(err, 0, kErrWaitConsumer);
              break;
            }
            __nanosleep(64);
          }
        }
        publish(slot, g, sm.titem[slot], __uint_as_float(ld_relaxed_u32(amax_bits + g)));
      };
      auto fill = [&](int slot, int other_it) {
        take(slot);
        if (sm.tk[slot] < total && sm.tenc[slot] && !sm.tready[slot]) resolve(slot, other_it);
        mbar_arrive(smem_u32(&sm.filled[slot]));
      };
      fill(0, -1);
      fill(1, 0);
      for (int it = 0;; ++it) {
        const int slot = it & 1;
        if (sm.tk[slot] >= total) break;
        mbar_wait(smem_u32(&sm.consumed[slot]), (it >> 1) & 1, err, kErrWaitConsumer, nullptr);
        if (!sm.tenc[slot] && !rel[slot]) release(sm.tg[slot], slot);
        rel[slot] = false;
        fill(slot, it + 1);
      }
    }
  } else {
    const int dw = warp - 1;
    for (int it = 0;; ++it) {
      const int slot = it & 1;
      if (!mbar_wait(smem_u32(&sm.filled[slot]), (it >> 1) & 1, err, kErrWaitConsumer, nullptr)) break;
      if (sm.tk[slot] >= total) break;
      const int g = sm.tg[slot];
      const int64_t item = sm.titem[slot];
      if (!sm.tenc[slot]) {
        // ---- amax item: rows [aoffs[g] + 32 item, +32) of scope group g
        const int64_t r0 = aoffs[g] + item * kItemRows;
        const int64_t r1 = r0 + kItemRows < aoffs[g + 1] ? r0 + kItemRows : aoffs[g + 1];
        uint32_t m = 0;
        if constexpr (kCh < 0) {
          for (int64_t row = r0 + 2 * dw; row < r1; row += 2 * kDataWarps)
            m = amax2(m, pair_absmax_lane<-kCh, true>(x, row, row + 1 < r1 ? row + 1 : -1, C32, ld, lane, keep));
        } else {
          for (int64_t row = r0 + dw; row < r1; row += kDataWarps)
            m = amax2(m, row_absmax_lane<kCh, true>(x + row * ld, C32, lane, keep));
        }
        const float wm = warp_max(abs_halves_max(m));
        if (lane == 0) sm.red[slot][dw] = wm;
      } else {
        // ---- encode item: scale rows [apref[g] + 32 item, +32) of scope group g
        const float senc = sm.tsenc[slot];
        const int64_t s0 = apref[g] + item * kItemRows;
        const int64_t grows = aoffs[g + 1] - aoffs[g];
        // scope groups are the layout groups: the data row follows directly
        auto row_of = [&](int64_t sr) -> int64_t {
          const int64_t local = sr - apref[g];
          return scope == 1 ? (local < grows ? aoffs[g] + local : -1) : data_row(sm.gs, grouped, G, R, sr);
        };
        if constexpr (kCh < 0) {
          for (int64_t sr = s0 + 2 * dw; sr < s0 + kItemRows; sr += 2 * kDataWarps)
            encode_pair<-kCh, true>(x, row_of(sr), row_of(sr + 1), C32, ld, false, senc, sm.tab, q, sblk, s32, sr,
                                    sr + 1, kt, lane, drop);
        } else {
          for (int64_t sr = s0 + dw; sr < s0 + kItemRows; sr += kDataWarps)
            process_row<kCh, true>(x, row_of(sr), C32, ld, false, senc, sm.tab, q, sblk, s32, sr, kt, lane, drop);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.consumed[slot]));
    }
  }
}

template <int kCh>
cudaError_t launch_dispatch(unsigned grid, cudaStream_t stream, const uint16_t* x, int64_t T, int64_t C,
                            int64_t ld, const int64_t* dest, int topk, const int64_t* offs, int G, int disp_codes,
                            uint8_t* q, uint8_t* sblk, float* s32) {
  auto k = nvfp4_dispatch_kernel<kCh>;
  const size_t smem = sizeof(GroupSmem);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, smem, stream>>>(x, T, C, ld, dest, topk, offs, G, disp_codes, q, sblk, s32);
  return cudaGetLastError();
}

template <int kCh>
cudaError_t launch_token(unsigned grid, size_t smem, cudaStream_t stream, const uint16_t* x, int64_t R,
                         int64_t C, int64_t ld, const int64_t* offs, int G, uint8_t* q, uint8_t* sblk,
                         float* s32, const uint32_t* tensor_amax) {
  auto k = nvfp4_token_kernel<kCh>;
  if (smem > 0) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  k<<<grid, kThreads, smem, stream>>>(x, R, C, ld, offs, G, q, sblk, s32, tensor_amax);
  return cudaGetLastError();
}

template <int kCh>
cudaError_t launch_scoped(int sm_count, cudaStream_t stream, const uint16_t* x, int64_t R, int64_t C,
                          int64_t ld, int scope, const int64_t* offs, int G, uint8_t* q, uint8_t* sblk,
                          float* s32, uint32_t* scratch, int* err) {
  auto k = nvfp4_scoped_kernel<kCh>;
  const size_t smem = sizeof(ScopedSmem);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kScopedThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  k<<<static_cast<unsigned>(sm_count * per_sm), kScopedThreads, smem, stream>>>(x, R, C, ld, scope, offs, G, q,
                                                                               sblk, s32, scratch, err);
  return cudaGetLastError();
}

}  // namespace

size_t nvfp4_scratch_bytes(int groups) {
  return (2 * static_cast<size_t>(scratch_gp(groups > 1 ? groups : 1)) + 2) * sizeof(uint32_t);
}

cudaError_t launch_nvfp4_quant(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int scope,
                               const int64_t* offs, int G, uint8_t* q, uint8_t* sblk, float* s32,
                               void* scratch, int* err, int sm_count, cudaStream_t stream) {
  const bool grouped = offs != nullptr;
  // tensor scope on a tensor that fits in L2: one abs-max launch, then the
  // token kernel encodes with the tensor's S_enc (its read of x hits L2);
  // larger tensors and group scope take the ticket kernel
  const uint32_t* tensor_amax = nullptr;
  if (scope == 2 && R * C * 2 <= (int64_t{64} << 20) && C % 8 == 0) {
    uint32_t* amax_word = static_cast<uint32_t*>(scratch);
    cudaError_t e = launch_absmax(x, R, C, ld, amax_word, sm_count, stream);
    if (e != cudaSuccess) return e;
    tensor_amax = amax_word;
    scope = 0;
  }
  if (scope != 0) {
    const int Gs = scope == 1 ? G : 1;
    cudaError_t e = cudaMemsetAsync(scratch, 0, nvfp4_scratch_bytes(Gs), stream);
    if (e != cudaSuccess) return e;
    uint32_t* sc = static_cast<uint32_t*>(scratch);
    if (C == 256) return launch_scoped<-1>(sm_count, stream, x, R, C, ld, scope, offs, G, q, sblk, s32, sc, err);
    if (C == 768) return launch_scoped<-3>(sm_count, stream, x, R, C, ld, scope, offs, G, q, sblk, s32, sc, err);
    if (C <= 1024) return launch_scoped<2>(sm_count, stream, x, R, C, ld, scope, offs, G, q, sblk, s32, sc, err);
    if (C <= 2048) return launch_scoped<4>(sm_count, stream, x, R, C, ld, scope, offs, G, q, sblk, s32, sc, err);
    return launch_scoped<0>(sm_count, stream, x, R, C, ld, scope, offs, G, q, sblk, s32, sc, err);
  }
  const int64_t tp_bound = grouped ? (R + 127 * static_cast<int64_t>(G) + 127) / 128 * 128
                                   : (R + 127) / 128 * 128;
  const int64_t want = (tp_bound + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (grid == 0) grid = 1;
  const size_t smem = grouped ? sizeof(GroupSmem) : 0;
  if (C == 256) return launch_token<-1>(grid, smem, stream, x, R, C, ld, offs, G, q, sblk, s32, tensor_amax);
  if (C == 768) return launch_token<-3>(grid, smem, stream, x, R, C, ld, offs, G, q, sblk, s32, tensor_amax);
  if (C <= 1024) return launch_token<2>(grid, smem, stream, x, R, C, ld, offs, G, q, sblk, s32, tensor_amax);
  if (C <= 2048) return launch_token<4>(grid, smem, stream, x, R, C, ld, offs, G, q, sblk, s32, tensor_amax);
  if (C <= 4096) return launch_token<8>(grid, smem, stream, x, R, C, ld, offs, G, q, sblk, s32, tensor_amax);
  return launch_token<0>(grid, smem, stream, x, R, C, ld, offs, G, q, sblk, s32, tensor_amax);
}

cudaError_t launch_nvfp4_dispatch(const uint16_t* x, int64_t T, int64_t C, int64_t ld, const int64_t* dest,
                                  int topk, const int64_t* offs, int G, int disp_codes, uint8_t* q, uint8_t* sblk,
                                  float* s32, int sm_count, cudaStream_t stream) {
  const int64_t units = T + (T * topk + 127 * static_cast<int64_t>(G) + 127) / 128 * 128;
  const int64_t want = (units + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (grid == 0) grid = 1;
  if (C <= 1024) return launch_dispatch<2>(grid, stream, x, T, C, ld, dest, topk, offs, G, disp_codes, q, sblk, s32);
  if (C <= 2048) return launch_dispatch<4>(grid, stream, x, T, C, ld, dest, topk, offs, G, disp_codes, q, sblk, s32);
  if (C <= 4096) return launch_dispatch<8>(grid, stream, x, T, C, ld, dest, topk, offs, G, disp_codes, q, sblk, s32);
  return launch_dispatch<0>(grid, stream, x, T, C, ld, dest, topk, offs, G, disp_codes, q, sblk, s32);
}

}  // namespace mx8q
