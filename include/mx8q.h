/*
 * mx8q -- microscaling quantization (MXFP8, per-token NVFP4, MXFP4), the
 * block-scaled tensor-core GEMM it feeds and the BF16 GEMM of the
 * dequantized-backward mode, for GB300 (sm_103a).
 *
 * Plain C ABI: device pointers, sizes and a CUDA stream; no framework types.
 *
 * Sources (page title -- section):
 *   [MRL] "Miles Blackwell RL Cambia la Uniformidad BF16 por MXFP8 y NVFP4
 *         Nativos" -- "La Compatibilidad de Miles Blackwell Ahora Abarca Todo
 *         el Ciclo de RL" (MXFP8 = 32 E4M3 values sharing one E8M0 scale,
 *         used by rollout, Fprop, Wgrad and Dgrad; NVFP4 = E2M1 with an E4M3
 *         scale per 16 values plus an FP32 scale computed per token; the
 *         dequantized-backward mode), and "Un Cuantizador Compartido Es el
 *         Mecanismo Real" (rowwise and columnwise copies made from the
 *         high-precision input; scale blocks along the reduction dimension;
 *         the FP32 token scale fused into the activation quantizer; gate and
 *         up projections quantized together).
 *   [NV4] "NVIDIA presenta una metodologia de preentrenamiento de 4 bits
 *         utilizando NVFP4" -- "Que es realmente NVFP4" (E2M1 grid, E4M3
 *         block scales, FP32 second-level scale; MXFP4 = 32 E2M1 values
 *         under one power-of-two scale), "La metodologia de
 *         formacion de cuatro partes" (1x16 blocks, round-to-nearest-even).
 *   [REC] "Miles Blackwell MXFP8 / NVFP4 RL recipes" (aib.vote) -- MXFP8
 *         row/column copies, NVFP4 on MoE routed experts with a tensor- or
 *         token-scope FP32 scale, the bit-exact quantizer contract.
 *
 * Numerical convention (bit-exact; the pages leave these points open):
 *   MXFP8 block exponent e = smallest integer with amax <= 448 * 2^e,
 *   clamped to [-127, 127]; scale byte = e + 127; element = RNE_E4M3(x*2^-e)
 *   saturating, signed zero kept.
 *   MXFP4: the same rule with 6 for 448 and RNE_E2M1 for RNE_E4M3.
 *   NVFP4 with scope amax A:  S_enc = min(RN(2688/A), FLT_MAX);
 *   S_dec = RN(A/2688) (stored); per 16-block: sb = RNE_E4M3(RN(RN(amax_b/6)
 *   * S_enc)); r = sb ? min(RN(S_enc/sb), FLT_MAX) : 0;
 *   element = RNE_E2M1(RN(x*r)) saturating.  All FP32, IEEE round-to-nearest
 *   (no approximate division, as the FP4 quantizer contract in [MRL] asks).
 *
 * Data layouts (all row-major, every buffer allocated and owned by the
 * caller; the library never allocates device memory):
 *   bf16 input x          : [rows, cols] with row stride ld elements.
 *   MXFP8 data            : uint8 E4M3 [rows, cols].
 *   MXFP8 columnwise data : uint8 E4M3 [cols, rows] -- stored transposed, so
 *                           its 1x32 blocks run along its contiguous axis.
 *   NVFP4 / MXFP4 data    : uint8 [rows, cols/2]; element 2j in the low
 *                           nibble of byte j, element 2j+1 in the high nibble
 *                           (an MXFP4 columnwise copy: [cols, rows/2]).
 *   Scale factors         : the tensor-core tile layout.  For a logical
 *                           [R, S] scale matrix (S = cols/32 for MXFP8 and
                           MXFP4, cols/16 for NVFP4),
 *                           scale (r, k) lives at byte
 *                             ((r/128)*ceil(S/4) + k/4)*512
 *                             + (r%32)*16 + ((r%128)/32)*4 + k%4
 *                           of a buffer of ceil(R/128)*128 * ceil(S/4)*4
 *                           bytes; padding bytes are written as zero.
 *                           With group offsets, group g's rows start at
 *                           padded row P_g = sum_{h<g} ceil(n_h/128)*128.
 *
 * Errors: arguments are validated on the host before any launch
 * (MX8_ERR_INVALID_ARG / MX8_ERR_ALIGNMENT / MX8_ERR_UNSUPPORTED); a failed
 * launch returns MX8_ERR_CUDA.  Every device-side wait is bounded (about one
 * second); a wait that runs out sets an error word in the caller's
 * workspace, and mx8_check_device_error() reports it as MX8_ERR_TIMEOUT.
 *
 * Workspace: a caller-owned device buffer of at least
 * mx8_workspace_bytes(num_groups) bytes, zero-filled once before first use.
 * Its first 16 bytes hold the error word; the rest is scratch for the call.
 * Calls are asynchronous on the given stream; two calls that share one
 * workspace must be ordered (same stream or synchronised).
 */
#ifndef MX8Q_H
#define MX8Q_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *mx8_stream_t; /* the same type as cudaStream_t */

typedef enum {
    MX8_OK = 0,
    MX8_ERR_INVALID_ARG = 1,  /* null pointer, bad size or mode           */
    MX8_ERR_ALIGNMENT = 2,    /* pointer or stride not 16-byte aligned     */
    MX8_ERR_UNSUPPORTED = 3,  /* valid request this build does not handle  */
    MX8_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed         */
    MX8_ERR_TIMEOUT = 5,      /* a bounded device wait ran out             */
    MX8_ERR_WORKSPACE = 6     /* workspace missing or too small            */
} mx8_status;

enum { MX8_ROWWISE = 1, MX8_COLWISE = 2 };
enum { NVFP4_SCOPE_TOKEN = 0, NVFP4_SCOPE_GROUP = 1, NVFP4_SCOPE_TENSOR = 2 };
enum { MX8_FMT_MXFP8 = 0, MX8_FMT_NVFP4 = 1, MX8_FMT_MXFP4 = 2 };
enum { MX8_OUT_F32 = 0, MX8_OUT_BF16 = 1 };
enum { MX8_EPI_NONE = 0, MX8_EPI_SWIGLU = 1 };
/* Where nvfp4_quantize_dispatch() puts codes and S_dec. */
enum { MX8_DISPATCH_TOKENS = 0, MX8_DISPATCH_ROWS = 1 };
/* How an FP32 decode scale vector applies to the rows of a matrix. */
enum { MX8_S32_NONE = 0, MX8_S32_ROW = 1, MX8_S32_TENSOR = 2, MX8_S32_GROUP = 3 };

/* Bytes of the tensor-core scale buffer for a [rows, cols] matrix in format
 * fmt (block 32 for MXFP8 and MXFP4, 16 for NVFP4). */
size_t mx8_scale_bytes(int fmt, int64_t rows, int64_t cols);

/* Upper bound of the grouped scale buffer (every group padded to whole
 * 128-row tiles) for total_rows rows split into num_groups groups. */
size_t mx8_scale_bytes_grouped(int fmt, int64_t total_rows, int num_groups, int64_t cols);

/* Workspace bytes needed by any call below with up to num_groups groups. */
size_t mx8_workspace_bytes(int num_groups);

/* Number of streaming multiprocessors the kernels size their grids for. */
int mx8_device_sm_count(void);

/*
 * MXFP8 quantization of a bf16 matrix, rowwise and/or columnwise in one pass
 * over the input ([MRL] "La Compatibilidad...": 32 E4M3 values share one E8M0
 * scale; [MRL] "Un Cuantizador Compartido...": both copies come from the
 * high-precision input; [REC] MXFP8 paragraph).
 *   x        : bf16 [rows, cols], row stride ld >= cols elements
 *   flags    : MX8_ROWWISE | MX8_COLWISE
 *   q_row    : E4M3 [rows, cols]                 (ROWWISE)
 *   s_row    : mx8_scale_bytes(MXFP8, rows, cols) (ROWWISE)
 *   q_col    : E4M3 [cols, rows], transposed     (COLWISE)
 *   s_col    : mx8_scale_bytes(MXFP8, cols, rows) (COLWISE)
 * Requires cols % 32 == 0, and rows % 32 == 0 for COLWISE; ld % 8 == 0;
 * x, q_*, s_* 16-byte aligned.  rows == 0 or cols == 0 is a no-op.
 */
mx8_status mx8_quantize(const void *x, int64_t rows, int64_t cols, int64_t ld, int flags,
                        uint8_t *q_row, uint8_t *s_row, uint8_t *q_col, uint8_t *s_col,
                        void *workspace, size_t workspace_bytes, mx8_stream_t stream);

/*
 * MXFP4 quantization of a bf16 matrix, rowwise and/or columnwise in one pass
 * over the input ([NV4] "Que es realmente NVFP4": 32 E2M1 values share one
 * power-of-two E8M0 scale).  Same arguments, checks and scale layout as
 * mx8_quantize(), with packed data:
 *   q_row    : uint8 [rows, cols/2]              (ROWWISE)
 *   s_row    : mx8_scale_bytes(MXFP4, rows, cols) (ROWWISE)
 *   q_col    : uint8 [cols, rows/2], transposed  (COLWISE)
 *   s_col    : mx8_scale_bytes(MXFP4, cols, rows) (COLWISE)
 */
mx8_status mxfp4_quantize(const void *x, int64_t rows, int64_t cols, int64_t ld, int flags,
                          uint8_t *q_row, uint8_t *s_row, uint8_t *q_col, uint8_t *s_col,
                          void *workspace, size_t workspace_bytes, mx8_stream_t stream);

/* One input of mx8_quantize_batch(): the arguments of one mx8_quantize()
 * (or mxfp4_quantize()) call. */
typedef struct {
    const void *x;
    int64_t rows, cols, ld;
    uint8_t *q_row, *s_row, *q_col, *s_col;
} mx8_quantize_item;

#define MX8_BATCH_MAX 4

/*
 * mx8_quantize() (fmt MX8_FMT_MXFP8) or mxfp4_quantize() (MX8_FMT_MXFP4) of
 * up to MX8_BATCH_MAX tensors in ONE launch, e.g. the input, weight and
 * output gradient of a linear layer ([MRL] "Un Cuantizador Compartido...":
 * each tensor's rowwise and columnwise copies come from its high-precision
 * values).  The tensors' 128x128 tiles form one work list for a persistent
 * grid, so the launch and memory latency of a small tensor hide behind the
 * others.  Results are byte for byte those of the separate calls; each item
 * obeys the same rules (items with rows == 0 or cols == 0 are skipped).
 * flags applies to every item.  n outside [1, MX8_BATCH_MAX] returns
 * MX8_ERR_INVALID_ARG.
 */
mx8_status mx8_quantize_batch(int fmt, const mx8_quantize_item *items, int n, int flags,
                              void *workspace, size_t workspace_bytes, mx8_stream_t stream);

/*
 * Two-level NVFP4 quantization of a bf16 matrix with the FP32 scale computed
 * online per token ([MRL] "La Compatibilidad..." and "Un Cuantizador
 * Compartido...": one FP32 activation scale per token, fused into the
 * activation quantizer that also emits the packed FP4 values and the block
 * scales; [NV4] "Que es realmente NVFP4"; [REC] NVFP4 paragraphs).
 *   x      : bf16 [rows, cols], row stride ld
 *   scope  : NVFP4_SCOPE_TOKEN  -> s32[rows], one decode scale per row
 *            NVFP4_SCOPE_GROUP  -> s32[num_groups] (e.g. one per expert
 *                                  weight, gate|up stored jointly)
 *            NVFP4_SCOPE_TENSOR -> s32[1]
 *   group_offsets : device int64 [num_groups+1], non-decreasing, 0..rows;
 *            when given, the scale buffer uses the grouped (per-group
 *            padded) tile layout; NULL means one group.  Required for
 *            NVFP4_SCOPE_GROUP.
 *   q      : uint8 [rows, cols/2]
 *   s_blk  : E4M3 scales, mx8_scale_bytes(NVFP4, rows, cols), or
 *            mx8_scale_bytes_grouped(...) with group_offsets
 * Requires cols % 16 == 0, ld % 8 == 0, 16-byte aligned x/q/s_blk;
 * cols > 2^30 returns MX8_ERR_UNSUPPORTED.
 */
mx8_status nvfp4_quantize_per_token(const void *x, int64_t rows, int64_t cols, int64_t ld,
                                    int scope, const int64_t *group_offsets, int num_groups,
                                    uint8_t *q, uint8_t *s_blk, float *s32,
                                    void *workspace, size_t workspace_bytes,
                                    mx8_stream_t stream);

/*
 * Per-token NVFP4 quantization of MoE tokens once, before dispatch ([MRL]
 * "La Compatibilidad..." / "Un Cuantizador Compartido...": the FP32 token
 * scale is computed per token inside the activation quantizer; per-token
 * scaling makes a token's codes independent of the batch, so quantizing
 * before the top-k dispatch gives the same bytes as quantizing every
 * dispatched copy, with 1/topk of the reads and of the encode work).
 *   x          : bf16 [tokens, cols], row stride ld
 *   dest_rows  : device int64 [tokens * topk]: the dispatched row of copy j
 *                of token t at [t * topk + j]; together the entries cover
 *                every dispatched row [0, group_offsets[G]) exactly once
 *                (entries outside that range are skipped)
 *   group_offsets : device int64 [num_groups + 1], the expert row ranges of
 *                the dispatched order
 *   layout     : MX8_DISPATCH_ROWS -> every copy written: q [R, cols/2]
 *                and s32 [R] in dispatched-row order (R = group_offsets[G]),
 *                the input of bs_grouped_gemm() / bs_grouped_gemm_fused()
 *                without a_rows;
 *                MX8_DISPATCH_TOKENS -> q [tokens, cols/2] and s32 [tokens]
 *                token-major, the input of bs_grouped_gemm_fused() with
 *                a_rows (the GEMM gathers the code rows)
 *   s_blk      : E4M3 scales of the DISPATCHED rows in the grouped layout,
 *                mx8_scale_bytes_grouped(NVFP4, tokens * topk, num_groups, cols)
 * Requires 1 <= topk <= 16, cols % 16 == 0, ld % 8 == 0, 16-byte aligned
 * x / q / s_blk.
 */
mx8_status nvfp4_quantize_dispatch(const void *x, int64_t tokens, int64_t cols, int64_t ld,
                                   const int64_t *dest_rows, int topk, const int64_t *group_offsets,
                                   int num_groups, int layout, uint8_t *q, uint8_t *s_blk, float *s32,
                                   void *workspace, size_t workspace_bytes, mx8_stream_t stream);

/*
 * NVFP4 weights with 2-D 16x16 block scaling ([NV4] "La metodologia de
 * formacion de cuatro partes": one quantized representation for the forward
 * weight and the transposed backward weight).  One FP32 tensor scale
 * (S_enc / S_dec from the tensor amax, as NVFP4_SCOPE_TENSOR); per 16x16
 * block the NVFP4 block scale and codes of that scale.
 *   flags  : MX8_ROWWISE | MX8_COLWISE
 *   q_row  : uint8 [rows, cols/2]; s_row: mx8_scale_bytes(NVFP4, rows, cols),
 *            each row holding its block's scale (the tensor cores read 1x16)
 *   q_col  : uint8 [cols, rows/2], the transposed copy; s_col:
 *            mx8_scale_bytes(NVFP4, cols, rows) -- codes and scales are the
 *            exact transposes of the rowwise ones
 *   s32    : float [1], S_dec
 * Requires rows % 32 == 0, cols % 32 == 0, ld % 8 == 0, 16-byte aligned
 * pointers.  Two launches (tensor amax, then encode).
 */
mx8_status nvfp4_quantize_2d(const void *x, int64_t rows, int64_t cols, int64_t ld, int flags,
                             uint8_t *q_row, uint8_t *s_row, uint8_t *q_col, uint8_t *s_col,
                             float *s32, void *workspace, size_t workspace_bytes, mx8_stream_t stream);

/*
 * The transposed NVFP4 copy of a Wgrad input with the 16x16 random Hadamard
 * transform ([NV4] "La metodologia de formacion de cuatro partes": Wgrad
 * inputs are multiplied, in 16-element tiles along the reduction dimension,
 * by a 16x16 Hadamard matrix combined with one random +-1 sign vector shared
 * by all linear layers; orthogonal, so no correction is needed in the GEMM
 * when both Wgrad operands use the same signs).
 *   x         : bf16 [rows, cols] (rows = the Wgrad reduction dimension,
 *               e.g. tokens), row stride ld
 *   sign_mask : bit i set -> sign -1 for element i of every 16-row tile
 *   stochastic: 1 -> codes by stochastic rounding (gradient inputs), as in
 *               nvfp4_quantize_per_token_sr(), element index = position in
 *               q_col (row * rows + column); 0 -> round to nearest even
 *   per 16 rows of a column: y = (1/4) H16 diag(s) x in binary32, evaluated
 *               as the natural-order fast Walsh-Hadamard butterfly; then
 *               NVFP4 of y with one FP32 tensor scale from the amax of y
 *   q_col     : uint8 [cols, rows/2]; s_col: mx8_scale_bytes(NVFP4, cols,
 *               rows); s32: float [1] S_dec
 * Requires rows % 32 == 0, cols % 8 == 0, ld % 8 == 0, 16-byte aligned
 * pointers.  Two launches (transformed amax, then encode).
 */
mx8_status nvfp4_quantize_rht_colwise(const void *x, int64_t rows, int64_t cols, int64_t ld,
                                      uint32_t sign_mask, int stochastic, uint64_t seed,
                                      uint8_t *q_col, uint8_t *s_col, float *s32,
                                      void *workspace, size_t workspace_bytes, mx8_stream_t stream);

/*
 * Per-token NVFP4 of a gradient with stochastically rounded codes ([NV4] "La
 * metodologia de formacion de cuatro partes": round-to-nearest-even biases
 * gradient tensors; stochastic rounding picks one of the two nearest values
 * with probability given by the distance to each; gradients only).  S_dec and
 * the block scales as nvfp4_quantize_per_token() with NVFP4_SCOPE_TOKEN; each
 * code is the E2M1 value below or above RN(x * r), chosen with 32 random
 * bits b: above when (b >> 8) < p * 2^24, p the distance to the value below
 * over the grid spacing; b = Philox4x32-10 (Salmon et al., SC 2011) with
 * counter (e / 4 split into two 32-bit words, 0, 0) and key (seed split into
 * two 32-bit words), word e % 4 of its four outputs, e = row * cols + column.  Same layouts and requirements as the token scope
 * of nvfp4_quantize_per_token() (plain scale layout, padding rows zero).
 */
mx8_status nvfp4_quantize_per_token_sr(const void *x, int64_t rows, int64_t cols, int64_t ld,
                                       uint64_t seed, uint8_t *q, uint8_t *s_blk, float *s32,
                                       mx8_stream_t stream);

/*
 * nvfp4_quantize_per_token() for callers that cannot allocate device memory
 * and so cannot provide a workspace (for instance a plugin whose host
 * application owns every allocation).  Same arguments and results, minus the
 * workspace: the per-group / per-tensor scratch is a fixed ~8 KB array
 * inside the library (at most 1024 groups; more return MX8_ERR_INVALID_ARG),
 * resident on each GPU that loads the library until the process exits.
 * No allocation of any kind happens in this call.  The first call on a device
 * looks up that array's device address; make it before any stream capture,
 * and do not use this entry point on a device after cudaDeviceReset().
 * All calls share the array (its scratch is cleared at the start of each
 * call), so calls that could run at the same time on the GPU race and must
 * be serialised.  A bounded device wait that runs out is recorded in the
 * array's error word, which nvfp4_noalloc_check_error() reads.
 * The pages describe no such variant; it exists for this library's callers.
 */
mx8_status nvfp4_quantize_per_token_noalloc(const void *x, int64_t rows, int64_t cols, int64_t ld,
                                            int scope, const int64_t *group_offsets, int num_groups,
                                            uint8_t *q, uint8_t *s_blk, float *s32,
                                            mx8_stream_t stream);

/* Synchronises the stream, then reads and clears the error word of the
 * library-owned array that nvfp4_quantize_per_token_noalloc() uses: MX8_OK,
 * or MX8_ERR_TIMEOUT if a bounded device wait of any such call since the
 * last check ran out (that call's outputs are then not valid).  Allocates
 * nothing.  (No counterpart in the pages.) */
mx8_status nvfp4_noalloc_check_error(mx8_stream_t stream);

/*
 * Dequantization back to f32 or bf16 (the dequantized-backward mode of [MRL]
 * "La Compatibilidad..." and [REC]: rebuild high-precision operands from the
 * exact low-precision forward values).
 *   MXFP8: out = e4m3 * 2^(scale-127)            (exact; may overflow to inf)
 *   MXFP4: out = e2m1 * 2^(scale-127)            (exact; may overflow to inf)
 *   NVFP4: out = RN((e2m1 * sb) * S_dec)
 *   q, s   : as produced by the quantizers (any rowwise-blocked matrix,
 *            including a transposed columnwise copy)
 *   s32, s32_mode : MX8_S32_NONE / ROW ([rows]) / TENSOR ([1]) / GROUP
 *            ([num_groups], needs group_offsets); NVFP4 only
 *   group_offsets : grouped scale layout (as in nvfp4_quantize_per_token)
 *   out    : [rows, cols] f32 or bf16 (out_dtype); bf16 = RNE of the f32 value
 */
mx8_status dequantize(int fmt, const uint8_t *q, const uint8_t *s, const float *s32, int s32_mode,
                      const int64_t *group_offsets, int num_groups,
                      int64_t rows, int64_t cols, int out_dtype, void *out,
                      mx8_stream_t stream);

/*
 * Block-scaled GEMM on the tcgen05 tensor cores:
 *     C[m, n] (+)= A32[m] * B32[n] * sum_k A^[m, k] * B^[n, k]
 * where A^ and B^ are the block-scaled decodes (MXFP8: E4M3 * E8M0 per 32
 * along K; NVFP4: E2M1 * E4M3 per 16 along K; MXFP4: E2M1 * E8M0 per 32
 * along K).  Both operands store K
 * contiguously, so Fprop (A = X rowwise, B = W rowwise), Dgrad (A = dY
 * rowwise, B = W columnwise copy) and Wgrad (A = dY columnwise copy,
 * B = X columnwise copy) are all this call ([MRL] "La Compatibilidad...":
 * MXFP8 in forward, weight-gradient and data-gradient GEMMs; [MRL] "Un
 * Cuantizador Compartido...": scale blocks follow the reduction dimension).
 *   A, SA : [M, K] data (K/2 bytes per row for NVFP4 and MXFP4) + scales
 *   B, SB : [N, K] data + scales
 *   A32 / a32_mode : MX8_S32_NONE, MX8_S32_ROW ([M], per-token scale),
 *                    MX8_S32_TENSOR ([1])
 *   B32 / b32_mode : MX8_S32_NONE, MX8_S32_ROW ([N]), MX8_S32_TENSOR ([1])
 *   C     : [M, N] with row stride ldc, f32 or bf16; accumulate=1 adds to C
 *           (f32 only)
 * Requires K % 32 == 0, ldc % 8 == 0, 16-byte aligned pointers.
 * Accumulation is FP32 in tensor memory.
 */
mx8_status bs_gemm(int fmt, int64_t M, int64_t N, int64_t K,
                   const uint8_t *A, const uint8_t *SA, const float *A32, int a32_mode,
                   const uint8_t *B, const uint8_t *SB, const float *B32, int b32_mode,
                   int out_dtype, void *C, int64_t ldc, int accumulate,
                   void *workspace, size_t workspace_bytes, mx8_stream_t stream);

/*
 * Grouped block-scaled GEMM for MoE routed experts ([REC] NVFP4 on MoE
 * experts; [MRL] "NVFP4 por token..."): rows [off[g], off[g+1]) of A are the
 * tokens routed to expert g and multiply that expert's weight B[g]:
 *     C[m, n] = A32[m] * B32[g] * sum_k A^[m, k] * B^_g[n, k]
 * The per-expert tile schedule is built on the device from group_offsets:
 * no host synchronisation on the routing.
 *   group_offsets : device int64 [num_groups+1]; total_rows = off[G]
 *   A, SA  : [total_rows, K] data + grouped scale layout (per-group padded)
 *   A32    : [total_rows] per-token FP32 decode scale, or NULL
 *   B, SB  : [G, N, K] data + scales ([G*N, K] tile layout, N % 128 == 0
 *            keeps groups on whole tiles; any N works since each group's
 *            scale block is laid out on its own)
 *   B32    : [G] per-expert FP32 decode scale, or NULL
 *   C      : [total_rows, N] with row stride ldc, f32 or bf16
 */
mx8_status bs_grouped_gemm(int fmt, int num_groups, const int64_t *group_offsets,
                           int64_t total_rows, int64_t N, int64_t K,
                           const uint8_t *A, const uint8_t *SA, const float *A32,
                           const uint8_t *B, const uint8_t *SB, const float *B32,
                           int out_dtype, void *C, int64_t ldc,
                           void *workspace, size_t workspace_bytes, mx8_stream_t stream);

/*
 * The MoE expert GEMM with the token dispatch and the SwiGLU fused in
 * ([MRL] "La Compatibilidad..." / "Un Cuantizador Compartido...": the FP32
 * token scale is fused into the activation quantizer, so each token is
 * quantized once, before dispatch -- per-token scaling makes the codes of a
 * token independent of the batch it sits in -- and SwiGLU experts compute
 * gate and up in one fused GEMM).  NVFP4 only.  As bs_grouped_gemm(), plus:
 *   a_rows     : device int64 [total_rows], the token (row of A) of each
 *                dispatched row, or NULL (A already dispatched, as in
 *                bs_grouped_gemm).  With a_rows, A and A32 are token-major
 *                (A [a_src_rows, K/2], A32 [a_src_rows] or NULL) and SA
 *                holds the dispatched rows' scales in the grouped layout --
 *                exactly what nvfp4_quantize_dispatch() writes; the GEMM
 *                gathers the code rows of each tile.  Indices outside
 *                [0, a_src_rows) are clamped into it.
 *   epilogue   : MX8_EPI_NONE -> C [total_rows, N] as bs_grouped_gemm();
 *                MX8_EPI_SWIGLU -> B [G, N, K] holds per expert the gate rows
 *                [0, F) and the up rows [F, 2F) (N = 2F, F % 128 == 0) and
 *                C [total_rows, F] bf16 receives
 *                  h = RN_bf16(silu(g) * u),  g = RN_bf16(gate), u = RN_bf16(up)
 *                (gate, up: the scaled FP32 GEMM outputs; silu in FP32 as in
 *                mx8_swiglu()), so the gate|up output never reaches memory.
 * Other formats return MX8_ERR_UNSUPPORTED.
 */
mx8_status bs_grouped_gemm_fused(int fmt, int num_groups, const int64_t *group_offsets,
                                 int64_t total_rows, int64_t N, int64_t K,
                                 const uint8_t *A, const uint8_t *SA, const float *A32,
                                 const int64_t *a_rows, int64_t a_src_rows,
                                 const uint8_t *B, const uint8_t *SB, const float *B32,
                                 int epilogue, int out_dtype, void *C, int64_t ldc,
                                 void *workspace, size_t workspace_bytes, mx8_stream_t stream);

/*
 * The gate|up expert GEMM of a SwiGLU MoE layer with the SwiGLU and the
 * per-token NVFP4 quantization of its output h fused into the epilogue
 * ([MRL] "Un Cuantizador Compartido...": the activation quantizer emits the
 * packed FP4 values, block scales and token scales in one operation, and
 * gate and up come out of one fused GEMM; "Las Curvas de Recompensa...":
 * a per-token scale computed as a separate step is what slowed NVFP4).
 * NVFP4 only, A already dispatched (as bs_grouped_gemm()).  Per row m:
 *     h = RN_bf16(silu(g) * u)   exactly as bs_grouped_gemm_fused() with
 *                                MX8_EPI_SWIGLU computes it, and
 *     q_h, s_h, s32_h = what nvfp4_quantize_per_token(h, NVFP4_SCOPE_TOKEN,
 *                       group_offsets) writes for h, byte for byte.
 *   B, SB, B32 : [G, N, K] gate rows [0, F) then up rows [F, 2F) per expert,
 *                N = 2F, N % 256 == 0 and F <= 1024 (the F / 128 column
 *                tiles of a 128-row band run as one thread-block cluster,
 *                which exchanges the rows' maxima; larger F returns
 *                MX8_ERR_UNSUPPORTED)
 *   q_h        : uint8 [total_rows, F/2] packed E2M1 codes of h
 *   s_h        : E4M3 block scales of h in the grouped tile layout,
 *                mx8_scale_bytes_grouped(NVFP4, total_rows, num_groups, F)
 *   s32_h      : float [total_rows] S_dec of h
 *   h, ld_h    : optional bf16 [total_rows, F] copy of h (NULL: h is never
 *                written to memory)
 * Requires K % 32 == 0 and 16-byte aligned A, SA, B, SB, q_h, s_h (and h).
 */
mx8_status bs_grouped_gemm_swiglu_nvfp4(int num_groups, const int64_t *group_offsets, int64_t total_rows,
                                        int64_t N, int64_t K, const uint8_t *A, const uint8_t *SA,
                                        const float *A32, const uint8_t *B, const uint8_t *SB,
                                        const float *B32, uint8_t *q_h, uint8_t *s_h, float *s32_h,
                                        void *h, int64_t ld_h, void *workspace, size_t workspace_bytes,
                                        mx8_stream_t stream);

/*
 * Dense BF16 GEMM on the tcgen05 tensor cores, for the dequantized-backward
 * mode ([MRL] "La Compatibilidad...": the backward GEMMs run in BF16 on
 * operands rebuilt by dequantize() from the low-precision copies, e.g.
 * Dgrad = deq(dY rowwise) x deq(W columnwise)^T, Wgrad = deq(dY columnwise)
 * x deq(X columnwise)^T):
 *     C[m, n] (+)= sum_k A[m, k] * B[n, k]
 *   A : bf16 [M, K], row stride lda >= K elements
 *   B : bf16 [N, K], row stride ldb >= K elements
 *   C : [M, N] with row stride ldc, f32 or bf16; accumulate=1 adds to C
 *       (f32 only)
 * Requires K % 8 == 0, lda/ldb/ldc % 8 == 0, 16-byte aligned pointers.
 * Accumulation is FP32 in tensor memory.
 */
mx8_status bf16_gemm(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                     const void *B, int64_t ldb, int out_dtype, void *C, int64_t ldc,
                     int accumulate, void *workspace, size_t workspace_bytes,
                     mx8_stream_t stream);

/*
 * SwiGLU between the joint gate|up GEMM and the down GEMM of a MoE expert
 * ([MRL] "Un Cuantizador Compartido...": SwiGLU experts compute gate and up
 * in one fused GEMM):
 *     h[r, j] = RN_bf16( silu(g) * u ),  g = gate_up[r, j], u = gate_up[r, ffn + j]
 * with silu(g) = g / (1 + exp(-g)) in FP32 (a few units of 2^-24 from the
 * exact value before the bf16 rounding, so h can differ from the correctly
 * rounded result by one bf16 unit).
 *   gate_up : bf16 [rows, 2*ffn], row stride ld_gate_up
 *   h       : bf16 [rows, ffn], row stride ld_h
 * Requires ffn % 8 == 0, 16-byte aligned pointers and strides % 8 == 0.
 */
mx8_status mx8_swiglu(const void *gate_up, int64_t rows, int64_t ffn, int64_t ld_gate_up,
                      void *h, int64_t ld_h, mx8_stream_t stream);

/*
 * MoE combine, the step that closes the routed-expert layer: each token's
 * top-k expert outputs, weighted by its router weights, summed back in token
 * order:
 *     out[t, h] = sum_{j<topk} w[t, j] * y[rows_of_slot[t, j], h]
 * in binary32 in the order j = 0, 1, ... (each product and each sum one
 * round-to-nearest operation), so the result is deterministic; a bf16 output
 * is the RNE of that value.
 *   y            : bf16 [rows_y, hidden], row stride ld_y (the down GEMM's
 *                  output in dispatched-row order)
 *   rows_of_slot : device int64 [tokens, topk]; rows outside [0, rows_y)
 *                  contribute nothing
 *   weights      : device float [tokens, topk]
 *   out          : [tokens, hidden] f32 or bf16, row stride ld_out
 * Requires hidden % 8 == 0, 1 <= topk <= 16, 16-byte aligned y / out,
 * strides % 8 == 0.
 */
mx8_status mx8_moe_combine(const void *y, int64_t rows_y, int64_t ld_y, const int64_t *rows_of_slot,
                           const float *weights, int64_t tokens, int64_t hidden, int topk,
                           int out_dtype, void *out, int64_t ld_out, mx8_stream_t stream);

/* Synchronises the stream, reads and clears the workspace error word:
 * MX8_OK, or MX8_ERR_TIMEOUT if a bounded device wait ran out. */
mx8_status mx8_check_device_error(void *workspace, mx8_stream_t stream);

/* Self-test of the bounded wait: launches one block that waits on a barrier
 * nothing will complete, with the given limit in nanoseconds; the wait gives
 * up, records the error and the kernel returns.  Follow with
 * mx8_check_device_error(), which then reports MX8_ERR_TIMEOUT. */
mx8_status mx8_selftest_bounded_wait(void *workspace, uint64_t limit_ns, mx8_stream_t stream);

const char *mx8_status_string(mx8_status s);

#ifdef __cplusplus
}
#endif

#endif /* MX8Q_H */
