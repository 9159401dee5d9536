/*
 * fsops.h -- C ABI of the GB300 (sm_103a) MXFP8 SwiGLU MLP library.
 *
 * The operation (Fish Audio, "How we made our TTS API free: the inference
 * engineering behind S2.1 Pro", and its copy on X, "We Made Our Best Voice
 * Model Free"): the feed-forward block of an autoregressive decoder at decode
 * shapes (M <= 128 tokens per step; X copy, "The GPU problem you're paying
 * for"), a SwiGLU MLP -- gate/up projection, SiLU(gate) * up, down projection
 * (X copy, "Custom kernels for the shapes TTS actually uses"; p2, "Por que
 * cuBLAS no era suficiente") -- computed on MXFP8 operands: OCP E4M3 elements
 * with one UE8M0 power-of-two scale per 32 consecutive elements along K (p2,
 * "Estrategia de cuantizacion FP8").  The fused entry point keeps the
 * intermediate on chip / in L2 instead of the bf16 round trip through HBM
 * that separate launches make (p2, "Resultados de benchmark del kernel").
 *
 * Quantisation rule (OCP MX): per 32-block, e = floor(log2(amax)) - 8 clamped
 * to [-127, 127] (amax == 0 gives e = -127); scale byte = e + 127; element =
 * E4M3 round-to-nearest-even of v * 2^-e, magnitudes above 448 saturate to
 * 448, sign kept (a negative value that rounds to zero is code 0x80).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller, 16-byte
 *     aligned.  The library never allocates, frees or synchronises inside a
 *     compute call; calls are asynchronous on `stream` (a cudaStream_t, NULL =
 *     legacy default stream) and may be captured in a CUDA graph.
 *   - Arguments are validated on the host before anything is launched; a
 *     rejected call launches nothing and touches no device memory.
 *   - Matrices are row-major.  Weights are [rows, K] with K contiguous
 *     (K-major); activations are [M, K].
 *   - Inputs must be finite; NaN or Inf inputs give unspecified results.
 *   - No C++ exception crosses this interface.
 *
 * Scale layouts (fsops_scale_layout):
 *   FSOPS_SCALES_ROWMAJOR: [rows, K/32] bytes, block index fastest.
 *   FSOPS_SCALES_TCGEN05:  the layout the tcgen05 block-scaled MMA reads.
 *     Rows are grouped in tiles of 128 and K-blocks in groups of 4; each
 *     (row tile rt, group kg) is 512 contiguous bytes at offset
 *     (rt * (K/128) + kg) * 512, and entry (r, kb) sits at
 *     (r % 32) * 16 + ((r % 128) / 32) * 4 + (kb % 4) inside it.  Rows past
 *     the end of the matrix inside the last tile are padding (byte 0).
 *     K must be a multiple of 128.  Buffer size: fsops_scale_bytes().
 *   Scales handed to the GEMM and MLP entry points must be in the TCGEN05
 *   layout.  Handing over another layout is not detected; it silently gives
 *   wrong numbers at normal speed (the failure the Fish Audio post describes
 *   for its own scale-layout bug, p2 "Estrategia de cuantizacion FP8").
 */
#ifndef FSOPS_H
#define FSOPS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FSOPS_OK = 0,
  FSOPS_ERR_INVALID_ARG = 1,      /* null pointer, bad enum, missing or too small workspace */
  FSOPS_ERR_UNSUPPORTED_SHAPE = 2,/* a size outside the documented limits */
  FSOPS_ERR_MISALIGNED = 3,       /* a pointer that is not 16-byte aligned */
  FSOPS_ERR_CUDA = 4,             /* a CUDA runtime call or a launch failed */
  FSOPS_ERR_TIMEOUT = 5,          /* a kernel wait ran out (read with fsops_read_kernel_status) */
  FSOPS_ERR_NO_DEVICE = 6         /* the current device is not an sm_100-class GPU */
} fsops_status;

typedef enum { FSOPS_SCALES_ROWMAJOR = 0, FSOPS_SCALES_TCGEN05 = 1 } fsops_scale_layout;

typedef enum { FSOPS_DTYPE_BF16 = 0, FSOPS_DTYPE_F32 = 1, FSOPS_DTYPE_MXFP8 = 2 } fsops_dtype;

/* Scales of the two MLP weights, both in the FSOPS_SCALES_TCGEN05 layout. */
typedef struct {
  const uint8_t* gateup; /* of W_gateup [2I, H] */
  const uint8_t* down;   /* of W_down [H, I] */
} fsops_mlp_scales;

/* ------------------------------------------------------------------------
 * fsops_quantize_mxfp8 -- bf16 -> MXFP8 (activation quantisation and scale
 * packing in one launch: the first of the two fused kernels in p2,
 * "Resultados de benchmark del kernel"; also the offline weight quantiser).
 *   x_bf16  [rows, ld] bf16, the first K columns are quantised; ld % 8 == 0.
 *   codes   [rows, K] E4M3 bytes (row stride K).
 *   scales  UE8M0 bytes in `layout`; fsops_scale_bytes(rows, K, layout) bytes.
 *   rows >= 0 (0 is a no-op), K % 32 == 0 (ROWMAJOR) or K % 128 == 0 (TCGEN05),
 *   rows * K < 2^31.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA.
 */
fsops_status fsops_quantize_mxfp8(const void* x_bf16, int rows, int K, int ld, uint8_t* codes,
                                  uint8_t* scales, fsops_scale_layout layout, void* stream);

/* fsops_quantize_mxfp8_gateup -- W_gate and W_up (bf16) to the MXFP8 W_gateup
 * that fsops_mxfp8_swiglu_mlp reads, in one launch: the rows are quantised
 * along H with the rule above and written in the paired order (rows
 * 128j..128j+63 from W_gate rows 64j..64j+63, rows 128j+64..128j+127 from
 * W_up rows 64j..64j+63), with TCGEN05 scales.  The pages do not say how
 * gate and up are stored; pairing keeps the gate and up sums of a feature in
 * one accumulator tile, and doing it here keeps a caller from handing over a
 * stacked [W_gate; W_up], which the MLP would not detect (p2 "Estrategia de
 * cuantizacion FP8": a weight layout mismatch gives wrong values at full
 * speed).
 *   w_gate_bf16, w_up_bf16  [I, ld] bf16 each, the first H columns used;
 *                           ld % 8 == 0.
 *   codes   [2I, H] E4M3;  scales fsops_scale_bytes(2I, H, TCGEN05) bytes.
 *   I % 64 == 0, H % 128 == 0, 2I * H < 2^31.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA. */
fsops_status fsops_quantize_mxfp8_gateup(const void* w_gate_bf16, const void* w_up_bf16, int I, int H, int ld,
                                         uint8_t* codes, uint8_t* scales, void* stream);

/* Size in bytes of a scale buffer for a [rows, K] matrix (0 for an invalid layout). */
size_t fsops_scale_bytes(int rows, int K, fsops_scale_layout layout);

/* ------------------------------------------------------------------------
 * fsops_mxfp8_gemm -- C[M, N] = A^[M, K] * B^[N, K]^T, the block-scaled
 * MXFP8 GEMM (p2 "Estrategia de cuantizacion FP8": mxfp8 1x32; the raw linear
 * that reads MXFP8 weights with a fixed scale stride).  A is bf16 and is
 * quantised inside the same launch; B is MXFP8 (codes + TCGEN05 scales);
 * C is bf16 (round-to-nearest-even of the fp32 accumulation).
 *   1 <= M <= 16384; N % 128 == 0; K % 128 == 0; N, K <= 65536.
 *   M <= 128 (decode): one launch, the K loop split over all SMs.  M > 128
 *   (prefill; p2 "Resultados de benchmark del kernel" runs the MLP from M = 1
 *   to 4096): A is quantised by its own launch when bf16, then every block
 *   computes whole 128 x 256 output tiles.
 *   workspace: device scratch of at least fsops_gemm_workspace_bytes(M, N, K)
 *   bytes, all zero before its first use.  Every call leaves its readiness
 *   counters and split-K accumulators zero again (a call whose wait ran out
 *   clears them before it returns), so the same workspace is reused without
 *   clearing; bytes 8..15 keep a running count of the blocks that have left
 *   the decode kernel.  One call at a time per workspace: calls that share a
 *   workspace must be ordered (same stream).
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA.
 */
fsops_status fsops_mxfp8_gemm(const void* a_bf16, const uint8_t* b_codes, const uint8_t* b_scales,
                              void* c_bf16, int M, int N, int K, void* workspace, size_t ws_bytes,
                              void* stream);

/* General form of fsops_mxfp8_gemm.
 *   a_dtype FSOPS_DTYPE_BF16: `a` is bf16 [M, K], quantised in-kernel, a_scales must be NULL.
 *   a_dtype FSOPS_DTYPE_MXFP8: `a` is E4M3 codes [M, K], a_scales its TCGEN05
 *     scales (ceil(M/128) x K/128 tiles of 512 bytes; rows past M are ignored).
 *   c_dtype FSOPS_DTYPE_BF16 or FSOPS_DTYPE_F32.  Other limits as above.
 */
fsops_status fsops_mxfp8_gemm_ex(const void* a, const uint8_t* a_scales, fsops_dtype a_dtype,
                                 const uint8_t* b_codes, const uint8_t* b_scales, void* c,
                                 fsops_dtype c_dtype, int M, int N, int K, void* workspace,
                                 size_t ws_bytes, void* stream);

size_t fsops_gemm_workspace_bytes(int M, int N, int K);

/* ------------------------------------------------------------------------
 * fsops_swiglu_quantize_mxfp8 -- h = SiLU(g) * u, requantised to MXFP8 along
 * I (the second fused kernel of p2 "Resultados de benchmark del kernel": the
 * SwiGLU prologue inside the down GEMM's activation quantisation).
 *   gu      [M, 2I] fp32 in the paired order of W_gateup's rows: columns
 *           128j..128j+63 are gate features 64j..64j+63, columns
 *           128j+64..128j+127 the up features 64j..64j+63 (this is what
 *           fsops_mxfp8_gemm_ex writes for A = x and B = W_gateup).
 *   h_codes [M, I] E4M3;  h_scales TCGEN05 layout, ceil(M/128) x I/128 tiles
 *   of 512 bytes (scales of rows past M within the last row tile may be left
 *   unwritten; the GEMMs ignore those rows).
 *   1 <= M <= 16384, I % 128 == 0.
 */
fsops_status fsops_swiglu_quantize_mxfp8(const float* gu, int M, int I, uint8_t* h_codes,
                                         uint8_t* h_scales, void* stream);

/* ------------------------------------------------------------------------
 * fsops_mxfp8_swiglu_mlp -- the whole block:
 *   x^ = MXFP8(x);  g = x^ Wg^T, u = x^ Wu^T (fp32 accumulate);
 *   h = SiLU(g) * u (fp32);  h^ = MXFP8(h) along I;  y = bf16(h^ Wd^T).
 *   M <= 128 (decode): ONE launch; h never leaves the chip except as split
 *   sums in L2.  M > 128 (prefill): three launches -- x quantised; the gate/up
 *   GEMM over whole 128 x 256 tiles whose epilogue forms h and requantises it
 *   (h^ goes to the workspace, M * I bytes plus scales); the down GEMM on h^.
 *   x_bf16   [M, H] bf16.
 *   w_gateup [2I, H] E4M3, W_gate and W_up paired in blocks of 64 rows:
 *            rows 128j..128j+63 are W_gate rows 64j..64j+63 and rows
 *            128j+64..128j+127 are W_up rows 64j..64j+63 (so every 128-row
 *            weight tile, and its one 512-byte scale tile, holds the gate and
 *            up rows of 64 features).
 *   w_down   [H, I] E4M3.
 *   scales   TCGEN05 scales of both.
 *   y_bf16   [M, H] bf16.
 *   1 <= M <= 16384; H % 128 == 0; I % 128 == 0; H, I <= 65536.
 * Uses the workspace registered with fsops_set_workspace for the current
 * device (INVALID_ARG if none or too small).  Calls on one device are ordered
 * by the caller (one stream, or events); concurrent calls would share the
 * workspace.
 * Launch order: the decode launch (M <= 128) may begin while the previous
 * kernel on the stream is finishing.  It starts streaming w_gateup, w_down
 * and their scales at once and waits for that kernel before it touches
 * anything else (x, y, the workspace).  So the weights must not be written
 * by the kernel launched just before this call on the same stream (the
 * library's own weight quantisers make their writes visible before they
 * finish, so they may precede it).
 */
fsops_status fsops_mxfp8_swiglu_mlp(const void* x_bf16, const uint8_t* w_gateup, const uint8_t* w_down,
                                    const fsops_mlp_scales* scales, void* y_bf16, int M, int H, int I,
                                    void* stream);

/* ------------------------------------------------------------------------
 * The decoder block around the MLP.  The pages name the MLP as a Qwen3-4B
 * SwiGLU MLP (p2, "Resultados de benchmark del kernel"): in that pre-norm
 * decoder the MLP's input is RMSNorm(x) * gamma and its output is added back
 * to x.  The pages do not write either step out; these entry points take the
 * standard definitions, in fp32:
 *   RMSNorm(x)[m, k] = x[m, k] * rsqrt(mean_j x[m, j]^2 + eps).
 *
 * fsops_rmsnorm_quantize_mxfp8 -- codes/scales of RMSNorm(x) * gamma, quantised
 * with the MXFP8 rule above (the normalised values are never rounded to bf16).
 *   x_bf16 [rows, ld] bf16 (first K columns used), gamma_bf16 [K] bf16,
 *   eps >= 0 (INVALID_ARG for negative, NaN or huge), codes [rows, K], scales
 *   as in fsops_quantize_mxfp8 (the tiled layout pads rows to 128 with scale 0).
 *   Limits as fsops_quantize_mxfp8; gamma 16-byte aligned.
 */
fsops_status fsops_rmsnorm_quantize_mxfp8(const void* x_bf16, const void* gamma_bf16, float eps, int rows, int K,
                                          int ld, uint8_t* codes, uint8_t* scales, fsops_scale_layout layout,
                                          void* stream);

/* fsops_mxfp8_swiglu_mlp_block -- the feed-forward half of a decoder layer:
 *   y = x + MLP(RMSNorm(x) * gamma)   (residual = 1)
 *   y = MLP(RMSNorm(x) * gamma)       (residual = 0)
 * with MLP the computation of fsops_mxfp8_swiglu_mlp and the sum rounded to
 * bf16 once.  ONE launch for M <= 128: the MLP kernel computes each row's
 * mean square in its x-quantisation prologue, quantises x * rsqrt(ms + eps) *
 * gamma straight to MXFP8 (never rounded to bf16) and adds x in its bf16
 * store.  Three launches above 128 rows (RMSNorm + quantisation, then the
 * tiled MLP).  Arguments, limits and workspace as fsops_mxfp8_swiglu_mlp,
 * plus gamma_bf16 [H] (16-byte aligned) and eps.
 * y_bf16 may equal x_bf16 (in place): every read of x for the norm and the
 * quantisation happens before any block writes y (each block reads x before
 * its gate/up products, and every tile of y needs every gate/up tile), and
 * the residual is read only by the thread that then writes the same element
 * of y.
 * Graph-capture safe, so a chain of layers (y of one block is x of the next)
 * can be captured once and replayed. */
fsops_status fsops_mxfp8_swiglu_mlp_block(const void* x_bf16, const void* gamma_bf16, float eps, int residual,
                                          const uint8_t* w_gateup, const uint8_t* w_down,
                                          const fsops_mlp_scales* scales, void* y_bf16, int M, int H, int I,
                                          void* stream);

/* ------------------------------------------------------------------------
 * fsops_mxfp8_paged_decode_attention -- one decode step of attention over a
 * paged KV cache held in MXFP8 (the library's MXFP8 FlashAttention with paged
 * decode and native GQA through a stride-0 K/V broadcast, p2 "Ya esta
 * disponible").  The pages do not write it out; read plainly:
 *   for sequence b, query head h, KV head hk = h / (Hq / Hkv):
 *   s[t] = sm_scale * q[b, h, :] . K^[t, hk, :]   for t < seq_lens[b],
 *   out[b, h, :] = bf16( sum_t softmax(s)[t] * V^[t, hk, :] ),
 * with K^ and V^ the dequantised cache (E4M3 codes times one UE8M0 scale per
 * 32 elements of the head dimension, the rule above) and q, s and the
 * probabilities in fp32.  The G = Hq / Hkv query heads of a KV head read its
 * K and V once.
 *   q_bf16      [B, Hq, D] bf16.
 *   k_codes, v_codes    [num_pages, Hkv, P, D] E4M3 (P = page_size tokens of
 *               one KV head contiguous per page).
 *   k_scales, v_scales  [num_pages, Hkv, P, D / 32] UE8M0, row-major per token
 *               (fsops_quantize_mxfp8's FSOPS_SCALES_ROWMAJOR of the
 *               [num_pages * Hkv * P, D] rows).
 *   block_table [B, max_pages] int32 page ids; token t of sequence b is slot
 *               t % P of page block_table[b, t / P].  Entries past a
 *               sequence's last page are not read.
 *   seq_lens    [B] int32, 1 <= seq_lens[b] <= max_pages * P.
 *   out_bf16    [B, Hq, D] bf16.
 *   Limits: D = 128; P in {16, 32, 64, 128}; Hq / Hkv in {1, 2, 4, 8};
 *   B, Hkv <= 65535.  Pointers 16-byte aligned (block_table, seq_lens 4).
 *   workspace: 256-byte aligned, fsops_paged_attention_workspace_bytes() of
 *   device memory whose first 256 bytes are zero before the first call: the
 *   status word, where a page id outside [0, num_pages) or a bad length is
 *   reported (fsops_read_kernel_status) instead of being read, and the
 *   counter from which the first launch's persistent blocks take their work
 *   (each call leaves it zero).  Two launches (the splits of each sequence,
 *   then their combination); graph-capture safe.  Calls sharing a workspace
 *   are serialised by their stream. */
fsops_status fsops_mxfp8_paged_decode_attention(const void* q_bf16, const uint8_t* k_codes, const uint8_t* k_scales,
                                                const uint8_t* v_codes, const uint8_t* v_scales, int num_pages,
                                                const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                                                void* out_bf16, int B, int Hq, int Hkv, int D, int page_size,
                                                float sm_scale, void* workspace, size_t ws_bytes, void* stream);

/* Workspace bytes of fsops_mxfp8_paged_decode_attention on the current device
 * (0 if the shape is unsupported). */
size_t fsops_paged_attention_workspace_bytes(int B, int Hq, int Hkv, int D, int page_size, int max_pages);

/* ------------------------------------------------------------------------
 * FP8 with 128 x 128 block scales -- the second scale format the Fish Audio
 * post names beside mxfp8 ("bsgemm", X copy "Custom kernels for the shapes
 * TTS actually uses"; p2 "Estrategia de cuantizacion FP8").  The pages give
 * no formula; read plainly:
 *   weights W [N, K]: one fp32 scale per 128 x 128 block, activations A [M, K]:
 *   one fp32 scale per 1 x 128 group along K (a 128 x 128 block of activations
 *   would span every token of a decode step); scale = amax / 448 in fp32 (1
 *   for an all-zero block); code = E4M3 round-to-nearest-even, saturating at
 *   448, of v / scale in fp32 (correctly rounded division), sign kept.
 *
 * fsops_quantize_fp8_blockscale -- bf16 x [rows, ld] (first K columns) to
 *   codes [rows, K] and fp32 scales [ceil(rows / block_rows), K / 128]
 *   (row-major), block_rows 1 (activations) or 128 (weights).  K % 128 == 0,
 *   ld % 8 == 0, rows * ld < 2^31.  Scales 4-byte aligned.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA. */
fsops_status fsops_quantize_fp8_blockscale(const void* x_bf16, int rows, int K, int ld, int block_rows, uint8_t* codes,
                                           float* scales, void* stream);

/* Number of fp32 scales of a [rows, K] matrix in blocks of block_rows x 128
 * (0 for an invalid argument). */
size_t fsops_blockscale_scale_count(int rows, int K, int block_rows);

/* fsops_fp8_blockscale_gemm -- C[M, N] = sum over 128-deep K-blocks kb of
 *   a_scales[m, kb] * w_scales[n / 128, kb] * (A^ W^T over kb), in fp32, for
 *   A = a_codes [M, K] with its 1 x 128 scales and W = w_codes [N, K] with its
 *   128 x 128 scales (as fsops_quantize_fp8_blockscale writes them).  C is
 *   bf16 (rounded once) or fp32.  One launch.  1 <= M <= 128, N % 128 == 0,
 *   K % 128 == 0, N, K <= 65536.
 *   workspace: 256-byte aligned, fsops_blockscale_gemm_workspace_bytes(M, N, K)
 *   bytes, zero before its first use; a successful call leaves it zero again
 *   (zero it again after a call that reported an error).  Calls that share a
 *   workspace must be ordered.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA. */
fsops_status fsops_fp8_blockscale_gemm(const uint8_t* a_codes, const float* a_scales, const uint8_t* w_codes,
                                       const float* w_scales, void* c, fsops_dtype c_dtype, int M, int N, int K,
                                       void* workspace, size_t ws_bytes, void* stream);

size_t fsops_blockscale_gemm_workspace_bytes(int M, int N, int K);

/* The same computation as three launches with the intermediates in HBM (the
 * unfused baseline of p2 "Por que cuBLAS no era suficiente"): GEMM gate/up
 * with fp32 output [M, 2I], SwiGLU + requantisation, GEMM down.  Same
 * arguments, limits and workspace as fsops_mxfp8_swiglu_mlp. */
fsops_status fsops_mxfp8_swiglu_mlp_unfused(const void* x_bf16, const uint8_t* w_gateup,
                                            const uint8_t* w_down, const fsops_mlp_scales* scales,
                                            void* y_bf16, int M, int H, int I, void* stream);

/* fsops_mxfp8_swiglu_mlp_noalloc -- the same single-launch MLP, for callers
 * that cannot allocate device memory: code running inside a framework or
 * plugin host that owns every device allocation, paths that must not call an
 * allocator (cudaMalloc may synchronise the device), or deployments with a
 * fixed memory budget.  It has no counterpart in the paper; it is a packaging
 * of fsops_mxfp8_swiglu_mlp.
 *   Arguments, layouts and limits as fsops_mxfp8_swiglu_mlp, with M <= 128
 *   only (the single-launch path; larger M is FSOPS_ERR_UNSUPPORTED_SHAPE),
 *   and no workspace is used: the scratch is one fixed 8 MiB buffer per device
 *   inside the library's device image, present from library load until
 *   process exit.  A shape whose scratch does not fit in 8 MiB is rejected
 *   with FSOPS_ERR_UNSUPPORTED_SHAPE before anything is launched.  The scratch
 *   is 16 KiB + M * (H + I) bytes (quantised x and h) + about
 *   (H + I) * 4 bytes of scales + the split-K sums: 1 KiB * M * ceil(H / TR1)
 *   for the down projection, with TR1 = 128 for M > 64 and 256 otherwise,
 *   plus 1 KiB * M * (2 I / 256) for M <= 32 (split gate/up tiles).  Example:
 *   M = 128, H = 4096, I = 12288 needs about 6.1 MiB.
 *   The first call on a device looks up the buffer's device address
 *   (cudaGetSymbolAddress) and clears the buffer (cudaMemsetAsync on
 *   `stream`); make that first call outside any stream capture.  A launch
 *   that succeeds leaves the buffer ready for the next call, so later calls
 *   only launch the kernel; the buffer is cleared again before the next call
 *   after a call that failed, or after fsops_read_noalloc_status reported a
 *   kernel error.  Neither step allocates.  All calls on a device share the
 *   one buffer, so calls whose execution overlaps on the GPU (different
 *   streams without ordering) race; order them. */
fsops_status fsops_mxfp8_swiglu_mlp_noalloc(const void* x_bf16, const uint8_t* w_gateup,
                                            const uint8_t* w_down, const fsops_mlp_scales* scales,
                                            void* y_bf16, int M, int H, int I, void* stream);

/* fsops_read_noalloc_status -- the status word of the fixed buffer of
 * fsops_mxfp8_swiglu_mlp_noalloc on the current device, read and cleared
 * like fsops_read_kernel_status (synchronises the device).  A nonzero word
 * (a kernel wait that ran out) also makes the next no-allocation call clear
 * the buffer first.  INVALID_ARG before the first no-allocation call on the
 * device. */
fsops_status fsops_read_noalloc_status(uint32_t* word);

/* Workspace bytes the MLP entry points need on the current device (0 if the
 * shape is unsupported).  It covers the unfused path's fp32 [M, 2I]
 * intermediate too (M * 8I bytes), which dominates for large M. */
size_t fsops_mlp_workspace_bytes(int M, int H, int I);

/* Register `ws` (device memory of `bytes` bytes, 256-byte aligned) as the MLP
 * workspace of the current device, replacing any earlier one.  Zeroes all of
 * it and synchronises the device: call it outside stream capture, before the
 * first MLP call, and again after a call that reported an error.
 * ws == NULL unregisters. */
fsops_status fsops_set_workspace(void* ws, size_t bytes);

/* ------------------------------------------------------------------------
 * Diagnostics.
 * fsops_read_kernel_status: synchronously reads and clears the status word
 * that the kernels write into a workspace when a bounded wait runs out
 * (workspace NULL = the registered MLP workspace of the current device).
 * *word is 0 when no kernel failed; otherwise bits 31..24 hold an
 * fsops_status, bits 23..16 the wait site and bits 15..0 the block index.
 * After a failure the workspace counters are reset by the kernel itself: the
 * blocks of a launch that gave up clear them once every block has left its
 * waits. */
fsops_status fsops_read_kernel_status(void* workspace, uint32_t* word);

/* Upper bound, in nanoseconds, for every wait inside the kernels launched
 * after this call (default 1e9).  Applies to the calling process. */
fsops_status fsops_set_wait_timeout_ns(uint64_t ns);

/* Test hook: kernels launched after this call wait for `n` more arrivals on
 * their cross-block readiness counters (quantised activations, finished
 * SwiGLU tiles) than any launch produces, so those waits run out and report
 * FSOPS_ERR_TIMEOUT.  0 (the default) disables it. */
fsops_status fsops_debug_set_extra_arrivals(uint32_t n);

/* Plan overrides for tests and tuning (fsops_debug_set_knob).  Each knob
 * holds -1 (the default: the library picks) or a forced value; a forced value
 * that a shape cannot use is ignored for that call.  They apply to calls made
 * after the change, in every thread of the process.
 *   TR0, TR1          weight tile rows of the gate/up and down phases of the
 *                     single-launch MLP on the grid-wide path: 128 or 256.
 *   WHOLE_TILES       1: one whole gate/up tile per block; 0: split-K.
 *   PAIRS             0: no 2-block cluster split of gate/up tiles.
 *   GEMM_FORM         tiled GEMM above 128 rows: 0 one block per 128 x 256
 *                     tile, 1 a 2-block cluster per 256 x 256 tile
 *                     (cta_group::2 MMA; N % 256 == 0, two or more row tiles).
 *   PRIME             weight loads in flight before the activations exist.
 *   MAX_INFLIGHT      weight loads in flight per block (1..8).
 *   LOCAL_XQ          0: quantise x grid-wide even for M <= 16; 2: every
 *                     block quantises x itself also with RMSNorm (by
 *                     default only where M * H <= 16384).
 *   DECODE_PATH       M <= 128: 0 the grid-wide two-phase kernel, 1 the
 *                     cluster-sliced kernel (M <= 32), 2 the small-M kernel
 *                     (M <= 8, one block per 32 intermediate features and
 *                     per 16 output rows on the SMs, each block's weights
 *                     in shared memory).  Default: the small-M kernel where
 *                     it applies, else the grid-wide kernel.
 *   COOPERATIVE       1: launch the grid-wide kernel cooperatively instead
 *                     of as a plain launch that may start while the previous
 *                     kernel on the stream finishes.
 *   EARLY_W           M > 16: 1 (the default) lets the weight producer
 *                     fill its stages before x is available (PRIME loads in
 *                     flight), 0 holds it until the block's x loads are
 *                     issued.
 *   ALIGNED           split phases: 1 gives each block K stages of one tile
 *                     only, 0 the even split over all tiles' stages.
 *   ATTN_CHUNKS       paged decode attention: 128-token chunks per work
 *                     item (8 by default; the workspace size depends on it:
 *                     query it again after a change). */
typedef enum {
  FSOPS_KNOB_TR0 = 0,
  FSOPS_KNOB_TR1 = 1,
  FSOPS_KNOB_WHOLE_TILES = 2,
  FSOPS_KNOB_PAIRS = 3,
  FSOPS_KNOB_GEMM_FORM = 4,
  FSOPS_KNOB_PRIME = 5,
  FSOPS_KNOB_MAX_INFLIGHT = 6,
  FSOPS_KNOB_LOCAL_XQ = 7,
  FSOPS_KNOB_DECODE_PATH = 8,
  FSOPS_KNOB_COOPERATIVE = 9,
  FSOPS_KNOB_EARLY_W = 10,
  FSOPS_KNOB_ALIGNED = 11,
  FSOPS_KNOB_ATTN_CHUNKS = 12,
  FSOPS_KNOB_COUNT = 13
} fsops_knob;

/* Set knob `knob` (an fsops_knob) to `value` (negative = back to the
 * default).  INVALID_ARG for an unknown knob. */
fsops_status fsops_debug_set_knob(int knob, int value);

const char* fsops_status_string(fsops_status s);

/* The CUDA runtime error (a cudaError_t value) behind the last
 * FSOPS_ERR_CUDA that a call on this thread returned, 0 if none.  With the
 * environment variable FSOPS_VERBOSE set, each such failure is also printed
 * to stderr with the step that failed. */
int fsops_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int fsops_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FSOPS_H */
