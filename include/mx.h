/*
 * mx.h -- C ABI of the GB300 (sm_103a) OCP-MX training-MLP library.
 *
 * The hot path of a microscaling (MX) mixture-of-experts / dense MLP
 * training step: block-of-32 quantization with E8M0 round-up scales, ragged
 * grouped block-scaled GEMMs on the 5th-generation tensor core with fused
 * SwiGLU / dSwiGLU epilogues that requantize from on-chip memory, and the
 * ragged-K weight-gradient GEMM.
 *
 * Sources (web pages, cited by title and passage):
 *   [MXFP8-PR]  torchao PR #5 "MXFP8 cudnn-fe Swiglu fused Grouped MLP
 *               fwd/bwd and wgrad group gemm" -- shared-infrastructure commit,
 *               correctness-first kernels commit, cudnn-fe ops commit,
 *               validation-memoization commit, hardening commit.
 *   [MXFP6-PR]  Primus PR #1064 "feat(mxfp6): MXFP6 (E2M3) Flux linears, a
 *               fused MLP, and the MLPerf recipe" -- first commit, fused-MLP
 *               commit, bias commits.
 *   [MXFP4-guide] ROCm Primus guide "MXFP4 training for Flux models",
 *               Overview.
 *   [PERMUTE-PR] Primus PR #1247 "Qwen3-30B-A3B FP8 on MI355X to 40k
 *               tokens/s/GPU" -- DeepEP permute section (tokens quantized
 *               as part of the permute; the un-permute's backward returns a
 *               quantized gradient).
 *
 * Common conventions
 *   - Every pointer named *_dev or held in an mx_tensor_t is DEVICE memory of
 *     the current CUDA device; nothing here allocates or frees device memory.
 *     The caller owns every input, output and workspace buffer.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  No call synchronises the host except
 *     mx_get_device_status and, when the environment variable
 *     MX_VALIDATE_OFFSETS=1 is set, the offsets value check ([MXFP8-PR]
 *     cudnn-fe ops commit: opt-in value checks that need a sync).
 *   - Errors: arguments are validated on the host before anything is
 *     launched.  On failure nothing is launched, the call returns a status
 *     and mx_last_error() returns a message naming the argument (per calling
 *     thread).  There is no fallback path: an unsupported combination is an
 *     error, never a slower route.
 *   - Device: compute capability 10.3 (GB300) only; anything else returns
 *     MX_ERR_UNSUPPORTED_DEVICE.
 *   - All device pointers must be 16-byte aligned ([MXFP8-PR] hardening
 *     commit: 16-byte data_ptr gate).
 */
#ifndef MX_H_
#define MX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MX_ABI_VERSION 1

#if defined(__GNUC__)
#define MX_API __attribute__((visibility("default")))
#else
#define MX_API
#endif

typedef struct CUstream_st *mx_stream_t; /* identical to cudaStream_t */

/* Element formats ([MXFP8-PR]: E4M3; [MXFP6-PR]: E2M3; [MXFP4-guide]: E2M1).
 * Payload packing: E4M3 one byte per element; E2M3 four elements per three
 * bytes, element i at bits [6i, 6i+6) of the little-endian 24-bit group;
 * E2M1 two per byte, even element in the low nibble. */
typedef enum { MX_E4M3 = 0, MX_E2M3 = 1, MX_E2M1 = 2 } mx_fmt_t;

typedef enum {
  MX_OK = 0,
  MX_ERR_INVALID_ARG = 1,        /* null pointer, bad enum, G == 0, ... */
  MX_ERR_SHAPE = 2,              /* dimension not a required multiple / mismatched */
  MX_ERR_ALIGNMENT = 3,          /* pointer or leading dimension not 16-byte aligned */
  MX_ERR_OFFSETS = 4,            /* offsets failed the opt-in value check */
  MX_ERR_UNSUPPORTED_DEVICE = 5, /* not a compute capability 10.3 device */
  MX_ERR_CUDA = 6,               /* a CUDA runtime / driver call failed */
  MX_ERR_DEVICE_TIMEOUT = 7,     /* a bounded on-device wait expired (see mx_get_device_status) */
  MX_ERR_WORKSPACE = 8,          /* workspace missing or too small */
  MX_ERR_NOT_SUPPORTED = 9       /* valid request outside what this build implements */
} mx_status_t;

/* A quantized MX tensor: logical [rows, cols], blocks of 32 run along cols.
 *   data   packed payload, row-major, mx_payload_bytes(rows, cols, fmt) bytes
 *   scale  E8M0 block scales (byte b = 2^(b-127), 0xFF = NaN block) in the
 *          blocked layout: scale (r, c) of the [rows, cols/32] scale matrix
 *          sits at ((r/128)*ceil(cols/128) + c/4)*512 + (r%32)*16 +
 *          ((r%128)/32)*4 + c%4, padding bytes zero; mx_scale_bytes() bytes.
 *          ([MXFP8-PR] shared-infrastructure commit: tcgen05 blocked-scale
 *          indexing with a constant 512-byte K stride per 128-row block.)
 *   hadamard  nonzero if each block carries the 32-point rotation.
 * A "columnwise" (32x1) quantization of a [R, C] tensor is stored as the
 * rowwise quantization of its transpose: an mx_tensor_t of shape [C, R]
 * whose scales are blocked over the whole [C, R/32] scale matrix
 * ([MXFP8-PR] shared-infrastructure commit: whole-matrix columnwise scales). */
typedef struct {
  void *data;
  uint8_t *scale;
  int64_t rows, cols;
  int32_t fmt;
  int32_t hadamard;
} mx_tensor_t;

/* mx_quantize flags */
enum { MX_ROWWISE = 1, MX_COLWISE = 2, MX_HADAMARD = 4, MX_COLSUM = 8 };

MX_API int mx_abi_version(void);
MX_API const char *mx_last_error(void);
MX_API const char *mx_status_string(mx_status_t status);

/* Sizes (bytes) of the payload and blocked scales of a [rows, cols] tensor. */
MX_API size_t mx_payload_bytes(int64_t rows, int64_t cols, int32_t fmt);
MX_API size_t mx_scale_bytes(int64_t rows, int64_t cols);
/* Workspace mx_quantize needs for `flags` on one [rows, cols] input. */
MX_API size_t mx_quantize_workspace_bytes(int64_t rows, int64_t cols, uint32_t flags);

/*
 * mx_quantize -- BF16 -> MX, rowwise and/or columnwise, in one pass.
 * [MXFP8-PR] shared-infrastructure commit (RCEIL E8M0, NaN-propagating
 * amax, rowwise 1x32 / columnwise 32x1); [MXFP6-PR] first and bias commits
 * (Hadamard folded into the packer; per-column sums for the bias gradient).
 *
 *   x_bf16     device BF16 [batch, rows, cols], row stride `ld` elements
 *              (ld >= cols, ld % 8 == 0); batches contiguous (stride rows*ld)
 *   fmt        element format
 *   flags      MX_ROWWISE | MX_COLWISE (at least one), optionally
 *              MX_HADAMARD (rotate each 32-block before quantizing) and
 *              MX_COLSUM (fp32 sum over rows of each column, of the
 *              unrotated input; needs MX_COLWISE and batch == 1)
 *   out_row    MX_ROWWISE: tensor [batch*rows, cols] of format fmt
 *   out_col    MX_COLWISE: tensor [batch*cols, rows] (per batch entry the
 *              transpose's rowwise quantization)
 *   colsum     MX_COLSUM: device fp32 [cols]
 *   workspace  MX_COLSUM: >= mx_quantize_workspace_bytes(rows, cols, flags)
 * Each 32-block's scale is the smallest power of two 2^e with
 * amax <= emax * 2^e (emax = 448 / 7.5 / 6); elements are x * 2^-e rounded
 * to nearest-even and saturated; amax == 0 -> 0x00, amax == Inf -> 0xFE,
 * NaN in the block -> 0xFF with every element code NaN (E4M3 0x7F) or +0.
 * Shapes: cols % 32 == 0; MX_COLWISE also rows % 32 == 0; batch > 1 needs
 * rows % 128 == 0 and cols % 128 == 0.  rows == 0: MX_OK; nothing is
 * quantized, and with MX_COLSUM colsum is set to zero (the sum over no
 * rows; the workspace may then be NULL).  Sizes past rows * batch < 2^31
 * or rows * batch * ld < 2^40 elements: MX_ERR_SHAPE.
 */
MX_API mx_status_t mx_quantize(const void *x_bf16, int64_t batch, int64_t rows, int64_t cols, int64_t ld,
                        int32_t fmt, uint32_t flags, const mx_tensor_t *out_row, const mx_tensor_t *out_col,
                        float *colsum, void *workspace, size_t workspace_bytes, mx_stream_t stream);

/*
 * mx_quantize_sr -- mx_quantize with stochastic rounding of the elements,
 * for gradients in E2M3 or E2M1 (ROCm Primus guide "MXFP4 training for Flux
 * models", knob semantics: optional stochastic rounding of the FP4 gradient
 * quantization; the guide names the option only, the rule below is our
 * reading).  Scales stay RCEIL.  Each scaled element a rounds to the lower
 * grid neighbour lo or to lo + spacing, the latter when (u >> 8) < frac *
 * 2^24 with frac = (|a| - lo) / spacing (exact), so E[result] = a; values
 * on the grid and beyond the largest finite value are deterministic.  u is
 * the 32-bit word idx % 4 of Philox4x32-10 (Salmon et al., SC 2011) at
 * counter (idx / 4 as two words, orientation, 0) with key (the seed's two
 * words), where idx is the element's row-major position in its output grid
 * ([batch*rows, cols] rowwise, orientation 0; [batch*cols, rows]
 * columnwise, orientation 1).  Same seed, same bytes.
 *   seed      the generator key
 *   other arguments as mx_quantize; flags MX_ROWWISE / MX_COLWISE /
 *   MX_HADAMARD
 * Errors as mx_quantize, plus MX_ERR_NOT_SUPPORTED for E4M3 or MX_COLSUM.
 */
MX_API mx_status_t mx_quantize_sr(const void *x_bf16, int64_t batch, int64_t rows, int64_t cols, int64_t ld,
                                  int32_t fmt, uint32_t flags, uint64_t seed, const mx_tensor_t *out_row,
                                  const mx_tensor_t *out_col, mx_stream_t stream);

/*
 * Token permute for the expert MLP ([PERMUTE-PR]).  Routed rows are grouped
 * by expert, experts ascending; within an expert in (token, choice) order;
 * each expert's segment is padded with empty rows to a multiple of 128 (the
 * grouped GEMMs' segment alignment).  An empty row has source -1 and is
 * all zeros.  Readings of ours where the page is silent: that order, the
 * padding, and -1 for empty rows.
 *
 * mx_moe_route_rows -- the routed-row capacity R_cap to allocate for T
 * tokens, k choices and G experts: T*k + 127*G rounded up to 128 (every
 * padded routing fits).  Negative arguments give 0.
 * mx_moe_route_workspace_bytes -- device workspace of mx_moe_route_index.
 */
MX_API int64_t mx_moe_route_rows(int64_t T, int32_t k, int32_t G);
MX_API size_t mx_moe_route_workspace_bytes(int64_t T, int32_t k, int32_t G);

/*
 * mx_moe_route_index -- the routing index from the router's choices.
 *   topk_dev     int32 [T, k]: expert id of each (token, choice), in [0, G)
 *   offsets_dev  out int32 [G]: cumulative padded segment ends (the grouped
 *                GEMMs' offsets); offsets[G-1] routed rows are in use
 *   src_dev      out int32 [R_cap]: source token of each routed row, -1 for
 *                an empty row (also every row from offsets[G-1] on)
 *   row_of_dev   out int32 [T, k]: routed row of each (token, choice), -1
 *                for an out-of-range expert id
 *   workspace    >= mx_moe_route_workspace_bytes(T, k, G) bytes
 * Deterministic (a stable counting sort, no order-dependent atomics); three
 * launches.  Expert ids outside [0, G) are skipped and reported as
 * MX_ERR_INVALID_ARG by mx_get_device_status.
 * Errors: MX_ERR_INVALID_ARG (null pointer, k < 1, G < 1 or G > 1024),
 * MX_ERR_SHAPE (R_cap < mx_moe_route_rows(T, k, G)), MX_ERR_WORKSPACE.
 */
MX_API mx_status_t mx_moe_route_index(const int32_t *topk_dev, int64_t T, int32_t k, int32_t G, int32_t *offsets_dev,
                                      int32_t *src_dev, int64_t R_cap, int32_t *row_of_dev, void *workspace,
                                      size_t workspace_bytes, mx_stream_t stream);

/*
 * mx_moe_route_rows_pad / mx_moe_route_index_pad -- the same with each
 * expert's segment padded to a multiple of `pad` rows, pad = 128 or 256
 * (256: the segment alignment the CTA-pair grouped GEMM needs, the torchao
 * PR #5 page's cudnn-fe ops commit: 256-row alignment for its kernels).
 * mx_moe_route_rows_pad gives T*k + (pad-1)*G rounded up to pad (0 for a
 * pad other than 128 or 256); mx_moe_route_index_pad returns
 * MX_ERR_INVALID_ARG for another pad, else behaves as mx_moe_route_index.
 */
MX_API int64_t mx_moe_route_rows_pad(int64_t T, int32_t k, int32_t G, int32_t pad);
MX_API mx_status_t mx_moe_route_index_pad(const int32_t *topk_dev, int64_t T, int32_t k, int32_t G, int32_t pad,
                                          int32_t *offsets_dev, int32_t *src_dev, int64_t R_cap,
                                          int32_t *row_of_dev, void *workspace, size_t workspace_bytes,
                                          mx_stream_t stream);

/*
 * mx_permute_quantize -- the quantizing permute: routed row r of the output
 * is the MX quantization of token src[r] of x (a zero row where src[r] <
 * 0), rowwise and/or columnwise, in one pass over the tokens with no
 * permuted BF16 copy.  The rowwise bytes equal the gathered rowwise
 * quantization of the tokens (blocks lie in one row); the columnwise blocks
 * are 32 consecutive routed rows, as the wgrad needs them.  Used for X
 * before FC1 and for dY after the un-permute's backward (a gather of the
 * tokens' gradient with unit weights).
 *   x_bf16       device BF16 [T, D], row stride ld elements (ld % 8 == 0)
 *   src_dev      int32 [R_cap] (from mx_moe_route_index)
 *   offsets_dev  int32 [G]: rows from offsets[G-1] on are not written (NULL:
 *                all R_cap rows are)
 *   fmt, flags   element format; MX_ROWWISE and/or MX_COLWISE only
 *   out_row      MX_ROWWISE: tensor [R_cap, D]
 *   out_col      MX_COLWISE: tensor [D, R_cap]
 * Shapes: D % 32 == 0, R_cap % 128 == 0.  A source index >= T is read as an
 * empty row and reported as MX_ERR_INVALID_ARG by mx_get_device_status.
 */
MX_API mx_status_t mx_permute_quantize(const void *x_bf16, int64_t T, int64_t D, int64_t ld, const int32_t *src_dev,
                                       int64_t R_cap, const int32_t *offsets_dev, int32_t G, int32_t fmt,
                                       uint32_t flags, const mx_tensor_t *out_row, const mx_tensor_t *out_col,
                                       mx_stream_t stream);

/*
 * mx_moe_unpermute -- out[t] = sum over j of w[t, j] * in[row_of[t, j]]
 * (w = 1 when weights_dev is NULL; choices with row -1 skipped): the
 * combine of the experts' outputs, and the backward of the permute (dX of
 * the tokens from dX of the routed rows).  fp32 accumulation in choice
 * order, one rounding to BF16.
 *   in_bf16      device BF16 [R, D], contiguous rows
 *   row_of_dev   int32 [T, k]
 *   weights_dev  fp32 [T, k] or NULL
 *   out_bf16     device BF16 [T, D], contiguous rows
 * Shapes: D % 8 == 0.  A row index >= R is skipped and reported as
 * MX_ERR_INVALID_ARG by mx_get_device_status.
 */
MX_API mx_status_t mx_moe_unpermute(const void *in_bf16, int64_t R, int64_t D, const int32_t *row_of_dev,
                                    const float *weights_dev, int64_t T, int32_t k, void *out_bf16,
                                    mx_stream_t stream);

/*
 * mx_quantize_colsum_noalloc -- mx_quantize with MX_COLSUM for callers that
 * cannot allocate device memory: a framework hook that runs under a memory
 * pool it may not grow, or an embedding that owns all device memory up
 * front.  The
 * per-tile column-sum partials, which mx_quantize keeps in the caller's
 * workspace, live here in a fixed scratch array inside this library instead
 * (MX_NOALLOC_COLSUM_MAX_PARTIALS fp32 values = 8 MiB, held by every GPU that
 * loads the library until the process exits).  The call allocates nothing.
 * No passage of the pages corresponds to it: it is a deployment variant.
 *   Arguments as mx_quantize with batch = 1 and no workspace; flags must
 *   include MX_COLSUM and MX_COLWISE.
 *   Limit: ceil(rows / 128) * cols <= MX_NOALLOC_COLSUM_MAX_PARTIALS, else
 *   MX_ERR_WORKSPACE (use mx_quantize with a workspace).
 *   The first call on a device looks up the scratch's device address
 *   (cudaGetSymbolAddress, a host-side query), later calls reuse it.
 *   Every call shares the scratch: the partials are fully rewritten by each
 *   call before they are read, so nothing needs clearing, but calls whose
 *   execution overlaps on the GPU (different streams, no ordering) race on
 *   it and must be serialised by the caller.
 */
#define MX_NOALLOC_COLSUM_MAX_PARTIALS (1u << 21)
MX_API mx_status_t mx_quantize_colsum_noalloc(const void *x_bf16, int64_t rows, int64_t cols, int64_t ld,
                                              int32_t fmt, uint32_t flags, const mx_tensor_t *out_row,
                                              const mx_tensor_t *out_col, float *colsum, mx_stream_t stream);

/*
 * Offsets (all grouped calls): device int32 [G], cumulative END offsets of
 * each expert's row segment, nondecreasing, each a multiple of 128,
 * offsets[G-1] <= R.  Rows in [offsets[G-1], R) are neither read nor
 * written (caller-allocated outputs keep their contents there).  An empty
 * segment is allowed; with G == 1 a NULL offsets means one segment of all R
 * rows.  ([MXFP8-PR] shared-infrastructure commit: per-expert
 * row counts are multiples of 128, so no tile straddles an expert and the
 * expert of a tile follows from its row base; cudnn-fe ops commit: rows past
 * offsets[-1] are untouched in caller-allocated outputs.)  Values are not
 * checked on the host unless MX_VALIDATE_OFFSETS=1; the kernels skip a tile
 * whose segment is malformed and report MX_ERR_OFFSETS through
 * mx_get_device_status.  G == 0 is MX_ERR_INVALID_ARG.
 */

/*
 * mx_grouped_gemm -- out[r, n] = sum_k A[r, k] * B[g(r)][n, k] in fp32,
 * stored as BF16 (round to nearest even).  The plain grouped GEMM on
 * prequantized operands (FC2 forward, FC1 dgrad; [MXFP8-PR] cudnn-fe ops
 * commit, grouped mm with b [G, N, K] blocked along K).
 *   a         [R, K] rowwise MX (blocks along K)
 *   b         [G*N, K] rowwise MX; expert g owns rows [g*N, (g+1)*N)
 *   out_bf16  device BF16 [R, ld_out], ld_out >= N, ld_out % 8 == 0
 * K % 128 == 0, N % 128 == 0, same format and rotation on both operands.
 */
MX_API mx_status_t mx_grouped_gemm(const mx_tensor_t *a, const mx_tensor_t *b, int32_t G, const int32_t *offsets_dev,
                            void *out_bf16, int64_t ld_out, mx_stream_t stream);

/*
 * mx_grouped_gemm_2sm -- mx_grouped_gemm on CTA pairs: two SMs take a
 * 256 x 256 output tile with tcgen05 .cta_group::2 MMAs (M = 256), each SM
 * loading its 128 rows of A and half of the tile's B slice ([MXFP8-PR]
 * cudnn-fe ops commit: 256-row MMA tiles and 256-row segment alignment).
 * Same arguments and output as mx_grouped_gemm, with:
 *   a, b     E4M3, E2M3 (.kind::mxf8f6f4, K = 32 per MMA) or packed E2M1
 *            (.kind::mxf4, K = 64 per MMA; ROCm Primus guide "MXFP4
 *            training for Flux models", backends section: FP4 GEMMs at
 *            twice the FP8 rate); N = b->rows / G a multiple of 256 (else
 *            MX_ERR_SHAPE)
 *   offsets  segments multiples of 128 rows, as for mx_grouped_gemm; each
 *            expert's rows are taken in 256-row tiles, and an expert with an
 *            odd number of 128-row blocks computes its last tile's upper
 *            half and discards it (no wasted half with 256-row segments:
 *            mx_moe_route_index_pad with pad 256).  A malformed segment is
 *            skipped on the device and reported as MX_ERR_OFFSETS by
 *            mx_get_device_status.  G <= 1024 (else MX_ERR_NOT_SUPPORTED).
 *            NULL: one segment of all R rows.
 * The products and their fp32 accumulation are those of mx_grouped_gemm
 * (bit-identical outputs).  A warp of the leader CTA copies each stage's
 * scale chunks into tensor memory, so the MMA thread issues only MMAs.
 */
MX_API mx_status_t mx_grouped_gemm_2sm(const mx_tensor_t *a, const mx_tensor_t *b, int32_t G,
                                       const int32_t *offsets_dev, void *out_bf16, int64_t ld_out,
                                       mx_stream_t stream);

/*
 * mx_grouped_gemm_bias -- mx_grouped_gemm with a per-expert bias added to
 * the fp32 accumulator before the single BF16 rounding ([MXFP6-PR] bias
 * commits: the bias add belongs in the GEMM's store epilogue; here each
 * expert has its own row).
 *   bias_bf16   device BF16 [G, N] (row g for the rows of segment g),
 *               16-byte aligned
 * Other arguments, shapes and errors as mx_grouped_gemm.
 */
MX_API mx_status_t mx_grouped_gemm_bias(const mx_tensor_t *a, const mx_tensor_t *b, int32_t G,
                                        const int32_t *offsets_dev, const void *bias_bf16, void *out_bf16,
                                        int64_t ld_out, mx_stream_t stream);

/*
 * mx_grouped_gemm_bias_2sm -- mx_grouped_gemm_bias on CTA pairs: the bias
 * row of the expert added to the fp32 accumulator before the single BF16
 * rounding, as in mx_grouped_gemm_bias (bit-identical outputs); shapes,
 * offsets and errors as mx_grouped_gemm_2sm.
 *   bias_bf16   device BF16 [G, N], 16-byte aligned
 */
MX_API mx_status_t mx_grouped_gemm_bias_2sm(const mx_tensor_t *a, const mx_tensor_t *b, int32_t G,
                                            const int32_t *offsets_dev, const void *bias_bf16, void *out_bf16,
                                            int64_t ld_out, mx_stream_t stream);

/*
 * mx_grouped_gemm_swiglu_fwd -- FC1 of the expert MLP with the SwiGLU
 * epilogue ([MXFP8-PR] correctness-first kernels commit: FC1 ragged grouped
 * GEMM + SwiGLU + dual 1x32 / 32x1 MXFP8 RCEIL quantization + BF16
 * pre-activation save, one launch).
 *   x_row     [R, D] rowwise E4M3
 *   w1_row    [G*2F, D] rowwise E4M3: expert g's rows [g*2F, g*2F+F) are the
 *             gate projection, [g*2F+F, (g+1)*2F) the up projection
 *   z_bf16    out, device BF16 [R, 2F] = [gate | up] pre-activation
 *   h_row     out, [R, F] rowwise E4M3 of h = gate * sigmoid(gate) * up
 *   h_col     out, [F, R] columnwise E4M3 of h
 * D % 128 == 0, F % 128 == 0, R % 128 == 0.  h is computed in fp32 from the
 * fp32 accumulators; sigmoid(x) = 1 / (1 + exp(-x)).  Runs on CTA pairs
 * (256-row tiles per expert, tcgen05 .cta_group::2) for G <= 1024 unless the
 * environment holds MX_FUSED_PAIRS=0 (one SM per 128-row tile); the output
 * bytes are the same either way.
 */
MX_API mx_status_t mx_grouped_gemm_swiglu_fwd(const mx_tensor_t *x_row, const mx_tensor_t *w1_row, int32_t G,
                                       const int32_t *offsets_dev, const mx_tensor_t *h_row,
                                       const mx_tensor_t *h_col, void *z_bf16, mx_stream_t stream);

/*
 * mx_grouped_gemm_dswiglu_bwd -- FC2 dgrad with the dSwiGLU epilogue
 * ([MXFP8-PR] correctness-first kernels commit: FC2 dgrad grouped GEMM +
 * dSwiGLU + dual quantization, one launch).
 *   dy_row    [R, D] rowwise E4M3 of the output gradient
 *   w2t_row   [G*F, D] rowwise E4M3 of each expert's W2^T (W2 is [D, F])
 *   z_bf16    device BF16 [R, 2F], the saved pre-activation
 *   dz_row    out, [R, 2F] rowwise E4M3 of dz = [dg | du]
 *   dz_col    out, [2F, R] columnwise E4M3 of dz
 * with dh = dY W2: dg = dh*u*s*(1 + g*(1-s)), du = dh*g*s, s = sigmoid(g),
 * g and u read from the BF16 z.  D % 128 == 0, F % 128 == 0, R % 128 == 0.
 * With MX_FUSED_PAIRS=1 in the environment and F % 256 == 0 it runs on CTA
 * pairs (its epilogue, not its mainloop, is the limit, so by default it
 * takes one SM per tile); the output bytes are the same either way.
 */
MX_API mx_status_t mx_grouped_gemm_dswiglu_bwd(const mx_tensor_t *dy_row, const mx_tensor_t *w2t_row,
                                        const void *z_bf16, int32_t G, const int32_t *offsets_dev,
                                        const mx_tensor_t *dz_row, const mx_tensor_t *dz_col,
                                        mx_stream_t stream);

/*
 * Routing probabilities fused into the activation (Primus PR #1247
 * "Qwen3-30B-A3B FP8 on MI355X to 40k tokens/s/GPU": the fused activation
 * with probabilities, which scales each routed row by its routing weight
 * before FC2 instead of after it).
 * mx_grouped_gemm_swiglu_probs_fwd -- mx_grouped_gemm_swiglu_fwd with
 *   h[r, :] = swiglu(g, u)[r, :] * probs[r] before both requants (z is
 *   saved unscaled).  probs: device fp32 [R], 16-byte aligned.
 * mx_grouped_gemm_dswiglu_probs_bwd -- the matching backward: the
 *   activation gradient is dh * probs[r]; dprobs[r] = sum over f of
 *   dh[r, f] * swiglu(g, u)[r, f] for the rows of the segments (rows past
 *   offsets[G-1] untouched), summed in a fixed order (deterministic).
 *   dprobs: device fp32 [R]; workspace: at least
 *   mx_dswiglu_probs_workspace_bytes(R, F) bytes for per-tile partial sums.
 *   Errors as mx_grouped_gemm_dswiglu_bwd, plus MX_ERR_WORKSPACE.
 */
MX_API mx_status_t mx_grouped_gemm_swiglu_probs_fwd(const mx_tensor_t *x_row, const mx_tensor_t *w1_row, int32_t G,
                                                    const int32_t *offsets_dev, const float *probs,
                                                    const mx_tensor_t *h_row, const mx_tensor_t *h_col,
                                                    void *z_bf16, mx_stream_t stream);
MX_API size_t mx_dswiglu_probs_workspace_bytes(int64_t R, int64_t F);
MX_API mx_status_t mx_grouped_gemm_dswiglu_probs_bwd(const mx_tensor_t *dy_row, const mx_tensor_t *w2t_row,
                                                     const void *z_bf16, const float *probs, int32_t G,
                                                     const int32_t *offsets_dev, const mx_tensor_t *dz_row,
                                                     const mx_tensor_t *dz_col, float *dprobs, void *workspace,
                                                     size_t workspace_bytes, mx_stream_t stream);

/*
 * mx_grouped_gemm_wgrad -- ragged-K weight gradient, BF16 out ([MXFP8-PR]
 * correctness-first kernels commit: generic ragged-K grouped wgrad, BF16
 * out; shared-infrastructure commit: zero-token experts give zeros).
 *   a_col     [N, R] columnwise operand (e.g. dY: [D, R])
 *   b_col     [K, R] columnwise operand (e.g. h: [F, R])
 *   out_bf16  device BF16 [G, N, K]: out[g, n, k] = sum over rows r of
 *             segment g of a_col[n, r] * b_col[k, r]; an empty segment
 *             writes exact zeros
 * N % 128 == 0, K % 128 == 0, R % 128 == 0.  out_bf16 may be the caller's
 * BF16 main-grad buffer itself: the gradient is stored there with no
 * separate gradient tensor and no add (Primus PR #1064 "feat(mxfp6): MXFP6
 * (E2M3) Flux linears, a fused MLP, and the MLPerf recipe", the commit that
 * writes wgrad into main_grad: a beta = 0 store, one microbatch per step).
 * With MX_FUSED_PAIRS=1 in the environment and N, K multiples of 256 (this
 * and the other weight-gradient calls) it runs on CTA pairs; the output
 * bytes are the same either way.
 */
MX_API mx_status_t mx_grouped_gemm_wgrad(const mx_tensor_t *a_col, const mx_tensor_t *b_col, int32_t G,
                                  const int32_t *offsets_dev, void *out_bf16, mx_stream_t stream);

/*
 * mx_grouped_gemm_wgrad_f32 -- the same weight gradient into a caller's
 * fp32 gradient buffer (the main-grad of mixed-precision training).  The
 * page's store overwrites, so it fits one microbatch per optimizer step;
 * accumulate = 1 is our extension for several microbatches (a beta = 1
 * variant).
 *   a_col, b_col, G, offsets_dev   as mx_grouped_gemm_wgrad
 *   grad_f32    device fp32 [G, N, K], 16-byte aligned
 *   accumulate  0: grad = a_col^T b_col per expert (an empty segment
 *               stores zeros); 1: grad += that product, one fp32 rounding
 *               per element (an empty segment leaves grad unchanged).
 *               Each element is written by exactly one tile, so the result
 *               does not depend on scheduling.
 * Errors: MX_ERR_INVALID_ARG if accumulate is not 0 or 1; otherwise as
 * mx_grouped_gemm_wgrad.
 */
MX_API mx_status_t mx_grouped_gemm_wgrad_f32(const mx_tensor_t *a_col, const mx_tensor_t *b_col, int32_t G,
                                             const int32_t *offsets_dev, float *grad_f32, int32_t accumulate,
                                             mx_stream_t stream);

/*
 * K-split of the largest experts' weight gradients (load balance under
 * skewed routing).  mx_grouped_gemm_wgrad_ws / _f32_ws are
 * mx_grouped_gemm_wgrad / _f32 with a workspace: experts whose token count
 * exceeds a split size (chosen from N, K, R and the SM count, in 128-token
 * chunks) have each output tile's K range cut into parts; every part writes
 * an fp32 partial tile to the workspace, and the part that completes the
 * tile's arrival counter sums all parts in part order and stores the tile
 * (BF16, or fp32 store / accumulate).  Deterministic: the same bits whichever
 * part finishes last; the sum order differs from the unsplit call's, so the
 * two agree to fp32 rounding, not bit for bit.  At most 16 experts are
 * split; with offsets NULL, G == 1, G > 1024 or a NULL workspace nothing is.
 * In the same cases the CTAs also claim output tiles (split parts first,
 * then experts by descending token count) from a counter in the workspace
 * instead of taking a fixed share; each tile is still computed by one CTA,
 * so with nothing split the result equals mx_grouped_gemm_wgrad's bit for
 * bit.
 * mx_grouped_gemm_wgrad_workspace_bytes(N, K, R, G) -- bytes for [N, K]
 * gradients over R routed rows (0: no split possible); N = a_col rows,
 * K = b_col rows.  The workspace starts with counters the call clears
 * itself (one memset per call, before its launch); its contents need no
 * preparation by the caller.
 * Errors as mx_grouped_gemm_wgrad / _f32, plus MX_ERR_WORKSPACE when a
 * non-NULL workspace is smaller than the query's bytes.
 */
MX_API size_t mx_grouped_gemm_wgrad_workspace_bytes(int64_t N, int64_t K, int64_t R, int32_t G);
MX_API mx_status_t mx_grouped_gemm_wgrad_ws(const mx_tensor_t *a_col, const mx_tensor_t *b_col, int32_t G,
                                            const int32_t *offsets_dev, void *out_bf16, void *workspace,
                                            size_t workspace_bytes, mx_stream_t stream);
MX_API mx_status_t mx_grouped_gemm_wgrad_f32_ws(const mx_tensor_t *a_col, const mx_tensor_t *b_col, int32_t G,
                                                const int32_t *offsets_dev, float *grad_f32, int32_t accumulate,
                                                void *workspace, size_t workspace_bytes, mx_stream_t stream);

/*
 * Dense (single-segment) calls of the MXFP6 Flux-style MLP ([MXFP6-PR]
 * fused-MLP commit: one unit owns fc1 -> activation -> fc2, the packer takes
 * the activation as an epilogue in the forward and its derivative in the
 * backward, the pre-activation gradient is never assembled in BF16, the bias
 * gradient comes back as a per-column sum; bias commits: the bias is added in
 * the fp32 accumulator before one rounding).  M, K and the output width are
 * multiples of 128; operands of any MX format, both operands alike.
 */

/* out[m, n] = sum_k A[m, k] B[n, k] + bias[n] (fp32), stored as BF16.
 *   a [M, K], b [N, K] rowwise MX; bias_bf16 device BF16 [N] or NULL. */
MX_API mx_status_t mx_gemm_bias(const mx_tensor_t *a, const mx_tensor_t *b, const void *bias_bf16, void *out_bf16,
                                int64_t ld_out, mx_stream_t stream);

/* FC1 forward with the tanh-GELU epilogue.
 *   x_row [M, D], w1_row [H, D] rowwise MX; b1_bf16 device BF16 [H] or NULL
 *   pre_bf16  out, device BF16 [M, H] = x W1^T + b1 (the saved pre-activation)
 *   act_row   out, [M, H] rowwise MX of act = gelu_tanh(pre) (fp32 pre)
 *   act_col   out, [H, M] columnwise MX of act
 * act_row / act_col: format E4M3 or E2M3, same format and rotation flag on
 * both; with the rotation, each 32-block is rotated before packing. */
MX_API mx_status_t mx_gemm_gelu_fwd(const mx_tensor_t *x_row, const mx_tensor_t *w1_row, const void *b1_bf16,
                                    void *pre_bf16, const mx_tensor_t *act_row, const mx_tensor_t *act_col,
                                    mx_stream_t stream);

/* FC2 dgrad with the dGELU epilogue.
 *   dy_row [M, D] rowwise MX; w2t_row [H, D] rowwise MX of W2^T (W2 [D, H])
 *   pre_bf16  device BF16 [M, H] from mx_gemm_gelu_fwd
 *   dpre_row  out, [M, H] rowwise MX of dpre = (dY W2) * gelu_tanh'(pre)
 *   dpre_col  out, [H, M] columnwise MX of dpre
 *   db1       out, device fp32 [H] = sum over rows of dpre (fixed order)
 *   workspace >= mx_gemm_dgelu_workspace_bytes(M, H), 16-byte aligned */
MX_API size_t mx_gemm_dgelu_workspace_bytes(int64_t M, int64_t H);
MX_API mx_status_t mx_gemm_dgelu_bwd(const mx_tensor_t *dy_row, const mx_tensor_t *w2t_row, const void *pre_bf16,
                                     const mx_tensor_t *dpre_row, const mx_tensor_t *dpre_col, float *db1,
                                     void *workspace, size_t workspace_bytes, mx_stream_t stream);

/* Activation of mx_mlp_fwd_bwd. */
typedef enum { MX_ACT_SWIGLU = 0, MX_ACT_GELU_TANH = 1 } mx_act_t;

/*
 * Arguments of the whole MLP step.  BF16 inputs / outputs, device memory.
 *   x   [R, D]        dy  [R, D]       y  out [R, D]     dx out [R, D]
 *   SwiGLU: w1 [G, 2F, D] (gate rows then up rows per expert), w2 [G, D, F],
 *           dw1 out [G, 2F, D], dw2 out [G, D, F]; b1, b2, db1, db2 unused.
 *   workspace  >= mx_mlp_workspace_bytes(args); holds every quantized
 *              operand and the saved pre-activation between the stages.
 */
typedef struct {
  int32_t act;
  int32_t fmt;
  int32_t hadamard;
  int32_t G;
  int64_t R, D, F;
  const int32_t *offsets;
  const void *x, *w1, *w2, *dy, *b1, *b2;
  void *y, *dx, *dw1, *dw2;
  float *db1, *db2;
  void *workspace;
  size_t workspace_bytes;
} mx_mlp_args_t;

MX_API size_t mx_mlp_workspace_bytes(const mx_mlp_args_t *args);

/*
 * mx_mlp_workspace_layout -- where mx_mlp_fwd_bwd keeps its intermediates
 * inside the caller's workspace, so a caller (a test, a debugger) can read
 * the quantized operands each stage consumed after the step has run.  Not
 * part of the method: the pages' fused MLP keeps these between its stages
 * too, but says nothing of where.
 *   args  as for mx_mlp_workspace_bytes (pointers are not read)
 *   out   receives, for each quantized tensor, the byte offsets of its
 *         payload and of its blocked scales from the workspace start and
 *         its logical [rows, cols] (columnwise tensors are stored as the
 *         rowwise quantization of the transpose, so rows = the source's
 *         columns):
 *           x_row [R, D], x_col [D, R], w1_row [G*F1, D], w1t_row [G*D, F1],
 *           w2_row [G*D, F], w2t_row [G*F, D], h_row [R, F], h_col [F, R],
 *           dy_row [R, D], dy_col [D, R], dz_row [R, F1], dz_col [F1, R],
 *         F1 = 2F for SwiGLU (FC1's gate and up halves), F for GELU (where
 *         h is the activation and dz the pre-activation gradient);
 *         z: the BF16 [R, F1] pre-activation (SwiGLU z, GELU pre);
 *         total: mx_mlp_workspace_bytes(args).
 * Returns MX_ERR_INVALID_ARG for a NULL pointer or a malformed shape (the
 * cases where mx_mlp_workspace_bytes returns 0).
 */
typedef struct {
  size_t data, scale;
  int64_t rows, cols;
} mx_mlp_slot_t;

typedef struct {
  mx_mlp_slot_t x_row, x_col, w1_row, w1t_row, w2_row, w2t_row;
  mx_mlp_slot_t h_row, h_col, dy_row, dy_col, dz_row, dz_col;
  size_t z;
  size_t total;
} mx_mlp_layout_t;

MX_API mx_status_t mx_mlp_workspace_layout(const mx_mlp_args_t *args, mx_mlp_layout_t *out);

/*
 * mx_mlp_fwd_bwd -- one training step of the MX MLP on one stream:
 * quantize X, W1, W2 (rowwise and per-expert columnwise); FC1 + SwiGLU
 * (mx_grouped_gemm_swiglu_fwd); FC2 (mx_grouped_gemm); quantize dY; FC2
 * dgrad + dSwiGLU (mx_grouped_gemm_dswiglu_bwd); FC1 dgrad
 * (mx_grouped_gemm); dW2 and dW1 (mx_grouped_gemm_wgrad_ws: the largest
 * experts' K range split, with the split workspace inside `workspace`).
 * 10 kernel launches (plus one small memset of the split counters per
 * weight gradient when the routing has more than one expert).
 * ([MXFP8-PR] cudnn-fe ops commit: the four ops of the routed-expert MLP;
 * [MXFP6-PR] fused-MLP commit: owning fc1 -> activation -> fc2 in one unit.)
 */
MX_API mx_status_t mx_mlp_fwd_bwd(const mx_mlp_args_t *args, mx_stream_t stream);

/*
 * Host-buffer pipeline of the step.  A runtime convenience for callers whose
 * tensors live in host memory; the pages' kernels have no counterpart (they
 * take device tensors).  Each mx_mlp_pipeline_run enqueues one step of
 * mx_mlp_fwd_bwd whose inputs (x, w1, w2, dy, the routing offsets, and b1, b2
 * for GELU) are copied from host memory and whose outputs (y, dx, dw1, dw2,
 * and db1, db2 for GELU) are copied back, with the two copy directions on
 * streams of their own: the next step's input copy starts as soon as this
 * step's only reader of that input has run, an output's copy back starts as
 * soon as its writer has run, and the next step's writer waits for that copy.
 * Consecutive runs therefore overlap host traffic in both directions with
 * the kernels, using one device buffer per tensor.
 *
 * mx_mlp_pipeline_create
 *   dev     device buffers and workspace exactly as for mx_mlp_fwd_bwd
 *           (validated here; the pointed-to arrays are staging buffers the
 *           pipeline overwrites; dev->offsets receives each step's routing);
 *           copied, the caller keeps ownership of every buffer
 *   stream  the stream the step's kernels run on
 *   out     receives the pipeline; creates two copy streams and events, no
 *           device memory
 * mx_mlp_pipeline_run
 *   io      host pointers, same shapes and element types as the device
 *           tensors (BF16, fp32 for db1/db2, int32 offsets [G]); pinned host
 *           memory is needed for the copies to run asynchronously.  Host
 *           buffers are read and written after the call returns: keep them
 *           alive and unchanged (inputs) or unread (outputs) until
 *           mx_mlp_pipeline_sync.  w1, w2, dw1 and dw2 may be NULL: those
 *           tensors then stay resident in the device buffers (weights the
 *           caller keeps and updates on the device, gradients it consumes
 *           there), as in a training loop with the optimizer on the device.
 *           Returns MX_ERR_INVALID_ARG for another missing host buffer,
 *           MX_ERR_CUDA if enqueuing failed (later runs then fail too).
 * mx_mlp_pipeline_sync     wait for every enqueued step, copies included
 * mx_mlp_pipeline_destroy  sync, then release streams and events
 */
typedef struct mx_mlp_pipeline mx_mlp_pipeline_t;
typedef struct {
  const void *x, *w1, *w2, *dy, *b1, *b2;
  const int32_t *offsets;
  void *y, *dx, *dw1, *dw2;
  float *db1, *db2;
} mx_mlp_host_io_t;

MX_API mx_status_t mx_mlp_pipeline_create(const mx_mlp_args_t *dev, mx_stream_t stream, mx_mlp_pipeline_t **out);
MX_API mx_status_t mx_mlp_pipeline_run(mx_mlp_pipeline_t *p, const mx_mlp_host_io_t *io);
MX_API mx_status_t mx_mlp_pipeline_sync(mx_mlp_pipeline_t *p);
MX_API void mx_mlp_pipeline_destroy(mx_mlp_pipeline_t *p);

/*
 * mx_get_device_status -- synchronise `stream`, then report and clear the
 * device-side status words: MX_ERR_DEVICE_TIMEOUT if a bounded wait inside
 * a kernel expired (the kernel unwound; its outputs are undefined),
 * MX_ERR_OFFSETS if a kernel saw a malformed offsets segment, else MX_OK.
 */
MX_API mx_status_t mx_get_device_status(mx_stream_t stream);

/*
 * mx_selftest_bounded_wait -- launch a kernel whose wait nothing completes;
 * it gives up after `budget_ns` and records the timeout, so the next
 * mx_get_device_status returns MX_ERR_DEVICE_TIMEOUT.  Exercises the
 * timeout path without hanging or faulting the device.
 */
MX_API mx_status_t mx_selftest_bounded_wait(uint64_t budget_ns, mx_stream_t stream);

/*
 * mx_debug_tap -- test instrument, not part of the method.  While attached
 * (tap_f32 != NULL) on the calling host thread, every fused-requant
 * epilogue (mx_grouped_gemm_swiglu_fwd: h [R, F]; mx_grouped_gemm_dswiglu_bwd:
 * dz = [dg | du] [R, 2F]; mx_gemm_gelu_fwd: act [M, H]; mx_gemm_dgelu_bwd:
 * dpre [M, H]) also writes the fp32 values it is about to quantize, row-major,
 * before any rotation.  Quantizing those values exactly must reproduce the
 * epilogue's payload and scale bytes bit for bit, which is how the tests
 * check the fused requant on random data.  Rows of empty tiles are not
 * written.
 *   tap_f32  device fp32 buffer of `elems` floats, 16-byte aligned, owned by
 *            the caller; NULL detaches
 *   elems    capacity; a fused call whose output is larger fails with
 *            MX_ERR_SHAPE before launching
 * Costs one store per value when attached; nothing when detached.
 */
MX_API mx_status_t mx_debug_tap(float *tap_f32, int64_t elems);

#ifdef __cplusplus
}
#endif

#endif /* MX_H_ */
