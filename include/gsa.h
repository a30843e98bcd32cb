/*
 * gsa.h -- C ABI of libgsa: grouped scaled activation fused with
 * block-scaled quantization (MXFP8 / NVFP4), forward and backward, for the
 * step between the FC1 and FC2 grouped GEMMs of an MoE expert FFN.
 *
 * Defining passages (NVIDIA/TransformerEngine pull-request pages):
 *   "Activation + GroupedLinear Fusion for MOE" -- Greptile Summary: one
 *     kernel pass fuses the per-row scale multiply, the activation (SwiGLU,
 *     clamped SwiGLU, SReLU) and grouped quantization; sequence diagram:
 *     forward grouped_scaled_{swiglu,srelu}(x, scales, quantizer,
 *     split_sizes) -> grouped_x, backward grouped_scaled_d{swiglu,srelu}
 *     (grad, input_, scales, quantizer) -> (grouped_dy, dense_dy,
 *     grad_scales); the "Crash when fc1 is frozen" note (grad_scales must be
 *     computable without the fc1 gradient).
 *   "[PyTorch] Enable fused activation recompute for ScaledTanhSReLU" --
 *     Description: ScaledTanhSReLU (SReLU bounded at s^2), activation
 *     recompute regenerating FC2's input from the saved FC1 output, MXFP8
 *     and NVFP4 (RHT) recipes.
 *
 * Conventions for every entry point
 *   - All tensors are row-major, contiguous, little-endian, in DEVICE memory
 *     of the current CUDA device, 16-byte aligned.  split_sizes is a HOST
 *     array.  The caller owns every buffer, including the workspace; the
 *     library never allocates, frees or synchronizes (except
 *     gsa_workspace_status, which synchronizes the given stream).
 *   - Rows are grouped by expert in expert order: expert e owns rows
 *     [o_e, o_e + M_e), o_e = sum of split_sizes before e.  M = sum M_e.
 *   - W_in = width of X.  W = width of Y: W_in for the unary activations,
 *     W_in / 2 for the GLU activations (X[:, :W] is the gate side, X[:, W:]
 *     the linear side).  W must be a multiple of 64 (the kernel's column
 *     tile): a W that is a multiple of the block size but not of 64 returns
 *     GSA_ERR_UNSUPPORTED.  So does a W whose W / 64 tiles cannot be split
 *     into at most 64 equal groups of 1, 2, 4, 8, 16 or 32 tiles (e.g.
 *     W = 64 * 195); every W up to 4096, and every W = 64 * 2^k up to 131072,
 *     is supported.
 *   - Block size B = 32 (MXFP8) or 16 (NVFP4).  Mp_e = ceil(M_e / B) * B.
 *   - Quantized copies of a [M, N] tensor (N = W for Y, W_in for dX):
 *       rowwise   data  MXFP8 [M, N] E4M3 bytes; NVFP4 [M, N/2] bytes, two
 *                       E2M1 codes per byte (element 2k low nibble)
 *                 scale MXFP8 [M, N/32] E8M0; NVFP4 [M, N/16] E4M3
 *       columnwise, per expert e, experts concatenated in expert order:
 *                 data  MXFP8 [N, Mp_e]; NVFP4 [N, Mp_e/2]
 *                 scale [N, Mp_e/B]
 *                 = the rowwise quantization of the zero-padded transpose
 *                 of the expert's rows; NVFP4 columnwise 16-chunks first go
 *                 through the random Hadamard transform (1/4) H16 diag(d)
 *                 when rht_colwise != 0, d_i = -1 where bit i of
 *                 rht_sign_mask is set.
 *       NVFP4 only: amax_row[E] = max |value| of each expert, amax_col[E] =
 *                 max |columnwise chunk value| of each expert (after the
 *                 RHT).  The per-expert encode scale is S = 2688 / amax
 *                 (1 for amax 0, capped at FLT_MAX); a block's element
 *                 multiplier S / E4M3(scale code) is capped at FLT_MAX too.
 *   - Errors in arguments are detected on the host before anything is
 *     enqueued and leave all outputs untouched.  Launch failures return
 *     GSA_ERR_CUDA.  Device-side bounded waits that run out set an error
 *     word in the workspace that gsa_workspace_status reports.
 */
#ifndef GSA_H
#define GSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st *gsa_stream_t;

typedef enum {
    GSA_OK = 0,
    GSA_ERR_INVALID_ARG = 1,    /* bad pointer, size, split or flag */
    GSA_ERR_UNSUPPORTED = 2,    /* valid but outside what the kernels cover */
    GSA_ERR_ALIGNMENT = 3,      /* a pointer is not 16-byte aligned */
    GSA_ERR_WORKSPACE = 4,      /* workspace missing or too small */
    GSA_ERR_CUDA = 5,           /* a CUDA runtime / driver call failed */
    GSA_ERR_DEVICE_TIMEOUT = 6  /* a device-side bounded wait ran out */
} gsa_status;

typedef enum {
    GSA_ACT_SRELU = 0,          /* relu(x)^2 */
    GSA_ACT_TANH_SRELU = 1,     /* s^2 tanh^2(relu(x) / s), bounded by s^2 */
    GSA_ACT_SWIGLU = 2,         /* silu(a) * b */
    GSA_ACT_CLAMPED_SWIGLU = 3, /* a' sigmoid(alpha a') (b' + offset), a' = min(a, L), b' = clamp(b, -L, L) */
    /* Further unary activations through the same kernel (the ScaledTanhSReLU
     * recompute page, review thread: nothing in the fused kernel or in
     * recompute is special to SReLU; GeLU, sigmoid or any unary activation
     * would do).  Results within 2 BF16 ULP of the correctly evaluated FP32
     * formula for GELU / SIGMOID (library erfcf / expf); IDENTITY is exact. */
    GSA_ACT_GELU = 4,           /* x Phi(x) = (x/2) erfc(-x / sqrt 2): the erf form, not the tanh fit */
    GSA_ACT_SIGMOID = 5,        /* 1 / (1 + exp(-x)) */
    GSA_ACT_IDENTITY = 6        /* x: with probs = NULL the forward is a plain grouped quantizer of a
                                 * BF16 tensor (the second step of the unfused two-step path) */
} gsa_act_kind;

typedef struct {
    float s;                    /* TanhSReLU bound parameter (> 0) */
    float limit;                /* clamped SwiGLU limit L (> 0) */
    float alpha;                /* clamped SwiGLU sigmoid slope */
    float glu_linear_offset;    /* clamped SwiGLU offset added to the linear side */
} gsa_act_params;

typedef enum { GSA_MXFP8 = 0, GSA_NVFP4 = 1 } gsa_recipe_kind;

/* Layout of the block scales (the codes are laid out the same in both).
 *   GSA_SCALES_COMPACT: rowwise [M, width / B] row-major; columnwise, per
 *     expert, [width, Mp_e / B] row-major, experts one after another.
 *   GSA_SCALES_TILED: the operand layout of block-scaled GEMMs (cuBLASLt's
 *     1D block-scaling factor layout, which the grouped GEMM that consumes the
 *     quantized tensor takes: "Activation + GroupedLinear Fusion for MOE",
 *     Greptile Summary, the pre-quantized GroupedTensorStorage handed to the
 *     GEMM; the scales are "handed to cuBLASLt", "Preserve FP8 recompute state
 *     for inner autocast", How much it costs).  Each expert's scale matrix
 *     ([M_e, width / B] rowwise, [width, Mp_e / B] columnwise) is padded to
 *     whole tiles of 128 rows x 4 columns, 512 bytes each, stored in row-major
 *     tile order; inside a tile, entry (r, c) sits at byte
 *     16 (r mod 32) + 4 floor(r / 32) + c.  The experts' tile blocks follow
 *     one another (offsets from gsa_layout_ex).  Padding entries are not
 *     written. */
typedef enum { GSA_SCALES_COMPACT = 0, GSA_SCALES_TILED = 1 } gsa_scale_layout;

typedef struct {
    int32_t kind;               /* gsa_recipe_kind */
    int32_t rht_colwise;        /* NVFP4: apply the 16-point RHT to the columnwise copy */
    uint32_t rht_sign_mask;     /* low 16 bits used */
    int32_t scale_layout;       /* gsa_scale_layout (0: compact) */
} gsa_recipe;

/* One quantized tensor.  Any member may be NULL to skip that part:
 * row_data/row_scale (both or neither) = rowwise copy, col_data/col_scale
 * (both or neither) = columnwise copy.  For NVFP4 amax_row is required with
 * the rowwise copy and amax_col with the columnwise copy ([E] floats). */
typedef struct {
    void *row_data;
    void *row_scale;
    void *col_data;
    void *col_scale;
    float *amax_row;
    float *amax_col;
} gsa_qout;

/* Byte sizes of the quantized copies of a [M, width] tensor. */
typedef struct {
    int64_t rows;               /* M */
    int64_t row_data_bytes;
    int64_t row_scale_bytes;
    int64_t col_data_bytes;
    int64_t col_scale_bytes;
    int64_t amax_floats;        /* E (NVFP4) or 0 */
} gsa_layout_info;

/* Layout of the quantized copies of a grouped [M, width] tensor.
 * col_data_offsets / col_scale_offsets (each E+1 entries, may be NULL)
 * receive the byte offset of each expert's columnwise block.
 * Errors: INVALID_ARG (E <= 0, NULL split_sizes, negative size,
 * width % B != 0, unknown recipe). */
gsa_status gsa_layout(int64_t E, const int64_t *split_sizes, int64_t width, int32_t recipe_kind,
                      gsa_layout_info *out, int64_t *col_data_offsets, int64_t *col_scale_offsets);

/* gsa_layout for a recipe, covering both scale layouts.  Sizes in *out as
 * gsa_layout's (scale sizes include the tiled layout's padding).  Each
 * offset array (E+1 entries, may be NULL) receives each expert's byte offset:
 *   col_data_offsets, col_scale_offsets: its columnwise block;
 *   row_scale_offsets: its rowwise scales (compact: row_off[e] * width / B;
 *   tiled: 512 ceil(width / (4 B)) * sum_{j<e} ceil(M_j / 128)); the tiled
 *   columnwise offset is 512 ceil(width / 128) * sum_{j<e} ceil(M_j / (4 B)).
 * The rowwise codes of expert e start at row_off[e] * width (MXFP8) or
 * row_off[e] * width / 2 (NVFP4) bytes in either layout.
 * Errors: as gsa_layout, and INVALID_ARG for a NULL recipe or an unknown
 * scale_layout. */
gsa_status gsa_layout_ex(int64_t E, const int64_t *split_sizes, int64_t width, const gsa_recipe *recipe,
                         gsa_layout_info *out, int64_t *col_data_offsets, int64_t *col_scale_offsets,
                         int64_t *row_scale_offsets);

/* Workspace bytes needed by grouped_scaled_act_fwd / _bwd for this problem
 * (covers both directions).  Returns 0 on invalid arguments. */
size_t gsa_workspace_size(int64_t E, const int64_t *split_sizes, int64_t W_in, int32_t act_kind,
                          int32_t recipe_kind);

/* Forward.  Y = bf16(p * act(X)) and its quantized copies.
 * Defined by "Activation + GroupedLinear Fusion for MOE": the sequence
 * diagram's forward call grouped_scaled_{swiglu,srelu}(x, scales, quantizer,
 * split_sizes) -> grouped_x, one kernel dispatch per the Greptile Summary
 * (per-row scale x activation x grouped quantization); the recompute mode
 * (no columnwise copy here) from "Enable fused activation recompute for
 * ScaledTanhSReLU", Description.
 *   x_bf16   [M, W_in] BF16, probs [M] FP32 (the per-row router scale p);
 *            probs may be NULL, meaning p = 1 for every row.
 *   y_q      quantized Y (at least one of its copies).  For activation
 *            recompute, pass col_data = col_scale = NULL and regenerate the
 *            columnwise copy in the backward.
 *   y_bf16_opt [M, W] BF16 Y, may be NULL.
 *   workspace >= gsa_workspace_size bytes, 256-byte aligned; its content
 *            on entry does not matter (the call clears what it uses).
 * Errors: INVALID_ARG, UNSUPPORTED (E > 256, W as above, M >= 2^31),
 *         ALIGNMENT, WORKSPACE, CUDA. */
gsa_status grouped_scaled_act_fwd(const void *x_bf16, const float *probs, const int64_t *split_sizes,
                                  int64_t E, int64_t W_in, int32_t act_kind,
                                  const gsa_act_params *act_params, const gsa_recipe *recipe,
                                  const gsa_qout *y_q, void *y_bf16_opt,
                                  void *workspace, size_t workspace_bytes, gsa_stream_t stream);

/* Backward, recomputing act(X) from the saved X.
 * Defined by "Activation + GroupedLinear Fusion for MOE": the sequence
 * diagram's backward call grouped_scaled_d{swiglu,srelu}(grad, input_,
 * scales, quantizer) -> (grouped_dy, dense_dy, grad_scales) -- here the
 * quantized dX, the dense dX and dprobs -- and its "Crash when fc1 is frozen"
 * note (dprobs alone is a valid request); the regenerated columnwise Y from
 * "Enable fused activation recompute for ScaledTanhSReLU", Description
 * (FC2's input regenerated from the saved FC1 output, bitwise equal to the
 * forward's).
 *   dy_bf16  [M, W] BF16 gradient w.r.t. Y.  probs may be NULL (p = 1).
 *   dx_bf16_opt [M, W_in] BF16 dX = bf16(dY * p * act'(X)) (GLU: both
 *            halves).  Required when dx_q_opt is given with NVFP4 (the
 *            per-expert scale needs every dX value first; the dense copy is
 *            re-read to encode).
 *   dx_q_opt quantized dX, may be NULL.
 *   dprobs_opt [M] FP32 dprobs[r] = sum_j dY[r, j] * act(X)[r, j], may be
 *            NULL (valid alone: the frozen-fc1 case).
 *   y_regen_col_opt  regenerated columnwise copy of Y (col_data, col_scale,
 *            and amax_col for NVFP4), bitwise equal to what the forward
 *            would have written; may be NULL.
 * At least one output must be requested.  Errors as for the forward. */
gsa_status grouped_scaled_act_bwd(const void *dy_bf16, const void *x_bf16, const float *probs,
                                  const int64_t *split_sizes, int64_t E, int64_t W_in, int32_t act_kind,
                                  const gsa_act_params *act_params, const gsa_recipe *recipe,
                                  void *dx_bf16_opt, const gsa_qout *dx_q_opt, float *dprobs_opt,
                                  const gsa_qout *y_regen_col_opt,
                                  void *workspace, size_t workspace_bytes, gsa_stream_t stream);

/* Forward without a caller-provided workspace and without any allocation.
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory at the point where they run the forward --
 * for example an operator executed from inside another runtime's allocator
 * or memory-planning callback, or a plugin whose execute hook gets no
 * workspace argument and must not call cudaMalloc (which can synchronize
 * the device and fragment a pre-planned pool).
 * Same arguments and results as grouped_scaled_act_fwd, minus the workspace:
 * the scratch counters live in a fixed 64 KiB device array inside libgsa
 * (every GPU that loads the library holds it until the process exits).
 *   - The first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress) with that device current; make the first call
 *     on each device before any stream capture.
 *   - Each call clears the counters it uses (cudaMemsetAsync on `stream`);
 *     the array keeps the last call's contents otherwise.  All calls share
 *     it: calls that overlap on the GPU (other streams, other threads) race
 *     and must be serialized by the caller.
 *   - Problems whose counters exceed the array (5 words per expert, one per
 *     128-row band, 64 words fixed: about 1.9 M rows at 256 experts) return
 *     GSA_ERR_WORKSPACE.
 *   - Never calls cudaMalloc, cudaFree or any allocating routine.
 * Device-side wait timeouts are recorded in the array; gsa_fwd_noalloc_status
 * reads them. */
gsa_status gsa_fwd_noalloc(const void *x_bf16, const float *probs, const int64_t *split_sizes, int64_t E,
                           int64_t W_in, int32_t act_kind, const gsa_act_params *act_params,
                           const gsa_recipe *recipe, const gsa_qout *y_q, void *y_bf16_opt, gsa_stream_t stream);

/* Status of the last gsa_fwd_noalloc call on the current device: synchronizes
 * `stream`, then reads the error word of the library's scratch array.
 * GSA_OK, or GSA_ERR_DEVICE_TIMEOUT if a bounded wait of that call ran out
 * (its outputs are then incomplete).  The next gsa_fwd_noalloc call clears
 * the word, so query before calling again.  Errors: CUDA. */
gsa_status gsa_fwd_noalloc_status(gsa_stream_t stream);

/* ------------------------------------------------------------------------
 * Graph-safe calls: split_sizes in DEVICE memory.
 *
 * The grouped-linear fusion page names a graph-safe fuser path (forward
 * under CUDA-graph capture, where the host cannot read the split).  These
 * calls take split_sizes_dev ([E] int64, device, 8-byte aligned) together
 * with the total row count M (the rows of X, known from its shape), so that
 * nothing enqueued depends on host knowledge of the split: a call can be
 * captured in a CUDA graph once and replayed after the split changes in
 * place.  Each call enqueues a one-CTA plan kernel (clears the workspace
 * counters, checks the split, builds the schedule on the device) and the
 * fused kernel over the full persistent grid.
 *   - Results are bitwise those of the host-split calls for the same split.
 *   - Output buffers are sized by gsa_layout_bound (rowwise copies as for M
 *     rows; columnwise copies for the largest padding any split of M rows
 *     over E experts can need).  The columnwise block of expert e starts at
 *     padded row pad[e] (data byte pad[e] * N for MXFP8, pad[e] * N / 2 for
 *     NVFP4; scale byte pad[e] * N / B), pad = the prefix sums of Mp_e,
 *     written to padded_row_offsets_opt ([E+1] int64, device, may be NULL).
 *   - The workspace is gsa_workspace_size_graph_safe(E, M, ...) bytes,
 *     256-byte aligned.
 *   - A device split with a negative entry or a sum other than M is not
 *     processed: every NVFP4 amax output is set to 0, nothing else is
 *     written, and gsa_workspace_status returns GSA_ERR_INVALID_ARG.
 * Other arguments, conventions and host-side errors as for the host-split
 * calls. */
gsa_status gsa_layout_bound(int64_t E, int64_t M, int64_t width, int32_t recipe_kind, gsa_layout_info *out);

/* gsa_layout_bound for a recipe, covering both scale layouts.  Tiled scales
 * are bounded by sum_e ceil(M_e / 128) <= floor((M + 127 E) / 128) row tiles
 * (rowwise) and sum_e ceil(M_e / (4 B)) <= floor((M + (4 B - 1) E) / (4 B))
 * tile columns (columnwise); an expert's tiled offsets follow from the split
 * by the formulas of gsa_layout_ex (the graph-safe calls use exactly those).
 * Errors: as gsa_layout_bound, and INVALID_ARG for a NULL recipe or an
 * unknown scale_layout. */
gsa_status gsa_layout_bound_ex(int64_t E, int64_t M, int64_t width, const gsa_recipe *recipe, gsa_layout_info *out);

/* Returns 0 on invalid arguments. */
size_t gsa_workspace_size_graph_safe(int64_t E, int64_t M, int64_t W_in, int32_t act_kind, int32_t recipe_kind);

gsa_status grouped_scaled_act_fwd_graph_safe(const void *x_bf16, const float *probs, const int64_t *split_sizes_dev,
                                             int64_t E, int64_t M, int64_t W_in, int32_t act_kind,
                                             const gsa_act_params *act_params, const gsa_recipe *recipe,
                                             const gsa_qout *y_q, void *y_bf16_opt, int64_t *padded_row_offsets_opt,
                                             void *workspace, size_t workspace_bytes, gsa_stream_t stream);

gsa_status grouped_scaled_act_bwd_graph_safe(const void *dy_bf16, const void *x_bf16, const float *probs,
                                             const int64_t *split_sizes_dev, int64_t E, int64_t M, int64_t W_in,
                                             int32_t act_kind, const gsa_act_params *act_params,
                                             const gsa_recipe *recipe, void *dx_bf16_opt, const gsa_qout *dx_q_opt,
                                             float *dprobs_opt, const gsa_qout *y_regen_col_opt,
                                             int64_t *padded_row_offsets_opt, void *workspace, size_t workspace_bytes,
                                             gsa_stream_t stream);

/* Failure-detection self-test.  Enqueues a one-thread kernel that runs one of
 * the library's bounded waits on something nothing signals -- which = 0: the
 * wait for a workspace counter (the encode pass's wait for its expert's amax
 * pass); which = 1: the wait on a shared-memory mbarrier (the stage waits) --
 * with a limit of limit_ms (1..2000) instead of the usual ~2 s.  The wait runs
 * out, records its error code in the workspace and the kernel returns; the
 * context stays usable.  Afterwards gsa_workspace_status returns
 * GSA_ERR_DEVICE_TIMEOUT.  workspace: any 256-byte aligned workspace of at
 * least 256 bytes (its first 256 bytes are cleared).
 * Errors: INVALID_ARG, ALIGNMENT, CUDA. */
gsa_status gsa_selftest_wait_timeout(void *workspace, int32_t which, uint32_t limit_ms, gsa_stream_t stream);

/* Synchronizes `stream`, then reads the workspace's device error word:
 * GSA_OK; GSA_ERR_DEVICE_TIMEOUT if a bounded wait of the last call using
 * this workspace ran out; GSA_ERR_INVALID_ARG if that call was graph-safe
 * and its device split was invalid.  Errors: INVALID_ARG, CUDA. */
gsa_status gsa_workspace_status(const void *workspace, gsa_stream_t stream);

/* Number of kernel launches the last successful fwd/bwd call made on the
 * calling thread (for launch accounting in benchmarks). */
int32_t gsa_last_launch_count(void);

const char *gsa_status_string(gsa_status status);

/* ABI version: (major << 16) | minor. */
int32_t gsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GSA_H */
