/*
 * ridgefill.h -- C ABI of the RidgeFill late-layer cache fill for GB300 (sm_103a).
 *
 * Method: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill"
 * (arXiv 2611.09709).  The lower layers run exactly up to a split layer S.  For
 * every late layer l >= S a ridge map predicts the layer's input from the split
 * state, x_hat_l = A_l x_S + b_l (section 2.2), and the layer's own norm and
 * key/value projections (rotary embedding on keys) write its cache for every
 * prefix row, i.e. every row before the exact tail (sections 2.1-2.2).  A Gated
 * DeltaNet layer instead folds the filled rows into its recurrent state
 * (section 2.3).  The maps come from a closed-form ridge fit over running sums
 * of one capture pass (section 2.2, "Fitting", "The penalty").
 *
 * Conventions shared by every call
 *  - All tensor arguments are plain pointers to dense row-major arrays.  The
 *    caller owns every buffer, including the workspace; the library allocates
 *    no device memory.  Device pointers must be 16-byte aligned.
 *  - bf16 is IEEE bfloat16 (1-8-7), f32/f64 IEEE single/double.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on it: it only enqueues work.  Argument errors are returned
 *    synchronously and nothing is enqueued; inputs are never modified.
 *  - A device-side wait that runs out (about two seconds) makes the kernel
 *    record a code in a device error word and return early; read it with
 *    ridgefill_device_error().  CUDA launch failures return RF_ERR_CUDA.
 *  - No call writes outside the output ranges it documents.
 *  - Not thread-safe for concurrent calls that share a workspace.
 */
#ifndef RIDGEFILL_H
#define RIDGEFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rf_status {
  RF_OK = 0,
  RF_ERR_ARG = 1,        /* null pointer where one is required, or a bad value   */
  RF_ERR_SHAPE = 2,      /* sizes the kernels do not support, or inconsistent   */
  RF_ERR_ALIGN = 3,      /* a device pointer is not 16-byte aligned             */
  RF_ERR_NOT_PINNED = 4, /* maps_on_host set but A is not page-locked host memory */
  RF_ERR_CUDA = 5,       /* a CUDA call failed; see ridgefill_last_error()      */
  RF_ERR_TIMEOUT = 6,    /* a device wait ran out (see ridgefill_device_error)  */
  RF_ERR_NUMERIC = 7,    /* the ridge system was not positive definite          */
  RF_ERR_WORKSPACE = 8,  /* workspace pointer NULL or smaller than required     */
  RF_ERR_SOURCE = 9,     /* a host map source (map_source) returned an error    */
  RF_ERR_BOUNDS = 10     /* debug library only: a kernel store fell outside its
                            buffer, or a workspace guard band was overwritten   */
} rf_status;

/* ------------------------------------------------------------------------ */
/* Attention late layers                                                     */
/* ------------------------------------------------------------------------ */

/*
 * rf_fill_args -- one fill of the prefix rows of L late attention layers.
 *
 * Paper section 2.2 (map x_hat = A_l x_S + b_l; "At inference the predicted
 * input goes through the layer's own normalization and projections ...") and
 * section 2.1 (rows before the tail).  For every layer l, row r and kv head h:
 *   x_hat = A_l h_r + b_l                                   (f32 accumulate)
 *   u     = x_hat / sqrt(mean(x_hat^2) + rms_eps) * gain_l  (RMSNorm)
 *   k     = RoPE(u Wk_l[h]^T, pos0 + r),  v = u Wv_l[h]^T
 *   Kc[l, h, pos0 + r, :] = k,  Vc[l, h, pos0 + r, :] = v   (bf16)
 * RoPE is rotate-half: pair (i, i + hd/2) turns by (pos0 + r) * theta^(-2i/hd).
 *
 * Layouts (row-major, bf16 unless noted):
 *   H     [rows, d_in]                  split state of the rows to fill
 *   A     [L, d_out, d_in]              maps in the paper's orientation: row j of
 *                                       A_l produces output channel j.  Device
 *                                       memory, or page-locked host memory when
 *                                       maps_on_host = 1 (copied one layer at a
 *                                       time while the previous layer computes;
 *                                       results are bitwise those of device maps)
 *   bias  [L, d_out] f32
 *   gain  [L, d_out]                    RMSNorm gain; NULL means all ones
 *   Wk,Wv [L, n_kv_heads*head_dim, d_out]  projection weights, [out, in]
 *   Kc,Vc [L, n_kv_heads, cache_len, head_dim]  caches; only positions
 *                                       [pos0, pos0 + rows) are written
 * Limits: d_in % 64 == 0, d_out % 128 == 0, head_dim in {64, 128},
 *   (n_kv_heads*head_dim) % 128 == 0, pos0 + rows <= cache_len < 2^24,
 *   rows_per_chunk == 0 (all rows in one pass) or a multiple of 128.
 * stage_events (optional, may be NULL): host array of three cudaEvent_t that
 *   the call records on `stream` before the first chunk's map GEMM, between
 *   its map GEMM and its K/V GEMM, and after its K/V GEMM (instrumentation for
 *   per-kernel timing; the events must have been created by the caller).
 * copy_events (optional, may be NULL; host maps only): host array of
 *   2 * n_layers cudaEvent_t recorded on the library's copy stream right before
 *   and after the first chunk's copy of map l (entries 2l and 2l + 1).
 * A_scale (optional, may be NULL): int8 maps.  When set, A holds int8 codes
 *   q [L, d_out, d_in] and A_scale the bf16 scales, one per 128 consecutive
 *   weights of a row (sections 2.2 "Size and cost" and 4.2), stored group-major
 *   [L, d_in / 128, d_out]: the scale of weights 128g .. 128g + 127 of row j
 *   is A_scale[l, g, j].  The map's weight is q * s, rounded once to bf16 as
 *   the GEMM stages it (the product has at most 16 significant bits).  d_in
 *   must be a multiple of 128.  Device memory, or page-locked host memory with
 *   maps_on_host = 1 (then both arrays are streamed, half the bytes of bf16
 *   maps).  ridgefill_quantize_maps makes them.
 * row_idx, h_rows (optional; row_idx may be NULL): exact prefix rows (section
 *   2.4).  When row_idx is set, H is [h_rows, d_in], the split states of every
 *   prefix row, and fill row r (0 <= r < rows) is prefix row row_idx[r]: its
 *   split state is H[row_idx[r]] and its keys and values go to cache position
 *   pos0 + row_idx[r], with RoPE at that position.  Positions not listed are
 *   not written (the exact rows the model computes).  row_idx is device int32
 *   [rows], 4-byte aligned, entries distinct and in [0, h_rows) (an entry
 *   outside is skipped and reported by ridgefill_device_error as
 *   RF_ERR_ARG); pos0 + h_rows <= cache_len.
 * h_on_host (0 or 1): H is page-locked host memory.  The call copies it into
 *   the workspace in groups of 4096 rows on the library's copy stream and the
 *   map GEMM starts on each group as soon as it has landed (a flag set by a
 *   stream memory write), so the copy overlaps the fill; later work on
 *   `stream` is ordered after the copy.  Not with row_idx.
 * k_scale, v_scale (optional, may be NULL): [L, n_kv_heads] f32 device arrays.
 *   When set, every key (value) of head h in layer l is multiplied by
 *   k_scale[l, h] (v_scale[l, h]) before its rounding to bf16: the value or
 *   key rescale of section 2.3 folded into the fill, with the scales from
 *   ridgefill_rescale called with rows = 0.
 * q8_group_layers (int8 maps in device memory; ignored otherwise): 0 or k > 0
 *   writes bf16(q * s) of 4 (or k) layers at a time into the workspace and runs
 *   the bf16 map GEMM on them (workspace grows by that many bf16 maps);
 *   -1 converts the codes inside the map GEMM's shared-memory stages instead
 *   (no extra workspace, bound by shared-memory bandwidth, about 9 % slower).
 *   Both give bitwise the same results.
 * map_source, map_source_user, map_staging, host_wait_ms (optional; map_source
 *   may be NULL): maps produced on the host one layer at a time, for maps that
 *   are not all held in page-locked memory (read from a file, decompressed,
 *   paged in): section 4.2's streamed maps with the host side as the source.
 *   Needs maps_on_host = 1; A (and A_scale) are then ignored and may be NULL,
 *   except that a non-NULL A_scale still selects int8 maps.  For every row
 *   chunk and layer l, in order, the call waits until staging half j (layers
 *   alternate between the two halves of map_staging) is no longer being
 *   copied, calls map_source(map_source_user, l, half j, slot_bytes), which
 *   must write layer l's map there and return 0, and enqueues the copy of
 *   half j into a device map slot.  slot_bytes = d_out * d_in * 2 for bf16
 *   maps; for int8 maps the codes [d_out, d_in] come first and the bf16 scales
 *   [d_in / 128, d_out] start at d_out * d_in rounded up to 256, slot_bytes =
 *   that offset + d_out * (d_in / 128) * 2.  map_staging is page-locked host
 *   memory of 2 * slot_bytes, 16-byte aligned.  Unlike every other use of
 *   this call, it returns only after the last layer's map has been handed to
 *   the copy engine (the kernels may still be running).
 *   Bounded host waits: a staging half that is still being copied after
 *   host_wait_ms milliseconds (0 means 10000), or a map_source call that takes
 *   longer than that, ends the call with RF_ERR_TIMEOUT; a non-zero return of
 *   map_source ends it with RF_ERR_SOURCE.  Work already enqueued for earlier
 *   layers then still completes normally (nothing waits for the missing
 *   layer), the K/V of the current row chunk are not written, and the caller
 *   should synchronise `stream` before reusing the buffers.  map_source runs
 *   on the calling thread and must return.
 */
typedef int32_t (*rf_map_source_fn)(void* user, int32_t layer, void* dst, size_t bytes);

typedef struct rf_fill_args {
  int32_t n_layers;
  int32_t d_in;
  int32_t d_out;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t maps_on_host;
  int64_t rows;
  int64_t pos0;
  int64_t cache_len;
  int64_t rows_per_chunk;
  double rope_theta;
  double rms_eps;
  const void* H;
  const void* A;
  const float* bias;
  const void* gain;
  const void* Wk;
  const void* Wv;
  void* Kc;
  void* Vc;
  void* const* stage_events;
  void* const* copy_events;
  const float* k_scale;
  const float* v_scale;
  const void* A_scale;
  const int32_t* row_idx;
  int64_t h_rows;
  int32_t h_on_host;
  int32_t q8_group_layers;
  rf_map_source_fn map_source;
  void* map_source_user;
  void* map_staging;
  int32_t host_wait_ms;
  int32_t reserved;
} rf_fill_args;

/* Bytes of device workspace ridgefill_fill needs for these arguments
 * (0 on invalid arguments).  Holds the predicted inputs of one row chunk
 * [L, chunk, d_out] bf16, their per-tile sums of squares, and, for host
 * maps, three map slots. */
size_t ridgefill_fill_workspace_size(const rf_fill_args* args);

/* Enqueue the fill described above on `stream`. */
rf_status ridgefill_fill(const rf_fill_args* args, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * ridgefill_fill_noalloc -- the same fill for callers that cannot allocate
 * device memory.  The paper has no counterpart: it is a packaging variant.
 *
 * Some callers have no allocator at hand (a host engine that owns every
 * device buffer and gives plugins none, or code running after the engine has
 * divided up all device memory).  They pass inputs and outputs exactly as for
 * ridgefill_fill but no workspace; the scratch lives in a library-owned
 * device array of RF_NOALLOC_SCRATCH_BYTES that every GPU loading the library
 * holds until exit.  The call allocates nothing.
 *  - Rows are processed in the largest 128-row multiple whose scratch fits
 *    (rows_per_chunk, if set, caps it); results equal ridgefill_fill's.
 *  - If one 128-row chunk does not fit (n_layers * d_out too large) the call
 *    returns RF_ERR_WORKSPACE with the required size in ridgefill_last_error().
 *  - maps_on_host = 1 and h_on_host = 1 are rejected (RF_ERR_ARG).
 *  - The array is shared by all calls on a device and keeps the last call's
 *    contents (nothing in it needs to start at zero); calls that overlap on
 *    the GPU race on it, so order them on one stream.
 *  - The first call on a device (and the first after its context changed)
 *    looks up the array's address with that device current; make it before
 *    any stream capture.
 */
#define RF_NOALLOC_SCRATCH_BYTES (64u << 20)
rf_status ridgefill_fill_noalloc(const rf_fill_args* args, void* stream);

/* ------------------------------------------------------------------------ */
/* Value / key rescale of the filled rows                                    */
/* ------------------------------------------------------------------------ */
/*
 * ridgefill_rescale -- RidgeFill section 2.3 "Value rescale" (and the key
 * scale of section 6.6).  In every late attention layer the first c tail
 * rows go through the layer's norm and value (or key) projection twice: from
 * their true late-layer inputs and from the map's prediction of the same
 * rows.  For each kv head, the mean over the c rows of
 * ||exact projection|| / ||predicted projection|| (rows whose predicted norm
 * is 0 are left out; a head with none keeps 1) is the head's scale, and the
 * filled rows' values (or keys) in the cache are multiplied by it.  Keys are
 * scaled after the rotary embedding, which preserves their norm.
 *
 *  which       RF_RESCALE_VALUES or RF_RESCALE_KEYS.
 *  tail_rows   c in [1, 2^23), the measured rows.
 *  rows, pos0  the filled rows scaled in place: cache positions
 *              [pos0, pos0 + rows) of every layer and kv head.  rows = 0
 *              computes the scales only; passed to ridgefill_fill as
 *              v_scale (k_scale) they are applied as the fill writes the
 *              rows, which saves the read and write of the filled rows here
 *              and rounds each value once instead of twice.
 *  H_tail      [c, d_in] bf16, split states of the c tail rows (device).
 *  X_true      [L, c, d_out] bf16, their true inputs to each late layer.
 *  A, A_scale, bias, gain, Wk, Wv, Kc, Vc, cache_len, rms_eps: as in
 *              rf_fill_args (maps resident in device memory).
 *  scale       optional [L, n_kv_heads] f32 output of the scales (device).
 * All pointers 16-byte aligned.  Asynchronous on `stream`; the cache rows
 * outside [pos0, pos0 + rows) and every other input are left unchanged.
 */
#define RF_RESCALE_VALUES 1
#define RF_RESCALE_KEYS 2
typedef struct {
  int32_t n_layers;
  int32_t d_in;
  int32_t d_out;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t which;
  int64_t tail_rows;
  int64_t rows;
  int64_t pos0;
  int64_t cache_len;
  double rms_eps;
  const void* H_tail;
  const void* X_true;
  const void* A;
  const float* bias;
  const void* gain;
  const void* Wk;
  const void* Wv;
  void* Kc;
  void* Vc;
  float* scale;
  const void* A_scale;
} rf_rescale_args;

/* Workspace bytes ridgefill_rescale needs (0 on invalid arguments): the
 * predicted and true inputs of the c rows stacked [L, 2c, d_out] bf16, their
 * sums of squares, the scaled projection of both [L, n_kv, 2c, head_dim] bf16
 * and the scales. */
size_t ridgefill_rescale_workspace_size(const rf_rescale_args* args);
rf_status ridgefill_rescale(const rf_rescale_args* args, void* workspace, size_t workspace_bytes,
                            void* stream);

/* ------------------------------------------------------------------------ */
/* int8 maps                                                                 */
/* ------------------------------------------------------------------------ */
/*
 * ridgefill_quantize_maps -- the int8 map format of sections 2.2 ("Size and
 * cost") and 4.2: int8 codes with one bf16 scale per 128 consecutive weights
 * of each map row.  For every group a[0..127] of a row:
 *   s = bf16(max|a| / 127)   (float32 division, then rounding to nearest even)
 *   q = clamp(rint(a / s), -127, 127)   (float32 division, ties to even)
 * and a group of zeros gets s = 0, q = 0.
 *
 *  A       [n_maps, d_out, d_in] f32 (src_bf16 = 0) or bf16 (src_bf16 = 1)
 *  q       [n_maps, d_out, d_in] int8 (output)
 *  scale   [n_maps, d_in / 128, d_out] bf16 (output), group-major: the
 *          scale of weights 128g .. 128g + 127 of row j is scale[l, g, j]
 * All device memory, 16-byte aligned; d_in a multiple of 128.  Asynchronous
 * on `stream`; the int8 maps then go to rf_fill_args.A / A_scale.
 */
typedef struct {
  int32_t n_maps;
  int32_t d_out;
  int32_t d_in;
  int32_t src_bf16;
  const void* A;
  void* q;
  void* scale;
} rf_quantize_args;

rf_status ridgefill_quantize_maps(const rf_quantize_args* args, void* stream);

/* ------------------------------------------------------------------------ */
/* Gated DeltaNet late layers                                                */
/* ------------------------------------------------------------------------ */

/*
 * rf_gdn_args -- end-of-fill recurrent state of L late Gated DeltaNet layers.
 *
 * Paper section 2.3 ("every filled row updates the shared state from its
 * predicted input") and section 2.1.  For every layer l and head h, over rows
 * r = 0 .. rows-1 in order, from u as in rf_fill_args:
 *   k = normalize(u Wk_l[h]^T)   (k / sqrt(sum k^2 + l2_eps))
 *   v = u Wv_l[h]^T,  alpha = sigmoid(u . Wa_l[h]),  beta = sigmoid(u . Wb_l[h])
 *   S <- alpha S (I - beta k k^T) + beta v k^T        (S is d_v x d_k, f32)
 * S starts from S0 (or zero) and the final S is written; with rows == 0 the
 * call writes S = S0 (or zero).  The state is carried in f32; `chunk` is the
 * row-chunk length of the state computation and must be 64.
 *
 * Layouts: H, A, bias, gain as in rf_fill_args; Wk [L, n_heads*d_k, d_out],
 *   Wv [L, n_heads*d_v, d_out], Wa/Wb [L, n_heads, d_out] (bf16);
 *   S0 (may be NULL) and S [L, n_heads, d_v, d_k] f32.
 * Limits: d_in % 64 == 0, d_out % 128 == 0, d_k == d_v == 128, chunk == 64,
 *   n_heads a multiple of 8 in [8, 64], rows_per_chunk 0 or a multiple of 128.
 * stage_events (optional): host array of four cudaEvent_t recorded on `stream`
 *   before the first chunk's map GEMM, after it, after its projection GEMM and
 *   after its state kernel.
 * A_scale (optional): int8 maps, as in rf_fill_args.
 * exact_idx, n_exact, X_exact (optional): exact prefix rows (section 2.4).
 *   Rows exact_idx[e] (device int32 [n_exact], 4-byte aligned, strictly
 *   increasing, in [0, rows)) enter the state in prompt order from their true
 *   inputs X_exact[l, e, :] ([L, n_exact, d_out] bf16) instead of the map's
 *   prediction; H still holds every prefix row.  An entry outside [0, rows) is
 *   skipped and reported by ridgefill_device_error as RF_ERR_ARG.
 * rho (optional): [L, n_heads] f32 output, section 2.3's share of the state at
 *   the end of the prefix that comes from filled rows: a row's weight is the
 *   product of the gates alpha of the rows after it, and rho is the filled
 *   rows' total weight over all rows' (1 with no exact rows, 0 with rows = 0).
 * delta_M (optional): [L, n_heads, d_v, d_k] f32, the terminal-state
 *   correction of section 2.3: S += rho * delta_M once, after the last row.
 * h_on_host (0 or 1): H is page-locked host memory, streamed as for
 *   rf_fill_args.h_on_host (with exact rows and one row chunk the copy
 *   completes before the filled rows are gathered).
 * q8_group_layers: as rf_fill_args.q8_group_layers.
 */
typedef struct rf_gdn_args {
  int32_t n_layers;
  int32_t d_in;
  int32_t d_out;
  int32_t n_heads;
  int32_t d_k;
  int32_t d_v;
  int32_t chunk;
  int32_t maps_on_host;
  int64_t rows;
  int64_t rows_per_chunk;
  double rms_eps;
  double l2_eps;
  const void* H;
  const void* A;
  const float* bias;
  const void* gain;
  const void* Wk;
  const void* Wv;
  const void* Wa;
  const void* Wb;
  const float* S0;
  float* S;
  void* const* stage_events;
  const void* A_scale;
  const int32_t* exact_idx;
  int64_t n_exact;
  const void* X_exact;
  float* rho;
  const float* delta_M;
  int32_t h_on_host;
  int32_t q8_group_layers;
} rf_gdn_args;

size_t ridgefill_gdn_workspace_size(const rf_gdn_args* args);
rf_status ridgefill_fill_gdn(const rf_gdn_args* args, void* workspace, size_t workspace_bytes,
                             void* stream);

/* ------------------------------------------------------------------------ */
/* Ridge fit                                                                 */
/* ------------------------------------------------------------------------ */

#define RF_FIT_ACCUMULATE 1
#define RF_FIT_SOLVE 2

/*
 * rf_fit_args -- closed-form ridge maps from running sums (section 2.2,
 * "The ridge map", "Fitting", "The penalty").
 *
 * RF_FIT_ACCUMULATE adds one batch of calibration pairs to caller-owned f64
 * running sums (products of bf16 inputs formed exactly and summed in f32
 * within the call, then added in f64):
 *   G += X^T X [d_in, d_in],  C_l += Y_l^T X (C is [L, d_out, d_in]),
 *   sx += sum_rows X [d_in],  sy += sum_rows Y_l [L, d_out],  count += rows.
 * Zero the sums before the first batch.  Batches add up: a split changes the
 * sums only by the f32 rounding inside each batch.  That rounding grows with
 * the batch: a Gram entry is rows / 16 tensor-core accumulation steps, each
 * within 2^-23 of its running sum (3e-4 low on the diagonal at 65,536 rows),
 * so callers that want tighter sums pass smaller batches.
 *
 * RF_FIT_SOLVE solves from the sums, centring them first:
 *   G~ = G - n mu_S mu_S^T, C~_l = C_l - n mu_l mu_S^T,
 *   alpha = lambda * tr(G~) / d_in,
 *   A_l = C~_l (G~ + alpha I)^-1,  b_l = mu_l - A_l mu_S.
 * The system is equilibrated by its diagonal, factored by a blocked f32
 * Cholesky and inverted; the product with C~ runs on the tensor cores with a
 * three-term bf16 split of both operands (about 16 significant bits each).
 * Outputs A in the fill's layout [L, d_out, d_in] (bf16 and/or f32) and b
 * [L, d_out] f32; alpha_out (device f64, may be NULL).  A non-positive pivot
 * is reported by ridgefill_device_error() as RF_ERR_NUMERIC.
 *
 * Layouts: X [rows, d_in] bf16; Y [L, rows, d_out] bf16.
 * Limits: d_in % 128 == 0, d_out % 128 == 0, d_in <= 16384.
 */
typedef struct rf_fit_args {
  int32_t n_layers;
  int32_t d_in;
  int32_t d_out;
  int32_t flags;
  int64_t rows;
  double lambda;
  const void* X;
  const void* Y;
  double* G;
  double* C;
  double* sx;
  double* sy;
  double* count;
  void* A_out;
  float* A_out_f32;
  float* b_out;
  double* alpha_out;
} rf_fit_args;

size_t ridgefill_fit_workspace_size(const rf_fit_args* args);
rf_status ridgefill_fit(const rf_fit_args* args, void* workspace, size_t workspace_bytes,
                        void* stream);

/* ------------------------------------------------------------------------ */
/* Workspace sizes through one entry                                         */
/* ------------------------------------------------------------------------ */

/* Which call ridgefill_workspace_size answers for. */
typedef enum {
  RF_CALL_FILL = 0,      /* args is a const rf_fill_args*  (ridgefill_fill)     */
  RF_CALL_FILL_GDN = 1,  /* args is a const rf_gdn_args*   (ridgefill_fill_gdn) */
  RF_CALL_FIT = 2,       /* args is a const rf_fit_args*   (ridgefill_fit)      */
  RF_CALL_RESCALE = 3    /* args is a const rf_rescale_args* (ridgefill_rescale) */
} rf_call;

/* Bytes of device workspace the call `which` needs for `args`: the same value
 * as ridgefill_fill_workspace_size, ridgefill_gdn_workspace_size,
 * ridgefill_fit_workspace_size or ridgefill_rescale_workspace_size.  0 for an unknown `which`, a NULL `args` or
 * arguments the call would reject (the reason is in ridgefill_last_error). */
size_t ridgefill_workspace_size(int32_t which, const void* args);

/* ------------------------------------------------------------------------ */
/* Status and host helpers                                                   */
/* ------------------------------------------------------------------------ */

/* Static description of a status code. */
const char* ridgefill_status_string(rf_status status);

/* Message of the last error returned on the calling thread ("" if none). */
const char* ridgefill_last_error(void);

/* Synchronises `stream`, stores the device error word in *code (0 = none,
 * otherwise the id of the wait that ran out, 7 for a non-positive Cholesky
 * pivot, 6 for an out-of-range row index) and clears it.  The status is
 * RF_ERR_TIMEOUT, RF_ERR_NUMERIC or RF_ERR_ARG accordingly. */
rf_status ridgefill_device_error(void* stream, int* code);

/* Section 2.5 compute ceiling: share of exact prefill work that remains,
 * r = (S (N - T) + L T) / (L N); the speedup is at most 1/r. */
double ridgefill_compute_share(int32_t split, int32_t n_layers, int64_t tail, int64_t prompt);

/* Failure-detection self-check.  Launches one small kernel whose bounded device
 * wait, the same helper the fill kernels use, runs out: which = 0 waits on an
 * mbarrier that nothing arrives at, which = 1 on a device flag that nothing
 * sets.  After about two seconds the wait records code 20 + which in the
 * device error word and the kernel returns; ridgefill_device_error() then
 * reports RF_ERR_TIMEOUT with that code, and the context stays usable.  For
 * tests of the error path.  Asynchronous on `stream`. */
rf_status ridgefill_wait_selftest(int32_t which, void* stream);

/* ABI version (incremented on any change to the structs above). */
int32_t ridgefill_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RIDGEFILL_H */
