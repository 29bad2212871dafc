/*
 * rf.h — C ABI of librf.so: the RidgeFill upper-layer KV fill, its calibration
 * statistics and closed-form ridge solve, and the cross-model per-head ridge
 * mapper, for one NVIDIA GB300 (sm_103a).
 *
 * Sources cited below:
 *   [RF] RidgeFill review (jaehun.me, English edition of the review of arXiv
 *        2611.09709): "Two numbers set the skip range", "Ridge map: predict the
 *        input, and the original projection runs unchanged", Table 3.
 *   [XM] "Cross-Model KV Cache Transfer in LLM Families: A Closed-Form Linear
 *        Mapping for Prefill Reuse" (digest): per-head ridge regression,
 *        cross-layer source selection, content-space mapping equation.
 *
 * Conventions shared by every call
 *   - Tensor arguments are DEVICE pointers owned by the caller, unless a comment
 *     says "host". bf16 values are passed as their 16-bit patterns (rf_bf16).
 *   - Every call is asynchronous on the caller's stream (a cudaStream_t passed
 *     as rf_stream_t; NULL is the legacy default stream). No call synchronises
 *     the host unless its comment says so.
 *   - The library allocates no device memory. Calls that need scratch memory
 *     take a caller workspace of at least rf_*_workspace_bytes(...) bytes,
 *     256-byte aligned; its contents are undefined after the call. Calls that
 *     share one workspace must be ordered on one stream.
 *   - Argument errors are detected on the host before any launch and return a
 *     status other than RF_OK; nothing is written then. rf_last_error() gives a
 *     thread-local text for the last failing call on the calling thread.
 *   - Errors found on the device (a bounded wait that gave up, a non-positive
 *     Cholesky pivot) are written to the optional device int32 *dev_status
 *     (first error wins; the caller zeroes it). A kernel that gives up returns
 *     without touching the outputs it had not written yet.
 *   - Functions are thread-safe; no call aborts the process or throws.
 *   - Rows of every matrix are contiguous; "ld" arguments are row strides in
 *     elements. Pointers must be 16-byte aligned and row/layer strides multiples
 *     of 8 elements, else RF_ERR_ALIGN.
 */
#ifndef RIDGE_MAP_KV_RF_H
#define RIDGE_MAP_KV_RF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rf_status {
  RF_OK = 0,
  RF_ERR_INVALID_ARG = 1,  /* null pointer, negative size, unknown mode        */
  RF_ERR_SHAPE = 2,        /* sizes the kernels do not support                */
  RF_ERR_ALIGN = 3,        /* pointer or stride alignment                      */
  RF_ERR_CUDA = 4,         /* CUDA runtime error; text in rf_last_error()      */
  RF_ERR_NOT_SPD = 5,      /* device status: Cholesky pivot <= 0               */
  RF_ERR_TIMEOUT = 6,      /* device status: a bounded device wait gave up      */
  RF_ERR_UNSUPPORTED = 7,  /* current device is not sm_100-family (tcgen05)    */
  RF_ERR_WORKSPACE = 8     /* workspace missing, too small or misaligned       */
} rf_status;

typedef uint16_t rf_bf16;   /* bfloat16 bit pattern                             */
typedef void* rf_stream_t;  /* cudaStream_t                                     */

/* Library version (major*10000 + minor*100 + patch). */
int rf_version(void);
/* Static text for a status code (never NULL). */
const char* rf_status_string(int status);
/* Thread-local text describing the last failing call on this thread ("" if none). */
const char* rf_last_error(void);
/* 1 if `device` has tcgen05 tensor cores (compute capability 10.x), else 0. */
int rf_device_supported(int device);
/* Bounded device waits give up after this many milliseconds (default 4000). Host
 * setting, read at each launch; values < 1 restore the default. */
void rf_set_wait_timeout_ms(int64_t ms);

/* Optional per-kernel timing. Between rf_profile_start and rf_profile_stop every
 * kernel the library launches (on any thread) is bracketed by two CUDA events
 * recorded on its launching stream, up to `max_records` kernels; later launches
 * are not recorded. rf_profile_stop waits for the recorded events, writes up to
 * `capacity` (stage id, milliseconds) pairs in launch order (host arrays) and
 * returns how many it wrote (-1 on a CUDA error). Recording adds two event
 * records per launch and no synchronisation. */
enum rf_stage {
  RF_STAGE_COMPACT = 1,      /* exact-row mask -> fill_idx                    */
  RF_STAGE_GATHER = 2,       /* x_S rows -> dense operand                      */
  RF_STAGE_ROPE_TABLE = 3,   /* (unused: RoPE angles are computed in the kernels) */
  RF_STAGE_MAP_GEMM = 4,     /* x̂ = x_S A_lᵀ + b_l, all upper layers           */
  RF_STAGE_KV_GEMM = 5,      /* K/V projection + norm scale + RoPE + scatter   */
  RF_STAGE_FOLD = 6,         /* gain fold into W_k / W_v                       */
  RF_STAGE_CALIB_GEMM = 7,   /* XᵀX and XᵀY_l                                  */
  RF_STAGE_COLSUM = 8,       /* Σx, Σy, n                                      */
  RF_STAGE_SOLVE = 9,        /* ridge solve: centring, Cholesky, H^-1          */
  RF_STAGE_UNROPE = 10,      /* RoPE / inverse RoPE on cache rows              */
  RF_STAGE_XMODEL_GEMM = 11, /* cross-model mapper GEMM                        */
  RF_STAGE_RESCALE = 12,     /* value rescale: value norms and their ratios   */
  RF_STAGE_EXPAND = 13,      /* int8 map codes -> bf16 before a layer's GEMM   */
  RF_STAGE_QUANTIZE = 14,    /* bf16 maps -> int8 codes and row scales         */
  RF_STAGE_SOLVE_PRODUCT = 15, /* solve: A_p = Cc_pᵀ H^-1 (split tensor-core GEMM) */
  RF_STAGE_SOLVE_REFINE = 16,  /* solve: fp64 residual and correction, per sweep */
  RF_STAGE_ROW_RMS = 17,       /* fill: per-row RMS scale from the map GEMM's sums */
  RF_STAGE_SELECT_GEMM = 18,   /* source selection: split tensor-core products    */
  RF_STAGE_SELECT_FACTOR = 19, /* source selection: batched Cholesky and inverse  */
  RF_STAGE_SELECT_SCORE = 20,  /* source selection: set-up, scores, argmax, copies */
  RF_STAGE_SELECT_SPLIT = 21   /* source selection: fp32 -> three bf16 planes      */
};
rf_status rf_profile_start(int max_records);
/* Diagnostic: runs the tensor-core GEMM kernel on a problem whose operand copies
 * are never issued, so its MMA thread's bounded wait runs out after the wait limit
 * (rf_set_wait_timeout_ms). The kernel then drains, frees its TMEM and writes
 * RF_ERR_TIMEOUT to *dev_status (device int32, must be 0 before the call). It
 * tests the library's failure path without faulting the GPU: nothing is ever in
 * flight, and the context stays usable.
 *   mode  bit 0: the CTA-pair kernel (else the single-CTA one); bit 1: the dynamic
 *         unit order (units posted through the shared-memory ring, from a counter
 *         inside the library's device code), else round-robin. */
rf_status rf_selftest_wait_timeout(int mode, int32_t* dev_status, rf_stream_t stream);
int rf_profile_stop(int32_t* stage_ids, float* ms, int capacity);
const char* rf_stage_name(int stage_id);

/* ===================================================================== *
 * Fill  ([RF] "Two numbers set the skip range"; "Ridge map", first equation
 * x̂_l = A_l x_S + b_l; the layer's own norm and K/V projections and RoPE)
 * ===================================================================== */
typedef struct rf_fill_desc {
  int64_t d;           /* hidden size: map output width, projection input; also the */
                       /* map input width unless d_in is set                        */
  int64_t L;           /* number of layers                                          */
  int64_t S;           /* split layer: maps exist for layers S .. L-1 (P = L - S)    */
  int64_t N;           /* prompt rows                                               */
  int64_t T;           /* tail rows: rows N-T .. N-1 are never filled (0 <= T <= N)  */
  int64_t n_kv_heads;  /* H                                                         */
  int64_t head_dim;    /* hd; KV = H*hd                                              */
  double rope_theta;   /* RoPE base (rotate-half pairs (i, i+hd/2), θ^(-2i/hd))      */
  double rms_eps;      /* RMSNorm ε: y = g ⊙ x / sqrt(mean(x²) + ε)                   */
  int64_t pos_offset;  /* RoPE position of row 0                                     */
  uint64_t flags;      /* RF_FLAG_* (0 = defaults)                                   */
  const float* v_scale;/* [P][H] device fp32 or NULL: the value rescale. Filled V of  */
                       /* layer S+p, head h is multiplied by v_scale[p*H + h] before */
                       /* rounding (see rf_value_scale). NULL = no rescale.         */
  const rf_bf16* k_norm_gain; /* [P][hd] device bf16 or NULL: key normalisation.      */
                       /* Each key head becomes g_p * k_h / sqrt(mean(k_h²) + ε)      */
                       /* (ε = rms_eps) before RoPE ("Qwen models normalize keys").  */
  int64_t d_in;        /* width of x_S rows and of the maps' input; 0 = d (square).  */
                       /* Non-square maps A_p [d][d_in] read a wider split state,    */
                       /* e.g. parallel residual streams ([RF] "Ridge map": 10,240 */
                       /* -> 2,560 for Flash-Next). Must be a multiple of 256.       */
} rf_fill_desc;

/* Flags of rf_fill_desc, rf_calib_desc and rf_xmodel_desc: which tensor-core GEMM
 * kernel runs. RF_FLAG_SINGLE_CTA: one CTA per 128 x 256 output tile
 * (cta_group::1). RF_FLAG_CTA_PAIR: a CTA pair per 256 x 256 tile (cta_group::2,
 * each CTA holding half of B). With neither bit set every operation runs on
 * CTA pairs, the measured-faster kernel. Results agree up to the order of fp32
 * additions. */
#define RF_FLAG_SINGLE_CTA 1u
#define RF_FLAG_CTA_PAIR 2u
/* Flag of rf_fill_desc: the K and V projections passed to the fill already hold
 * the RMSNorm gain, Wk[p][j][i] = W_k,p[j][i] g_p[i] (likewise Wv), for example
 * from rf_fold_kv_weights; `gain` is then ignored and may be NULL. Without it the
 * fill folds the gain into its workspace on every call. */
#define RF_WEIGHTS_PREFOLDED 4u
/* Flag of rf_calib_desc for rf_solve: the refinement's residual cuts its operands
 * into 7-bit digits at every width. By default it takes 8-bit digits up to
 * d_in = 21845 and 7-bit ones above, where the int32 sums of 8-bit digit products
 * could overflow; the flag runs the wider widths' arithmetic at any size (the
 * result meets the same accuracy, with more digit products). */
#define RF_SOLVE_DIGITS7 8u

/* Supported fill shapes: d % 256 == 0, head_dim in {64, 128}, KV % 128 == 0,
 * N - T <= 2^24. */

/* Workspace bytes rf_fill_kv needs for `desc` (0 on invalid desc). Without
 * RF_WEIGHTS_PREFOLDED in desc->flags this includes 2*P*KV*d bf16 for the folded
 * projections. */
size_t rf_fill_workspace_bytes(const rf_fill_desc* desc);

/* Weight preparation for the fill (run once per weight set, then pass the results
 * with RF_WEIGHTS_PREFOLDED): folds each layer's RMSNorm gain into its K and V
 * projections,
 *   Wk_folded[p][j][i] = bf16(Wk[p][j][i] * gain[p][i]),
 *   Wv_folded[p][j][i] = bf16(Wv[p][j][i] * gain[p][i]),
 * gain [P][d], Wk, Wv, Wk_folded, Wv_folded [P][KV][d] (row = output channel),
 * all device. The bf16 x bf16 product is exact in fp32, so the only rounding is
 * the last one. In place (Wk_folded == Wk, Wv_folded == Wv) is allowed. */
rf_status rf_fold_kv_weights(const rf_fill_desc* desc, const rf_bf16* gain,
                             const rf_bf16* Wk, const rf_bf16* Wv,
                             rf_bf16* Wk_folded, rf_bf16* Wv_folded, rf_stream_t stream);

/* The fill. For every filled row t (t < N-T, exact_mask[t] == 0, ascending) and
 * every layer l = S + p:
 *   x̂ = A_p x_S[t] + b_p;  r = (mean(x̂²) + ε)^-1/2;
 *   k = r · (Wk_p ⊙ g_p) x̂,  v = r · (Wv_p ⊙ g_p) x̂   (g_p scales the input channels);
 *   k_h <- g_k,p ⊙ k_h / sqrt(mean(k_h²) + ε)   when desc->k_norm_gain is set;
 *   v_h <- v_scale[p][h] · v_h                  when desc->v_scale is set;
 *   k_h <- RoPE(k_h, t + pos_offset) per head;
 *   k_cache[l][t][h][:] = bf16(k_h),  v_cache[l][t][h][:] = bf16(v_h).
 * Nothing else in the caches is written: not the tail, not exact rows, not
 * layers < S ([RF] Table 3). x̂ is rounded to bf16 before the projection.
 *   x_S        [N][ld_x] bf16 rows of width d_in (d if d_in = 0), the state entering layer S
 *   exact_mask [N-T] uint8, nonzero = exact row (never filled); NULL = none
 *   A          [P][d][d_in] bf16, A_p[o][i] (row = output)
 *   b          [P][d] fp32
 *   gain       [P][d] bf16, the layers' RMSNorm gains (ignored with RF_WEIGHTS_PREFOLDED)
 *   Wk, Wv     [P][KV][d] bf16, the layers' K and V projections (row = output
 *              channel); with RF_WEIGHTS_PREFOLDED they already include the gain
 *              (rf_fold_kv_weights), else the call folds it into its workspace
 *   k_cache, v_cache: element (l, t, h, c) at l*layer_stride + t*row_stride + h*hd + c
 *   n_fill_out device int32 (may be NULL): number of filled rows
 * Kernels: the gain fold (unless prefolded), row compaction + gather, one tcgen05
 * GEMM for all maps (bias, bf16 x̂ and per-row sum-of-squares in its epilogue), one
 * tcgen05 GEMM for all K/V projections (RMS scale, RoPE and cache scatter in its
 * epilogue). */
rf_status rf_fill_kv(const rf_fill_desc* desc,
                     const rf_bf16* x_S, int64_t ld_x,
                     const uint8_t* exact_mask,
                     const rf_bf16* A, const float* b,
                     const rf_bf16* gain, const rf_bf16* Wk, const rf_bf16* Wv,
                     rf_bf16* k_cache, rf_bf16* v_cache,
                     int64_t layer_stride, int64_t row_stride,
                     int32_t* n_fill_out, int32_t* dev_status,
                     void* workspace, size_t workspace_bytes, rf_stream_t stream);

/* Fill for callers that cannot allocate device memory (the pages have no
 * counterpart; this is a library convenience). Some callers have no way to get
 * scratch memory on the GPU: a plugin inside a serving engine whose device memory
 * all belongs to the engine's own pool, or a latency-critical path where a
 * cudaMalloc would synchronise the device. This call computes exactly what
 * rf_fill_kv computes, with the same arguments minus the workspace: its scratch
 * (including the gain fold, unless the weights are prefolded) is a fixed 256-byte
 * aligned array of RF_STATIC_SCRATCH_BYTES inside the
 * library's device code, which every GPU that loads the library keeps until the
 * process exits. It makes no allocating call.
 *   - Fills whose rf_fill_workspace_bytes(desc) exceeds RF_STATIC_SCRATCH_BYTES
 *     are rejected with RF_ERR_WORKSPACE before anything runs.
 *   - Every call looks up the array's device address in the current context (a
 *     host call; the first one in a context may load the library's device code
 *     there), so a cudaDeviceReset or another context never sees a stale address.
 *     Make the first call in each context before any stream capture.
 *   - All calls on a device share the array, which keeps the previous call's
 *     contents; nothing in it needs clearing between calls. Calls that overlap
 *     on the GPU race on it: order them on one stream. */
#define RF_STATIC_SCRATCH_BYTES (64u * 1024u * 1024u)
rf_status rf_fill_kv_static(const rf_fill_desc* desc,
                            const rf_bf16* x_S, int64_t ld_x,
                            const uint8_t* exact_mask,
                            const rf_bf16* A, const float* b,
                            const rf_bf16* gain, const rf_bf16* Wk, const rf_bf16* Wv,
                            rf_bf16* k_cache, rf_bf16* v_cache,
                            int64_t layer_stride, int64_t row_stride,
                            int32_t* n_fill_out, int32_t* dev_status, rf_stream_t stream);

/* Value rescale ([RF] "Hybrid layers and two corrections", value rescale; the
 * 27B deployment uses it with c = 512, "Two numbers set the skip range"). For
 * each upper layer l = S + p and KV head h:
 *   v_scale[p*H + h] = mean over t in [0, c) of ||v_exact_h(t)|| / ||v_pred_h(t)||
 *   v_pred(t)  = r(x̂) · Wv'_p x̂,  x̂ = bf16(A_p x_S[N-T+t] + b_p)   (as in the fill)
 *   v_exact(t) = r(x)  · Wv'_p x,  x  = x_exact[p][t]
 * where Wv'_p = bf16(Wv_p ⊙ g_p) is the gain-folded V projection (Wv as given with
 * RF_WEIGHTS_PREFOLDED in desc->flags, else folded into the workspace from `gain`
 * and `Wv`, both [P][KV][d] / [P][d] bf16), r(x) = (mean(x²) + ε)^-1/2 and
 * ||.|| is the L2 norm of the head's hd values. Rows whose predicted norm is 0 are
 * left out of a head's mean (scale 1 if none is left). The result is meant for
 * rf_fill_desc.v_scale.
 *   c         number of tail rows used, 1 <= c <= T (rows N-T .. N-T+c-1)
 *   x_S, ld_x as for rf_fill_kv (only rows N-T .. N-T+c-1 are read)
 *   x_exact   [P][c][ld_e] bf16 (device): the exact inputs of layers S .. L-1
 *             at those rows (the tail runs every layer exactly)
 *   A, b, gain, Wv as for rf_fill_kv;  v_scale  [P][H] fp32 (device), written
 * Requires d % 256 == 0, head_dim 64 or 128, KV % 128 == 0, S < L. Kernels: the
 * fill's map GEMM on the c tail rows, one tcgen05 GEMM for the V projections of
 * the predicted and the exact rows with per-head norms in its epilogue, and a
 * small reduction. The workspace is rf_value_scale_workspace_bytes(desc, c). */
size_t rf_value_scale_workspace_bytes(const rf_fill_desc* desc, int64_t c);
rf_status rf_value_scale(const rf_fill_desc* desc, int64_t c,
                         const rf_bf16* x_S, int64_t ld_x,
                         const rf_bf16* x_exact, int64_t ld_e,
                         const rf_bf16* A, const float* b,
                         const rf_bf16* gain, const rf_bf16* Wv,
                         float* v_scale, int32_t* dev_status,
                         void* workspace, size_t workspace_bytes, rf_stream_t stream);

/* ===================================================================== *
 * Map storage ([RF] "Ridge map": the 27B maps "in int8 total 1.2 GiB"; "maps can
 * be kept resident in GPU memory or streamed from host memory one layer at a time")
 * ===================================================================== */
/* int8 code of the maps, symmetric per output row (the pages give no scheme):
 *   s[p][o] = max_i |A[p][o][i]| / 127,  q[p][o][i] = rint(A[p][o][i] / s[p][o])
 * (ties to even; both in fp32; a zero row gives s = 0 and q = 0), so that
 * A[p][o][i] ≈ s[p][o] q[p][o][i]. A [P][d][d_in] bf16, q [P][d][d_in] int8,
 * s [P][d] fp32, all device. */
rf_status rf_quantize_maps_int8(const rf_fill_desc* desc, const rf_bf16* A, int8_t* q, float* s,
                                rf_stream_t stream);

#define RF_MAPS_BF16 0 /* A is [P][d][d_in] bf16                                   */
#define RF_MAPS_INT8 1 /* A is q [P][d][d_in] int8 with row_scale s [P][d] fp32    */
typedef struct rf_map_source {
  int32_t kind;           /* RF_MAPS_BF16 or RF_MAPS_INT8                               */
  int32_t on_host;        /* nonzero: A is in host memory. Page-locked memory lets the */
                          /* copy of layer p+1 overlap the GEMMs of layer p; pageable  */
                          /* memory works but its copies may block the calling thread. */
  const void* A;          /* the maps, layer after layer (p = 0 .. P-1)                 */
  const float* row_scale; /* RF_MAPS_INT8: [P][d] fp32 on the device; else unused       */
} rf_map_source;

/* The fill of rf_fill_kv, a few layers at a time: for each step of up to 4
 * layers the map GEMM of those layers and then their K/V GEMM, so x̂ exists for
 * 4 layers only (workspace 4*M_pad*d instead of P*M_pad*d bf16). Maps on the host
 * or in int8 pass through a two-slot bf16 ring in the workspace: the library's
 * copy stream copies the next step's maps (and expands int8 codes to bf16, exact
 * for |q| <= 127) while the caller's stream computes the current step; int8 row
 * scales are applied to the map GEMM's output
 * columns with the bias. Device bf16 maps are read in place. The results equal
 * rf_fill_kv's bit for bit when the maps are the same bf16 values (same kernels,
 * same summation order). Arguments as for rf_fill_kv, with `maps` replacing A
 * (gain, Wk, Wv and RF_WEIGHTS_PREFOLDED as there); the workspace is
 * rf_fill_layered_workspace_bytes(desc, maps). Everything is asynchronous on
 * `stream`. */
size_t rf_fill_layered_workspace_bytes(const rf_fill_desc* desc, const rf_map_source* maps);
rf_status rf_fill_kv_layered(const rf_fill_desc* desc,
                             const rf_bf16* x_S, int64_t ld_x,
                             const uint8_t* exact_mask,
                             const rf_map_source* maps, const float* b,
                             const rf_bf16* gain, const rf_bf16* Wk, const rf_bf16* Wv,
                             rf_bf16* k_cache, rf_bf16* v_cache,
                             int64_t layer_stride, int64_t row_stride,
                             int32_t* n_fill_out, int32_t* dev_status,
                             void* workspace, size_t workspace_bytes, rf_stream_t stream);

/* ===================================================================== *
 * Calibration statistics ([RF] "Ridge map": only XᵀX, XᵀY_l and the two means
 * are accumulated in one pass; [XM]: XᵀX is the dominant fitting cost)
 * ===================================================================== */
typedef struct rf_calib_desc {
  int64_t d_in;    /* width of x (map input)        */
  int64_t d_out;   /* width of each y_p (map output) */
  int64_t n_maps;  /* P                              */
  uint64_t flags;  /* RF_FLAG_* (0 = defaults)       */
} rf_calib_desc;

/* Raw one-pass sums, all device fp64 (n as int64), caller-owned.
 *   G   [d_in][d_in]          Σ x xᵀ   (both triangles)
 *   C   [n_maps][d_in][d_out] Σ x y_pᵀ
 *   sx  [d_in]                Σ x
 *   sy  [n_maps][d_out]       Σ y_p
 *   n   [1]                   rows seen
 *   syy [n_maps][d_out]       Σ y_p² per column (optional, NULL = not kept; the
 *                             total sums of squares that rf_select_sources needs)
 * Zero them to start; saved and reloaded sums resume accumulation. */
typedef struct rf_calib_stats {
  double* G;
  double* C;
  double* sx;
  double* sy;
  int64_t* n;
  double* syy;
} rf_calib_stats;

/* Supported: d_in % 128 == 0, d_out % 256 == 0 (or n_maps == 0), n_rows % 8 == 0.
 * The workspace is optional (see rf_calib_accumulate); this is its size (256). */
size_t rf_calib_workspace_bytes(const rf_calib_desc* desc, int64_t n_rows);

/* Adds one batch of rows: G += XᵀX, C_p += XᵀY_p, sx += Σx, sy_p += Σy_p, n += n_rows
 * (and syy_p += Σy_p² when stats->syy is set).
 *   X [n_rows][ld_x] bf16; Y_p at Y + p*y_map_stride, [n_rows][ld_y] bf16.
 * Products are exact in fp32, summed in fp32 over chunks of rows on the tensor
 * cores and added to the fp64 totals.
 *   workspace  NULL, or rf_calib_workspace_bytes(...) bytes, 256-byte aligned: with
 *              it the GEMM takes its output tiles in dynamic order (a device
 *              counter), which keeps the CTAs that share operand rows together in
 *              L2; without it, in a fixed round-robin order. The sums are the same
 *              bit for bit either way (each tile is added to the totals once per
 *              16 chunks of rows, in stream order). */
rf_status rf_calib_accumulate(const rf_calib_desc* desc,
                              const rf_bf16* X, int64_t ld_x,
                              const rf_bf16* Y, int64_t ld_y, int64_t y_map_stride,
                              int64_t n_rows, const rf_calib_stats* stats,
                              int32_t* dev_status,
                              void* workspace, size_t workspace_bytes, rf_stream_t stream);

/* ===================================================================== *
 * Ridge solve ([RF] "Ridge map": A_l = Y_lᵀX (XᵀX + αI)^-1, b_l = μ_l − A_l μ_S,
 * α = λ·tr(XᵀX)/d_in on centred X; a new λ only needs a re-solve)
 * ===================================================================== */
enum { RF_ALPHA_TRACE = 0, RF_ALPHA_ABSOLUTE = 1 };

size_t rf_solve_workspace_bytes(const rf_calib_desc* desc);

/* Solves every map from the statistics (read only, so re-solving at another λ
 * is legal):
 *   Gc = G − n μ_x μ_xᵀ, Cc_p = C_p − n μ_x μ_pᵀ, α = λ tr(Gc)/d_in (TRACE) or λ,
 *   Gc + αI = L Lᵀ (fp32 Cholesky), A_p = Cc_pᵀ (Gc + αI)^-1 (fp32), then
 *   `refine_iters` sweeps of A_p += (Cc_pᵀ − A_p (Gc + αI)) (Gc + αI)^-1 with the
 *   residual computed beyond fp32 accuracy (exact integer digit products on the
 *   tensor cores); b_p = μ_p − A_p μ_x (compensated, to about 2^-44 of Σ|A||μ|,
 *   rounded to fp32). How accurate the residual and the correction are is chosen on
 *   the device from κ(Gc + αI), estimated once by power iteration (24 steps, whose
 *   estimate is taken twice over): accurate enough for a sweep to bring A to fp32
 *   accuracy, the residual to at least 2^-(25 + log2 2κ) of Σ|A||Gc + αI| (with
 *   8-bit digits 2^-31.7 for κ up to about 51, 2^-39.4 up to about 10,800, else
 *   2^-47.2, its limit; with 7-bit digits, above d_in = 21845 or under
 *   RF_SOLVE_DIGITS7, 2^-27.7 up to about 3, 2^-34.4 up to about 330, else 2^-41.2),
 *   the correction to fp32 when 4κ > 2^10, else to about 2^-16 of its terms.
 *   A [n_maps][d_out][d_in] fp32, b [n_maps][d_out] fp32,
 *   A_bf16 (may be NULL) bf16 copy of A for rf_fill_kv, alpha_out (device, may be NULL).
 * A non-positive pivot sets RF_ERR_NOT_SPD in *dev_status. */
rf_status rf_solve(const rf_calib_desc* desc, const rf_calib_stats* stats,
                   double lambda, int alpha_mode, int refine_iters,
                   float* A, float* b, rf_bf16* A_bf16, double* alpha_out,
                   int32_t* dev_status,
                   void* workspace, size_t workspace_bytes, rf_stream_t stream);

/* ===================================================================== *
 * Cross-model mapper ([XM] content-space mapping
 *   K̂_t = (K_s R_s^-1(t) W_K + b_K) R_t(t), V mapped without RoPE;
 * the k source layers chosen for a target layer are concatenated, all heads)
 * ===================================================================== */
typedef struct rf_xmodel_desc {
  int64_t L_src;       /* source layers                                  */
  int64_t L_tgt;       /* target layers                                  */
  int64_t k;           /* source layers concatenated per target layer     */
  int64_t n_kv_heads;  /* H (same on both sides: KV-matched pair)         */
  int64_t head_dim;    /* hd                                             */
  int64_t N;           /* rows (tokens)                                  */
  double theta_src;    /* source RoPE base                                */
  double theta_tgt;    /* target RoPE base                                */
  int64_t pos_offset;  /* position of row 0                               */
  uint64_t flags;      /* RF_FLAG_* (0 = defaults)                        */
} rf_xmodel_desc;

/* Supported: head_dim in {64, 128}, KV % 256 == 0, N >= 1. */
size_t rf_xmodel_workspace_bytes(const rf_xmodel_desc* desc);

/* For every target layer l and row t:
 *   F_K = [RoPE_src^-1(k_src[s_j][t]) for j < k] (feature order: j, head, dim),
 *   F_V = [v_src[s_j][t] for j < k],  s_j = src_layers[l*k + j],
 *   k_tgt[l][t] = bf16(RoPE_tgt(F_K Wk_lᵀ + bk_l)),  v_tgt[l][t] = bf16(F_V Wv_lᵀ + bv_l).
 *   src_layers  device int32 [L_tgt][k], each in [0, L_src) (e.g. rf_select_sources'
 *               output, used with no host round trip). The table is checked on the
 *               device: an entry outside [0, L_src) writes RF_ERR_INVALID_ARG to
 *               *dev_status and the call then writes no target entry.
 *   k_src, v_src [L_src][N][KV] bf16;  k_tgt, v_tgt [L_tgt][N][KV] bf16
 *   Wk, Wv [L_tgt][KV][k*KV] bf16 (row = output);  bk, bv [L_tgt][KV] fp32 */
rf_status rf_xmodel_map(const rf_xmodel_desc* desc, const int32_t* src_layers,
                        const rf_bf16* k_src, const rf_bf16* v_src,
                        const rf_bf16* Wk, const float* bk,
                        const rf_bf16* Wv, const float* bv,
                        rf_bf16* k_tgt, rf_bf16* v_tgt, int32_t* dev_status,
                        void* workspace, size_t workspace_bytes, rf_stream_t stream);

/* RoPE (inverse = 0) or its inverse (inverse = 1) on rows of heads, out of place
 * or in place: out[t][h][:] = R^{±1}(t + pos_offset) in[t][h][:]. The angle
 * (t + pos_offset)·θ^(-2i/hd) is reduced mod 2π exactly in 64-bit fixed point,
 * then its sine and cosine are taken in fp32 (absolute error about 2^-21); the
 * fill and the mapper rotate the same way.
 * in, out [n_rows][ld] bf16 with H*hd <= ld. Used to build cross-model
 * calibration features (un-roped keys). [XM] content-space mapping. */
rf_status rf_rope_rows(const rf_bf16* in, rf_bf16* out, int64_t n_rows, int64_t ld,
                       int64_t n_heads, int64_t head_dim, double theta,
                       int64_t pos_offset, int inverse, rf_stream_t stream);

/* Side-by-side features of several layers, for cross-model calibration:
 *   out[t][l*W + j] = f(src[l*layer_stride + t*ld_src + j]),  W = n_heads*head_dim,
 *   f = inverse RoPE at position t + pos_offset with base theta (theta > 0: keys)
 *   or the identity (theta == 0: values), for l < n_layers, t < n_rows, j < W.
 * src, out bf16 device; ld_src >= W, ld_out >= n_layers*W, strides multiples of 8.
 * [XM] "층 교차 소스 선택": a target layer's features are all heads of its source
 * layers side by side; content-space mapping: keys are un-roped first. */
rf_status rf_concat_layers(const rf_bf16* src, int64_t n_layers, int64_t layer_stride,
                           int64_t n_rows, int64_t ld_src, int64_t n_heads, int64_t head_dim,
                           double theta, int64_t pos_offset,
                           rf_bf16* out, int64_t ld_out, rf_stream_t stream);

/* ===================================================================== *
 * Cross-layer source selection ([XM] "소스 층은 몇 개가 필요한가": greedy
 * forward selection adding the source layer that raises the head-mean R² most;
 * "층 교차 소스 선택": k layers per target layer, chosen by the head-mean R² of
 * the un-roped keys and of the values, shared by all heads of the target layer)
 * ===================================================================== */
typedef struct rf_select_desc {
  int64_t L_src;      /* candidate source layers                                       */
  int64_t F;          /* features per source layer (the statistics' d_in = L_src * F)  */
  int64_t n_targets;  /* target layers (the statistics' n_maps)                        */
  int64_t d_out;      /* columns per target layer                                      */
  int64_t head_dim;   /* columns per target head; R² is averaged over d_out/head_dim   */
  int64_t k;          /* layers chosen per target layer, 1 <= k <= L_src               */
  int64_t n_kinds;    /* statistics sets scored together: 1, or 2 (keys and values)    */
  int64_t group;      /* target layers per pass, 0 = all; the workspace grows with it  */
  uint64_t flags;     /* RF_FLAG_* (0 = defaults)                                      */
} rf_select_desc;

/* Supported: F % 256 == 0, d_out % 256 == 0, d_out % head_dim == 0,
 * L_src * F <= 65536, n_targets <= 65535. */
size_t rf_select_workspace_bytes(const rf_select_desc* desc);

/* Greedy forward selection for every target layer t, from calibration sums
 * (stats[kind], one set per kind, each with d_in = L_src*F, d_out, n_maps =
 * n_targets and syy set):
 *   per kind: Gc, Cc_t centred as in rf_solve, TSS_t[o] = syy_t[o] − n μ_t[o]²,
 *   α = λ·tr(Gc)/(L_src*F) (RF_ALPHA_TRACE, over ALL source features) or λ;
 *   the score of a layer set S for target t and kind: the mean over heads h of
 *     R²_h = Σ_{o∈h} Cc_t[S,o]ᵀ (Gc[S,S] + αI)^-1 Cc_t[S,o] / Σ_{o∈h} TSS_t[o],
 *   i.e. 1 − (RSS + α‖w‖²)/TSS of the ridge fit (the least-squares R² at λ = 0);
 *   a head with TSS = 0 counts as R² = 0;
 *   step j adds the layer s not yet chosen whose set S ∪ {s} has the highest mean
 *   score over kinds (the lowest index among equal scores).
 * Outputs (device): src_layers [n_targets][k] int32, the layer chosen at each step;
 * r2 [n_kinds][n_targets][k][L_src] fp32 (may be NULL): each candidate's score at
 * each step, NaN for layers already chosen (step 0 is the single-layer R² table).
 * Arithmetic: the Gram and cross terms in fp32, products as fp32-accurate split
 * bf16 tensor-core GEMMs, Schur blocks factored in fp32; scores in fp64.
 * A non-positive pivot sets RF_ERR_NOT_SPD in *dev_status. */
rf_status rf_select_sources(const rf_select_desc* desc, const rf_calib_stats* stats,
                            double lambda, int alpha_mode,
                            int32_t* src_layers, float* r2, int32_t* dev_status,
                            void* workspace, size_t workspace_bytes, rf_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* RIDGE_MAP_KV_RF_H */
