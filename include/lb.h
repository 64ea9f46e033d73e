/*
 * lb.h — C ABI of the GB300 layer-boundary library (liblb.so).
 *
 * A layer boundary completes the producer's owed sum, folds it into the residual
 * stream and prepares the consumer's input ("Layer boundaries", sglang developer
 * guide, opening section and section "Residual stream").  On one GPU the owed
 * cross-rank sum is recast as K partial-contribution buffers resident in device
 * memory; every call below does the whole boundary in one pass over HBM.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - bf16 tensors are raw IEEE bfloat16, row-major, rows contiguous (row stride H).
 *    gamma is float32 [H].  FP8 codes are OCP E4M3 ("fn": max 448, no infinity).
 *  - All tensor pointers are DEVICE pointers.  Arrays of pointers (`partials`) and
 *    the ragged-set metadata are HOST arrays, read during the call only.
 *  - Ownership: the caller allocates and owns every buffer.  The library allocates
 *    nothing, keeps no per-call state and never synchronises the stream.
 *  - Execution: kernels are enqueued asynchronously on `stream` (NULL = the legacy
 *    default stream), on the device that owns the stream; every buffer must live on
 *    (or be accessible from) that device.  If the stream's device is not the calling
 *    thread's current device, the call makes it current for the launch and restores
 *    the caller's device before returning.  While the stream is being captured into
 *    a CUDA graph its device cannot be queried, and the call then launches on the
 *    current device: capture on a stream of the current device.  A returned LB_OK
 *    means the launch was enqueued.
 *  - Arithmetic ("Residual update and input read": the fused add+norm keeps its FP32
 *    accumulation and normalises it, not a rounded snapshot):
 *      o[t,h]  = (+0 + p_0[t,h] + p_1[t,h] + ... + p_{K-1}[t,h]) + res[t,h]
 *                (binary32, left to right; no residual term in the Initial state)
 *      res'    = bf16_rne(o)
 *      r_t     = 1 / sqrt(sum_h o[t,h]^2 / H + eps)
 *      yf      = (o * r_t) * gamma[h]         y = bf16_rne(yf)
 *      FP8:    scale_t = max_h |yf| / 448,   q = e4m3_rne_satfinite(yf / scale_t)
 *              (an all-zero row gets scale 0 and codes 0x00)
 *    res' is bit-identical to a sequential binary32 evaluation; y and the FP8 scale
 *    differ from it only through the order of the sum of squares.
 *  - Aliasing: residual_out may equal residual_in (in-place fold).  Any other
 *    overlap between an output and any buffer is rejected (LB_ERR_INVALID_ARGUMENT).
 *  - Alignment: every tensor pointer must be 16-byte aligned and H a multiple of 8,
 *    else LB_ERR_MISALIGNED / LB_ERR_UNSUPPORTED.
 *  - Validation before writes: every argument is checked before anything is
 *    launched; on any error nothing is written ("Fusion providers and output
 *    decisions": a candidate that declines must do so before touching its inputs).
 *  - Empty batch: zero rows returns LB_OK and launches nothing ("Enter and leave the
 *    layer stack": an empty batch still completes owed work and skips the norm).
 *    Only the scalar arguments are checked then; buffer pointers may be NULL.
 */
#ifndef LB_H
#define LB_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
struct CUstream_st;
typedef struct CUstream_st *lb_stream_t;

#define LB_MAX_K 16       /* partial buffers per call */
#define LB_MAX_TOPK 16    /* routed experts per token in the MoE finalize */
#define LB_MAX_SETS 64    /* token sets in a ragged batch */
#define LB_MAX_H 131072   /* hidden size */
#define LB_MAX_ROWS 134217728 /* rows of one call (2^27: every launch grid fits) */

typedef enum {
    LB_OK = 0,
    LB_ERR_INVALID_ARGUMENT = 1, /* NULL where a buffer is required, bad sizes, overlap */
    LB_ERR_MISALIGNED = 2,       /* a tensor pointer is not 16-byte aligned */
    LB_ERR_UNSUPPORTED = 3,      /* K, topk, sets or H outside the supported range */
    LB_ERR_CUDA = 4,             /* the CUDA launch failed; see lb_last_cuda_error() */
    /* residual stream misuse (lb_residual.h; "Layer boundaries", section "Integration
     * checklist and common errors") */
    LB_ERR_NOT_STARTED = 5,      /* start the layer stack before entering a stage */
    LB_ERR_FOREIGN_OUTPUT = 6,   /* the output does not belong to this residual stream */
    LB_ERR_UPDATE_PENDING = 7    /* write the residual update before taking the output */
} lb_status;

/* Static, human-readable name of a status. */
const char *lb_status_string(lb_status status);

/* cudaError_t value of the most recent LB_ERR_CUDA on the calling thread (0 if none). */
int lb_last_cuda_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int lb_version(void);

/*
 * Optional behaviour of a call; pass NULL for the defaults (plain gamma, no snapshot).
 *   flags              LB_OPT_GEMMA_WEIGHT: the read's weight is 1 + gamma (the Gemma
 *                      form of RMSNorm that the fused final-norm handoff reads,
 *                      "Layer boundaries", section "Enter and leave the layer stack")
 *   residual_snapshot  bf16 output [rows, H] receiving a second copy of residual'
 *                      (an owned snapshot of the updated residual, section "Auxiliary
 *                      capture and extra contributions"), or NULL; 16-byte aligned
 * An extra contribution added exactly once ("add_to_output") is one more partial.
 */
#define LB_OPT_GEMMA_WEIGHT 1u
/*
 * LB_OPT_ROUTING_READY (lb_moe_finalize_fold_norm only; other calls return
 * LB_ERR_UNSUPPORTED): the caller promises that idx and w were complete before the
 * kernel that immediately precedes this call on its stream began, as they are when the
 * router runs ahead of the expert GEMMs.  The call then reads its first tokens' indices
 * and weights without waiting for that kernel to finish (the call's kernels are
 * programmatic dependents of it); every other read still waits.  Without the promise
 * (default) nothing is read before the preceding kernel has finished.
 */
#define LB_OPT_ROUTING_READY 2u
/*
 * LB_OPT_RESIDUAL_READY (every call): the caller promises that residual_in and gamma
 * were complete before the kernel that immediately precedes this call on its stream
 * began, as they are between two layer boundaries (GEMMs run in between; gamma is a
 * weight).  The call may then read them without waiting for that kernel to finish.
 * The partials (or expert rows) and every output still wait for it.
 * Every kernel of this library lets its own dependent start as soon as it begins
 * (programmatic dependent launch), so a preceding call of this library counts as having
 * begun while its own predecessor was still running.  Do not set the flag when
 * residual_in (or gamma) was written by a call of this library earlier in the same
 * chain of back-to-back launches, unless another kernel runs in between (the usual
 * case: the layer's GEMMs separate two boundaries).
 */
#define LB_OPT_RESIDUAL_READY 4u

typedef struct {
    unsigned int flags;
    void *residual_snapshot;
} lb_options;

/* Kernels of the library (lb_plan.kernel). */
#define LB_KERNEL_ROW 0     /* one CTA, or a cluster of up to 8 CTAs, per token row */
#define LB_KERNEL_STREAM 1  /* persistent CTAs streaming rows through TMA stages */

/* How a call of `rows` rows is launched. */
typedef struct {
    int kernel;             /* LB_KERNEL_ROW or LB_KERNEL_STREAM */
    int grid;               /* CTAs launched */
    int threads;            /* threads per CTA */
    int vectors_per_thread; /* 16-byte vectors of a row per (consumer) thread */
    int ctas_per_row;       /* row kernel: CTAs (cluster size) per row; else 1 */
    int stages;             /* stream kernel: shared-memory stages; else 0 */
    int smem_bytes;         /* stream kernel: dynamic shared memory per CTA; else 0 */
    int groups;             /* stream kernel: consumer groups (rows reduced at once) */
    int chunks;             /* stream kernel: stages per row (column chunks); else 0 */
} lb_plan;

/*
 * The launch the library makes for `rows` rows of width H, each reading `n_inputs`
 * input rows (K partials or topk expert rows, plus one if there is a residual), on a
 * GPU with `num_sms` SMs and `smem_per_block` bytes of opt-in shared memory per CTA.
 * Host-only, pure.  Calls with more rows than SMs stream through the
 * persistent TMA kernel when a double-buffered stage fits (a stage holds a whole row
 * of every input, or for rows of more than 8192 elements, up to 16384, one of 2-4
 * column chunks of it); smaller calls use the row kernel, one CTA per row, splitting
 * a row over a cluster only when it is longer than one CTA holds (16384 elements).
 * Returns LB_ERR_UNSUPPORTED for an H that no launch covers.
 */
lb_status lb_launch_plan(int64_t rows, int64_t H, int n_inputs, int num_sms,
                         int smem_per_block, lb_plan *plan);

/* Device-side error flags (lb_device_error). */
#define LB_DEVICE_ERR_TIMEOUT 1u  /* a bounded wait in the stream kernel gave up */
#define LB_DEVICE_ERR_LAUNCH 2u   /* the stream kernel refused an inconsistent launch */

/*
 * Synchronises the current device, then returns in *flags the OR of the device-side
 * error flags raised by the library's kernels since they were last cleared, and
 * clears them when `clear` is nonzero.  A set flag means that some call since then
 * produced incomplete outputs.  Not for use during stream capture.
 */
lb_status lb_device_error(unsigned int *flags, int clear);

/*
 * lb_fold_norm — complete K partial sums, fold into the residual, RMSNorm read.
 * "Layer boundaries": section "Residual stream" (state table and the helpers
 * complete_output / fold) and section "Residual update and input read" (fused
 * update_and_read); "SGLang flashinfer_allreduce_fusion精读", section forward
 * (all-reduce + residual add + RMSNorm in one kernel at fusion points A and B).
 *
 *   partials     host array of K device pointers, each bf16 [T,H]; K in [0, LB_MAX_K]
 *   residual_in  bf16 [T,H], or NULL for the Initial state (o = sum of partials)
 *   residual_out bf16 [T,H] receives bf16(o), or NULL to skip (read-only boundary)
 *   gamma        float32 [H]; required when y_out is given
 *   y_out        bf16 [T,H] receives the RMSNorm read, or NULL for no read
 *   T, H         rows and hidden size; 0 <= T <= LB_MAX_ROWS, 8 <= H <= LB_MAX_H,
 *                H % 8 == 0 (LB_ERR_UNSUPPORTED outside these ranges)
 *   eps          >= 0 and finite
 *
 * The stream operations of the Residual stream section map to argument patterns:
 *   enter (Initial)     residual_in = NULL
 *   complete_output     residual_in = NULL, y_out = NULL  (residual_out = the sum)
 *   fold                residual_in != NULL, y_out = NULL
 *   read (Written)      K = 0, residual_out = NULL
 *   fold + read         every buffer given (the hot path)
 * K = 0 needs residual_in; at least one of residual_out, y_out must be given.
 */
lb_status lb_fold_norm(const void *const *partials, int K, const void *residual_in,
                       void *residual_out, const float *gamma, void *y_out, int64_t T,
                       int64_t H, float eps, const lb_options *options, lb_stream_t stream);

/*
 * lb_fold_norm_fp8 — lb_fold_norm whose read is quantised per token to FP8 E4M3
 * with a dynamic scale ("Layer boundaries", section "Execute a layer": prepare()
 * returns input in the consumer read's format, which can be quantized).
 *
 *   q_out        uint8 [T,H] E4M3 codes (required)
 *   scale_out    float32 [T] per-token scale, max|yf| / 448 (required)
 *   y_out        bf16 [T,H] unquantised read, or NULL
 * Other arguments as lb_fold_norm; gamma is required.
 */
lb_status lb_fold_norm_fp8(const void *const *partials, int K, const void *residual_in,
                           void *residual_out, const float *gamma, uint8_t *q_out,
                           float *scale_out, void *y_out, int64_t T, int64_t H, float eps,
                           const lb_options *options, lb_stream_t stream);

/*
 * lb_moe_finalize_fold_norm — deferred MoE finalize fused with the fold and read.
 * "Layer boundaries": section "Producer contracts and output state" (HandoffOutput,
 * a deferred MoE finalize consumed by the next boundary) and section "Enter and
 * leave the layer stack" (finalize(handoff, residual, gamma) fuses finalize,
 * all-reduce, residual add and norm).
 *
 *   o[t,h] = (+0 + w[t,0]*E[idx[t,0],h] + ... + w[t,topk-1]*E[idx[t,topk-1],h])
 *            + res[t,h]      (each product rounded to binary32, then added)
 *
 *   expert_out     bf16 [n_expert_rows, H], expert-sorted rows of the routed tokens
 *   idx            int32 [T, topk], row of expert_out for (token, slot)
 *   w              float32 [T, topk], routing weights
 *   topk           1 .. LB_MAX_TOPK
 *   residual_in    bf16 [T,H] or NULL (Initial);  residual_out bf16 [T,H] or NULL
 *   y_out          bf16 [T,H] or NULL;  q_out uint8 [T,H] + scale_out float32 [T]
 *                  together or both NULL (FP8 read)
 *   bad_index_flag int32 device word or NULL.  An index outside [0, n_expert_rows)
 *                  is skipped (contributes nothing) and, when the flag is given, the
 *                  kernel stores 1 into it; the caller zeroes it beforehand.
 */
lb_status lb_moe_finalize_fold_norm(const void *expert_out, int64_t n_expert_rows,
                                    const int32_t *idx, const float *w, int topk,
                                    const void *residual_in, void *residual_out,
                                    const float *gamma, void *y_out, uint8_t *q_out,
                                    float *scale_out, int64_t T, int64_t H, float eps,
                                    int32_t *bad_index_flag, const lb_options *options,
                                    lb_stream_t stream);

/*
 * lb_slice_fold_norm — one rank's row slice of a padded, ragged token batch after a
 * fixed-size reduce-scatter ("Layer boundaries", section "Choose a reduction
 * policy", value rs, and section "Token layouts and sums": ATTN_DP token sets whose
 * padding and counts come from batch metadata; "SGLang flashinfer_allreduce_fusion
 * 精读", section forward: with reduce-scatter RMSNorm runs on the rank's slice only).
 *
 *   partials       K device pointers, each bf16 [T_pad,H] over the padded batch
 *   T_pad          padded rows; num_slices >= 1 divides T_pad; S = T_pad/num_slices
 *   slice          0 <= slice < num_slices; global rows [slice*S, (slice+1)*S)
 *   set_offsets    host int32 [num_sets]: first padded row of each token set
 *   set_counts     host int32 [num_sets]: valid rows of each set; set i holds valid
 *                  rows [offset_i, offset_i + count_i); sets ascending, disjoint,
 *                  inside [0, T_pad).  num_sets = 0: every row is valid.
 *   residual_in    bf16 [S,H] compact slice rows, or NULL (Initial)
 *   residual_out, y_out, q_out/scale_out: compact [S,...] outputs as above
 * Padding rows are neither computed nor written: their output bytes are untouched.
 */
lb_status lb_slice_fold_norm(const void *const *partials, int K, int64_t T_pad,
                             int num_slices, int slice, const int32_t *set_offsets,
                             const int32_t *set_counts, int num_sets,
                             const void *residual_in, void *residual_out,
                             const float *gamma, void *y_out, uint8_t *q_out,
                             float *scale_out, int64_t H, float eps,
                             const lb_options *options, lb_stream_t stream);

/*
 * lb_slice_fold_norm_v — one rank's rows of a padded, ragged token batch after a
 * variable-size attention-DP reduce-scatter ("Layer boundaries", section "Choose a
 * reduction policy", value rsv; section "Token layouts and sums": ATTN_DP token
 * sets): rank `set` receives exactly the valid rows of its own token set, global
 * rows [set_offsets[set], set_offsets[set] + set_counts[set]), no padding.
 *
 *   partials       K device pointers, each bf16 [T_pad,H] over the padded batch
 *   set            0 <= set < num_sets (1 <= num_sets <= LB_MAX_SETS)
 *   set_offsets, set_counts   host int32 [num_sets], as for lb_slice_fold_norm
 *   residual_in    bf16 [set_counts[set], H] or NULL (Initial)
 *   residual_out, y_out, q_out/scale_out: compact [set_counts[set], ...] outputs
 */
lb_status lb_slice_fold_norm_v(const void *const *partials, int K, int64_t T_pad, int set,
                               const int32_t *set_offsets, const int32_t *set_counts,
                               int num_sets, const void *residual_in, void *residual_out,
                               const float *gamma, void *y_out, uint8_t *q_out,
                               float *scale_out, int64_t H, float eps,
                               const lb_options *options, lb_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LB_H */
