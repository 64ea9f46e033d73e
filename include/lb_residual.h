/*
 * lb_residual.h — host-side residual stream over the boundary calls of lb.h.
 *
 * "Layer boundaries" (sglang developer guide) carries the residual and the producer's
 * owed contribution from one boundary to the next in a residual stream:
 *   section "Residual stream": the states Initial / Written / Pending, the rule that a
 *     model passes back exactly the value each boundary call returned, and the helpers
 *     complete_output, fold, written and take_output;
 *   section "Enter and leave the layer stack": start() before the stack, the final
 *     norm that releases the stream, and the MoE finalize handoff consumed by the next
 *     read or by the final norm;
 *   section "Auxiliary capture and extra contributions": add_to_output adds an extra
 *     contribution exactly once and keeps the update pending;
 *   section "Integration checklist and common errors": the errors below.
 *
 * This header mirrors that object for C callers.  An lb_residual_stream records the
 * state, the owed contribution (K partial buffers, or a MoE finalize handoff) and the
 * handle of the output the model must pass next; every device operation is one call of
 * lb.h, enqueued on the caller's stream.  The stream is a plain host struct owned by the
 * caller; nothing is allocated and no device state is kept.  A call that returns an
 * error changes nothing (the underlying lb.h call validates before it launches).
 *
 * Handles: an lb_output is the identity of a value handed to the model.  Every call
 * that hands on an output returns a new handle in *out; the next call must pass that
 * handle, else LB_ERR_FOREIGN_OUTPUT (the page's "output does not belong to this
 * residual stream": a rebound or another microbatch's output).
 *
 * Buffers: `residual` (bf16 [T,H], caller-owned, 16-byte aligned) holds the residual;
 * updates are written into it in place.  Partial buffers and handoff tensors must stay
 * valid until the contribution is consumed.
 */
#ifndef LB_RESIDUAL_H
#define LB_RESIDUAL_H

#include "lb.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Stream states ("Residual stream" state table). */
#define LB_RESIDUAL_INITIAL 0  /* neither residual nor contribution */
#define LB_RESIDUAL_WRITTEN 1  /* residual, no pending contribution */
#define LB_RESIDUAL_PENDING 2  /* contribution owed, optionally an existing residual */

/* Kind of the owed contribution. */
#define LB_CONTRIB_PARTIALS 0  /* K partial buffers whose sum is owed */
#define LB_CONTRIB_MOE 1       /* a deferred MoE finalize (HandoffOutput) */

typedef uint64_t lb_output;

typedef struct {
    uint32_t magic;            /* set by lb_residual_init */
    int started;               /* between lb_residual_start and the stack's exit */
    int state;                 /* LB_RESIDUAL_* */
    int has_residual;          /* `residual` holds a residual */
    uint64_t serial;           /* handle the model must pass next */
    void *residual;            /* bf16 [T,H] device buffer */
    int64_t T, H;
    int kind;                  /* LB_CONTRIB_* of a pending contribution */
    int K;                     /* partials: buffers owed */
    const void *partials[LB_MAX_K];
    const void *expert_out;    /* MoE handoff: lb_moe_finalize_fold_norm's inputs */
    int64_t n_expert_rows;
    const int32_t *idx;
    const float *w;
    int topk;
} lb_residual_stream;

/* Bind `residual` (bf16 [T,H]) to a fresh, not yet started stream. */
lb_status lb_residual_init(lb_residual_stream *s, void *residual, int64_t T, int64_t H);

/* Start the layer stack ("Enter and leave the layer stack": start()): the stream becomes
 * Initial; *out is the handle of the stack's input. */
lb_status lb_residual_start(lb_residual_stream *s, lb_output *out);

/* A producer leaves an owed sum of K partial buffers (bf16 [T,H] each, 1 <= K <=
 * LB_MAX_K): the stream becomes Pending.  A stream that is already Pending is refused
 * with LB_ERR_UPDATE_PENDING (its contribution would be lost). */
lb_status lb_residual_leave(lb_residual_stream *s, lb_output h, const void *const *partials,
                            int K, lb_output *out);

/* A producer leaves a deferred MoE finalize (HandoffOutput): the arguments of
 * lb_moe_finalize_fold_norm.  The stream becomes Pending. */
lb_status lb_residual_leave_moe(lb_residual_stream *s, lb_output h, const void *expert_out,
                                int64_t n_expert_rows, const int32_t *idx, const float *w,
                                int topk, lb_output *out);

/* The consumer's input read ("Residual update and input read": update_and_read).
 * Pending: complete the owed work, fold it into the residual (or, with no residual yet,
 * make it the residual: enter) and read, in one fused call; the stream becomes Written.
 * Written: read without another update.  Initial: LB_ERR_INVALID_ARGUMENT (no input).
 * The read is y_out (bf16 [T,H]) and/or q_out + scale_out (FP8 E4M3 codes [T,H] and
 * float32 scales [T]), as in lb_fold_norm / lb_fold_norm_fp8; options as in lb.h. */
lb_status lb_residual_prepare(lb_residual_stream *s, lb_output h, const float *gamma,
                              void *y_out, uint8_t *q_out, float *scale_out, float eps,
                              const lb_options *options, lb_stream_t stream, lb_output *out);

/* "complete_output": finish the owed sum into `sum_out` (bf16 [T,H]) and leave the
 * update pending, now owed as the single buffer `sum_out`.  Written: nothing is owed,
 * nothing is written. */
lb_status lb_residual_complete_output(lb_residual_stream *s, lb_output h, void *sum_out,
                                      lb_stream_t stream, lb_output *out);

/* "fold": complete the contribution and fold it into the residual; the stream becomes
 * Written.  Written: nothing to do. */
lb_status lb_residual_fold(lb_residual_stream *s, lb_output h, lb_stream_t stream,
                           lb_output *out);

/* "add_to_output": add `extra` (bf16 [T,H]) to the output exactly once, keeping the
 * update pending (a Written stream becomes Pending with `extra` owed).  A MoE handoff
 * must be completed first (LB_ERR_UNSUPPORTED); more than LB_MAX_K owed buffers is
 * LB_ERR_UNSUPPORTED. */
lb_status lb_residual_add_to_output(lb_residual_stream *s, lb_output h, const void *extra,
                                    lb_stream_t stream, lb_output *out);

/* "written": the stream becomes Written with `hidden` (bf16 [T,H], caller-owned) as its
 * residual, discarding any pending contribution.  The stream's residual buffer is
 * `hidden` from then on. */
lb_status lb_residual_written(lb_residual_stream *s, lb_output h, void *hidden,
                              lb_output *out);

/* "take_output": release the stream at a terminal exit whose output is already
 * written; *residual receives the residual buffer.  Pending: LB_ERR_UPDATE_PENDING
 * ("write the residual update before taking the final output"); Initial:
 * LB_ERR_INVALID_ARGUMENT. */
lb_status lb_residual_take_output(lb_residual_stream *s, lb_output h, void **residual);

/* The stack's final norm: lb_residual_prepare, then release the stream.  A pending MoE
 * handoff is finalized by the same fused call (pass LB_OPT_GEMMA_WEIGHT for a Gemma
 * final norm). */
lb_status lb_residual_norm(lb_residual_stream *s, lb_output h, const float *gamma,
                           void *y_out, uint8_t *q_out, float *scale_out, float eps,
                           const lb_options *options, lb_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LB_RESIDUAL_H */
