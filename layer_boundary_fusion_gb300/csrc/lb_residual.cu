// Host-side residual stream (include/lb_residual.h): the state, owed contribution and
// output handle of "Layer boundaries", sections "Residual stream", "Enter and leave the
// layer stack", "Auxiliary capture and extra contributions" and "Integration checklist
// and common errors".  Every device operation is one call of the boundary entry points
// in lb_api.cu; nothing here touches device memory itself.
#include "lb_residual.h"

#include <cstring>

namespace {

constexpr uint32_t kMagic = 0x4C425253u;   // "LBRS"

bool bound(const lb_residual_stream *s) { return s != nullptr && s->magic == kMagic; }

// The checks every operation on a model-held output makes, in the page's order: the
// stack must have started, and the handle must be the one handed out last.
lb_status check_handle(const lb_residual_stream *s, lb_output h) {
    if (!bound(s))
        return LB_ERR_INVALID_ARGUMENT;
    if (!s->started)
        return LB_ERR_NOT_STARTED;
    if (h != s->serial)
        return LB_ERR_FOREIGN_OUTPUT;
    return LB_OK;
}

lb_output hand_on(lb_residual_stream *s, lb_output *out) {
    ++s->serial;
    if (out != nullptr)
        *out = s->serial;
    return s->serial;
}

void clear_contribution(lb_residual_stream *s) {
    s->kind = LB_CONTRIB_PARTIALS;
    s->K = 0;
    std::memset(s->partials, 0, sizeof s->partials);
    s->expert_out = nullptr;
    s->n_expert_rows = 0;
    s->idx = nullptr;
    s->w = nullptr;
    s->topk = 0;
}

// Complete the owed contribution into residual_out (in place over the residual when
// residual_out is the residual) together with the optional read, in one boundary call.
lb_status complete_and_read(lb_residual_stream *s, void *residual_out, bool fold,
                            const float *gamma, void *y_out, uint8_t *q_out,
                            float *scale_out, float eps, const lb_options *options,
                            lb_stream_t stream) {
    const void *res_in = (fold && s->has_residual) ? s->residual : nullptr;
    if (s->kind == LB_CONTRIB_MOE)
        return lb_moe_finalize_fold_norm(s->expert_out, s->n_expert_rows, s->idx, s->w,
                                         s->topk, res_in, residual_out, gamma, y_out, q_out,
                                         scale_out, s->T, s->H, eps, nullptr, options, stream);
    if (q_out != nullptr || scale_out != nullptr)
        return lb_fold_norm_fp8(s->partials, s->K, res_in, residual_out, gamma, q_out,
                                scale_out, y_out, s->T, s->H, eps, options, stream);
    return lb_fold_norm(s->partials, s->K, res_in, residual_out, gamma, y_out, s->T, s->H,
                        eps, options, stream);
}

}  // namespace

extern "C" {

lb_status lb_residual_init(lb_residual_stream *s, void *residual, int64_t T, int64_t H) {
    if (s == nullptr || T < 0 || H <= 0)
        return LB_ERR_INVALID_ARGUMENT;
    if (T > 0 && residual == nullptr)
        return LB_ERR_INVALID_ARGUMENT;
    std::memset(s, 0, sizeof *s);
    s->magic = kMagic;
    s->residual = residual;
    s->T = T;
    s->H = H;
    s->state = LB_RESIDUAL_INITIAL;
    return LB_OK;
}

lb_status lb_residual_start(lb_residual_stream *s, lb_output *out) {
    if (!bound(s))
        return LB_ERR_INVALID_ARGUMENT;
    s->started = 1;
    s->state = LB_RESIDUAL_INITIAL;
    s->has_residual = 0;
    clear_contribution(s);
    hand_on(s, out);
    return LB_OK;
}

lb_status lb_residual_leave(lb_residual_stream *s, lb_output h, const void *const *partials,
                            int K, lb_output *out) {
    const lb_status st = check_handle(s, h);
    if (st != LB_OK)
        return st;
    if (s->state == LB_RESIDUAL_PENDING)
        return LB_ERR_UPDATE_PENDING;
    if (K < 1 || partials == nullptr)
        return LB_ERR_INVALID_ARGUMENT;
    if (K > LB_MAX_K)
        return LB_ERR_UNSUPPORTED;
    for (int k = 0; k < K; ++k)
        if (partials[k] == nullptr && s->T > 0)
            return LB_ERR_INVALID_ARGUMENT;
    clear_contribution(s);
    s->kind = LB_CONTRIB_PARTIALS;
    s->K = K;
    for (int k = 0; k < K; ++k)
        s->partials[k] = partials[k];
    s->state = LB_RESIDUAL_PENDING;
    hand_on(s, out);
    return LB_OK;
}

lb_status lb_residual_leave_moe(lb_residual_stream *s, lb_output h, const void *expert_out,
                                int64_t n_expert_rows, const int32_t *idx, const float *w,
                                int topk, lb_output *out) {
    const lb_status st = check_handle(s, h);
    if (st != LB_OK)
        return st;
    if (s->state == LB_RESIDUAL_PENDING)
        return LB_ERR_UPDATE_PENDING;
    if (topk < 1 || n_expert_rows < 0)
        return LB_ERR_INVALID_ARGUMENT;
    if (topk > LB_MAX_TOPK)
        return LB_ERR_UNSUPPORTED;
    if (s->T > 0 && (expert_out == nullptr || idx == nullptr || w == nullptr))
        return LB_ERR_INVALID_ARGUMENT;
    clear_contribution(s);
    s->kind = LB_CONTRIB_MOE;
    s->expert_out = expert_out;
    s->n_expert_rows = n_expert_rows;
    s->idx = idx;
    s->w = w;
    s->topk = topk;
    s->state = LB_RESIDUAL_PENDING;
    hand_on(s, out);
    return LB_OK;
}

lb_status lb_residual_prepare(lb_residual_stream *s, lb_output h, const float *gamma,
                              void *y_out, uint8_t *q_out, float *scale_out, float eps,
                              const lb_options *options, lb_stream_t stream, lb_output *out) {
    lb_status st = check_handle(s, h);
    if (st != LB_OK)
        return st;
    if (y_out == nullptr && q_out == nullptr && scale_out == nullptr)
        return LB_ERR_INVALID_ARGUMENT;            // a read produces something
    switch (s->state) {
    case LB_RESIDUAL_PENDING:
        // update_and_read: complete, fold (or enter) and read in one call
        st = complete_and_read(s, s->residual, true, gamma, y_out, q_out, scale_out, eps,
                               options, stream);
        if (st != LB_OK)
            return st;
        clear_contribution(s);
        s->has_residual = 1;
        s->state = LB_RESIDUAL_WRITTEN;
        break;
    case LB_RESIDUAL_WRITTEN:
        // read without another update: K = 0, no residual output
        if (q_out != nullptr || scale_out != nullptr)
            st = lb_fold_norm_fp8(nullptr, 0, s->residual, nullptr, gamma, q_out, scale_out,
                                  y_out, s->T, s->H, eps, options, stream);
        else
            st = lb_fold_norm(nullptr, 0, s->residual, nullptr, gamma, y_out, s->T, s->H, eps,
                              options, stream);
        if (st != LB_OK)
            return st;
        break;
    default:
        return LB_ERR_INVALID_ARGUMENT;            // Initial: no input to read
    }
    hand_on(s, out);
    return LB_OK;
}

lb_status lb_residual_complete_output(lb_residual_stream *s, lb_output h, void *sum_out,
                                      lb_stream_t stream, lb_output *out) {
    lb_status st = check_handle(s, h);
    if (st != LB_OK)
        return st;
    if (s->state == LB_RESIDUAL_PENDING) {
        if (sum_out == nullptr && s->T > 0)
            return LB_ERR_INVALID_ARGUMENT;
        // complete_output mode of the boundary call: no residual, no read
        st = complete_and_read(s, sum_out, false, nullptr, nullptr, nullptr, nullptr, 0.0f,
                               nullptr, stream);
        if (st != LB_OK)
            return st;
        clear_contribution(s);
        s->kind = LB_CONTRIB_PARTIALS;
        s->K = 1;
        s->partials[0] = sum_out;                  // the update stays pending
    } else if (s->state != LB_RESIDUAL_WRITTEN) {
        return LB_ERR_INVALID_ARGUMENT;            // Initial: nothing produced yet
    }
    hand_on(s, out);
    return LB_OK;
}

lb_status lb_residual_fold(lb_residual_stream *s, lb_output h, lb_stream_t stream,
                           lb_output *out) {
    lb_status st = check_handle(s, h);
    if (st != LB_OK)
        return st;
    if (s->state == LB_RESIDUAL_PENDING) {
        st = complete_and_read(s, s->residual, true, nullptr, nullptr, nullptr, nullptr, 0.0f,
                               nullptr, stream);
        if (st != LB_OK)
            return st;
        clear_contribution(s);
        s->has_residual = 1;
        s->state = LB_RESIDUAL_WRITTEN;
    } else if (s->state != LB_RESIDUAL_WRITTEN) {
        return LB_ERR_INVALID_ARGUMENT;
    }
    hand_on(s, out);
    return LB_OK;
}

lb_status lb_residual_add_to_output(lb_residual_stream *s, lb_output h, const void *extra,
                                    lb_stream_t stream, lb_output *out) {
    (void)stream;                                  // the extra buffer joins the owed sum
    const lb_status st = check_handle(s, h);
    if (st != LB_OK)
        return st;
    if (extra == nullptr && s->T > 0)
        return LB_ERR_INVALID_ARGUMENT;
    if (s->state == LB_RESIDUAL_PENDING) {
        if (s->kind == LB_CONTRIB_MOE)
            return LB_ERR_UNSUPPORTED;             // complete the handoff first
        if (s->K >= LB_MAX_K)
            return LB_ERR_UNSUPPORTED;
        s->partials[s->K++] = extra;
    } else if (s->state == LB_RESIDUAL_WRITTEN) {
        clear_contribution(s);
        s->K = 1;
        s->partials[0] = extra;
        s->state = LB_RESIDUAL_PENDING;
    } else {
        return LB_ERR_INVALID_ARGUMENT;
    }
    hand_on(s, out);
    return LB_OK;
}

lb_status lb_residual_written(lb_residual_stream *s, lb_output h, void *hidden,
                              lb_output *out) {
    const lb_status st = check_handle(s, h);
    if (st != LB_OK)
        return st;
    if (hidden == nullptr && s->T > 0)
        return LB_ERR_INVALID_ARGUMENT;
    clear_contribution(s);                          // a pending contribution is discarded
    s->residual = hidden;
    s->has_residual = 1;
    s->state = LB_RESIDUAL_WRITTEN;
    hand_on(s, out);
    return LB_OK;
}

lb_status lb_residual_take_output(lb_residual_stream *s, lb_output h, void **residual) {
    const lb_status st = check_handle(s, h);
    if (st != LB_OK)
        return st;
    if (s->state == LB_RESIDUAL_PENDING)
        return LB_ERR_UPDATE_PENDING;
    if (s->state != LB_RESIDUAL_WRITTEN)
        return LB_ERR_INVALID_ARGUMENT;
    if (residual != nullptr)
        *residual = s->residual;
    s->started = 0;                                 // released
    ++s->serial;
    return LB_OK;
}

lb_status lb_residual_norm(lb_residual_stream *s, lb_output h, const float *gamma,
                           void *y_out, uint8_t *q_out, float *scale_out, float eps,
                           const lb_options *options, lb_stream_t stream) {
    const lb_status st = lb_residual_prepare(s, h, gamma, y_out, q_out, scale_out, eps,
                                             options, stream, nullptr);
    if (st != LB_OK)
        return st;
    s->started = 0;                                 // the final norm releases the stream
    return LB_OK;
}

}  // extern "C"
