// C-ABI entry points of liblb.so: argument validation, launch shape, dispatch.
//
// Every check runs before anything is enqueued, so a rejected call writes nothing
// ("Layer boundaries", section "Fusion providers and output decisions": a candidate
// that declines must do so before modifying inputs).  The contract of each entry
// point is documented in include/lb.h.
#include <cmath>
#include <cstdint>
#include <atomic>
#include <climits>
#include <cstring>

#include "lb_internal.h"

namespace {

thread_local int g_last_cuda_error = 0;

enum BufId { kOther = 0, kResIn = 1, kResOut = 2 };

struct Buf {
    const void *ptr;
    uint64_t bytes;
    bool output;
    int id;
};

struct BufList {
    Buf b[LB_MAX_K + 16];
    int n = 0;
    void add(const void *ptr, uint64_t bytes, bool output, int id = kOther) {
        b[n++] = Buf{ptr, bytes, output, id};
    }
};

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// An output may not overlap any other buffer, except residual_out == residual_in
// (the in-place fold, element for element).
lb_status check_overlaps(const BufList &l) {
    for (int i = 0; i < l.n; ++i) {
        const Buf &o = l.b[i];
        if (!o.output || o.ptr == nullptr || o.bytes == 0)
            continue;
        const uintptr_t o0 = reinterpret_cast<uintptr_t>(o.ptr), o1 = o0 + o.bytes;
        for (int j = 0; j < l.n; ++j) {
            const Buf &x = l.b[j];
            if (j == i || x.ptr == nullptr || x.bytes == 0)
                continue;
            const uintptr_t x0 = reinterpret_cast<uintptr_t>(x.ptr), x1 = x0 + x.bytes;
            if (o0 >= x1 || x0 >= o1)
                continue;
            const bool in_place = ((o.id == kResOut && x.id == kResIn) ||
                                   (o.id == kResIn && x.id == kResOut)) &&
                                  o0 == x0 && o.bytes == x.bytes;
            if (!in_place)
                return LB_ERR_INVALID_ARGUMENT;
        }
    }
    return LB_OK;
}

lb_status check_shape(int64_t T, int64_t H, float eps) {
    if (T < 0 || H <= 0 || !(eps >= 0.0f) || !std::isfinite(eps))
        return LB_ERR_INVALID_ARGUMENT;
    if (H % 8 != 0 || H > LB_MAX_H)
        return LB_ERR_UNSUPPORTED;
    if (T > LB_MAX_ROWS)                 // grid: rows x 8 CTAs must fit in 2^31 - 1
        return LB_ERR_UNSUPPORTED;
    return LB_OK;
}

lb_status check_tensor(const void *p) {
    return aligned(p, 16) ? LB_OK : LB_ERR_MISALIGNED;
}

#define LB_TRY(expr)                       \
    do {                                   \
        const lb_status s_ = (expr);       \
        if (s_ != LB_OK)                   \
            return s_;                     \
    } while (0)

// Per-device SM count and opt-in shared memory per block, cached after first use.
struct DeviceInfo {
    int sms;
    int smem_optin;
    int device;
};

int device_info(int dev, DeviceInfo *out) {
    static std::atomic<int> cached[64];
    static DeviceInfo info[64];
    if (dev >= 0 && dev < 64 && cached[dev].load(std::memory_order_acquire)) {
        *out = info[dev];
        return 0;
    }
    DeviceInfo d{};
    d.device = dev;
    cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess)
        return static_cast<int>(e);
    if (dev >= 0 && dev < 64) {
        info[dev] = d;
        cached[dev].store(1, std::memory_order_release);
    }
    *out = d;
    return 0;
}

// The launch goes to the device that owns `stream` (the current device for the legacy
// and per-thread default streams); while it is made, that device is current, and the
// caller's current device is restored afterwards.  A stream that is being captured
// into a CUDA graph cannot be asked for its device (cudaStreamGetDevice fails with
// cudaErrorStreamCaptureUnsupported and invalidates the capture), so a capturing
// stream is taken to belong to the current device.
struct StreamDevice {
    int stream_dev = 0;
    int prev_dev = 0;
    bool switched = false;
    int open(cudaStream_t stream) {
        cudaError_t e = cudaGetDevice(&prev_dev);
        stream_dev = prev_dev;
        const bool default_stream = stream == nullptr || stream == cudaStreamLegacy ||
                                    stream == cudaStreamPerThread;
        if (e != cudaSuccess || default_stream)
            return static_cast<int>(e);
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        e = cudaStreamIsCapturing(stream, &cap);
        if (e != cudaSuccess || cap != cudaStreamCaptureStatusNone)
            return static_cast<int>(e);
        e = cudaStreamGetDevice(stream, &stream_dev);
        if (e == cudaSuccess && stream_dev != prev_dev) {
            e = cudaSetDevice(stream_dev);
            switched = e == cudaSuccess;
        }
        return static_cast<int>(e);
    }
    ~StreamDevice() {
        if (switched)
            cudaSetDevice(prev_dev);
    }
};

#ifdef LB_TEST_HOOKS
// Test builds only: the row whose copies the next stream-kernel launches withhold.
static int64_t g_test_withhold_row = -1;
#endif

lb_status launch(const lb::Params &p, lb::Mode mode, bool fp8, int n_inputs,
                 cudaStream_t stream) {
    StreamDevice sd;
    int e0 = sd.open(stream);
    DeviceInfo d;
    if (e0 == 0)
        e0 = device_info(sd.stream_dev, &d);
    if (e0 != 0) {
        g_last_cuda_error = e0;
        return LB_ERR_CUDA;
    }
    lb::Params q = p;
    q.inv_H = 1.0f / static_cast<float>(p.H);
#ifdef LB_TEST_HOOKS
    q.test_withhold_row = g_test_withhold_row;
#endif
    cudaError_t e;
    lb::StreamShape ss;
    if (lb::use_stream_kernel(p.rows, d.sms) &&
        lb::choose_stream_shape(p.rows, p.H, n_inputs, d.sms, d.smem_optin, &ss)) {
        ss.device = d.device;
        ss.smem_optin = d.smem_optin;
        q.stages = ss.stages;
        q.groups = ss.groups;
        q.consumer_warps = ss.consumer_warps;
        e = (mode == lb::kFold) ? lb::launch_fold_stream(q, ss, fp8, stream)
                                : lb::launch_moe_stream(q, ss, fp8, stream);
    } else {
        lb::Shape s;
        if (!lb::choose_shape(p.rows, p.H, d.sms, &s))
            return LB_ERR_UNSUPPORTED;
        q.vec_per_cta = static_cast<int>(((p.H / 8) + s.ctas_per_row - 1) / s.ctas_per_row);
        e = (mode == lb::kFold) ? lb::launch_fold(q, s, fp8, stream)
                                : lb::launch_moe(q, s, fp8, stream);
    }
    if (e != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(e);
        return LB_ERR_CUDA;
    }
    return LB_OK;
}

// Shared validation of the fold family (dense and slice).
lb_status check_fold_inputs(const void *const *partials, int K, int64_t rows_in,
                            const void *residual_in, BufList *l, int64_t H) {
    if (K < 0)
        return LB_ERR_INVALID_ARGUMENT;
    if (K > LB_MAX_K)
        return LB_ERR_UNSUPPORTED;
    if (K > 0 && partials == nullptr)
        return LB_ERR_INVALID_ARGUMENT;
    if (K == 0 && residual_in == nullptr)
        return LB_ERR_INVALID_ARGUMENT;    // nothing to read
    for (int k = 0; k < K; ++k) {
        if (partials[k] == nullptr)
            return LB_ERR_INVALID_ARGUMENT;
        LB_TRY(check_tensor(partials[k]));
        l->add(partials[k], static_cast<uint64_t>(rows_in * H * 2), false);
    }
    return LB_OK;
}

// Residual, gamma and outputs of a call that produces `rows` rows.
lb_status check_stream_buffers(const void *residual_in, void *residual_out,
                               const float *gamma, void *y_out, uint8_t *q_out,
                               float *scale_out, int64_t rows, int64_t H, BufList *l) {
    const bool fp8 = q_out != nullptr || scale_out != nullptr;
    if (fp8 && (q_out == nullptr || scale_out == nullptr))
        return LB_ERR_INVALID_ARGUMENT;
    if (residual_out == nullptr && y_out == nullptr && !fp8)
        return LB_ERR_INVALID_ARGUMENT;    // nothing to produce
    if ((y_out != nullptr || fp8) && gamma == nullptr)
        return LB_ERR_INVALID_ARGUMENT;
    const uint64_t row_bytes = static_cast<uint64_t>(rows * H * 2);
    for (const void *t : {residual_in, static_cast<const void *>(residual_out),
                          static_cast<const void *>(gamma), static_cast<const void *>(y_out),
                          static_cast<const void *>(q_out)})
        if (t != nullptr)
            LB_TRY(check_tensor(t));
    if (scale_out != nullptr && !aligned(scale_out, 4))
        return LB_ERR_MISALIGNED;
    l->add(residual_in, row_bytes, false, kResIn);
    l->add(residual_out, row_bytes, true, kResOut);
    if (y_out != nullptr || fp8)
        l->add(gamma, static_cast<uint64_t>(H * 4), false);
    l->add(y_out, row_bytes, true);
    l->add(q_out, static_cast<uint64_t>(rows * H), true);
    l->add(scale_out, static_cast<uint64_t>(rows * 4), true);
    return LB_OK;
}

// Options: known flags only (the routing promise on the MoE call alone); the snapshot
// is one more output of residual's shape.
lb_status check_options(const lb_options *opt, int64_t rows, int64_t H, BufList *l,
                        bool moe = false) {
    if (opt == nullptr)
        return LB_OK;
    const unsigned int known = LB_OPT_GEMMA_WEIGHT | LB_OPT_RESIDUAL_READY |
                               (moe ? static_cast<unsigned int>(LB_OPT_ROUTING_READY) : 0u);
    if (opt->flags & ~known)
        return LB_ERR_UNSUPPORTED;
    if (opt->residual_snapshot != nullptr) {
        LB_TRY(check_tensor(opt->residual_snapshot));
        l->add(opt->residual_snapshot, static_cast<uint64_t>(rows * H * 2), true);
    }
    return LB_OK;
}

void set_options(lb::Params *p, const lb_options *opt) {
    p->gemma = (opt != nullptr && (opt->flags & LB_OPT_GEMMA_WEIGHT)) ? 1 : 0;
    p->routing_ready = (opt != nullptr && (opt->flags & LB_OPT_ROUTING_READY)) ? 1 : 0;
    p->residual_ready = (opt != nullptr && (opt->flags & LB_OPT_RESIDUAL_READY)) ? 1 : 0;
    p->snapshot = opt != nullptr ? static_cast<uint16_t *>(opt->residual_snapshot) : nullptr;
}

void set_stream_params(lb::Params *p, const void *residual_in, void *residual_out,
                       const float *gamma, void *y_out, uint8_t *q_out, float *scale_out,
                       int64_t rows, int64_t H, float eps) {
    p->residual_in = static_cast<const uint16_t *>(residual_in);
    p->residual_out = static_cast<uint16_t *>(residual_out);
    p->gamma = gamma;
    p->y_out = static_cast<uint16_t *>(y_out);
    p->q_out = q_out;
    p->scale_out = scale_out;
    p->rows = rows;
    p->H = H;
    p->eps = eps;
}

lb_status fold_common(const void *const *partials, int K, const void *residual_in,
                      void *residual_out, const float *gamma, void *y_out, uint8_t *q_out,
                      float *scale_out, int64_t T, int64_t H, float eps,
                      const lb_options *opt, lb_stream_t stream) {
    LB_TRY(check_shape(T, H, eps));
    if (K < 0)
        return LB_ERR_INVALID_ARGUMENT;
    if (K > LB_MAX_K)
        return LB_ERR_UNSUPPORTED;
    if (T == 0)
        return LB_OK;                          // empty batch: no pointer is used
    BufList l;
    LB_TRY(check_fold_inputs(partials, K, T, residual_in, &l, H));
    LB_TRY(check_stream_buffers(residual_in, residual_out, gamma, y_out, q_out, scale_out, T,
                                H, &l));
    LB_TRY(check_options(opt, T, H, &l));
    LB_TRY(check_overlaps(l));
    lb::Params p;
    std::memset(&p, 0, sizeof p);
    for (int k = 0; k < K; ++k)
        p.partials[k] = static_cast<const uint16_t *>(partials[k]);
    p.K = K;
    set_stream_params(&p, residual_in, residual_out, gamma, y_out, q_out, scale_out, T, H,
                      eps);
    set_options(&p, opt);
    return launch(p, lb::kFold, q_out != nullptr, K + (residual_in != nullptr ? 1 : 0),
                  reinterpret_cast<cudaStream_t>(stream));
}

// Shared validation of the ragged set metadata: sets ascending, disjoint, inside.
lb_status check_sets(const int32_t *set_offsets, const int32_t *set_counts, int num_sets,
                     int64_t T_pad) {
    if (num_sets < 0)
        return LB_ERR_INVALID_ARGUMENT;
    if (num_sets > LB_MAX_SETS)
        return LB_ERR_UNSUPPORTED;
    if (num_sets > 0 && (set_offsets == nullptr || set_counts == nullptr))
        return LB_ERR_INVALID_ARGUMENT;
    int64_t prev_end = 0;
    for (int s = 0; s < num_sets; ++s) {
        const int64_t lo = set_offsets[s], n = set_counts[s];
        if (lo < prev_end || n < 0 || lo + n > T_pad)
            return LB_ERR_INVALID_ARGUMENT;
        prev_end = lo + n;
    }
    return LB_OK;
}

}  // namespace

namespace lb {

bool use_stream_kernel(int64_t rows, int num_sms) {
    // More rows than SMs; up to one row per SM the row kernel (one CTA per row, all in
    // one wave; a cluster only for rows longer than one CTA holds) measured faster
    // (K=8 T=152 H=4096: 4.24 against 5.24 us), beyond that the stream kernel (254
    // rows: 6.63 against 7.29 us).
    return rows > num_sms;
}

bool choose_stream_shape(int64_t rows, int64_t H, int n_inputs, int num_sms,
                         int smem_per_block, StreamShape *out) {
    if (rows <= 0 || H <= 0 || H % 8 != 0 || n_inputs < 1 || n_inputs > LB_MAX_K + 1 ||
        num_sms <= 0)
        return false;
    const int64_t nvec = H / 8;
    if (nvec <= LB_STREAM_MIN_ROW_VECS)
        return false;                          // short rows: the row kernel measured faster
    const int64_t wide = LB_STREAM_CONSUMER_WARPS_WIDE;
    int64_t per_cta = LB_SMEM_PER_SM / LB_STREAM_CTAS_PER_SM - 1024;
    if (per_cta > smem_per_block)
        per_cta = smem_per_block;
    const int64_t reserve = 1024;              // static shared memory and mbarriers
    // Stages that fit when a stage holds `width` columns of every input row: per
    // stage its input rows, two mbarriers and two row-metadata blocks, plus (chunked
    // rows) the read weight of H floats once.
    auto stages_for = [&](int64_t width, int64_t weight_bytes) {
        const int64_t per_stage =
            static_cast<int64_t>(n_inputs) * width * 2 + 16 + 2 * LB_STREAM_META_BYTES;
        int64_t ns = (per_cta - reserve - weight_bytes) / per_stage;
        return ns > LB_STREAM_MAX_STAGES ? static_cast<int64_t>(LB_STREAM_MAX_STAGES) : ns;
    };
    int ncw = 0;                               // warps per consumer group (even)
    int64_t vpt = 0;                           // vectors per thread; 4 = chunked rows
    int64_t chunks = 1;                        // stages per row
    int64_t groups_cap = LB_STREAM_GROUPS;
    int64_t ns = 0;
    if (nvec < LB_STREAM_CHUNK_FROM) {
        // Whole rows per stage.
        if (nvec <= 2 * 32 * LB_STREAM_CONSUMER_WARPS) {
            const int64_t maxw = LB_STREAM_CONSUMER_WARPS;
            ncw = static_cast<int>(nvec >= 32 * maxw ? maxw : (nvec + 31) / 32);
            ncw += ncw & 1;                    // an even number of warps per group
            vpt = (nvec + ncw * 32 - 1) / (ncw * 32) <= 1 ? 1 : 2;
        } else {
            // Rows of up to 2 x 32 x `wide` vectors keep two vectors per thread with
            // wider groups (as many as fit the two-vector thread budget).
            ncw = static_cast<int>((nvec + 63) / 64);
            ncw += ncw & 1;
            vpt = 2;
            groups_cap = (LB_STREAM_THREADS_2 / 32 - 1) / ncw;   // consumer warps left
        }
        ns = groups_cap >= 1 ? stages_for(H, 0) : 0;
    }
    if (ns < 2 && nvec < LB_STREAM_CHUNK_FROM)
        return false;                          // many inputs: the row kernel measured faster
    if (ns < 2) {
        // Long rows: 2-4 column chunks of 32 x ncw vectors, one group of up to `wide`
        // warps; chunk c holds the row's vectors [c, c + 1) x 32 x ncw and thread t
        // keeps vector t of each.
        ns = 0;
        for (chunks = 2; chunks <= 4 && ns < 2; ++chunks) {
            ncw = static_cast<int>((nvec + 32 * chunks - 1) / (32 * chunks));
            ncw += ncw & 1;
            if (ncw > wide)
                continue;
            ns = stages_for(static_cast<int64_t>(ncw) * 256, H * 4);
        }
        if (ns < 2)
            return false;
        chunks = (nvec + 32 * ncw - 1) / (32 * ncw);   // the last chunk may be short
        vpt = 4;
        groups_cap = 1;
    }
    // Row i uses stage i % ns and consumer group i % groups (chunked rows: chunk c of
    // row i uses stage (i x chunks + c) % ns, one group).  The stage count is a
    // multiple of the group count, so that every stage belongs to one group and its
    // uses are consumed in order: a parity wait on an mbarrier tells only two
    // consecutive phases apart.
    int64_t groups = groups_cap > LB_STREAM_GROUPS ? LB_STREAM_GROUPS : groups_cap;
    if (groups > ns)
        groups = ns;
    ns -= ns % groups;
    const int64_t width = chunks > 1 ? static_cast<int64_t>(ncw) * 256 : H;
    const int64_t per_stage =
        static_cast<int64_t>(n_inputs) * width * 2 + 16 + 2 * LB_STREAM_META_BYTES;
    const int64_t ctas = static_cast<int64_t>(num_sms) * LB_STREAM_CTAS_PER_SM;
    out->grid = static_cast<int>(rows < ctas ? rows : ctas);
    out->groups = static_cast<int>(groups);
    out->consumer_warps = ncw;
    out->vpt = static_cast<int>(vpt);
    out->chunks = static_cast<int>(chunks);
    out->stages = static_cast<int>(ns);
    out->smem_bytes = static_cast<int>(ns * per_stage + (chunks > 1 ? H * 4 : 0));
    return true;
}

bool choose_shape(int64_t rows, int64_t H, int num_sms, Shape *out) {
    if (rows < 0 || H <= 0 || H % 8 != 0 || num_sms <= 0)
        return false;
    const int64_t nvec = H / 8;
    // One CTA per row: splitting short rows over a cluster measured slower at decode
    // sizes (cluster scheduling and barriers cost more than the extra SMs give).
    int cs = 1;
    (void)rows;
    (void)num_sms;
    // Long rows: at most 512 threads x 4 vectors per CTA, else a cluster splits them.
    while (cs < 8 && (nvec + cs - 1) / cs > 2048)
        cs *= 2;
    const int64_t vpc = (nvec + cs - 1) / cs;
    if (vpc > 2048)
        return false;
    const int vpt = vpc <= 512 ? 1 : (vpc <= 1024 ? 2 : 4);
    int64_t threads = (vpc + vpt - 1) / vpt;
    threads = ((threads + 31) / 32) * 32;
    out->threads = static_cast<int>(threads);
    out->vpt = vpt;
    out->ctas_per_row = cs;
    return true;
}

}  // namespace lb

extern "C" {

const char *lb_status_string(lb_status status) {
    switch (status) {
    case LB_OK: return "LB_OK";
    case LB_ERR_INVALID_ARGUMENT: return "LB_ERR_INVALID_ARGUMENT";
    case LB_ERR_MISALIGNED: return "LB_ERR_MISALIGNED";
    case LB_ERR_UNSUPPORTED: return "LB_ERR_UNSUPPORTED";
    case LB_ERR_CUDA: return "LB_ERR_CUDA";
    case LB_ERR_NOT_STARTED: return "LB_ERR_NOT_STARTED";
    case LB_ERR_FOREIGN_OUTPUT: return "LB_ERR_FOREIGN_OUTPUT";
    case LB_ERR_UPDATE_PENDING: return "LB_ERR_UPDATE_PENDING";
    }
    return "LB_ERR_UNKNOWN";
}

int lb_last_cuda_error(void) { return g_last_cuda_error; }

int lb_version(void) { return 100; }

#ifdef LB_TEST_HOOKS
// Test builds only (not declared in the public headers): make the stream kernel post a
// row's bytes without issuing its copies (-1: none), to exercise the bounded waits.
void lb_test_withhold_row(int64_t row) { g_test_withhold_row = row; }
#endif

lb_status lb_launch_plan(int64_t rows, int64_t H, int n_inputs, int num_sms,
                         int smem_per_block, lb_plan *plan) {
    if (plan == nullptr || n_inputs < 1 || n_inputs > LB_MAX_K + 1)
        return LB_ERR_INVALID_ARGUMENT;
    std::memset(plan, 0, sizeof *plan);
    lb::StreamShape ss;
    if (lb::use_stream_kernel(rows, num_sms) &&
        lb::choose_stream_shape(rows, H, n_inputs, num_sms, smem_per_block, &ss)) {
        plan->kernel = LB_KERNEL_STREAM;
        plan->grid = ss.grid;
        plan->threads = 32 * (1 + ss.groups * ss.consumer_warps);
        plan->vectors_per_thread = ss.vpt;
        plan->ctas_per_row = 1;
        plan->stages = ss.stages;
        plan->smem_bytes = ss.smem_bytes;
        plan->groups = ss.groups;
        plan->chunks = ss.chunks;
        return LB_OK;
    }
    lb::Shape s;
    if (!lb::choose_shape(rows, H, num_sms, &s))
        return LB_ERR_UNSUPPORTED;
    plan->kernel = LB_KERNEL_ROW;
    plan->grid = static_cast<int>(rows * s.ctas_per_row);
    plan->threads = s.threads;
    plan->vectors_per_thread = s.vpt;
    plan->ctas_per_row = s.ctas_per_row;
    return LB_OK;
}

lb_status lb_device_error(unsigned int *flags, int clear) {
    if (flags == nullptr)
        return LB_ERR_INVALID_ARGUMENT;
    cudaError_t e = cudaDeviceSynchronize();
    unsigned int a = 0, b = 0;
    if (e == cudaSuccess)
        e = lb::fold_device_error(&a, clear != 0);
    if (e == cudaSuccess)
        e = lb::moe_device_error(&b, clear != 0);
    if (e != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(e);
        return LB_ERR_CUDA;
    }
    *flags = a | b;
    return LB_OK;
}

lb_status lb_fold_norm(const void *const *partials, int K, const void *residual_in,
                       void *residual_out, const float *gamma, void *y_out, int64_t T,
                       int64_t H, float eps, const lb_options *options, lb_stream_t stream) {
    return fold_common(partials, K, residual_in, residual_out, gamma, y_out, nullptr,
                       nullptr, T, H, eps, options, stream);
}

lb_status lb_fold_norm_fp8(const void *const *partials, int K, const void *residual_in,
                           void *residual_out, const float *gamma, uint8_t *q_out,
                           float *scale_out, void *y_out, int64_t T, int64_t H, float eps,
                           const lb_options *options, lb_stream_t stream) {
    if (q_out == nullptr || scale_out == nullptr)
        return LB_ERR_INVALID_ARGUMENT;
    return fold_common(partials, K, residual_in, residual_out, gamma, y_out, q_out,
                       scale_out, T, H, eps, options, stream);
}

lb_status lb_moe_finalize_fold_norm(const void *expert_out, int64_t n_expert_rows,
                                    const int32_t *idx, const float *w, int topk,
                                    const void *residual_in, void *residual_out,
                                    const float *gamma, void *y_out, uint8_t *q_out,
                                    float *scale_out, int64_t T, int64_t H, float eps,
                                    int32_t *bad_index_flag, const lb_options *options,
                                    lb_stream_t stream) {
    LB_TRY(check_shape(T, H, eps));
    if (topk < 1 || n_expert_rows < 0)
        return LB_ERR_INVALID_ARGUMENT;
    if (topk > LB_MAX_TOPK || n_expert_rows > (int64_t(1) << 31))
        return LB_ERR_UNSUPPORTED;
    if (T == 0)
        return LB_OK;                          // empty batch: no pointer is used
    if (expert_out == nullptr || idx == nullptr || w == nullptr)
        return LB_ERR_INVALID_ARGUMENT;
    LB_TRY(check_tensor(expert_out));
    if (!aligned(idx, 4) || !aligned(w, 4) ||
        (bad_index_flag != nullptr && !aligned(bad_index_flag, 4)))
        return LB_ERR_MISALIGNED;
    BufList l;
    l.add(expert_out, static_cast<uint64_t>(n_expert_rows * H * 2), false);
    l.add(idx, static_cast<uint64_t>(T * topk * 4), false);
    l.add(w, static_cast<uint64_t>(T * topk * 4), false);
    l.add(bad_index_flag, 4, true);
    LB_TRY(check_stream_buffers(residual_in, residual_out, gamma, y_out, q_out, scale_out, T,
                                H, &l));
    LB_TRY(check_options(options, T, H, &l, true));
    LB_TRY(check_overlaps(l));
    lb::Params p;
    std::memset(&p, 0, sizeof p);
    p.expert_out = static_cast<const uint16_t *>(expert_out);
    p.n_expert_rows = n_expert_rows;
    p.idx = idx;
    p.w = w;
    p.topk = topk;
    p.bad_index = bad_index_flag;
    set_stream_params(&p, residual_in, residual_out, gamma, y_out, q_out, scale_out, T, H,
                      eps);
    set_options(&p, options);
    return launch(p, lb::kMoe, q_out != nullptr, topk + (residual_in != nullptr ? 1 : 0),
                  reinterpret_cast<cudaStream_t>(stream));
}

lb_status lb_slice_fold_norm(const void *const *partials, int K, int64_t T_pad,
                             int num_slices, int slice, const int32_t *set_offsets,
                             const int32_t *set_counts, int num_sets,
                             const void *residual_in, void *residual_out,
                             const float *gamma, void *y_out, uint8_t *q_out,
                             float *scale_out, int64_t H, float eps,
                             const lb_options *options, lb_stream_t stream) {
    if (T_pad < 0 || num_slices < 1 || T_pad % num_slices != 0 || slice < 0 ||
        slice >= num_slices || num_sets < 0)
        return LB_ERR_INVALID_ARGUMENT;
    if (num_sets > LB_MAX_SETS || T_pad > INT32_MAX)
        return LB_ERR_UNSUPPORTED;
    LB_TRY(check_sets(set_offsets, set_counts, num_sets, T_pad));
    const int64_t S = T_pad / num_slices;
    LB_TRY(check_shape(S, H, eps));
    if (K < 0)
        return LB_ERR_INVALID_ARGUMENT;
    if (K > LB_MAX_K)
        return LB_ERR_UNSUPPORTED;
    if (S == 0)
        return LB_OK;                          // empty batch: no pointer is used
    BufList l;
    LB_TRY(check_fold_inputs(partials, K, T_pad, residual_in, &l, H));
    LB_TRY(check_stream_buffers(residual_in, residual_out, gamma, y_out, q_out, scale_out, S,
                                H, &l));
    LB_TRY(check_options(options, S, H, &l));
    LB_TRY(check_overlaps(l));
    lb::Params p;
    std::memset(&p, 0, sizeof p);
    for (int k = 0; k < K; ++k)
        p.partials[k] = static_cast<const uint16_t *>(partials[k]);
    p.K = K;
    p.in_row0 = static_cast<int64_t>(slice) * S;
    p.num_sets = num_sets;
    bool any_valid = num_sets == 0;
    for (int s = 0; s < num_sets; ++s) {
        p.set_lo[s] = set_offsets[s];
        p.set_hi[s] = set_offsets[s] + set_counts[s];
        any_valid |= (p.set_lo[s] < p.in_row0 + S) && (p.set_hi[s] > p.in_row0) &&
                     (set_counts[s] > 0);
    }
    if (!any_valid)
        return LB_OK;                          // the slice holds padding only
    set_stream_params(&p, residual_in, residual_out, gamma, y_out, q_out, scale_out, S, H,
                      eps);
    set_options(&p, options);
    return launch(p, lb::kFold, q_out != nullptr, K + (residual_in != nullptr ? 1 : 0),
                  reinterpret_cast<cudaStream_t>(stream));
}

lb_status lb_slice_fold_norm_v(const void *const *partials, int K, int64_t T_pad, int set,
                               const int32_t *set_offsets, const int32_t *set_counts,
                               int num_sets, const void *residual_in, void *residual_out,
                               const float *gamma, void *y_out, uint8_t *q_out,
                               float *scale_out, int64_t H, float eps,
                               const lb_options *options, lb_stream_t stream) {
    if (T_pad < 0 || num_sets < 1 || set < 0 || set >= num_sets)
        return LB_ERR_INVALID_ARGUMENT;
    if (num_sets > LB_MAX_SETS || T_pad > INT32_MAX)
        return LB_ERR_UNSUPPORTED;
    LB_TRY(check_sets(set_offsets, set_counts, num_sets, T_pad));
    const int64_t rows = set_counts[set];
    LB_TRY(check_shape(rows, H, eps));
    if (K < 0)
        return LB_ERR_INVALID_ARGUMENT;
    if (K > LB_MAX_K)
        return LB_ERR_UNSUPPORTED;
    if (rows == 0)
        return LB_OK;                          // empty set: no pointer is used
    BufList l;
    LB_TRY(check_fold_inputs(partials, K, T_pad, residual_in, &l, H));
    LB_TRY(check_stream_buffers(residual_in, residual_out, gamma, y_out, q_out, scale_out,
                                rows, H, &l));
    LB_TRY(check_options(options, rows, H, &l));
    LB_TRY(check_overlaps(l));
    lb::Params p;
    std::memset(&p, 0, sizeof p);
    for (int k = 0; k < K; ++k)
        p.partials[k] = static_cast<const uint16_t *>(partials[k]);
    p.K = K;
    p.in_row0 = set_offsets[set];              // every row of the set is valid
    set_stream_params(&p, residual_in, residual_out, gamma, y_out, q_out, scale_out, rows, H,
                      eps);
    set_options(&p, options);
    return launch(p, lb::kFold, q_out != nullptr, K + (residual_in != nullptr ? 1 : 0),
                  reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
