// Persistent, warp-specialised boundary kernel for sm_103a: TMA bulk copies stream
// every input row of the boundary into a ring of shared-memory stages while the
// consumer warps fold, reduce and store earlier rows.
//
//   warp 0 (producer): for each of this CTA's rows, wait until its stage is free,
//     post the byte count on the stage's "full" mbarrier and issue one
//     cp.async.bulk (global -> shared) per input row: the K partial rows (or the
//     gathered expert rows of a MoE finalize) and the residual row (lane 0 in turn,
//     or one lane per row for short slots and for expert rows).  A MoE token's
//     expert indices and routing weights are fetched two rows ahead (cp.async) into
//     a ring of per-row metadata blocks beside the stages.  On the caller's promises
//     the first rows' routing and residual rows go out before griddepcontrol.wait.
//   consumer groups of W warps (rows dealt to the groups in turn, so that several
//     rows are reduced at once): wait on "full", fold the stage's rows in binary32 in
//     the definition's order, hand the stage back ("empty" mbarrier, one arrive per
//     warp), store residual', reduce sum(o^2) (and max|o*gamma| for FP8) across the
//     group with shuffles and ONE named barrier per row, and store the bf16 read or
//     the FP8 codes and scale.  gamma stays in registers for the whole kernel (in
//     shared memory for rows split into column chunks, one chunk per stage).
//
// Loads in flight per SM are bounded by the stages (up to ~220 KB), not by
// registers, and the fixed per-row costs (one barrier, one rsqrt) are spread over
// 8-32 elements per consumer thread.
//
// Every wait is bounded: after about a second without progress the waiting thread
// records LB_DEVICE_ERR_TIMEOUT in the library's device error word, the CTA stops
// taking rows, the producer waits (again bounded) for the copies it has in flight,
// and the kernel returns.
//
// Sources: "Layer boundaries" (sglang developer guide), sections "Residual stream"
// and "Residual update and input read"; "SGLang flashinfer_allreduce_fusion精读",
// section forward.  The pipeline itself is this library's GB300 design.
#pragma once

#include "lb_kernel.cuh"

namespace lb {

// Device error word of this translation unit (bit flags: LB_DEVICE_ERR_*), read and
// cleared through lb_device_error().  Each kernel translation unit has its own copy.
static __device__ unsigned int g_device_error = 0;
constexpr unsigned int kDeviceErrTimeout = 1u;
constexpr unsigned int kDeviceErrLaunch = 2u;

// Host side: synchronise nothing, read and optionally clear this unit's word.
static inline cudaError_t read_device_error(unsigned int *out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(unsigned int));
    if (e == cudaSuccess && clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
    }
    return e;
}

// ------------------------------------------------------------------------------------
// mbarrier / bulk-copy primitives
// ------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Post bytes that the current phase must also receive, without arriving: the phase
// still completes only at the (single) arrival and once every posted byte has landed.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// As mbar_try_wait, but the thread may stay suspended in the instruction until the
// phase completes or about `hint_ns` have passed: a waiter then issues a handful of
// instructions per wait instead of polling, leaving the SM's issue slots to the
// warps that are working.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity,
                                                      uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase with the given parity: at most 2^24 suspending waits of
// up to 20 us each and about one second in all.  `abort_flag` (shared) is read after
// every wait, so a waiter gives up early once another warp of the CTA has given up.
// Returns false on time-out or abort.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0; it < (1u << 24); ++it) {
        if (mbar_try_wait_suspend(bar, parity, 20000u))
            return true;
        if (abort_flag != nullptr && *abort_flag)
            return false;
        if (global_timer_ns() - t0 > 1000000000ull)
            return false;
    }
    return false;
}

// 16 bytes from this CTA's shared memory (32-bit shared-window address).
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// One bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 4 bytes global -> shared by the issuing thread (cp.async), in the thread's current
// group; the copy is complete for that thread after a wait covering its group.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most `n` of this thread's committed groups are pending (n <= 7;
// larger n waits for all of them).
__device__ __forceinline__ void cp_async_wait_pending(int n) {
    switch (n) {
    case 7: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    }
}

// Streaming stores (st.global.cs: evict-first in L2) for outputs nothing in this
// launch reads back.
__device__ __forceinline__ void st_stream16(void *ptr, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_stream8(void *ptr, uint2 v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(ptr), "r"(v.x), "r"(v.y)
                 : "memory");
}

// ------------------------------------------------------------------------------------
// Row schedule shared by producer and consumers
// ------------------------------------------------------------------------------------

__device__ __forceinline__ bool row_valid(const Params &p, int64_t row) {
    if (p.num_sets == 0)
        return true;
    const int64_t g = p.in_row0 + row;
    bool v = false;
    for (int s = 0; s < p.num_sets; ++s)
        v |= (g >= p.set_lo[s]) & (g < p.set_hi[s]);
    return v;
}

// Next valid row of this CTA at or after `row` (rows are dealt round-robin).
__device__ __forceinline__ int64_t next_row(const Params &p, int64_t row) {
    while (row < p.rows && !row_valid(p, row))
        row += gridDim.x;
    return row;
}

// The valid row `n` places after `row` in this CTA's sequence.
__device__ __forceinline__ int64_t advance(const Params &p, int64_t row, int n) {
    if (p.num_sets == 0)
        return row + static_cast<int64_t>(n) * gridDim.x;
    for (int t = 0; t < n && row < p.rows; ++t)
        row = next_row(p, row + gridDim.x);
    return row;
}

// ------------------------------------------------------------------------------------
// The kernel
// ------------------------------------------------------------------------------------

struct StageMeta {
    int32_t idx[LB_MAX_TOPK];
    float w[LB_MAX_TOPK];
    uint32_t valid;
    uint32_t pad[3];
};
static_assert(sizeof(StageMeta) == LB_STREAM_META_BYTES, "stage metadata size");

// Threads per CTA the kernel is compiled for: one producer warp plus the consumer
// groups.  kVpt == 4 is the chunked-row variant: one group, one vector per chunk.
template <int kVpt>
struct StreamThreads {
    static constexpr bool chunked = kVpt >= 4;
    static constexpr int value = chunked ? LB_STREAM_THREADS_CHUNKED : LB_STREAM_THREADS_2;
};
// Warps of one consumer group at most (the wide-row shapes use up to 16).
constexpr int kMaxGroupWarps = LB_STREAM_CONSUMER_WARPS > LB_STREAM_CONSUMER_WARPS_WIDE
                                   ? LB_STREAM_CONSUMER_WARPS
                                   : LB_STREAM_CONSUMER_WARPS_WIDE;
constexpr int kGroupsMax = LB_STREAM_GROUPS;

// Group-local barrier that also ORs a predicate over the group (barrier id 1 + g).
__device__ __forceinline__ bool group_sync_or(bool pred, int id, int nthreads) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return out != 0;
}

// Shared-memory layout (dynamic): [stages][slot][slot_bytes], the mbarriers (full,
// empty), then a ring of 2 x stages StageMeta blocks: row i's metadata is in block
// i % (2 stages), fetched up to `stages` rows before row i is issued.
// Slot j < n_main holds partial j (fold) or routed row j (MoE); the residual row, if
// any, is slot n_main.  The CTA's rows are numbered i = 0, 1, ... in the order the
// producer streams them; stage i % stages holds row i, and consumer group i % groups
// processes it, so that `groups` rows are folded and reduced at the same time.
// `stages` is a multiple of `groups`: stage s then belongs to group s % groups alone
// and each stage's uses are waited for in order, which the one-bit phase parity of
// an mbarrier wait requires (a group that skipped ahead to use k of a stage whose use
// k-1 had not landed would see phase k-1's parity as complete).
// Chunked rows (kVpt == 4): a slot holds one column chunk of 32 x 8 x W elements of an
// input row, row i's chunk c is stage (i x chunks + c) % stages, and the single group
// folds the chunks in order; thread t keeps vector t of every chunk in registers
// until the row's reduction, so the thread-to-column map is the whole-row one.
template <int kMode, bool kFp8, int kVpt>
__global__ void __launch_bounds__(StreamThreads<kVpt>::value, 1)
    stream_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(16) float2 red[kGroupsMax][2][kMaxGroupWarps];
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int W = p.consumer_warps;                      // warps per consumer group
    const int G = p.groups;
    const int ns = p.stages;
    const bool has_res = p.residual_in != nullptr;
    const int n_main = (kMode == kFold) ? p.K : p.topk;
    const int n_slots = n_main + (has_res ? 1 : 0);
    constexpr bool kChunked = StreamThreads<kVpt>::chunked;
    // elements of an input row per stage, and stages per row
    const int64_t chunk = kChunked ? static_cast<int64_t>(W) * 256 : p.H;
    const int nch = kChunked ? static_cast<int>((p.H + chunk - 1) / chunk) : 1;
    const uint32_t slot_bytes = static_cast<uint32_t>(chunk * 2);
    const uint32_t stage_bytes = slot_bytes * n_slots;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(ns) * stage_bytes);
    const uint32_t full0 = smem_addr(bars);
    const uint32_t empty0 = smem_addr(bars + ns);
    const uint32_t stage0 = smem_addr(smem);
    // MoE: per row, its expert indices and routing weights (cp.async by the producer,
    // d <= ns rows ahead) and the mask of valid indices (written before the producer
    // arms the row's first "full" barrier).  Row i uses block i % (2 ns): the block of
    // row i + d last served row i + d - 2 ns, whose last stage lies at least ns stage
    // uses before row i's last one and was released before that one was issued, so
    // it is free when the fetch is issued (and when row i's mask is written).
    StageMeta *meta = reinterpret_cast<StageMeta *>(bars + 2 * ns);
    // Chunked rows: the read weight (gamma, or 1 + gamma) after the metadata ring, H
    // floats; each consumer thread writes and reads back only its own vectors' eight,
    // which keeps them out of the registers that the four folded vectors need.
    float4 *wsm = reinterpret_cast<float4 *>(meta + 2 * ns);

    if (G < 1 || ns % G != 0 || nch > (kChunked ? kVpt : 1) ||
        (kChunked && G != 1)) {                          // launch contract, see above
        if (threadIdx.x == 0)
            atomicOr(&g_device_error, kDeviceErrLaunch);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, W);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Each role reads its launch parameters before griddepcontrol.wait, so that their
    // first (cache-missing) reads overlap the previous kernel; no global memory is
    // touched before the wait.
    pdl_launch_dependents();

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        int issued = 0;
        bool ok = true;
        // Lane j's source base: partial j (fold), the residual (lane n_main), or the
        // expert rows (MoE, row chosen per token below).
        const uint16_t *lane_base = nullptr;
        int64_t lane_row0 = 0;
        if (kMode == kFold && lane < n_main) {
            lane_base = p.partials[lane];
            lane_row0 = p.in_row0;
        } else if (lane == n_main && has_res) {
            lane_base = p.residual_in;
        }
        const uint16_t *experts = p.expert_out;
        const int64_t n_experts = p.n_expert_rows;
        const int32_t *idx = p.idx;
        const int topk = p.topk;
        const int64_t H = p.H;
        const int64_t rows = p.rows;
        int64_t row = next_row(p, blockIdx.x);
        // MoE: lane j < topk fetches slot j's index and weight of a row into the row's
        // metadata block, one cp.async group per row, LB_MOE_META_AHEAD rows ahead of
        // its issue, so that no index load sits between a free stage and its copies
        // (the first rows' metadata is fetched at once).  Two rows ahead measured
        // faster than one (the load latency under a saturated memory system outlasts
        // a row) and than a full ring of stages ahead.  With the caller's promise that
        // the routing was complete before the preceding kernel began, the first rows'
        // metadata is fetched before griddepcontrol.wait.
        int64_t ahead = row;             // next row whose metadata is fetched
        auto fetch_meta = [&](int blk) {
            if (kMode != kMoe)
                return;
            if (lane < n_main && ahead < rows) {
                cp_async4(smem_addr(&meta[blk].idx[lane]), idx + ahead * topk + lane);
                cp_async4(smem_addr(&meta[blk].w[lane]), p.w + ahead * topk + lane);
            }
            cp_async_commit();
            if (ahead < rows)
                ahead = next_row(p, ahead + gridDim.x);
        };
        const int ahead_rows = ns < LB_MOE_META_AHEAD ? ns : LB_MOE_META_AHEAD;
        const bool early_meta = kMode == kMoe && p.routing_ready;
        if (early_meta)
            for (int b = 0; b < ahead_rows; ++b)
                fetch_meta(b);
        // With the caller's promise that the residual was complete before the previous
        // kernel began, the residual rows of the first (up to ns) rows are copied into
        // their stages before griddepcontrol.wait; their bytes are posted without an
        // arrival, which those rows' own arrive.expect_tx (for the other slots) adds.
        int early_rows = 0;
        if (!kChunked && p.residual_ready && has_res) {
            int64_t r = row;
            for (; early_rows < ns && r < rows; ++early_rows) {
                if (lane == 0) {
                    const uint32_t bar = full0 + 8 * early_rows;
                    mbar_expect_tx(bar, slot_bytes);
                    bulk_g2s(stage0 + static_cast<uint32_t>(early_rows) * stage_bytes +
                                 static_cast<uint32_t>(n_main) * slot_bytes,
                             p.residual_in + r * H, slot_bytes, bar);
                }
                r = next_row(p, r + gridDim.x);
            }
        }
        pdl_wait();
        if (!early_meta)
            for (int b = 0; b < ahead_rows; ++b)
                fetch_meta(b);
        // Who issues a stage's copies.  Lane 0 issuing them one after another measured
        // best for the fold's copies of 6 KB and more (rows of 3072 elements and up);
        // for shorter slots the issue itself (about 0.15 us per copy from one lane)
        // bounds the kernel, and each lane issues its own slot's copy, as it does for
        // the gathered expert rows of a MoE finalize at any size.
        const bool lane_issue = kMode == kMoe || slot_bytes <= LB_STREAM_LANE_ISSUE_BYTES;
        int s = 0;                       // stage of the next chunk to issue
        uint32_t k = 0;                  // use of that stage
        int units = 0;                   // chunks issued (one per row unless chunked)
        for (; row < rows; ++issued) {
            const int blk = issued % (2 * ns);          // this row's metadata block
            const void *src = nullptr;
            unsigned valid = 0;
            for (int c = 0; c < nch; ++c) {
                bool free_ok = true;
                if (k > 0 && lane == 0)
                    free_ok = mbar_wait_bounded(empty0 + 8 * s, (k - 1) & 1u, &abort_flag);
                if (!__shfl_sync(0xFFFFFFFFu, free_ok, 0)) {
                    ok = false;
                    break;
                }
                if (c == 0) {
                    // sources of this row: lane j handles slot j (n_slots <= 17 <= 32)
                    if (kMode == kMoe && lane < n_main) {
                        cp_async_wait_pending(ahead_rows - 1);   // this row's group landed
                        const int32_t e = meta[blk].idx[lane];
                        if (e >= 0 && static_cast<int64_t>(e) < n_experts)
                            src = experts + static_cast<int64_t>(e) * H;
                    } else if (lane_base != nullptr) {
                        src = lane_base + (lane_row0 + row) * H;
                    }
                    valid = __ballot_sync(0xFFFFFFFFu, src != nullptr);
                    if (kMode == kMoe) {
                        if (lane == 0) {
                            const unsigned main_mask =
                                (n_main >= 32) ? 0xFFFFFFFFu : ((1u << n_main) - 1u);
                            meta[blk].valid = valid & main_mask;
                            if ((valid & main_mask) != main_mask && p.bad_index != nullptr)
                                *p.bad_index = 1;
                        }
                        __syncwarp();
                    }
                }
                const uint32_t full = full0 + 8 * s;
                const int64_t c0 = static_cast<int64_t>(c) * chunk;    // first column
                const uint32_t bytes =
                    static_cast<uint32_t>((H - c0 < chunk ? H - c0 : chunk) * 2);
                // (a row whose residual went out early posts and copies the rest)
                const bool res_early = issued < early_rows;
                const unsigned posted = res_early ? valid & ~(1u << n_main) : valid;
                if (lane == 0)
                    mbar_arrive_expect_tx(full, bytes * __popc(posted));
#ifdef LB_TEST_HOOKS
                if (row == p.test_withhold_row)
                    src = nullptr;               // the posted bytes never arrive
#endif
                const uint32_t dst = stage0 + static_cast<uint32_t>(s) * stage_bytes;
                if (lane_issue) {
                    // short slots: lane j issues slot j's copy, all at once
                    __syncwarp();
                    if (src != nullptr && !(res_early && lane == n_main))
                        bulk_g2s(dst + lane * slot_bytes,
                                 reinterpret_cast<const uint16_t *>(src) + c0, bytes, full);
                } else {
                    for (int j = 0; j < n_slots; ++j) {
                        const uint16_t *sj = reinterpret_cast<const uint16_t *>(__shfl_sync(
                            0xFFFFFFFFu, reinterpret_cast<unsigned long long>(src), j));
                        if (lane == 0 && sj != nullptr && !(res_early && j == n_main))
                            bulk_g2s(dst + j * slot_bytes, sj + c0, bytes, full);
                    }
                }
                ++units;
                if (++s == ns) {
                    s = 0;
                    ++k;
                }
            }
            if (!ok)
                break;
            row = next_row(p, row + gridDim.x);
            fetch_meta((issued + ahead_rows) % (2 * ns));   // block of row i + ahead_rows
        }
        if (kMode == kMoe)
            cp_async_wait_pending(0);    // no metadata copy outlives the CTA
        if (!ok && lane == 0) {
            atomicOr(&g_device_error, kDeviceErrTimeout);
            abort_flag = 1;
        }
        // Drain: the copies of the last stages issued must land before the CTA ends.
        if (lane == 0) {
            const int first = units > ns ? units - ns : 0;
            for (int u = first; u < units; ++u)
                if (!mbar_wait_bounded(full0 + 8 * (u % ns), (u / ns) & 1u, nullptr))
                    atomicOr(&g_device_error, kDeviceErrTimeout);
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    const int g = (warp - 1) / W;                        // consumer group
    const int cw = (warp - 1) % W;                       // warp within the group
    const int ct = cw * 32 + lane;                       // thread within the group
    const int gthreads = W * 32;
    const int bar_id = 1 + g;
    const int64_t nvec = p.H >> 3;
    const bool need_read = kFp8 || p.y_out != nullptr;
    int64_t col[kVpt];
    uint32_t soff[kVpt];                                 // byte offset within a slot
    bool act[kVpt];
    float2 gm[kVpt][4];
#pragma unroll
    for (int i = 0; i < kVpt; ++i) {
        const int64_t v = ct + static_cast<int64_t>(i) * gthreads;
        act[i] = v < nvec;
        col[i] = v * 8;
        // chunked rows: vector i is vector ct of chunk i
        soff[i] = static_cast<uint32_t>((kChunked ? ct : v) * 16);
    }
    // gamma before griddepcontrol.wait only on the caller's promise that it was complete
    // before the previous kernel began
    const bool early_gamma = p.residual_ready != 0;
    if (!early_gamma)
        pdl_wait();
#pragma unroll
    for (int i = 0; i < kVpt; ++i) {
        if (act[i] && need_read) {
            float4 a = __ldg(reinterpret_cast<const float4 *>(p.gamma + col[i]));
            float4 b = __ldg(reinterpret_cast<const float4 *>(p.gamma + col[i]) + 1);
            if (p.gemma) {                         // GemmaRMSNorm: weight = 1 + gamma
                a = make_float4(1.0f + a.x, 1.0f + a.y, 1.0f + a.z, 1.0f + a.w);
                b = make_float4(1.0f + b.x, 1.0f + b.y, 1.0f + b.z, 1.0f + b.w);
            }
            if (kChunked) {
                wsm[col[i] >> 2] = a;
                wsm[(col[i] >> 2) + 1] = b;
            } else {
                gm[i][0] = make_float2(a.x, a.y);
                gm[i][1] = make_float2(a.z, a.w);
                gm[i][2] = make_float2(b.x, b.y);
                gm[i][3] = make_float2(b.z, b.w);
            }
        } else if (!kChunked) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                gm[i][e] = make_float2(0.0f, 0.0f);
        }
    }
    if (early_gamma)
        pdl_wait();
    // the weight of vector v's elements 2e, 2e + 1
    auto weight = [&](int v, int e) -> float2 {
        if (!kChunked)
            return gm[v][e];
        const float4 t = wsm[(col[v] >> 2) + (e >> 1)];
        return (e & 1) ? make_float2(t.z, t.w) : make_float2(t.x, t.y);
    };

    // This group's rows are the CTA's valid rows g, g + G, g + 2G, ...; with the
    // stage count a multiple of G, the group's stage advances by G per stage use (one
    // use per row, or per chunk of a chunked row with G = 1) and the phase parity
    // flips each time it wraps.
    int s = g;
    uint32_t phase = 0;
    int par = 0;
    int blk = g;                                         // this row's metadata block
    int64_t row = next_row(p, blockIdx.x);
    for (int t = 0; t < g && row < p.rows; ++t)
        row = next_row(p, row + gridDim.x);
    for (; row < p.rows; blk = (blk + G < 2 * ns) ? blk + G : blk + G - 2 * ns) {
        // o in binary32 pairs: acc[v][i] holds elements 2i, 2i+1 of vector v.  Mixed
        // add.rn.f32.bf16 adds, scalar mul.rn products and packed f32x2 adds all round
        // like the scalar binary32 ops, so the order of the definition -- and residual'
        // bit for bit -- is kept.
        float2 acc[kVpt][4];
#pragma unroll
        for (int v = 0; v < kVpt; ++v)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                acc[v][e] = make_float2(0.0f, 0.0f);
        // A thread whose wait fails reads nothing from the stage and writes nothing;
        // the group learns of it at its row barrier and leaves together.
        bool ok = true;
#pragma unroll
        for (int c = 0; c < (kChunked ? kVpt : 1); ++c) {
            if (c >= nch)
                break;
            if (s >= ns) {
                s -= ns;
                phase ^= 1u;
            }
            if (ok)
                ok = mbar_wait_bounded(full0 + 8 * s, phase, &abort_flag);
            if (ok) {
                const uint32_t stage = stage0 + static_cast<uint32_t>(s) * stage_bytes;
                const uint32_t valid = (kMode == kMoe) ? meta[blk].valid : 0u;
#pragma unroll
                for (int j = 0; j < LB_MAX_K; ++j) {
                    if (j >= n_main)
                        break;
                    if (kMode == kMoe && !((valid >> j) & 1u))
                        continue;
                    const float wj = (kMode == kMoe) ? meta[blk].w[j] : 1.0f;
                    const uint32_t slot = stage + static_cast<uint32_t>(j) * slot_bytes;
#pragma unroll
                    for (int v = 0; v < kVpt; ++v)
                        if ((!kChunked || v == c) && act[v]) {
                            const uint4 x = lds128(slot + soff[v]);
                            if (kMode == kMoe) {
                                float2 f[4];
                                unpack8x2(x, f);
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    acc[v][e] = add_mul2_rn(acc[v][e], wj, f[e]);
                            } else {
                                add_bf16x8(acc[v], x);
                            }
                        }
                }
                if (has_res) {
                    const uint32_t slot = stage + static_cast<uint32_t>(n_main) * slot_bytes;
#pragma unroll
                    for (int v = 0; v < kVpt; ++v)
                        if ((!kChunked || v == c) && act[v])
                            add_bf16x8(acc[v], lds128(slot + soff[v]));
                }
            }
            // the stage's data is in registers: hand it back to the producer
            __syncwarp();
            if (ok && lane == 0)
                mbar_arrive(empty0 + 8 * s);
            s += G;
            if (ok && (p.residual_out != nullptr || p.snapshot != nullptr)) {
                const int64_t roff = row * p.H;
#pragma unroll
                for (int v = 0; v < kVpt; ++v)
                    if ((!kChunked || v == c) && act[v]) {
                        const uint4 packed = pack8x2(acc[v]);
                        if (p.residual_out != nullptr)
                            st_stream16(p.residual_out + roff + col[v], packed);
                        if (p.snapshot != nullptr)
                            *reinterpret_cast<uint4 *>(p.snapshot + roff + col[v]) = packed;
                    }
            }
        }
        if (!need_read) {
            if (!ok) {
                atomicOr(&g_device_error, kDeviceErrTimeout);
                abort_flag = 1;
                return;
            }
            row = advance(p, row, G);
            continue;
        }

        const int64_t roff = row * p.H;
        // One barrier per row: sum(o^2) and, for FP8, max|o * gamma| (amax of the read
        // is r * max|o * gamma| since r > 0), plus the group's verdict on the waits.
        float2 ss2 = make_float2(0.0f, 0.0f);
        float mg = 0.0f;
#pragma unroll
        for (int v = 0; v < kVpt; ++v)
            if (act[v])
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    ss2 = __ffma2_rn(acc[v][e], acc[v][e], ss2);
                    if (kFp8) {
                        const float2 t = __fmul2_rn(acc[v][e], weight(v, e));
                        mg = fmaxf(mg, fmaxf(fabsf(t.x), fabsf(t.y)));
                    }
                }
        float ss = ss2.x + ss2.y;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
        if (kFp8)
            mg = warp_max(mg);
        if (lane == 0)
            red[g][par][cw] = make_float2(ss, mg);
        if (group_sync_or(!ok, bar_id, gthreads)) {
            if (ct == 0) {
                atomicOr(&g_device_error, kDeviceErrTimeout);
                abort_flag = 1;
            }
            return;
        }
        // the group's W (even, at most 16) slots, two per 16-byte read, summed in warp
        // order: passes of four reads, each pass's reads issued before its first add (a
        // missing pair adds +0, which leaves the sum bit for bit as it is)
        static_assert(kMaxGroupWarps <= 16, "two passes of four pairs");
        const float4 *slots = reinterpret_cast<const float4 *>(&red[g][par][0]);
        ss = 0.0f;
        mg = 0.0f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (8 * h >= W)
                break;
            float4 pair[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int w = 4 * h + i;
                pair[i] = (w < (W >> 1)) ? slots[w] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ss += pair[i].x;
                ss += pair[i].z;
                mg = fmaxf(mg, fmaxf(pair[i].y, pair[i].w));
            }
        }
        par ^= 1;
        const float r = rsqrtf(__fmaf_rn(ss, p.inv_H, p.eps));
        const float2 r2 = make_float2(r, r);

        // yf = (o * r) * gamma, for this thread's vectors of the row only (a chunked
        // row keeps no weight for the others)
#pragma unroll
        for (int v = 0; v < kVpt; ++v)
            if (act[v])
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc[v][e] = __fmul2_rn(__fmul2_rn(acc[v][e], r2), weight(v, e));

        if (p.y_out != nullptr) {
#pragma unroll
            for (int v = 0; v < kVpt; ++v)
                if (act[v])
                    *reinterpret_cast<uint4 *>(p.y_out + roff + col[v]) = pack8x2(acc[v]);
        }
        if (!kFp8) {
            row = advance(p, row, G);
            continue;
        }

        // FP8 read: scale = amax / 448, q = E4M3(yf * 448 / amax) (yf / scale for a
        // subnormal scale); an all-zero row (amax = 0) gets scale 0 and codes 0x00.
        const float amax = __fmul_rn(r, mg);
        if (ct == 0)
            p.scale_out[row] = amax / 448.0f;
        if (amax > 0.0f) {
            bool direct;
            const float inv = fp8_inverse(amax, &direct);
#pragma unroll
            for (int v = 0; v < kVpt; ++v)
                if (act[v])
                    st_stream8(p.q_out + roff + col[v], e4m3x8(acc[v], inv, amax, direct));
        } else {
#pragma unroll
            for (int v = 0; v < kVpt; ++v)
                if (act[v])
                    *reinterpret_cast<uint2 *>(p.q_out + roff + col[v]) = make_uint2(0u, 0u);
        }
        row = advance(p, row, G);
    }
}

}  // namespace lb
