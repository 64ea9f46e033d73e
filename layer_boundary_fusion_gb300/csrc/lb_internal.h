// Internal interface between the C-ABI layer (lb_api.cu) and the kernel
// translation units.  Not installed; the public contract is include/lb.h.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "lb.h"

// Stream-kernel launch parameters (compile-time, so that the kernel's register
// budget matches the launch): persistent CTAs per SM, consumer warps per CTA, and the
// largest number of shared-memory stages per CTA.
#ifndef LB_STREAM_CTAS_PER_SM
#define LB_STREAM_CTAS_PER_SM 1
#endif
#ifndef LB_STREAM_CONSUMER_WARPS
#define LB_STREAM_CONSUMER_WARPS 8
#endif
#ifndef LB_STREAM_GROUPS
#define LB_STREAM_GROUPS 3
#endif
// Consumer warps of one group for long rows: rows of up to 2 x 32 x this many vectors
// keep two vectors per thread in one stage (hidden sizes up to 8192 at 16); rows of up
// to twice that are split into column chunks of 32 x (group warps) vectors, one chunk
// per stage, in a single group whose threads keep one vector of every chunk.
#ifndef LB_STREAM_CONSUMER_WARPS_WIDE
#define LB_STREAM_CONSUMER_WARPS_WIDE 16
#endif
// Rows of at least this many 16-byte vectors are split into chunks (at most 4).
#ifndef LB_STREAM_CHUNK_FROM
#define LB_STREAM_CHUNK_FROM (2 * 32 * LB_STREAM_CONSUMER_WARPS_WIDE + 1)
#endif
// threads per CTA the stream kernel is compiled for (launch bounds): whole-row stages
// (1 or 2 vectors per thread) and chunked rows (4 chunks per thread at most)
#define LB_STREAM_THREADS_2 (32 * (1 + LB_STREAM_GROUPS * LB_STREAM_CONSUMER_WARPS))
#define LB_STREAM_THREADS_CHUNKED (32 * (1 + LB_STREAM_CONSUMER_WARPS_WIDE))
// Stream-kernel slots of at most this many bytes (one input row, or chunk, per slot)
// are copied by one producer lane each, larger ones by lane 0 in turn.
#ifndef LB_STREAM_LANE_ISSUE_BYTES
#define LB_STREAM_LANE_ISSUE_BYTES 4096
#endif
// Rows of at most this many 16-byte vectors take the row kernel at any row count: the
// stream kernel's per-row copies cost more than such rows carry.
#ifndef LB_STREAM_MIN_ROW_VECS
#define LB_STREAM_MIN_ROW_VECS 128
#endif
#ifndef LB_STREAM_MAX_STAGES
#define LB_STREAM_MAX_STAGES 8
#endif
// MoE finalize: rows of routing metadata (indices, weights) the stream kernel's
// producer fetches ahead of the row it issues (at most the stage count).
#ifndef LB_MOE_META_AHEAD
#define LB_MOE_META_AHEAD 2
#endif
// Bytes of one row-metadata block of the stream kernel (MoE expert indices, routing
// weights, valid mask); the kernel keeps two blocks per stage.
#define LB_STREAM_META_BYTES 144
// Shared memory of one SM (GB300: 228 KB), shared by the CTAs resident on it.
#ifndef LB_SMEM_PER_SM
#define LB_SMEM_PER_SM 233472
#endif

namespace lb {

enum Mode : int { kFold = 0, kMoe = 1 };

// Everything one launch needs, passed to the kernel by value (__grid_constant__).
struct Params {
    // fold: K partial buffers; row of the partials = in_row0 + local row
    const uint16_t *partials[LB_MAX_K];
    int K;
    int64_t in_row0;
    // MoE finalize: gathered expert rows
    const uint16_t *expert_out;
    int64_t n_expert_rows;
    const int32_t *idx;
    const float *w;
    int topk;
    int32_t *bad_index;
    int routing_ready;         // idx, w may be read before griddepcontrol.wait
    int residual_ready;        // residual_in, gamma may be read before it
    // residual stream and read
    const uint16_t *residual_in;
    uint16_t *residual_out;
    const float *gamma;
    int gemma;                 // read weight = 1 + gamma
    uint16_t *snapshot;        // optional second copy of residual'
    uint16_t *y_out;
    uint8_t *q_out;
    float *scale_out;
    int64_t rows;      // local rows of this call (T, or S for a slice)
    int64_t H;
    float eps;
    // ragged placement: global row g is valid iff lo[i] <= g < hi[i] for some set;
    // num_sets == 0 makes every row valid
    int num_sets;
    int32_t set_lo[LB_MAX_SETS];
    int32_t set_hi[LB_MAX_SETS];
    // row kernel: 16-byte vectors of one row handled by one CTA
    int vec_per_cta;
    // stream kernel: shared-memory stages, consumer groups x warps, 1/H
    int stages;
    int groups;
    int consumer_warps;
    float inv_H;
#ifdef LB_TEST_HOOKS
    // test builds only: the stream kernel posts this row's bytes but issues none of its
    // copies, so that the row's consumers wait until their bounded wait runs out
    int64_t test_withhold_row;
#endif
};

// Row kernel: one CTA (or a cluster of CTAs) per row.
struct Shape {
    int threads;
    int vpt;           // vectors per thread (1, 2 or 4)
    int ctas_per_row;  // thread-block cluster size along the row (1..8)
};

// Stream kernel: persistent CTAs, one producer warp + consumer warps, TMA stages.
struct StreamShape {
    int grid;
    int groups;          // consumer groups, each folding its own rows
    int consumer_warps;  // warps per group
    int vpt;             // vectors per consumer thread (1, 2; 4 = chunked rows)
    int chunks;          // stages per row: 1, or 2..4 column chunks when vpt == 4
    int stages;          // 2..8
    int smem_bytes;      // dynamic shared memory per CTA
    int device;          // launch: the current device (-1 if unknown)
    int smem_optin;      // launch: the device's opt-in shared memory per CTA
};

// Pure host functions choosing the launch.  n_inputs = input rows read per output row.
bool choose_shape(int64_t rows, int64_t H, int num_sms, Shape *out);
bool choose_stream_shape(int64_t rows, int64_t H, int n_inputs, int num_sms,
                         int smem_per_block, StreamShape *out);
bool use_stream_kernel(int64_t rows, int num_sms);

// Kernel launchers (one pair per translation unit).  Return the CUDA launch status.
cudaError_t launch_fold(const Params &p, const Shape &s, bool fp8, cudaStream_t stream);
cudaError_t launch_moe(const Params &p, const Shape &s, bool fp8, cudaStream_t stream);
cudaError_t launch_fold_stream(const Params &p, const StreamShape &s, bool fp8,
                               cudaStream_t stream);
cudaError_t launch_moe_stream(const Params &p, const StreamShape &s, bool fp8,
                              cudaStream_t stream);
// Read (and optionally clear) the device error word of each translation unit.
cudaError_t fold_device_error(unsigned int *out, bool clear);
cudaError_t moe_device_error(unsigned int *out, bool clear);

}  // namespace lb
