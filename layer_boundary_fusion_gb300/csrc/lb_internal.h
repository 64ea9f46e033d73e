// Internal interface between the C-ABI layer (lb_api.cu) and the kernel
// translation units.  Not installed; the public contract is include/lb.h.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "lb.h"

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
    // residual stream and read
    const uint16_t *residual_in;
    uint16_t *residual_out;
    const float *gamma;
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
    // launch shape: 16-byte vectors of one row handled by one CTA
    int vec_per_cta;
};

struct Shape {
    int threads;
    int vpt;           // vectors per thread (1, 2 or 4)
    int ctas_per_row;  // thread-block cluster size along the row (1..8)
};

// Pure host function: the launch shape for `rows` rows of width H.
bool choose_shape(int64_t rows, int64_t H, int num_sms, Shape *out);

// Kernel launchers (one per translation unit).  Return the CUDA launch status.
cudaError_t launch_fold(const Params &p, const Shape &s, bool fp8, cudaStream_t stream);
cudaError_t launch_moe(const Params &p, const Shape &s, bool fp8, cudaStream_t stream);

}  // namespace lb
