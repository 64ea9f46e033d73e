// MoE-mode kernels: the deferred finalize over gathered expert rows
// (lb_moe_finalize_fold_norm).
#include "lb_kernel.cuh"

namespace lb {

cudaError_t launch_moe(const Params &p, const Shape &s, bool fp8, cudaStream_t stream) {
    return launch_mode<kMoe>(p, s, fp8, stream);
}

}  // namespace lb
