// MoE-mode kernels: the deferred finalize over gathered expert rows
// (lb_moe_finalize_fold_norm), row and stream variants.
#include "lb_launch.cuh"

namespace lb {

cudaError_t launch_moe(const Params &p, const Shape &s, bool fp8, cudaStream_t stream) {
    return launch_mode<kMoe>(p, s, fp8, stream);
}

cudaError_t launch_moe_stream(const Params &p, const StreamShape &s, bool fp8,
                              cudaStream_t stream) {
    return launch_stream_mode<kMoe>(p, s, fp8, stream);
}

cudaError_t moe_device_error(unsigned int *out, bool clear) {
    return read_device_error(out, clear);
}

}  // namespace lb
