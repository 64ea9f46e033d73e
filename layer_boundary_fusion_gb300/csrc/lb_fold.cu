// Fold-mode kernels: K partial buffers (lb_fold_norm, lb_fold_norm_fp8 and the row
// slice of a ragged batch, lb_slice_fold_norm), row and stream variants.
#include "lb_launch.cuh"

namespace lb {

cudaError_t launch_fold(const Params &p, const Shape &s, bool fp8, cudaStream_t stream) {
    return launch_mode<kFold>(p, s, fp8, stream);
}

cudaError_t launch_fold_stream(const Params &p, const StreamShape &s, bool fp8,
                               cudaStream_t stream) {
    return launch_stream_mode<kFold>(p, s, fp8, stream);
}

cudaError_t fold_device_error(unsigned int *out, bool clear) {
    return read_device_error(out, clear);
}

}  // namespace lb
