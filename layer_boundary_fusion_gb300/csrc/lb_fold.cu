// Fold-mode kernels: K partial buffers (lb_fold_norm, lb_fold_norm_fp8 and the row
// slice of a ragged batch, lb_slice_fold_norm).
#include "lb_kernel.cuh"

namespace lb {

cudaError_t launch_fold(const Params &p, const Shape &s, bool fp8, cudaStream_t stream) {
    return launch_mode<kFold>(p, s, fp8, stream);
}

}  // namespace lb
