// Host-side launches of the two boundary kernels (templated on the kernel variant):
// launch shape, dynamic shared memory, programmatic dependent launch and, for long
// rows, the thread-block cluster.  Included by the kernel translation units.
#pragma once

#include <atomic>

#include "lb_stream.cuh"

namespace lb {

// Row kernel

template <int kMode, bool kFp8, int kVpt>
cudaError_t launch_variant(const Params &p, const Shape &s, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.rows * s.ctas_per_row), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(s.threads), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (s.ctas_per_row > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(s.ctas_per_row);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, boundary_kernel<kMode, kFp8, kVpt>, p);
}

template <int kMode>
cudaError_t launch_mode(const Params &p, const Shape &s, bool fp8, cudaStream_t stream) {
    switch (s.vpt) {
    case 1:
        return fp8 ? launch_variant<kMode, true, 1>(p, s, stream)
                   : launch_variant<kMode, false, 1>(p, s, stream);
    case 2:
        return fp8 ? launch_variant<kMode, true, 2>(p, s, stream)
                   : launch_variant<kMode, false, 2>(p, s, stream);
    case 4:
        return fp8 ? launch_variant<kMode, true, 4>(p, s, stream)
                   : launch_variant<kMode, false, 4>(p, s, stream);
    default:
        return cudaErrorInvalidConfiguration;
    }
}

// Stream kernel

template <int kMode, bool kFp8, int kVpt>
cudaError_t launch_stream_variant(const Params &p, const StreamShape &s, cudaStream_t stream) {
    auto kern = stream_kernel<kMode, kFp8, kVpt>;
    // The kernel may use up to the device's opt-in shared memory: set once per device
    // (a function attribute, kept by the context), not on every launch.
    static std::atomic<int> opted_in[64];
    const int dev = s.device;
    if (dev < 0 || dev >= 64 || !opted_in[dev].load(std::memory_order_acquire)) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess)
            return e;
        int bytes = s.smem_optin - static_cast<int>(fa.sharedSizeBytes);
        if (bytes < s.smem_bytes)
            bytes = s.smem_bytes;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            opted_in[dev].store(1, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s.grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(32 * (1 + s.groups * s.consumer_warps)), 1, 1);
    if (cfg.blockDim.x > static_cast<unsigned>(StreamThreads<kVpt>::value))
        return cudaErrorInvalidConfiguration;
    cfg.dynamicSmemBytes = static_cast<size_t>(s.smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int kMode>
cudaError_t launch_stream_mode(const Params &p, const StreamShape &s, bool fp8,
                               cudaStream_t stream) {
    switch (s.vpt) {
    case 1:
        return fp8 ? launch_stream_variant<kMode, true, 1>(p, s, stream)
                   : launch_stream_variant<kMode, false, 1>(p, s, stream);
    case 2:
        return fp8 ? launch_stream_variant<kMode, true, 2>(p, s, stream)
                   : launch_stream_variant<kMode, false, 2>(p, s, stream);
    case 4:
        return fp8 ? launch_stream_variant<kMode, true, 4>(p, s, stream)
                   : launch_stream_variant<kMode, false, 4>(p, s, stream);
    default:
        return cudaErrorInvalidConfiguration;
    }
}

}  // namespace lb
