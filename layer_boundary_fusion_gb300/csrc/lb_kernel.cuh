// Fused layer-boundary kernel for sm_103a.
//
// One token row per CTA, or per thread-block cluster of up to 8 CTAs when there are
// too few rows to fill the GPU (each CTA then owns a contiguous column range and the
// row's reductions are combined through distributed shared memory).  Each thread
// owns whole 16-byte vectors (8 bf16) of the row and makes exactly one pass over
// HBM:
//   1. issue the residual load and every partial (or gathered expert-row) load of a
//      chunk before consuming any, so that (chunk + 1) x 16 B are in flight per
//      vector;
//   2. accumulate in binary32 in a fixed order (+0, then k or j ascending, then the
//      residual) -- the order of the binary32 definition, so residual' is
//      bit-identical to it;
//   3. store residual' and the thread's share of sum(o^2) in the same pass;
//   4. reduce sum(o^2) over the row (warp shuffles, shared memory across warps,
//      DSMEM across the cluster), r = 1/sqrt(ss/H + eps) with IEEE sqrt and divide;
//   5. store y = bf16((o*r)*gamma) from registers, and for the FP8 read reduce
//      max|yf| the same way and store E4M3 codes and the per-token scale.
// Nothing is re-read and nothing is staged in global memory.  Launches are
// programmatic dependents of the previous kernel in the stream: the launch overlaps
// its tail, and every global access waits for it (griddepcontrol.wait).
//
// Sources: "Layer boundaries" (sglang developer guide), sections "Residual stream"
// and "Residual update and input read" (fused add+norm, FP32 accumulation);
// "SGLang flashinfer_allreduce_fusion精读", section forward (AR + add + RMSNorm as
// one kernel).  The GB300 design (register-resident rows, cluster split for small
// batches, no cross-GPU workspace) is this library's own.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lb_internal.h"

namespace lb {

// ------------------------------------------------------------------------------------
// Memory access
// ------------------------------------------------------------------------------------

// Data read exactly once (partials, expert rows): bypass L1, 256-byte L2 prefetch.
__device__ __forceinline__ uint4 ld_once(const void *ptr) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr));
    return v;
}

// The residual may be overwritten in place by this same kernel, so it is read
// through the coherent path.
__device__ __forceinline__ uint4 ld_residual(const void *ptr) {
    return *reinterpret_cast<const uint4 *>(ptr);
}

__device__ __forceinline__ void ld_gamma8(const float *g, float out[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(g));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(g) + 1);
    out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
    out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}

// ------------------------------------------------------------------------------------
// Programmatic dependent launch
// ------------------------------------------------------------------------------------

// Lets the next kernel of the stream (if launched as a programmatic dependent) be
// scheduled now, so that its launch and prologue overlap the rest of this kernel.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Waits until the kernels this one depends on have completed and their memory is
// visible.  Every global memory access of a boundary kernel comes after this call,
// so inputs produced by the previous kernel (a GEMM, the last boundary) are safe.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------------------------
// Number formats
// ------------------------------------------------------------------------------------

// 8 bf16 (element 0 in the low half of .x) -> 8 floats; widening is exact.
__device__ __forceinline__ void unpack8(const uint4 &v, float f[8]) {
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xFFFF0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xFFFF0000u);
    f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xFFFF0000u);
    f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);   // round to nearest even
    return *reinterpret_cast<uint32_t *>(&b);
}

__device__ __forceinline__ uint4 pack8(const float f[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

// Two floats -> two E4M3 codes (round to nearest even, saturate to +-448); the first
// argument lands in the low byte.  cvt puts its first source in the high half.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------------------------------------------
// Reductions
// ------------------------------------------------------------------------------------

template <bool kMax>
__device__ __forceinline__ float combine(float a, float b) {
    return kMax ? fmaxf(a, b) : a + b;
}

// Every thread of the CTA returns the same value.  `red` holds one slot per warp;
// each call site owns its own array, so no slot is reused within a launch.
template <bool kMax>
__device__ __forceinline__ float block_reduce(float v, float *red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v = combine<kMax>(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = v;
    __syncthreads();
    const int nwarps = blockDim.x >> 5;
    float r = red[0];
    for (int i = 1; i < nwarps; ++i)
        r = combine<kMax>(r, red[i]);
    return r;
}

__device__ __forceinline__ int cluster_size() {
    uint32_t n;
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return (int)n;
}

__device__ __forceinline__ int cluster_rank() {
    uint32_t r;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return (int)r;
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Combines one value per CTA across the cluster (same value in every thread of a
// CTA).  Every CTA reads the slots in rank order, so all CTAs get the same result.
template <bool kMax>
__device__ __forceinline__ float cluster_reduce(float v, float *slot, int cs) {
    if (threadIdx.x == 0)
        *slot = v;
    cluster_arrive();
    cluster_wait();
    const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(slot));
    float r = 0.0f;
    for (int c = 0; c < cs; ++c) {
        uint32_t remote;
        float x;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(c));
        asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(x) : "r"(remote) : "memory");
        r = (c == 0) ? x : combine<kMax>(r, x);
    }
    return r;
}

// ------------------------------------------------------------------------------------
// The kernel
// ------------------------------------------------------------------------------------

// Loads in flight per vector: the residual plus a chunk of kChunk partials.
template <int kVpt>
struct Chunk {
    static constexpr int value = (kVpt >= 4) ? 2 : 4;
};

// At most 512 threads per CTA; one-vector threads are held to 64 registers so that two
// 512-thread CTAs fit on an SM, wider threads get room for their extra vectors.
template <int kVpt>
struct MinBlocks {
    static constexpr int value = (kVpt == 1) ? 2 : 1;
};

template <int kMode, bool kFp8, int kVpt>
__global__ void __launch_bounds__(512, MinBlocks<kVpt>::value)
    boundary_kernel(const __grid_constant__ Params p) {
    constexpr int kChunk = Chunk<kVpt>::value;
    __shared__ float red_ss[32];
    __shared__ float red_mx[32];
    __shared__ float cl_ss;
    __shared__ float cl_mx;

    pdl_launch_dependents();
    pdl_wait();
    const int cs = cluster_size();                 // 1 without a cluster launch
    const int crank = (cs > 1) ? cluster_rank() : 0;
    const int64_t row = blockIdx.x / cs;           // all CTAs of a cluster share it
    const int64_t H = p.H;

    // Ragged placement: padding rows are neither computed nor written.  The whole
    // cluster leaves together, before any cluster barrier.
    const int64_t g = p.in_row0 + row;
    if (p.num_sets > 0) {
        bool valid = false;
        for (int s = 0; s < p.num_sets; ++s)
            valid |= (g >= p.set_lo[s]) & (g < p.set_hi[s]);
        if (!valid)
            return;
    }

    const int64_t nvec = H >> 3;
    const int64_t vbeg = static_cast<int64_t>(crank) * p.vec_per_cta;
    const int64_t vend = min(nvec, vbeg + p.vec_per_cta);
    int64_t col[kVpt];      // first element of each owned vector
    bool act[kVpt];
#pragma unroll
    for (int i = 0; i < kVpt; ++i) {
        const int64_t v = vbeg + threadIdx.x + static_cast<int64_t>(i) * blockDim.x;
        act[i] = v < vend;
        col[i] = v * 8;
    }

    const bool has_res = p.residual_in != nullptr;
    uint4 rv[kVpt];
    if (has_res) {
#pragma unroll
        for (int i = 0; i < kVpt; ++i)
            if (act[i])
                rv[i] = ld_residual(p.residual_in + row * H + col[i]);
    }

    float acc[kVpt][8];
#pragma unroll
    for (int i = 0; i < kVpt; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            acc[i][e] = 0.0f;

    if (kMode == kFold) {
        // o = +0 + p_0 + p_1 + ... (k ascending)
        const int64_t base = g * H;
        for (int k0 = 0; k0 < p.K; k0 += kChunk) {
            uint4 buf[kChunk][kVpt];
#pragma unroll
            for (int kk = 0; kk < kChunk; ++kk)
                if (k0 + kk < p.K) {
                    const uint16_t *src = p.partials[k0 + kk] + base;
#pragma unroll
                    for (int i = 0; i < kVpt; ++i)
                        if (act[i])
                            buf[kk][i] = ld_once(src + col[i]);
                }
#pragma unroll
            for (int kk = 0; kk < kChunk; ++kk)
                if (k0 + kk < p.K) {
#pragma unroll
                    for (int i = 0; i < kVpt; ++i)
                        if (act[i]) {
                            float f[8];
                            unpack8(buf[kk][i], f);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                acc[i][e] = __fadd_rn(acc[i][e], f[e]);
                        }
                }
        }
    } else {
        // o = +0 + w_0 * E[idx_0] + w_1 * E[idx_1] + ... (j ascending, no FMA)
        const int64_t tk = row * p.topk;
        for (int j0 = 0; j0 < p.topk; j0 += kChunk) {
            uint4 buf[kChunk][kVpt];
            float wj[kChunk];
            bool ok[kChunk];
#pragma unroll
            for (int jj = 0; jj < kChunk; ++jj) {
                ok[jj] = false;
                wj[jj] = 0.0f;
                if (j0 + jj < p.topk) {
                    const int32_t e = __ldg(p.idx + tk + j0 + jj);
                    wj[jj] = __ldg(p.w + tk + j0 + jj);
                    ok[jj] = (e >= 0) & (static_cast<int64_t>(e) < p.n_expert_rows);
                    if (ok[jj]) {
                        const uint16_t *src = p.expert_out + static_cast<int64_t>(e) * H;
#pragma unroll
                        for (int i = 0; i < kVpt; ++i)
                            if (act[i])
                                buf[jj][i] = ld_once(src + col[i]);
                    } else if (p.bad_index != nullptr && threadIdx.x == 0 && crank == 0) {
                        *p.bad_index = 1;
                    }
                }
            }
#pragma unroll
            for (int jj = 0; jj < kChunk; ++jj)
                if (ok[jj]) {
#pragma unroll
                    for (int i = 0; i < kVpt; ++i)
                        if (act[i]) {
                            float f[8];
                            unpack8(buf[jj][i], f);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                acc[i][e] = __fadd_rn(acc[i][e], __fmul_rn(wj[jj], f[e]));
                        }
                }
        }
    }

    // Fold the residual in, store residual' = bf16(o).
    if (has_res) {
#pragma unroll
        for (int i = 0; i < kVpt; ++i)
            if (act[i]) {
                float f[8];
                unpack8(rv[i], f);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[i][e] = __fadd_rn(acc[i][e], f[e]);
            }
    }
    if (p.residual_out != nullptr) {
#pragma unroll
        for (int i = 0; i < kVpt; ++i)
            if (act[i])
                *reinterpret_cast<uint4 *>(p.residual_out + row * H + col[i]) = pack8(acc[i]);
    }

    if (!kFp8 && p.y_out == nullptr)
        return;                                    // complete_output / fold only

    // gamma is re-read by every row: cached loads, issued before the reduction.
    float gm[kVpt][8];
#pragma unroll
    for (int i = 0; i < kVpt; ++i)
        if (act[i])
            ld_gamma8(p.gamma + col[i], gm[i]);

    // r = 1 / sqrt(mean(o^2) + eps) over the whole row
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < kVpt; ++i)
        if (act[i])
#pragma unroll
            for (int e = 0; e < 8; ++e)
                ss = __fmaf_rn(acc[i][e], acc[i][e], ss);
    ss = block_reduce<false>(ss, red_ss);
    if (cs > 1)
        ss = cluster_reduce<false>(ss, &cl_ss, cs);
    const float r = 1.0f / sqrtf(ss / static_cast<float>(H) + p.eps);

    // yf = (o * r) * gamma
#pragma unroll
    for (int i = 0; i < kVpt; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            acc[i][e] = __fmul_rn(__fmul_rn(acc[i][e], r), act[i] ? gm[i][e] : 0.0f);

    if (!kFp8) {
        if (cs > 1)
            cluster_arrive();                      // done with the peers' slots
#pragma unroll
        for (int i = 0; i < kVpt; ++i)
            if (act[i])
                *reinterpret_cast<uint4 *>(p.y_out + row * H + col[i]) = pack8(acc[i]);
        if (cs > 1)
            cluster_wait();                        // keep our slot alive for them
        return;
    }

    // FP8 read: scale = max|yf| / 448, q = E4M3(yf * 448 / max|yf|)
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < kVpt; ++i)
        if (act[i])
#pragma unroll
            for (int e = 0; e < 8; ++e)
                mx = fmaxf(mx, fabsf(acc[i][e]));
    mx = block_reduce<true>(mx, red_mx);
    if (cs > 1) {
        mx = cluster_reduce<true>(mx, &cl_mx, cs);
        cluster_arrive();
    }
    if (p.y_out != nullptr) {
#pragma unroll
        for (int i = 0; i < kVpt; ++i)
            if (act[i])
                *reinterpret_cast<uint4 *>(p.y_out + row * H + col[i]) = pack8(acc[i]);
    }
    const bool nonzero = mx > 0.0f;
    const float inv = nonzero ? 448.0f / mx : 0.0f;
    if (threadIdx.x == 0 && crank == 0)
        p.scale_out[row] = mx / 448.0f;
#pragma unroll
    for (int i = 0; i < kVpt; ++i)
        if (act[i]) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                v[e] = nonzero ? __fmul_rn(acc[i][e], inv) : 0.0f;
            const uint32_t lo = cvt_e4m3x2(v[0], v[1]) | (cvt_e4m3x2(v[2], v[3]) << 16);
            const uint32_t hi = cvt_e4m3x2(v[4], v[5]) | (cvt_e4m3x2(v[6], v[7]) << 16);
            *reinterpret_cast<uint2 *>(p.q_out + row * H + col[i]) = make_uint2(lo, hi);
        }
    if (cs > 1)
        cluster_wait();
}

// ------------------------------------------------------------------------------------
// Host-side launch
// ------------------------------------------------------------------------------------

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

}  // namespace lb
