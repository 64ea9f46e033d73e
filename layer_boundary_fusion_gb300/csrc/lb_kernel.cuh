// Row kernel for sm_103a: the boundary for calls with fewer rows than SMs (decode).
//
// One CTA per token row (a thread-block cluster of up to 8 CTAs splits only rows too
// long for one CTA, with the row's reduction combined through distributed shared
// memory).  Each thread owns whole 16-byte vectors (8 bf16) of the row and makes one
// pass over HBM:
//   1. issue the residual, gamma and every partial (or gathered expert-row) load of
//      a chunk -- all of a decode boundary's K <= 8 partials -- before consuming any;
//   2. accumulate in binary32 in a fixed order: +0, then k or j ascending, then the
//      residual -- the order of the definition, so residual' is bit-identical to it
//      (bf16 inputs are added by one mixed-precision add.rn.f32.bf16 each; MoE
//      products are rounded by scalar mul.rn before a packed f32x2 add);
//   3. store residual', and reduce sum(o^2) (and max|o*gamma| for the FP8 read) over
//      the row in one warp-shuffle + shared-memory step;
//   4. r = rsqrt(sum/H + eps); store y = bf16((o*r)*gamma), or the E4M3 codes and the
//      per-token scale with amax = r * max|o*gamma|.
// Nothing is re-read and nothing is staged in global memory.  Launches are
// programmatic dependents of the previous kernel in the stream: the launch overlaps
// its tail, and every global access waits for it (griddepcontrol.wait).
//
// Sources: "Layer boundaries" (sglang developer guide), sections "Residual stream"
// and "Residual update and input read" (fused add+norm, FP32 accumulation);
// "SGLang flashinfer_allreduce_fusion精读", section forward (AR + add + RMSNorm as
// one kernel).  The GB300 design is this library's own.
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

// The same load under a predicate: no memory access (and zeros) when `pred` is false,
// so that a run of data-dependent loads needs no branches between them.
__device__ __forceinline__ uint4 ld_once_if(const void *ptr, bool pred) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    asm("{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %5, 0;\n\t"
        "@p ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}"
        : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
        : "l"(ptr), "r"(static_cast<uint32_t>(pred)));
    return v;
}

// The residual may be overwritten in place by this same kernel, so it is read
// through the coherent path.
__device__ __forceinline__ uint4 ld_residual(const void *ptr) {
    return *reinterpret_cast<const uint4 *>(ptr);
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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);   // round to nearest even
    return *reinterpret_cast<uint32_t *>(&b);
}

// 8 bf16 (element 0 in the low half of .x) -> 4 binary32 pairs; widening is exact.
__device__ __forceinline__ void unpack8x2(const uint4 &w, float2 f[4]) {
    f[0] = make_float2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
    f[1] = make_float2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
    f[2] = make_float2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u));
    f[3] = make_float2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u));
}

// acc += the 8 bf16 values of w (element 2e in acc[e].x, 2e+1 in acc[e].y), each add
// one mixed-precision add.rn.f32.bf16: the bf16 operand widens exactly, so every add
// rounds like the binary32 add of the definition, in one instruction per element.
__device__ __forceinline__ void add_bf16x8(float2 acc[4], const uint4 &w) {
    asm("{\n\t.reg .b16 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
        "mov.b32 {l0, h0}, %8;\n\t"
        "mov.b32 {l1, h1}, %9;\n\t"
        "mov.b32 {l2, h2}, %10;\n\t"
        "mov.b32 {l3, h3}, %11;\n\t"
        "add.rn.f32.bf16 %0, l0, %0;\n\t"
        "add.rn.f32.bf16 %1, h0, %1;\n\t"
        "add.rn.f32.bf16 %2, l1, %2;\n\t"
        "add.rn.f32.bf16 %3, h1, %3;\n\t"
        "add.rn.f32.bf16 %4, l2, %4;\n\t"
        "add.rn.f32.bf16 %5, h2, %5;\n\t"
        "add.rn.f32.bf16 %6, l3, %6;\n\t"
        "add.rn.f32.bf16 %7, h3, %7;\n\t}"
        : "+f"(acc[0].x), "+f"(acc[0].y), "+f"(acc[1].x), "+f"(acc[1].y),
          "+f"(acc[2].x), "+f"(acc[2].y), "+f"(acc[3].x), "+f"(acc[3].y)
        : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w));
}

__device__ __forceinline__ uint4 pack8x2(const float2 f[4]) {
    return make_uint4(pack_bf16x2(f[0].x, f[0].y), pack_bf16x2(f[1].x, f[1].y),
                      pack_bf16x2(f[2].x, f[2].y), pack_bf16x2(f[3].x, f[3].y));
}

// acc + w * f with the product rounded to binary32 before the add, per lane (the
// MoE finalize's definition).  ptxas turns a packed f32x2 multiply feeding a packed
// add into a packed fused multiply-add even when both carry .rn, so the two
// products are formed with scalar mul.rn.f32 (never fused) and only the add is
// packed; the parity tests check residual' bit for bit against the definition.
__device__ __forceinline__ float2 add_mul2_rn(float2 acc, float w, float2 f) {
    float2 r;
    asm("{\n\t.reg .b64 a, t;\n\t.reg .f32 px, py;\n\t"
        "mul.rn.f32 px, %4, %5;\n\t"
        "mul.rn.f32 py, %4, %6;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 t, {px, py};\n\t"
        "add.rn.f32x2 t, a, t;\n\t"
        "mov.b64 {%0, %1}, t;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(acc.x), "f"(acc.y), "f"(w), "f"(f.x), "f"(f.y));
    return r;
}

// Maximum over the warp of a non-negative float (one redux instruction).
__device__ __forceinline__ float warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// E4M3 codes of 8 read values (element 2e in x[e].x, 2e+1 in x[e].y), packed low byte
// first.  Normally x * (448 / amax); when that reciprocal is not a finite positive
// binary32 (a read so small that its scale amax / 448 is subnormal) the codes come from
// x / scale, the definition's own division, out of line since ordinary data never
// takes that path.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi);

static __device__ __noinline__ uint2 e4m3x8_divided(float2 x0, float2 x1, float2 x2, float2 x3,
                                                    float amax) {
    const float scale = amax / 448.0f;
    return make_uint2(cvt_e4m3x2(__fdiv_rn(x0.x, scale), __fdiv_rn(x0.y, scale)) |
                          (cvt_e4m3x2(__fdiv_rn(x1.x, scale), __fdiv_rn(x1.y, scale)) << 16),
                      cvt_e4m3x2(__fdiv_rn(x2.x, scale), __fdiv_rn(x2.y, scale)) |
                          (cvt_e4m3x2(__fdiv_rn(x3.x, scale), __fdiv_rn(x3.y, scale)) << 16));
}

__device__ __forceinline__ uint2 e4m3x8(const float2 x[4], float inv, float amax,
                                        bool direct) {
    if (direct)
        return e4m3x8_divided(x[0], x[1], x[2], x[3], amax);
    float2 q[4];
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int e = 0; e < 4; ++e)
        q[e] = __fmul2_rn(x[e], inv2);
    return make_uint2(cvt_e4m3x2(q[0].x, q[0].y) | (cvt_e4m3x2(q[1].x, q[1].y) << 16),
                      cvt_e4m3x2(q[2].x, q[2].y) | (cvt_e4m3x2(q[3].x, q[3].y) << 16));
}

// 448 / amax, and whether it must be replaced by dividing by the scale.
__device__ __forceinline__ float fp8_inverse(float amax, bool *direct) {
    const float inv = __fdividef(448.0f, amax);
    *direct = !(inv > 0.0f && inv <= 3.40282347e38f);
    return inv;
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

// ------------------------------------------------------------------------------------
// The kernel
// ------------------------------------------------------------------------------------

// Loads in flight per vector: the residual, gamma and a chunk of up to kChunk
// partials (every partial of a decode boundary, K <= 8, in one batch).
template <int kVpt>
struct Chunk {
    static constexpr int value = (kVpt >= 4) ? 2 : (kVpt == 2 ? 4 : 8);
};

template <int kMode, bool kFp8, int kVpt>
__global__ void __launch_bounds__(512, 1) boundary_kernel(const __grid_constant__ Params p) {
    constexpr int kChunk = Chunk<kVpt>::value;
    __shared__ __align__(16) float2 red[16];       // one (sum o^2, max|o*gamma|) per warp
    __shared__ __align__(8) float2 cl_red;         // this CTA's share, for the cluster

    pdl_launch_dependents();
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
    const bool need_read = kFp8 || p.y_out != nullptr;
    // MoE with the caller's promise that the routing was complete before the preceding
    // kernel began: the first chunk's indices and weights are read before the wait
    // (not by the four-vector variant, whose registers are full).
    int32_t e_early[kChunk];
    float w_early[kChunk];
    const bool early_meta = kMode == kMoe && kVpt <= 2 && p.routing_ready;
    if (early_meta) {
#pragma unroll
        for (int jj = 0; jj < kChunk; ++jj)
            if (jj < p.topk) {
                e_early[jj] = __ldg(p.idx + row * p.topk + jj);
                w_early[jj] = __ldg(p.w + row * p.topk + jj);
            }
    }
    // Every global access after griddepcontrol.wait, but for what the caller promised
    // was complete before the previous kernel began: the routing above, and with
    // residual_ready the residual and gamma, which then load while that kernel drains.
    const bool early_res = p.residual_ready != 0;
    if (!early_res)
        pdl_wait();

    // Residual and gamma loads go out with the first chunk of partials.
    uint4 rv[kVpt];
    if (has_res) {
#pragma unroll
        for (int i = 0; i < kVpt; ++i)
            if (act[i])
                rv[i] = ld_residual(p.residual_in + row * H + col[i]);
    }
    float2 gm[kVpt][4];
#pragma unroll
    for (int i = 0; i < kVpt; ++i) {
        if (act[i] && need_read) {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(p.gamma + col[i]));
            const float4 b = __ldg(reinterpret_cast<const float4 *>(p.gamma + col[i]) + 1);
            gm[i][0] = make_float2(a.x, a.y);
            gm[i][1] = make_float2(a.z, a.w);
            gm[i][2] = make_float2(b.x, b.y);
            gm[i][3] = make_float2(b.z, b.w);
            if (p.gemma) {                         // GemmaRMSNorm: weight = 1 + gamma
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    gm[i][e] = __fadd2_rn(make_float2(1.0f, 1.0f), gm[i][e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                gm[i][e] = make_float2(0.0f, 0.0f);
        }
    }

    if (early_res)
        pdl_wait();

    // o in binary32 pairs, summed in the definition's order (mixed-precision and packed
    // adds round each element like the scalar binary32 add)
    float2 acc[kVpt][4];
#pragma unroll
    for (int i = 0; i < kVpt; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            acc[i][e] = make_float2(0.0f, 0.0f);

    if (kMode == kFold) {
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
                            if (kVpt >= 4) {       // (keeps the 4-vector variant unspilled)
                                float2 f[4];
                                unpack8x2(buf[kk][i], f);
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    acc[i][e] = __fadd2_rn(acc[i][e], f[e]);
                            } else {
                                add_bf16x8(acc[i], buf[kk][i]);
                            }
                        }
                }
        }
    } else {
        // o = +0 + w_0 * E[idx_0] + w_1 * E[idx_1] + ... (j ascending, each product
        // rounded before its add)
        const int64_t tk = row * p.topk;
        for (int j0 = 0; j0 < p.topk; j0 += kChunk) {
            // the chunk's routing first, then every expert-row load under a predicate
            // (no branch between the loads), then the products in slot order
            int32_t ev[kChunk];
            float wj[kChunk];
            bool ok[kChunk];
#pragma unroll
            for (int jj = 0; jj < kChunk; ++jj) {
                const bool in = j0 + jj < p.topk;
                const bool pre = early_meta && j0 == 0;
                ev[jj] = -1;
                wj[jj] = 0.0f;
                if (in) {
                    ev[jj] = pre ? e_early[jj] : __ldg(p.idx + tk + j0 + jj);
                    wj[jj] = pre ? w_early[jj] : __ldg(p.w + tk + j0 + jj);
                }
            }
            uint4 buf[kChunk][kVpt];
#pragma unroll
            for (int jj = 0; jj < kChunk; ++jj) {
                ok[jj] = (ev[jj] >= 0) & (static_cast<int64_t>(ev[jj]) < p.n_expert_rows);
                const uint16_t *src =
                    p.expert_out + static_cast<int64_t>(ok[jj] ? ev[jj] : 0) * H;
#pragma unroll
                for (int i = 0; i < kVpt; ++i)
                    buf[jj][i] = ld_once_if(src + col[i], ok[jj] && act[i]);
            }
            if (p.bad_index != nullptr && threadIdx.x == 0 && crank == 0) {
#pragma unroll
                for (int jj = 0; jj < kChunk; ++jj)
                    if (j0 + jj < p.topk && !ok[jj])
                        *p.bad_index = 1;
            }
#pragma unroll
            for (int jj = 0; jj < kChunk; ++jj)
                if (ok[jj]) {
#pragma unroll
                    for (int i = 0; i < kVpt; ++i)
                        if (act[i]) {
                            float2 f[4];
                            unpack8x2(buf[jj][i], f);
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                acc[i][e] = add_mul2_rn(acc[i][e], wj[jj], f[e]);
                        }
                }
        }
    }

    // Fold the residual in, store residual' = bf16(o).
    if (has_res) {
#pragma unroll
        for (int i = 0; i < kVpt; ++i)
            if (act[i])
                add_bf16x8(acc[i], rv[i]);
    }
    if (p.residual_out != nullptr || p.snapshot != nullptr) {
#pragma unroll
        for (int i = 0; i < kVpt; ++i)
            if (act[i]) {
                const uint4 packed = pack8x2(acc[i]);
                if (p.residual_out != nullptr)
                    *reinterpret_cast<uint4 *>(p.residual_out + row * H + col[i]) = packed;
                if (p.snapshot != nullptr)
                    *reinterpret_cast<uint4 *>(p.snapshot + row * H + col[i]) = packed;
            }
    }
    if (!need_read)
        return;                                    // complete_output / fold only

    // One reduction for the row: sum(o^2) and, for FP8, max|o * gamma| (the read's
    // amax is r * max|o * gamma| since r > 0).
    float2 ss2 = make_float2(0.0f, 0.0f);
    float mg = 0.0f;
#pragma unroll
    for (int i = 0; i < kVpt; ++i)
        if (act[i])
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                ss2 = __ffma2_rn(acc[i][e], acc[i][e], ss2);
                if (kFp8) {
                    const float2 t = __fmul2_rn(acc[i][e], gm[i][e]);
                    mg = fmaxf(mg, fmaxf(fabsf(t.x), fabsf(t.y)));
                }
            }
    float ss = ss2.x + ss2.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
    if (kFp8)
        mg = warp_max(mg);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = make_float2(ss, mg);
    __syncthreads();
    const int nwarps = blockDim.x >> 5;
    ss = 0.0f;
    mg = 0.0f;
    for (int w = 0; w < nwarps; ++w) {
        const float2 t = red[w];
        ss += t.x;
        mg = fmaxf(mg, t.y);
    }
    if (cs > 1) {
        // across the cluster (long rows): every CTA sums the CTAs' shares in rank order
        if (threadIdx.x == 0)
            cl_red = make_float2(ss, mg);
        cluster_arrive();
        cluster_wait();
        const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(&cl_red));
        ss = 0.0f;
        mg = 0.0f;
        for (int c = 0; c < cs; ++c) {
            uint32_t remote;
            float x, y;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(c));
            asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                         : "=f"(x), "=f"(y)
                         : "r"(remote)
                         : "memory");
            ss += x;
            mg = fmaxf(mg, y);
        }
        cluster_arrive();                          // done with the peers' shares
    }
    const float r = rsqrtf(__fmaf_rn(ss, p.inv_H, p.eps));
    const float2 r2 = make_float2(r, r);

    // yf = (o * r) * gamma
#pragma unroll
    for (int i = 0; i < kVpt; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            acc[i][e] = __fmul2_rn(__fmul2_rn(acc[i][e], r2), gm[i][e]);

    if (p.y_out != nullptr) {
#pragma unroll
        for (int i = 0; i < kVpt; ++i)
            if (act[i])
                *reinterpret_cast<uint4 *>(p.y_out + row * H + col[i]) = pack8x2(acc[i]);
    }
    if (kFp8) {
        // FP8 read: scale = amax / 448, q = E4M3(yf * 448 / amax) (yf / scale for a
        // subnormal scale); an all-zero row gets scale 0 and codes 0x00.
        const float amax = __fmul_rn(r, mg);
        if (threadIdx.x == 0 && crank == 0)
            p.scale_out[row] = amax / 448.0f;
        bool direct = false;
        const float inv = amax > 0.0f ? fp8_inverse(amax, &direct) : 0.0f;
#pragma unroll
        for (int i = 0; i < kVpt; ++i)
            if (act[i]) {
                const uint2 out =
                    amax > 0.0f ? e4m3x8(acc[i], inv, amax, direct) : make_uint2(0u, 0u);
                *reinterpret_cast<uint2 *>(p.q_out + row * H + col[i]) = out;
            }
    }
    if (cs > 1)
        cluster_wait();                            // keep our share alive for the peers
}

}  // namespace lb
