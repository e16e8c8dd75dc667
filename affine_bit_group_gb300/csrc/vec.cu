// Activation producers: group sums (gsum), RMS norm with group sums (rmsq) and
// SwiGLU with group sums (swq).
//
// Source: "Metal: queued rmsq, swq, gdn and atq kernels and a 4-row q4mv ..."
// (bendlang/bend #1440), Change: Array.rmsq ("RMS norm with weights ... plus
// the 64-value group sums that Array.q4mv reads") and Array.swq(a, o, n)
// ("round(silu(a[i]) * a[n + i]), plus the group sums").
//
// Every 64-value group is one warp: lane l holds elements 2l and 2l+1, adds
// them (the tree's first level) and a 5-step butterfly finishes the group's
// pairwise tree.  rmsq needs the sum of squares of the whole vector before it
// can scale, so it runs in one thread block; gsum and swq spread groups over
// as many blocks as needed.
#include "abg_dev.cuh"
#include "abg_kernels.cuh"

#include <algorithm>

namespace abg {

namespace {

template <bool kTree>
__device__ __forceinline__ float add_(float a, float b) {
    return kTree ? __fadd_rn(a, b) : a + b;
}

template <bool kTree>
__global__ void __launch_bounds__(256) gsum_kernel(const float *__restrict__ v, float *__restrict__ s, int64_t G) {
    grid_dep_wait();
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); g < G; g += nwarps) {
        const float2 p = reinterpret_cast<const float2 *>(v)[32 * g + lane];
        float t = add_<kTree>(p.x, p.y);
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) t = add_<kTree>(t, __shfl_xor_sync(0xffffffffu, t, d));
        if (lane == 0) s[g] = t;
    }
}

template <bool kTree>
__global__ void __launch_bounds__(256) swq_kernel(const float *__restrict__ a, float *__restrict__ o,
                                                  float *__restrict__ osum, int64_t n) {
    grid_dep_wait();
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int64_t G = n / 64;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); g < G; g += nwarps) {
        const float2 gg = reinterpret_cast<const float2 *>(a)[32 * g + lane];
        const float2 uu = reinterpret_cast<const float2 *>(a + n)[32 * g + lane];
        const float o0 = swiglu<kTree>(gg.x, uu.x);
        const float o1 = swiglu<kTree>(gg.y, uu.y);
        reinterpret_cast<float2 *>(o)[32 * g + lane] = make_float2(o0, o1);
        float t = add_<kTree>(o0, o1);
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) t = add_<kTree>(t, __shfl_xor_sync(0xffffffffu, t, d));
        if (lane == 0) osum[g] = t;
    }
}

// One block; dynamic shared memory holds next_pow2(G) floats for the
// per-group sums of squares.
template <bool kTree>
__global__ void __launch_bounds__(1024) rmsq_kernel(const float *__restrict__ x, const float *__restrict__ wt,
                                                    float eps, float *__restrict__ xn, float *__restrict__ xsum,
                                                    int64_t n) {
    extern __shared__ float red[];
    __shared__ float s_r;
    grid_dep_wait();
    grid_dep_launch();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int G = static_cast<int>(n / 64);
    for (int g = warp; g < G; g += nwarps) {
        const float2 p = reinterpret_cast<const float2 *>(x)[32 * g + lane];
        float t = __fadd_rn(__fmul_rn(p.x, p.x), __fmul_rn(p.y, p.y));
        t = warp_tree<32>(t);
        if (lane == 0) red[g] = t;
    }
    __syncthreads();
    if (warp == 0) {
        const float ss = warp_tree_smem(red, G);
        if (lane == 0) {
            if (kTree) {
                const float mean = __fdiv_rn(ss, static_cast<float>(n));
                s_r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
            } else {
                s_r = rsqrtf(ss / static_cast<float>(n) + eps);
            }
        }
    }
    __syncthreads();
    const float r = s_r;
    for (int g = warp; g < G; g += nwarps) {
        const float2 p = reinterpret_cast<const float2 *>(x)[32 * g + lane];
        const float2 w = reinterpret_cast<const float2 *>(wt)[32 * g + lane];
        const float v0 = __fmul_rn(__fmul_rn(p.x, r), w.x);
        const float v1 = __fmul_rn(__fmul_rn(p.y, r), w.y);
        reinterpret_cast<float2 *>(xn)[32 * g + lane] = make_float2(v0, v1);
        float t = add_<kTree>(v0, v1);
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) t = add_<kTree>(t, __shfl_xor_sync(0xffffffffu, t, d));
        if (lane == 0) xsum[g] = t;
    }
}

cudaError_t launch(void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl, void **params) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, params);
}

unsigned groups_grid(int64_t G) {
    const int64_t blocks = (G + 7) / 8;  // 8 warps per block
    return static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(blocks, 4 * sm_count())));
}

}  // namespace

cudaError_t launch_gsum(const float *v, float *s, int64_t n, bool tree, cudaStream_t stream, bool pdl) {
    int64_t G = n / 64;
    void *params[] = {&v, &s, &G};
    void *fn = tree ? reinterpret_cast<void *>(&gsum_kernel<true>) : reinterpret_cast<void *>(&gsum_kernel<false>);
    return launch(fn, dim3(groups_grid(G)), dim3(256), 0, stream, pdl, params);
}

cudaError_t launch_swq(const float *a, float *o, float *osum, int64_t n, bool tree, cudaStream_t stream, bool pdl) {
    void *params[] = {&a, &o, &osum, &n};
    void *fn = tree ? reinterpret_cast<void *>(&swq_kernel<true>) : reinterpret_cast<void *>(&swq_kernel<false>);
    return launch(fn, dim3(groups_grid(n / 64)), dim3(256), 0, stream, pdl, params);
}

cudaError_t launch_rmsq(const float *x, const float *wt, float eps, float *xn, float *xsum, int64_t n, bool tree,
                        cudaStream_t stream, bool pdl) {
    const int G = static_cast<int>(n / 64);
    int gp = 32;
    while (gp < G) gp <<= 1;
    const size_t smem = static_cast<size_t>(gp) * sizeof(float);
    const int threads = std::min(1024, std::max(32, 32 * G));
    void *fn = tree ? reinterpret_cast<void *>(&rmsq_kernel<true>) : reinterpret_cast<void *>(&rmsq_kernel<false>);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    void *params[] = {&x, &wt, &eps, &xn, &xsum, &n};
    return launch(fn, dim3(1), dim3(threads), smem, stream, pdl, params);
}

cudaError_t vec_status(unsigned *bits, bool clear) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof v);
    if (e == cudaSuccess && clear && v) {
        const unsigned z = 0;
        e = cudaMemcpyToSymbol(g_status, &z, sizeof z);
    }
    *bits |= v;
    return e;
}

}  // namespace abg
