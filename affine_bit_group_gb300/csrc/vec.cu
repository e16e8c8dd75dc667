// Activation producers: group sums (gsum), RMS norm with group sums (rmsq) and
// SwiGLU with group sums (swq).
//
// Source: "Metal: queued rmsq, swq, gdn and atq kernels and a 4-row q4mv ..."
// (bendlang/bend #1440), Change: Array.rmsq ("RMS norm with weights ... plus
// the 64-value group sums that Array.q4mv reads") and Array.swq(a, o, n)
// ("round(silu(a[i]) * a[n + i]), plus the group sums").
//
// Every group of GS values (32, 64 or 128) is one warp: lane l holds the K =
// GS/32 consecutive elements K*l .. K*l+K-1, sums them by the pairwise tree
// (the tree's first log2 K levels) and a 5-step butterfly finishes the
// group's tree.  rmsq needs the sum of squares of the whole vector before it
// can scale, so it runs in one thread block; its squares are summed per
// 64-value group whatever GS is (a tree over power-of-two blocks is the tree
// over the whole vector).  gsum and swq spread groups over as many blocks as
// needed.
#include "abg_dev.cuh"
#include "abg_kernels.cuh"

#include <algorithm>

namespace abg {

namespace {

template <bool kTree>
__device__ __forceinline__ float add_(float a, float b) {
    return kTree ? __fadd_rn(a, b) : a + b;
}

// K consecutive floats at p (p aligned to 4K bytes).
template <int K>
__device__ __forceinline__ void load_k(const float *p, float (&v)[K]) {
    if constexpr (K == 1) {
        v[0] = *p;
    } else if constexpr (K == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        v[0] = t.x, v[1] = t.y;
    } else {
        const float4 t = *reinterpret_cast<const float4 *>(p);
        v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
    }
}

template <int K>
__device__ __forceinline__ void store_k(float *p, const float (&v)[K]) {
    if constexpr (K == 1) {
        *p = v[0];
    } else if constexpr (K == 2) {
        *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
    } else {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// The group's tree sum: the lane's K values, then the butterfly over lanes.
template <int K, bool kTree>
__device__ __forceinline__ float group_tree(const float (&v)[K]) {
    float t;
    if constexpr (K == 1) {
        t = v[0];
    } else if constexpr (K == 2) {
        t = add_<kTree>(v[0], v[1]);
    } else {
        t = add_<kTree>(add_<kTree>(v[0], v[1]), add_<kTree>(v[2], v[3]));
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) t = add_<kTree>(t, __shfl_xor_sync(0xffffffffu, t, d));
    return t;
}

template <int GS, bool kTree>
__global__ void __launch_bounds__(256) gsum_kernel(const float *__restrict__ v, float *__restrict__ s, int64_t G) {
    constexpr int K = GS / 32;
    grid_dep_wait();
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); g < G; g += nwarps) {
        float p[K];
        load_k<K>(v + GS * g + K * lane, p);
        const float t = group_tree<K, kTree>(p);
        if (lane == 0) s[g] = t;
    }
}

template <int GS, bool kTree>
__global__ void __launch_bounds__(256) swq_kernel(const float *__restrict__ a, float *__restrict__ o,
                                                  float *__restrict__ osum, int64_t n) {
    constexpr int K = GS / 32;
    grid_dep_wait();
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int64_t G = n / GS;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); g < G; g += nwarps) {
        const int64_t i0 = GS * g + K * lane;
        float gg[K], uu[K], ov[K];
        load_k<K>(a + i0, gg);
        load_k<K>(a + n + i0, uu);
#pragma unroll
        for (int i = 0; i < K; ++i) ov[i] = swiglu<kTree>(gg[i], uu[i]);
        store_k<K>(o + i0, ov);
        const float t = group_tree<K, kTree>(ov);
        if (lane == 0) osum[g] = t;
    }
}

// One block; dynamic shared memory holds next_pow2(n/64) floats for the
// per-64-value sums of squares.
template <int GS, bool kTree>
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
    constexpr int K = GS / 32;
    const int GG = static_cast<int>(n / GS);
    for (int g = warp; g < GG; g += nwarps) {
        const int64_t i0 = static_cast<int64_t>(GS) * g + K * lane;
        float p[K], w[K], v[K];
        load_k<K>(x + i0, p);
        load_k<K>(wt + i0, w);
#pragma unroll
        for (int i = 0; i < K; ++i) v[i] = __fmul_rn(__fmul_rn(p[i], r), w[i]);
        store_k<K>(xn + i0, v);
        const float t = group_tree<K, kTree>(v);
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

// Instantiation for a group size (32, 64 or 128) and mode.
#define ABG_VEC_PICK(kernel, group, tree)                                                                \
    ((group) == 32    ? ((tree) ? reinterpret_cast<void *>(&kernel<32, true>) : reinterpret_cast<void *>(&kernel<32, false>))   \
     : (group) == 128 ? ((tree) ? reinterpret_cast<void *>(&kernel<128, true>) : reinterpret_cast<void *>(&kernel<128, false>)) \
                      : ((tree) ? reinterpret_cast<void *>(&kernel<64, true>) : reinterpret_cast<void *>(&kernel<64, false>)))

cudaError_t launch_gsum(const float *v, float *s, int64_t n, int group, bool tree, cudaStream_t stream, bool pdl) {
    int64_t G = n / group;
    void *params[] = {&v, &s, &G};
    void *fn = ABG_VEC_PICK(gsum_kernel, group, tree);
    return launch(fn, dim3(groups_grid(G)), dim3(256), 0, stream, pdl, params);
}

cudaError_t launch_swq(const float *a, float *o, float *osum, int64_t n, int group, bool tree, cudaStream_t stream,
                       bool pdl) {
    void *params[] = {&a, &o, &osum, &n};
    void *fn = ABG_VEC_PICK(swq_kernel, group, tree);
    return launch(fn, dim3(groups_grid(n / group)), dim3(256), 0, stream, pdl, params);
}

cudaError_t launch_rmsq(const float *x, const float *wt, float eps, float *xn, float *xsum, int64_t n, int group,
                        bool tree, cudaStream_t stream, bool pdl) {
    const int G = static_cast<int>(n / 64);
    int gp = 32;
    while (gp < G) gp <<= 1;
    const size_t smem = static_cast<size_t>(gp) * sizeof(float);
    const int threads = std::min(1024, std::max(32, 32 * G));
    void *fn = ABG_VEC_PICK(rmsq_kernel, group, tree);
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
