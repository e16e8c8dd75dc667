// gdn: one token of a gated DeltaNet mixer ("Metal: queued rmsq, swq, gdn and
// atq kernels and a 4-row q4mv ...", bendlang/bend #1440, Change, the
// Array.gdn bullet: conv window and activation, q/k L2 norms, decay and beta,
// the delta-rule rows, the gated norm and group sums; one threadgroup per
// value head, every phase local to its head).
//
// One thread block per head, one thread per value column j (D threads).  The
// steps are the library's reading of the published gated DeltaNet recurrence
// (see abg_gdn in abg.h), every one a single binary32 operation rounded to
// nearest and every sum the pairwise tree in index order, so each output is
// bit-identical to the oracle's:
//   - the conv window of the thread's three channels (q, k, v) and SiLU;
//   - block sums for the L2 norms and the gated norm: a 5-step butterfly in
//     each warp, then the tree over the warps' sums;
//   - the state column S[.][j]: for D <= 128 the head's state is brought into
//     shared memory by one bulk copy at the start (overlapping the conv window,
//     the norms and the decay), otherwise read from global memory; read twice,
//     the decay recomputed on the second read, each column's sums over the
//     keys i taken in blocks of 32 keys, and the new column written to global
//     memory (coalesced over j).
#include "abg_dev.cuh"
#include "abg_kernels.cuh"

namespace abg {

namespace {

// The library's binary32 natural logarithm, from its written definition:
// NaN -> NaN; v < 0 -> NaN; v == 0 -> -inf; +inf -> +inf; a subnormal v is
// scaled by 2^23 first (e -= 23).  With v = m * 2^e, m in [1, 2), and m
// halved (e + 1) when m > RN(sqrt 2): f = m - 1 (exact), s = f / (2 + f),
// t = s*s, p = Horner(t; RN(2/9), RN(2/7), RN(2/5), RN(2/3), 2) (multiply,
// then add), and the result e*LN2HI + (s*p + e*LN2LO): log(m) = 2 atanh(s)
// by the atanh series to s^9 (|s| <= 0.1716).  LN2HI and LN2LO as in EXP.
__device__ __forceinline__ float log_tree(float v) {
    if (v != v) return v;
    if (v < 0.0f) return __int_as_float(0x7fc00000);
    if (v == 0.0f) return __int_as_float(0xff800000);
    if (v == __int_as_float(0x7f800000)) return v;
    int e = 0;
    uint32_t b = __float_as_uint(v);
    if ((b >> 23) == 0u) {  // subnormal: scale by 2^23 (exact)
        b = __float_as_uint(__fmul_rn(v, pow2i(23)));
        e = -23;
    }
    e += static_cast<int>(b >> 23) - 127;
    float m = __uint_as_float((b & 0x007FFFFFu) | 0x3F800000u);
    if (m > __int_as_float(0x3FB504F3)) {
        m = __fmul_rn(m, 0.5f);
        e += 1;
    }
    const float f = __fadd_rn(m, -1.0f);
    const float s = __fdiv_rn(f, __fadd_rn(2.0f, f));
    const float t = __fmul_rn(s, s);
    float p = 2.0f / 9.0f;
    p = __fadd_rn(__fmul_rn(p, t), 2.0f / 7.0f);
    p = __fadd_rn(__fmul_rn(p, t), 2.0f / 5.0f);
    p = __fadd_rn(__fmul_rn(p, t), 2.0f / 3.0f);
    p = __fadd_rn(__fmul_rn(p, t), 2.0f);
    const float ef = static_cast<float>(e);
    const float hi = __fmul_rn(ef, __int_as_float(0x3F317000));
    const float lo = __fmul_rn(ef, __int_as_float(0x3805FDF4));
    return __fadd_rn(hi, __fadd_rn(__fmul_rn(s, p), lo));
}

// 1 / (1 + EXP(-u)), u / (1 + EXP(-u)), and u if u > 20 else LOG(1 + EXP(u)).
__device__ __forceinline__ float sigmoid_tree(float u) {
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, exp_tree(-u)));
}
__device__ __forceinline__ float silu_tree(float u) { return __fdiv_rn(u, __fadd_rn(1.0f, exp_tree(-u))); }
__device__ __forceinline__ float softplus_tree(float u) {
    return u > 20.0f ? u : log_tree(__fadd_rn(1.0f, exp_tree(u)));
}

// The pairwise tree over v[0 .. K), an odd last element carried (K <= 8).
__device__ __forceinline__ float tree_upto8(float (&v)[8], int K) {
    int m = K;
    while (m > 1) {
        const int half = m >> 1;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (i < half) v[i] = __fadd_rn(v[2 * i], v[2 * i + 1]);
        if (m & 1) v[half] = v[m - 1];
        m = half + (m & 1);
    }
    return v[0];
}

// Sum over the block's D threads (one value each, in thread order) by the
// pairwise tree: butterfly steps within each warp, then the tree over the
// D/32 warp sums (every thread computes it from shared memory).  Every
// thread of the block calls it; `red` holds D/32 floats.
template <int D>
__device__ __forceinline__ float block_tree(float v, float *red) {
    constexpr int NW = D / 32;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, d));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float w[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = red[i];
#pragma unroll
    for (int h = NW / 2; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) w[i] = __fadd_rn(w[2 * i], w[2 * i + 1]);
    __syncthreads();  // red is reused by the next call
    return w[0];
}

// Pairwise tree over 32 values in index order.
__device__ __forceinline__ float tree32v(float (&v)[32]) {
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) v[i] = __fadd_rn(v[2 * i], v[2 * i + 1]);
    return v[0];
}

// Pairwise tree over NB <= 8 values (NB a power of two).
template <int NB>
__device__ __forceinline__ float tree_blocks(float (&v)[8]) {
#pragma unroll
    for (int h = NB / 2; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) v[i] = __fadd_rn(v[2 * i], v[2 * i + 1]);
    return v[0];
}

template <int D>
__global__ void __launch_bounds__(D) gdn_kernel(const float *__restrict__ x, const float *__restrict__ conv,
                                                float *state, const float *__restrict__ a,
                                                const float *__restrict__ b, const float *__restrict__ z,
                                                const float *__restrict__ A_log, const float *__restrict__ dt_bias,
                                                const float *__restrict__ nw, float *S, float *y, float *ysum,
                                                int H, int K, float eps, float eps_n) {
    // D <= 128: the head's state (D*D floats, at most 64 KB) is brought into
    // shared memory by one bulk copy issued at the start, which overlaps the
    // conv window, the norms and the decay; both passes over the state then
    // read shared memory.  D = 256 reads its 256 KB state from global memory.
    constexpr bool kStage = D <= 128;
    extern __shared__ __align__(128) float Ss[];
    __shared__ float qh_s[D], kh_s[D];
    __shared__ float red[D / 32];
    __shared__ uint64_t bar;
    const int h = blockIdx.x, j = threadIdx.x;
    const int64_t HD = static_cast<int64_t>(H) * D;
    float *const Sh = S + static_cast<int64_t>(h) * D * D;
    if constexpr (kStage) {
        if (j == 0) {
            mbar_init(&bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (j == 0) {
            mbar_arrive_expect_tx(&bar, D * D * 4);
            bulk_g2s(Ss, Sh, D * D * 4, &bar, l2_evict_first());
        }
    }
    // conv window and SiLU of the thread's q, k and v channels
    float act[3];
#pragma unroll
    for (int part = 0; part < 3; ++part) {
        const int64_t c = part * HD + static_cast<int64_t>(h) * D + j;
        float w[8], p[8];
        for (int t = 0; t < K - 1; ++t) w[t] = state[c * (K - 1) + t];
        w[K - 1] = x[c];
        for (int t = 0; t < K; ++t) p[t] = __fmul_rn(conv[c * K + t], w[t]);
        act[part] = silu_tree(tree_upto8(p, K));
        for (int t = 0; t < K - 1; ++t) state[c * (K - 1) + t] = w[t + 1];
    }
    const float q = act[0], k = act[1], v = act[2];
    // L2 norms; the query also scaled by RN(1 / RN(sqrt D))
    const float rq = __frcp_rn(__fsqrt_rn(__fadd_rn(block_tree<D>(__fmul_rn(q, q), red), eps)));
    const float rk = __frcp_rn(__fsqrt_rn(__fadd_rn(block_tree<D>(__fmul_rn(k, k), red), eps)));
    const float qscale = __frcp_rn(__fsqrt_rn(static_cast<float>(D)));
    qh_s[j] = __fmul_rn(__fmul_rn(q, rq), qscale);
    kh_s[j] = __fmul_rn(k, rk);
    // decay and beta
    const float alpha = exp_tree(-__fmul_rn(exp_tree(A_log[h]), softplus_tree(__fadd_rn(a[h], dt_bias[h]))));
    const float beta = sigmoid_tree(b[h]);
    __syncthreads();
    // the state, staged: a bounded wait (on a timeout the status word records
    // it and the block leaves its state and outputs untouched)
    if constexpr (kStage) {
        if (!mbar_wait(&bar, 0)) return;
    }
    const float *Src = kStage ? Ss : Sh;
    // the delta rule on column j of the head's state (S[i][j]: key i, value
    // j), its sums over the keys taken in blocks of 32 (the pairwise tree
    // over D is the tree over the blocks' trees)
    constexpr int NB = D / 32;
    float bs[8];
#pragma unroll 1
    for (int ib = 0; ib < NB; ++ib) {
        float p[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const int i = ib * 32 + t;
            p[t] = __fmul_rn(__fmul_rn(Src[i * D + j], alpha), kh_s[i]);
        }
        bs[ib] = tree32v(p);
    }
    const float d = __fmul_rn(beta, __fadd_rn(v, -tree_blocks<NB>(bs)));
#pragma unroll 1
    for (int ib = 0; ib < NB; ++ib) {
        float p[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const int i = ib * 32 + t;
            const float sv = __fadd_rn(__fmul_rn(Src[i * D + j], alpha), __fmul_rn(kh_s[i], d));
            Sh[static_cast<int64_t>(i) * D + j] = sv;
            p[t] = __fmul_rn(sv, qh_s[i]);
        }
        bs[ib] = tree32v(p);
    }
    const float o = tree_blocks<NB>(bs);
    // gated RMS norm and the output's group sums
    const float mean = __fdiv_rn(block_tree<D>(__fmul_rn(o, o), red), static_cast<float>(D));
    const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(mean, eps_n)));
    const int64_t yi = static_cast<int64_t>(h) * D + j;
    const float yv = __fmul_rn(__fmul_rn(__fmul_rn(o, r), nw[j]), silu_tree(z[yi]));
    y[yi] = yv;
    float g = yv;
#pragma unroll
    for (int dd = 1; dd < 32; dd <<= 1) g = __fadd_rn(g, __shfl_xor_sync(0xffffffffu, g, dd));
    if ((j & 31) == 0) red[j >> 5] = g;
    __syncthreads();
    if ((j & 63) == 0) ysum[yi >> 6] = __fadd_rn(red[j >> 5], red[(j >> 5) + 1]);
}

template <int D>
cudaError_t launch_gdn_d(const float *x, const float *conv, float *state, const float *a, const float *b,
                         const float *z, const float *A_log, const float *dt_bias, const float *nw, float *S,
                         float *y, float *ysum, int H, int K, float eps, float eps_n, cudaStream_t stream) {
    constexpr int kSmem = D <= 128 ? D * D * 4 : 0;
    static const cudaError_t attr =
        cudaFuncSetAttribute(gdn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (attr != cudaSuccess) return attr;
    gdn_kernel<D><<<H, D, kSmem, stream>>>(x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, H, K, eps,
                                           eps_n);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gdn(const float *x, const float *conv, float *state, const float *a, const float *b,
                       const float *z, const float *A_log, const float *dt_bias, const float *nw, float *S, float *y,
                       float *ysum, int H, int D, int K, float eps, float eps_n, cudaStream_t stream) {
    switch (D) {
    case 64: return launch_gdn_d<64>(x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, H, K, eps, eps_n, stream);
    case 128:
        return launch_gdn_d<128>(x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, H, K, eps, eps_n, stream);
    case 256:
        return launch_gdn_d<256>(x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, H, K, eps, eps_n, stream);
    default: return cudaErrorInvalidValue;
    }
}

// This unit's device status word (OR-ed into *bits).
cudaError_t mixer_status(unsigned *bits, bool clear) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof v);
    if (e == cudaSuccess && clear && v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_status, &zero, sizeof zero);
    }
    *bits |= v;
    return e;
}

}  // namespace abg
