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
#include "mixer.cuh"

#include <mutex>

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
constexpr int gdn_smem() {
    return D <= 128 ? D * D * 4 : 0;
}

// the shared-memory attribute, set once (before any stream capture when a
// stage graph holds the launch)
template <int D>
cudaError_t gdn_attr() {
    static const cudaError_t attr =
        cudaFuncSetAttribute(gdn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, gdn_smem<D>());
    return attr;
}

template <int D>
cudaError_t launch_gdn_d(const float *x, const float *conv, float *state, const float *a, const float *b,
                         const float *z, const float *A_log, const float *dt_bias, const float *nw, float *S,
                         float *y, float *ysum, int H, int K, float eps, float eps_n, cudaStream_t stream) {
    constexpr int kSmem = gdn_smem<D>();
    const cudaError_t attr = gdn_attr<D>();
    if (attr != cudaSuccess) return attr;
    gdn_kernel<D><<<H, D, kSmem, stream>>>(x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, H, K, eps,
                                           eps_n);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ atq ----
// One token of gated attention ("Metal: queued rmsq, swq, gdn and atq
// kernels ...", Change, the Array.atq bullet: q/k RMS norm and rotation, the
// new k/v into the caches, scores, softmax, weighted values, sigmoid gate and
// group sums; one threadgroup per query head, the first head of each KV group
// writing the cache row while the others use the new k/v).
//
// The positions t = 0..pos are split into chunks of 256 (one block per query
// head and chunk), in four launches on the stream: scores and the
// chunk's maximum; the exponentials and the chunk's sum; the probabilities
// and the chunk's weighted values; the tree over the chunks, the gate and the
// group sums.  Every sum over positions is the pairwise tree with an odd
// element carried, which equals the tree over the positions padded with -0
// to a power of two (carrying is adding -0); the padded tree's subtrees are
// the aligned 32-position blocks and 256-position chunks, so the chunks'
// sums, combined by the tree, give the oracle's bits.
constexpr int kAtqMaxPositions = 8192;
constexpr int kAtqChunk = 256;
constexpr int kAtqMaxChunks = kAtqMaxPositions / kAtqChunk;

// The maximum over the block's D threads (exact in any order).
template <int D>
__device__ __forceinline__ float block_max(float v, float *red) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float m = red[0];
#pragma unroll
    for (int i = 1; i < D / 32; ++i) m = fmaxf(m, red[i]);
    __syncthreads();
    return m;
}

// RMS norm with weights, then the rotation of column pairs (i, i + D/2):
// thread j's rotated value.  `un` (D floats of shared memory) carries the
// normed values between the threads.
template <int D>
__device__ __forceinline__ float rms_rotate(float u, float w, const float *cs, const float *sn, float eps,
                                            float *un, float *red) {
    const int j = threadIdx.x;
    const float mean = __fdiv_rn(block_tree<D>(__fmul_rn(u, u), red), static_cast<float>(D));
    const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(mean, eps)));
    un[j] = __fmul_rn(__fmul_rn(u, r), w);
    __syncthreads();
    float out;
    if (j < D / 2) {
        out = __fsub_rn(__fmul_rn(un[j], cs[j]), __fmul_rn(un[j + D / 2], sn[j]));
    } else {
        const int i = j - D / 2;
        out = __fadd_rn(__fmul_rn(un[j], cs[i]), __fmul_rn(un[i], sn[i]));
    }
    __syncthreads();  // un is reused
    return out;
}

// The same two steps in a block wider than D: only threads j < D hold a
// column (the others pass 0 and get 0); every thread of the block calls them.
template <int D>
__device__ __forceinline__ float block_tree_first(float v, float *red) {
    constexpr int NW = D / 32;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, d));
    if ((threadIdx.x & 31) == 0 && (threadIdx.x >> 5) < NW) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float w[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = red[i];
#pragma unroll
    for (int h = NW / 2; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) w[i] = __fadd_rn(w[2 * i], w[2 * i + 1]);
    __syncthreads();
    return w[0];
}

template <int D>
__device__ __forceinline__ float rms_rotate_first(float u, float w, const float *cs, const float *sn, float eps,
                                                  float *un, float *red) {
    const int j = threadIdx.x;
    const float mean = __fdiv_rn(block_tree_first<D>(__fmul_rn(u, u), red), static_cast<float>(D));
    const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(mean, eps)));
    if (j < D) un[j] = __fmul_rn(__fmul_rn(u, r), w);
    __syncthreads();
    float out = 0.0f;
    if (j < D / 2) {
        out = __fsub_rn(__fmul_rn(un[j], cs[j]), __fmul_rn(un[j + D / 2], sn[j]));
    } else if (j < D) {
        const int i = j - D / 2;
        out = __fadd_rn(__fmul_rn(un[j], cs[i]), __fmul_rn(un[i], sn[i]));
    }
    __syncthreads();
    return out;
}

// The pairwise tree over v[0 .. m), padded with -0 to a power of two (m <= 32).
__device__ __forceinline__ float tree_padded32(const float *v, int m) {
    float e[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) e[i] = i < m ? v[i] : -0.0f;
    int p = 1;
    while (p < m) p <<= 1;
    for (int h = p / 2; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i < h) e[i] = __fadd_rn(e[2 * i], e[2 * i + 1]);
    return e[0];
}

struct AtqArgs {
    const float *q, *gate, *k, *v, *qn_w, *kn_w, *cs, *sn;
    float *Kc, *Vc, *y, *ysum;
    float *sc;    // [Hq][C*256] scores, then exponentials
    float *cmax;  // [Hq][C] the chunks' maxima
    float *csum;  // [Hq][C] the chunks' sums of exponentials
    float *opart; // [Hq][C][D] the chunks' weighted values
    int Hq, Hkv, P, pos, C;
    float eps;
};

// 1: the rotated query (and key), the cache row (written by the group's first
// head, in the chunk holding pos), the chunk's scores and their maximum.  32
// warps, 8 rows each: the chunk's 256 rows are loaded in one step.
constexpr int kAtqScoreThreads = 1024;

template <int D>
__global__ void __launch_bounds__(kAtqScoreThreads) atq_scores_kernel(const __grid_constant__ AtqArgs a) {
    constexpr int NW = kAtqScoreThreads / 32, CPL = D / 32, kRows = kAtqChunk / NW;
    __shared__ float un[D], qr_s[D], kr_s[D];
    __shared__ float red[NW];
    const int h = blockIdx.x, c = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j = tid < D ? tid : 0;
    const int g = h / (a.Hq / a.Hkv), n = a.pos + 1;
    const float qr = rms_rotate_first<D>(tid < D ? a.q[static_cast<int64_t>(h) * D + j] : 0.0f, a.qn_w[j], a.cs,
                                         a.sn, a.eps, un, red);
    const float kr = rms_rotate_first<D>(tid < D ? a.k[static_cast<int64_t>(g) * D + j] : 0.0f, a.kn_w[j], a.cs,
                                         a.sn, a.eps, un, red);
    if (tid < D) {
        qr_s[j] = qr;
        kr_s[j] = kr;
        if (h % (a.Hq / a.Hkv) == 0 && c == a.C - 1) {
            a.Kc[(static_cast<int64_t>(g) * a.P + a.pos) * D + j] = kr;
            a.Vc[(static_cast<int64_t>(g) * a.P + a.pos) * D + j] = a.v[static_cast<int64_t>(g) * D + j];
        }
    }
    __syncthreads();
    // warp w takes rows t_lo + kRows*w ..; lane l the columns l*CPL .. l*CPL +
    // CPL-1 (their tree, then the butterfly: the tree over D).  Row pos is this
    // block's own key (the cache row may be written by another block).
    const float *Kg = a.Kc + static_cast<int64_t>(g) * a.P * D;
    const float scale = __frcp_rn(__fsqrt_rn(static_cast<float>(D)));
    const int t_lo = c * kAtqChunk, t_hi = min(t_lo + kAtqChunk, n);
    float mx = -__int_as_float(0x7f800000);
    // (at most 32 loaded values a lane at a time: 64 registers a thread)
    constexpr int kPass = 32 / CPL < kRows ? 32 / CPL : kRows;
#pragma unroll
    for (int r0 = 0; r0 < kRows; r0 += kPass) {
        const int t0 = t_lo + warp * kRows + r0;
        float kv[kPass][CPL];
#pragma unroll
        for (int r = 0; r < kPass; ++r) {
            const int t = t0 + r;
            const float *kt = t == a.pos ? kr_s : Kg + static_cast<int64_t>(t < t_hi ? t : t_lo) * D;
#pragma unroll
            for (int cc = 0; cc < CPL; ++cc) kv[r][cc] = kt[lane * CPL + cc];
        }
#pragma unroll
        for (int r = 0; r < kPass; ++r) {
            float pr[CPL];
#pragma unroll
            for (int cc = 0; cc < CPL; ++cc) pr[cc] = __fmul_rn(qr_s[lane * CPL + cc], kv[r][cc]);
#pragma unroll
            for (int hh = CPL / 2; hh >= 1; hh >>= 1)
#pragma unroll
                for (int cc = 0; cc < hh; ++cc) pr[cc] = __fadd_rn(pr[2 * cc], pr[2 * cc + 1]);
            float dot = pr[0];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) dot = __fadd_rn(dot, __shfl_xor_sync(0xffffffffu, dot, d));
            const float sv = __fmul_rn(dot, scale);
            if (t0 + r < t_hi) {
                mx = fmaxf(mx, sv);
                if (lane == 0) a.sc[static_cast<int64_t>(h) * a.C * kAtqChunk + t0 + r] = sv;
            }
        }
    }
    const float m = block_max<kAtqScoreThreads>(mx, red);
    if (tid == 0) a.cmax[h * a.C + c] = m;
}

// 2: the exponentials of the chunk (against the head's maximum) and their sum.
template <int D>
__global__ void __launch_bounds__(D) atq_exp_kernel(const __grid_constant__ AtqArgs a) {
    __shared__ float es[kAtqChunk];
    __shared__ float red[D / 32];
    const int h = blockIdx.x, c = blockIdx.y, j = threadIdx.x;
    const int n = a.pos + 1, t_lo = c * kAtqChunk;
    float mx = -__int_as_float(0x7f800000);
    for (int i = j; i < a.C; i += D) mx = fmaxf(mx, a.cmax[h * a.C + i]);
    const float m = block_max<D>(mx, red);
    float *sh = a.sc + static_cast<int64_t>(h) * a.C * kAtqChunk;
    for (int i = j; i < kAtqChunk; i += D) {
        const int t = t_lo + i;
        float e = -0.0f;
        if (t < n) {
            e = exp_tree(__fsub_rn(sh[t], m));
            sh[t] = e;
        }
        es[i] = e;
    }
    __syncthreads();
    if (j < 32) {
        // lane l < 8: the tree over block l's 32 positions; then the tree over
        // the 8 blocks
        float b = j < kAtqChunk / 32 ? tree_padded32(es + 32 * j, 32) : -0.0f;
#pragma unroll
        for (int d = 1; d < kAtqChunk / 32; d <<= 1) b = __fadd_rn(b, __shfl_xor_sync(0xffffffffu, b, d));
        if (j == 0) a.csum[h * a.C + c] = b;
    }
}

// 3: the probabilities of the chunk and its weighted values.  NG thread
// groups of D threads (threads qg*D + j: column j): group qg sums the chunk's
// 32-position blocks qg*BPG .. qg*BPG + BPG-1 (an aligned subtree of the
// chunk's tree), then the NG parts are combined by the tree.
template <int D>
__host__ __device__ constexpr int atq_value_groups() { return D == 64 ? 8 : 1024 / D; }

template <int D>
__global__ void __launch_bounds__(D * atq_value_groups<D>()) atq_values_kernel(const __grid_constant__ AtqArgs a) {
    constexpr int NG = atq_value_groups<D>(), BPG = kAtqChunk / 32 / NG;
    __shared__ float ps[kAtqChunk];
    __shared__ float part[NG][D];
    const int h = blockIdx.x, c = blockIdx.y, tid = threadIdx.x, qg = tid / D, j = tid % D;
    const int g = h / (a.Hq / a.Hkv), n = a.pos + 1, t_lo = c * kAtqChunk;
    const float Z = tree_padded32(a.csum + h * a.C, a.C);
    const float *sh = a.sc + static_cast<int64_t>(h) * a.C * kAtqChunk;
    for (int i = tid; i < kAtqChunk; i += D * NG) {
        const int t = t_lo + i;
        ps[i] = t < n ? __fdiv_rn(sh[t], Z) : 0.0f;
    }
    __syncthreads();
    const float *Vg = a.Vc + static_cast<int64_t>(g) * a.P * D + j;
    float bsum[BPG];
#pragma unroll
    for (int bb = 0; bb < BPG; ++bb) {
        const int b = qg * BPG + bb;
        float e[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int t = t_lo + 32 * b + i;
            e[i] = t < n ? __fmul_rn(ps[32 * b + i], Vg[static_cast<int64_t>(t) * D]) : -0.0f;
        }
        bsum[bb] = tree32v(e);
    }
#pragma unroll
    for (int hh = BPG / 2; hh >= 1; hh >>= 1)
#pragma unroll
        for (int bb = 0; bb < hh; ++bb) bsum[bb] = __fadd_rn(bsum[2 * bb], bsum[2 * bb + 1]);
    part[qg][j] = bsum[0];
    __syncthreads();
    if (tid < D) {
        float w[NG];
#pragma unroll
        for (int i = 0; i < NG; ++i) w[i] = part[i][tid];
#pragma unroll
        for (int hh = NG / 2; hh >= 1; hh >>= 1)
#pragma unroll
            for (int i = 0; i < hh; ++i) w[i] = __fadd_rn(w[2 * i], w[2 * i + 1]);
        a.opart[(static_cast<int64_t>(h) * a.C + c) * D + tid] = w[0];
    }
}

// 4: the tree over the chunks, the gate and the group sums.
template <int D>
__global__ void __launch_bounds__(D) atq_out_kernel(const __grid_constant__ AtqArgs a) {
    __shared__ float red[D / 32];
    const int h = blockIdx.x, j = threadIdx.x;
    float o[kAtqMaxChunks];
    for (int c = 0; c < a.C; ++c) o[c] = a.opart[(static_cast<int64_t>(h) * a.C + c) * D + j];
    const float ov = tree_padded32(o, a.C);
    const int64_t yi = static_cast<int64_t>(h) * D + j;
    const float yv = __fmul_rn(ov, sigmoid_tree(a.gate[yi]));
    a.y[yi] = yv;
    float gsm = yv;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) gsm = __fadd_rn(gsm, __shfl_xor_sync(0xffffffffu, gsm, d));
    if ((j & 31) == 0) red[j >> 5] = gsm;
    __syncthreads();
    if ((j & 63) == 0) a.ysum[yi >> 6] = __fadd_rn(red[j >> 5], red[(j >> 5) + 1]);
}

template <int D>
cudaError_t launch_atq_d(const AtqArgs &a, cudaStream_t stream) {
    const dim3 grid(a.Hq, a.C);
    atq_scores_kernel<D><<<grid, kAtqScoreThreads, 0, stream>>>(a);
    atq_exp_kernel<D><<<grid, D, 0, stream>>>(a);
    atq_values_kernel<D><<<grid, D * atq_value_groups<D>(), 0, stream>>>(a);
    atq_out_kernel<D><<<a.Hq, D, 0, stream>>>(a);
    return cudaGetLastError();
}

// Device scratch for the chunk results, per device, grown when a call needs
// more (freed only at exit).
std::mutex g_atq_mu;
float *g_atq_scratch[64];
size_t g_atq_bytes[64];

cudaError_t atq_scratch(size_t bytes, float **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_atq_mu);
    if (g_atq_bytes[dev] < bytes) {
        if (g_atq_scratch[dev]) {
            e = cudaDeviceSynchronize();  // a launch may still use the old buffer
            if (e == cudaSuccess) e = cudaFree(g_atq_scratch[dev]);
            if (e != cudaSuccess) return e;
            g_atq_scratch[dev] = nullptr;
            g_atq_bytes[dev] = 0;
        }
        void *p = nullptr;
        e = cudaMalloc(&p, bytes);
        if (e != cudaSuccess) return e;
        g_atq_scratch[dev] = static_cast<float *>(p);
        g_atq_bytes[dev] = bytes;
    }
    *out = g_atq_scratch[dev];
    return cudaSuccess;
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

cudaError_t prepare_gdn(int D) {
    switch (D) {
    case 64: return gdn_attr<64>();
    case 128: return gdn_attr<128>();
    case 256: return gdn_attr<256>();
    default: return cudaErrorInvalidValue;
    }
}

size_t atq_scratch_bytes(int Hq, int D, int pos) {
    const size_t nc = static_cast<size_t>(Hq) * ((pos + kAtqChunk) / kAtqChunk);
    return (nc * kAtqChunk + 2 * nc + nc * D) * sizeof(float);
}

cudaError_t launch_atq(const float *q, const float *gate, const float *k, const float *v, const float *qn_w,
                       const float *kn_w, const float *cs, const float *sn, float *Kc, float *Vc, float *y,
                       float *ysum, int Hq, int Hkv, int D, int P, int pos, float eps, float *scratch,
                       cudaStream_t stream) {
    if (pos + 1 > kAtqMaxPositions || (D != 64 && D != 128 && D != 256)) return cudaErrorInvalidValue;
    AtqArgs a{q, gate, k, v, qn_w, kn_w, cs, sn, Kc, Vc, y, ysum, nullptr, nullptr, nullptr, nullptr,
              Hq, Hkv, P, pos, (pos + kAtqChunk) / kAtqChunk, eps};
    const size_t nsc = static_cast<size_t>(Hq) * a.C * kAtqChunk, nc = static_cast<size_t>(Hq) * a.C;
    float *base = scratch;
    cudaError_t e = scratch ? cudaSuccess : atq_scratch(atq_scratch_bytes(Hq, D, pos), &base);
    if (e != cudaSuccess) return e;
    a.sc = base;
    a.cmax = base + nsc;
    a.csum = a.cmax + nc;
    a.opart = a.csum + nc;
    switch (D) {
    case 64: return launch_atq_d<64>(a, stream);
    case 128: return launch_atq_d<128>(a, stream);
    default: return launch_atq_d<256>(a, stream);
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
