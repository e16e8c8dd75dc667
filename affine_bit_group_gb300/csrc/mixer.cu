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

// ------------------------------------------------------------------ atq ----
// One token of gated attention ("Metal: queued rmsq, swq, gdn and atq
// kernels ...", Change, the Array.atq bullet: q/k RMS norm and rotation, the
// new k/v into the caches, scores, softmax, weighted values, sigmoid gate and
// group sums; one threadgroup per query head, the first head of each KV group
// writing the cache row while the others use the new k/v).
//
// One block per query head, one thread per column j (D threads).  Sums over
// the positions t = 0..pos (pos + 1 of them, the pairwise tree with an odd
// element carried) are taken over blocks of 32 positions padded with -0,
// then over the blocks' sums padded with -0 to a power of two: carrying an
// element is adding -0, so this is the same tree.
constexpr int kAtqMaxPositions = 8192;

// The block's maximum of one value per thread (exact in any order).
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

template <int D>
__global__ void __launch_bounds__(D) atq_kernel(const float *__restrict__ q, const float *__restrict__ gate,
                                                const float *__restrict__ k, const float *__restrict__ v,
                                                const float *__restrict__ qn_w, const float *__restrict__ kn_w,
                                                const float *__restrict__ cs, const float *__restrict__ sn,
                                                float *Kc, float *Vc, float *y, float *ysum, int Hq, int Hkv, int P,
                                                int pos, float eps) {
    constexpr int NW = D / 32, CPL = D / 32;  // warps; columns per lane in a score
    extern __shared__ float sc[];            // scores, then probabilities (pos + 1)
    __shared__ float un[D], qr_s[D], kr_s[D], vn_s[D];
    __shared__ float red[NW];
    __shared__ float bs[2][kAtqMaxPositions / 32];
    const int h = blockIdx.x, j = threadIdx.x, warp = j >> 5, lane = j & 31;
    const int g = h / (Hq / Hkv);
    const int n = pos + 1;
    const float *Kg = Kc + static_cast<int64_t>(g) * P * D;
    const float *Vg = Vc + static_cast<int64_t>(g) * P * D;
    // normed, rotated query and key; the new value
    const float qr = rms_rotate<D>(q[static_cast<int64_t>(h) * D + j], qn_w[j], cs, sn, eps, un, red);
    const float kr = rms_rotate<D>(k[static_cast<int64_t>(g) * D + j], kn_w[j], cs, sn, eps, un, red);
    const float vn = v[static_cast<int64_t>(g) * D + j];
    qr_s[j] = qr;
    kr_s[j] = kr;
    vn_s[j] = vn;
    if (h % (Hq / Hkv) == 0) {  // the first head of the group appends the row
        Kc[(static_cast<int64_t>(g) * P + pos) * D + j] = kr;
        Vc[(static_cast<int64_t>(g) * P + pos) * D + j] = vn;
    }
    __syncthreads();
    // scores: warp w takes positions w, w + NW, ...; lane l the columns
    // l*CPL .. l*CPL + CPL-1 (their tree, then the butterfly: the tree over D)
    const float scale = __frcp_rn(__fsqrt_rn(static_cast<float>(D)));
    for (int t = warp; t < n; t += NW) {
        const float *kt = t == pos ? kr_s : Kg + static_cast<int64_t>(t) * D;
        float pr[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) pr[c] = __fmul_rn(qr_s[lane * CPL + c], kt[lane * CPL + c]);
#pragma unroll
        for (int hh = CPL / 2; hh >= 1; hh >>= 1)
#pragma unroll
            for (int c = 0; c < hh; ++c) pr[c] = __fadd_rn(pr[2 * c], pr[2 * c + 1]);
        float dot = pr[0];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) dot = __fadd_rn(dot, __shfl_xor_sync(0xffffffffu, dot, d));
        if (lane == 0) sc[t] = __fmul_rn(dot, scale);
    }
    __syncthreads();
    // softmax
    float mx = -__int_as_float(0x7f800000);
    for (int t = j; t < n; t += D) mx = fmaxf(mx, sc[t]);
    const float m = block_max<D>(mx, red);
    for (int t = j; t < n; t += D) sc[t] = exp_tree(__fsub_rn(sc[t], m));
    __syncthreads();
    const int nb = (n + 31) / 32;
    int p2 = 1;
    while (p2 < nb) p2 <<= 1;
    for (int b = j; b < p2; b += D) {
        float e[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) e[i] = (b < nb && 32 * b + i < n) ? sc[32 * b + i] : -0.0f;
        bs[0][b] = tree32v(e);
    }
    __syncthreads();
    int cur = 0;
    for (int half = p2 / 2; half >= 1; half >>= 1) {
        for (int b = j; b < half; b += D) bs[cur ^ 1][b] = __fadd_rn(bs[cur][2 * b], bs[cur][2 * b + 1]);
        cur ^= 1;
        __syncthreads();
    }
    const float Z = bs[cur][0];
    for (int t = j; t < n; t += D) sc[t] = __fdiv_rn(sc[t], Z);
    __syncthreads();
    // weighted values of column j: blocks of 32 positions, their sums combined
    // by a running pairwise tree over p2 blocks (-0 past the last)
    float lv[10];
    for (int b = 0; b < p2; ++b) {
        float blk = -0.0f;
        if (b < nb) {
            float e[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int t = 32 * b + i;
                e[i] = t < n ? __fmul_rn(sc[t], t == pos ? vn_s[j] : Vg[static_cast<int64_t>(t) * D + j]) : -0.0f;
            }
            blk = tree32v(e);
        }
        int l = 0;
        while ((b >> l) & 1) {
            blk = __fadd_rn(lv[l], blk);
            ++l;
        }
        lv[l] = blk;
    }
    int top = 0;
    while ((1 << top) < p2) ++top;
    const float o = lv[top];
    const int64_t yi = static_cast<int64_t>(h) * D + j;
    const float yv = __fmul_rn(o, sigmoid_tree(gate[yi]));
    y[yi] = yv;
    float gsm = yv;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) gsm = __fadd_rn(gsm, __shfl_xor_sync(0xffffffffu, gsm, d));
    if (lane == 0) red[warp] = gsm;
    __syncthreads();
    if ((j & 63) == 0) ysum[yi >> 6] = __fadd_rn(red[warp], red[warp + 1]);
}

template <int D>
cudaError_t launch_atq_d(const float *q, const float *gate, const float *k, const float *v, const float *qn_w,
                         const float *kn_w, const float *cs, const float *sn, float *Kc, float *Vc, float *y,
                         float *ysum, int Hq, int Hkv, int P, int pos, float eps, cudaStream_t stream) {
    atq_kernel<D><<<Hq, D, static_cast<size_t>(pos + 1) * 4, stream>>>(q, gate, k, v, qn_w, kn_w, cs, sn, Kc, Vc,
                                                                       y, ysum, Hq, Hkv, P, pos, eps);
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

cudaError_t launch_atq(const float *q, const float *gate, const float *k, const float *v, const float *qn_w,
                       const float *kn_w, const float *cs, const float *sn, float *Kc, float *Vc, float *y,
                       float *ysum, int Hq, int Hkv, int D, int P, int pos, float eps, cudaStream_t stream) {
    if (pos + 1 > kAtqMaxPositions) return cudaErrorInvalidValue;
    switch (D) {
    case 64: return launch_atq_d<64>(q, gate, k, v, qn_w, kn_w, cs, sn, Kc, Vc, y, ysum, Hq, Hkv, P, pos, eps, stream);
    case 128:
        return launch_atq_d<128>(q, gate, k, v, qn_w, kn_w, cs, sn, Kc, Vc, y, ysum, Hq, Hkv, P, pos, eps, stream);
    case 256:
        return launch_atq_d<256>(q, gate, k, v, qn_w, kn_w, cs, sn, Kc, Vc, y, ysum, Hq, Hkv, P, pos, eps, stream);
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
