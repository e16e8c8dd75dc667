// gdn: one token of a gated DeltaNet mixer ("Metal: queued rmsq, swq, gdn and
// atq kernels and a 4-row q4mv ...", bendlang/bend #1440, Change, the
// Array.gdn bullet: conv window and activation, q/k L2 norms, decay and beta,
// the delta-rule rows, the gated norm and group sums; one threadgroup per
// value head, every phase local to its head).
//
// One thread block per head, four threads per value column j (4*D threads,
// one per quarter of the keys).  The steps are the library's reading of the
// published gated DeltaNet recurrence (see abg_gdn in abg.h), every one a
// single binary32 operation rounded to nearest and every sum the pairwise
// tree in index order, so each output is bit-identical to the oracle's:
//   - the conv window of column j's three channels (q, k, v; one quarter
//     each) and SiLU;
//   - block sums for the L2 norms and the gated norm: a 5-step butterfly in
//     each warp, then the tree over the warps' sums;
//   - the state column S[.][j]: for D <= 128 the head's state is brought into
//     shared memory by one bulk copy at the start (overlapping the conv window,
//     the norms and the decay), otherwise read from global memory; read twice,
//     the decay recomputed on the second read, each quarter of the keys summed
//     by its own thread (a subtree of the tree over the keys, in blocks of at
//     most 32 keys) and the quarters combined by the tree, and the new column
//     written to global memory (coalesced over j).
#include "abg_dev.cuh"
#include "abg_kernels.cuh"
#include "mixer.cuh"

#include <mutex>
#include <type_traits>

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

// Channel c's conv window (the K-1 stored inputs, then x[c]) into w, and
// SiLU of its K products' pairwise tree (padded with -0 to 8: the odd element
// carried); indices fixed at compile time so w stays in registers.
__device__ __forceinline__ float conv_window(const float *x, const float *conv, const float *state, int64_t c,
                                             int K, float (&w)[8]) {
    float p[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        w[t] = t < K - 1 ? state[c * (K - 1) + t] : (t == K - 1 ? x[c] : 0.0f);
        p[t] = t < K ? __fmul_rn(conv[c * K + t], w[t]) : -0.0f;
    }
#pragma unroll
    for (int hh = 4; hh >= 1; hh >>= 1)
#pragma unroll
        for (int t = 0; t < hh; ++t) p[t] = __fadd_rn(p[2 * t], p[2 * t + 1]);
    return silu_tree(p[0]);
}

// The window moves on: inputs 1 .. K-1 become the stored ones.
__device__ __forceinline__ void conv_shift(float *state, int64_t c, int K, const float (&w)[8]) {
#pragma unroll
    for (int t = 0; t < 7; ++t)
        if (t < K - 1) state[c * (K - 1) + t] = w[t + 1];
}

// A warp-sum over the first D threads of the block (one value each, thread
// order) by the pairwise tree: the butterfly in each warp, then the tree over
// the D/32 warp sums, returned to every thread of the block.  `red` holds
// D/32 floats; every thread of the block calls it.
template <int D>
__device__ __forceinline__ float first_d_tree(float v, float *red) {
    constexpr int NW = D / 32;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, d));
    if ((threadIdx.x & 31) == 0 && threadIdx.x < D) red[threadIdx.x >> 5] = v;
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

// The pairwise tree over KQ (8, 16, 32 or 64) values f(t), t < KQ: trees of
// at most 32, then their sum.
template <int KQ, typename F>
__device__ __forceinline__ float quarter_tree(F f) {
    constexpr int B = KQ < 32 ? KQ : 32;
    float bsum[KQ / B];
#pragma unroll 1
    for (int ib = 0; ib < KQ / B; ++ib) {
        float p[B];
#pragma unroll
        for (int t = 0; t < B; ++t) p[t] = f(ib * B + t);
#pragma unroll
        for (int h = B / 2; h >= 1; h >>= 1)
#pragma unroll
            for (int i = 0; i < h; ++i) p[i] = __fadd_rn(p[2 * i], p[2 * i + 1]);
        bsum[ib] = p[0];
    }
    return KQ / B == 2 ? __fadd_rn(bsum[0], bsum[1]) : bsum[0];
}

// Key groups per state column (8 for D = 128 measured slower).
template <int D>
__host__ __device__ constexpr int gdn_groups() {
    return 4;
}

// G*D threads (G = gdn_groups<D>()): thread (group r, column j) with j = tid %
// D, r = tid / D walks keys r*D/G .. (r+1)*D/G - 1 of state column j (a
// subtree of the pairwise tree over the D keys; the groups' sums are combined
// by the tree).  The conv windows of the q, k and v channels of column j run
// in groups 0, 1 and 2, the decay, beta and the output gate's SiLU in group
// 3; the norms use the first D threads.
template <int D>
__global__ void __launch_bounds__(gdn_groups<D>() * D, 1) gdn_kernel(
    const float *__restrict__ x, const float *__restrict__ conv, float *state, const float *__restrict__ a,
    const float *__restrict__ b, const float *__restrict__ z, const float *__restrict__ A_log,
    const float *__restrict__ dt_bias, const float *__restrict__ nw, float *S, float *y, float *ysum, int H, int K,
    float eps, float eps_n) {
    // D <= 128: the head's state (D*D floats, at most 64 KB) is brought into
    // shared memory by one bulk copy issued at the start, which overlaps the
    // conv window, the norms and the decay; both passes over the state then
    // read shared memory.  D = 256 reads its 256 KB state from global memory.
    constexpr bool kStage = D <= 128;
    constexpr int G = gdn_groups<D>(), KQ = D / G;
    extern __shared__ __align__(128) float Ss[];
    __shared__ float act_s[3][D], qh_s[D], kh_s[D], gate_s[D];
    __shared__ float part[G][D];
    __shared__ float red[D / 32], red2[2][D / 32];
    __shared__ float s_ab[2];
    __shared__ uint64_t bar;
    const int h = blockIdx.x, tid = threadIdx.x, j = tid % D, r = tid / D;
    const int64_t HD = static_cast<int64_t>(H) * D;
    const int64_t yi = static_cast<int64_t>(h) * D + j;
    float *const Sh = S + static_cast<int64_t>(h) * D * D;
    if constexpr (kStage) {
        if (tid == 0) {
            mbar_init(&bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
    }
    // every input may come from the launch before (programmatic dependent
    // launch: this block was scheduled while it ran)
    grid_dep_wait();
    grid_dep_launch();
    if constexpr (kStage) {
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar, D * D * 4);
            bulk_g2s(Ss, Sh, D * D * 4, &bar, l2_evict_first());
        }
    }
    if (r < 3) {
        // conv window and SiLU of channel r (q, k, v) of column j
        const int64_t c = r * HD + static_cast<int64_t>(h) * D + j;
        float w[8];
        act_s[r][j] = conv_window(x, conv, state, c, K, w);
        conv_shift(state, c, K, w);
    } else if (r == 3) {
        // decay and beta
        const float alpha = exp_tree(-__fmul_rn(exp_tree(A_log[h]), softplus_tree(__fadd_rn(a[h], dt_bias[h]))));
        const float beta = sigmoid_tree(b[h]);
        if (j == 0) {
            s_ab[0] = alpha;
            s_ab[1] = beta;
        }
        gate_s[j] = silu_tree(z[yi]);
    }
    __syncthreads();
    // L2 norms (both sums in one pass: the butterflies in each warp, then the
    // tree over the warps' sums); the query also scaled by RN(1 / RN(sqrt D))
    const float q = act_s[0][j], k = act_s[1][j], v = act_s[2][j];
    float qq = __fmul_rn(q, q), kk = __fmul_rn(k, k);
#pragma unroll
    for (int dd = 1; dd < 32; dd <<= 1) {
        qq = __fadd_rn(qq, __shfl_xor_sync(0xffffffffu, qq, dd));
        kk = __fadd_rn(kk, __shfl_xor_sync(0xffffffffu, kk, dd));
    }
    if ((tid & 31) == 0 && tid < D) {
        red2[0][tid >> 5] = qq;
        red2[1][tid >> 5] = kk;
    }
    __syncthreads();
    float wsq[D / 32], wsk[D / 32];
#pragma unroll
    for (int i = 0; i < D / 32; ++i) wsq[i] = red2[0][i], wsk[i] = red2[1][i];
#pragma unroll
    for (int hh = D / 64; hh >= 1; hh >>= 1)
#pragma unroll
        for (int i = 0; i < hh; ++i) {
            wsq[i] = __fadd_rn(wsq[2 * i], wsq[2 * i + 1]);
            wsk[i] = __fadd_rn(wsk[2 * i], wsk[2 * i + 1]);
        }
    const float rq = __frcp_rn(__fsqrt_rn(__fadd_rn(wsq[0], eps)));
    const float rk = __frcp_rn(__fsqrt_rn(__fadd_rn(wsk[0], eps)));
    if (tid < D) {
        const float qscale = __frcp_rn(__fsqrt_rn(static_cast<float>(D)));
        qh_s[j] = __fmul_rn(__fmul_rn(q, rq), qscale);
        kh_s[j] = __fmul_rn(k, rk);
    }
    const float alpha = s_ab[0], beta = s_ab[1];
    __syncthreads();
    // the state, staged: a bounded wait (on a timeout the status word records
    // it and the block leaves its state and outputs untouched)
    if constexpr (kStage) {
        if (!mbar_wait(&bar, 0)) return;
    }
    const float *Src = kStage ? Ss : Sh;
    const int i0 = r * KQ;
    auto groups_tree = [&](int jj) {
        float t[G];
#pragma unroll
        for (int g = 0; g < G; ++g) t[g] = part[g][jj];
#pragma unroll
        for (int hh = G / 2; hh >= 1; hh >>= 1)
#pragma unroll
            for (int g = 0; g < hh; ++g) t[g] = __fadd_rn(t[2 * g], t[2 * g + 1]);
        return t[0];
    };
    // the delta rule on column j (S[i][j]: key i, value j); with at most 32
    // keys a group, RN(S*alpha) stays in registers between the two passes
    constexpr bool kKeep = KQ <= 32;
    float sa[kKeep ? KQ : 1];
    part[r][j] = quarter_tree<KQ>([&](int t) {
        const float v1 = __fmul_rn(Src[(i0 + t) * D + j], alpha);
        if constexpr (kKeep) sa[t] = v1;
        return __fmul_rn(v1, kh_s[i0 + t]);
    });
    __syncthreads();
    const float d = __fmul_rn(beta, __fadd_rn(v, -groups_tree(j)));
    __syncthreads();  // part is rewritten
    part[r][j] = quarter_tree<KQ>([&](int t) {
        const int i = i0 + t;
        float v1;
        if constexpr (kKeep) {
            v1 = sa[t];
        } else {
            v1 = __fmul_rn(Src[i * D + j], alpha);
        }
        const float sv = __fadd_rn(v1, __fmul_rn(kh_s[i], d));
        Sh[static_cast<int64_t>(i) * D + j] = sv;
        return __fmul_rn(sv, qh_s[i]);
    });
    __syncthreads();
    const float o = groups_tree(j);
    // gated RMS norm and the output's group sums (the first D threads)
    const float mean =
        __fdiv_rn(first_d_tree<D>(tid < D ? __fmul_rn(o, o) : 0.0f, red), static_cast<float>(D));
    if (tid >= D) return;
    const float rn = __frcp_rn(__fsqrt_rn(__fadd_rn(mean, eps_n)));
    const float yv = __fmul_rn(__fmul_rn(__fmul_rn(o, rn), nw[j]), gate_s[j]);
    y[yi] = yv;
    float g = yv;
#pragma unroll
    for (int dd = 1; dd < 32; dd <<= 1) g = __fadd_rn(g, __shfl_xor_sync(0xffffffffu, g, dd));
    if ((j & 31) == 0) red[j >> 5] = g;
    named_bar(2, D);
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
                         float *y, float *ysum, int H, int K, float eps, float eps_n, bool pdl, cudaStream_t stream) {
    const cudaError_t attr = gdn_attr<D>();
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(H));
    cfg.blockDim = dim3(gdn_groups<D>() * D);
    cfg.dynamicSmemBytes = gdn_smem<D>();
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gdn_kernel<D>, x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, H, K,
                              eps, eps_n);
}

// ------------------------------------------------------------------ atq ----
// One token of gated attention ("Metal: queued rmsq, swq, gdn and atq
// kernels ...", Change, the Array.atq bullet: q/k RMS norm and rotation, the
// new k/v into the caches, scores, softmax, weighted values, sigmoid gate and
// group sums; the first head of each KV group writing the cache row while the
// others use the new k/v).
//
// A block takes GB query heads of one KV group (GB = 4, 2 or 1, dividing the
// group) and one chunk of 64 positions.  Four launches, the last three
// started early by programmatic dependent launch (the first too: it reads
// its cache rows below pos before waiting for the launch before it):
//   scores (one block a half chunk): the normed, rotated queries (and, in
//     the block holding pos, the key, written to the cache row with the new
//     value by the group's first block), the block's scores (each row of
//     keys read once for the GB heads) and each head's maximum over them;
//   exponentials: each head's maximum over the half chunks' maxima, the
//     chunk's exponentials (in place of the scores) and their sum;
//   values: before its wait it copies the chunk's value rows into shared
//     memory (rows below pos, which no earlier launch of the call writes; row
//     pos is the new v); then Z, the tree over the chunks' sums, the
//     probabilities e/Z and the chunk's weighted values;
//   out (one block a head): the tree over the chunks' weighted values (one
//     bulk copy of them), the sigmoid gate and the group sums.
// Every sum over positions is the pairwise tree with an odd element carried,
// which equals the tree over the positions padded with -0 to a power of two
// (carrying is adding -0); its aligned subtrees of 32 and 64 positions are
// the warps' and chunks' sums, so the pieces, combined by the tree over the
// chunks (padded with -0 to 128), give the oracle's bits.
constexpr int kAtqMaxPositions = 8192;
constexpr int kAtqL = 64;          // positions per chunk
constexpr int kAtqSL = 32;         // positions per scores block (half a chunk)
constexpr int kAtqRW = 4;          // positions per warp of a scores block
constexpr int kAtqThreads = 256;   // scores: 8 warps of 4 positions
constexpr int kAtqValThreads = 1024;
constexpr int kAtqMaxChunks = kAtqMaxPositions / kAtqL;

struct AtqArgs {
    const float *q, *gate, *k, *v, *qn_w, *kn_w, *cs, *sn;
    float *Kc, *Vc, *y, *ysum;
    float *sc;     // [Hq][C*64] scores, then their exponentials
    float *cmax;   // [Hq][2C] the half chunks' maxima
    float *csum;   // [Hq][C] the chunks' sums of exponentials
    float *opart;  // [Hq][C][D] the chunks' weighted values
    int Hq, Hkv, P, pos, C;
    float eps;
};

// Query heads per block: 4, 2 or 1, dividing the heads of a KV group.
__host__ __device__ constexpr int atq_heads_per_block(int per) { return per % 4 == 0 ? 4 : (per % 2 == 0 ? 2 : 1); }

// Sums each of a lane's N values (N a power of two, at most 32) over the
// warp's 32 lanes by the pairwise tree in lane order.  At distances 1, 2, ...
// N/2 each lane keeps half of its values and adds the partner's partial sums
// of them (a transposed butterfly); the rest is a plain butterfly.  Lane l
// ends with the sum of value rev(l mod N) (its log2 N low bits reversed).
template <int N>
__device__ __forceinline__ float warp_sums(float (&v)[N], int lane) {
#pragma unroll
    for (int d = 1; d < N; d <<= 1) {
        const int cnt = N / (2 * d);
        const bool up = (lane & d) != 0;
#pragma unroll
        for (int i = 0; i < cnt; ++i) {
            const float send = up ? v[i] : v[i + cnt];
            const float keep = up ? v[i + cnt] : v[i];
            v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, d));
        }
    }
    float x = v[0];
#pragma unroll
    for (int d = N; d < 32; d <<= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, d));
    return x;
}

template <int N>
__device__ __forceinline__ int rev_low_bits(int l) {
    int r = 0;
#pragma unroll
    for (int b = 1; b < N; b <<= 1) r = (r << 1) | ((l & b) ? 1 : 0);
    return r;
}

// CPL consecutive floats at p (CPL * 4 bytes aligned).
template <int CPL>
__device__ __forceinline__ void load_cols(const float *p, float (&o)[CPL]) {
    if constexpr (CPL % 4 == 0) {
#pragma unroll
        for (int i = 0; i < CPL / 4; ++i) {
            const float4 t = reinterpret_cast<const float4 *>(p)[i];
            o[4 * i] = t.x, o[4 * i + 1] = t.y, o[4 * i + 2] = t.z, o[4 * i + 3] = t.w;
        }
    } else {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        o[0] = t.x, o[1] = t.y;
    }
}

// The maximum over v[0 .. C) by one warp (exact in any order).
__device__ __forceinline__ float warp_max_of(const float *v, int C, int lane) {
    float mx = -__int_as_float(0x7f800000);
    for (int i = lane; i < C; i += 32) mx = fmaxf(mx, __ldcg(v + i));
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    return mx;
}

template <int D, int GB>
__global__ void __launch_bounds__(kAtqThreads) atq_scores_kernel(const __grid_constant__ AtqArgs a) {
    constexpr int CPL = D / 32, NV = kAtqRW * GB, NR = GB + 1, kStep = kAtqThreads / D;
    constexpr int kRows = (NR + kStep - 1) / kStep;  // norm rows a thread takes
    __shared__ __align__(16) float un[NR][D];
    __shared__ __align__(16) float rot[NR][D];
    __shared__ float red[NR][D / 32];
    __shared__ float ssc[GB][kAtqSL];
    const int s = blockIdx.x, c = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int per = a.Hq / a.Hkv, h0 = s * GB, g = h0 / per, n = a.pos + 1, t_lo = c * kAtqSL;
    const bool holds_pos = c == a.pos / kAtqSL;
    const int nr = GB + (holds_pos ? 1 : 0);  // the query rows, and the key in the block holding pos
    // cache rows t_lo + 4 warp + r (r < 4) below pos, read before waiting for
    // the previous launch (which must not write them); lane l holds columns
    // l*CPL .. l*CPL+CPL-1 (row pos is this block's own key)
    const float *Kg = a.Kc + static_cast<int64_t>(g) * a.P * D + lane * CPL;
    const int tw = t_lo + kAtqRW * warp;
    float kv[kAtqRW][CPL];
#pragma unroll
    for (int r = 0; r < kAtqRW; ++r) {
        if (tw + r < a.pos) {
            load_cols<CPL>(Kg + static_cast<int64_t>(tw + r) * D, kv[r]);
        } else {
#pragma unroll
            for (int cc = 0; cc < CPL; ++cc) kv[r][cc] = 0.0f;
        }
    }
    grid_dep_wait();
    grid_dep_launch();
    // the rows to norm (row r of the thread's column j: r0 + k*kStep), their
    // weights and this column's rotation
    const int j = tid % D, r0 = tid / D, ji = j % (D / 2);
    float u[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
        const int r = r0 + k * kStep;
        u[k] = r < nr ? (r < GB ? a.q[static_cast<int64_t>(h0 + r) * D + j] : a.k[static_cast<int64_t>(g) * D + j])
                      : 0.0f;
    }
    const float wq = a.qn_w[j], wk = a.kn_w[j], cj = a.cs[ji], sj = a.sn[ji];
    // RMS norms: the rows' sums of squares (a warp holds 32 consecutive
    // columns of one row: the butterfly, then the tree over the warps)
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
        const int r = r0 + k * kStep;
        if (r < nr) {
            float sq = __fmul_rn(u[k], u[k]);
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, d));
            if (lane == 0) red[r][j >> 5] = sq;
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
        const int r = r0 + k * kStep;
        if (r < nr) {
            float w[D / 32];
#pragma unroll
            for (int i = 0; i < D / 32; ++i) w[i] = red[r][i];
#pragma unroll
            for (int h = D / 64; h >= 1; h >>= 1)
#pragma unroll
                for (int i = 0; i < h; ++i) w[i] = __fadd_rn(w[2 * i], w[2 * i + 1]);
            const float mean = __fdiv_rn(w[0], static_cast<float>(D));
            const float f = __frcp_rn(__fsqrt_rn(__fadd_rn(mean, a.eps)));
            un[r][j] = __fmul_rn(__fmul_rn(u[k], f), r < GB ? wq : wk);
        }
    }
    __syncthreads();
    // the rotation of column pairs (i, i + D/2)
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
        const int r = r0 + k * kStep;
        if (r < nr)
            rot[r][j] = j < D / 2 ? __fsub_rn(__fmul_rn(un[r][j], cj), __fmul_rn(un[r][j + D / 2], sj))
                                  : __fadd_rn(__fmul_rn(un[r][j], cj), __fmul_rn(un[r][ji], sj));
    }
    __syncthreads();
    if (holds_pos && h0 % per == 0) {
        const int64_t row = (static_cast<int64_t>(g) * a.P + a.pos) * D;
        for (int jj = tid; jj < D; jj += kAtqThreads) {
            a.Kc[row + jj] = rot[GB][jj];
            a.Vc[row + jj] = a.v[static_cast<int64_t>(g) * D + jj];
        }
    }
    float qv[GB][CPL];
#pragma unroll
    for (int hh = 0; hh < GB; ++hh)
#pragma unroll
        for (int cc = 0; cc < CPL; ++cc) qv[hh][cc] = rot[hh][lane * CPL + cc];
#pragma unroll
    for (int r = 0; r < kAtqRW; ++r)
        if (tw + r == a.pos)
#pragma unroll
            for (int cc = 0; cc < CPL; ++cc) kv[r][cc] = rot[GB][lane * CPL + cc];
    // value hh*4 + r: the lane's tree over its columns of q_hh . k_r
    float vals[NV];
#pragma unroll
    for (int hh = 0; hh < GB; ++hh)
#pragma unroll
        for (int r = 0; r < kAtqRW; ++r) {
            float pr[CPL];
#pragma unroll
            for (int cc = 0; cc < CPL; ++cc) pr[cc] = __fmul_rn(qv[hh][cc], kv[r][cc]);
#pragma unroll
            for (int h = CPL / 2; h >= 1; h >>= 1)
#pragma unroll
                for (int cc = 0; cc < h; ++cc) pr[cc] = __fadd_rn(pr[2 * cc], pr[2 * cc + 1]);
            vals[hh * kAtqRW + r] = pr[0];
        }
    const float dot = warp_sums<NV>(vals, lane);
    if (lane < NV) {
        const int idx = rev_low_bits<NV>(lane), hh = idx / kAtqRW, r = idx % kAtqRW;
        const float scale = __frcp_rn(__fsqrt_rn(static_cast<float>(D)));
        ssc[hh][kAtqRW * warp + r] = __fmul_rn(dot, scale);
    }
    __syncthreads();
    if (warp < GB) {
        const int h = h0 + warp;
        float mx = -__int_as_float(0x7f800000);
        float *sh = a.sc + static_cast<int64_t>(h) * a.C * kAtqL + t_lo;
        if (t_lo + lane < n) {
            const float sv = ssc[warp][lane];
            sh[lane] = sv;
            mx = sv;
        }
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
        if (lane == 0) a.cmax[h * 2 * a.C + c] = mx;
    }
}

// Thread i < GB*64: head i / 64, position t_lo + i % 64 (a warp holds 32
// consecutive positions: its butterfly is their tree).
template <int GB>
__global__ void __launch_bounds__(kAtqThreads) atq_exp_kernel(const __grid_constant__ AtqArgs a) {
    __shared__ float s_m[GB];
    __shared__ float red[kAtqThreads / 32];
    // the values launch may start and copy its value rows meanwhile
    grid_dep_launch();
    const int s = blockIdx.x, c = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h0 = s * GB, n = a.pos + 1, t_lo = c * kAtqL;
    const int hh = tid / kAtqL, i = tid % kAtqL, t = t_lo + i;
    const bool act = hh < GB && t < n;
    float *const sp = a.sc + static_cast<int64_t>(h0 + hh) * a.C * kAtqL + t;
    grid_dep_wait();
    const float sv = act ? __ldcg(sp) : 0.0f;
    if (warp < GB) {
        const float mx = warp_max_of(a.cmax + (h0 + warp) * 2 * a.C, a.pos / kAtqSL + 1, lane);
        if (lane == 0) s_m[warp] = mx;
    }
    __syncthreads();
    float e = -0.0f;
    if (act) {
        e = exp_tree(__fsub_rn(sv, s_m[hh]));
        *sp = e;
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) e = __fadd_rn(e, __shfl_xor_sync(0xffffffffu, e, d));
    if (lane == 0) red[warp] = e;
    __syncthreads();
    if (hh < GB && i == 0) a.csum[(h0 + hh) * a.C + c] = __fadd_rn(red[warp], red[warp + 1]);
}

// 1024 threads, thread i < GB*D holding output (head i / D, column i % D);
// dynamic shared memory: the chunk's value rows [64][D].
template <int D, int GB>
__global__ void __launch_bounds__(kAtqValThreads) atq_values_kernel(const __grid_constant__ AtqArgs a) {
    extern __shared__ __align__(128) float vs[];
    __shared__ uint64_t bar;
    __shared__ float s_z[GB];
    __shared__ __align__(16) float s_p[GB][kAtqL];
    __shared__ float s_part[4][GB][D];
    const int s = blockIdx.x, c = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int per = a.Hq / a.Hkv, h0 = s * GB, g = h0 / per, n = a.pos + 1, t_lo = c * kAtqL;
    const int rows_old = max(0, min(t_lo + kAtqL, a.pos) - t_lo);  // cache rows below pos
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0 && rows_old > 0) {
        const uint32_t bytes = static_cast<uint32_t>(rows_old) * D * 4u;
        mbar_arrive_expect_tx(&bar, bytes);
        bulk_g2s(vs, a.Vc + (static_cast<int64_t>(g) * a.P + t_lo) * D, bytes, &bar, l2_evict_first());
    }
    if (a.pos < t_lo + kAtqL && tid < D) vs[(a.pos - t_lo) * D + tid] = a.v[static_cast<int64_t>(g) * D + tid];
    grid_dep_wait();
    grid_dep_launch();
    // the chunk's exponentials; Z, the tree over the chunks' sums (padded
    // with -0 to 128 chunks: lane l takes chunks 4l .. 4l+3)
    const int ph = tid / kAtqL, pi = tid % kAtqL, pt = t_lo + pi;
    const bool pact = ph < GB && pt < n;
    const float ev = pact ? __ldcg(a.sc + static_cast<int64_t>(h0 + ph) * a.C * kAtqL + pt) : 0.0f;
    if (warp < GB) {
        const float *cs = a.csum + (h0 + warp) * a.C;
        float e4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) e4[q] = 4 * lane + q < a.C ? __ldcg(cs + 4 * lane + q) : -0.0f;
        float z = __fadd_rn(__fadd_rn(e4[0], e4[1]), __fadd_rn(e4[2], e4[3]));
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) z = __fadd_rn(z, __shfl_xor_sync(0xffffffffu, z, d));
        if (lane == 0) s_z[warp] = z;
    }
    __syncthreads();
    if (ph < GB) s_p[ph][pi] = pact ? __fdiv_rn(ev, s_z[ph]) : 0.0f;
    if (rows_old > 0) mbar_wait(&bar, 0);
    __syncthreads();
    // the chunk's weighted values: quarter q = tid / 256 of the chunk (16
    // positions), thread tid % 256 column j and heads hs, hs + 256/D, ...
    // (each value row read once for them); then the tree over the quarters
    constexpr int kHS = kAtqThreads / D, kHPT = GB / kHS > 0 ? GB / kHS : 1;
    const int q = tid >> 8, hs = (tid & 255) / D, j = tid % D;
    // (positions past pos only in the chunk holding it: a separate copy of
    // the loop, so full chunks run without the per-position test)
    auto weighted = [&](auto ragged_c) {
        constexpr bool kRagged = decltype(ragged_c)::value;
        float vv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) vv[i] = vs[(16 * q + i) * D + j];
#pragma unroll
        for (int k = 0; k < kHPT; ++k) {
            const int hh = hs + k * kHS;
            if (hh >= GB) break;
            float e[16];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float4 p4 = *reinterpret_cast<const float4 *>(&s_p[hh][16 * q + 4 * m]);
                const float p[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int ti = 16 * q + 4 * m + i;
                    e[4 * m + i] = !kRagged || t_lo + ti < n ? __fmul_rn(p[i], vv[4 * m + i]) : -0.0f;
                }
            }
#pragma unroll
            for (int h = 8; h >= 1; h >>= 1)
#pragma unroll
                for (int i = 0; i < h; ++i) e[i] = __fadd_rn(e[2 * i], e[2 * i + 1]);
            s_part[q][hh][j] = e[0];
        }
    };
    if (hs < GB) {
        if (t_lo + kAtqL <= n) {
            weighted(std::false_type{});
        } else {
            weighted(std::true_type{});
        }
    }
    __syncthreads();
    if (tid < GB * D) {
        const int hh = tid / D, jj = tid % D;
        a.opart[(static_cast<int64_t>(h0 + hh) * a.C + c) * D + jj] =
            __fadd_rn(__fadd_rn(s_part[0][hh][jj], s_part[1][hh][jj]), __fadd_rn(s_part[2][hh][jj], s_part[3][hh][jj]));
    }
}

// One block a head, thread j its column; dynamic shared memory: the head's
// chunk results [C][D], brought in by one bulk copy.
template <int D>
__global__ void __launch_bounds__(D) atq_out_kernel(const __grid_constant__ AtqArgs a) {
    extern __shared__ __align__(128) float op[];
    __shared__ uint64_t bar;
    __shared__ float red[D / 32];
    const int h = blockIdx.x, j = threadIdx.x;
    const int64_t yi = static_cast<int64_t>(h) * D + j;
    if (j == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const float sg = sigmoid_tree(a.gate[yi]);
    grid_dep_wait();
    grid_dep_launch();
    if (j == 0) {
        const uint32_t bytes = static_cast<uint32_t>(a.C) * D * 4u;
        mbar_arrive_expect_tx(&bar, bytes);
        bulk_g2s(op, a.opart + static_cast<int64_t>(h) * a.C * D, bytes, &bar, l2_evict_first());
    }
    mbar_wait(&bar, 0);
    // the tree over 128 chunks padded with -0: trees of 8, then of the 16
    float b[16];
#pragma unroll
    for (int cb = 0; cb < 16; ++cb) {
        b[cb] = -0.0f;
        if (8 * cb < a.C) {
            float e[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) e[i] = 8 * cb + i < a.C ? op[(8 * cb + i) * D + j] : -0.0f;
#pragma unroll
            for (int hh = 4; hh >= 1; hh >>= 1)
#pragma unroll
                for (int i = 0; i < hh; ++i) e[i] = __fadd_rn(e[2 * i], e[2 * i + 1]);
            b[cb] = e[0];
        }
    }
#pragma unroll
    for (int hh = 8; hh >= 1; hh >>= 1)
#pragma unroll
        for (int i = 0; i < hh; ++i) b[i] = __fadd_rn(b[2 * i], b[2 * i + 1]);
    const float yv = __fmul_rn(b[0], sg);
    a.y[yi] = yv;
    float gsm = yv;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) gsm = __fadd_rn(gsm, __shfl_xor_sync(0xffffffffu, gsm, d));
    if ((j & 31) == 0) red[j >> 5] = gsm;
    __syncthreads();
    if ((j & 63) == 0) a.ysum[yi >> 6] = __fadd_rn(red[j >> 5], red[(j >> 5) + 1]);
}

template <int D, int GB>
cudaError_t atq_attr() {
    static const cudaError_t e = [] {
        cudaError_t r = cudaFuncSetAttribute(atq_values_kernel<D, GB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kAtqL * D * 4);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(atq_out_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kAtqMaxChunks * D * 4);
        return r;
    }();
    return e;
}

cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, size_t smem, const AtqArgs &a, bool pdl,
                       cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    void *params[] = {const_cast<AtqArgs *>(&a)};
    return cudaLaunchKernelExC(&cfg, fn, params);
}

template <int D, int GB>
cudaError_t launch_atq_dg(const AtqArgs &a, bool pdl, cudaStream_t stream) {
    cudaError_t e = atq_attr<D, GB>();
    if (e != cudaSuccess) return e;
    const dim3 grid(a.Hq / GB, a.C);
    if ((e = launch_pdl(reinterpret_cast<const void *>(atq_scores_kernel<D, GB>), dim3(a.Hq / GB, a.pos / kAtqSL + 1),
                        dim3(kAtqThreads), 0, a, pdl, stream)) != cudaSuccess)
        return e;
    if ((e = launch_pdl(reinterpret_cast<const void *>(atq_exp_kernel<GB>), grid, dim3(kAtqThreads), 0, a, pdl,
                        stream)) != cudaSuccess)
        return e;
    if ((e = launch_pdl(reinterpret_cast<const void *>(atq_values_kernel<D, GB>), grid, dim3(kAtqValThreads),
                        kAtqL * D * 4, a, pdl, stream)) != cudaSuccess)
        return e;
    return launch_pdl(reinterpret_cast<const void *>(atq_out_kernel<D>), dim3(a.Hq), dim3(D),
                      static_cast<size_t>(a.C) * D * 4, a, pdl, stream);
}

template <int D>
cudaError_t launch_atq_d(const AtqArgs &a, bool pdl, cudaStream_t stream) {
    switch (atq_heads_per_block(a.Hq / a.Hkv)) {
    case 4: return launch_atq_dg<D, 4>(a, pdl, stream);
    case 2: return launch_atq_dg<D, 2>(a, pdl, stream);
    default: return launch_atq_dg<D, 1>(a, pdl, stream);
    }
}

template <int D>
cudaError_t prepare_atq_d(int per) {
    switch (atq_heads_per_block(per)) {
    case 4: return atq_attr<D, 4>();
    case 2: return atq_attr<D, 2>();
    default: return atq_attr<D, 1>();
    }
}

// The scratch layout (offsets in floats, each a multiple of 4): the scores,
// the half chunks' maxima, the chunks' sums and weighted values.
struct AtqLayout {
    size_t sc, cmax, csum, opart, total;
};

AtqLayout atq_layout(int Hq, int D, int pos) {
    const size_t C = static_cast<size_t>(pos + kAtqL) / kAtqL, nc = static_cast<size_t>(Hq) * C;
    const size_t nc4 = (nc + 3) / 4 * 4;
    AtqLayout l;
    l.sc = 0;
    l.cmax = nc * kAtqL;
    l.csum = l.cmax + 2 * nc4;
    l.opart = l.csum + nc4;
    l.total = l.opart + nc * D;
    return l;
}

// Device scratch for direct calls, per device, grown when a call needs more
// (freed only at exit).
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
                       float *ysum, int H, int D, int K, float eps, float eps_n, bool pdl, cudaStream_t stream) {
    switch (D) {
    case 64:
        return launch_gdn_d<64>(x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, H, K, eps, eps_n, pdl, stream);
    case 128:
        return launch_gdn_d<128>(x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, H, K, eps, eps_n, pdl,
                                 stream);
    case 256:
        return launch_gdn_d<256>(x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, H, K, eps, eps_n, pdl,
                                 stream);
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

size_t atq_scratch_bytes(int Hq, int D, int pos) { return atq_layout(Hq, D, pos).total * sizeof(float); }

cudaError_t prepare_atq(int Hq, int Hkv, int D) {
    if (Hkv < 1 || Hq % Hkv) return cudaErrorInvalidValue;
    switch (D) {
    case 64: return prepare_atq_d<64>(Hq / Hkv);
    case 128: return prepare_atq_d<128>(Hq / Hkv);
    case 256: return prepare_atq_d<256>(Hq / Hkv);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_atq(const float *q, const float *gate, const float *k, const float *v, const float *qn_w,
                       const float *kn_w, const float *cs, const float *sn, float *Kc, float *Vc, float *y,
                       float *ysum, int Hq, int Hkv, int D, int P, int pos, float eps, float *scratch, bool pdl,
                       cudaStream_t stream) {
    if (pos < 0 || pos + 1 > kAtqMaxPositions || (D != 64 && D != 128 && D != 256) || Hkv < 1 || Hq % Hkv)
        return cudaErrorInvalidValue;
    const AtqLayout l = atq_layout(Hq, D, pos);
    float *base = scratch;
    const cudaError_t e = scratch ? cudaSuccess : atq_scratch(l.total * sizeof(float), &base);
    if (e != cudaSuccess) return e;
    const AtqArgs a{q, gate, k, v, qn_w, kn_w, cs, sn, Kc, Vc, y, ysum, base + l.sc, base + l.cmax, base + l.csum,
                    base + l.opart, Hq, Hkv, P, pos, (pos + kAtqL) / kAtqL, eps};
    switch (D) {
    case 64: return launch_atq_d<64>(a, pdl, stream);
    case 128: return launch_atq_d<128>(a, pdl, stream);
    default: return launch_atq_d<256>(a, pdl, stream);
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
