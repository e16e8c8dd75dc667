// q4mm kernel: the affine 4-bit product for a batch of T decode tokens that
// share the weights, Y[t] = W x[t] for t < T, each token's result bit-identical
// to its own single-token product (q4mv).  Groups of 64 columns, f32 scale and
// bias.
//
// Source: the product of "Array.q4mv on Metal: one kernel thread per row ..."
// (bendlang/bend #1435) and "Metal: queued rmsq, swq, gdn and atq kernels and
// a 4-row q4mv ..." (#1440, Change: the 4-row q4mv reads each group's
// activations once for all of its rows); here the weights are read once for all
// of a batch's tokens.
//
// Layout.  The tile machinery is the single-token kernel's (a producer warp
// streams row tiles into a ring of shared-memory stages with bulk copies;
// computing warps own column chunks and take row blocks of each tile; chunk
// partials meet in shared memory and are summed per row by the tree).  What
// changes is the lane mapping: a lane covers LC = 32/T columns (16 for a pair
// of tokens), so the slices of all T activations still fit in 32
// registers, and a warp's chunk is 32*LC columns.  Each nibble is unpacked once
// (one logic op) and used for all T tokens (one packed FMA per two products per
// token).  A 64-column group spans 64/LC lanes; the transposed butterflies now
// reduce R*T values per lane (row-major over (row, token)), and the affine
// term of a (row, token) value reads the row's scale and bias and the token's
// group sum.  The sums pair the same leaves as the single-token tree, so every
// token's output equals its q4mv output bit for bit.
#pragma once

#include "q4mv_kernel.cuh"

namespace abg {

namespace {

// Columns per lane for T token slots (the pair kernel uses T = 2: 16).
template <int T>
__host__ __device__ constexpr int mm_lane_cols() {
    return 32 / T;
}

// The float -(1 + q * 2^(4k-23)) for nibble J of a word (see neg_u2).
template <int J>
__device__ __forceinline__ float neg_u1(uint32_t w, uint32_t wh) {
    constexpr uint32_t kMask = 0xFu << (4 * nib_k(J));
    return __uint_as_float(and_or<kMask>(J <= 4 ? w : wh, 0xBF800000u));
}

// Word and nibble of lane column c (LC columns = LC/8 words).
template <int C>
__device__ __forceinline__ float neg_u_col(const uint32_t (&w)[2], const uint32_t (&h)[2]) {
    return neg_u1<C % 8>(w[C / 8], h[C / 8]);
}

// Pairwise tree over N packed pairs (N a power of two), returning the pair of
// the two half sums.
template <int N>
__device__ __forceinline__ float2 tree_pairs(float2 (&P)[N]) {
#pragma unroll
    for (int h = N / 2; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) P[i] = __fadd2_rn(P[2 * i], P[2 * i + 1]);
    return P[0];
}

// Pairwise tree over N scalars (N a power of two).
template <int N, bool kTree>
__device__ __forceinline__ float tree_n(const float (&v)[N]) {
    float t[N];
#pragma unroll
    for (int i = 0; i < N; ++i) t[i] = v[i];
#pragma unroll
    for (int h = N / 2; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) t[i] = kTree ? __fadd_rn(t[2 * i], t[2 * i + 1]) : t[2 * i] + t[2 * i + 1];
    return t[0];
}

// One lane's slices of the T activations: X[t][m] = {x_t(m), x_t(m + LC/2)}
// of the lane's LC columns (scaled by -2^(23-4k) on the exact path).
template <int T, int LC>
struct MSlice {
    float2 X[T][LC / 2];
    float xs[T];  // group sums of the lane's group, per token
    bool exact;
    int negs;     // tree mode, bit t: every value of the lane's group of token t is negative
    bool anyneg;  // warp-uniform: negs != 0 in some lane
};

// Activation slices for chunk ch: x of token t at a.xt[t]; group sums given
// (kProNone, a.xst[t]) or computed (kProGsum).
template <int T, int LC, bool kTree>
__device__ __forceinline__ void load_mslice(const Q4ArgsT<kMmProbs> &a, int ch, int lane, MSlice<T, LC> &sl) {
    constexpr int kL = 64 / LC, GPC = 32 / kL;
    const int C = a.cols, base = ch * 32 * LC + lane * LC;
    const bool active = base < C;
    float v[T][LC];
    bool sp = false;
    int negs = 0;  // bit t: every value of this lane's slice of token t is negative
#pragma unroll
    for (int t = 0; t < T; ++t) {
#pragma unroll
        for (int i = 0; i < LC / 4; ++i) {
            float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
            if (active) q = reinterpret_cast<const float4 *>(a.xt[t] + base)[i];
            v[t][4 * i] = q.x, v[t][4 * i + 1] = q.y, v[t][4 * i + 2] = q.z, v[t][4 * i + 3] = q.w;
        }
        bool allneg = true;
#pragma unroll
        for (int j = 0; j < LC; ++j) {
            sp |= !x_ordinary(v[t][j]);
            allneg &= v[t][j] < 0.f;
        }
        if (active && allneg) negs |= 1 << t;
    }
    if (!active) sp = false;
    // a group spans kL lanes: all-negative groups per token (every lane
    // takes part in the shuffles)
#pragma unroll
    for (int d = 1; d < kL; d <<= 1) negs &= __shfl_xor_sync(0xffffffffu, negs, d);
    sl.exact = !__any_sync(0xffffffffu, sp);
    sl.negs = kTree ? negs : 0;
    sl.anyneg = __any_sync(0xffffffffu, sl.negs != 0);
    const int g = ch * GPC + lane / kL;
#pragma unroll
    for (int t = 0; t < T; ++t) {
        if (a.prologue == kProNone) {
            sl.xs[t] = active ? a.xst[t][g] : 0.f;
        } else {
            float s = tree_n<LC, kTree>(v[t]);
#pragma unroll
            for (int d = 1; d < kL; d <<= 1) {
                const float o = __shfl_xor_sync(0xffffffffu, s, d);
                s = kTree ? __fadd_rn(s, o) : s + o;
            }
            sl.xs[t] = s;
        }
#pragma unroll
        for (int m = 0; m < LC / 2; ++m) {
            if (sl.exact) {
                sl.X[t][m] = f2(__fmul_rn(v[t][m], -nib_scale(m % 8)), __fmul_rn(v[t][m + LC / 2], -nib_scale((m + LC / 2) % 8)));
            } else {
                sl.X[t][m] = f2(v[t][m], v[t][m + LC / 2]);
            }
        }
    }
}

// u pairs of the lane's LC columns for one row: U[m] = {u(m), u(m + LC/2)}.
template <int LC, int M = 0>
__device__ __forceinline__ void unpack_pairs(float2 (&U)[LC / 2], const uint32_t (&w)[2], const uint32_t (&h)[2]) {
    if constexpr (M < LC / 2) {
        U[M] = f2(neg_u_col<M>(w, h), neg_u_col<M + LC / 2>(w, h));
        unpack_pairs<LC, M + 1>(U, w, h);
    }
}

// Lane sums of one row for all T tokens into v[T].
template <int T, int LC, bool kExact>
__device__ __forceinline__ void lane_sums(const uint32_t (&w)[2], const MSlice<T, LC> &sl, float *v) {
    uint32_t h[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) h[i] = __umulhi(w[i], 1u << 20);
    if constexpr (kExact) {
        float2 U[LC / 2];
        unpack_pairs<LC>(U, w, h);
#pragma unroll
        for (int t = 0; t < T; ++t) {
            float2 P[LC / 2];
#pragma unroll
            for (int m = 0; m < LC / 2; ++m) P[m] = __ffma2_rn(U[m], sl.X[t][m], sl.X[t][m]);
            const float2 r = tree_pairs<LC / 2>(P);
            v[t] = __fadd_rn(r.x, r.y);
        }
    } else {
        float q[LC];
#pragma unroll
        for (int c = 0; c < LC; ++c) q[c] = q_exact(w[c / 8], h[c / 8], c % 8);
#pragma unroll
        for (int t = 0; t < T; ++t) {
            float2 P[LC / 4];
#pragma unroll
            for (int i = 0; i < LC / 4; ++i) {
                // first tree level in scalar RN ops (never contracted)
                const int m = 2 * i;
                const float a0 = __fmul_rn(q[m], sl.X[t][m].x), a1 = __fmul_rn(q[m + 1], sl.X[t][m + 1].x);
                const float b0 = __fmul_rn(q[m + LC / 2], sl.X[t][m].y), b1 = __fmul_rn(q[m + 1 + LC / 2], sl.X[t][m + 1].y);
                P[i] = f2(__fadd_rn(a0, a1), __fadd_rn(b0, b1));
            }
            const float2 r = tree_pairs<LC / 4>(P);
            v[t] = __fadd_rn(r.x, r.y);
        }
    }
}

// The token's group sum among the lane's T (t warp-divergent: selects, no
// indexed register array).
template <int T>
__device__ __forceinline__ float pick(const float (&xs)[T], int t) {
    float r = xs[0];
#pragma unroll
    for (int i = 1; i < T; ++i) r = (t == i) ? xs[i] : r;
    return r;
}

template <int T, int R, bool kTree, bool kSbSmem>
__global__ void __launch_bounds__(288, 2) q4mm_kernel(const __grid_constant__ Q4ArgsT<kMmProbs> a) {
    constexpr int LC = mm_lane_cols<T>();
    constexpr int CW = 32 * LC;      // columns of a warp's chunk
    constexpr int kL = 64 / LC;      // lanes per 64-column group
    constexpr int GPC = 32 / kL;     // groups per chunk
    constexpr int NV = R * T;        // (row, token) values per lane
    static_assert(NV <= 32, "lanes 0..NV-1 hold the final values");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ volatile int s_abort;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_bar);
    uint64_t *empty = full + a.stages;
    uint64_t *done = empty + a.stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.stages, TR = a.tile_rows, W = a.W, G = a.G, nch = a.nch, nw = a.nw;
    const int ntok = a.ntok;  // real tokens (slots past it are padding)

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], nw);
        }
        for (int i = 0; i < a.parts; ++i) mbar_init(&done[i], nw);
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const bool wait_first = a.wait_first != 0;
    if (!wait_first) grid_dep_launch();
    if (warp == 0) {
        // ------------------------------------------------ producer warp ----
        if (lane != 0) return;
        const uint64_t policy = l2_evict_first();
        bool released = !wait_first;
        ProbCursor cur;
        const int total = static_cast<int>(a.total_tiles);
        int k = 0, s = 0;
        uint32_t eph = 1;  // ((k / S) & 1) ^ 1 for k >= S
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++k) {
            if (k == S) {
                grid_dep_wait();
                grid_dep_launch();
                released = true;
            }
            if (k >= S && !wait_or_abort(&empty[s], eph, &s_abort, kSiteEmpty)) break;
            if (s_abort) break;
            int tile;
            const Q4Prob &P = a.prob[cur.find(a, t, tile)];
            const int64_t r0 = static_cast<int64_t>(tile) * TR;
            const int rows = static_cast<int>(min(static_cast<int64_t>(TR), P.n - r0));
            unsigned char *st = smem + a.off_stage + static_cast<size_t>(s) * a.stage_bytes;
            const uint32_t wb = static_cast<uint32_t>(rows) * W * 4u;
            const uint32_t sbb = kSbSmem ? static_cast<uint32_t>(rows) * G * 4u : 0u;
            mbar_arrive_expect_tx(&full[s], wb + 2 * sbb);
            bulk_g2s(st, P.w + r0 * W, wb, &full[s], policy);
            if (kSbSmem) {
                const size_t sbo = static_cast<size_t>(r0) * G * 4u;
                bulk_g2s(st + a.stage_w_bytes, static_cast<const unsigned char *>(P.scale) + sbo, sbb, &full[s],
                         policy);
                bulk_g2s(st + a.stage_w_bytes + a.stage_sb_bytes, static_cast<const unsigned char *>(P.bias) + sbo,
                         sbb, &full[s], policy);
            }
            if (++s == S) {
                s = 0;
                eph ^= 1u;
            }
        }
        if (!released) {
            grid_dep_wait();
            grid_dep_launch();
        }
        for (int j = max(0, k - S); j < k; ++j) mbar_wait(&full[j % S], static_cast<uint32_t>((j / S) & 1));
        return;
    }

    // ---------------------------------------------------- consumer warps ----
    const int ct = threadIdx.x - 32, cw = warp - 1;
    float *part = reinterpret_cast<float *>(smem + a.off_part);
    const bool fixed_ch = nch <= nw;
    const int kk = fixed_ch ? nw / nch : 1;
    const bool idle = fixed_ch && cw >= nch * kk;
    const int ch0 = fixed_ch ? cw % nch : cw;
    const int rb0 = fixed_ch ? cw / nch : 0;
    const int chstep = fixed_ch ? nch : nw;

    if (wait_first) {
        grid_dep_wait();
        grid_dep_launch();
    }
    MSlice<T, LC> sl;
    int cur_ch = -1;
    // Final sums of tile tj: thread ct < rows*T adds value (row, token) =
    // (ct / T, ct % T) over the chunks by the tree.
    ProbCursor cur, fcur;
    auto finish = [&](int tj, int pi, uint32_t dph) -> bool {
        if (!wait_or_abort(&done[pi], dph, &s_abort, kSiteDone)) return false;
        int tile;
        const Q4Prob &P = a.prob[fcur.find(a, tj, tile)];
        const int64_t r0 = static_cast<int64_t>(tile) * TR;
        const int rows = static_cast<int>(min(static_cast<int64_t>(TR), P.n - r0));
        if (ct < rows * T) {
            const int row = ct / T, tk = ct - row * T;
            float *pr = part + static_cast<size_t>(pi) * TR * nch * T;
            const int base = row * nch * T + tk;  // element c at base + c*T
            int m = nch;
            while (m > 1) {
                const int hh = m >> 1;
                for (int i = 0; i < hh; ++i) {
                    const float l = pr[base + 2 * i * T], r = pr[base + (2 * i + 1) * T];
                    pr[base + i * T] = kTree ? __fadd_rn(l, r) : l + r;
                }
                if (m & 1) pr[base + hh * T] = pr[base + (m - 1) * T];
                m = hh + (m & 1);
            }
            if (tk < ntok) P.y[static_cast<int64_t>(tk) * P.n + r0 + row] = pr[base];
        }
        return true;
    };

    const int total = static_cast<int>(a.total_tiles), NP = a.parts;
    const bool finisher = cw * 32 < TR * T;
    int tprev = -1, s = 0, pi = 0, ppi = 0;
    uint32_t fph = 0, dph = 0, pdph = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
        if (!wait_or_abort(&full[s], fph, &s_abort, kSiteFull)) break;
        int tile;
        const Q4Prob &P = a.prob[cur.find(a, t, tile)];
        const int64_t r0 = static_cast<int64_t>(tile) * TR;
        const int rows = static_cast<int>(min(static_cast<int64_t>(TR), P.n - r0));
        const unsigned char *stg = smem + a.off_stage + static_cast<size_t>(s) * a.stage_bytes;
        const uint32_t *sw = reinterpret_cast<const uint32_t *>(stg);
        const float *ssc = reinterpret_cast<const float *>(stg + a.stage_w_bytes);
        const float *sbi = reinterpret_cast<const float *>(stg + a.stage_w_bytes + a.stage_sb_bytes);
        float *prt = part + static_cast<size_t>(pi) * TR * nch * T;
        const int nrb = (rows + R - 1) / R;
        if (!idle) {
            for (int ch = ch0; ch < nch; ch += chstep) {
                if (ch != cur_ch) {
                    load_mslice<T, LC, kTree>(a, ch, lane, sl);
                    cur_ch = ch;
                }
                const bool active = (ch * CW + lane * LC) < a.cols;
                const int g = active ? ch * GPC + lane / kL : 0;
                // this lane's LC/8 words in row 0 of the stage (row 0's first
                // words past the row end; their sums are replaced by -0)
                const uint32_t *wl = sw + (active ? ch * (CW / 8) + lane * (LC / 8) : 0);
                for (int rb = rb0; rb < nrb; rb += kk) {
                    float v[NV];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t *wr = wl + (rb * R + r) * W;  // rows past a ragged end: stale, discarded
                        uint32_t w[2];
                        if constexpr (LC == 16) {
                            const uint2 q = *reinterpret_cast<const uint2 *>(wr);
                            w[0] = q.x, w[1] = q.y;
                        } else {
                            w[0] = wr[0], w[1] = 0u;
                        }
                        if (sl.exact)
                            lane_sums<T, LC, true>(w, sl, v + r * T);
                        else
                            lane_sums<T, LC, false>(w, sl, v + r * T);
                    }
                    constexpr int H = lv_count<NV, 1, kL>();
                    int sel = 0;
                    float d[H];
                    levels<NV, 1, kL, kTree>(v, d, lane, sel);
                    const int ofs = sel;
                    if (kTree && sl.exact && sl.anyneg) {
                        // zero sums are +0 on the exact path; in an all-negative
                        // group a zero sum means every q is 0, and RN's sum is -0
#pragma unroll
                        for (int i = 0; i < H; ++i)
                            d[i] = (((sl.negs >> ((ofs + i) % T)) & 1) && d[i] == 0.f) ? kNegZero : d[i];
                    }
                    float tv[H];
#pragma unroll
                    for (int i = 0; i < H; ++i) {
                        const int c = ofs + i, row = rb * R + c / T, tk = c % T;
                        const int64_t idx = kSbSmem ? static_cast<int64_t>(row * G + g)
                                                    : (r0 + min(row, rows - 1)) * G + g;
                        const float sc = kSbSmem ? ssc[idx] : __ldg(reinterpret_cast<const float *>(P.scale) + idx);
                        const float bi = kSbSmem ? sbi[idx] : __ldg(reinterpret_cast<const float *>(P.bias) + idx);
                        const float xs = pick<T>(sl.xs, tk);
                        const float tt = kTree ? __fadd_rn(__fmul_rn(sc, d[i]), __fmul_rn(bi, xs)) : fmaf(sc, d[i], bi * xs);
                        tv[i] = active ? tt : kNegZero;
                    }
                    float fin[1];
                    levels<H, kL, 32, kTree>(tv, fin, lane, sel);
                    // lanes 0..NV-1 hold (row, token) value sel
                    const int row = rb * R + sel / T, tk = sel % T;
                    if (lane < NV && row < rows) prt[(row * nch + ch) * T + tk] = fin[0];
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&empty[s]);
            mbar_arrive(&done[pi]);
        }
        if (finisher && tprev >= 0 && !finish(tprev, ppi, pdph)) break;
        tprev = t;
        ppi = pi;
        pdph = dph;
        if (++s == S) {
            s = 0;
            fph ^= 1u;
        }
        if (++pi == NP) {
            pi = 0;
            dph ^= 1u;
        }
    }
    if (finisher && tprev >= 0) finish(tprev, ppi, pdph);
    if (!wait_first) grid_dep_wait();
}

}  // namespace

}  // namespace abg
