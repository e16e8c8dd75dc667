// q4mv: affine 4-bit group-quantized matrix-vector product for sm_103a.
//
// Source: "Array.q4mv on Metal: one kernel thread per row ..." (bendlang/bend
// #1435, Change and Limits), "Metal: queued rmsq, swq, gdn and atq kernels and
// a 4-row q4mv ..." (#1440, Change: bend_q4mv bullet) and the product
//     y[r] = sum_g ( scale[r][g] * sum_j q[r][64g+j] * x[64g+j] + bias[r][g] * xsum[g] ).
//
// Data flow (one thread block per SM slot, persistent over row tiles):
//   warp 0 (producer)  streams tiles of whole rows -- packed words, and scale
//                      and bias where their rows are 16-byte aligned -- from
//                      HBM into a ring of shared-memory stages with 1-D bulk
//                      copies (cp.async.bulk) completing on mbarriers.  The
//                      weights are read once, so the copies carry an
//                      evict-first L2 policy.  They start before the kernel
//                      waits on its predecessor (programmatic dependent
//                      launch): weights never depend on an earlier stage.
//   warps 1..nw        wait for the predecessor, stage the activation row x
//                      (or compute it: group sums, RMS norm or SwiGLU) in
//                      shared memory, then work on (row block, 1024-column
//                      chunk) items.  A warp keeps its chunk of x in registers
//                      across items, so the activation is read from shared
//                      memory once per kernel, not once per row.
//
// Per lane and row a chunk is one 16-byte word quad (32 columns).  Nibble j of
// a word is turned into the float 2^(23-4(j%4)) + q by OR-ing an exponent into
// the masked word (the high half-word is shifted down first), and one fused
// multiply-add with c = -2^(23-4(j%4)) * x gives RN(q * x) exactly: the exact
// value (2^E + q)x - 2^E x = qx is rounded once.  So the product is the
// correctly rounded q*x that the tree order calls for, at one logic op and one
// FMA per weight (packed two at a time with the f32x2 ops).  The identity
// needs x finite, not -0 and |x| < 2^100; a block whose x has any other value
// takes the plain path (convert, then multiply), which is bit-identical.
//
// Reduction, tree order: the lane's 32 products are summed by the pairwise
// tree (16 packed adds carry two columns 16 apart, so every level pairs the
// right leaves), a shuffle with the neighbouring lane completes the 64-column
// group, the affine term is RN(RN(scale*d) + RN(bias*xsum)), and a 4-step
// butterfly over lane pairs sums the chunk's 16 groups.  Chunk partials meet
// in shared memory, where one thread per row sums them with the same tree
// (odd element carried).  Groups past the end of the row contribute -0, which
// leaves every tree sum unchanged.
#include "../../include/abg.h"
#include "abg_dev.cuh"
#include "abg_kernels.cuh"

#include <algorithm>
#include <mutex>
#include <set>

namespace abg {

namespace {

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Nibble j (0..7) of a word is read at bit position 4k of the word itself
// (j <= 4, k = j) or of the word shifted right by 12 (j >= 5, k = j - 3), so
// it always sits inside the 23 significand bits.
__host__ __device__ constexpr int nib_k(int j) { return j <= 4 ? j : j - 3; }

// (w & mask) | c as one three-input logic op (mask an immediate).
template <uint32_t kMask>
__device__ __forceinline__ uint32_t and_or(uint32_t w, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(w), "n"(kMask), "r"(c));
    return d;
}

// The pair of floats -(1 + q * 2^(4k-23)) for nibble J of words a and b
// (sign and exponent of -1.0, held in `neg_one`, OR-ed onto the masked nibble).
template <int J>
__device__ __forceinline__ float2 neg_u2(uint32_t a, uint32_t ah, uint32_t b, uint32_t bh, uint32_t neg_one) {
    constexpr uint32_t kMask = 0xFu << (4 * nib_k(J));
    const uint32_t sa = (J <= 4) ? a : ah, sb = (J <= 4) ? b : bh;
    return f2(__uint_as_float(and_or<kMask>(sa, neg_one)), __uint_as_float(and_or<kMask>(sb, neg_one)));
}

// q of nibble j as a float, exactly: (2^(23-4k) + q) - 2^(23-4k).
__device__ __forceinline__ float q_exact(uint32_t w, uint32_t wh, int j) {
    const int k = nib_k(j);
    const uint32_t src = (j <= 4) ? w : wh;
    const float v = __uint_as_float((src & (0xFu << (4 * k))) | (static_cast<uint32_t>(150 - 4 * k) << 23));
    return __fadd_rn(v, -__uint_as_float(static_cast<uint32_t>(150 - 4 * k) << 23));
}

// 2^(23-4k) for nibble j: the factor that turns q * 2^(4k-23) back into q.
__device__ __forceinline__ float nib_scale(int j) {
    return __uint_as_float(static_cast<uint32_t>(150 - 4 * nib_k(j)) << 23);
}

// Pairwise tree over the lane's 32 products, given as P[m] = {p_m, p_(m+16)}:
// adding P[2i] and P[2i+1] pairs leaves (2i, 2i+1) in both halves, and the
// halves stay aligned level after level.
__device__ __forceinline__ float tree32_pairs(float2 (&P)[16]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) P[i] = __fadd2_rn(P[2 * i], P[2 * i + 1]);
#pragma unroll
    for (int i = 0; i < 4; ++i) P[i] = __fadd2_rn(P[2 * i], P[2 * i + 1]);
#pragma unroll
    for (int i = 0; i < 2; ++i) P[i] = __fadd2_rn(P[2 * i], P[2 * i + 1]);
    P[0] = __fadd2_rn(P[0], P[1]);
    return __fadd_rn(P[0].x, P[0].y);
}

template <int M>
__device__ __forceinline__ void exact_products(float2 (&P)[16], uint32_t w0, uint32_t h0, uint32_t w1, uint32_t h1,
                                               uint32_t w2, uint32_t h2, uint32_t w3, uint32_t h3,
                                               const float2 (&X)[16], uint32_t neg_one) {
    if constexpr (M < 16) {
        const float2 u = (M < 8) ? neg_u2<M & 7>(w0, h0, w2, h2, neg_one) : neg_u2<M & 7>(w1, h1, w3, h3, neg_one);
        P[M] = __ffma2_rn(u, X[M], X[M]);
        exact_products<M + 1>(P, w0, h0, w1, h1, w2, h2, w3, h3, X, neg_one);
    }
}

// Tree sum of q*x over the lane's 32 columns of one row chunk (words wq).
//   exact path: X[m] = {-x(m) S_m, -x(m+16) S_m} with S_m = 2^(23-4k); the
//     product fma(-(1 + q 2^(4k-23)), -x S, -x S) = q x exactly before its one
//     rounding, so it is RN(q*x), at one logic op and half a packed FMA per
//     weight.
//   plain path (activations with zeros of either sign, infinities, NaN, huge
//     values, or a group of all-negative values): X[m] = {x(m), x(m+16)}; q is
//     converted exactly and multiplied with scalar RN ops.  (The compiler may
//     fuse a packed multiply into the packed add after it; the scalar
//     __fmul_rn / __fadd_rn intrinsics are never contracted.)
template <bool kExact>
__device__ __forceinline__ float lane_sum32(uint4 wq, const float2 (&X)[16]) {
    const uint32_t w0 = wq.x, w1 = wq.y, w2 = wq.z, w3 = wq.w;
    const uint32_t h0 = w0 >> 12, h1 = w1 >> 12, h2 = w2 >> 12, h3 = w3 >> 12;
    float2 P[16];
    if constexpr (kExact) {
        exact_products<0>(P, w0, h0, w1, h1, w2, h2, w3, h3, X, 0xBF800000u);
        return tree32_pairs(P);
    } else {
    float p[32];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int j = m & 7;
        const float qa = (m < 8) ? q_exact(w0, h0, j) : q_exact(w1, h1, j);
        const float qb = (m < 8) ? q_exact(w2, h2, j) : q_exact(w3, h3, j);
        p[m] = __fmul_rn(qa, X[m].x);
        p[m + 16] = __fmul_rn(qb, X[m].y);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        P[i] = f2(__fadd_rn(p[2 * i], p[2 * i + 1]), __fadd_rn(p[16 + 2 * i], p[17 + 2 * i]));
#pragma unroll
    for (int i = 0; i < 4; ++i) P[i] = add2(P[2 * i], P[2 * i + 1]);
#pragma unroll
    for (int i = 0; i < 2; ++i) P[i] = add2(P[2 * i], P[2 * i + 1]);
    P[0] = add2(P[0], P[1]);
    return __fadd_rn(P[0].x, P[0].y);
    }
}

// True when the exact path gives RN(q*x) for this activation value (finite,
// not a zero of either sign... +0 is fine for the identity but a zero is
// cheap to route to the plain path, and |x| < 2^100 so x * 2^23 cannot overflow).
__device__ __forceinline__ bool x_ordinary(float v) { return fabsf(v) < 1.2676506e30f && v != 0.0f; }

// Pairwise tree over 32 values in index order (scalar RN adds).
__device__ __forceinline__ float tree32(const float (&v)[32]) {
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = __fadd_rn(v[2 * i], v[2 * i + 1]);
#pragma unroll
    for (int h = 8; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) t[i] = __fadd_rn(t[2 * i], t[2 * i + 1]);
    return t[0];
}

// The same factor computed by all computing warps of a block together: each
// 64-value group is summed by 8 lanes (8 consecutive squares each, then a
// 3-step butterfly: the pairwise tree over 8 blocks of 8), group sums meet in
// shared memory, one warp takes the tree over groups (padded with -0).  Uses
// named barrier 1 over the nct computing threads (all of them call this).
template <bool kTree>
__device__ float block_rms_factor(const float *__restrict__ x, int C, float eps, int cw, int nw, int lane,
                                  float *red, float *rbox) {
    const int G = C / 64, nct = nw * 32;
    for (int g0 = 4 * cw; g0 < G; g0 += 4 * nw) {
        const int g = g0 + (lane >> 3);
        float s = kNegZero;
        if (g < G) {
            const float4 *p4 = reinterpret_cast<const float4 *>(x + 64 * g + 8 * (lane & 7));
            const float4 a = p4[0], b = p4[1];
            const float t0 = __fadd_rn(__fmul_rn(a.x, a.x), __fmul_rn(a.y, a.y));
            const float t1 = __fadd_rn(__fmul_rn(a.z, a.z), __fmul_rn(a.w, a.w));
            const float t2 = __fadd_rn(__fmul_rn(b.x, b.x), __fmul_rn(b.y, b.y));
            const float t3 = __fadd_rn(__fmul_rn(b.z, b.z), __fmul_rn(b.w, b.w));
            s = __fadd_rn(__fadd_rn(t0, t1), __fadd_rn(t2, t3));
        }
#pragma unroll
        for (int d = 1; d < 8; d <<= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, d));
        if (g < G && (lane & 7) == 0) red[g] = s;
    }
    named_bar(1, nct);
    if (cw == 0) {
        const float ss = warp_tree_smem(red, G);
        if (lane == 0) {
            float r;
            if (kTree) {
                const float mean = __fdiv_rn(ss, static_cast<float>(C));
                r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
            } else {
                r = rsqrtf(ss / static_cast<float>(C) + eps);
            }
            *rbox = r;
        }
    }
    named_bar(1, nct);
    return *rbox;
}

// One warp's slice of the activation: columns ch*1024 + lane*32 + (0..31).
struct Slice {
    float2 X[16];  // see lane_sum32
    float xs;      // group sum of the lane's 64-column group
    bool exact;    // warp-uniform: the exact path applies to the whole slice
};

template <bool kTree>
__device__ __forceinline__ void load_slice(const Q4Args &a, int ch, int lane, float rms_r, Slice &sl) {
    const int C = a.cols, base = ch * 1024 + lane * 32;
    const bool active = base < C;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
    if (active) {
        const float4 *x4 = reinterpret_cast<const float4 *>(a.x + base);
        if (a.prologue == kProNone || a.prologue == kProGsum) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 q = x4[i];
                v[4 * i] = q.x, v[4 * i + 1] = q.y, v[4 * i + 2] = q.z, v[4 * i + 3] = q.w;
            }
        } else if (a.prologue == kProRmsq) {
            const float4 *w4 = reinterpret_cast<const float4 *>(a.wt + base);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 q = x4[i], w = w4[i];
                v[4 * i] = __fmul_rn(__fmul_rn(q.x, rms_r), w.x);
                v[4 * i + 1] = __fmul_rn(__fmul_rn(q.y, rms_r), w.y);
                v[4 * i + 2] = __fmul_rn(__fmul_rn(q.z, rms_r), w.z);
                v[4 * i + 3] = __fmul_rn(__fmul_rn(q.w, rms_r), w.w);
            }
        } else {  // kProSwq: x = [gate | up]
            const float4 *u4 = reinterpret_cast<const float4 *>(a.x + C + base);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 g = x4[i], u = u4[i];
                v[4 * i] = swiglu<kTree>(g.x, u.x);
                v[4 * i + 1] = swiglu<kTree>(g.y, u.y);
                v[4 * i + 2] = swiglu<kTree>(g.z, u.z);
                v[4 * i + 3] = swiglu<kTree>(g.w, u.w);
            }
        }
    }
    // special values, and groups whose 64 values are all negative (there the
    // exact path's q = 0 products would be +0 where RN(0 * x) is -0, and a
    // whole group of them could leave -0 in the sum)
    bool sp = false, allneg = true;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        sp |= !x_ordinary(v[i]);
        allneg &= v[i] < 0.f;
    }
    if (!active) sp = false, allneg = false;
    // every lane takes part in the shuffle (a full-mask shuffle that only some
    // lanes reach, e.g. behind a short-circuit &&, stalls the warp for good)
    const bool partner_neg = __shfl_xor_sync(0xffffffffu, allneg ? 1 : 0, 1) != 0;
    const bool grpneg = allneg && partner_neg;
    sl.exact = !__any_sync(0xffffffffu, sp || grpneg);
    // group sum of the lane's group: given, or the tree over the slice's values
    if (a.prologue == kProNone) {
        sl.xs = active ? a.xsum[ch * 16 + (lane >> 1)] : 0.f;
    } else {
        const float t = kTree ? tree32(v) : [&] {
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) s += v[i];
            return s;
        }();
        const float o = __shfl_xor_sync(0xffffffffu, t, 1);
        sl.xs = kTree ? __fadd_rn(t, o) : t + o;
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        if (sl.exact) {
            const float s = -nib_scale(m & 7);
            sl.X[m] = f2(__fmul_rn(v[m], s), __fmul_rn(v[m + 16], s));
        } else {
            sl.X[m] = f2(v[m], v[m + 16]);
        }
    }
}

// Locates tiles of a grouped launch.  A block visits its tiles in increasing
// order, so the problem index only moves forward.
struct ProbCursor {
    int p = 0;
    int64_t base = 0;  // first tile of problem p
    __device__ __forceinline__ int find(const Q4Args &a, int64_t t, int64_t &tile) {
        while (p + 1 < a.nprob && t >= base + a.prob[p].tiles) {
            base += a.prob[p].tiles;
            ++p;
        }
        tile = t - base;
        return p;
    }
};

// Bounded mbarrier wait that also gives up when another warp has aborted.
// On a timeout it sets the timeout bit plus `site` (which wait gave up).
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              unsigned site) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(&g_status, kStatusTimeout | site);
            *abort_flag = 1;
            return false;
        }
    }
}
// wait sites recorded in the status word
constexpr unsigned kSiteEmpty = 1u << 4, kSiteFull = 1u << 5, kSiteDone = 1u << 6;

// One step of a transposed butterfly over N values (N -> N/2): lanes whose
// `d` bit is clear keep the first half and send the second, their partners
// the other way round, so each lane adds N/2 pairs with N/2 shuffles.  The
// sums pair the same two leaves as a plain butterfly step.
template <int N, bool kTree>
__device__ __forceinline__ void tstep(float (&v)[N], int d, bool hi) {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float send = hi ? v[i] : v[N / 2 + i];
        const float keep = hi ? v[N / 2 + i] : v[i];
        const float recv = __shfl_xor_sync(0xffffffffu, send, d);
        v[i] = kTree ? __fadd_rn(keep, recv) : keep + recv;
    }
}

// Butterfly levels from distance `dist` up to 16 over N held values: while
// N > 1 each level is a transposed step (the lane keeps the half selected by
// its `dist` bit, recorded in rowsel); then plain butterfly steps.
template <int N, bool kTree>
__device__ __forceinline__ float group_levels(float (&v)[N], int lane, int dist, int &rowsel) {
    if constexpr (N == 1) {
        float val = v[0];
        for (int dd = dist; dd < 32; dd <<= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, val, dd);
            val = kTree ? __fadd_rn(val, o) : val + o;
        }
        return val;
    } else {
        const bool hi = (lane & dist) != 0;
        tstep<N, kTree>(v, dist, hi);
        rowsel += hi ? N / 2 : 0;
        float w[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i) w[i] = v[i];
        return group_levels<N / 2, kTree>(w, lane, dist * 2, rowsel);
    }
}

// Partial-sum buffers (and their barriers) rotate over 4 tiles: a warp writes
// a tile's buffer only after every warp has finished the final sums of the
// tile four back.
constexpr int kParts = 4;

// Block layouts (the register file is split over the SM's four schedulers,
// so the warps per SM set the registers per thread):
//   kLayout 0: up to 8 computing warps, two blocks per SM (96 registers);
//   kLayout 1: up to 16 computing warps, one block per SM;
//   kLayout 2: up to 6 computing warps, two blocks per SM (128 registers).
// With two blocks per SM the next launch of a chain can start beside this one.
constexpr int layout_threads(int l) { return l == 1 ? 544 : (l == 2 ? 224 : 288); }
constexpr int layout_blocks(int l) { return l == 1 ? 1 : 2; }

template <int R, bool kTree, bool kSbSmem, int kLayout>
__global__ void __launch_bounds__(layout_threads(kLayout), layout_blocks(kLayout))
    q4mv_kernel(const __grid_constant__ Q4Args a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ volatile int s_abort;
    __shared__ float s_red[ABG_MAX_COLS / 64];  // group sums of squares (RMS-norm prologue)
    __shared__ float s_rbox;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_bar);
    uint64_t *empty = full + a.stages;
    uint64_t *done = empty + a.stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.stages, TR = a.tile_rows, W = a.W, G = a.G, nch = a.nch, nw = a.nw;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], nw);
        }
        for (int i = 0; i < kParts; ++i) mbar_init(&done[i], nw);
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // Programmatic dependent launch.  When the activation comes from the
    // preceding launch (wait_first), the first S tiles of weights are fetched
    // before waiting for it (weights never depend on it) and every thread
    // signals its dependents only after that wait has returned.  A sibling
    // launch of the same stage signals at once, computes, and waits for its
    // predecessor only before exiting.
    const bool wait_first = a.wait_first != 0;
    if (!wait_first) grid_dep_launch();
    if (warp == 0) {
        // ------------------------------------------------ producer warp ----
        if (lane != 0) return;
        const uint64_t policy = l2_evict_first();
        bool released = !wait_first;
        ProbCursor cur;
        int64_t k = 0;
        for (int64_t t = blockIdx.x; t < a.total_tiles; t += gridDim.x, ++k) {
            const int s = static_cast<int>(k % S);
            if (k == S) {
                grid_dep_wait();
                grid_dep_launch();
                released = true;
            }
            if (k >= S && !wait_or_abort(&empty[s], static_cast<uint32_t>(((k / S) & 1) ^ 1), &s_abort, kSiteEmpty))
                break;
            if (s_abort) break;
            int64_t tile;
            const Q4Prob &P = a.prob[cur.find(a, t, tile)];
            const int64_t r0 = tile * TR;
            const int rows = static_cast<int>(min(static_cast<int64_t>(TR), P.n - r0));
            unsigned char *st = smem + a.off_stage + static_cast<size_t>(s) * a.stage_bytes;
            const uint32_t wb = static_cast<uint32_t>(rows) * W * 4u;
            const uint32_t sbb = kSbSmem ? static_cast<uint32_t>(rows) * G * 4u : 0u;
            mbar_arrive_expect_tx(&full[s], wb + 2 * sbb);
            bulk_g2s(st, P.w + r0 * W, wb, &full[s], policy);
            if (kSbSmem) {
                bulk_g2s(st + a.stage_w_bytes, P.scale + r0 * G, sbb, &full[s], policy);
                bulk_g2s(st + a.stage_w_bytes + a.stage_sb_bytes, P.bias + r0 * G, sbb, &full[s], policy);
            }
        }
        if (!released) {
            grid_dep_wait();
            grid_dep_launch();
        }
        // Drain: the block may not exit while a copy into its shared memory is
        // in flight.  Waiting on a phase that already completed returns at once.
        for (int64_t j = max(static_cast<int64_t>(0), k - S); j < k; ++j)
            mbar_wait(&full[j % S], static_cast<uint32_t>((j / S) & 1));
        return;
    }

    // ---------------------------------------------------- consumer warps ----
    const int ct = threadIdx.x - 32, cw = warp - 1;
    float *part = reinterpret_cast<float *>(smem + a.off_part);
    // chunk positions and row blocks of this warp
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
    float rms_r = 0.f;
    if (a.prologue == kProRmsq) rms_r = block_rms_factor<kTree>(a.x, a.cols, a.eps, cw, nw, lane, s_red, &s_rbox);
    Slice sl;
    int cur_ch = -1;
    // Final sums of tile j: thread ct adds row ct's chunk partials by the tree.
    ProbCursor cur, fcur;
    auto finish = [&](int64_t j, int64_t tj) -> bool {
        const int pi = static_cast<int>(j % kParts);
        if (!wait_or_abort(&done[pi], static_cast<uint32_t>((j / kParts) & 1), &s_abort, kSiteDone)) return false;
        int64_t tile;
        const Q4Prob &P = a.prob[fcur.find(a, tj, tile)];
        const int64_t r0 = tile * TR;
        const int rows = static_cast<int>(min(static_cast<int64_t>(TR), P.n - r0));
        if (ct < rows) {
            float *pr = part + (static_cast<size_t>(pi) * TR + ct) * nch;
            int m = nch;
            while (m > 1) {
                const int h = m >> 1;
                for (int i = 0; i < h; ++i) pr[i] = kTree ? __fadd_rn(pr[2 * i], pr[2 * i + 1]) : pr[2 * i] + pr[2 * i + 1];
                if (m & 1) pr[h] = pr[m - 1];
                m = h + (m & 1);
            }
            P.y[r0 + ct] = pr[0];
        }
        return true;
    };

    int64_t k = 0, tprev = -1;
    for (int64_t t = blockIdx.x; t < a.total_tiles; t += gridDim.x, ++k) {
        const int s = static_cast<int>(k % S);
        if (!wait_or_abort(&full[s], static_cast<uint32_t>((k / S) & 1), &s_abort, kSiteFull)) break;
        int64_t tile;
        const Q4Prob &P = a.prob[cur.find(a, t, tile)];
        const int64_t r0 = tile * TR;
        const int rows = static_cast<int>(min(static_cast<int64_t>(TR), P.n - r0));
        const unsigned char *stg = smem + a.off_stage + static_cast<size_t>(s) * a.stage_bytes;
        const uint4 *sw = reinterpret_cast<const uint4 *>(stg);
        const float *ssc = reinterpret_cast<const float *>(stg + a.stage_w_bytes);
        const float *sbi = reinterpret_cast<const float *>(stg + a.stage_w_bytes + a.stage_sb_bytes);
        float *prt = part + static_cast<size_t>(k % kParts) * TR * nch;
        const int nrb = (rows + R - 1) / R;
        if (!idle) {
            for (int ch = ch0; ch < nch; ch += chstep) {
                if (ch != cur_ch) {
                    load_slice<kTree>(a, ch, lane, rms_r, sl);
                    cur_ch = ch;
                }
                const bool active = (ch * 1024 + lane * 32) < a.cols;
                const int g = ch * 16 + (lane >> 1);
                // this lane's 16-byte column quad in row 0 of the stage; lanes
                // past the row end (last chunk only) read row 0's first quad
                // instead and their sums are discarded
                const uint4 *wl = sw + (active ? ch * 32 + lane : 0);
                const int wq_stride = W / 4;
                for (int rb = rb0; rb < nrb; rb += kk) {
                    // lane sums of R rows, four rows at a time: their loads
                    // first, then the arithmetic
                    float v[R];
                    const int nr = min(R, rows - rb * R);  // uniform; R except in the last block
                    constexpr int B = (R < 4) ? R : 4;
#pragma unroll
                    for (int bq = 0; bq < R; bq += B) {
                        uint4 wq[B];
#pragma unroll
                        for (int r = 0; r < B; ++r)
                            wq[r] = wl[(bq + r < nr ? rb * R + bq + r : 0) * wq_stride];
                        if (sl.exact) {
#pragma unroll
                            for (int r = 0; r < B; ++r) v[bq + r] = lane_sum32<true>(wq[r], sl.X);
                        } else {
#pragma unroll
                            for (int r = 0; r < B; ++r) v[bq + r] = lane_sum32<false>(wq[r], sl.X);
                        }
                    }
                    // group completion (lane pair), transposed when R > 1: this
                    // lane keeps rows [ofs, ofs + R/2)
                    constexpr int H = (R > 1) ? R / 2 : 1;
                    int ofs = 0;
                    float d[H];
                    if constexpr (R > 1) {
                        const bool hi = lane & 1;
                        tstep<R, kTree>(v, 1, hi);
                        ofs = hi ? R / 2 : 0;
#pragma unroll
                        for (int i = 0; i < H; ++i) d[i] = v[i];
                    } else {
                        const float o = __shfl_xor_sync(0xffffffffu, v[0], 1);
                        d[0] = kTree ? __fadd_rn(v[0], o) : v[0] + o;
                    }
                    // affine term per (row, group); groups past the row end add -0
                    float tv[H];
#pragma unroll
                    for (int i = 0; i < H; ++i) {
                        const int row = rb * R + ofs + i;
                        tv[i] = kNegZero;
                        if (active && row < rows) {
                            float sc, bi;
                            if (kSbSmem) {
                                sc = ssc[row * G + g];
                                bi = sbi[row * G + g];
                            } else {
                                sc = __ldg(P.scale + (r0 + row) * G + g);
                                bi = __ldg(P.bias + (r0 + row) * G + g);
                            }
                            tv[i] = kTree ? __fadd_rn(__fmul_rn(sc, d[i]), __fmul_rn(bi, sl.xs))
                                          : fmaf(sc, d[i], bi * sl.xs);
                        }
                    }
                    // the chunk's 16 groups: butterfly over lane pairs (distances
                    // 2..16), transposed while more than one row is held
                    int rowsel = ofs;
                    const float val = group_levels<H, kTree>(tv, lane, 2, rowsel);
                    // lanes 0..R-1 hold the R rows (row rb*R + rowsel)
                    const int row = rb * R + rowsel;
                    if (lane < R && row < rows) prt[row * nch + ch] = val;
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&empty[s]);       // weights of this stage no longer needed
            mbar_arrive(&done[k % kParts]);  // this warp's partials are written
        }
        if (tprev >= 0 && !finish(k - 1, tprev)) break;
        tprev = t;
    }
    if (tprev >= 0) finish(k - 1, tprev);
    if (!wait_first) grid_dep_wait();
}

template <int R, bool kTree, bool kSb, int kLayout>
void *kernel_ptr() {
    return reinterpret_cast<void *>(&q4mv_kernel<R, kTree, kSb, kLayout>);
}

void *select_kernel(int R, bool tree, bool sb, int layout) {
    if (layout != 0) {  // built for 8 rows per item only
        if (R != 8) return nullptr;
        if (layout == 1) {
            if (tree) return sb ? kernel_ptr<8, true, true, 1>() : kernel_ptr<8, true, false, 1>();
            return sb ? kernel_ptr<8, false, true, 1>() : kernel_ptr<8, false, false, 1>();
        }
        if (tree) return sb ? kernel_ptr<8, true, true, 2>() : kernel_ptr<8, true, false, 2>();
        return sb ? kernel_ptr<8, false, true, 2>() : kernel_ptr<8, false, false, 2>();
    }
#define ABG_SEL(RR)                                                                                  \
    if (R == RR) {                                                                                   \
        if (tree) return sb ? kernel_ptr<RR, true, true, 0>() : kernel_ptr<RR, true, false, 0>();    \
        return sb ? kernel_ptr<RR, false, true, 0>() : kernel_ptr<RR, false, false, 0>();            \
    }
    ABG_SEL(1)
    ABG_SEL(2)
    ABG_SEL(4)
    ABG_SEL(8)
#undef ABG_SEL
    return nullptr;
}

inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

cudaError_t raise_smem_limit(void *fn);

}  // namespace

cudaError_t q4mv_status(unsigned *bits, bool clear) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof v);
    if (e == cudaSuccess && clear && v) {
        const unsigned z = 0;
        e = cudaMemcpyToSymbol(g_status, &z, sizeof z);
    }
    *bits |= v;
    return e;
}

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

namespace {
bool plan_once(Q4Plan *plan, const Q4Prob *probs, int nprob, int cols, int prologue, const float *x,
               const float *xsum, const float *wt, float eps, bool tree, int rows_per_warp, bool sb_smem,
               const Q4Tuning &tune) {
    Q4Args &a = plan->args;
    a = Q4Args{};
    const int R = rows_per_warp;
    const int C = cols, W = C / 8, G = C / 64, nch = (C + 1023) / 1024;
    // consumer warps: a multiple of the chunk count (each warp keeps one
    // 1024-column slice of x), at most 8 (the kernel's launch bound)
    // layout: tuned consumer_warps > 8 selects one block per SM; 1..6 with 8
    // rows per item selects the 128-register two-block layout
    const int layout = (R != 8 || tune.consumer_warps == 0) ? 0 : (tune.consumer_warps > 8 ? 1 : (tune.consumer_warps <= 6 ? 2 : 0));
    const bool wide = layout == 1;
    const int nw_max = wide ? 16 : (layout == 2 ? 6 : 8);
    int nw = tune.consumer_warps;
    if (nw <= 0) nw = nch <= 8 ? nch * (8 / nch) : 8;
    if (nch <= nw_max) nw = nch * (std::min(nw, nw_max) / nch);
    nw = std::min(std::max(nw, 1), nw_max);
    const int kk = (nch <= nw) ? nw / nch : 1;  // warps per chunk position
    const uint32_t row_bytes = static_cast<uint32_t>(C / 2 + (sb_smem ? 8 * G : 0));
    const uint32_t fixed = 1024;  // barriers and alignment slack
    uint32_t budget = static_cast<uint32_t>(tune.smem_kb > 0 ? tune.smem_kb : (wide ? 220 : 110)) * 1024u;
    const uint32_t hard_max = 225u * 1024u;  // leaves room for the static shared memory
    // tile rows: a multiple of R*kk so row blocks spread evenly over the warps
    const int unit = R * kk;
    int TR = unit;
    const uint32_t stage_target = static_cast<uint32_t>(tune.stage_kb > 0 ? tune.stage_kb : 40) * 1024u;
    while (TR * 2 <= nw * 32 && (TR * 2) * row_bytes <= stage_target) TR *= 2;
    TR = std::min(TR, nw * 32);
    if (TR < R) return false;
    auto stage_bytes = [&](int tr) {
        return align_up(static_cast<uint32_t>(tr) * (C / 2), 16) +
               2u * align_up(sb_smem ? static_cast<uint32_t>(tr) * G * 4u : 0u, 16);
    };
    auto part_bytes = [&](int tr) { return align_up(static_cast<uint32_t>(kParts * tr * nch) * 4u, 16); };
    int S = 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
        for (;;) {
            const uint32_t sb = stage_bytes(TR);
            S = 0;
            while (S < 8 && fixed + (S + 1) * sb + part_bytes(TR) + 16u * (S + 1) + 8u * kParts <= budget) ++S;
            if (S >= 2 || TR <= unit) break;
            TR = std::max(unit, TR / 2);
        }
        if (S >= 2) break;
        budget = hard_max;
    }
    if (S < 2) return false;

    a.nprob = nprob;
    a.total_tiles = 0;
    for (int i = 0; i < nprob; ++i) {
        a.prob[i] = probs[i];
        a.prob[i].tiles = (probs[i].n + TR - 1) / TR;
        a.total_tiles += a.prob[i].tiles;
    }
    a.x = x;
    a.xsum = xsum;
    a.wt = wt;
    a.eps = eps;
    a.prologue = prologue;
    a.wait_first = 1;
    a.cols = C;
    a.W = W;
    a.G = G;
    a.nch = nch;
    a.tile_rows = TR;
    a.stages = S;
    a.nw = nw;
    a.off_stage = 0;
    a.stage_w_bytes = align_up(static_cast<uint32_t>(TR) * (C / 2), 16);
    a.stage_sb_bytes = align_up(sb_smem ? static_cast<uint32_t>(TR) * G * 4u : 0u, 16);
    a.stage_bytes = a.stage_w_bytes + 2 * a.stage_sb_bytes;
    a.off_part = a.off_stage + S * a.stage_bytes;
    a.off_bar = align_up(a.off_part + part_bytes(TR), 16);
    a.smem_bytes = a.off_bar + 16u * S + 8u * kParts;

    // blocks per SM: what fits (registers and shared memory), at most 2 unless tuned
    int fit = 1;
    void *fn = select_kernel(R, tree, sb_smem, layout);
    if (fn && raise_smem_limit(fn) == cudaSuccess) {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, static_cast<int>(32 * (1 + nw)), a.smem_bytes) ==
                cudaSuccess &&
            nb > 0)
            fit = nb;
    }
    cudaGetLastError();
    int bps = std::min(fit, wide ? 1 : (tune.blocks_per_sm > 0 ? tune.blocks_per_sm : 2));
    bps = std::max(bps, 1);
    const int64_t cap = static_cast<int64_t>(sm_count()) * bps;
    plan->grid = dim3(static_cast<unsigned>(std::max<int64_t>(1, std::min(a.total_tiles, cap))));
    plan->block = dim3(32u * (1 + nw));
    plan->rows_per_warp = R;
    plan->tree = tree;
    plan->sb_smem = sb_smem;
    plan->layout = layout;
    return true;
}

// Every instantiation gets the device's largest dynamic shared-memory limit
// once, so launches with different plans (different sizes) of one kernel can
// share it (a per-plan limit would be overwritten by the last plan prepared).
cudaError_t raise_smem_limit(void *fn) {
    static std::mutex mu;
    static std::set<void *> done;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count(fn)) return cudaSuccess;
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, fn);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - static_cast<int>(fa.sharedSizeBytes));
    if (e == cudaSuccess) done.insert(fn);
    return e;
}

}  // namespace

// Plans with the requested rows per item; if the stages do not fit in shared
// memory (very wide rows), retries with fewer rows per item (same results).
bool plan_q4mv(Q4Plan *plan, const Q4Prob *probs, int nprob, int cols, int prologue, const float *x,
               const float *xsum, const float *wt, float eps, bool tree, int rows_per_warp, bool sb_smem,
               const Q4Tuning &tune) {
    for (int R = rows_per_warp; R >= 1; R /= 2)
        if (plan_once(plan, probs, nprob, cols, prologue, x, xsum, wt, eps, tree, R, sb_smem, tune)) return true;
    return false;
}

cudaError_t prepare_q4mv(const Q4Plan &plan) {
    void *fn = select_kernel(plan.rows_per_warp, plan.tree, plan.sb_smem, plan.layout);
    if (!fn) return cudaErrorInvalidValue;
    return raise_smem_limit(fn);
}

cudaError_t launch_q4mv(const Q4Plan &plan, cudaStream_t stream, bool pdl) {
    if (plan.args.total_tiles == 0) return cudaSuccess;
    void *fn = select_kernel(plan.rows_per_warp, plan.tree, plan.sb_smem, plan.layout);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = plan.grid;
    cfg.blockDim = plan.block;
    cfg.dynamicSmemBytes = plan.args.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void *params[] = {const_cast<Q4Args *>(&plan.args)};
    return cudaLaunchKernelExC(&cfg, fn, params);
}

}  // namespace abg
