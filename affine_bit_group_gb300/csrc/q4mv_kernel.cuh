// q4mv kernel: affine 4-bit group-quantized matrix-vector product for sm_103a.
// Included by each translation unit that instantiates it for a weight format.
//
// Source: "Array.q4mv on Metal: one kernel thread per row ..." (bendlang/bend
// #1435, Change and Limits), "Metal: queued rmsq, swq, gdn and atq kernels and
// a 4-row q4mv ..." (#1440, Change: bend_q4mv bullet; Why: the MLX 4-bit
// formats) and the product, for groups of gs columns,
//     y[r] = sum_g ( scale[r][g] * sum_j q[r][gs*g+j] * x[gs*g+j] + bias[r][g] * xsum[g] ).
// Formats (template parameters): gs = 32 << kLg (32, 64 or 128 columns) and
// scale/bias stored as f32 or, with kHalf, as 16-bit bf16 or f16 (chosen at
// run time), widened to f32 exactly before use.
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
// a word sits at bit 4k of the word (j <= 4, k = j) or of the word shifted
// right by 12 (j >= 5, k = j - 3); masking it and OR-ing in the sign and
// exponent of -1.0 gives u = -(1 + q 2^(4k-23)), and with the activation held
// as x' = -x 2^(23-4k) one fused multiply-add u x' + x' is q x exactly before
// its single rounding: RN(q * x), the product the tree order calls for, at one
// logic op and half a packed FMA per weight.  The identity needs x finite,
// nonzero and |x| < 2^100; a warp whose slice holds any other value takes the
// plain path (convert, then multiply).  Its one difference from RN is the sign
// of a zero (q = 0 gives +0 where RN(0 * x) is -0 for x < 0), which can reach
// the output only through a zero group sum of an all-negative group; there the
// sum is set to -0 (see the product loop).  Both paths are bit-identical to
// the plain definition.
//
// Reduction, tree order: the lane's 32 products are summed by the pairwise
// tree (16 packed adds carry two columns 16 apart, so every level pairs the
// right leaves); a group of gs columns spans gs/32 lanes, and as many
// butterfly steps (0, 1 or 2) complete its sum d; the affine term is
// RN(RN(scale*d) + RN(bias*xsum)), and the remaining butterfly steps sum the
// chunk's 1024/gs groups.  Chunk partials meet in shared memory, where one
// thread per row sums them with the same tree (odd element carried).  Groups
// past the end of the row contribute -0, which leaves every tree sum
// unchanged.  Since every group and chunk is a power-of-two block of the
// row, these steps are exactly the pairwise tree over the groups.
#pragma once

#include "../../include/abg.h"
#include "abg_dev.cuh"
#include "abg_kernels.cuh"

#include <cuda_fp16.h>

#include <type_traits>

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

// 2^(4k-23) for nibble j, the inverse of nib_scale (exact).
__device__ __forceinline__ float nib_unscale(int j) {
    return __uint_as_float(static_cast<uint32_t>(104 + 4 * nib_k(j)) << 23);
}

// A stored 16-bit scale or bias widened to f32 (exact for both types).
__device__ __forceinline__ float widen16(unsigned short h, bool f16) {
    return f16 ? __half2float(__ushort_as_half(h)) : __uint_as_float(static_cast<uint32_t>(h) << 16);
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
//   plain path (activations with zeros of either sign, infinities, NaN or
//     huge values): X[m] = {x(m), x(m+16)}; q is
//     converted exactly and multiplied with scalar RN ops.  (The compiler may
//     fuse a packed multiply into the packed add after it; the scalar
//     __fmul_rn / __fadd_rn intrinsics are never contracted.)
template <bool kExact>
__device__ __forceinline__ float lane_sum32(uint4 wq, const float2 (&X)[16]) {
    const uint32_t w0 = wq.x, w1 = wq.y, w2 = wq.z, w3 = wq.w;
    // w >> 12 as the high word of w * 2^20: the multiplier pipe, not the
    // logic pipe that the unpacking keeps busy
    const uint32_t h0 = __umulhi(w0, 1u << 20), h1 = __umulhi(w1, 1u << 20), h2 = __umulhi(w2, 1u << 20),
                   h3 = __umulhi(w3, 1u << 20);
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

// The factor from the C/64 block sums of squares posted in red: one warp takes
// the tree over them, every computing thread (nct, named barrier 1) reads it.
template <bool kTree>
__device__ __forceinline__ float rms_from_blocks(float *red, int C, float eps, int cw, int nct, float *rbox) {
    named_bar(1, nct);
    if (cw == 0) {
        const float ss = warp_tree_smem(red, C / 64);
        if ((threadIdx.x & 31) == 0) {
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
    return rms_from_blocks<kTree>(red, C, eps, cw, nct, rbox);
}

// One warp's slice of the activation: columns ch*1024 + lane*32 + (0..31).
struct Slice {
    float2 X[16];  // see lane_sum32
    float xs;      // group sum of the group the lane's columns belong to
    float xsp;     // group sum of the partner group (the other group of its pair)
    bool exact;    // warp-uniform: the exact path applies to the whole slice
    bool neg;      // tree mode: every activation of this lane's group is negative
    bool anyneg;   // tree mode, warp-uniform: some lane's group is all negative
    bool act;      // the lane's columns lie inside the row
    bool actp;     // the partner group's columns lie inside the row
    bool full;     // warp-uniform: every lane's columns lie inside the row
};

// The rest of a slice from its activation values v (zero where inactive):
// the product path, the group sums, and the pairs X of lane_sum32.
template <bool kTree, int kLg, class A>
__device__ __forceinline__ void finish_slice(const A &a, int ch, int lane, bool active, float (&v)[32],
                                             Slice &sl) {
    // special values take the plain path; groups whose values are all
    // negative are marked for the sign of a zero group sum (see the product
    // loop)
    bool sp = false, allneg = true;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        sp |= !x_ordinary(v[i]);
        allneg &= v[i] < 0.f;
    }
    if (!active) sp = false, allneg = false;
    // a group spans 1 << kLg lanes; every lane takes part in the shuffles (a
    // full-mask shuffle that only some lanes reach, e.g. behind a
    // short-circuit &&, stalls the warp for good)
    int grpneg = allneg ? 1 : 0;
#pragma unroll
    for (int d = 1; d < (1 << kLg); d <<= 1) grpneg &= __shfl_xor_sync(0xffffffffu, grpneg, d);
    sl.exact = !__any_sync(0xffffffffu, sp);
    sl.neg = kTree && grpneg != 0;
    sl.anyneg = __any_sync(0xffffffffu, sl.neg);
    // group sum of the lane's group: given, or the tree over the slice's values
    // completed across the group's lanes
    if (a.prologue == kProNone) {
        sl.xs = active ? a.xsum[ch * (32 >> kLg) + (lane >> kLg)] : 0.f;
    } else {
        float t = kTree ? tree32(v) : [&] {
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) s += v[i];
            return s;
        }();
#pragma unroll
        for (int d = 1; d < (1 << kLg); d <<= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, t, d);
            t = kTree ? __fadd_rn(t, o) : t + o;
        }
        sl.xs = t;
    }
    // the partner group g ^ 1 sits kL lanes away (groups are aligned pairs of
    // 2 kL lanes); its sum and activity feed the paired affine term
    sl.xsp = __shfl_xor_sync(0xffffffffu, sl.xs, 1 << kLg);
    sl.act = active;
    sl.actp = __shfl_xor_sync(0xffffffffu, active ? 1 : 0, 1 << kLg) != 0;
    sl.full = __all_sync(0xffffffffu, active);
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

template <bool kTree, int kLg, class A>
__device__ __forceinline__ void load_slice(const A &a, int ch, int lane, float rms_r, Slice &sl) {
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
    finish_slice<kTree, kLg>(a, ch, lane, active, v, sl);
}

// RMS-norm prologue in one pass over x, for warps that keep one chunk for the
// whole launch: each lane loads its 32 values of x and of the weights once; the
// 64-value block sums of squares come from those registers (the lane's 32
// squares by the pairwise tree, then the partner lane's half: the same tree as
// block_rms_factor's), one warp per chunk posts them (post), and the factor
// scales the values in place.  Every computing warp calls this, idle ones with
// has = false, since it holds the block barriers.
template <bool kTree, int kLg, class A>
__device__ __forceinline__ void rms_slice(const A &a, int ch, bool has, bool post, int cw, int nw, int lane,
                                          float *red, float *rbox, Slice &sl) {
    const int C = a.cols, base = ch * 1024 + lane * 32;
    const bool active = has && base < C;
    float v[32], w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f, w[i] = 0.f;
    if (active) {
        const float4 *x4 = reinterpret_cast<const float4 *>(a.x + base);
        const float4 *w4 = reinterpret_cast<const float4 *>(a.wt + base);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 q = x4[i], u = w4[i];
            v[4 * i] = q.x, v[4 * i + 1] = q.y, v[4 * i + 2] = q.z, v[4 * i + 3] = q.w;
            w[4 * i] = u.x, w[4 * i + 1] = u.y, w[4 * i + 2] = u.z, w[4 * i + 3] = u.w;
        }
    }
    float sq[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) sq[i] = __fmul_rn(v[i], v[i]);
    float s2 = tree32(sq);
    s2 = __fadd_rn(s2, __shfl_xor_sync(0xffffffffu, s2, 1));
    if (post && active && (lane & 1) == 0) red[base >> 6] = s2;
    const float r = rms_from_blocks<kTree>(red, C, a.eps, cw, nw * 32, rbox);
    if (active) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(__fmul_rn(v[i], r), w[i]);
    }
    finish_slice<kTree, kLg>(a, ch, lane, active, v, sl);
}

// The fixed-shape prologue.  The block's computing threads produce the
// activation once, cooperatively, and stage it in shared memory for the
// warps' slices:
//   act  column c = 1024 ch + 32 l + 4 i + e at float index 4 (32 (8 ch + i)
//        + l) + e: lane l of a warp with chunk ch reads its 32 columns with 8
//        conflict-free 16-byte loads;
//   gs   the group sums (computed by the prologue);
//   gneg 1 where every value of the group is negative;
//   spec 1 where a 128-column block holds a value outside the exact path's
//        range (zero of either sign, infinite, NaN or |x| >= 2^100).
// Thread t takes the 4-column units u = t, t + nct, ...; the 16 units of a
// 64-column group are 16 consecutive threads of one half-warp, so a group's
// sum is the thread's pairwise sum of its 4 values followed by butterfly
// steps at distances 1, 2, 4 and 8: the pairwise tree over the 64 values.
// The RMS-norm factor takes the tree over the group sums of squares in
// shared memory between two barriers (rms_from_blocks).  All three sums are
// the oracle's trees, so the staged values are the producers' bits.
template <int kNU>
struct CoopIn {
    float4 w[kNU];  // RMS-norm weights of the thread's units, read before the dependency wait
};

// The RMS-norm factor of a fixed-shape prologue, computed by every warp from
// the group sums of squares in red[0 .. kC/64) (one barrier; no broadcast):
// each lane takes the pairwise tree over its V consecutive group sums (the
// groups padded with -0 to 32 V), then a 5-step butterfly finishes the tree.
// The mean divides by kC; for a power of two that is the exact product with
// 1/kC, the same correctly rounded value.  The factor is the correctly
// rounded reciprocal of the correctly rounded square root.
template <bool kTree, int kC>
__device__ __forceinline__ float rms_factor_all(const float *red, float eps, int nct) {
    constexpr int G = kC / 64;
    constexpr int V = G <= 32 ? 1 : (G <= 64 ? 2 : (G <= 128 ? 4 : 8));
    static_assert(G <= 32 * V, "group sums fit the lanes");
    named_bar(1, nct);
    const int lane = threadIdx.x & 31;
    float t[V];
#pragma unroll
    for (int j = 0; j < V; ++j) t[j] = lane * V + j < G ? red[lane * V + j] : kNegZero;
#pragma unroll
    for (int h = V / 2; h >= 1; h >>= 1)
#pragma unroll
        for (int j = 0; j < h; ++j) t[j] = kTree ? __fadd_rn(t[2 * j], t[2 * j + 1]) : t[2 * j] + t[2 * j + 1];
    float ss = t[0];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, ss, d);
        ss = kTree ? __fadd_rn(ss, o) : ss + o;
    }
    if constexpr (kTree) {
        constexpr bool kPow2 = (kC & (kC - 1)) == 0;
        const float mean = kPow2 ? __fmul_rn(ss, 1.0f / static_cast<float>(kC)) : __fdiv_rn(ss, static_cast<float>(kC));
        return __frcp_rn(__fsqrt_rn(__fadd_rn(mean, eps)));
    } else {
        return rsqrtf(ss / static_cast<float>(kC) + eps);
    }
}

// Group sums of NU units at once: the thread's pairwise sum of a unit's 4
// values, then butterfly steps at distances 1, 2, .. UG/2 over the UG threads
// of the unit's group (the pairwise tree over its 4 UG values: UG = 16 for 64
// values); the steps of the NU units are interleaved so that their shuffles
// overlap.
template <bool kTree, int NU, int UG = 16>
__device__ __forceinline__ void sum4_groups(const float4 (&v)[NU], float (&s)[NU]) {
#pragma unroll
    for (int k = 0; k < NU; ++k)
        s[k] = kTree ? __fadd_rn(__fadd_rn(v[k].x, v[k].y), __fadd_rn(v[k].z, v[k].w))
                     : (v[k].x + v[k].y) + (v[k].z + v[k].w);
#pragma unroll
    for (int d = 1; d < UG; d <<= 1) {
        float o[NU];
#pragma unroll
        for (int k = 0; k < NU; ++k) o[k] = __shfl_xor_sync(0xffffffffu, s[k], d);
#pragma unroll
        for (int k = 0; k < NU; ++k) s[k] = kTree ? __fadd_rn(s[k], o[k]) : s[k] + o[k];
    }
}

template <bool kTree, int UG = 16>
__device__ __forceinline__ float sum4_group(float4 v) {
    float s = kTree ? __fadd_rn(__fadd_rn(v.x, v.y), __fadd_rn(v.z, v.w)) : (v.x + v.y) + (v.z + v.w);
#pragma unroll
    for (int d = 1; d < UG; d <<= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, s, d);
        s = kTree ? __fadd_rn(s, o) : s + o;
    }
    return s;
}

// Stages unit k of a thread (4 columns from c): the block flags, and the
// values in the per-lane layout.  A 128-column block of ordinary values (a
// warp's 32 units) is staged times -2^(23-4k) of its columns' nibbles, the
// exact path's operands; a block with a special value is staged as it is.
// gneg is per group of UG units (the format's group: 32, 64 or 128 columns).
template <int UG>
__device__ __forceinline__ void stage_unit(float4 q, int u, int lane, unsigned bsp, unsigned bneg, float *act,
                                           unsigned *gneg, unsigned *spec) {
    constexpr unsigned kMask = UG == 32 ? 0xffffffffu : (1u << UG) - 1u;
    const int c = 4 * u;
    if (lane == 0) spec[u >> 5] = bsp != 0u;
    if ((u & (UG - 1)) == 0) gneg[u / UG] = ((bneg >> (lane & (32 - UG))) & kMask) == kMask;
    const int ch = c >> 10, l = (c & 1023) >> 5, i = (c & 31) >> 2;
    float4 st = q;
    if (bsp == 0u) {
        const int j0 = c & 4;
        st = make_float4(__fmul_rn(q.x, -nib_scale(j0)), __fmul_rn(q.y, -nib_scale(j0 + 1)),
                         __fmul_rn(q.z, -nib_scale(j0 + 2)), __fmul_rn(q.w, -nib_scale(j0 + 3)));
    }
    reinterpret_cast<float4 *>(act)[(ch * 8 + i) * 32 + l] = st;
}

// kLatency (the few-tiles layout, whose launches are latency-bound): every
// warp computes the RMS-norm factor after one barrier, and the butterflies of
// a thread's units are interleaved.  Otherwise one warp computes the factor
// between two barriers and the units go one after the other (the throughput
// layout's product loop measured faster with this prologue).
template <bool kTree, int kC, int kNct, bool kLatency, int kLg, class A>
__device__ __forceinline__ void coop_prologue(const A &a, const CoopIn<(kC / 4 + kNct - 1) / kNct> &in,
                                              float *act, float *gs, unsigned *gneg, unsigned *spec, int cw,
                                              float *red, float *rbox) {
    constexpr int NU = (kC / 4 + kNct - 1) / kNct;
    constexpr int UG = 8 << kLg;  // units of the format's group (the sums of squares use groups of 64)
    // units per thread: NU, or in a block whose threads do not divide the
    // units, NU - 1 for the threads of the last round's idle warps (whole
    // warps: the units and the threads are multiples of 32)
    constexpr bool kWhole = (kC / 4) % kNct == 0;
    static_assert((kC / 4) % 32 == 0 && kNct % 32 == 0 && (kWhole || !kLatency), "whole warps of units");
    const int t = threadIdx.x - 32, lane = threadIdx.x & 31;
    auto has = [&](int k) { return kWhole || t + k * kNct < kC / 4; };
    const float4 *x4 = reinterpret_cast<const float4 *>(a.x);
    float4 v[NU];
    if (a.prologue == kProSwq) {
        const float4 *u4 = reinterpret_cast<const float4 *>(a.x + kC);
#pragma unroll
        for (int k = 0; k < NU; ++k) {
            v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!has(k)) continue;
            const float4 g = x4[t + k * kNct], u = u4[t + k * kNct];
            v[k] = make_float4(swiglu<kTree>(g.x, u.x), swiglu<kTree>(g.y, u.y), swiglu<kTree>(g.z, u.z),
                               swiglu<kTree>(g.w, u.w));
        }
    } else {
#pragma unroll
        for (int k = 0; k < NU; ++k) v[k] = has(k) ? x4[t + k * kNct] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (a.prologue == kProRmsq) {
        float4 sq[NU];
#pragma unroll
        for (int k = 0; k < NU; ++k)
            sq[k] = make_float4(__fmul_rn(v[k].x, v[k].x), __fmul_rn(v[k].y, v[k].y), __fmul_rn(v[k].z, v[k].z),
                                __fmul_rn(v[k].w, v[k].w));
        float r;
        if constexpr (kLatency) {
            float ss[NU];
            sum4_groups<kTree, NU>(sq, ss);
#pragma unroll
            for (int k = 0; k < NU; ++k) {
                const int u = t + k * kNct;
                if ((u & 15) == 0) red[u >> 4] = ss[k];
            }
            r = rms_factor_all<kTree, kC>(red, a.eps, kNct);
        } else {
#pragma unroll
            for (int k = 0; k < NU; ++k) {
                if (!has(k)) continue;
                const float s = sum4_group<kTree>(sq[k]);
                const int u = t + k * kNct;
                if ((u & 15) == 0) red[u >> 4] = s;
            }
            r = rms_from_blocks<kTree>(red, kC, a.eps, cw, kNct, rbox);
        }
#pragma unroll
        for (int k = 0; k < NU; ++k) {
            if (!has(k)) continue;
            const float4 q = v[k], w = in.w[k];
            v[k] = make_float4(__fmul_rn(__fmul_rn(q.x, r), w.x), __fmul_rn(__fmul_rn(q.y, r), w.y),
                               __fmul_rn(__fmul_rn(q.z, r), w.z), __fmul_rn(__fmul_rn(q.w, r), w.w));
        }
    }
    if constexpr (kLatency) {
        if (a.prologue != kProNone) {
            float gsum[NU];
            sum4_groups<kTree, NU, UG>(v, gsum);
#pragma unroll
            for (int k = 0; k < NU; ++k) {
                const int u = t + k * kNct;
                if ((u & (UG - 1)) == 0) gs[u / UG] = gsum[k];
            }
        }
        unsigned bspk[NU], bnegk[NU];
#pragma unroll
        for (int k = 0; k < NU; ++k) {
            const float4 q = v[k];
            const bool sp = !x_ordinary(q.x) || !x_ordinary(q.y) || !x_ordinary(q.z) || !x_ordinary(q.w);
            const bool neg = q.x < 0.f && q.y < 0.f && q.z < 0.f && q.w < 0.f;
            bspk[k] = __ballot_sync(0xffffffffu, sp);
            bnegk[k] = __ballot_sync(0xffffffffu, neg);
        }
#pragma unroll
        for (int k = 0; k < NU; ++k) stage_unit<UG>(v[k], t + k * kNct, lane, bspk[k], bnegk[k], act, gneg, spec);
    } else {
#pragma unroll
        for (int k = 0; k < NU; ++k) {
            if (!has(k)) continue;
            const int u = t + k * kNct;
            const float4 q = v[k];
            if (a.prologue != kProNone) {
                const float s = sum4_group<kTree, UG>(q);
                if ((u & (UG - 1)) == 0) gs[u / UG] = s;
            }
            const bool sp = !x_ordinary(q.x) || !x_ordinary(q.y) || !x_ordinary(q.z) || !x_ordinary(q.w);
            const bool neg = q.x < 0.f && q.y < 0.f && q.z < 0.f && q.w < 0.f;
            const unsigned bsp = __ballot_sync(0xffffffffu, sp), bneg = __ballot_sync(0xffffffffu, neg);
            stage_unit<UG>(q, u, lane, bsp, bneg, act, gneg, spec);
        }
    }
    named_bar(1, kNct);
}

// A warp's slice of the staged activation (chunk ch; fixed shapes: every
// lane's columns lie inside the row).  Blocks of ordinary values were staged
// as the exact path's operands; on the plain path (a special value somewhere
// in the chunk) a lane whose own 128-column block was scaled takes the
// scaling back, which is exact (ordinary values were scaled up by at least
// 2^7 without overflow).
template <bool kTree, int kLg, class A>
__device__ __forceinline__ void slice_from_stage(const A &a, int ch, int lane, const float *act,
                                                 const float *gs, const unsigned *gneg, const unsigned *spec,
                                                 Slice &sl) {
    float v[32];
    const float4 *s4 = reinterpret_cast<const float4 *>(act);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 q = s4[(ch * 8 + i) * 32 + lane];
        v[4 * i] = q.x, v[4 * i + 1] = q.y, v[4 * i + 2] = q.z, v[4 * i + 3] = q.w;
    }
    const uint4 f0 = reinterpret_cast<const uint4 *>(spec + ch * 8)[0];
    const uint4 f1 = reinterpret_cast<const uint4 *>(spec + ch * 8)[1];
    const bool sp = (f0.x | f0.y | f0.z | f0.w | f1.x | f1.y | f1.z | f1.w) != 0u;
    const int g = ch * (32 >> kLg) + (lane >> kLg);
    sl.exact = !sp;
    sl.xs = a.prologue == kProNone ? a.xsum[g] : gs[g];
    sl.xsp = __shfl_xor_sync(0xffffffffu, sl.xs, 1 << kLg);
    sl.neg = kTree && gneg[g] != 0u;
    sl.anyneg = __any_sync(0xffffffffu, sl.neg);
    sl.act = sl.actp = sl.full = true;
    if (sp && spec[ch * 8 + (lane >> 2)] == 0u) {
#pragma unroll
        for (int m = 0; m < 32; ++m) v[m] = __fmul_rn(v[m], -nib_unscale(m & 7));
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) sl.X[m] = f2(v[m], v[m + 16]);
}

// Locates tiles of a grouped launch.  A block visits its tiles in increasing
// order, so the problem index only moves forward.
// Tile counts fit in 32 bits (the planner checks the launch's total).
struct ProbCursor {
    int p = 0;
    int base = 0;  // first tile of problem p
    template <class A>
    __device__ __forceinline__ int find(const A &a, int t, int &tile) {
        while (p + 1 < a.nprob && t >= base + static_cast<int>(a.prob[p].tiles)) {
            base += static_cast<int>(a.prob[p].tiles);
            ++p;
        }
        tile = t - base;
        return p;
    }
};

// Bounded mbarrier wait that also gives up when another warp has aborted.
// On a timeout it sets the timeout bit plus `site` (which wait gave up).  The
// abort flag and the clock are looked at every 16th poll (a poll suspends the
// warp for at most the sleep hint), which keeps short waits cheap.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              unsigned site) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (unsigned i = 1;; ++i) {
        if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
        if ((i & 15u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                atomicOr(&g_status, kStatusTimeout | site);
                *abort_flag = 1;
                return false;
            }
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

// Values a lane still holds after the butterfly levels at distances D, 2D,
// ... below E, starting from N (each transposed step halves them).
template <int N, int D, int E>
__host__ __device__ constexpr int lv_count() {
    if constexpr (D >= E || N == 1) {
        return N;
    } else {
        return lv_count<N / 2, 2 * D, E>();
    }
}

// Butterfly levels at distances D, 2D, ... below E over N held values: while
// N > 1 each level is a transposed step (the lane keeps the half selected by
// its distance bit, and rowsel records the offset of the rows it keeps);
// then plain butterfly steps.
template <int N, int D, int E, bool kTree>
__device__ __forceinline__ void levels(float (&v)[N], float (&out)[lv_count<N, D, E>()], int lane, int &rowsel) {
    if constexpr (D >= E) {
#pragma unroll
        for (int i = 0; i < N; ++i) out[i] = v[i];
    } else if constexpr (N == 1) {
        float val = v[0];
#pragma unroll
        for (int dd = D; dd < E; dd <<= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, val, dd);
            val = kTree ? __fadd_rn(val, o) : val + o;
        }
        out[0] = val;
    } else {
        const bool hi = (lane & D) != 0;
        tstep<N, kTree>(v, D, hi);
        rowsel += hi ? N / 2 : 0;
        float w[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i) w[i] = v[i];
        levels<N / 2, 2 * D, E, kTree>(w, out, lane, rowsel);
    }
}

// Partial-sum buffers (and their `done` barriers) rotate over S + 2 tiles.
// Only the warps that compute a tile's final sums (threads ct < tile rows)
// wait for every warp's partials of that tile.  The others never wait on
// `done`: a warp reaches tile k only after the producer refilled its stage,
// i.e. after every warp released tile k - S, by which time the finishing
// warps have completed the final sums of tile k - S - 2.  Tiles k - S - 1 .. k
// hold S + 2 distinct buffers, so no buffer is rewritten while still read.
// A launch whose rows fit in one 1024-column chunk writes y directly.

// Block layouts (the register file is split over the SM's four schedulers,
// so the warps per SM set the registers per thread):
//   kLayout 0: up to 8 computing warps, two blocks per SM (96 registers);
//   kLayout 1: up to 16 computing warps, one block per SM;
//   kLayout 2: up to 6 computing warps, two blocks per SM (128 registers);
//   kLayout 4: up to 18 computing warps, one block per SM (rows of 6144
//              columns: three warps per 1024-column chunk).
// With two blocks per SM the next launch of a chain can start beside this one.
constexpr int layout_threads(int l) { return l == 1 ? 544 : (l == 2 ? 224 : (l == 4 ? 608 : 288)); }
constexpr int layout_blocks(int l) { return (l == 1 || l == 4) ? 1 : 2; }
// The launch-bounds thread count: layout 4 declares 21 warps (it launches
// 19) so that the register cap is 96, which keeps the 5 warps of its fullest
// SM sub-partition within the sub-partition's 16K registers.
constexpr int layout_bound_threads(int l) { return l == 4 ? 672 : layout_threads(l); }
// computing warps at most per block
__host__ __device__ constexpr int layout_max_warps(int l) { return l == 1 ? 16 : (l == 4 ? 18 : (l == 2 ? 6 : 8)); }

// Where a tile's results go.  The producer writes the header of a block's
// k-th tile into slot k mod (S + 2) -- the slot of the tile's partial-sum
// buffer -- before it arms the tile's `full` barrier (that arrival releases
// the write; the computing warps' wait on the barrier acquires it).  The slot
// is rewritten for tile k + S + 2 only after every warp has released tile
// k + 2, and a warp reads it at tile k and, for the final sums, before it
// starts tile k + 2.
struct TileHdr {
    float *y;        // output of the tile's first row (a SwiGLU pair: of its gate rows)
    float *y2;       // a SwiGLU pair: output of the tile's first up row
    float *epi;      // a SwiGLU pair: SwiGLU output of the tile's first row
    const void *sc;  // scale and bias of the tile's first row in global memory
    const void *bi;  // (read there when they are not staged)
    int rows;        // rows of the tile (a SwiGLU pair: of each product); fewer at a problem's end
    int pad;
};

// The i-th tile of this block: tiles blockIdx.x, blockIdx.x + gridDim.x, ...
template <class A>
__device__ __forceinline__ int tile_of(const A &, int i) {
    return static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
}
constexpr int kMaxStages = 8;
constexpr int kMaxHdr = kMaxStages + 2;

__host__ __device__ constexpr int log2_rows(int r) { return r >= 8 ? 3 : (r >= 4 ? 2 : (r >= 2 ? 1 : 0)); }

// The lane's row permutation pi: the low log2(R) bits of the lane index,
// reversed.  Item value v[i] holds row (i ^ pi) of its row block, so two lanes
// kL apart (a butterfly level's partners) hold each row in registers whose
// indices differ exactly in the bit that level splits.
template <int kBits>
__device__ __forceinline__ int rev_lane_bits(int lane) {
    int r = 0;
#pragma unroll
    for (int b = 0; b < kBits; ++b) r |= ((lane >> b) & 1) << (kBits - 1 - b);
    return r;
}

// Butterfly levels over lanes at distances D, 2D, ... below E, on N held
// values with the row permutation above: while N > 1 every lane keeps v[i]
// (i < N/2) plus its partner's v[N/2 + i], which is the same row (transposed
// step, no lane-dependent selection); with one value left the remaining
// levels are plain butterfly steps.  Each sum pairs the same two leaves as
// the pairwise tree.
template <int N, int D, int E, bool kTree>
__device__ __forceinline__ void plevels(const float (&v)[N], float (&out)[lv_count<N, D, E>()]) {
    if constexpr (D >= E) {
#pragma unroll
        for (int i = 0; i < N; ++i) out[i] = v[i];
    } else if constexpr (N == 1) {
        float val = v[0];
#pragma unroll
        for (int dd = D; dd < E; dd <<= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, val, dd);
            val = kTree ? __fadd_rn(val, o) : val + o;
        }
        out[0] = val;
    } else {
        float w[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, v[N / 2 + i], D);
            w[i] = kTree ? __fadd_rn(v[i], o) : v[i] + o;
        }
        plevels<N / 2, 2 * D, E, kTree>(w, out);
    }
}

// Tree sum of a row's m chunk partials p[0..m) (m <= 16): the pairwise tree,
// odd element carried, as the tree over the partials padded with -0.
template <bool kTree>
__device__ __forceinline__ float tree_chunks(const float *p, int m) {
    auto add = [](float x, float y) { return kTree ? __fadd_rn(x, y) : x + y; };
    if (m == 2) return add(p[0], p[1]);
    float v[16];
    if (m <= 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = i < m ? p[i] : kNegZero;
        return add(add(v[0], v[1]), add(v[2], v[3]));
    }
    const int n = m <= 8 ? 8 : 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = i < m ? p[i] : kNegZero;
    for (int h = n / 2; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < h) v[i] = add(v[2 * i], v[2 * i + 1]);
    return v[0];
}

// Compile-time tile shape of a product of kC columns in groups of 64 with f32
// scale and bias staged, R rows per item and block layout 0 (at most 8
// computing warps) or 1 (at most 16), following the planner's rule for the
// default tuning: computing warps a multiple of the chunk count, tile rows
// doubled from R times the warps per chunk while a tile stays within one row
// per computing thread and a 40 KB stage.  A launch whose plan has exactly
// this shape may use the kC instantiation, in which the shape's sizes and
// offsets are constants.
__host__ __device__ constexpr int fixed_nch(int C) { return (C + 1023) / 1024; }
__host__ __device__ constexpr int fixed_nw(int C, int layout = 0) {
    return fixed_nch(C) <= layout_max_warps(layout) ? fixed_nch(C) * (layout_max_warps(layout) / fixed_nch(C))
                                                    : layout_max_warps(layout);
}
__host__ __device__ constexpr int fixed_tr(int C, int R, int layout = 0) {
    const int nch = fixed_nch(C), nw = fixed_nw(C, layout), kk = nch <= nw ? nw / nch : 1;
    const int row_bytes = C / 2 + 2 * (C / 64) * 4;
    int tr = R * kk;
    while (tr * 2 <= nw * 32 && tr * 2 * row_bytes <= 40 * 1024) tr *= 2;
    return tr < nw * 32 ? tr : nw * 32;
}

// Pairwise tree over N values (odd element carried), N a compile-time count.
template <int N, bool kTree>
__device__ __forceinline__ float tree_fixed(const float (&v)[N]) {
    if constexpr (N == 1) {
        return v[0];
    } else {
        constexpr int M = (N + 1) / 2;
        float w[M];
#pragma unroll
        for (int i = 0; i < N / 2; ++i) w[i] = kTree ? __fadd_rn(v[2 * i], v[2 * i + 1]) : v[2 * i] + v[2 * i + 1];
        if constexpr (N % 2 == 1) w[M - 1] = v[N - 1];
        return tree_fixed<M, kTree>(w);
    }
}

// The product table of an instantiation: the few-tiles fixed shapes (block
// layout 1 with a compile-time row length, a decode token's launches) take
// kFewProbs products, every other instantiation kMaxProbs.
__host__ __device__ constexpr int kernel_probs(int layout, int c) {
    return layout == 1 && c != 0 ? kFewProbs : kMaxProbs;
}

template <int R, bool kTree, bool kSbSmem, int kLayout, int kLg, bool kHalf, int kC = 0>
__global__ void __launch_bounds__(layout_bound_threads(kLayout), layout_blocks(kLayout))
    q4mv_kernel(const __grid_constant__ Q4ArgsT<kernel_probs(kLayout, kC)> a) {
    static_assert(kC == 0 || (kLayout != 2 && kSbSmem), "fixed shapes: staged scale/bias");
    constexpr bool kFix = kC != 0;
    constexpr int kL = 1 << kLg;                  // lanes per group
    constexpr uint32_t kElem = kHalf ? 2u : 4u;   // bytes per stored scale or bias
    constexpr int kLogR = log2_rows(R);
    // values a lane holds after the group completion (levels below kL) and
    // after the exchange with the partner group (level kL), each then a pair
    constexpr int NA = lv_count<R, 1, kL>();
    constexpr bool kSplitB = NA > 1;
    constexpr int NB = kSplitB ? NA / 2 : 1;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ volatile int s_abort;
    __shared__ float s_red[ABG_MAX_COLS / 64];  // group sums of squares (RMS-norm prologue)
    __shared__ float s_rbox;
    __shared__ TileHdr s_hdr[kMaxHdr];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_bar);
    uint64_t *empty = full + a.stages;
    uint64_t *done = empty + a.stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // shape: constants in a fixed-shape instantiation, else from the plan
    const int S = a.stages;
    constexpr int kTRf = kFix ? fixed_tr(kC, R, kLayout) : 0;
    static_assert(!kFix || kTRf == R * (fixed_nw(kC, kLayout) / fixed_nch(kC)), "one item per warp and tile");
    const int TR = kFix ? kTRf : a.tile_rows, W = kFix ? kC / 8 : a.W, G = kFix ? kC / (32 << kLg) : a.G;
    const int nch = kFix ? fixed_nch(kC) : a.nch, nw = kFix ? fixed_nw(kC, kLayout) : a.nw;
    const uint32_t stage_w_bytes = kFix ? static_cast<uint32_t>(kTRf * kC / 2) : a.stage_w_bytes;
    const uint32_t stage_sb_bytes = kFix ? static_cast<uint32_t>(kTRf * (kC / (32 << kLg))) * kElem : a.stage_sb_bytes;
    const uint32_t stage_bytes = kFix ? stage_w_bytes + 2 * stage_sb_bytes : a.stage_bytes;

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
        const int total = static_cast<int>(a.total_tiles);
        // eph: parity of the empty phase that frees stage s for round k / S,
        // i.e. ((k / S) & 1) ^ 1 (the consumers' release of the round before)
        int k = 0, s = 0, hs = 0;
        const int NP = a.parts;
        uint32_t eph = 1;
        for (int t = tile_of(a, 0); t < total; t = tile_of(a, ++k)) {
            if (a.withhold) break;  // self-test: nothing is copied, nothing is in flight
            if (k == S) {
                grid_dep_wait();
                grid_dep_launch();
                released = true;
            }
            if (k >= S && !wait_or_abort(&empty[s], eph, &s_abort, kSiteEmpty)) break;
            if (s_abort) break;
            int tile = t;
            const int pidx = a.paired ? 0 : cur.find(a, t, tile);
            const Q4Prob &P = a.prob[pidx];
            // a SwiGLU pair's tile: TR/2 rows of the gate product into the
            // stage's first half, the same rows of the up product after them;
            // otherwise the problem's tile rows (at most TR)
            const int trp = a.paired ? TR / 2 : (kFix && kLayout != 1 ? TR : static_cast<int>(P.tr));
            const int64_t r0 = static_cast<int64_t>(tile) * trp;
            const int rows = static_cast<int>(min(static_cast<int64_t>(trp), P.n - r0));
            unsigned char *st = smem + a.off_stage + static_cast<size_t>(s) * stage_bytes;
            const uint32_t wb = static_cast<uint32_t>(rows) * W * 4u;
            const uint32_t sbb = kSbSmem ? static_cast<uint32_t>(rows) * G * kElem : 0u;
            const size_t sbo = static_cast<size_t>(r0) * G * kElem;
            TileHdr &h = s_hdr[hs];
            if (++hs == NP) hs = 0;
            h.y = P.y + r0;
            h.y2 = a.paired ? a.prob[1].y + r0 : nullptr;
            h.epi = a.paired ? a.epi + r0 : nullptr;
            h.sc = static_cast<const unsigned char *>(P.scale) + sbo;
            h.bi = static_cast<const unsigned char *>(P.bias) + sbo;
            h.rows = rows;
            mbar_arrive_expect_tx(&full[s], (a.paired ? 2u : 1u) * (wb + 2 * sbb));
            for (int q = 0; q < (a.paired ? 2 : 1); ++q) {
                const Q4Prob &Q = a.prob[pidx + q];
                const uint32_t hw = q ? static_cast<uint32_t>(trp) * W * 4u : 0u;
                const uint32_t hsb = q ? static_cast<uint32_t>(trp) * G * kElem : 0u;
                bulk_g2s(st + hw, Q.w + r0 * W, wb, &full[s], policy);
                if (kSbSmem) {
                    bulk_g2s(st + stage_w_bytes + hsb, static_cast<const unsigned char *>(Q.scale) + sbo, sbb,
                             &full[s], policy);
                    bulk_g2s(st + stage_w_bytes + stage_sb_bytes + hsb,
                             static_cast<const unsigned char *>(Q.bias) + sbo, sbb, &full[s], policy);
                }
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
        // Drain: the block may not exit while a copy into its shared memory is
        // in flight.  Waiting on a phase that already completed returns at once.
        for (int j = max(0, k - S); j < k; ++j) mbar_wait(&full[j % S], static_cast<uint32_t>((j / S) & 1));
        return;
    }

    // ---------------------------------------------------- consumer warps ----
    const int ct = threadIdx.x - 32, cw = warp - 1;
    float *const part = reinterpret_cast<float *>(smem + a.off_part);
    const unsigned char *const stage0 = smem + a.off_stage;
    // chunk positions and row blocks of this warp
    const bool fixed_ch = nch <= nw;
    const int kk = fixed_ch ? nw / nch : 1;
    const bool idle = fixed_ch && cw >= nch * kk;
    const int ch0 = fixed_ch ? cw % nch : cw;
    const int rb0 = fixed_ch ? cw / nch : 0;
    const int chstep = fixed_ch ? nch : nw;
    const bool direct = nch == 1;  // one chunk per row: y is written by the item

    // fixed shapes: the RMS-norm weights are read before the dependency wait
    // (the preceding launch does not produce them)
    constexpr int kNct = kFix ? 32 * fixed_nw(kC, kLayout) : 32;
    constexpr int kNU = kFix ? (kC / 4 + kNct - 1) / kNct : 1;
    CoopIn<kNU> cin;
    if (kFix && a.prologue == kProRmsq) {
        const float4 *w4 = reinterpret_cast<const float4 *>(a.wt);
#pragma unroll
        for (int k = 0; k < kNU; ++k)
            if ((kC / 4) % kNct == 0 || ct + k * kNct < kC / 4) cin.w[k] = __ldg(w4 + ct + k * kNct);
    }
    Slice sl;
    int cur_ch = -1;
    float rms_r = 0.f;
    if constexpr (!kFix) {
        if (wait_first) {
            grid_dep_wait();
            grid_dep_launch();
        }
        if (a.prologue == kProRmsq) {
            // one pass over x, after which the warp's slice is ready for every
            // tile; only in the main instantiations (tree mode, 8 rows per item,
            // block layout 0, staged scale/bias): in the others the product
            // loop would lose registers to it, so they keep the two passes
            constexpr bool kOnePass = kTree && R == 8 && kLayout == 0 && kSbSmem;
            if (kOnePass && fixed_ch) {
                rms_slice<kTree, kLg>(a, ch0, !idle, rb0 == 0, cw, nw, lane, s_red, &s_rbox, sl);
                if (!idle) cur_ch = ch0;
            } else {
                rms_r = block_rms_factor<kTree>(a.x, a.cols, a.eps, cw, nw, lane, s_red, &s_rbox);
            }
        }
    }
    // Lane constants of the current chunk position (set with its slice):
    // byte offsets in a row block of the item rows' 16-byte column quads,
    // v[i] <- row (i ^ pi), and the lane's and its partner's group.
    // Rows are loaded in batches of B = min(R, 4): batch b's row i is row
    // (4b + i) ^ pi = (i ^ pi) + 4b or - 4b, so one set of B offsets and the
    // batch step serve all batches.
    // (The fixed shapes' few-tiles layout sets them before the dependency
    // wait; the other instantiations wait and compute their prologue before
    // setting them.)
    constexpr int B = R < 4 ? R : 4;
    const int pi = rev_lane_bits<kLogR>(lane);
    const uint32_t rowW = static_cast<uint32_t>(W) * 4u;
    const int bstep = (pi & 4) ? -4 * static_cast<int>(rowW) : 4 * static_cast<int>(rowW);
    uint32_t roff[B];
    // staged scale/bias of the item's affine rows (i ^ pi), i < NB: byte
    // offsets of the lane's own group in a row block, and the step to the
    // partner group
    uint32_t sbo[NB];
    int sbd = 0;
    int gown = 0, gpar = 0;
    // item row j -> stage row (relative to the item's first row): j, or in a
    // SwiGLU pair (R = 4: gate rows 0..R/2-1, then the same up rows in the
    // stage's second half) j < R/2 ? j : TR/2 + j - R/2
    const bool paired = R == 4 && a.paired != 0;
    const int rbm = paired ? R / 2 : R;  // stage rows per item block
    auto srow = [&](int j) -> uint32_t {
        return static_cast<uint32_t>(paired && j >= R / 2 ? TR / 2 + j - R / 2 : j);
    };
    auto set_chunk = [&](int ch) {
        const uint32_t quad = sl.act ? static_cast<uint32_t>(ch * 32 + lane) * 16u : 0u;
#pragma unroll
        for (int i = 0; i < B; ++i) roff[i] = srow(i ^ pi) * rowW + quad;
        // a lane past the row end keeps its group index only to name its
        // partner; its own term is replaced by -0 and reads group 0
        const int gv = ch * (32 >> kLg) + (lane >> kLg);
        gown = sl.act ? gv : 0;
        gpar = sl.actp ? (gv ^ 1) : gown;
#pragma unroll
        for (int i = 0; i < NB; ++i) sbo[i] = (srow(i ^ pi) * G + gown) * kElem;
        sbd = (gpar - gown) * static_cast<int>(kElem);
    };
    if constexpr (kFix) {
        // a fixed shape's lane constants need no activation: the few-tiles
        // layout, bound by latency, sets them before the wait
        sl.act = sl.actp = sl.full = true;
        if constexpr (kLayout == 1) set_chunk(ch0);
        if (wait_first) {
            grid_dep_wait();
            grid_dep_launch();
        }
        // the activation once per block, staged in shared memory
        float *act = reinterpret_cast<float *>(smem + a.off_act);
        float *gs = act + kC;
        unsigned *gneg = reinterpret_cast<unsigned *>(gs + kC / (32 << kLg));
        unsigned *spec = gneg + kC / (32 << kLg);
        coop_prologue<kTree, kC, kNct, kLayout == 1, kLg>(a, cin, act, gs, gneg, spec, cw, s_red, &s_rbox);
        slice_from_stage<kTree, kLg>(a, ch0, lane, act, gs, gneg, spec, sl);
        if constexpr (kLayout != 1) set_chunk(ch0);
        cur_ch = ch0;
    }
    if (!kFix && cur_ch >= 0) set_chunk(cur_ch);  // slice computed by the prologue
    const bool f16 = a.sb_f16 != 0;
    // stored scale or bias i (elements) from the stage or from global memory
    auto sb_at = [&](const void *base, int64_t i) -> float {
        if constexpr (kHalf) {
            const unsigned short h = kSbSmem ? static_cast<const unsigned short *>(base)[i]
                                             : __ldg(static_cast<const unsigned short *>(base) + i);
            return widen16(h, f16);
        } else {
            return kSbSmem ? static_cast<const float *>(base)[i] : __ldg(static_cast<const float *>(base) + i);
        }
    };

    // One item: rows rb*R .. rb*R + R-1 of the tile in the stage at stg, for
    // the lane's 32 columns of chunk ch.  Rows past a ragged tile's end are
    // computed from the stage's stale words and discarded.
    auto item = [&](auto exact_c, auto partial_c, const unsigned char *stg, const TileHdr &h, float *prt, int ch,
                    int rb, bool keep) -> float {
        constexpr bool kExact = decltype(exact_c)::value;
        constexpr bool kPartial = decltype(partial_c)::value;
        const unsigned char *blk = stg + static_cast<uint32_t>(rb * rbm) * rowW;
        float v[R];
#pragma unroll
        for (int b = 0; b < R / B; ++b) {
            const unsigned char *bb = blk + b * bstep;
            uint4 wq[B];
#pragma unroll
            for (int i = 0; i < B; ++i) wq[i] = *reinterpret_cast<const uint4 *>(bb + roff[i]);
#pragma unroll
            for (int i = 0; i < B; ++i) v[B * b + i] = lane_sum32<kExact>(wq[i], sl.X);
        }
        // group completion over the group's kL lanes
        float d[NA];
        plevels<R, 1, kL, kTree>(v, d);
        if (kTree && kExact && sl.anyneg) {
            // The exact path's tree values equal RN's except that a zero is
            // always +0 (q = 0 products are x' - x').  In an all-negative
            // group every product is <= 0, so the sum is zero only when
            // every q is 0, and then RN's products and sum are all -0.
            // Elsewhere a zero sum holds a +0 product or a cancellation: +0
            // either way.
#pragma unroll
            for (int i = 0; i < NA; ++i) d[i] = (sl.neg && d[i] == 0.f) ? kNegZero : d[i];
        }
        // exchange with the partner group (kL lanes away): pairs {own, partner}
        // for rows (i ^ pi), i < NB
        float2 dp[NB];
        if constexpr (kSplitB) {
#pragma unroll
            for (int i = 0; i < NB; ++i) dp[i] = f2(d[i], __shfl_xor_sync(0xffffffffu, d[NB + i], kL));
        } else {
            dp[0] = f2(d[0], __shfl_xor_sync(0xffffffffu, d[0], kL));
        }
        // affine terms of the group pair and their sum (the first level of the
        // groups' tree: t(2j) + t(2j+1), in either order, is the same sum)
        float tv[NB];
        const int rows = h.rows;
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int row = rb * R + (i ^ pi);
            float2 sc, bi;
            if constexpr (kSbSmem) {
                const unsigned char *so = stg + stage_w_bytes + static_cast<uint32_t>(rb * rbm * G) * kElem + sbo[i];
                const unsigned char *sp = so + sbd;
                sc = f2(sb_at(so, 0), sb_at(sp, 0));
                bi = f2(sb_at(so + stage_sb_bytes, 0), sb_at(sp + stage_sb_bytes, 0));
            } else {
                const int64_t e = static_cast<int64_t>(min(row, rows - 1)) * G;
                sc = f2(sb_at(h.sc, e + gown), sb_at(h.sc, e + gpar));
                bi = f2(sb_at(h.bi, e + gown), sb_at(h.bi, e + gpar));
            }
            float2 t2;
            if constexpr (kTree) {
                // scalar RN intrinsics: the compiler fuses a packed multiply
                // into a following packed add, and these must round twice
                t2 = f2(__fadd_rn(__fmul_rn(sc.x, dp[i].x), __fmul_rn(bi.x, sl.xs)),
                        __fadd_rn(__fmul_rn(sc.y, dp[i].y), __fmul_rn(bi.y, sl.xsp)));
            } else {
                t2 = __ffma2_rn(sc, dp[i], __fmul2_rn(bi, f2(sl.xs, sl.xsp)));
            }
            if constexpr (kPartial) {
                // groups past the row end contribute -0
                if (!sl.act) t2.x = kNegZero;
                if (!sl.actp) t2.y = kNegZero;
            }
            tv[i] = kTree ? __fadd_rn(t2.x, t2.y) : t2.x + t2.y;
        }
        // the rest of the chunk's group tree
        float fin[1];
        plevels<NB, 2 * kL, 32, kTree>(tv, fin);
        // lane l < R holds row pi of the block
        if (lane < R && !keep) {
            const int row = rb * R + pi;
            if (direct) {
                if (row < rows) h.y[row] = fin[0];
            } else {
                prt[row * nch + ch] = fin[0];
            }
        }
        return fin[0];
    };

    // Final sums of a finished tile: thread ct adds row ct's chunk partials by
    // the tree (q: the tile's slot, i.e. its partial buffer, header and done
    // barrier; ph: the parity of that barrier's phase).
    auto finish = [&](int q, uint32_t ph) -> bool {
        if (!wait_or_abort(&done[q], ph, &s_abort, kSiteDone)) return false;
        const TileHdr &fh = s_hdr[q];
        if (ct < fh.rows) {
            const float *pr = part + (q * TR + ct) * nch;
            if (nch == 2) {
                const float2 v2 = *reinterpret_cast<const float2 *>(pr);
                fh.y[ct] = kTree ? __fadd_rn(v2.x, v2.y) : v2.x + v2.y;
            } else {
                fh.y[ct] = tree_chunks<kTree>(pr, nch);
            }
        }
        return true;
    };

    const int total = static_cast<int>(a.total_tiles), NP = a.parts;
    const bool finisher = !direct && cw * 32 < TR;  // holds final-sum threads (ct < rows)
    int s = 0, p = 0, pp = -1;
    uint32_t fph = 0, dph = 0, pdph = 0;  // full and done phase parities (current and previous tile)
    if constexpr (kFix) {
        // One item per warp and tile: rows rb0*R .. rb0*R + R-1 of chunk ch0
        // (the tile has R rows per warp of a chunk).  In a tile of fewer rows
        // the items wholly past its end are skipped; a partly filled item's
        // rows past the end are computed from stale words into values that
        // are never written to y.  Warps of chunk 0 keep their chunk totals
        // in a register and, one tile later (once every warp's partials of
        // that tile are in), add the other chunks' partials by the tree and
        // write y for their own rows.  The path (exact or plain) is chosen
        // once: each has its own copy of the loop.
        if (cur_ch != ch0) {
            load_slice<kTree, kLg>(a, ch0, lane, rms_r, sl);
            cur_ch = ch0;
            set_chunk(ch0);
        }
        const bool lead = ch0 == 0;
        const int frow = rb0 * R + pi;  // the row whose final sum this lane writes (lane < R)
        auto final_rows = [&](int q, uint32_t ph, float own) -> bool {
            if (!wait_or_abort(&done[q], ph, &s_abort, kSiteDone)) return false;
            const TileHdr &fh = s_hdr[q];
            float yv = 0.f;
            if (lane < R) {
                const float *pr = part + (q * TR + frow) * nch;
                float c[fixed_nch(kC)];
                c[0] = own;
#pragma unroll
                for (int i = 1; i < fixed_nch(kC); ++i) c[i] = pr[i];
                yv = tree_fixed<fixed_nch(kC), kTree>(c);
            }
            if (paired) {
                // item row j = pi: gate row rb0*R/2 + j (j < R/2) or up row
                // rb0*R/2 + j - R/2; the up value of a gate lane's row sits one
                // lane away (pi reverses the lane bits)
                const float up = __shfl_xor_sync(0xffffffffu, yv, 1);
                const int j = pi, prow = rb0 * (R / 2) + (j & (R / 2 - 1));
                if (lane < R && prow < fh.rows) {
                    if (j < R / 2) {
                        fh.y[prow] = yv;
                        fh.epi[prow] = swiglu<kTree>(yv, up);
                    } else {
                        fh.y2[prow] = yv;
                    }
                }
            } else if (lane < R && frow < fh.rows) {
                fh.y[frow] = yv;
            }
            return true;
        };
        auto run = [&](auto exact_c) {
            float own = 0.f;
            int i = 0;
            for (int t = tile_of(a, 0); t < total; t = tile_of(a, ++i)) {
                if (!wait_or_abort(&full[s], fph, &s_abort, kSiteFull)) break;
                const unsigned char *stg = stage0 + static_cast<uint32_t>(s) * stage_bytes;
                float *prt = part + p * TR * nch;
                // in the few-tiles layout, where the planner cuts quarter
                // tiles (a quarter of the tile is a whole number of items), a
                // tile of fewer rows skips the items wholly past its rows
                constexpr bool kQuarter = kLayout == 1 && kTRf / 4 >= R && (kTRf / 4) % R == 0;
                const float v = (!kQuarter || rb0 * rbm < s_hdr[p].rows)
                                    ? item(exact_c, std::false_type{}, stg, s_hdr[p], prt, ch0, rb0, lead)
                                    : 0.f;
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&empty[s]);
                    mbar_arrive(&done[p]);
                }
                if (lead && pp >= 0 && !final_rows(pp, pdph, own)) break;
                own = v;
                pp = p;
                pdph = dph;
                if (++s == S) {
                    s = 0;
                    fph ^= 1u;
                }
                if (++p == NP) {
                    p = 0;
                    dph ^= 1u;
                }
            }
            if (lead && pp >= 0) final_rows(pp, pdph, own);
        };
        if (sl.exact) {
            run(std::true_type{});
        } else {
            run(std::false_type{});
        }
    } else {
        int ti = 0;
        for (int t = tile_of(a, 0); t < total; t = tile_of(a, ++ti)) {
            if (!wait_or_abort(&full[s], fph, &s_abort, kSiteFull)) break;
            const unsigned char *stg = stage0 + static_cast<uint32_t>(s) * stage_bytes;
            const TileHdr &h = s_hdr[p];
            const int nrb = (h.rows + R - 1) >> kLogR;
            float *prt = part + p * TR * nch;
            if (!idle) {
                for (int ch = ch0; ch < nch; ch += chstep) {
                    if (ch != cur_ch) {
                        load_slice<kTree, kLg>(a, ch, lane, rms_r, sl);
                        cur_ch = ch;
                        set_chunk(ch);
                    }
                    for (int rb = rb0; rb < nrb; rb += kk) {
                        if (sl.exact) {
                            if (sl.full) {
                                item(std::true_type{}, std::false_type{}, stg, h, prt, ch, rb, false);
                            } else {
                                item(std::true_type{}, std::true_type{}, stg, h, prt, ch, rb, false);
                            }
                        } else {
                            item(std::false_type{}, std::true_type{}, stg, h, prt, ch, rb, false);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s]);               // weights of this stage no longer needed
                if (!direct) mbar_arrive(&done[p]);   // this warp's partials are written
            }
            if (finisher && pp >= 0 && !finish(pp, pdph)) break;
            pp = p;
            pdph = dph;
            if (++s == S) {
                s = 0;
                fph ^= 1u;
            }
            if (++p == NP) {
                p = 0;
                dph ^= 1u;
            }
        }
        if (finisher && pp >= 0) finish(pp, pdph);
    }
    if (!wait_first) grid_dep_wait();
}

// Kernel entry for one instantiation, as an untyped pointer.
template <int R, bool kTree, bool kSb, int kLayout, int kLg, bool kHalf, int kC = 0>
void *kernel_ptr() {
    return reinterpret_cast<void *>(&q4mv_kernel<R, kTree, kSb, kLayout, kLg, kHalf, kC>);
}

// Layout-0 instantiations of one format for rows per item 1, 2, 4 or 8.
template <int kLg, bool kHalf>
void *select_layout0(int R, bool tree, bool sb) {
#define ABG_SEL(RR)                                                                                              \
    if (R == RR) {                                                                                               \
        if (tree) return sb ? kernel_ptr<RR, true, true, 0, kLg, kHalf>() : kernel_ptr<RR, true, false, 0, kLg, kHalf>(); \
        return sb ? kernel_ptr<RR, false, true, 0, kLg, kHalf>() : kernel_ptr<RR, false, false, 0, kLg, kHalf>();        \
    }
    ABG_SEL(1)
    ABG_SEL(2)
    ABG_SEL(4)
    ABG_SEL(8)
#undef ABG_SEL
    return nullptr;
}

// This translation unit's device status word (OR-ed into *bits).  Internal
// linkage: every unit that includes this header has its own word.
cudaError_t read_status_word(unsigned *bits, bool clear) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof v);
    if (e == cudaSuccess && clear && v) {
        const unsigned z = 0;
        e = cudaMemcpyToSymbol(g_status, &z, sizeof z);
    }
    *bits |= v;
    return e;
}

}  // namespace

// Defines the kernel selector and status reader of a unit that instantiates
// one format (block layout 0).
#define ABG_Q4MV_FORMAT_UNIT(tag, lg, half)                                                        \
    void *q4mv_select_##tag(int R, bool tree, bool sb) { return select_layout0<lg, half>(R, tree, sb); } \
    cudaError_t q4mv_status_##tag(unsigned *bits, bool clear) { return read_status_word(bits, clear); }

}  // namespace abg
