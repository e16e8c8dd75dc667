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
#include "abg_dev.cuh"
#include "abg_kernels.cuh"

#include <algorithm>
#include <mutex>
#include <set>

namespace abg {

namespace {

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Exponent bits of 2^(23-4k), k = 0..3: the float 2^(23-4k) + q sits in the
// low 23 bits when q occupies bits 4k..4k+3.
__device__ __forceinline__ uint32_t magic_bits(int k) { return static_cast<uint32_t>(150 - 4 * k) << 23; }

// The pair of magic floats for nibble j (0..7) of words a and b.
__device__ __forceinline__ float2 nib2(uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi, int j) {
    const int k = j & 3;
    const uint32_t mask = 0xFu << (4 * k);
    const uint32_t a = (j < 4) ? a_lo : a_hi;
    const uint32_t b = (j < 4) ? b_lo : b_hi;
    return f2(__uint_as_float((a & mask) | magic_bits(k)), __uint_as_float((b & mask) | magic_bits(k)));
}

// Sum over the lane's 32 columns of one row chunk.
//   X[m] = {x(m), x(m+16)}, Cc[m] = {c(m), c(m+16)} for lane-local columns m.
//   kExact: the fused-multiply-add identity (x is ordinary); else convert and multiply.
//   kTree: pairwise tree in column order; else FMA accumulation (fast mode).
template <bool kTree, bool kExact>
__device__ __forceinline__ float lane_sum32(uint4 wq, const float2 (&X)[16], const float2 (&Cc)[16]) {
    const uint32_t w0 = wq.x, w1 = wq.y, w2 = wq.z, w3 = wq.w;
    const uint32_t h0 = w0 >> 16, h1 = w1 >> 16, h2 = w2 >> 16, h3 = w3 >> 16;
    if (kTree) {
        float2 P[16];
        if (kExact) {
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float2 v = (m < 8) ? nib2(w0, h0, w2, h2, m & 7) : nib2(w1, h1, w3, h3, m & 7);
                P[m] = fma2(v, X[m], Cc[m]);
            }
            // P[m] = {p_m, p_(m+16)}: adding P[2i] and P[2i+1] pairs leaves (2i, 2i+1)
            // in both halves; the halves stay aligned level after level.
#pragma unroll
            for (int i = 0; i < 8; ++i) P[i] = add2(P[2 * i], P[2 * i + 1]);
        } else {
            // Plain path: q converted exactly, products and the first tree level
            // as scalar RN operations.  (The compiler may fuse a packed multiply
            // or a packed fma with a -0 addend into the packed add after it; the
            // scalar __fmul_rn / __fadd_rn intrinsics are never contracted.)
            float p[32];
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float2 v = (m < 8) ? nib2(w0, h0, w2, h2, m & 7) : nib2(w1, h1, w3, h3, m & 7);
                const float e = -__uint_as_float(magic_bits(m & 3));
                p[m] = __fmul_rn(__fadd_rn(v.x, e), X[m].x);
                p[m + 16] = __fmul_rn(__fadd_rn(v.y, e), X[m].y);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
                P[i] = f2(__fadd_rn(p[2 * i], p[2 * i + 1]), __fadd_rn(p[16 + 2 * i], p[17 + 2 * i]));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) P[i] = add2(P[2 * i], P[2 * i + 1]);
#pragma unroll
        for (int i = 0; i < 2; ++i) P[i] = add2(P[2 * i], P[2 * i + 1]);
        P[0] = add2(P[0], P[1]);
        return __fadd_rn(P[0].x, P[0].y);
    } else {
        float2 acc[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float2 v = (m < 8) ? nib2(w0, h0, w2, h2, m & 7) : nib2(w1, h1, w3, h3, m & 7);
            const float e = -__uint_as_float(magic_bits(m & 3));
            acc[m & 3] = fma2(add2(v, f2(e, e)), X[m], acc[m & 3]);
        }
        const float2 s = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
        return s.x + s.y;
    }
}

// Location of column `col` in the staged activation: chunk ch = col/1024, lane
// L = (col/32)%32, lane-local m = col%32.  Quad i (0..7) of (ch, L) holds
// {x(2i), x(2i+16), x(2i+1), x(2i+17)} so one 16-byte load gives X[2i], X[2i+1]
// and consecutive lanes read consecutive 16-byte words.
__device__ __forceinline__ int xc_index(int col) {
    const int ch = col >> 10, L = (col >> 5) & 31, m = col & 31;
    const int half = m >> 4, mm = m & 15;
    const int quad = ((ch * 8 + (mm >> 1)) * 32 + L);
    return quad * 4 + (((mm & 1) << 1) | half);
}

// True when the fused-multiply-add identity gives RN(q*x) for this x.
__device__ __forceinline__ bool x_ordinary(float v) {
    const uint32_t b = __float_as_uint(v);
    return fabsf(v) < 1.2676506e30f /* 2^100 */ && b != 0x80000000u;
}

struct Staging {
    float *xc;   // activation quads
    float *xs;   // group sums [G]
    float *red;  // reduction scratch [next_pow2(G)]
    int *flags;  // [0] = some x is not ordinary, [1] = rms factor bits
};

// Emits the activation pair (v0, v1) at columns (col, col+1) and returns its
// contribution to the special-value flag.
__device__ __forceinline__ int emit_x(const Staging &st, int col, float v0, float v1) {
    st.xc[xc_index(col)] = v0;
    st.xc[xc_index(col + 1)] = v1;
    return (x_ordinary(v0) && x_ordinary(v1)) ? 0 : 1;
}

// Stages (or computes) the activation for a product block.  Runs on the
// consumer threads only (ct = consumer thread index, nct threads, ncw warps);
// ends with those threads synchronized on named barrier 1.
template <bool kTree>
__device__ void stage_activation(const Q4Args &a, const Staging &st, int ct, int nct) {
    const int cw = ct >> 5, lane = ct & 31, ncw = nct >> 5;
    const int C = a.cols, G = a.G;
    int special = 0;
    if (ct == 0) st.flags[0] = 0;
    named_bar(1, nct);
    if (a.prologue == kProNone) {
        for (int p = ct; p < C / 2; p += nct) {
            const float2 v = reinterpret_cast<const float2 *>(a.x)[p];
            special |= emit_x(st, 2 * p, v.x, v.y);
        }
        for (int g = ct; g < G; g += nct) st.xs[g] = a.xsum[g];
    } else if (a.prologue == kProGsum || a.prologue == kProSwq) {
        for (int g = cw; g < G; g += ncw) {
            const int col = 64 * g + 2 * lane;
            float v0, v1;
            if (a.prologue == kProGsum) {
                const float2 v = reinterpret_cast<const float2 *>(a.x)[col / 2];
                v0 = v.x, v1 = v.y;
            } else {
                const float2 gg = reinterpret_cast<const float2 *>(a.x)[col / 2];
                const float2 uu = reinterpret_cast<const float2 *>(a.x + C)[col / 2];
                v0 = swiglu<kTree>(gg.x, uu.x);
                v1 = swiglu<kTree>(gg.y, uu.y);
            }
            special |= emit_x(st, col, v0, v1);
            const float s = warp_tree<32>(kTree ? __fadd_rn(v0, v1) : v0 + v1);
            if (lane == 0) st.xs[g] = s;
        }
    } else {  // kProRmsq
        for (int g = cw; g < G; g += ncw) {
            const float2 v = reinterpret_cast<const float2 *>(a.x)[32 * g + lane];
            const float s = warp_tree<32>(__fadd_rn(__fmul_rn(v.x, v.x), __fmul_rn(v.y, v.y)));
            if (lane == 0) st.red[g] = s;
        }
        named_bar(1, nct);
        if (cw == 0) {
            const float ss = warp_tree_smem(st.red, G);
            if (lane == 0) {
                float r;
                if (kTree) {
                    const float mean = __fdiv_rn(ss, static_cast<float>(C));
                    r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.eps)));
                } else {
                    r = rsqrtf(ss / static_cast<float>(C) + a.eps);
                }
                st.flags[1] = __float_as_int(r);
            }
        }
        named_bar(1, nct);
        const float r = __int_as_float(st.flags[1]);
        for (int g = cw; g < G; g += ncw) {
            const float2 v = reinterpret_cast<const float2 *>(a.x)[32 * g + lane];
            const float2 wt = reinterpret_cast<const float2 *>(a.wt)[32 * g + lane];
            const float v0 = __fmul_rn(__fmul_rn(v.x, r), wt.x);
            const float v1 = __fmul_rn(__fmul_rn(v.y, r), wt.y);
            special |= emit_x(st, 64 * g + 2 * lane, v0, v1);
            const float s = warp_tree<32>(kTree ? __fadd_rn(v0, v1) : v0 + v1);
            if (lane == 0) st.xs[g] = s;
        }
    }
    if (special) atomicOr(st.flags, 1);
    named_bar(1, nct);
}

// Locates tile t of a grouped launch.
__device__ __forceinline__ int find_prob(const Q4Args &a, int64_t t, int64_t &tile) {
    int p = 0;
    while (p + 1 < a.nprob && t >= a.prob[p].tiles) {
        t -= a.prob[p].tiles;
        ++p;
    }
    tile = t;
    return p;
}

// Bounded mbarrier wait that also gives up when another warp has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (unsigned spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 255u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                atomicOr(&g_status, kStatusTimeout);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

template <int R, bool kTree, bool kSbSmem>
__global__ void __launch_bounds__(416, 1) q4mv_kernel(const __grid_constant__ Q4Args a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_flags[2];
    __shared__ volatile int s_abort;
    float4 *xc4 = reinterpret_cast<float4 *>(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_bar);
    uint64_t *empty = full + a.stages;
    uint64_t *done = empty + a.stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.stages, TR = a.tile_rows, W = a.W, G = a.G, nch = a.nch;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], a.nw);
            mbar_init(&done[s], a.nw);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dep_launch();

    if (warp == 0) {
        // ------------------------------------------------ producer warp ----
        if (lane != 0) return;
        const uint64_t policy = l2_evict_first();
        int64_t k = 0;
        for (int64_t t = blockIdx.x; t < a.total_tiles; t += gridDim.x, ++k) {
            const int s = static_cast<int>(k % S);
            if (k >= S && !wait_or_abort(&empty[s], static_cast<uint32_t>(((k / S) & 1) ^ 1), &s_abort)) break;
            if (s_abort) break;
            int64_t tile;
            const Q4Prob &P = a.prob[find_prob(a, t, tile)];
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
        // Drain: the CTA may not exit while a copy into its shared memory is in
        // flight.  Waiting on a phase that already completed returns at once.
        for (int64_t j = max(static_cast<int64_t>(0), k - S); j < k; ++j)
            mbar_wait(&full[j % S], static_cast<uint32_t>((j / S) & 1));
        return;
    }

    // ---------------------------------------------------- consumer warps ----
    const int ct = threadIdx.x - 32, nct = a.nw * 32, cw = warp - 1;
    grid_dep_wait();
    Staging st;
    st.xc = reinterpret_cast<float *>(smem);
    st.xs = reinterpret_cast<float *>(smem + a.off_xs);
    st.red = reinterpret_cast<float *>(smem + a.off_red);
    st.flags = s_flags;
    stage_activation<kTree>(a, st, ct, nct);
    const bool exact = (s_flags[0] == 0);
    const float *xs = st.xs;
    float *part = reinterpret_cast<float *>(smem + a.off_part);

    float2 X[16], Cc[16];
    float xsg = 0.f;
    int cur_ch = -1;
    int64_t k = 0;
    for (int64_t t = blockIdx.x; t < a.total_tiles; t += gridDim.x, ++k) {
        const int s = static_cast<int>(k % S);
        const uint32_t ph = static_cast<uint32_t>((k / S) & 1);
        if (!wait_or_abort(&full[s], ph, &s_abort)) return;
        int64_t tile;
        const Q4Prob &P = a.prob[find_prob(a, t, tile)];
        const int64_t r0 = tile * TR;
        const int rows = static_cast<int>(min(static_cast<int64_t>(TR), P.n - r0));
        const unsigned char *stg = smem + a.off_stage + static_cast<size_t>(s) * a.stage_bytes;
        const uint4 *sw = reinterpret_cast<const uint4 *>(stg);
        const float *ssc = reinterpret_cast<const float *>(stg + a.stage_w_bytes);
        const float *sbi = reinterpret_cast<const float *>(stg + a.stage_w_bytes + a.stage_sb_bytes);
        float *prt = part + static_cast<size_t>(s) * TR * nch;
        const int nrb = (rows + R - 1) / R;
        const int items = nrb * nch;
        for (int item = cw; item < items; item += a.nw) {
            const int ch = item % nch, rb = item / nch;
            const bool active = (ch * 1024 + lane * 32) < a.cols;
            const int g = ch * 16 + (lane >> 1);
            if (ch != cur_ch) {
                cur_ch = ch;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 q = xc4[(ch * 8 + i) * 32 + lane];
                    X[2 * i] = f2(q.x, q.y);
                    X[2 * i + 1] = f2(q.z, q.w);
                }
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float e = -__uint_as_float(magic_bits(m & 3));
                    Cc[m] = f2(__fmul_rn(X[m].x, e), __fmul_rn(X[m].y, e));
                }
                xsg = active ? xs[g] : 0.f;
            }
            // Lanes past the end of the row (last chunk only) come in whole
            // groups (lane pairs); they contribute -0 to the group butterfly.
            float tv[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int row = rb * R + r;  // uniform across the warp
                tv[r] = kNegZero;
                if (row < rows) {
                    float part32 = 0.f, sc = 0.f, bi = 0.f;
                    if (active) {
                        const uint4 wq = sw[static_cast<size_t>(row) * (W / 4) + ch * 32 + lane];
                        part32 = exact ? lane_sum32<kTree, true>(wq, X, Cc) : lane_sum32<kTree, false>(wq, X, Cc);
                        if (kSbSmem) {
                            sc = ssc[row * G + g];
                            bi = sbi[row * G + g];
                        } else {
                            sc = __ldg(P.scale + (r0 + row) * G + g);
                            bi = __ldg(P.bias + (r0 + row) * G + g);
                        }
                    }
                    const float o = __shfl_xor_sync(0xffffffffu, part32, 1);
                    if (active) {
                        if (kTree) {
                            const float d = __fadd_rn(part32, o);
                            tv[r] = __fadd_rn(__fmul_rn(sc, d), __fmul_rn(bi, xsg));
                        } else {
                            tv[r] = fmaf(sc, part32 + o, bi * xsg);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float v = tv[r];
#pragma unroll
                for (int d = 2; d < 32; d <<= 1) {
                    const float o = __shfl_xor_sync(0xffffffffu, v, d);
                    v = kTree ? __fadd_rn(v, o) : v + o;
                }
                const int row = rb * R + r;
                if (lane == 0 && row < rows) prt[row * nch + ch] = v;
            }
        }
        // all chunk partials of the tile are in shared memory
        __syncwarp();
        if (lane == 0) mbar_arrive(&done[s]);
        if (!wait_or_abort(&done[s], ph, &s_abort)) return;
        if (ct < rows) {
            float *pr = prt + ct * nch;
            int m = nch;
            while (m > 1) {
                const int h = m >> 1;
                for (int i = 0; i < h; ++i) pr[i] = kTree ? __fadd_rn(pr[2 * i], pr[2 * i + 1]) : pr[2 * i] + pr[2 * i + 1];
                if (m & 1) pr[h] = pr[m - 1];
                m = h + (m & 1);
            }
            P.y[r0 + ct] = pr[0];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

template <int R, bool kTree, bool kSb>
void *kernel_ptr() {
    return reinterpret_cast<void *>(&q4mv_kernel<R, kTree, kSb>);
}

void *select_kernel(int R, bool tree, bool sb) {
#define ABG_SEL(RR)                                                                            \
    if (R == RR) {                                                                             \
        if (tree) return sb ? kernel_ptr<RR, true, true>() : kernel_ptr<RR, true, false>();    \
        return sb ? kernel_ptr<RR, false, true>() : kernel_ptr<RR, false, false>();            \
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
    int nw = tune.consumer_warps;
    if (nw <= 0) nw = nch <= 8 ? std::min(12, nch * ((8 + nch - 1) / nch)) : 8;
    nw = std::min(std::max(nw, 1), 12);
    const int kk = (nw % nch == 0) ? nw / nch : 1;  // warps per chunk position
    const uint32_t row_bytes = static_cast<uint32_t>(C / 2 + (sb_smem ? 8 * G : 0));
    int gp = 1;
    while (gp < G) gp <<= 1;
    const uint32_t xc_bytes = static_cast<uint32_t>(nch) * 8u * 32u * 16u;
    const uint32_t xs_bytes = align_up(static_cast<uint32_t>(G) * 4u, 16);
    const uint32_t red_bytes = align_up(static_cast<uint32_t>(std::max(gp, 32)) * 4u, 16);
    const uint32_t fixed = xc_bytes + xs_bytes + red_bytes + 1024;  // + barriers and slack
    uint32_t budget = static_cast<uint32_t>(tune.smem_kb > 0 ? tune.smem_kb : 110) * 1024u;
    const uint32_t hard_max = 227u * 1024u;
    // tile rows: a multiple of R*kk so items spread evenly over the warps
    const int unit = R * kk;
    int TR = unit;
    const uint32_t stage_target = 48u * 1024u;
    while (TR * 2 <= nw * 32 && (TR * 2) * row_bytes <= stage_target) TR *= 2;
    TR = std::min(TR, nw * 32);
    if (TR < R) return false;
    auto stage_bytes = [&](int tr) {
        return align_up(static_cast<uint32_t>(tr) * (C / 2), 16) +
               2u * align_up(sb_smem ? static_cast<uint32_t>(tr) * G * 4u : 0u, 16);
    };
    auto part_bytes = [&](int tr, int s) { return align_up(static_cast<uint32_t>(s * tr * nch) * 4u, 16); };
    int S = 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
        for (;;) {
            const uint32_t sb = stage_bytes(TR);
            S = 0;
            while (S < 8 && fixed + (S + 1) * sb + part_bytes(TR, S + 1) + 24u * (S + 1) <= budget) ++S;
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
    a.cols = C;
    a.W = W;
    a.G = G;
    a.nch = nch;
    a.tile_rows = TR;
    a.stages = S;
    a.nw = nw;
    a.off_xs = xc_bytes;
    a.off_red = a.off_xs + xs_bytes;
    a.off_stage = align_up(a.off_red + red_bytes, 128);
    a.stage_w_bytes = align_up(static_cast<uint32_t>(TR) * (C / 2), 16);
    a.stage_sb_bytes = align_up(sb_smem ? static_cast<uint32_t>(TR) * G * 4u : 0u, 16);
    a.stage_bytes = a.stage_w_bytes + 2 * a.stage_sb_bytes;
    a.off_part = a.off_stage + S * a.stage_bytes;
    a.off_bar = align_up(a.off_part + part_bytes(TR, S), 16);
    a.smem_bytes = a.off_bar + 24u * S;

    // blocks per SM: what fits (registers and shared memory), at most 2 unless tuned
    int fit = 1;
    void *fn = select_kernel(R, tree, sb_smem);
    if (fn && raise_smem_limit(fn) == cudaSuccess) {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, static_cast<int>(32 * (1 + nw)), a.smem_bytes) ==
                cudaSuccess &&
            nb > 0)
            fit = nb;
    }
    cudaGetLastError();
    int bps = std::min(fit, tune.blocks_per_sm > 0 ? tune.blocks_per_sm : 2);
    bps = std::max(bps, 1);
    const int64_t cap = static_cast<int64_t>(sm_count()) * bps;
    plan->grid = dim3(static_cast<unsigned>(std::max<int64_t>(1, std::min(a.total_tiles, cap))));
    plan->block = dim3(32u * (1 + nw));
    plan->rows_per_warp = R;
    plan->tree = tree;
    plan->sb_smem = sb_smem;
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
    void *fn = select_kernel(plan.rows_per_warp, plan.tree, plan.sb_smem);
    if (!fn) return cudaErrorInvalidValue;
    return raise_smem_limit(fn);
}

cudaError_t launch_q4mv(const Q4Plan &plan, cudaStream_t stream, bool pdl) {
    if (plan.args.total_tiles == 0) return cudaSuccess;
    void *fn = select_kernel(plan.rows_per_warp, plan.tree, plan.sb_smem);
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
