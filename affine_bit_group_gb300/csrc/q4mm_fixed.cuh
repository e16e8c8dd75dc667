// Fixed-shape batched product: a pair of tokens (T = 2) sharing the weights,
// rows of 2048 or 4096 columns in groups of 64 with f32 scale and bias staged
// in shared memory.  Each token's output equals its single-token product bit
// for bit.
//
// The lane mapping is the pair kernel's (q4mm_kernel.cuh): a lane covers 16
// columns, so the two tokens' activation slices fit in 32 registers, a warp's
// chunk is 512 columns and a 64-column group spans 4 lanes.  What changes is
// the item (4 rows x 2 tokens = 8 values per lane) and the loop:
//   - value v[2r + t] of a lane holds the (row, token) index (2r + t) ^ pi,
//     pi the lane's low 3 bits reversed: the row part comes from the order in
//     which the lane loads its rows, the token part from the order in which it
//     keeps the two tokens' activation registers.  Every transposed butterfly
//     step is then the same shuffle-and-add in every lane (no selects), as in
//     the single-token kernel;
//   - the group completion (2 levels over the group's 4 lanes) leaves 2
//     values; the exchange with the partner group (4 lanes away) leaves one
//     pair {own group, partner group}, whose two affine terms and their sum
//     are the first level of the groups' tree;
//   - the tile shape and shared-memory offsets are compile-time constants,
//     each warp takes 4 items per tile, and the chunk-0 warps write the final
//     sums of their own rows one tile later.
//
// A second kernel takes four tokens (T = 4) on rows of 2048 columns: a lane
// covers 8 columns (one word, unpacked once for four tokens), a 64-column
// group spans 8 lanes and a warp's chunk 256 columns, so the 8 computing
// warps own one chunk each and take every row block of a tile.  Value
// v[4r + t] holds (row, token) index (4r + t) ^ pi, pi the lane's low 4 bits
// reversed: the row bits from the lane's row order, the token bits from a
// per-lane XOR permutation of the four activation slices.  Three transposed
// steps complete a group, the exchange with the partner group (8 lanes away)
// leaves one pair of affine terms, and the step at 16 lanes finishes the
// chunk.  Each warp writes the final sums of an eighth of the tile's rows
// one tile later.
#pragma once

#include "q4mm_kernel.cuh"

namespace abg {

namespace {

__host__ __device__ constexpr int mmf_nch(int C) { return C / 512; }
__host__ __device__ constexpr int mmf_kk(int C) { return 8 / mmf_nch(C); }
__host__ __device__ constexpr int mmf_tr(int C) { return C == 2048 ? 32 : 16; }  // the pair planner's tile rows
constexpr int kMmfItems = 4;  // items per warp and tile

template <bool kTree, int kC>
__global__ void __launch_bounds__(288, 2) q4mm_fixed_kernel(const __grid_constant__ Q4ArgsT<kMmProbs> a) {
    constexpr int T = 2, R = 4, LC = 16, kL = 4, GPC = 8;
    constexpr int W = kC / 8, G = kC / 64, NCH = mmf_nch(kC), NW = 8, KK = mmf_kk(kC), TR = mmf_tr(kC);
    static_assert(TR == R * KK * kMmfItems, "4 items per warp and tile");
    constexpr uint32_t kStageW = TR * W * 4, kStageSb = TR * G * 4, kStage = kStageW + 2 * kStageSb;
    constexpr uint32_t kRowW = W * 4;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ volatile int s_abort;
    __shared__ TileHdr s_hdr[kMaxHdr];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_bar);
    uint64_t *empty = full + a.stages;
    uint64_t *done = empty + a.stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.stages, NP = a.parts;
    const int total = static_cast<int>(a.total_tiles);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        for (int i = 0; i < NP; ++i) mbar_init(&done[i], NW);
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
        int k = 0, s = 0, hs = 0;
        uint32_t eph = 1;
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
            unsigned char *st = smem + a.off_stage + static_cast<size_t>(s) * kStage;
            const uint32_t wb = static_cast<uint32_t>(rows) * kRowW, sbb = static_cast<uint32_t>(rows) * G * 4u;
            const size_t sbo = static_cast<size_t>(r0) * G * 4u;
            TileHdr &h = s_hdr[hs];
            if (++hs == NP) hs = 0;
            h.y = P.y + r0;
            h.y2 = nullptr;
            h.epi = nullptr;
            h.sc = nullptr;
            h.bi = nullptr;
            h.rows = rows;
            h.pad = static_cast<int>(P.n);  // stride between the tokens' outputs
            mbar_arrive_expect_tx(&full[s], wb + 2 * sbb);
            bulk_g2s(st, P.w + r0 * W, wb, &full[s], policy);
            bulk_g2s(st + kStageW, static_cast<const unsigned char *>(P.scale) + sbo, sbb, &full[s], policy);
            bulk_g2s(st + kStageW + kStageSb, static_cast<const unsigned char *>(P.bias) + sbo, sbb, &full[s], policy);
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
    const int cw = warp - 1;
    float *const part = reinterpret_cast<float *>(smem + a.off_part);
    const unsigned char *const stage0 = smem + a.off_stage;
    const int ch0 = cw % NCH, rb0 = cw / NCH;
    const bool lead = ch0 == 0;
    const int ntok = a.ntok;
    if (wait_first) {
        grid_dep_wait();
        grid_dep_launch();
    }
    MSlice<T, LC> sl;
    load_mslice<T, LC, kTree>(a, ch0, lane, sl);
    // pi = the lane's low 3 bits reversed; value v[2r + t] holds (row, token)
    // index (2r + t) ^ pi: rows loaded in the order r ^ (pi >> 1), the two
    // tokens' activation registers swapped when pi & 1
    const int pi = ((lane & 1) << 2) | (lane & 2) | ((lane >> 2) & 1);
    const int rp = pi >> 1, tsw = pi & 1;
    if (tsw) {
#pragma unroll
        for (int m = 0; m < LC / 2; ++m) {
            const float2 q = sl.X[0][m];
            sl.X[0][m] = sl.X[1][m];
            sl.X[1][m] = q;
        }
    }
    // the lane's final value: row rb*R + rp, token tsw (lanes 0..7)
    const int g = ch0 * GPC + lane / kL;
    // the pair's token is tsw in this lane and tsw ^ 1 in the partner lane
    // (kL lanes away): the partner sends its group sum of token tsw
    const float xs_own = tsw ? sl.xs[1] : sl.xs[0];
    const float xs_par = __shfl_xor_sync(0xffffffffu, tsw ? sl.xs[0] : sl.xs[1], kL);
    // group completion leaves d[i] = (row, token) index i ^ pi: token i ^ tsw
    const bool neg0 = kTree && ((sl.negs >> tsw) & 1), neg1 = kTree && ((sl.negs >> (tsw ^ 1)) & 1);
    const uint32_t quad = static_cast<uint32_t>(ch0 * 64 + lane * 2) * 4u;  // the lane's 2 words in a row
    uint32_t roff[R];
#pragma unroll
    for (int r = 0; r < R; ++r) roff[r] = static_cast<uint32_t>(r ^ rp) * kRowW + quad;
    const uint32_t sbo = (static_cast<uint32_t>(rp) * G + g) * 4u;  // the pair's own scale, relative to its item
    const int sbd = ((g ^ 1) - g) * 4;

    auto item = [&](auto exact_c, const unsigned char *stg, float *prt, int rb) -> float {
        constexpr bool kExact = decltype(exact_c)::value;
        const unsigned char *blk = stg + static_cast<uint32_t>(rb * R) * kRowW;
        float v[R * T];
        uint2 wq[R];
#pragma unroll
        for (int r = 0; r < R; ++r) wq[r] = *reinterpret_cast<const uint2 *>(blk + roff[r]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t w[2] = {wq[r].x, wq[r].y};
            lane_sums<T, LC, kExact>(w, sl, v + r * T);
        }
        float d[2];
        plevels<R * T, 1, kL, kTree>(v, d);
        if (kTree && kExact && sl.anyneg) {
            // zero sums are +0 on the exact path; in an all-negative group a
            // zero sum means every q is 0, and RN's sum is -0
            d[0] = (neg0 && d[0] == 0.f) ? kNegZero : d[0];
            d[1] = (neg1 && d[1] == 0.f) ? kNegZero : d[1];
        }
        // the pair {own group, partner group} of (row, token) index pi
        const float dpar = __shfl_xor_sync(0xffffffffu, d[1], kL);
        const unsigned char *so = stg + kStageW + static_cast<uint32_t>(rb * R * G) * 4u + sbo;
        const unsigned char *sp = so + sbd;
        const float sco = *reinterpret_cast<const float *>(so), scp = *reinterpret_cast<const float *>(sp);
        const float bio = *reinterpret_cast<const float *>(so + kStageSb);
        const float bip = *reinterpret_cast<const float *>(sp + kStageSb);
        float t0, t1;
        if constexpr (kTree) {
            t0 = __fadd_rn(__fmul_rn(sco, d[0]), __fmul_rn(bio, xs_own));
            t1 = __fadd_rn(__fmul_rn(scp, dpar), __fmul_rn(bip, xs_par));
        } else {
            t0 = fmaf(sco, d[0], bio * xs_own);
            t1 = fmaf(scp, dpar, bip * xs_par);
        }
        float tv[1] = {kTree ? __fadd_rn(t0, t1) : t0 + t1};
        float fin[1];
        plevels<1, 2 * kL, 32, kTree>(tv, fin);
        if (lane < R * T && !lead) prt[((rb * R + rp) * NCH + ch0) * T + tsw] = fin[0];
        return fin[0];
    };

    // chunk-0 warps: final sums of the previous tile's rows of this warp
    auto final_rows = [&](int q, uint32_t ph, const float (&own)[kMmfItems]) -> bool {
        if (!wait_or_abort(&done[q], ph, &s_abort, kSiteDone)) return false;
        if (lane < R * T) {
            const TileHdr &fh = s_hdr[q];
            const float *pq = part + q * TR * NCH * T;
#pragma unroll
            for (int j = 0; j < kMmfItems; ++j) {
                const int row = (rb0 + j * KK) * R + rp;
                float c[NCH];
                c[0] = own[j];
#pragma unroll
                for (int i = 1; i < NCH; ++i) c[i] = pq[(row * NCH + i) * T + tsw];
                const float yv = tree_fixed<NCH, kTree>(c);
                if (row < fh.rows && tsw < ntok) fh.y[static_cast<int64_t>(tsw) * fh.pad + row] = yv;
            }
        }
        return true;
    };

    auto run = [&](auto exact_c) {
        int s = 0, p = 0, pp = -1;
        uint32_t fph = 0, dph = 0, pdph = 0;
        float own[kMmfItems], pown[kMmfItems];
#pragma unroll
        for (int j = 0; j < kMmfItems; ++j) own[j] = pown[j] = 0.f;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            if (!wait_or_abort(&full[s], fph, &s_abort, kSiteFull)) break;
            const unsigned char *stg = stage0 + static_cast<uint32_t>(s) * kStage;
            float *prt = part + p * TR * NCH * T;
#pragma unroll
            for (int j = 0; j < kMmfItems; ++j) own[j] = item(exact_c, stg, prt, rb0 + j * KK);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s]);
                mbar_arrive(&done[p]);
            }
            if (lead && pp >= 0 && !final_rows(pp, pdph, pown)) break;
#pragma unroll
            for (int j = 0; j < kMmfItems; ++j) pown[j] = own[j];
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
        if (lead && pp >= 0) final_rows(pp, pdph, pown);
    };
    if (sl.exact) {
        run(std::true_type{});
    } else {
        run(std::false_type{});
    }
    if (!wait_first) grid_dep_wait();
}


// ---------------------------------------------------------------- T = 4 ----
constexpr int kMm4Cols = 2048;
constexpr int kMm4Rows = 32;  // tile rows (8 items of 4 rows per warp)

template <bool kTree>
__global__ void __launch_bounds__(288, 2) q4mm4_fixed_kernel(const __grid_constant__ Q4ArgsT<kMmProbs> a) {
    constexpr int T = 4, R = 4, LC = 8, kL = 8, GPC = 4, kC = kMm4Cols;
    constexpr int W = kC / 8, G = kC / 64, NCH = kC / 256, NW = 8, TR = kMm4Rows, NI = TR / R;
    static_assert(NCH == NW, "one chunk per computing warp");
    constexpr uint32_t kStageW = TR * W * 4, kStageSb = TR * G * 4, kStage = kStageW + 2 * kStageSb;
    constexpr uint32_t kRowW = W * 4;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ volatile int s_abort;
    __shared__ TileHdr s_hdr[kMaxHdr];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_bar);
    uint64_t *empty = full + a.stages;
    uint64_t *done = empty + a.stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.stages, NP = a.parts;
    const int total = static_cast<int>(a.total_tiles);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        for (int i = 0; i < NP; ++i) mbar_init(&done[i], NW);
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
        int k = 0, s = 0, hs = 0;
        uint32_t eph = 1;
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
            unsigned char *st = smem + a.off_stage + static_cast<size_t>(s) * kStage;
            const uint32_t wb = static_cast<uint32_t>(rows) * kRowW, sbb = static_cast<uint32_t>(rows) * G * 4u;
            const size_t sbo = static_cast<size_t>(r0) * G * 4u;
            TileHdr &h = s_hdr[hs];
            if (++hs == NP) hs = 0;
            h.y = P.y + r0;
            h.y2 = nullptr;
            h.epi = nullptr;
            h.sc = nullptr;
            h.bi = nullptr;
            h.rows = rows;
            h.pad = static_cast<int>(P.n);  // stride between the tokens' outputs
            mbar_arrive_expect_tx(&full[s], wb + 2 * sbb);
            bulk_g2s(st, P.w + r0 * W, wb, &full[s], policy);
            bulk_g2s(st + kStageW, static_cast<const unsigned char *>(P.scale) + sbo, sbb, &full[s], policy);
            bulk_g2s(st + kStageW + kStageSb, static_cast<const unsigned char *>(P.bias) + sbo, sbb, &full[s], policy);
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
    const int ch = warp - 1;
    float *const part = reinterpret_cast<float *>(smem + a.off_part);
    const unsigned char *const stage0 = smem + a.off_stage;
    const int ntok = a.ntok;
    if (wait_first) {
        grid_dep_wait();
        grid_dep_launch();
    }
    MSlice<T, LC> sl;
    load_mslice<T, LC, kTree>(a, ch, lane, sl);
    // pi = the lane's low 4 bits reversed; value v[4r + t] holds (row, token)
    // index (4r + t) ^ pi: rows loaded in the order r ^ (pi >> 2), activation
    // slice t holding token t ^ (pi & 3)
    const int pi = ((lane & 1) << 3) | ((lane & 2) << 1) | ((lane >> 1) & 2) | ((lane >> 3) & 1);
    const int rp = pi >> 2, tp = pi & 3;
    if (tp & 1) {
#pragma unroll
        for (int m = 0; m < LC / 2; ++m) {
            float2 q = sl.X[0][m];
            sl.X[0][m] = sl.X[1][m];
            sl.X[1][m] = q;
            q = sl.X[2][m];
            sl.X[2][m] = sl.X[3][m];
            sl.X[3][m] = q;
        }
    }
    if (tp & 2) {
#pragma unroll
        for (int m = 0; m < LC / 2; ++m) {
            float2 q = sl.X[0][m];
            sl.X[0][m] = sl.X[2][m];
            sl.X[2][m] = q;
            q = sl.X[1][m];
            sl.X[1][m] = sl.X[3][m];
            sl.X[3][m] = q;
        }
    }
    // the lane's final value: row rb*R + rp, token tp (lanes 0..15).  The
    // partner lane (kL away) holds token tp ^ 1 and sends its group sum of
    // token tp.
    const float xs_own = pick<T>(sl.xs, tp);
    const float xs_par = __shfl_xor_sync(0xffffffffu, pick<T>(sl.xs, tp ^ 1), kL);
    // group completion leaves d[i] = (row, token) index i ^ pi: token tp ^ i
    const bool neg0 = kTree && ((sl.negs >> tp) & 1), neg1 = kTree && ((sl.negs >> (tp ^ 1)) & 1);
    const int g = ch * GPC + lane / kL;
    const uint32_t word = static_cast<uint32_t>(ch * 32 + lane) * 4u;  // the lane's word in a row
    uint32_t roff[R];
#pragma unroll
    for (int r = 0; r < R; ++r) roff[r] = static_cast<uint32_t>(r ^ rp) * kRowW + word;
    const uint32_t sbo = (static_cast<uint32_t>(rp) * G + g) * 4u;
    const int sbd = ((g ^ 1) - g) * 4;

    auto item = [&](auto exact_c, const unsigned char *stg, float *prt, int rb) {
        constexpr bool kExact = decltype(exact_c)::value;
        const unsigned char *blk = stg + static_cast<uint32_t>(rb * R) * kRowW;
        float v[R * T];
        uint32_t wq[R];
#pragma unroll
        for (int r = 0; r < R; ++r) wq[r] = *reinterpret_cast<const uint32_t *>(blk + roff[r]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t w[2] = {wq[r], 0u};
            lane_sums<T, LC, kExact>(w, sl, v + r * T);
        }
        float d[2];
        plevels<R * T, 1, kL, kTree>(v, d);
        if (kTree && kExact && sl.anyneg) {
            // zero sums are +0 on the exact path; in an all-negative group a
            // zero sum means every q is 0, and RN's sum is -0
            d[0] = (neg0 && d[0] == 0.f) ? kNegZero : d[0];
            d[1] = (neg1 && d[1] == 0.f) ? kNegZero : d[1];
        }
        // the pair {own group, partner group} of (row, token) index pi
        const float dpar = __shfl_xor_sync(0xffffffffu, d[1], kL);
        const unsigned char *so = stg + kStageW + static_cast<uint32_t>(rb * R * G) * 4u + sbo;
        const unsigned char *sp = so + sbd;
        const float sco = *reinterpret_cast<const float *>(so), scp = *reinterpret_cast<const float *>(sp);
        const float bio = *reinterpret_cast<const float *>(so + kStageSb);
        const float bip = *reinterpret_cast<const float *>(sp + kStageSb);
        float t0, t1;
        if constexpr (kTree) {
            t0 = __fadd_rn(__fmul_rn(sco, d[0]), __fmul_rn(bio, xs_own));
            t1 = __fadd_rn(__fmul_rn(scp, dpar), __fmul_rn(bip, xs_par));
        } else {
            t0 = fmaf(sco, d[0], bio * xs_own);
            t1 = fmaf(scp, dpar, bip * xs_par);
        }
        float tv[1] = {kTree ? __fadd_rn(t0, t1) : t0 + t1};
        float fin[1];
        plevels<1, 2 * kL, 32, kTree>(tv, fin);
        // chunk partials: (row, token) value i at prt[i * NCH + chunk]
        if (lane < R * T) prt[((rb * R + rp) * T + tp) * NCH + ch] = fin[0];
    };

    // Final sums of a finished tile: warp c adds the chunk partials of rows
    // c, c + 8, c + 16, c + 24 (lane l < 16: row c + 8 (l >> 2), token l & 3)
    // by the tree.
    auto finals = [&](int q, uint32_t ph) -> bool {
        if (!wait_or_abort(&done[q], ph, &s_abort, kSiteDone)) return false;
        if (lane < 16) {
            const TileHdr &fh = s_hdr[q];
            const int row = ch + 8 * (lane >> 2), tk = lane & 3;
            const float4 *pq = reinterpret_cast<const float4 *>(part + q * TR * T * NCH + (row * T + tk) * NCH);
            const float4 lo = pq[0], hi = pq[1];
            const float c[NCH] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
            const float yv = tree_fixed<NCH, kTree>(c);
            if (row < fh.rows && tk < ntok) fh.y[static_cast<int64_t>(tk) * fh.pad + row] = yv;
        }
        return true;
    };

    auto run = [&](auto exact_c) {
        int s = 0, p = 0, pp = -1;
        uint32_t fph = 0, dph = 0, pdph = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            if (!wait_or_abort(&full[s], fph, &s_abort, kSiteFull)) break;
            const unsigned char *stg = stage0 + static_cast<uint32_t>(s) * kStage;
            float *prt = part + p * TR * T * NCH;
            for (int rb = 0; rb < NI; ++rb) item(exact_c, stg, prt, rb);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s]);
                mbar_arrive(&done[p]);
            }
            if (pp >= 0 && !finals(pp, pdph)) break;
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
        if (pp >= 0) finals(pp, pdph);
    };
    if (sl.exact) {
        run(std::true_type{});
    } else {
        run(std::false_type{});
    }
    if (!wait_first) grid_dep_wait();
}

}  // namespace

}  // namespace abg
