// q4mv host side: planning and launching of the product kernel
// (q4mv_kernel.cuh), and its instantiations for the default format -- groups
// of 64 columns with f32 scale and bias -- in all three block layouts.  The
// other formats are instantiated, in block layout 0, by q4mv_g32.cu,
// q4mv_g32h.cu, q4mv_g64h.cu, q4mv_g128.cu and q4mv_g128h.cu.
#include "q4mv_kernel.cuh"

#include <algorithm>
#include <mutex>
#include <set>

namespace abg {

// kernel selectors and status words of the other format units
void *q4mv_select_g32(int R, bool tree, bool sb);
void *q4mv_select_g32h(int R, bool tree, bool sb);
void *q4mv_select_g64h(int R, bool tree, bool sb);
void *q4mv_select_g128(int R, bool tree, bool sb);
void *q4mv_select_g128h(int R, bool tree, bool sb);
cudaError_t q4mv_status_g32(unsigned *bits, bool clear);
cudaError_t q4mv_status_g32h(unsigned *bits, bool clear);
cudaError_t q4mv_status_g64h(unsigned *bits, bool clear);
cudaError_t q4mv_status_g128(unsigned *bits, bool clear);
cudaError_t q4mv_status_g128h(unsigned *bits, bool clear);
void *q4mv_select_fixed(int cols, bool tree, int R, int layout);
void *q4mv_select_fixed_half(int cols, bool tree, int R, int layout);
void *q4mv_select_fixed_g32(int cols, bool tree, int R, int layout, bool half);
void *q4mv_select_fixed_g128(int cols, bool tree, int R, int layout, bool half);
cudaError_t q4mv_status_fixed(unsigned *bits, bool clear);
cudaError_t q4mv_status_fixed_half(unsigned *bits, bool clear);
cudaError_t q4mv_status_fixed_g32(unsigned *bits, bool clear);
cudaError_t q4mv_status_fixed_g128(unsigned *bits, bool clear);

namespace {

// The instantiation for a format (group = 32 << lg columns; 16-bit scale and
// bias when half), rows per item, mode, scale/bias staging and block layout;
// nullptr if it is not built (layouts 1 and 2 exist for the default format
// with 8 rows per item only).  shape != 0 selects the fixed-shape
// instantiation for that row length (q4mv_fixed.cu).
void *select_kernel(int lg, bool half, int R, bool tree, bool sb, int layout, int shape = 0) {
    if (shape != 0) {
        if (lg == 0) return q4mv_select_fixed_g32(shape, tree, R, layout, half);
        if (lg == 2) return q4mv_select_fixed_g128(shape, tree, R, layout, half);
        return half ? q4mv_select_fixed_half(shape, tree, R, layout) : q4mv_select_fixed(shape, tree, R, layout);
    }
    if (lg == 1 && !half) {
        if (layout == 0) return select_layout0<1, false>(R, tree, sb);
        if (R != 8) return nullptr;
        if (layout == 1) {
            if (tree) return sb ? kernel_ptr<8, true, true, 1, 1, false>() : kernel_ptr<8, true, false, 1, 1, false>();
            return sb ? kernel_ptr<8, false, true, 1, 1, false>() : kernel_ptr<8, false, false, 1, 1, false>();
        }
        if (layout == 2) {
            if (tree) return sb ? kernel_ptr<8, true, true, 2, 1, false>() : kernel_ptr<8, true, false, 2, 1, false>();
            return sb ? kernel_ptr<8, false, true, 2, 1, false>() : kernel_ptr<8, false, false, 2, 1, false>();
        }
        return nullptr;
    }
    if (layout != 0) return nullptr;
    switch (lg) {
    case 0: return half ? q4mv_select_g32h(R, tree, sb) : q4mv_select_g32(R, tree, sb);
    case 1: return q4mv_select_g64h(R, tree, sb);
    case 2: return half ? q4mv_select_g128h(R, tree, sb) : q4mv_select_g128(R, tree, sb);
    default: return nullptr;
    }
}

inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

}  // namespace

cudaError_t q4mv_status(unsigned *bits, bool clear) {
    cudaError_t (*const units[])(unsigned *, bool) = {read_status_word,   q4mv_status_g32,  q4mv_status_g32h,
                                                      q4mv_status_g64h,   q4mv_status_g128, q4mv_status_g128h,
                                                      q4mv_status_fixed,  q4mv_status_fixed_half,
                                                      q4mv_status_fixed_g32, q4mv_status_fixed_g128};
    for (auto f : units) {
        const cudaError_t e = f(bits, clear);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
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
constexpr int kFewTilesPerSm = 4;

// A launch of one block per SM whose tiles exceed the SMs by a little (a
// decode token's q/k/v products: 160 tiles on 152 SMs) would run a second
// round of whole tiles on a few SMs.  Its last problems are cut into quarter
// tiles instead (TR/4 rows, a whole number of items), as long as the whole
// tiles left number at most the SMs and all tiles at most twice that: tile t
// runs on block t mod SMs, so no block then takes more than one whole and one
// quarter tile.  Results are unchanged (a tile's rows are summed as before).
void quarter_tail(Q4Args &a, int TR, int R, int64_t sms) {
    const int tq = TR / 4;
    if (tq < R || tq % R != 0 || a.paired || a.total_tiles <= sms) return;
    int64_t whole = a.total_tiles, quarter = 0;
    int first = a.nprob;
    while (first > 0 && whole > sms) {
        --first;
        whole -= a.prob[first].tiles;
        quarter += (a.prob[first].n + tq - 1) / tq;
    }
    if (whole > sms || whole + quarter > 2 * sms) return;
    for (int i = first; i < a.nprob; ++i) {
        a.prob[i].tr = tq;
        a.prob[i].tiles = static_cast<int>((a.prob[i].n + tq - 1) / tq);
    }
    a.total_tiles = whole + quarter;
}

bool plan_once(Q4Plan *plan, const Q4Prob *probs, int nprob, int cols, int group, int sb_type, int prologue,
               const float *x, const float *xsum, const float *wt, float eps, bool tree, int rows_per_warp,
               bool sb_smem, const Q4Tuning &tune, bool allow_few, int force_layout = -1) {
    if (nprob < 1 || nprob > kMaxProbs) return false;
    Q4Args &a = plan->args;
    a = Q4Args{};
    const int R = rows_per_warp;
    const int lg = group == 32 ? 0 : (group == 64 ? 1 : 2);
    const bool half = sb_type != ABG_SB_F32;
    const uint32_t elem = half ? 2u : 4u;
    const int C = cols, W = C / 8, G = C / group, nch = (C + 1023) / 1024;
    // consumer warps: a multiple of the chunk count (each warp keeps one
    // 1024-column slice of x), at most 8 (the kernel's launch bound)
    // layout (default format only): tuned consumer_warps > 8 selects one
    // block per SM; 1..6 with 8 rows per item selects the 128-register
    // two-block layout
    const bool fmt_default = lg == 1 && !half;
    const int layout = force_layout >= 0 ? force_layout
                       : (!fmt_default || R != 8 || tune.consumer_warps == 0)
                           ? 0
                           : (tune.consumer_warps > 8 ? 1 : (tune.consumer_warps <= 6 ? 2 : 0));
    const bool wide = layout == 1 || layout == 4;  // one block per SM, the large shared-memory budget
    const int nw_max = layout_max_warps(layout);
    int nw = force_layout >= 0 ? 0 : tune.consumer_warps;
    if (nw <= 0) nw = nch <= nw_max ? nch * (nw_max / nch) : nw_max;
    if (nch <= nw_max) nw = nch * (std::min(nw, nw_max) / nch);
    nw = std::min(std::max(nw, 1), nw_max);
    const int kk = (nch <= nw) ? nw / nch : 1;  // warps per chunk position
    const uint32_t row_bytes = static_cast<uint32_t>(C / 2) + (sb_smem ? 2u * G * elem : 0u);
    // the fixed-shape prologue stages the activation: cols floats, G group
    // sums, G group flags and a flag per 128 columns
    const bool fmt_fixed = lg >= 0 && lg <= 2;  // every format has fixed-shape instantiations
    const bool act_stage = fmt_fixed && sb_smem && (C == 2048 || C == 4096 || C == 6144);
    const uint32_t act_bytes = act_stage ? align_up(static_cast<uint32_t>(C * 4 + G * 8 + C / 32), 128) : 0u;
    const uint32_t fixed = 1024 + act_bytes;  // barriers, alignment slack and the staged activation
    // tile rows: a multiple of R*kk so row blocks spread evenly over the warps
    const int unit = R * kk;
    int TR = unit;
    const uint32_t stage_target = static_cast<uint32_t>(tune.stage_kb > 0 ? tune.stage_kb : 40) * 1024u;
    while (TR * 2 <= nw * 32 && (TR * 2) * row_bytes <= stage_target) TR *= 2;
    TR = std::min(TR, nw * 32);
    if (TR < R) return false;
    // A launch of few tiles (at most kFewTilesPerSm per SM, e.g. a decode
    // token's products) runs one block per SM with a larger stage ring: two
    // blocks of a small launch would share some SMs and leave others idle,
    // and those SMs finish last.  Large launches keep two blocks per SM,
    // which hides each block's per-tile bubbles behind the other.
    int64_t tiles_est = 0;
    for (int i = 0; i < nprob; ++i) tiles_est += (probs[i].n + TR - 1) / TR;
    const bool few = allow_few && !wide && tune.smem_kb == 0 && tune.blocks_per_sm == 0 &&
                     tiles_est <= static_cast<int64_t>(kFewTilesPerSm) * sm_count();
    uint32_t budget =
        static_cast<uint32_t>(tune.smem_kb > 0 ? tune.smem_kb : (wide ? 220 : (few ? 160 : 110))) * 1024u;
    const uint32_t hard_max = 225u * 1024u;  // leaves room for the static shared memory
    auto stage_bytes = [&](int tr) {
        return align_up(static_cast<uint32_t>(tr) * (C / 2), 16) +
               2u * align_up(sb_smem ? static_cast<uint32_t>(tr) * G * elem : 0u, 16);
    };
    auto part_bytes = [&](int tr, int stages) {
        return align_up(static_cast<uint32_t>((stages + 2) * tr * nch) * 4u, 16);
    };
    int S = 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
        for (;;) {
            const uint32_t sb = stage_bytes(TR);
            S = 0;
            while (S < 8 && fixed + (S + 1) * sb + part_bytes(TR, S + 1) + 8u * (3 * (S + 1) + 2) <= budget) ++S;
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
        const int64_t tiles = (probs[i].n + TR - 1) / TR;
        if (tiles > 0x7fffffff) return false;
        a.prob[i].tr = TR;
        a.prob[i].tiles = static_cast<int>(tiles);
        a.total_tiles += tiles;
    }
    if (a.total_tiles > 0x7fffffff) return false;  // the kernel counts tiles in 32 bits
    // the budget loop may have halved the tile rows after the few-tiles
    // decision: a launch that has more tiles than that rule admits is planned
    // again with two blocks per SM
    if (few && a.total_tiles > static_cast<int64_t>(kFewTilesPerSm) * sm_count())
        return plan_once(plan, probs, nprob, cols, group, sb_type, prologue, x, xsum, wt, eps, tree, rows_per_warp,
                         sb_smem, tune, false, force_layout);
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
    a.stage_sb_bytes = align_up(sb_smem ? static_cast<uint32_t>(TR) * G * elem : 0u, 16);
    a.sb_f16 = sb_type == ABG_SB_F16 ? 1 : 0;
    a.stage_bytes = a.stage_w_bytes + 2 * a.stage_sb_bytes;
    a.off_part = a.off_stage + S * a.stage_bytes;
    a.off_bar = align_up(a.off_part + part_bytes(TR, S), 16);
    a.parts = S + 2;
    a.off_act = align_up(a.off_bar + 8u * (2 * S + a.parts), 128);
    a.act_bytes = act_bytes;
    a.smem_bytes = a.off_act + act_bytes;

    // a plan with the compile-time shape of its row length runs the
    // fixed-shape instantiation (same results, constant sizes) if its product
    // table holds the launch's products
    int shape = 0;
    if (fmt_fixed && sb_smem && nprob <= kernel_probs(layout, C) &&
        ((layout == 0 && R == 8) || (layout == 1 && R == 4) || (layout == 4 && R == 8 && C == 6144)) &&
        (C == 2048 || C == 4096 || C == 6144) && TR == fixed_tr(C, R, layout) && nw == fixed_nw(C, layout) &&
        nch == fixed_nch(C) && a.stage_w_bytes == static_cast<uint32_t>(TR * C / 2) &&
        a.stage_sb_bytes == static_cast<uint32_t>(TR * G) * elem)
        shape = C;

    // blocks per SM: what fits (registers and shared memory), at most 2 (1 for a
    // launch of few tiles) unless tuned
    int fit = 1;
    void *fn = select_kernel(lg, half, R, tree, sb_smem, layout, shape);
    if (!fn) return false;
    if (raise_smem_limit(fn) == cudaSuccess) {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, static_cast<int>(32 * (1 + nw)), a.smem_bytes) ==
                cudaSuccess &&
            nb > 0)
            fit = nb;
    }
    cudaGetLastError();
    int bps = std::min(fit, wide ? 1 : (tune.blocks_per_sm > 0 ? tune.blocks_per_sm : (few ? 1 : 2)));
    bps = std::max(bps, 1);
    // (fixed shapes skip a quarter tile's empty items only in the few-tiles
    // layout; elsewhere the generic kernel does)
    if (bps == 1 && (shape == 0 || layout == 1)) quarter_tail(a, TR, R, sm_count());
    const int64_t cap = static_cast<int64_t>(sm_count()) * bps;
    plan->grid = dim3(static_cast<unsigned>(std::max<int64_t>(1, std::min(a.total_tiles, cap))));
    plan->block = dim3(32u * (1 + nw));
    plan->rows_per_warp = R;
    plan->tree = tree;
    plan->sb_smem = sb_smem;
    plan->layout = layout;
    plan->shape = shape;
    plan->lg = lg;
    plan->half = half;
    plan->mm = 0;
    return true;
}


}  // namespace

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

// Plans with the requested rows per item; if the stages do not fit in shared
// memory (very wide rows), retries with fewer rows per item (same results).
// rows_per_warp 0 chooses: a launch of few tiles (a decode token's products)
// of a row length with a fixed-shape instantiation runs 16 computing warps
// with 4 rows per item in one block per SM, so each tile is split over twice
// as many warps and finishes sooner; every other launch runs 8 rows per item.
bool plan_q4mv(Q4Plan *plan, const Q4Prob *probs, int nprob, int cols, int group, int sb_type, int prologue,
               const float *x, const float *xsum, const float *wt, float eps, bool tree, int rows_per_warp,
               bool sb_smem, const Q4Tuning &tune) {
    if (rows_per_warp == 0) {
        const bool plain_tuning = tune.smem_kb == 0 && tune.consumer_warps == 0 && tune.blocks_per_sm == 0 &&
                                  tune.stage_kb == 0;
        if (plain_tuning && sb_smem && (cols == 2048 || cols == 4096 || cols == 6144)) {
            const int tr = fixed_tr(cols, 4, 1);
            int64_t tiles = 0;
            for (int i = 0; i < nprob; ++i) tiles += (probs[i].n + tr - 1) / tr;
            if (tiles <= static_cast<int64_t>(kFewTilesPerSm) * sm_count() &&
                plan_once(plan, probs, nprob, cols, group, sb_type, prologue, x, xsum, wt, eps, tree, 4, sb_smem,
                          tune, false, 1) &&
                plan->shape == cols)
                return true;
        }
        rows_per_warp = 8;
    }
    // rows of 6144 columns in a launch of many tiles: 18 computing warps in one
    // block per SM (three per chunk), where the two-block layout has six
    if (rows_per_warp == 8 && cols == 6144 && group != 32 && sb_smem &&
        tune.smem_kb == 0 && tune.consumer_warps == 0 && tune.blocks_per_sm == 0 && tune.stage_kb == 0) {
        const int tr = fixed_tr(cols, 8, 4);
        int64_t tiles = 0;
        for (int i = 0; i < nprob; ++i) tiles += (probs[i].n + tr - 1) / tr;
        if (tiles > static_cast<int64_t>(kFewTilesPerSm) * sm_count() &&
            plan_once(plan, probs, nprob, cols, group, sb_type, prologue, x, xsum, wt, eps, tree, 8, sb_smem, tune,
                      false, 4) &&
            plan->shape == cols)
            return true;
    }
    for (int R = rows_per_warp; R >= 1; R /= 2)
        if (plan_once(plan, probs, nprob, cols, group, sb_type, prologue, x, xsum, wt, eps, tree, R, sb_smem, tune,
                      true))
            return true;
    return false;
}

cudaError_t prepare_q4mv(const Q4Plan &plan) {
    void *fn = select_kernel(plan.lg, plan.half, plan.rows_per_warp, plan.tree, plan.sb_smem, plan.layout, plan.shape);
    if (!fn) return cudaErrorInvalidValue;
    return raise_smem_limit(fn);
}

cudaError_t launch_q4mv(const Q4Plan &plan, cudaStream_t stream, bool pdl) {
    if (plan.args.total_tiles == 0) return cudaSuccess;
    void *fn = select_kernel(plan.lg, plan.half, plan.rows_per_warp, plan.tree, plan.sb_smem, plan.layout, plan.shape);
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
    if (kernel_probs(plan.layout, plan.shape) == kFewProbs) {
        Q4ArgsT<kFewProbs> few{};
        narrow_args(few, plan.args);
        void *params[] = {&few};
        return cudaLaunchKernelExC(&cfg, fn, params);
    }
    void *params[] = {const_cast<Q4Args *>(&plan.args)};
    return cudaLaunchKernelExC(&cfg, fn, params);
}

}  // namespace abg
