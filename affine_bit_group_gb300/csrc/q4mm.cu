// q4mm host side: planning, instantiation and launch of the batched product
// kernel (q4mm_kernel.cuh) for pairs of tokens.  The product is bound by the
// computing warps' instruction stream, not by HBM, so larger batches run as
// several pair launches: a 4-token lane mapping (8 columns per lane) was
// measured slower per token than pairs, its butterflies and register pressure
// outweighing the shared unpacking.
#include "q4mm_fixed.cuh"

#include <algorithm>

namespace abg {

namespace {

template <int T, int R, bool kTree, bool kSb>
void *mm_ptr() {
    return reinterpret_cast<void *>(&q4mm_kernel<T, R, kTree, kSb>);
}

template <bool kTree, int kC>
void *mmf_ptr() {
    return reinterpret_cast<void *>(&q4mm_fixed_kernel<kTree, kC>);
}

template <bool kTree>
void *mm4_ptr() {
    return reinterpret_cast<void *>(&q4mm4_fixed_kernel<kTree>);
}

// Rows per item: T * R = 8 values per lane.  shape != 0: the fixed-shape
// kernel for rows of `shape` columns (T = 4: only the fixed shape exists).
void *select_mm(int T, bool tree, bool sb, int shape = 0) {
    if (T == 4) return (sb && shape == kMm4Cols) ? (tree ? mm4_ptr<true>() : mm4_ptr<false>()) : nullptr;
    if (T == 2 && sb && shape == 2048) return tree ? mmf_ptr<true, 2048>() : mmf_ptr<false, 2048>();
    if (T == 2 && sb && shape == 4096) return tree ? mmf_ptr<true, 4096>() : mmf_ptr<false, 4096>();
    if (T == 2) {
        if (tree) return sb ? mm_ptr<2, 4, true, true>() : mm_ptr<2, 4, true, false>();
        return sb ? mm_ptr<2, 4, false, true>() : mm_ptr<2, 4, false, false>();
    }
    return nullptr;
}

constexpr int mm_rows(int T) { return 8 / T; }

inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

}  // namespace

bool plan_q4mm(Q4Plan *plan, const Q4Prob *probs, int nprob, int cols, int T, int ntok, const float *const *xt,
               const float *const *xst, int prologue, bool tree, int rows_per_warp, bool sb_smem) {
    (void)rows_per_warp;  // rows per item follow from T (T * R = 8 values per lane)
    if ((T == 2 ? !select_mm(T, tree, sb_smem) : !(T == 4 && cols == kMm4Cols && sb_smem)) || ntok < 1 || ntok > T ||
        nprob < 1 || nprob > kMmProbs)
        return false;
    Q4Args &a = plan->args;
    a = Q4Args{};
    const int R = mm_rows(T);
    const int LC = 32 / T, CW = 32 * LC;
    const int C = cols, W = C / 8, G = C / 64, nch = (C + CW - 1) / CW;
    int nw = nch <= 8 ? nch * (8 / nch) : 8;
    const int kk = (nch <= nw) ? nw / nch : 1;
    const uint32_t row_bytes = static_cast<uint32_t>(C / 2) + (sb_smem ? 8u * G : 0u);
    const uint32_t fixed = 1024, budget = 110u * 1024u, hard_max = 225u * 1024u;
    const int unit = R * kk;
    int TR = unit;
    // final-sum threads: TR * T <= computing threads
    while (TR * 2 * T <= nw * 32 && (TR * 2) * row_bytes <= 40u * 1024u) TR *= 2;
    if (TR * T > nw * 32) return false;
    auto stage_bytes = [&](int tr) {
        return align_up(static_cast<uint32_t>(tr) * (C / 2), 16) +
               2u * align_up(sb_smem ? static_cast<uint32_t>(tr) * G * 4u : 0u, 16);
    };
    auto part_bytes = [&](int tr, int stages) {
        return align_up(static_cast<uint32_t>((stages + 2) * tr * nch * T) * 4u, 16);
    };
    int S = 0;
    uint32_t bud = budget;
    for (int attempt = 0; attempt < 2; ++attempt) {
        for (;;) {
            const uint32_t sb = stage_bytes(TR);
            S = 0;
            while (S < 8 && fixed + (S + 1) * sb + part_bytes(TR, S + 1) + 8u * (3 * (S + 1) + 2) <= bud) ++S;
            if (S >= 2 || TR <= unit) break;
            TR = std::max(unit, TR / 2);
        }
        if (S >= 2) break;
        bud = hard_max;
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
    if (a.total_tiles > 0x7fffffff) return false;
    for (int t = 0; t < T; ++t) {
        a.xt[t] = xt[std::min(t, ntok - 1)];
        a.xst[t] = xst ? xst[std::min(t, ntok - 1)] : nullptr;
    }
    a.ntok = ntok;
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
    a.off_bar = align_up(a.off_part + part_bytes(TR, S), 16);
    a.parts = S + 2;
    a.smem_bytes = a.off_bar + 8u * (2 * S + a.parts);
    // the fixed-shape kernel when the plan has its shape (its stage layout and
    // tile rows are compile-time constants equal to these)
    const bool fixed_shape =
        a.parts <= kMaxHdr && sb_smem && nw == 8 &&
        ((T == 2 && (C == 2048 || C == 4096) && TR == mmf_tr(C)) || (T == 4 && C == kMm4Cols && TR == kMm4Rows));
    plan->shape = fixed_shape ? C : 0;
    void *fn = select_mm(T, tree, sb_smem, plan->shape);
    if (!fn) return false;
    int fit = 1;
    if (raise_smem_limit(fn) == cudaSuccess) {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, 32 * (1 + nw), a.smem_bytes) == cudaSuccess &&
            nb > 0)
            fit = nb;
    }
    cudaGetLastError();
    const int64_t cap = static_cast<int64_t>(sm_count()) * std::min(fit, 2);
    plan->grid = dim3(static_cast<unsigned>(std::max<int64_t>(1, std::min(a.total_tiles, cap))));
    plan->block = dim3(32u * (1 + nw));
    plan->rows_per_warp = R;
    plan->tree = tree;
    plan->sb_smem = sb_smem;
    plan->layout = 0;
    plan->lg = 1;
    plan->half = false;
    plan->mm = T;
    return true;
}

cudaError_t launch_q4mm(const Q4Plan &plan, cudaStream_t stream, bool pdl) {
    if (plan.args.total_tiles == 0) return cudaSuccess;
    void *fn = select_mm(plan.mm, plan.tree, plan.sb_smem, plan.shape);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = raise_smem_limit(fn);
    if (e != cudaSuccess) return e;
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
    Q4ArgsT<kMmProbs> mm{};
    narrow_args(mm, plan.args);
    void *params[] = {&mm};
    return cudaLaunchKernelExC(&cfg, fn, params);
}

cudaError_t q4mm_status(unsigned *bits, bool clear) { return read_status_word(bits, clear); }

}  // namespace abg
