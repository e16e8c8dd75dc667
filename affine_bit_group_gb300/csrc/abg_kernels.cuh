// Launch descriptors and host-side launchers of the library's kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

namespace abg {

// Products that share one activation in a grouped launch: the table of the
// planner and of the throughput kernels.  A kernel's argument block costs
// launch time in proportion to its size (about 0.02 us per KB on every
// launch), so each kernel family takes the smallest table its launches need:
// the few-tiles instantiations (a decode token's products) kFewProbs, the
// batched product's kernels (one product a launch) kMmProbs.
constexpr int kMaxProbs = 256;
constexpr int kFewProbs = 16;
constexpr int kMmProbs = 1;

enum Prologue { kProNone = 0, kProGsum = 1, kProRmsq = 2, kProSwq = 3 };

// One matrix of a (grouped) product launch.  Pointers already point at row row0.
struct Q4Prob {
    const uint32_t *w;
    const void *scale;  // f32, or bf16 / f16 bit patterns
    const void *bias;
    float *y;
    int64_t n;  // rows to compute
    int tiles;  // ceil(n / tr) (a launch's tiles fit in 32 bits)
    int tr;     // rows per tile of this problem: tile_rows, or a quarter of it (see plan_q4mv)
};

// Everything the product kernel needs, passed by value (__grid_constant__),
// with a table of kP products after the other fields (so every table size
// lays those fields out alike).
template <int kP>
struct Q4ArgsT {
    int nprob;
    int64_t total_tiles;
    // activation: x/xsum for kProNone; producer inputs otherwise (see abg.h)
    const float *x;
    const float *xsum;
    const float *wt;
    float eps;
    int prologue;
    // 1: read the activation only after the preceding launch has finished
    // (it produced it).  0: the preceding launch is a sibling of the same
    // stage, the activation is ready at start; wait for that launch only
    // before exiting, so finishing still implies every earlier launch finished.
    int wait_first;
    // shape (G = cols / group size)
    int cols, W, G, nch;
    int sb_f16;  // 16-bit scale and bias: 1 = f16, 0 = bf16
    // tiling (parts: partial-sum buffers, stages + 2)
    int tile_rows, stages, nw, parts;
    // shared-memory layout (byte offsets)
    uint32_t off_stage, stage_w_bytes, stage_sb_bytes, stage_bytes, off_part, off_bar;
    // the activation staged by the fixed-shape prologue (0 bytes when unused):
    // cols floats in the per-lane layout, then group sums and group flags
    uint32_t off_act, act_bytes;
    uint32_t smem_bytes;
    // failure-detection self-test only: the producer delivers no tile, so the
    // computing warps' bounded waits run out (see abg_selftest_wait_timeout)
    int withhold;
    // SwiGLU pair (fixed shapes, 4 rows per item): problems 0 and 1 are the
    // gate and up products of one activation, with equal shapes; a tile holds
    // tile_rows/2 rows of each (the same row indices), every item 2 gate rows
    // and the same 2 up rows, and the computing warps write
    // epi[r] = silu(gate y[r]) * up y[r] besides both outputs
    int paired;
    float *epi;
    // batched product only: activation and group-sum rows of the T token
    // slots, and how many of them are real tokens
    const float *xt[4];
    const float *xst[4];
    int ntok;
    Q4Prob prob[kP];
};
using Q4Args = Q4ArgsT<kMaxProbs>;

// A plan's arguments with a smaller table (nprob <= kP, which the planners
// ensure for the kernels that take one).
template <int kP>
void narrow_args(Q4ArgsT<kP> &dst, const Q4Args &src) {
    static_assert(offsetof(Q4ArgsT<kP>, prob) == offsetof(Q4Args, prob), "fields laid out alike");
    std::memcpy(&dst, &src, offsetof(Q4Args, prob));
    std::memcpy(dst.prob, src.prob, static_cast<size_t>(src.nprob < kP ? src.nprob : kP) * sizeof(Q4Prob));
}

struct Q4Tuning {
    int smem_kb = 0;
    int consumer_warps = 0;
    int blocks_per_sm = 0;
    int stage_kb = 0;
};

struct Q4Plan {
    Q4Args args;
    dim3 grid, block;
    int rows_per_warp;
    bool tree;
    bool sb_smem;
    int layout;  // block layout (see the kernel)
    int shape = 0;  // row length of a fixed-shape instantiation (0: sizes from the arguments)
    int lg;      // group size 32 << lg
    bool half;   // 16-bit scale and bias
    int mm = 0;  // batched product: kernel width in tokens (0: single token)
};

// Fills plan->args layout, grid and block for products sharing one activation
// and one weight format (group 32, 64 or 128; sb_type an abg_sb_type).
// Returns false if the shape cannot be planned (cols too large for shared memory).
bool plan_q4mv(Q4Plan *plan, const Q4Prob *probs, int nprob, int cols, int group, int sb_type, int prologue,
               const float *x, const float *xsum, const float *wt, float eps, bool tree, int rows_per_warp,
               bool sb_smem, const Q4Tuning &tune);

// Sets the kernel's shared-memory limit for a plan (not a stream operation;
// call it before stream capture).
cudaError_t prepare_q4mv(const Q4Plan &plan);

// Launches a planned product on `stream`; `pdl` marks it as a programmatic
// dependent of the previous launch on the stream (plan.args.wait_first says
// whether it also depends on that launch's results).
cudaError_t launch_q4mv(const Q4Plan &plan, cudaStream_t stream, bool pdl);

// Producers; their group sums cover `group` (32, 64 or 128) values each.
cudaError_t launch_gsum(const float *v, float *s, int64_t n, int group, bool tree, cudaStream_t stream, bool pdl);
cudaError_t launch_rmsq(const float *x, const float *wt, float eps, float *xn, float *xsum, int64_t n, int group,
                        bool tree, cudaStream_t stream, bool pdl);
cudaError_t launch_swq(const float *a, float *o, float *osum, int64_t n, int group, bool tree, cudaStream_t stream,
                       bool pdl);

int sm_count();

// Raises a kernel's dynamic shared-memory limit to the device maximum (once).
cudaError_t raise_smem_limit(void *fn);

// Batched product (q4mm.cu): plan and launch for kernel width T (2 or 4)
// tokens, of which ntok are real (x and y rows of the others are never read
// or written beyond the duplicated pointers the caller passes).
bool plan_q4mm(Q4Plan *plan, const Q4Prob *probs, int nprob, int cols, int T, int ntok, const float *const *xt,
               const float *const *xst, int prologue, bool tree, int rows_per_warp, bool sb_smem);
cudaError_t launch_q4mm(const Q4Plan &plan, cudaStream_t stream, bool pdl);
cudaError_t q4mm_status(unsigned *bits, bool clear);

// Each translation unit's device status word (OR-ed into *bits).
cudaError_t q4mv_status(unsigned *bits, bool clear);
cudaError_t vec_status(unsigned *bits, bool clear);

}  // namespace abg
