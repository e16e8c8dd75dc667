// The library's C ABI (include/abg.h): argument validation, the single calls,
// and the stage graph that records a decode token's dependent stages into one
// CUDA graph.
//
// Stage semantics follow "Array.q4go/Array.q4wait queue Metal Q4 products in
// one command buffer and wait once on a flag" (bendlang/bend #1437, Change:
// queued products run concurrently, none may read another's y, dependent
// stages need a wait) and "Metal: queued rmsq, swq, gdn and atq kernels ..."
// (#1440, Why: a decode token as one command buffer with one wait).  Here a
// token is one graph launch; the caller's single stream synchronization is
// the one wait.
#include "../../include/abg.h"
#include "abg_kernels.cuh"
#include "mixer.cuh"

#include <algorithm>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <string>
#include <vector>

using namespace abg;

namespace {

thread_local std::string g_cuda_error;

// Live stage-graph handles: launching or destroying a handle that was never
// created here, or was destroyed already, is refused with ABG_EINVAL instead
// of touching freed memory.
std::mutex g_graphs_mu;
std::set<void *> g_graphs;

bool graph_live(void *g) {
    std::lock_guard<std::mutex> lock(g_graphs_mu);
    return g && g_graphs.count(g) != 0;
}
Q4Tuning g_tuning;

abg_status cuda_fail(cudaError_t e, const char *where = nullptr) {
    if (e == cudaSuccess) return ABG_OK;
    g_cuda_error = where ? std::string(where) + ": " + cudaGetErrorString(e) : std::string(cudaGetErrorString(e));
    return ABG_ECUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
    uintptr_t lo = 0, hi = 0;  // [lo, hi) in bytes; empty when lo == hi
};
Range rng(const void *p, int64_t count, size_t elem) {
    Range r;
    r.lo = reinterpret_cast<uintptr_t>(p);
    r.hi = r.lo + static_cast<uintptr_t>(count) * elem;
    return r;
}
bool overlap(Range a, Range b) { return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi; }

bool valid_group(int group) { return group == 32 || group == 64 || group == 128; }
// a vector length: whole 64-value groups and whole groups of `group`
bool valid_len(int64_t n, int group = 64) { return n > 0 && n % 64 == 0 && n % group == 0; }
// node field: 0 means 64
int node_group(int32_t g) { return g == 0 ? 64 : g; }

// ------------------------------------------------------------ products ----
struct Q4Call {
    const uint32_t *w;
    const void *scale, *bias;
    int64_t rows, cols, row0, n;
    float *y;
    int prologue;
    const float *x, *xsum, *wt;
    float eps;
    int group = 64;
    int sb_type = ABG_SB_F32;
};

int64_t act_len(const Q4Call &c) { return c.prologue == kProSwq ? 2 * c.cols : c.cols; }
size_t sb_elem(const Q4Call &c) { return c.sb_type == ABG_SB_F32 ? 4 : 2; }
int64_t groups(const Q4Call &c) { return c.cols / c.group; }

// the weight arrays of a product (packed words, scale, bias)
std::vector<Range> q4_weights(const Q4Call &c) {
    const int64_t W = c.cols / 8, G = groups(c);
    return {rng(c.w, c.rows * W, 4), rng(c.scale, c.rows * G, sb_elem(c)), rng(c.bias, c.rows * G, sb_elem(c))};
}

std::vector<Range> q4_inputs(const Q4Call &c) {
    std::vector<Range> in = q4_weights(c);
    in.push_back(rng(c.x, act_len(c), 4));
    if (c.prologue == kProNone) in.push_back(rng(c.xsum, groups(c), 4));
    if (c.prologue == kProRmsq) in.push_back(rng(c.wt, c.cols, 4));
    return in;
}

abg_status check_q4(const Q4Call &c, int mode, int rpw) {
    if (mode != ABG_TREE && mode != ABG_FAST) return ABG_EINVAL;
    if (rpw != 0 && rpw != 1 && rpw != 2 && rpw != 4 && rpw != 8) return ABG_EINVAL;
    if (c.prologue < kProNone || c.prologue > kProSwq) return ABG_EINVAL;
    if (!valid_group(c.group) || c.sb_type < ABG_SB_F32 || c.sb_type > ABG_SB_F16) return ABG_EINVAL;
    if (c.cols <= 0 || c.cols % 64 != 0 || c.cols % c.group != 0 || c.cols > ABG_MAX_COLS) return ABG_ESHAPE;
    if (c.rows < 0 || c.row0 < 0 || c.n < 0 || c.row0 > c.rows || c.n > c.rows - c.row0) return ABG_ESHAPE;
    if (c.n == 0) return ABG_OK;
    if (!c.w || !c.scale || !c.bias || !c.x || !c.y) return ABG_EINVAL;
    if (c.prologue == kProNone && !c.xsum) return ABG_EINVAL;
    if (c.prologue == kProRmsq && !c.wt) return ABG_EINVAL;
    if (!aligned(c.w, 16) || !aligned(c.x, 16) || !aligned(c.scale, sb_elem(c)) || !aligned(c.bias, sb_elem(c)) ||
        !aligned(c.y, 4))
        return ABG_EALIGN;
    if (c.prologue == kProNone && !aligned(c.xsum, 4)) return ABG_EALIGN;
    if (c.prologue == kProRmsq && !aligned(c.wt, 16)) return ABG_EALIGN;
    const Range out = rng(c.y, c.n, 4);
    for (const Range &r : q4_inputs(c))
        if (overlap(out, r)) return ABG_EALIAS;
    return ABG_OK;
}

// Scale and bias rows are bulk-copied when every row starts on 16 bytes.
bool sb_bulk(const Q4Call &c) {
    return (groups(c) * static_cast<int64_t>(sb_elem(c))) % 16 == 0 && aligned(c.scale, 16) && aligned(c.bias, 16);
}

Q4Prob make_prob(const Q4Call &c) {
    Q4Prob p = {};
    const size_t sbo = static_cast<size_t>(c.row0 * groups(c)) * sb_elem(c);
    p.w = c.w + c.row0 * (c.cols / 8);
    p.scale = static_cast<const unsigned char *>(c.scale) + sbo;
    p.bias = static_cast<const unsigned char *>(c.bias) + sbo;
    p.y = c.y;
    p.n = c.n;
    return p;
}

abg_status plan_calls(Q4Plan *plan, const std::vector<Q4Call> &calls, int mode, int rpw) {
    // rows per item: chosen by the planner unless asked for (it never
    // changes results)
    Q4Prob probs[kMaxProbs];
    for (size_t i = 0; i < calls.size(); ++i) probs[i] = make_prob(calls[i]);
    const Q4Call &c0 = calls[0];
    if (!plan_q4mv(plan, probs, static_cast<int>(calls.size()), static_cast<int>(c0.cols), c0.group, c0.sb_type,
                   c0.prologue, c0.x, c0.xsum, c0.wt, c0.eps, mode == ABG_TREE, rpw, sb_bulk(c0),
                   g_tuning))
        return ABG_ESHAPE;
    return ABG_OK;
}

// -------------------------------------------------------------- vectors ----
abg_status check_gsum(const float *v, const float *s, int64_t n, int group, int mode) {
    if (mode != ABG_TREE && mode != ABG_FAST) return ABG_EINVAL;
    if (!v || !s || !valid_group(group)) return ABG_EINVAL;
    if (!valid_len(n, group)) return ABG_ESHAPE;
    if (!aligned(v, 16) || !aligned(s, 4)) return ABG_EALIGN;
    if (overlap(rng(s, n / group, 4), rng(v, n, 4))) return ABG_EALIAS;
    return ABG_OK;
}

abg_status check_rmsq(const float *x, const float *wt, const float *xn, const float *xsum, int64_t n, int group,
                      int mode) {
    if (mode != ABG_TREE && mode != ABG_FAST) return ABG_EINVAL;
    if (!x || !wt || !xn || !xsum || !valid_group(group)) return ABG_EINVAL;
    if (!valid_len(n, group) || n > (int64_t(1) << 20)) return ABG_ESHAPE;
    if (!aligned(x, 16) || !aligned(wt, 16) || !aligned(xn, 16) || !aligned(xsum, 4)) return ABG_EALIGN;
    const Range rx = rng(x, n, 4), rw = rng(wt, n, 4), rn = rng(xn, n, 4), rs = rng(xsum, n / group, 4);
    if (overlap(rn, rx) || overlap(rn, rw) || overlap(rs, rx) || overlap(rs, rw) || overlap(rs, rn)) return ABG_EALIAS;
    return ABG_OK;
}

abg_status check_swq(const float *a, const float *o, const float *osum, int64_t n, int group, int mode) {
    if (mode != ABG_TREE && mode != ABG_FAST) return ABG_EINVAL;
    if (!a || !o || !osum || !valid_group(group)) return ABG_EINVAL;
    if (!valid_len(n, group)) return ABG_ESHAPE;
    if (!aligned(a, 16) || !aligned(o, 16) || !aligned(osum, 4)) return ABG_EALIGN;
    const Range ra = rng(a, 2 * n, 4), ro = rng(o, n, 4), rs = rng(osum, n / group, 4);
    if (overlap(ro, ra) || overlap(rs, ra) || overlap(rs, ro)) return ABG_EALIAS;
    return ABG_OK;
}

// A copy node: len floats from x to out, each device memory or page-locked
// host memory (a captured copy from pageable memory would not be an
// asynchronous graph node).
bool copyable(const void *p) {
    cudaPointerAttributes at{};
    const cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeManaged;
}

abg_status check_copy(const float *x, const float *out, int64_t len) {
    if (!x || !out) return ABG_EINVAL;
    if (len <= 0) return ABG_ESHAPE;
    if (!aligned(x, 4) || !aligned(out, 4)) return ABG_EALIGN;
    if (overlap(rng(x, len, 4), rng(out, len, 4))) return ABG_EALIAS;
    if (!copyable(x) || !copyable(out)) return ABG_EINVAL;
    return ABG_OK;
}

// the ranges a gdn call reads and writes (state and S are read and written)
void gdn_io(const abg_gdn_args &g, std::vector<Range> &in, std::vector<Range> &out) {
    const int64_t C = 3 * g.H * g.D;
    in = {rng(g.x, C, 4),     rng(g.conv, C * g.K, 4),  rng(g.a, g.H, 4),  rng(g.b, g.H, 4),
          rng(g.z, g.H * g.D, 4), rng(g.A_log, g.H, 4), rng(g.dt_bias, g.H, 4), rng(g.nw, g.D, 4)};
    out = {rng(g.state, C * (g.K - 1), 4), rng(g.S, g.H * g.D * g.D, 4), rng(g.y, g.H * g.D, 4),
           rng(g.ysum, g.H * g.D / 64, 4)};
}

// the ranges an atq call reads and writes (the caches are read and written)
void atq_io(const abg_atq_args &t, std::vector<Range> &in, std::vector<Range> &out) {
    in = {rng(t.q, t.Hq * t.D, 4),  rng(t.gate, t.Hq * t.D, 4), rng(t.k, t.Hkv * t.D, 4),
          rng(t.v, t.Hkv * t.D, 4), rng(t.qn_w, t.D, 4),        rng(t.kn_w, t.D, 4),
          rng(t.cos, t.D / 2, 4),   rng(t.sin, t.D / 2, 4)};
    out = {rng(t.Kc, t.Hkv * t.P * t.D, 4), rng(t.Vc, t.Hkv * t.P * t.D, 4), rng(t.y, t.Hq * t.D, 4),
           rng(t.ysum, t.Hq * t.D / 64, 4)};
}

// no output overlaps an input or another output
abg_status disjoint_outputs(const std::vector<Range> &in, const std::vector<Range> &out) {
    for (size_t i = 0; i < out.size(); ++i) {
        for (const Range &r : in)
            if (overlap(out[i], r)) return ABG_EALIAS;
        for (size_t k = i + 1; k < out.size(); ++k)
            if (overlap(out[i], out[k])) return ABG_EALIAS;
    }
    return ABG_OK;
}

abg_status check_gdn(const abg_gdn_args &g, int mode) {
    if (mode != ABG_TREE && mode != ABG_FAST) return ABG_EINVAL;
    if (!g.x || !g.conv || !g.state || !g.a || !g.b || !g.z || !g.A_log || !g.dt_bias || !g.nw || !g.S || !g.y ||
        !g.ysum)
        return ABG_EINVAL;
    if (g.H < 1 || (g.D != 64 && g.D != 128 && g.D != 256) || g.K < 2 || g.K > 8 || g.H * g.D > (int64_t(1) << 20))
        return ABG_ESHAPE;
    const void *all[] = {g.x, g.conv, g.state, g.a, g.b, g.z, g.A_log, g.dt_bias, g.nw, g.S, g.y, g.ysum};
    for (const void *p : all)
        if (!aligned(p, 4)) return ABG_EALIGN;
    if (!aligned(g.S, 16)) return ABG_EALIGN;  // a head's state is one bulk copy
    std::vector<Range> in, out;
    gdn_io(g, in, out);
    return disjoint_outputs(in, out);
}

abg_status check_atq(const abg_atq_args &t, int mode) {
    if (mode != ABG_TREE && mode != ABG_FAST) return ABG_EINVAL;
    if (!t.q || !t.gate || !t.k || !t.v || !t.qn_w || !t.kn_w || !t.cos || !t.sin || !t.Kc || !t.Vc || !t.y ||
        !t.ysum)
        return ABG_EINVAL;
    if (t.Hq < 1 || t.Hkv < 1 || t.Hq % t.Hkv || (t.D != 64 && t.D != 128 && t.D != 256) || t.pos < 0 ||
        t.pos >= t.P || t.pos + 1 > 8192 || t.Hq * t.D > (int64_t(1) << 20))
        return ABG_ESHAPE;
    const void *all[] = {t.q, t.gate, t.k, t.v, t.qn_w, t.kn_w, t.cos, t.sin, t.Kc, t.Vc, t.y, t.ysum};
    for (const void *p : all)
        if (!aligned(p, 4)) return ABG_EALIGN;
    if (!aligned(t.Kc, 16) || !aligned(t.Vc, 16)) return ABG_EALIGN;  // cache rows are read as 16-byte units
    std::vector<Range> in, out;
    atq_io(t, in, out);
    return disjoint_outputs(in, out);
}

bool pdl_enabled();

cudaError_t run_gdn(const abg_gdn_args &g, cudaStream_t s, bool pdl) {
    return launch_gdn(g.x, g.conv, g.state, g.a, g.b, g.z, g.A_log, g.dt_bias, g.nw, g.S, g.y, g.ysum,
                      static_cast<int>(g.H), static_cast<int>(g.D), static_cast<int>(g.K), g.eps, g.eps_n, pdl, s);
}

cudaError_t run_atq(const abg_atq_args &t, float *scratch, cudaStream_t s, bool pdl) {
    return launch_atq(t.q, t.gate, t.k, t.v, t.qn_w, t.kn_w, t.cos, t.sin, t.Kc, t.Vc, t.y, t.ysum,
                      static_cast<int>(t.Hq), static_cast<int>(t.Hkv), static_cast<int>(t.D), static_cast<int>(t.P),
                      static_cast<int>(t.pos), t.eps, scratch, pdl, s);
}

// --------------------------------------------------------------- graphs ----
struct Launch {
    int kind;  // abg_node_kind
    int stage = 0;
    Q4Plan plan;
    std::vector<Q4Call> calls;  // the products of a Q4MV launch
    const float *a = nullptr, *b = nullptr;
    float *o = nullptr, *os = nullptr;
    float eps = 0.f;
    int64_t len = 0;
    int group = 64;
    abg_gdn_args gdn{};
    abg_atq_args atq{};
    float *atq_scratch = nullptr;  // owned by the graph
};

struct StageGraph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int64_t launches = 0;
    int64_t swiglu_pairs = 0;
    std::vector<void *> scratch;  // device buffers: fused SwiGLU vectors, atq chunk results
};

void free_scratch(StageGraph *g) {
    for (void *p : g->scratch) cudaFree(p);
    g->scratch.clear();
}

// SwiGLU pairs.  A product launch D whose activation is the SwiGLU of a =
// [gate | up] (the SwiGLU prologue), right after a launch GU of the previous
// stage that holds exactly the two products writing a[0, n) (gate) and
// a[n, 2n) (up), gets that vector from GU's epilogue: each of GU's tiles holds
// the same rows of both products, and the warp that finishes a gate row and
// its up row writes silu(gate) * up, once per element, into a buffer the graph
// owns; D reads it with the group-sum prologue instead of recomputing the
// SwiGLU in every thread block.  Both write the same outputs as before, bit
// for bit (the same SwiGLU of the same values, the same group-sum tree).  Only
// launches planned with a fixed shape and 4 rows per item are paired.
abg_status fuse_swiglu_pairs(std::vector<Launch> &launches, StageGraph *g, int mode, int rpw) {
    for (size_t d = 1; d < launches.size(); ++d) {
        Launch &D = launches[d], &GU = launches[d - 1];
        if (D.kind != ABG_NODE_Q4MV || D.calls.empty() || D.calls[0].prologue != kProSwq) continue;
        if (GU.kind != ABG_NODE_Q4MV || GU.calls.size() != 2 || GU.stage + 1 != D.stage) continue;
        const float *a = D.calls[0].x;
        const int64_t n = D.calls[0].cols;
        if (D.calls[0].group != 64) continue;
        int gi = -1, ui = -1;
        for (int i = 0; i < 2; ++i) {
            const Q4Call &c = GU.calls[i];
            if (c.n != n) continue;
            if (c.y == a) gi = i;
            if (c.y == a + n) ui = i;
        }
        if (gi < 0 || ui < 0 || gi == ui) continue;
        Q4Plan pair_plan;
        const std::vector<Q4Call> gu = {GU.calls[gi], GU.calls[ui]};
        if (plan_calls(&pair_plan, gu, mode, rpw) != ABG_OK || pair_plan.shape == 0 || pair_plan.rows_per_warp != 4)
            continue;
        void *o = nullptr;
        const cudaError_t e = cudaMalloc(&o, static_cast<size_t>(n) * sizeof(float));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc (SwiGLU vector)");
        g->scratch.push_back(o);
        std::vector<Q4Call> dc = D.calls;
        for (Q4Call &c : dc) {
            c.prologue = kProGsum;
            c.x = static_cast<const float *>(o);
        }
        Q4Plan d_plan;
        const abg_status st = plan_calls(&d_plan, dc, mode, rpw);
        if (st != ABG_OK) return st;
        // a tile holds tile_rows/2 rows of each product
        Q4Args &pa = pair_plan.args;
        pa.paired = 1;
        pa.epi = static_cast<float *>(o);
        const int64_t half_rows = pa.tile_rows / 2;
        pa.total_tiles = (n + half_rows - 1) / half_rows;
        pair_plan.grid.x = static_cast<unsigned>(std::min<int64_t>(pair_plan.grid.x, pa.total_tiles));
        GU.plan = pair_plan;
        GU.calls = gu;
        D.plan = d_plan;
        D.calls = dc;
        ++g->swiglu_pairs;
    }
    return ABG_OK;
}

cudaError_t prepare(const Launch &L) {
    if (L.kind == ABG_NODE_GDN) return prepare_gdn(static_cast<int>(L.gdn.D));
    if (L.kind == ABG_NODE_ATQ)
        return prepare_atq(static_cast<int>(L.atq.Hq), static_cast<int>(L.atq.Hkv), static_cast<int>(L.atq.D));
    if (L.kind != ABG_NODE_Q4MV) return cudaSuccess;
    return prepare_q4mv(L.plan);
}

// The mixers' launches start early like the products' (programmatic
// dependent launch): gdn reads every input after its wait; atq's first
// launch reads only its own key cache rows before it (no other node writes
// them).  No launch starts early after a copy (`after_copy`): early start
// overlaps a kernel with the kernel before it only.
cudaError_t run(const Launch &L, cudaStream_t s, bool pdl, bool tree, bool after_copy) {
    switch (L.kind) {
    case ABG_NODE_Q4MV: return launch_q4mv(L.plan, s, pdl);
    case ABG_NODE_GDN: return run_gdn(L.gdn, s, pdl_enabled() && !after_copy);
    case ABG_NODE_ATQ: return run_atq(L.atq, L.atq_scratch, s, pdl_enabled() && !after_copy);
    case ABG_NODE_COPY:
        return cudaMemcpyAsync(L.o, L.a, static_cast<size_t>(L.len) * sizeof(float), cudaMemcpyDefault, s);
    case ABG_NODE_RMSQ: return launch_rmsq(L.a, L.b, L.eps, L.o, L.os, L.len, L.group, tree, s, pdl);
    case ABG_NODE_SWQ: return launch_swq(L.a, L.o, L.os, L.len, L.group, tree, s, pdl);
    default: return launch_gsum(L.a, L.os, L.len, L.group, tree, s, pdl);
    }
}

Q4Call call_of(const abg_node &nd) {
    Q4Call c;
    c.w = nd.w;
    c.scale = nd.scale;
    c.bias = nd.bias;
    c.rows = nd.rows;
    c.cols = nd.cols;
    c.row0 = nd.row0;
    c.n = nd.n;
    c.y = nd.y;
    c.prologue = nd.prologue;
    c.x = nd.x;
    c.xsum = nd.xsum;
    c.wt = nd.wt;
    c.eps = nd.eps;
    c.group = node_group(nd.group);
    c.sb_type = nd.sb_type;
    return c;
}

void node_io(const abg_node &nd, std::vector<Range> &in, std::vector<Range> &out) {
    switch (nd.kind) {
    case ABG_NODE_Q4MV: {
        const Q4Call c = call_of(nd);
        in = q4_inputs(c);
        out = {rng(c.y, c.n, 4)};
        break;
    }
    case ABG_NODE_RMSQ:
        in = {rng(nd.x, nd.len, 4), rng(nd.wt, nd.len, 4)};
        out = {rng(nd.out, nd.len, 4), rng(nd.out_sum, nd.len / node_group(nd.group), 4)};
        break;
    case ABG_NODE_SWQ:
        in = {rng(nd.x, 2 * nd.len, 4)};
        out = {rng(nd.out, nd.len, 4), rng(nd.out_sum, nd.len / node_group(nd.group), 4)};
        break;
    case ABG_NODE_GDN: gdn_io(*static_cast<const abg_gdn_args *>(nd.args), in, out); break;
    case ABG_NODE_ATQ: atq_io(*static_cast<const abg_atq_args *>(nd.args), in, out); break;
    case ABG_NODE_COPY:
        in = {rng(nd.x, nd.len, 4)};
        out = {rng(nd.out, nd.len, 4)};
        break;
    default:
        in = {rng(nd.x, nd.len, 4)};
        out = {rng(nd.out_sum, nd.len / node_group(nd.group), 4)};
        break;
    }
}

// one grouped launch: same activation, same format, same scale/bias staging
bool same_activation(const Q4Call &a, const Q4Call &b) {
    return a.prologue == b.prologue && a.cols == b.cols && a.x == b.x && a.group == b.group &&
           a.sb_type == b.sb_type &&
           (a.prologue != kProNone || a.xsum == b.xsum) && (a.prologue != kProRmsq || (a.wt == b.wt && a.eps == b.eps)) &&
           sb_bulk(a) == sb_bulk(b);
}

// ------------------------------------------------- allocation-free MLP ----
// abg_swiglu_mlp_static keeps its intermediate vectors in this array instead
// of memory it would have to allocate: the gate outputs, the up outputs and
// their SwiGLU, kMlpMaxHidden floats each (192 KB).  Every device that loads
// the library holds one copy until the process exits.  In host code the
// name is only a stand-in for the device symbol: its device address comes
// from cudaGetSymbolAddress, once per device (mlp_scratch below).
constexpr int64_t kMlpMaxHidden = 16384;
static __device__ __align__(256) float g_mlp_scratch[3 * kMlpMaxHidden];

std::mutex g_mlp_mu;
constexpr int kMlpMaxDevices = 64;
float *g_mlp_ptr[kMlpMaxDevices] = {};

// The device address of g_mlp_scratch on the current device (looked up on
// the first call per device, with that device current).
abg_status mlp_scratch(float **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMlpMaxDevices) return ABG_EINVAL;
    std::lock_guard<std::mutex> lock(g_mlp_mu);
    if (!g_mlp_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_mlp_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress (MLP scratch)");
        g_mlp_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_mlp_ptr[dev];
    return ABG_OK;
}

// ABG_PDL=0: plain stream-ordered launches (no early start of a dependent
// launch) in stage graphs and between the launches of one batched call;
// results are the same.
bool pdl_enabled() {
    static const bool on = [] {
        const char *v = std::getenv("ABG_PDL");
        return !(v && std::strcmp(v, "0") == 0);
    }();
    return on;
}

}  // namespace

extern "C" {

abg_status abg_q4mv(const uint32_t *w, const float *scale, const float *bias, const float *x, const float *xsum,
                    float *y, int64_t rows, int64_t cols, int64_t row0, int64_t n, int mode, int rows_per_warp,
                    void *stream) {
    return abg_q4mv_ex(w, scale, bias, ABG_SB_F32, 64, x, xsum, y, rows, cols, row0, n, mode, rows_per_warp, stream);
}

abg_status abg_q4mv_ex(const uint32_t *w, const void *scale, const void *bias, int sb_type, int group, const float *x,
                       const float *xsum, float *y, int64_t rows, int64_t cols, int64_t row0, int64_t n, int mode,
                       int rows_per_warp, void *stream) {
    Q4Call c{w, scale, bias, rows, cols, row0, n, y, kProNone, x, xsum, nullptr, 0.f, group, sb_type};
    abg_status st = check_q4(c, mode, rows_per_warp);
    if (st != ABG_OK || n == 0) return st;
    Q4Plan plan;
    st = plan_calls(&plan, {c}, mode, rows_per_warp);
    if (st != ABG_OK) return st;
    cudaError_t e = prepare_q4mv(plan);
    if (e != cudaSuccess) return cuda_fail(e, "kernel attributes");
    return cuda_fail(launch_q4mv(plan, static_cast<cudaStream_t>(stream), false), "q4mv launch");
}

abg_status abg_q4mm(const uint32_t *w, const float *scale, const float *bias, const float *x, const float *xsum,
                    float *y, int64_t rows, int64_t cols, int64_t row0, int64_t n, int64_t T, int mode,
                    int rows_per_warp, void *stream) {
    if (T < 1 || T > 8) return ABG_EINVAL;
    // token 0 validates the matrix, row range, pointers and alignment
    Q4Call c{w, scale, bias, rows, cols, row0, n, y, kProNone, x, xsum, nullptr, 0.f};
    abg_status st = check_q4(c, mode, rows_per_warp);
    if (st != ABG_OK || n == 0) return st;
    // y [T][n] overlaps no input, x [T][cols] or xsum [T][cols/64] included
    const Range out = rng(y, T * n, 4);
    Q4Call all = c;
    const int64_t G = cols / 64;
    std::vector<Range> in = q4_weights(all);
    in.push_back(rng(x, T * cols, 4));
    in.push_back(rng(xsum, T * G, 4));
    for (const Range &r : in)
        if (overlap(out, r)) return ABG_EALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The first launch waits for the work queued before the call; the later
    // ones share its inputs and write other outputs, so they may start early
    // (programmatic launch) without waiting for it.
    const bool pdl = pdl_enabled();
    for (int64_t t0 = 0; t0 < T;) {
        // four tokens share a launch on rows of 2048 columns with staged
        // scale and bias, otherwise pairs; an odd last token runs alone
        int width = (T - t0 >= 2) ? 2 : 1;
        if (T - t0 >= 4 && cols == 2048 && sb_bulk(c)) width = 4;
        const bool sibling = pdl && t0 > 0;
        const int ntok = width;
        Q4Call ct = c;
        ct.x = x + t0 * cols;
        ct.xsum = xsum + t0 * G;
        ct.y = y + t0 * n;
        Q4Plan plan;
        if (width == 1) {
            st = plan_calls(&plan, {ct}, mode, rows_per_warp);
            if (st != ABG_OK) return st;
            if (sibling) plan.args.wait_first = 0;
            cudaError_t e = prepare_q4mv(plan);
            if (e == cudaSuccess) e = launch_q4mv(plan, s, sibling);
            if (e != cudaSuccess) return cuda_fail(e, "q4mm launch");
        } else {
            const float *xt[4], *xst[4];
            for (int i = 0; i < ntok; ++i) {
                xt[i] = ct.x + i * cols;
                xst[i] = ct.xsum + i * G;
            }
            Q4Prob p = make_prob(ct);
            if (!plan_q4mm(&plan, &p, 1, static_cast<int>(cols), width, ntok, xt, xst, kProNone, mode == ABG_TREE,
                           rows_per_warp == 0 ? 8 : rows_per_warp, sb_bulk(ct)))
                return ABG_ESHAPE;
            if (sibling) plan.args.wait_first = 0;
            const cudaError_t e = launch_q4mm(plan, s, sibling);
            if (e != cudaSuccess) return cuda_fail(e, "q4mm launch");
        }
        t0 += ntok;
    }
    return ABG_OK;
}

abg_status abg_gsum(const float *v, float *s, int64_t n, int mode, void *stream) {
    return abg_gsum_ex(v, s, n, 64, mode, stream);
}

abg_status abg_gsum_ex(const float *v, float *s, int64_t n, int group, int mode, void *stream) {
    abg_status st = check_gsum(v, s, n, group, mode);
    if (st != ABG_OK) return st;
    return cuda_fail(launch_gsum(v, s, n, group, mode == ABG_TREE, static_cast<cudaStream_t>(stream), false));
}

abg_status abg_rmsq(const float *x, const float *wt, float eps, float *xn, float *xsum, int64_t n, int mode,
                    void *stream) {
    return abg_rmsq_ex(x, wt, eps, xn, xsum, n, 64, mode, stream);
}

abg_status abg_rmsq_ex(const float *x, const float *wt, float eps, float *xn, float *xsum, int64_t n, int group,
                       int mode, void *stream) {
    abg_status st = check_rmsq(x, wt, xn, xsum, n, group, mode);
    if (st != ABG_OK) return st;
    return cuda_fail(
        launch_rmsq(x, wt, eps, xn, xsum, n, group, mode == ABG_TREE, static_cast<cudaStream_t>(stream), false));
}

abg_status abg_swq(const float *a, float *o, float *osum, int64_t n, int mode, void *stream) {
    return abg_swq_ex(a, o, osum, n, 64, mode, stream);
}

abg_status abg_swq_ex(const float *a, float *o, float *osum, int64_t n, int group, int mode, void *stream) {
    abg_status st = check_swq(a, o, osum, n, group, mode);
    if (st != ABG_OK) return st;
    return cuda_fail(launch_swq(a, o, osum, n, group, mode == ABG_TREE, static_cast<cudaStream_t>(stream), false));
}

abg_status abg_gdn(const float *x, const float *conv, float *state, const float *a, const float *b, const float *z,
                   const float *A_log, const float *dt_bias, const float *nw, float *S, float *y, float *ysum,
                   int64_t H, int64_t D, int64_t K, float eps, float eps_n, int mode, void *stream) {
    const abg_gdn_args g{x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, H, D, K, eps, eps_n};
    const abg_status st = check_gdn(g, mode);
    if (st != ABG_OK) return st;
    return cuda_fail(run_gdn(g, static_cast<cudaStream_t>(stream), pdl_enabled()), "gdn launch");
}

abg_status abg_atq(const float *q, const float *gate, const float *k, const float *v, const float *qn_w,
                   const float *kn_w, const float *cos, const float *sin, float *Kc, float *Vc, float *y, float *ysum,
                   int64_t Hq, int64_t Hkv, int64_t D, int64_t P, int64_t pos, float eps, int mode, void *stream) {
    const abg_atq_args t{q, gate, k, v, qn_w, kn_w, cos, sin, Kc, Vc, y, ysum, Hq, Hkv, D, P, pos, eps};
    const abg_status st = check_atq(t, mode);
    if (st != ABG_OK) return st;
    return cuda_fail(run_atq(t, nullptr, static_cast<cudaStream_t>(stream), pdl_enabled()), "atq launch");
}

abg_status abg_stage_graph_create(const abg_node *nodes, int64_t count, int mode, int rows_per_warp,
                                  void **graph_out) {
    if (!graph_out) return ABG_EINVAL;
    *graph_out = nullptr;
    if (!nodes || count <= 0) return ABG_EINVAL;
    if (mode != ABG_TREE && mode != ABG_FAST) return ABG_EINVAL;
    if (rows_per_warp != 0 && rows_per_warp != 1 && rows_per_warp != 2 && rows_per_warp != 4 && rows_per_warp != 8)
        return ABG_EINVAL;
    // 1. every node on its own
    for (int64_t i = 0; i < count; ++i) {
        const abg_node &nd = nodes[i];
        abg_status st;
        switch (nd.kind) {
        case ABG_NODE_Q4MV: st = check_q4(call_of(nd), mode, rows_per_warp); break;
        case ABG_NODE_RMSQ: st = check_rmsq(nd.x, nd.wt, nd.out, nd.out_sum, nd.len, node_group(nd.group), mode); break;
        case ABG_NODE_SWQ: st = check_swq(nd.x, nd.out, nd.out_sum, nd.len, node_group(nd.group), mode); break;
        case ABG_NODE_GSUM: st = check_gsum(nd.x, nd.out_sum, nd.len, node_group(nd.group), mode); break;
        case ABG_NODE_GDN:
            st = nd.args ? check_gdn(*static_cast<const abg_gdn_args *>(nd.args), mode) : ABG_EINVAL;
            break;
        case ABG_NODE_ATQ:
            st = nd.args ? check_atq(*static_cast<const abg_atq_args *>(nd.args), mode) : ABG_EINVAL;
            break;
        case ABG_NODE_COPY: st = check_copy(nd.x, nd.out, nd.len); break;
        default: st = ABG_EINVAL;
        }
        if (st != ABG_OK) return st;
    }
    // 2. stages: no node reads or writes what another node of its stage writes,
    //    and no node writes any product's weights or RMS-norm prologue weights
    //    (they are fetched before the wait for the previous stage)
    std::map<int, std::vector<int64_t>> stages;
    for (int64_t i = 0; i < count; ++i) stages[nodes[i].stage].push_back(i);
    std::vector<std::vector<Range>> ins(count), outs(count);
    for (int64_t i = 0; i < count; ++i) node_io(nodes[i], ins[i], outs[i]);
    for (auto &kv : stages) {
        const auto &idx = kv.second;
        for (int64_t i : idx)
            for (int64_t j : idx) {
                if (i == j) continue;
                for (const Range &o : outs[i]) {
                    for (const Range &r : ins[j])
                        if (overlap(o, r)) return ABG_EALIAS;
                    for (const Range &r : outs[j])
                        if (overlap(o, r)) return ABG_EALIAS;
                }
            }
    }
    for (int64_t i = 0; i < count; ++i) {
        if (nodes[i].kind != ABG_NODE_Q4MV || nodes[i].n == 0) continue;
        std::vector<Range> wr = q4_weights(call_of(nodes[i]));
        // an RMS-norm prologue's weights are read early too
        if (nodes[i].prologue == ABG_PRO_RMSQ) wr.push_back(rng(nodes[i].wt, nodes[i].cols, 4));
        for (int64_t j = 0; j < count; ++j)
            for (const Range &o : outs[j])
                for (const Range &r : wr)
                    if (overlap(o, r)) return ABG_EALIAS;
    }
    // an atq node reads its key cache rows before waiting for the launch
    // before it: no other node writes its caches
    for (int64_t i = 0; i < count; ++i) {
        if (nodes[i].kind != ABG_NODE_ATQ) continue;
        const Range caches[2] = {outs[i][0], outs[i][1]};  // Kc, Vc (atq_io's first two outputs)
        for (int64_t j = 0; j < count; ++j) {
            if (j == i) continue;
            for (const Range &o : outs[j])
                for (const Range &r : caches)
                    if (overlap(o, r)) return ABG_EALIAS;
        }
    }
    // 3. launches: stage by stage; products of a stage that share their
    //    activation become one grouped launch
    std::vector<Launch> launches;
    for (auto &kv : stages) {
        std::vector<bool> used(kv.second.size(), false);
        for (size_t a = 0; a < kv.second.size(); ++a) {
            if (used[a]) continue;
            const abg_node &nd = nodes[kv.second[a]];
            used[a] = true;
            Launch L;
            L.kind = nd.kind;
            L.stage = kv.first;
            if (nd.kind == ABG_NODE_Q4MV) {
                if (nd.n == 0) continue;
                std::vector<Q4Call> group = {call_of(nd)};
                for (size_t b = a + 1; b < kv.second.size() && group.size() < static_cast<size_t>(kMaxProbs); ++b) {
                    const abg_node &nb = nodes[kv.second[b]];
                    if (used[b] || nb.kind != ABG_NODE_Q4MV || nb.n == 0) continue;
                    const Q4Call cb = call_of(nb);
                    if (!same_activation(group[0], cb)) continue;
                    group.push_back(cb);
                    used[b] = true;
                }
                abg_status st = plan_calls(&L.plan, group, mode, rows_per_warp);
                if (st != ABG_OK) return st;
                L.calls = group;
            } else if (nd.kind == ABG_NODE_GDN) {
                L.gdn = *static_cast<const abg_gdn_args *>(nd.args);
            } else if (nd.kind == ABG_NODE_ATQ) {
                L.atq = *static_cast<const abg_atq_args *>(nd.args);
            } else {
                L.a = nd.x;
                L.b = nd.wt;
                L.o = nd.out;
                L.os = nd.out_sum;
                L.eps = nd.eps;
                L.len = nd.len;
                L.group = node_group(nd.group);
            }
            launches.push_back(L);
        }
    }
    auto *g = new StageGraph();
    for (const Launch &L : launches) g->launches += L.kind == ABG_NODE_COPY ? 0 : (L.kind == ABG_NODE_ATQ ? 4 : 1);
    {
        const abg_status st = fuse_swiglu_pairs(launches, g, mode, rows_per_warp);
        if (st != ABG_OK) {
            free_scratch(g);
            delete g;
            return st;
        }
    }
    cudaError_t e = cudaSuccess;
    std::string where;
    // each atq launch gets its own buffer for the chunk results
    for (Launch &L : launches) {
        if (L.kind != ABG_NODE_ATQ || e != cudaSuccess) continue;
        void *p = nullptr;
        const size_t bytes = atq_scratch_bytes(static_cast<int>(L.atq.Hq), static_cast<int>(L.atq.D),
                                               static_cast<int>(L.atq.pos));
        if ((e = cudaMalloc(&p, bytes)) != cudaSuccess) {
            where = "cudaMalloc (atq chunk results)";
            break;
        }
        g->scratch.push_back(p);
        L.atq_scratch = static_cast<float *>(p);
    }
    for (const Launch &L : launches)
        if (e == cudaSuccess && (e = prepare(L)) != cudaSuccess) where = "kernel attributes";
    cudaStream_t cs = nullptr;
    if (e == cudaSuccess && (e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking)) != cudaSuccess)
        where = "cudaStreamCreateWithFlags";
    if (e == cudaSuccess && (e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal)) != cudaSuccess)
        where = "cudaStreamBeginCapture";
    const bool pdl_on = pdl_enabled();
    // a product launch that follows a launch of its own stage does not depend
    // on it (siblings of one stage share their inputs)
    for (size_t i = 1; i < launches.size(); ++i)
        if (launches[i].kind == ABG_NODE_Q4MV && launches[i].stage == launches[i - 1].stage)
            launches[i].plan.args.wait_first = 0;
    if (e == cudaSuccess) {
        for (size_t i = 0; i < launches.size() && e == cudaSuccess; ++i) {
            const bool after_copy = i > 0 && launches[i - 1].kind == ABG_NODE_COPY;
            if ((e = run(launches[i], cs, pdl_on && i > 0 && !after_copy, mode == ABG_TREE, after_copy)) !=
                cudaSuccess)
                where = "launch " + std::to_string(i) + " (kind " + std::to_string(launches[i].kind) + ")";
        }
        cudaGraph_t graph = nullptr;
        const cudaError_t e2 = cudaStreamEndCapture(cs, &graph);
        if (e == cudaSuccess && (e = e2) != cudaSuccess) where = "cudaStreamEndCapture";
        g->graph = graph;
    }
    if (e == cudaSuccess && (e = cudaGraphInstantiate(&g->exec, g->graph, 0)) != cudaSuccess)
        where = "cudaGraphInstantiate";
    if (cs) cudaStreamDestroy(cs);
    if (e != cudaSuccess) {
        if (g->exec) cudaGraphExecDestroy(g->exec);
        if (g->graph) cudaGraphDestroy(g->graph);
        free_scratch(g);
        delete g;
        cudaGetLastError();
        return cuda_fail(e, where.c_str());
    }
    {
        std::lock_guard<std::mutex> lock(g_graphs_mu);
        g_graphs.insert(g);
    }
    *graph_out = g;
    return ABG_OK;
}

abg_status abg_stage_graph_launch(void *graph, void *stream) {
    if (!graph_live(graph)) return ABG_EINVAL;
    auto *g = static_cast<StageGraph *>(graph);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    static const bool trace = [] {
        const char *v = std::getenv("ABG_TRACE");
        return v && std::strcmp(v, "1") == 0;
    }();
    if (!trace) return cuda_fail(cudaGraphLaunch(g->exec, s));
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    const auto t0 = std::chrono::steady_clock::now();
    if (e == cudaSuccess) e = cudaEventRecord(e0, s);
    if (e == cudaSuccess) e = cudaGraphLaunch(g->exec, s);
    if (e == cudaSuccess) e = cudaEventRecord(e1, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    const auto t1 = std::chrono::steady_clock::now();
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (e == cudaSuccess)
        std::fprintf(stderr, "abg: stage graph %lld launches, GPU %.3f ms, wall %.3f ms\n",
                     static_cast<long long>(g->launches), ms,
                     std::chrono::duration<double, std::milli>(t1 - t0).count());
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    return cuda_fail(e);
}

abg_status abg_stage_graph_launches(void *graph, int64_t *launches) {
    if (!graph_live(graph) || !launches) return ABG_EINVAL;
    *launches = static_cast<StageGraph *>(graph)->launches;
    return ABG_OK;
}

abg_status abg_stage_graph_swiglu_pairs(void *graph, int64_t *pairs) {
    if (!graph_live(graph) || !pairs) return ABG_EINVAL;
    *pairs = static_cast<StageGraph *>(graph)->swiglu_pairs;
    return ABG_OK;
}

abg_status abg_stage_graph_destroy(void *graph) {
    {
        std::lock_guard<std::mutex> lock(g_graphs_mu);
        if (!graph || g_graphs.erase(graph) == 0) return ABG_EINVAL;
    }
    auto *g = static_cast<StageGraph *>(graph);
    cudaError_t e = cudaSuccess;
    if (g->exec) e = cudaGraphExecDestroy(g->exec);
    if (g->graph) {
        const cudaError_t e2 = cudaGraphDestroy(g->graph);
        if (e == cudaSuccess) e = e2;
    }
    free_scratch(g);
    delete g;
    return cuda_fail(e);
}

abg_status abg_selftest_wait_timeout(void *stream) {
    // one 64x1024 product whose producer withholds its only tile; the
    // computing warps touch no memory before that wait, so no pointer is read
    Q4Prob p = {};
    p.n = 64;
    Q4Plan plan;
    Q4Tuning none;
    if (!plan_q4mv(&plan, &p, 1, 1024, 64, ABG_SB_F32, kProNone, nullptr, nullptr, nullptr, 0.f, true, 8, false,
                   none))
        return ABG_ESHAPE;
    plan.args.withhold = 1;
    cudaError_t e = prepare_q4mv(plan);
    if (e != cudaSuccess) return cuda_fail(e, "kernel attributes");
    return cuda_fail(launch_q4mv(plan, static_cast<cudaStream_t>(stream), false), "self-test launch");
}

abg_status abg_device_status(uint32_t *bits, int clear) {
    if (!bits) return ABG_EINVAL;
    *bits = 0;
    cudaError_t e = cudaDeviceSynchronize();
    unsigned v = 0;
    if (e == cudaSuccess) e = q4mv_status(&v, clear != 0);
    if (e == cudaSuccess) e = vec_status(&v, clear != 0);
    if (e == cudaSuccess) e = q4mm_status(&v, clear != 0);
    if (e == cudaSuccess) e = mixer_status(&v, clear != 0);
    if (e != cudaSuccess) return cuda_fail(e);
    *bits = v;
    return (v & 1u) ? ABG_ETIMEOUT : ABG_OK;  // bit 0: a bounded wait timed out
}

abg_status abg_set_q4mv_tuning(int smem_kb, int consumer_warps, int blocks_per_sm, int stage_kb) {
    if (smem_kb < 0 || smem_kb > 227 || consumer_warps < 0 || consumer_warps > 16 || blocks_per_sm < 0 ||
        blocks_per_sm > 4 || stage_kb < 0 || stage_kb > 200)
        return ABG_EINVAL;
    g_tuning.smem_kb = smem_kb;
    g_tuning.consumer_warps = consumer_warps;
    g_tuning.blocks_per_sm = blocks_per_sm;
    g_tuning.stage_kb = stage_kb;
    return ABG_OK;
}

const char *abg_status_str(int status) {
    switch (status) {
    case ABG_OK: return "ok";
    case ABG_EINVAL: return "invalid argument";
    case ABG_EALIGN: return "misaligned pointer";
    case ABG_ESHAPE: return "bad shape";
    case ABG_EALIAS: return "output overlaps an input";
    case ABG_ECUDA: return "CUDA error";
    case ABG_ETIMEOUT: return "device wait timed out";
    default: return "unknown status";
    }
}

const char *abg_last_cuda_error(void) { return g_cuda_error.c_str(); }

abg_status abg_swiglu_mlp_static(const uint32_t *wg, const float *sg, const float *bg, const uint32_t *wu,
                                 const float *su, const float *bu, const uint32_t *wd, const float *sd,
                                 const float *bd, const float *x, const float *xsum, float *y, int64_t n,
                                 int64_t cols, int64_t rows, int mode, void *stream) {
    // Checked before any device work (this call allocates no device memory
    // and takes no buffer from the caller for its intermediate vectors).
    if (mode != ABG_TREE && mode != ABG_FAST) return ABG_EINVAL;
    if (n <= 0 || n % 64 != 0) return ABG_ESHAPE;
    if (n > kMlpMaxHidden) return ABG_ESHAPE;  // larger than the static scratch
    if (cols <= 0 || cols % 64 != 0 || cols > ABG_MAX_COLS || rows < 0) return ABG_ESHAPE;
    if (rows == 0) return ABG_OK;
    if (!wg || !sg || !bg || !wu || !su || !bu || !wd || !sd || !bd || !x || !xsum || !y) return ABG_EINVAL;
    const void *a16[] = {wg, wu, wd, x};
    for (const void *q : a16)
        if (!aligned(q, 16)) return ABG_EALIGN;
    const void *a4[] = {sg, bg, su, bu, sd, bd, xsum, y};
    for (const void *q : a4)
        if (!aligned(q, 4)) return ABG_EALIGN;
    const int64_t G = cols / 64, Gd = n / 64;
    const Range ins[] = {rng(wg, n * (cols / 8), 4), rng(sg, n * G, 4), rng(bg, n * G, 4),
                         rng(wu, n * (cols / 8), 4), rng(su, n * G, 4), rng(bu, n * G, 4),
                         rng(wd, rows * (n / 8), 4), rng(sd, rows * Gd, 4), rng(bd, rows * Gd, 4),
                         rng(x, cols, 4),           rng(xsum, G, 4)};
    const Range out = rng(y, rows, 4);
    for (const Range &r : ins)
        if (overlap(out, r)) return ABG_EALIAS;
    float *sp = nullptr;
    abg_status st = mlp_scratch(&sp);
    if (st != ABG_OK) return st;
    // scratch: gate outputs [0, n), up outputs [n, 2n), SwiGLU [2n, 3n);
    // every element is written before it is read, so nothing is cleared
    const Q4Call gc{wg, sg, bg, n, cols, 0, n, sp, kProNone, x, xsum, nullptr, 0.f};
    const Q4Call uc{wu, su, bu, n, cols, 0, n, sp + n, kProNone, x, xsum, nullptr, 0.f};
    const bool tree = mode == ABG_TREE;
    Q4Prob probs[2] = {make_prob(gc), make_prob(uc)};
    Q4Plan pu, pd;
    if (!plan_q4mv(&pu, probs, 2, static_cast<int>(cols), 64, ABG_SB_F32, kProNone, x, xsum, nullptr, 0.f, tree, 0,
                   sb_bulk(gc) && sb_bulk(uc), g_tuning))
        return ABG_ESHAPE;
    Q4Call dc{wd, sd, bd, rows, n, 0, rows, y, kProSwq, sp, nullptr, nullptr, 0.f};
    if (pu.shape != 0 && pu.rows_per_warp == 4) {
        // the gate/up launch writes the SwiGLU itself (a tile holds the same
        // rows of both products) and the down product reads it with the
        // group-sum prologue
        Q4Args &pa = pu.args;
        pa.paired = 1;
        pa.epi = sp + 2 * n;
        const int64_t half_rows = pa.tile_rows / 2;
        pa.total_tiles = (n + half_rows - 1) / half_rows;
        pu.grid.x = static_cast<unsigned>(std::min<int64_t>(pu.grid.x, pa.total_tiles));
        dc.prologue = kProGsum;
        dc.x = sp + 2 * n;
    }  // else the down product computes the SwiGLU of [gate | up] in its prologue
    Q4Prob pdown = make_prob(dc);
    if (!plan_q4mv(&pd, &pdown, 1, static_cast<int>(n), 64, ABG_SB_F32, dc.prologue, dc.x, nullptr, nullptr, 0.f, tree,
                   0, sb_bulk(dc), g_tuning))
        return ABG_ESHAPE;
    cudaError_t e = prepare_q4mv(pu);
    if (e == cudaSuccess) e = prepare_q4mv(pd);
    if (e != cudaSuccess) return cuda_fail(e, "kernel attributes");
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((e = launch_q4mv(pu, s, false)) != cudaSuccess) return cuda_fail(e, "gate/up launch");
    return cuda_fail(launch_q4mv(pd, s, false), "down launch");
}

}  // extern "C"
