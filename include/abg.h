/*
 * abg.h -- C ABI of the GB300 (sm_103a) affine 4-bit group-quantized
 * matrix-vector product and its two activation producers.
 *
 * The operation comes from three Bend pull-request pages by one author:
 *   [q4mv-metal]  "Array.q4mv on Metal: one kernel thread per row for products
 *                 of 4M weights or more, bit-identical" (bendlang/bend #1435)
 *   [q4go]        "Array.q4go/Array.q4wait queue Metal Q4 products in one
 *                 command buffer and wait once on a flag" (#1437)
 *   [fused-token] "Metal: queued rmsq, swq, gdn and atq kernels and a 4-row
 *                 q4mv, so a decode token is one command buffer with one wait"
 *                 (#1440)
 *
 * Weight format ([fused-token] Why and Change; [q4go] Verification): MLX-style
 * 4-bit affine weights, w = scale*q + bias with q in 0..15, in groups of 64
 * columns.  q is packed 8 nibbles per u32: column 8k+j of a row is bits
 * 4j..4j+3 of word k (low nibble first).  scale and bias are f32, one per row
 * and 64-column group.  The product reads the activation x together with its
 * 64-value group sums xsum, so that
 *
 *     y[r] = sum_g ( scale[r][g] * sum_j q[r][64g+j] * x[64g+j]
 *                    + bias[r][g] * xsum[g] ).
 *
 * Modes.  ABG_TREE reproduces a fixed summation order bit for bit ([fused-token]
 * Change, bend_q4mv bullet: "sums in a fixed tree order").  Every sum is a
 * balanced pairwise tree in index order: at each level elements (2i, 2i+1)
 * are added and an odd last element is carried up unchanged.  Products are
 * rounded once (RN binary32), the affine term is RN(RN(scale*d) + RN(bias*xsum))
 * without fused multiply-add, and each row's group terms are summed by the
 * same tree.  ABG_FAST may reorder and contract; its outputs stay within
 * 1e-5 * max(|y|, sum_g |scale*d| + |bias*xsum|) of the tree result.
 *
 * Conventions shared by every call:
 *   - Pointers are DEVICE pointers owned by the caller (the library allocates
 *     nothing per call).  Packed weights and every vector read in pairs
 *     (x, wt, a, and the xn / o outputs) must be 16-byte aligned; group sums,
 *     scale, bias and y 4-byte aligned (else ABG_EALIGN).  scale and bias
 *     rows are streamed with bulk copies when both are 16-byte aligned and
 *     cols is a multiple of 256, and read with ordinary loads otherwise.
 *   - Calls are asynchronous: they enqueue on `stream` (a cudaStream_t, NULL =
 *     the legacy default stream) and return.  The caller synchronizes.
 *   - Lifetime ([q4go] Change, last paragraph; Limits): every buffer a call
 *     reads or writes must stay allocated and unmodified by others until the
 *     stream work has completed.  Freeing w early was seen to corrupt row 0.
 *   - An output may not overlap any input of the same call (else ABG_EALIAS):
 *     concurrent products must not read one another's y ([q4go] Change).
 *   - Lengths that are not whole 64-value groups are rejected (ABG_ESHAPE).
 *     The pages' GPU kernels silently left such outputs untouched
 *     ([fused-token] reviewer reply); here it is an error.
 *   - A device-side wait that exceeds its time limit (0.5 s) stops the
 *     kernel and sets a bit in the library's device status word; read it with
 *     abg_device_status().  No call hangs the GPU.
 */
#ifndef ABG_H
#define ABG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ABG_OK = 0,
    ABG_EINVAL = 1,   /* null pointer, bad mode, bad enum, bad count */
    ABG_EALIGN = 2,   /* a pointer is not aligned as the call requires */
    ABG_ESHAPE = 3,   /* size not a positive multiple of 64, row range out of bounds, cols too large */
    ABG_EALIAS = 4,   /* an output overlaps an input (or, in a graph, a same-stage read) */
    ABG_ECUDA = 5,    /* a CUDA runtime call failed; see abg_last_cuda_error() */
    ABG_ETIMEOUT = 6  /* a device-side wait ran out of time (reported by abg_device_status) */
} abg_status;

typedef enum { ABG_TREE = 0, ABG_FAST = 1 } abg_mode;

/* Storage type of scale and bias ([fused-token] Why: the MLX 4-bit formats).
 * 16-bit values are widened to f32 exactly before use (bf16: the upper half
 * of an f32; f16: IEEE binary16), so the arithmetic is the same as for f32
 * storage of the widened values. */
typedef enum { ABG_SB_F32 = 0, ABG_SB_BF16 = 1, ABG_SB_F16 = 2 } abg_sb_type;

/* Largest `cols` a product accepts: the activation row is staged once per
 * thread block in shared memory. */
#define ABG_MAX_COLS 16384

/*
 * q4mv: rows row0 .. row0+n-1 of the packed rows x cols matrix times x.
 * ([q4go] Change: Array.q4go(w, x, y, r, n, cols, rows) -- reading: r is the
 *  first row, n the number of rows computed, rows the matrix height that
 *  locates each row's words, scale and bias.)
 *
 *   w      u32 [rows][cols/8]   packed nibbles (see the header comment)
 *   scale  f32 [rows][cols/64]
 *   bias   f32 [rows][cols/64]
 *   x      f32 [cols]
 *   xsum   f32 [cols/64]        xsum[g] = tree sum of x[64g .. 64g+63]
 *   y      f32 [n]              y[i] = row row0+i
 *   cols   positive multiple of 64, at most ABG_MAX_COLS
 *   0 <= row0, 0 <= n, row0 + n <= rows.  n == 0 enqueues nothing.
 *   mode   ABG_TREE or ABG_FAST
 *   rows_per_warp  1, 2, 4 or 8 rows share one staging of each 1024-column
 *          slice of x in a warp's registers ([fused-token] Change: a SIMD
 *          group does 4 rows and reads each group's activations once); 0 picks
 *          the default (8).  It never changes the result.
 */
abg_status abg_q4mv(const uint32_t *w, const float *scale, const float *bias,
                    const float *x, const float *xsum, float *y,
                    int64_t rows, int64_t cols, int64_t row0, int64_t n,
                    int mode, int rows_per_warp, void *stream);

/*
 * q4mv_ex: the same product for the other MLX 4-bit formats ([fused-token]
 * Why): groups of `group` columns (32, 64 or 128) and scale/bias stored as
 * `sb_type` (abg_sb_type).
 *
 *     y[r] = sum_g ( scale[r][g] * sum_j q[r][group*g+j] * x[group*g+j]
 *                    + bias[r][g] * xsum[g] ),   g < cols/group,
 *
 * with the same tree order and rounding as abg_q4mv (which is this call with
 * group 64 and ABG_SB_F32).
 *   scale, bias  [rows][cols/group] of f32, or of 16-bit bf16 / f16 patterns;
 *                aligned to their element size (4 or 2 bytes)
 *   xsum   f32 [cols/group]   xsum[g] = tree sum of x[group*g .. group*g+group-1]
 *   cols   a positive multiple of 64 and of group, at most ABG_MAX_COLS
 * scale and bias rows are streamed with bulk copies when both pointers are
 * 16-byte aligned and a row of them is a multiple of 16 bytes.  Other
 * arguments and errors as abg_q4mv; a bad group or sb_type is ABG_EINVAL.
 */
abg_status abg_q4mv_ex(const uint32_t *w, const void *scale, const void *bias, int sb_type, int group,
                       const float *x, const float *xsum, float *y,
                       int64_t rows, int64_t cols, int64_t row0, int64_t n,
                       int mode, int rows_per_warp, void *stream);

/*
 * q4mm: the product for a batch of T decode tokens that share the weights
 * (the 4-row q4mv of [fused-token] Change reads each activation group once for
 * several rows; here each weight is read once for several tokens):
 *
 *     y[t*n + i] = q4mv row row0+i of x[t*cols .. t*cols+cols-1],  t < T,
 *
 * each token's result bit-identical to abg_q4mv on that token alone (ABG_TREE).
 *   x     f32 [T][cols], 16-byte aligned (rows follow each other)
 *   xsum  f32 [T][cols/64]   xsum[t][g] = tree sum of token t's group g
 *   y     f32 [T][n]
 *   T     1..8.  Each group of four tokens (rows of 2048 columns with
 *         bulk-copied scale and bias) or pair of tokens is one launch that
 *         reads the weights once for all of them; an odd last token runs as
 *         a single-token product.
 *         The first launch waits for the stream's earlier work; the later
 *         ones may start while it runs (programmatic dependent launch, off
 *         with ABG_PDL=0), since they read the same inputs and write other
 *         rows of y.
 * Groups of 64 columns with f32 scale and bias; other arguments and errors as
 * abg_q4mv.
 */
abg_status abg_q4mm(const uint32_t *w, const float *scale, const float *bias,
                    const float *x, const float *xsum, float *y,
                    int64_t rows, int64_t cols, int64_t row0, int64_t n, int64_t T,
                    int mode, int rows_per_warp, void *stream);

/*
 * gsum: s[g] = tree sum of v[64g .. 64g+63], g < n/64.  The group sums a
 * product reads for its bias term ([fused-token] Change, Array.rmsq bullet:
 * "the 64-value group sums that Array.q4mv reads").  n a positive multiple of 64.
 */
abg_status abg_gsum(const float *v, float *s, int64_t n, int mode, void *stream);
/* gsum_ex: s[g] = tree sum of v[group*g .. group*g+group-1], group 32, 64 or
 * 128; n a positive multiple of 64 and of group. */
abg_status abg_gsum_ex(const float *v, float *s, int64_t n, int group, int mode, void *stream);

/*
 * rmsq: RMS norm with weights plus the group sums of its output
 * ([fused-token] Change, Array.rmsq bullet).
 *   ss      = tree over groups of (tree over the group of x[i]*x[i])
 *   r       = 1 / sqrt(ss / n + eps)
 *   xn[i]   = (x[i] * r) * wt[i]
 *   xsum[g] = tree sum of xn over group g
 * x, wt, xn f32 [n]; xsum f32 [n/64]; n a positive multiple of 64, at most
 * 2^20.  Runs in one thread block.
 */
abg_status abg_rmsq(const float *x, const float *wt, float eps, float *xn, float *xsum,
                    int64_t n, int mode, void *stream);
/* rmsq_ex: the same with xsum over groups of `group` values (32, 64 or 128;
 * xsum f32 [n/group]; n also a multiple of group).  The norm factor does not
 * depend on the group size: the two-level tree of squares is the pairwise tree
 * over all n values. */
abg_status abg_rmsq_ex(const float *x, const float *wt, float eps, float *xn, float *xsum,
                       int64_t n, int group, int mode, void *stream);

/*
 * swq: SwiGLU plus the group sums of its output ([fused-token] Change,
 * Array.swq(a, o, n) bullet).  a = [gate (n) | up (n)].
 *   o[i]    = silu(a[i]) * a[n+i],  silu(g) = g / (1 + EXP(-g))
 *   osum[g] = tree sum of o over group g
 * In ABG_TREE mode EXP is the library's own binary32 exponential (Cody-Waite
 * reduction with a two-part ln 2, degree-7 Taylor polynomial with RN(1/i!)
 * coefficients, exact scaling by 2^k), so the result is bit-exact across
 * devices; a vendor exp moves the last bits ([fused-token] Change, last
 * paragraph).  a f32 [2n]; o f32 [n]; osum f32 [n/64]; n a positive multiple
 * of 64.
 */
abg_status abg_swq(const float *a, float *o, float *osum, int64_t n, int mode, void *stream);
/* swq_ex: the same with osum over groups of `group` values (32, 64 or 128;
 * osum f32 [n/group]; n also a multiple of group). */
abg_status abg_swq_ex(const float *a, float *o, float *osum, int64_t n, int group, int mode, void *stream);

/*
 * gdn: one token of a gated DeltaNet mixer ([fused-token] Change, Array.gdn
 * bullet: conv window and activation, q/k L2 norms, decay and beta, the
 * delta-rule rows, the gated norm and group sums; one threadgroup per value
 * head, every phase local to its head).  The page gives no formulas; this is
 * the published gated DeltaNet recurrence with one key head per value head,
 * every step one binary32 operation rounded to nearest, every sum the
 * library's pairwise tree, EXP as in swq and LOG the library's own logarithm
 * (reduction to [sqrt(1/2), sqrt(2)) times 2^e, 2 atanh(s) by its series to
 * s^9, e*ln2 in two parts):
 *   SIGMOID(u) = 1/(1 + EXP(-u)), SILU(u) = u/(1 + EXP(-u)),
 *   SOFTPLUS(u) = u if u > 20, else LOG(1 + EXP(u))
 *   channel c of x = [q | k | v]: window w = [state[c][0..K-2], x[c]],
 *     a_c = SILU(tree_t conv[c][t]*w[t]), state[c] <- w[1..K-1]
 *   head h: qh = q * (1/sqrt(tree q*q + eps)) * RN(1/sqrt(D)),
 *     kh = k * (1/sqrt(tree k*k + eps)),
 *     alpha = EXP(-(EXP(A_log[h]) * SOFTPLUS(a[h] + dt_bias[h]))),
 *     beta = SIGMOID(b[h]),
 *     S <- alpha*S;  d_j = beta*(v_j - tree_i S[i][j]*kh_i);
 *     S[i][j] <- S[i][j] + kh_i*d_j;  o_j = tree_i S[i][j]*qh_i,
 *     y_j = ((o_j * 1/sqrt(tree(o*o)/D + eps_n)) * nw_j) * SILU(z[h*D+j])
 *   ysum = 64-value group sums of y.
 *   x        f32 [3*H*D] (q, then k, then v; head h's block at h*D)
 *   conv     f32 [3*H*D][K]         state  f32 [3*H*D][K-1], updated in place
 *   a, b, A_log, dt_bias f32 [H]    z      f32 [H*D]      nw  f32 [D]
 *   S        f32 [H][D][D] (key i, value j), updated in place; 16-byte aligned
 *   y        f32 [H*D]              ysum   f32 [H*D/64]
 *   D = 64, 128 or 256; 2 <= K <= 8; H >= 1, H*D <= 2^20.
 * Both modes compute the same bits.  One launch, started early by
 * programmatic dependent launch unless ABG_PDL=0 (it reads every input after
 * the launch before it has finished).  Errors: null pointer or mode
 * ABG_EINVAL; shape ABG_ESHAPE; a pointer not 4-byte aligned, or S not
 * 16-byte aligned, ABG_EALIGN; an
 * output (state, S, y, ysum) overlapping an input or another output
 * ABG_EALIAS.  Asynchronous on `stream`.
 */
abg_status abg_gdn(const float *x, const float *conv, float *state, const float *a, const float *b, const float *z,
                   const float *A_log, const float *dt_bias, const float *nw, float *S, float *y, float *ysum,
                   int64_t H, int64_t D, int64_t K, float eps, float eps_n, int mode, void *stream);

/*
 * atq: one token of gated attention over key and value caches ([fused-token]
 * Change, Array.atq bullet: q/k RMS norm and rotation, the new k/v into the
 * caches, scores, softmax, weighted values, sigmoid gate and group sums; one
 * threadgroup per query head, the first head of each KV group writing the
 * cache row while the others use the new k/v).  The page gives no formulas;
 * this is grouped-query attention at position pos (query head h reads
 * key/value head h / (Hq/Hkv)) with the library's steps (one RN binary32 op
 * each, pairwise trees, EXP and SIGMOID as in gdn):
 *   RMS(u) = 1/sqrt(tree(u*u)/D + eps);  qn = (q_h*RMS(q_h))*qn_w,
 *     kn = (k_g*RMS(k_g))*kn_w
 *   rotation of column pairs (i, i + D/2) by this position's cos_i, sin_i:
 *     r_i = u_i*cos_i - u_{i+D/2}*sin_i, r_{i+D/2} = u_{i+D/2}*cos_i + u_i*sin_i
 *   Kc[g][pos] = rot(kn), Vc[g][pos] = v_g
 *   s_t = tree_j(rot(qn)_j*Kc[g][t][j]) * RN(1/sqrt D), t = 0..pos
 *   p_t = EXP(s_t - max s) / tree_t EXP(s_t - max s)
 *   y_j = tree_t(p_t*Vc[g][t][j]) * SIGMOID(gate[h*D+j]);  ysum = 64-value
 *   group sums of y
 *   q, gate  f32 [Hq*D]    k, v  f32 [Hkv*D]    qn_w, kn_w  f32 [D]
 *   cos, sin f32 [D/2]     Kc, Vc f32 [Hkv][P][D], rows < pos filled; row pos
 *                          written (by the call)
 *   y        f32 [Hq*D]    ysum  f32 [Hq*D/64]
 *   D = 64, 128 or 256; Hq a multiple of Hkv; 0 <= pos < P; pos + 1 <= 8192;
 *   Hq*D <= 2^20.
 * Both modes compute the same bits.  The positions run in chunks of 64 (four
 * launches, started early by programmatic dependent launch unless
 * ABG_PDL=0): the first reads the key cache rows below pos before it waits
 * for the launch before it on the stream, which therefore must not write
 * them.  The chunks' partial results live in a device buffer the library
 * allocates on a device's first call and grows when a call needs more (the
 * growth synchronizes the device, so a call recorded into a stream capture
 * must not need more than an earlier call outside it: ABG_ECUDA otherwise);
 * calls that can overlap on the GPU (on different streams or host threads)
 * share it and must be ordered by the caller.  A stage graph's atq nodes
 * have buffers of their own.  Errors: null pointer
 * or mode ABG_EINVAL; shape ABG_ESHAPE; a pointer not 4-byte aligned, or Kc
 * or Vc not 16-byte aligned, ABG_EALIGN; an output (Kc, Vc, y, ysum)
 * overlapping an input or another output ABG_EALIAS.  Asynchronous on
 * `stream`.
 */
abg_status abg_atq(const float *q, const float *gate, const float *k, const float *v, const float *qn_w,
                   const float *kn_w, const float *cos, const float *sin, float *Kc, float *Vc, float *y, float *ysum,
                   int64_t Hq, int64_t Hkv, int64_t D, int64_t P, int64_t pos, float eps, int mode, void *stream);

/* ---------------------------------------------------------------------------
 * Stage graph: one decode token's dependent stages recorded into one CUDA
 * graph, replayed with one launch and synchronized once by the caller
 * ([fused-token] Why and Verification: one command buffer, one wait per
 * token; [q4go] Change: products queued together run concurrently, and a
 * dependent stage needs the previous one finished).
 *
 * Nodes carry a stage index.  Nodes with the same index form one stage and
 * may run concurrently; every node of stage s+1 runs after every node of
 * stage s has finished.  Products of one stage that read the same x (for
 * example q/k/v, or gate/up) are run as grouped launches of up to 256
 * products each (abg_stage_graph_launches counts them).  Consecutive
 * launches overlap through programmatic dependent launch: a product fetches
 * its weights before the previous stage has finished and waits only before
 * it reads its activation.  Weights, and the norm weights of an RMS-norm
 * prologue, must therefore not be written by any node of the graph (checked:
 * ABG_EALIAS).
 *
 * Node kinds and the fields each reads (unused fields are ignored):
 *   ABG_NODE_Q4MV  w, scale, bias, rows, cols, row0, n, y, prologue, and
 *                  prologue ABG_PRO_NONE: x [cols], xsum [cols/64]
 *                  prologue ABG_PRO_GSUM: x [cols]; xsum computed in-kernel
 *                  prologue ABG_PRO_RMSQ: x [cols] (un-normalized), wt [cols],
 *                                         eps; the product reads rmsq(x, wt)
 *                  prologue ABG_PRO_SWQ:  x [2*cols] = [gate | up]; the
 *                                         product reads swq(x)
 *                  A prologue recomputes the producer inside each thread
 *                  block with the same trees, so the product's result is
 *                  bit-identical to running the producer node first.
 *   ABG_NODE_RMSQ  x, wt, eps, len -> out (xn), out_sum (xsum)
 *   ABG_NODE_SWQ   x (2*len), len -> out (o), out_sum (osum)
 *   ABG_NODE_GSUM  x, len -> out_sum
 *   ABG_NODE_GDN   args (abg_gdn_args): as abg_gdn; reads and writes state
 *                  and S in place
 *   ABG_NODE_ATQ   args (abg_atq_args): as abg_atq; writes row pos of Kc, Vc
 *                  (the graph owns the buffer of the chunk results of each
 *                  ATQ node, so replays of different graphs do not share it);
 *                  no other node may write its Kc or Vc (ABG_EALIAS)
 *   ABG_NODE_COPY  x, len -> out: copies len floats (a memory copy, no
 *                  arithmetic), so that a replay can take its inputs from
 *                  host memory and return its results there: each of x and
 *                  out is device memory or page-locked host memory (pinned or
 *                  registered); pageable host memory, len <= 0, a pointer not
 *                  4-byte aligned or overlapping ranges give ABG_EINVAL,
 *                  ABG_ESHAPE, ABG_EALIGN and ABG_EALIAS.  The kernel launch
 *                  that follows a copy does not start early.
 * Every kind also reads `group` (0 means 64): the group size of the product's
 * scale, bias and xsum (Q4MV, including the group sums its prologue
 * computes) or of out_sum (RMSQ, SWQ, GSUM); Q4MV reads `sb_type` (an
 * abg_sb_type; scale and bias then point at that type).  Sizes given above
 * as cols/64 or len/64 are cols/group and len/group.
 * ------------------------------------------------------------------------- */
typedef enum {
    ABG_NODE_Q4MV = 0,
    ABG_NODE_RMSQ = 1,
    ABG_NODE_SWQ = 2,
    ABG_NODE_GSUM = 3,
    ABG_NODE_GDN = 4, /* args -> abg_gdn_args */
    ABG_NODE_ATQ = 5, /* args -> abg_atq_args */
    ABG_NODE_COPY = 6 /* x -> out, len floats */
} abg_node_kind;

/* The arguments of abg_gdn and abg_atq, for their stage-graph nodes (the
 * struct is read when the graph is created; the pointers must stay valid for
 * the graph's lifetime, like every node's). */
typedef struct abg_gdn_args {
    const float *x, *conv;
    float *state;
    const float *a, *b, *z, *A_log, *dt_bias, *nw;
    float *S, *y, *ysum;
    int64_t H, D, K;
    float eps, eps_n;
} abg_gdn_args;

typedef struct abg_atq_args {
    const float *q, *gate, *k, *v, *qn_w, *kn_w, *cos, *sin;
    float *Kc, *Vc, *y, *ysum;
    int64_t Hq, Hkv, D, P, pos;
    float eps;
} abg_atq_args;
typedef enum { ABG_PRO_NONE = 0, ABG_PRO_GSUM = 1, ABG_PRO_RMSQ = 2, ABG_PRO_SWQ = 3 } abg_prologue;

typedef struct abg_node {
    int32_t kind;      /* abg_node_kind */
    int32_t stage;     /* stage index; any order, grouped by value */
    const uint32_t *w; /* Q4MV */
    const void *scale; /* f32, or 16-bit patterns (sb_type) */
    const void *bias;
    int64_t rows, cols, row0, n;
    float *y;
    int32_t prologue;  /* abg_prologue, Q4MV only */
    float eps;         /* RMSQ node and ABG_PRO_RMSQ */
    const float *x;    /* activation / producer input (see above) */
    const float *xsum; /* Q4MV with ABG_PRO_NONE */
    const float *wt;   /* RMSQ node and ABG_PRO_RMSQ */
    float *out;        /* RMSQ, SWQ, COPY */
    float *out_sum;    /* RMSQ, SWQ, GSUM */
    int64_t len;       /* RMSQ, SWQ, GSUM vector length n; COPY floats */
    int32_t group;     /* group size 32, 64 or 128; 0 = 64 */
    int32_t sb_type;   /* Q4MV: abg_sb_type of scale and bias */
    const void *args;  /* GDN: abg_gdn_args; ATQ: abg_atq_args */
} abg_node;

/* Validates every node (same rules as the single calls), checks that no node
 * reads an output of its own stage, records the launches on a private stream
 * and instantiates the graph.  *graph_out receives an opaque handle.  The
 * graph owns its executable graph and, for SwiGLU pairs (see
 * abg_stage_graph_swiglu_pairs), one device buffer of n floats per pair. */
abg_status abg_stage_graph_create(const abg_node *nodes, int64_t count, int mode, int rows_per_warp,
                                  void **graph_out);
/* With the environment variable ABG_PDL=0 at creation, launches are recorded
 * without programmatic dependent launch (each waits for the previous one to
 * finish before starting); results are identical. */
/* Enqueues one replay of the whole graph on `stream`; the caller syncs once.
 * With the environment variable ABG_TRACE=1 each launch also synchronizes and
 * prints the launch count, GPU milliseconds and wall milliseconds to stderr. */
abg_status abg_stage_graph_launch(void *graph, void *stream);
/* Number of kernel launches one replay performs (after sibling grouping; an
 * ATQ node performs four, a COPY node none). */
abg_status abg_stage_graph_launches(void *graph, int64_t *launches);
/* SwiGLU pairs: when a Q4MV node with the ABG_PRO_SWQ prologue reads a =
 * [gate | up] (2n values) written by the only two products of the launch
 * right before it (gate y = a[0, n), up y = a[n, 2n), one activation, n rows
 * each, groups of 64 with f32 scale and bias, 2048, 4096 or 6144 columns), the
 * gate/up launch also writes silu(gate) * up once per element into a device
 * buffer of n floats that the graph allocates at creation and frees in
 * abg_stage_graph_destroy, and the reading product takes its group sums from
 * that buffer instead of recomputing the SwiGLU in every thread block.  Every
 * node's outputs keep their bits.  *pairs receives how many were formed. */
abg_status abg_stage_graph_swiglu_pairs(void *graph, int64_t *pairs);
abg_status abg_stage_graph_destroy(void *graph);

/* Reads (and, if clear != 0, resets) the device status word on the current
 * device: bit 0 = a device-side wait timed out; bits 4.. name the wait that
 * gave up (16: a stage's release, 32: a stage's arrival, 64: the partial sums
 * of a tile, 128: a final drain of copies).  Synchronizes the device.
 * Returns ABG_ETIMEOUT when bit 0 was set, else ABG_OK. */
abg_status abg_device_status(uint32_t *bits, int clear);

/* Failure-detection self-test (no counterpart on the pages, whose queued
 * kernels had no bounded waits): enqueues one small product whose producer
 * warp withholds its only tile, so the computing warps' bounded waits run out
 * after the 0.5 s limit.  The kernel then sets bits 0 and 32 of the device
 * status word and exits with no copy in flight; the GPU context stays usable.
 * Reads no caller memory.  Expect abg_device_status to return ABG_ETIMEOUT
 * (and clear it there) after syncing the stream. */
abg_status abg_selftest_wait_timeout(void *stream);

/* Tuning of the product kernel, process-wide; 0 keeps the default.  Applies
 * to calls and graphs created afterwards.
 *   smem_kb          shared-memory budget per thread block (default 110, so
 *                    two blocks fit on an SM and a dependent launch can start
 *                    while its predecessor still runs)
 *   consumer_warps   warps that compute, 1..16 (default: chosen from cols, at
 *                    most 8); above 8 selects one block per SM (with 8 rows
 *                    per warp item)
 *   blocks_per_sm    thread blocks per SM in the grid, at most what fits
 *                    (default: 2)
 *   stage_kb         target size of one pipeline stage of streamed rows
 *                    (default 40)
 * It never changes results. */
abg_status abg_set_q4mv_tuning(int smem_kb, int consumer_warps, int blocks_per_sm, int stage_kb);

/*
 * swiglu_mlp_static: the MLP block y = down( silu(gate x) * (up x) ) with
 * no device allocation and no buffer from the caller for the intermediate
 * vectors.  The pages have no counterpart of this call: it exists for callers
 * that cannot allocate device memory themselves, such as code whose device
 * memory all belongs to another allocator (a framework's caching allocator,
 * or a server that reserves its memory up front), or code on a latency path
 * where cudaMalloc/cudaFree would synchronize the device.
 *   wg, sg, bg  gate product: u32 [n][cols/8], f32 [n][cols/64] x2
 *   wu, su, bu  up product:   the same shapes
 *   wd, sd, bd  down product: u32 [rows][n/8], f32 [rows][n/64] x2
 *   x     f32 [cols], xsum f32 [cols/64] (x's group sums)
 *   y     f32 [rows]  y[i] = row i of the down product of o[j] =
 *                     silu(gate_y[j]) * up_y[j], silu(g) = g / (1 + EXP(-g))
 *   n     rows of gate and up, columns of down: a positive multiple of 64, at
 *         most 16384 (else ABG_ESHAPE)
 * Groups of 64 columns with f32 scale and bias; every result, tree order and
 * error rule as the separate calls (abg_q4mv twice, abg_swq, abg_q4mv), whose
 * results it equals bit for bit in ABG_TREE mode.
 * The intermediate vectors (gate_y, up_y and o, 3n floats) live in one
 * static device array of 3 * 16384 floats inside the library, which every
 * device that loads the library holds until the process exits.  The first
 * call on a device looks up that array's device address (with the device
 * current), so make the first call on each device before any stream capture
 * begins.  Every call uses the same array: calls that can overlap on the GPU
 * (on different streams, or different host threads) race on it and must be
 * ordered by the caller.  Nothing in the array needs clearing: each call
 * writes every element it reads.  Asynchronous like the other calls.
 */
abg_status abg_swiglu_mlp_static(const uint32_t *wg, const float *sg, const float *bg,
                                 const uint32_t *wu, const float *su, const float *bu,
                                 const uint32_t *wd, const float *sd, const float *bd,
                                 const float *x, const float *xsum, float *y,
                                 int64_t n, int64_t cols, int64_t rows, int mode, void *stream);

const char *abg_status_str(int status);
/* Text of the last CUDA error seen by any call on this thread ("" if none). */
const char *abg_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* ABG_H */
