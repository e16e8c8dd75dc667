/*
 * Plain CPU oracle for the affine 4-bit group-quantized matrix-vector product
 * (q4mv) and its two activation producers (rmsq, swq), plus the group sum
 * (gsum) and the output hash used by the measurements.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it.  It shares
 * no source, header, table or helper with the CUDA library.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fPIC -shared.  Every float
 * operation below is one IEEE binary32 operation rounded to nearest even; with
 * contraction off no multiply is fused into an add, so each line is exactly
 * the rounded operation it names.  (C's FLT_EVAL_METHOD is 0 on both x86-64
 * and aarch64, so float expressions are evaluated in float.)
 *
 * Sources (Bend pull requests by the same author, all closed unmerged):
 *   [q4mv-metal]  "Array.q4mv on Metal: one kernel thread per row for products
 *                 of 4M weights or more, bit-identical" (bendlang/bend #1435)
 *   [q4go]        "Array.q4go/Array.q4wait queue Metal Q4 products in one
 *                 command buffer and wait once on a flag" (#1437)
 *   [fused-token] "Metal: queued rmsq, swq, gdn and atq kernels and a 4-row
 *                 q4mv, so a decode token is one command buffer with one wait"
 *                 (#1440)
 * The pages state the product (MLX-style 4-bit affine weights, groups of 64
 * columns, a per-group activation sum for the bias term) and that the sum runs
 * in a fixed tree order, but not the tree itself; the readings taken where the
 * pages are silent are named at each function.
 *
 * parity unpinned: or_hash32 against the pages' printed hash (their input
 * generator and hash function are not given).  Every other function is pinned
 * by the CPU tests.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* TREE: the fixed summation order.                                          */
/* [fused-token] Change, the bend_q4mv bullet, and the #1436 title it cites:  */
/* sums run in a fixed tree order.  Reading: a balanced pairwise tree in      */
/* index order.  At each level elements (2i, 2i+1) are added; an odd last    */
/* element is carried to the next level unchanged (not added to a zero).      */
/* For a power-of-two count this is recursive halving.                        */
/* ------------------------------------------------------------------------ */
float or_tree(const float *v, int64_t m)
{
    if (m <= 0) return -0.0f; /* never used by the method; -0 is the additive identity */
    float local[128];
    float *buf = m <= 128 ? local : (float *)malloc((size_t)m * sizeof(float));
    memcpy(buf, v, (size_t)m * sizeof(float));
    const int64_t m0 = m;
    while (m > 1) {
        const int64_t half = m / 2;
        for (int64_t i = 0; i < half; ++i)
            buf[i] = buf[2 * i] + buf[2 * i + 1];
        if (m & 1) buf[half] = buf[m - 1];
        m = half + (m & 1);
    }
    const float s = buf[0];
    if (m0 > 128) free(buf);
    return s;
}

/* ------------------------------------------------------------------------ */
/* gsum: s[g] = TREE(v[64g .. 64g+63]).                                       */
/* [fused-token] Change, Array.rmsq bullet: producers emit the 64-value      */
/* group sums that Array.q4mv reads.                                          */
/* ------------------------------------------------------------------------ */
void or_gsum(const float *v, float *s, int64_t n)
{
    for (int64_t g = 0; g < n / 64; ++g)
        s[g] = or_tree(v + 64 * g, 64);
}

/* ------------------------------------------------------------------------ */
/* q4mv.  Weight format ([fused-token] Why; [q4go] Verification, whole       */
/* model): MLX-style 4-bit affine weights w = scale*q + bias in groups of 64 */
/* columns.  Packing: 8 nibbles per u32, column 8k+j is nibble j of word k,  */
/* low nibble first; scale and bias are f32 [rows][cols/64].                 */
/*                                                                          */
/* For each row r and group g:                                              */
/*   p_j = (float)q[r][64g+j] * x[64g+j]          (one rounding each)        */
/*   d   = TREE(p_0 .. p_63)                                                 */
/*   t_g = scale[r][g]*d + bias[r][g]*xsum[g]     (two products, one add)    */
/* and y = TREE(t_0 .. t_{G-1}).  This is the dequantize-then-dot product     */
/* with the bias folded into the activation's group sum:                     */
/*   sum_j (s*q_j + b)*x_j = s*sum_j q_j*x_j + b*sum_j x_j.                  */
/* Row range ([q4go] Change, Array.q4go(w, x, y, r, n, cols, rows)): rows    */
/* row0 .. row0+n-1 of a rows x cols matrix; y[i] receives row row0+i.       */
/* ------------------------------------------------------------------------ */
void or_q4mv(const uint32_t *w, const float *scale, const float *bias,
             const float *x, const float *xsum, float *y,
             int64_t rows, int64_t cols, int64_t row0, int64_t n)
{
    (void)rows;
    const int64_t W = cols / 8, G = cols / 64;
    float *t = (float *)malloc((size_t)(G > 0 ? G : 1) * sizeof(float));
    float p[64];
    for (int64_t i = 0; i < n; ++i) {
        const int64_t r = row0 + i;
        for (int64_t g = 0; g < G; ++g) {
            for (int j = 0; j < 64; ++j) {
                const int64_t c = 64 * g + j;
                const uint32_t word = w[r * W + c / 8];
                const uint32_t q = (word >> (4 * (c % 8))) & 0xFu;
                p[j] = (float)q * x[c];
            }
            const float d = or_tree(p, 64);
            const float sd = scale[r * G + g] * d;
            const float bx = bias[r * G + g] * xsum[g];
            t[g] = sd + bx;
        }
        y[i] = or_tree(t, G);
    }
    free(t);
}

/* Magnitude of the terms of each output, in double: A_r = sum_g |scale*d| +
 * |bias*xsum| with d = sum_j q*x in double.  Used only to scale the error
 * allowed to the reordered (fast) mode, whose per-output error is bounded by
 * a multiple of this sum, not of |y| (the bias term cancels most of y). */
void or_q4mv_absmag(const uint32_t *w, const float *scale, const float *bias,
                    const float *x, const float *xsum, double *a,
                    int64_t rows, int64_t cols, int64_t row0, int64_t n)
{
    (void)rows;
    const int64_t W = cols / 8, G = cols / 64;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t r = row0 + i;
        double acc = 0.0;
        for (int64_t g = 0; g < G; ++g) {
            double d = 0.0;
            for (int j = 0; j < 64; ++j) {
                const int64_t c = 64 * g + j;
                const uint32_t q = (w[r * W + c / 8] >> (4 * (c % 8))) & 0xFu;
                d += (double)q * (double)x[c];
            }
            acc += fabs((double)scale[r * G + g] * d) + fabs((double)bias[r * G + g] * (double)xsum[g]);
        }
        a[i] = acc;
    }
}

/* ------------------------------------------------------------------------ */
/* rmsq: RMS norm with f32 weights plus the group sums of its output.        */
/* [fused-token] Change, Array.rmsq bullet.  Readings: weights multiply the  */
/* normalised value directly (not 1+w); the sum of squares uses the same     */
/* two-level tree as every other sum (per 64-group, then across groups).     */
/*   ss   = TREE_g( TREE_j( x_i*x_i ) )                                      */
/*   mean = ss / n;  r = 1 / sqrt(mean + eps)                                */
/*   xn_i = (x_i * r) * wt_i;  xsum[g] = TREE(xn in group g)                  */
/* n must be a multiple of 64.                                               */
/* ------------------------------------------------------------------------ */
void or_rmsq(const float *x, const float *wt, float eps, float *xn, float *xsum, int64_t n)
{
    const int64_t G = n / 64;
    float *gs = (float *)malloc((size_t)(G > 0 ? G : 1) * sizeof(float));
    float sq[64];
    for (int64_t g = 0; g < G; ++g) {
        for (int j = 0; j < 64; ++j) {
            const float v = x[64 * g + j];
            sq[j] = v * v;
        }
        gs[g] = or_tree(sq, 64);
    }
    const float ss = or_tree(gs, G);
    const float mean = ss / (float)n;
    const float r = 1.0f / sqrtf(mean + eps);
    for (int64_t i = 0; i < n; ++i) {
        const float xr = x[i] * r;
        xn[i] = xr * wt[i];
    }
    or_gsum(xn, xsum, n);
    free(gs);
}

/* ------------------------------------------------------------------------ */
/* EXP: an exponential both sides compute from this written definition, so  */
/* that the SwiGLU product can be bit-exact ([fused-token] Change, last      */
/* paragraph: a vendor exp moves the last bits).  Cody-Waite reduction with  */
/* a two-part ln 2, degree-7 Taylor polynomial in Horner form, exact scaling */
/* by 2^k.  Constants (IEEE binary32 bit patterns):                          */
/*   L2E   = RN(log2 e)                         0x3FB8AA3B                   */
/*   LN2HI = RN(ln 2) with its low 12 mantissa bits cleared  0x3F317000      */
/*           (so k*LN2HI is exact for |k| < 2^12)                            */
/*   LN2LO = RN(ln 2 - LN2HI)                   0x3805FDF4                   */
/*   C_i   = RN(1/i!), i = 0..7                                              */
/* Steps: NaN -> NaN; v > 89 -> +inf; v < -104 -> +0; otherwise              */
/*   k  = round-half-even(v*L2E)                                             */
/*   rr = (v + (-k)*LN2HI) + (-k)*LN2LO                                      */
/*   p  = C_0 + rr*(C_1 + rr*(... + rr*C_7))   (Horner, mul then add)         */
/*   result = p*2^k, applied as one multiply for -126 <= k <= 127, as        */
/*   (p*2^(k+126))*2^-126 for k < -126 (first product exact) and as          */
/*   (p*2^127)*2^(k-127) for k > 127, so the result is rounded once.         */
/* ------------------------------------------------------------------------ */
static float f32_from_bits(uint32_t b)
{
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

static float pow2i(int e) /* 2^e for -126 <= e <= 127 */
{
    return f32_from_bits((uint32_t)(e + 127) << 23);
}

float or_exp(float v)
{
    if (v != v) return v;
    if (v > 89.0f) return INFINITY;
    if (v < -104.0f) return 0.0f;
    const float L2E = f32_from_bits(0x3FB8AA3Bu);
    const float LN2HI = f32_from_bits(0x3F317000u);
    const float LN2LO = f32_from_bits(0x3805FDF4u);
    const float C[8] = {
        f32_from_bits(0x3F800000u), f32_from_bits(0x3F800000u), f32_from_bits(0x3F000000u),
        f32_from_bits(0x3E2AAAABu), f32_from_bits(0x3D2AAAABu), f32_from_bits(0x3C088889u),
        f32_from_bits(0x3AB60B61u), f32_from_bits(0x39500D01u),
    };
    const float kf = rintf(v * L2E); /* default rounding mode: nearest even */
    const int k = (int)kf;
    const float nk = -kf;
    const float a = nk * LN2HI;
    const float b = nk * LN2LO;
    const float rr = (v + a) + b;
    float p = C[7];
    for (int i = 6; i >= 0; --i) {
        const float pr = p * rr;
        p = pr + C[i];
    }
    if (k > 127) {
        const float t = p * pow2i(127);
        return t * pow2i(k - 127);
    }
    if (k < -126) {
        const float t = p * pow2i(k + 126);
        return t * pow2i(-126);
    }
    return p * pow2i(k);
}

void or_exp_array(const float *v, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = or_exp(v[i]);
}

/* ------------------------------------------------------------------------ */
/* swq: SwiGLU of a = [gate (n) | up (n)] plus the group sums of its output. */
/* [fused-token] Change, Array.swq(a, o, n) bullet: o[i] is silu(a[i]) times */
/* a[n+i], rounded (to binary32: every step here is an RN binary32 op).      */
/* Reading: silu(g) = g / (1 + EXP(-g)).  n must be a multiple of 64.        */
/* ------------------------------------------------------------------------ */
void or_swq(const float *a, float *o, float *osum, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        const float g = a[i];
        const float e = or_exp(-g);
        const float den = 1.0f + e;
        const float silu = g / den;
        o[i] = silu * a[n + i];
    }
    or_gsum(o, osum, n);
}

/* ------------------------------------------------------------------------ */
/* Hash of an output vector's bits ([q4mv-metal] Verification: the scratch   */
/* program prints a hash of y's bits).  The pages do not name the function;  */
/* reading: 32-bit FNV-1a over the little-endian bytes of y in index order.  */
/* ------------------------------------------------------------------------ */
uint32_t or_fnv1a(const uint8_t *bytes, int64_t nbytes)
{
    uint32_t h = 2166136261u;
    for (int64_t i = 0; i < nbytes; ++i) {
        h ^= bytes[i];
        h *= 16777619u;
    }
    return h;
}

uint32_t or_hash32(const float *y, int64_t n)
{
    /* byte order fixed explicitly, so the hash does not depend on the host */
    uint32_t h = 2166136261u;
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b;
        memcpy(&b, &y[i], sizeof b);
        for (int s = 0; s < 32; s += 8) {
            h ^= (b >> s) & 0xFFu;
            h *= 16777619u;
        }
    }
    return h;
}

/* ------------------------------------------------------------------------ */
/* Other formats of the same product (the MLX 4-bit family the pages name:  */
/* [fused-token] Why, "MLX 4-bit"): group size gs in {32, 64, 128} columns   */
/* and scale/bias stored as f32, bf16 or f16.  Every stored scale and bias   */
/* is widened to f32 exactly, then the product is the one above with gs in   */
/* place of 64:                                                              */
/*   d = TREE_gs(RN(q*x)),  t = RN(RN(s*d) + RN(b*xsum[g])),  y = TREE_G(t)  */
/* with G = cols/gs and xsum[g] = TREE(x over group g).                      */
/* ------------------------------------------------------------------------ */
enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2 };

/* bf16 is the upper half of an f32 */
float or_bf16_to_f32(uint16_t h)
{
    return f32_from_bits((uint32_t)h << 16);
}

/* f16 (1 sign, 5 exponent, 10 significand bits, bias 15) to f32, exactly */
float or_f16_to_f32(uint16_t h)
{
    const uint32_t sign = (uint32_t)(h >> 15) << 31;
    const uint32_t e = (h >> 10) & 0x1Fu;
    uint32_t m = h & 0x3FFu;
    if (e == 0x1Fu) return f32_from_bits(sign | 0x7F800000u | (m << 13)); /* inf, NaN */
    if (e != 0) return f32_from_bits(sign | ((e - 15u + 127u) << 23) | (m << 13));
    if (m == 0) return f32_from_bits(sign); /* signed zero */
    /* subnormal: m * 2^-24, normalised */
    int ex = -14;
    while (!(m & 0x400u)) {
        m <<= 1;
        --ex;
    }
    m &= 0x3FFu;
    return f32_from_bits(sign | ((uint32_t)(ex + 127) << 23) | (m << 13));
}

static float or_load_sb(const void *p, int dtype, int64_t i)
{
    if (dtype == OR_BF16) return or_bf16_to_f32(((const uint16_t *)p)[i]);
    if (dtype == OR_F16) return or_f16_to_f32(((const uint16_t *)p)[i]);
    return ((const float *)p)[i];
}

void or_gsum_ex(const float *v, float *s, int64_t n, int gs)
{
    for (int64_t g = 0; g < n / gs; ++g)
        s[g] = or_tree(v + gs * g, gs);
}

void or_q4mv_ex(const uint32_t *w, const void *scale, const void *bias, int sb_dtype, int gs,
                const float *x, const float *xsum, float *y,
                int64_t rows, int64_t cols, int64_t row0, int64_t n)
{
    (void)rows;
    const int64_t W = cols / 8, G = cols / gs;
    float *t = (float *)malloc((size_t)(G > 0 ? G : 1) * sizeof(float));
    float p[128];
    for (int64_t i = 0; i < n; ++i) {
        const int64_t r = row0 + i;
        for (int64_t g = 0; g < G; ++g) {
            for (int j = 0; j < gs; ++j) {
                const int64_t c = gs * g + j;
                const uint32_t q = (w[r * W + c / 8] >> (4 * (c % 8))) & 0xFu;
                p[j] = (float)q * x[c];
            }
            const float d = or_tree(p, gs);
            const float sd = or_load_sb(scale, sb_dtype, r * G + g) * d;
            const float bx = or_load_sb(bias, sb_dtype, r * G + g) * xsum[g];
            t[g] = sd + bx;
        }
        y[i] = or_tree(t, G);
    }
    free(t);
}

/* ------------------------------------------------------------------------ */
/* LOG: a natural logarithm both sides compute from this written definition */
/* (the gdn mixer's softplus needs one; as with EXP, a vendor log would move */
/* the last bits).  Reduction to m in [sqrt(1/2), sqrt(2)) times 2^e, then   */
/* log(m) = 2 atanh(s) with s = (m - 1)/(m + 1), the atanh series summed to  */
/* the s^9 term (|s| <= 0.1716, so the first omitted term is below 1e-9 of    */
/* the result), and e*ln2 added in two parts:                                */
/*   special: NaN -> NaN; v < 0 -> NaN; v == 0 -> -inf; +inf -> +inf         */
/*   subnormal v: v*2^23 (exact), e -= 23                                     */
/*   m = v's significand in [1, 2), e = its exponent                          */
/*   if m > RN(sqrt 2) (0x3FB504F3): m = m*0.5, e = e + 1   (exact)           */
/*   f = m - 1 (exact);  s = f / (2 + f);  t = s*s                            */
/*   p = D9;  p = p*t + D7;  p = p*t + D5;  p = p*t + D3;  p = p*t + 2        */
/*   (D_k = RN(2/k); each step a multiply then an add)                        */
/*   result = e*LN2HI + (s*p + e*LN2LO)     (LN2HI, LN2LO as in EXP; e*LN2HI */
/*   and e*LN2LO are exact for |e| < 2^12)                                    */
/* ------------------------------------------------------------------------ */
float or_log(float v)
{
    if (v != v) return v;
    if (v < 0.0f) return NAN;
    if (v == 0.0f) return -INFINITY;
    if (v == INFINITY) return v;
    int e = 0;
    uint32_t b;
    memcpy(&b, &v, sizeof b);
    if ((b >> 23) == 0) { /* subnormal */
        const float vs = v * pow2i(23);
        memcpy(&b, &vs, sizeof b);
        e = -23;
    }
    e += (int)(b >> 23) - 127;
    float m = f32_from_bits((b & 0x007FFFFFu) | 0x3F800000u);
    if (m > f32_from_bits(0x3FB504F3u)) {
        m = m * 0.5f;
        e = e + 1;
    }
    const float LN2HI = f32_from_bits(0x3F317000u);
    const float LN2LO = f32_from_bits(0x3805FDF4u);
    const float D9 = 2.0f / 9.0f, D7 = 2.0f / 7.0f, D5 = 2.0f / 5.0f, D3 = 2.0f / 3.0f;
    const float f = m - 1.0f;
    const float den = 2.0f + f;
    const float s = f / den;
    const float t = s * s;
    float p = D9;
    p = p * t;
    p = p + D7;
    p = p * t;
    p = p + D5;
    p = p * t;
    p = p + D3;
    p = p * t;
    p = p + 2.0f;
    const float ef = (float)e;
    const float hi = ef * LN2HI;
    const float lo = ef * LN2LO;
    const float sp = s * p;
    const float r = sp + lo;
    return hi + r;
}

void or_log_array(const float *v, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = or_log(v[i]);
}

/* ------------------------------------------------------------------------ */
/* gdn: one token of a gated DeltaNet mixer.  [fused-token] Change, the      */
/* Array.gdn bullet, lists the phases -- conv window and activation, q/k L2  */
/* norms, decay and beta, the delta-rule rows, the gated norm and group      */
/* sums -- with one threadgroup per value head, every phase local to its     */
/* head.  The pages give no formulas; the reading (the published gated       */
/* DeltaNet recurrence, one key head per value head, head dimension D for q, */
/* k and v, K conv taps, every sum a TREE, every step one RN binary32 op):   */
/*   SIGMOID(u) = 1 / (1 + EXP(-u));  SILU(u) = u / (1 + EXP(-u)) (as swq)   */
/*   SOFTPLUS(u) = u if u > 20, else LOG(1 + EXP(u))                         */
/* Channels c of x = [q | k | v] (3*H*D values, head h's block at h*D):       */
/*   window w = [state[c][0..K-2], x[c]];  a_c = SILU(TREE_j(conv[c][j]*w[j])) */
/*   state[c] <- w[1..K-1]                                                   */
/* Head h (q, k, v its D activations; i indexes keys, j values):             */
/*   rq = 1 / sqrt(TREE_i(q_i*q_i) + eps);  qh_i = (q_i*rq) * RN(1/sqrt(D))   */
/*   rk = 1 / sqrt(TREE_i(k_i*k_i) + eps);  kh_i = k_i*rk                    */
/*   alpha = EXP(-(EXP(A_log[h]) * SOFTPLUS(a[h] + dt_bias[h])))              */
/*   beta  = SIGMOID(b[h])                                                   */
/*   S[i][j] <- S[i][j]*alpha                                                */
/*   kv_j = TREE_i(S[i][j]*kh_i);  d_j = beta*(v_j - kv_j)                    */
/*   S[i][j] <- S[i][j] + kh_i*d_j                                           */
/*   o_j = TREE_i(S[i][j]*qh_i)                                              */
/*   r = 1 / sqrt(TREE_j(o_j*o_j) / D + eps_n)                               */
/*   y_j = ((o_j*r) * nw_j) * SILU(z_j)                                      */
/* ysum = the 64-value group sums of y.  S [H][D][D] and state [3HD][K-1]    */
/* are updated in place.  D a multiple of 64 (<= 1024), K <= 8.               */
/* ------------------------------------------------------------------------ */
static float or_sigmoid(float u)
{
    const float e = or_exp(-u);
    const float den = 1.0f + e;
    return 1.0f / den;
}

static float or_silu(float u)
{
    const float e = or_exp(-u);
    const float den = 1.0f + e;
    return u / den;
}

static float or_softplus(float u)
{
    if (u > 20.0f) return u;
    const float e = or_exp(u);
    const float one_e = 1.0f + e;
    return or_log(one_e);
}

void or_gdn(const float *x, const float *conv, float *state, const float *a, const float *b, const float *z,
            const float *A_log, const float *dt_bias, const float *nw, float *S, float *y, float *ysum,
            int64_t H, int64_t D, int64_t K, float eps, float eps_n)
{
    const int64_t C = 3 * H * D;
    float *act = (float *)malloc((size_t)C * sizeof(float));
    float *tmp = (float *)malloc((size_t)(D > K ? D : K) * sizeof(float));
    float *qh = (float *)malloc((size_t)D * sizeof(float));
    float *kh = (float *)malloc((size_t)D * sizeof(float));
    float *o = (float *)malloc((size_t)D * sizeof(float));
    float wv[8];
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t j = 0; j < K - 1; ++j) wv[j] = state[c * (K - 1) + j];
        wv[K - 1] = x[c];
        for (int64_t j = 0; j < K; ++j) tmp[j] = conv[c * K + j] * wv[j];
        act[c] = or_silu(or_tree(tmp, K));
        for (int64_t j = 0; j < K - 1; ++j) state[c * (K - 1) + j] = wv[j + 1];
    }
    const float qscale = 1.0f / sqrtf((float)D);
    for (int64_t h = 0; h < H; ++h) {
        const float *q = act + h * D, *k = act + H * D + h * D, *v = act + 2 * H * D + h * D;
        for (int64_t i = 0; i < D; ++i) tmp[i] = q[i] * q[i];
        const float rq = 1.0f / sqrtf(or_tree(tmp, D) + eps);
        for (int64_t i = 0; i < D; ++i) {
            const float t = q[i] * rq;
            qh[i] = t * qscale;
        }
        for (int64_t i = 0; i < D; ++i) tmp[i] = k[i] * k[i];
        const float rk = 1.0f / sqrtf(or_tree(tmp, D) + eps);
        for (int64_t i = 0; i < D; ++i) kh[i] = k[i] * rk;
        const float dec = or_exp(A_log[h]) * or_softplus(a[h] + dt_bias[h]);
        const float alpha = or_exp(-dec);
        const float beta = or_sigmoid(b[h]);
        float *Sh = S + h * D * D;
        for (int64_t i = 0; i < D * D; ++i) Sh[i] = Sh[i] * alpha;
        for (int64_t j = 0; j < D; ++j) {
            for (int64_t i = 0; i < D; ++i) tmp[i] = Sh[i * D + j] * kh[i];
            const float kv = or_tree(tmp, D);
            const float dv = v[j] - kv;
            const float d = beta * dv;
            for (int64_t i = 0; i < D; ++i) {
                const float u = kh[i] * d;
                Sh[i * D + j] = Sh[i * D + j] + u;
            }
        }
        for (int64_t j = 0; j < D; ++j) {
            for (int64_t i = 0; i < D; ++i) tmp[i] = Sh[i * D + j] * qh[i];
            o[j] = or_tree(tmp, D);
        }
        for (int64_t j = 0; j < D; ++j) tmp[j] = o[j] * o[j];
        const float mean = or_tree(tmp, D) / (float)D;
        const float r = 1.0f / sqrtf(mean + eps_n);
        for (int64_t j = 0; j < D; ++j) {
            const float on = o[j] * r;
            const float ow = on * nw[j];
            y[h * D + j] = ow * or_silu(z[h * D + j]);
        }
    }
    or_gsum(y, ysum, H * D);
    free(act);
    free(tmp);
    free(qh);
    free(kh);
    free(o);
}

/* ------------------------------------------------------------------------ */
/* atq: one token of gated attention over key and value caches.              */
/* [fused-token] Change, the Array.atq bullet, lists the phases -- q/k RMS   */
/* norm and rotation, the new k/v into the caches, scores, softmax, weighted */
/* values, sigmoid gate and group sums -- with one threadgroup per query     */
/* head; the first head of each KV group writes the cache row and the others */
/* use the new k/v, so no head reads a row another head writes.  The page    */
/* gives no formulas; the reading (grouped-query attention at position pos,  */
/* Hq query heads sharing Hkv key/value heads, head dimension D, the         */
/* rotation given as this position's cos/sin of each column pair):           */
/*   RMS(u) = 1 / sqrt(TREE(u*u) / D + eps)                                  */
/*   qn = (q_h * RMS(q_h)) * qn_w;  kn = (k_g * RMS(k_g)) * kn_w  (g = h/(Hq/Hkv)) */
/*   rotation of pairs (i, i + D/2), i < D/2:                                */
/*     r_i = u_i*cos_i - u_{i+D/2}*sin_i;  r_{i+D/2} = u_{i+D/2}*cos_i + u_i*sin_i */
/*   Kc[g][pos] = rot(kn), Vc[g][pos] = v_g                                  */
/*   s_t = TREE_j(rot(qn)_j * Kc[g][t][j]) * RN(1/RN(sqrt D)),  t = 0..pos    */
/*   m = max_t s_t;  e_t = EXP(s_t - m);  p_t = e_t / TREE_t(e_t)             */
/*   y_j = TREE_t(p_t * Vc[g][t][j]) * SIGMOID(gate_hj);  ysum = group sums  */
/* Caches [Hkv][P][D], pos < P; D a multiple of 64, at most 1024.            */
/* ------------------------------------------------------------------------ */
static void or_rms_rot(const float *u, const float *w, const float *cs, const float *sn, float eps, int64_t D,
                       float *tmp, float *out)
{
    for (int64_t i = 0; i < D; ++i) tmp[i] = u[i] * u[i];
    const float mean = or_tree(tmp, D) / (float)D;
    const float r = 1.0f / sqrtf(mean + eps);
    for (int64_t i = 0; i < D; ++i) {
        const float t = u[i] * r;
        tmp[i] = t * w[i];
    }
    const int64_t h = D / 2;
    for (int64_t i = 0; i < h; ++i) {
        const float a = tmp[i] * cs[i], b = tmp[i + h] * sn[i];
        const float c = tmp[i + h] * cs[i], d = tmp[i] * sn[i];
        out[i] = a - b;
        out[i + h] = c + d;
    }
}

void or_atq(const float *q, const float *gate, const float *k, const float *v, const float *qn_w,
            const float *kn_w, const float *cs, const float *sn, float *Kc, float *Vc, float *y, float *ysum,
            int64_t Hq, int64_t Hkv, int64_t D, int64_t P, int64_t pos, float eps)
{
    const int64_t n = pos + 1, per = Hq / Hkv;
    float *tmp = (float *)malloc((size_t)D * sizeof(float));
    float *qr = (float *)malloc((size_t)D * sizeof(float));
    float *s = (float *)malloc((size_t)n * sizeof(float));
    float *pv = (float *)malloc((size_t)n * sizeof(float));
    for (int64_t g = 0; g < Hkv; ++g) {
        or_rms_rot(k + g * D, kn_w, cs, sn, eps, D, tmp, Kc + (g * P + pos) * D);
        memcpy(Vc + (g * P + pos) * D, v + g * D, (size_t)D * sizeof(float));
    }
    const float scale = 1.0f / sqrtf((float)D);
    for (int64_t h = 0; h < Hq; ++h) {
        const int64_t g = h / per;
        or_rms_rot(q + h * D, qn_w, cs, sn, eps, D, tmp, qr);
        float m = -INFINITY;
        for (int64_t t = 0; t < n; ++t) {
            const float *kr = Kc + (g * P + t) * D;
            for (int64_t j = 0; j < D; ++j) tmp[j] = qr[j] * kr[j];
            s[t] = or_tree(tmp, D) * scale;
            if (s[t] > m) m = s[t];
        }
        for (int64_t t = 0; t < n; ++t) s[t] = or_exp(s[t] - m);
        const float Z = or_tree(s, n);
        for (int64_t t = 0; t < n; ++t) s[t] = s[t] / Z;
        for (int64_t j = 0; j < D; ++j) {
            for (int64_t t = 0; t < n; ++t) pv[t] = s[t] * Vc[(g * P + t) * D + j];
            const float o = or_tree(pv, n);
            y[h * D + j] = o * or_sigmoid(gate[h * D + j]);
        }
    }
    or_gsum(y, ysum, Hq * D);
    free(tmp);
    free(qr);
    free(s);
    free(pv);
}
