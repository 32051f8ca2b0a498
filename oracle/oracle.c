/*
 * oracle.c -- plain, slow, scalar CPU oracle for the deterministic gated BF16 FFN.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only tests/, the smoke check and the CPU-baseline leg of the benchmark load it.
 * It shares no code, header or table with the CUDA library; it has its own
 * BF16/FP16 rounding helpers and its own SiLU tables.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread (no -ffast-math,
 * no FTZ/DAZ), so every float operation below is one IEEE-754 binary32
 * operation rounded to nearest-even.
 *
 * Source of the method (RL-Kernel PR #325, "feat(ffn): add deterministic
 * distributed Triton FFN for ROCm"):
 *   - Design: "canonical FP32-leaf/BF16-node midpoint reduction tree in
 *     deterministic GEMM", "preserve BF16 stage boundaries in forward and
 *     backward", "each contiguous TP K shard the same subtree used by TP=1",
 *     "fixed balanced BF16 rank reduction tree".
 * Rank tree arithmetic ((rank0 + rank1) + (rank2 + rank3)) + ... for FP32,
 * FP16 and BF16: PR #357 "optimize deterministic ROCm collectives with HIP
 * IPC", Design; PR #356 "add deterministic ROCm/RCCL transport collectives",
 * Design.
 *
 * Readings of points the pages leave open (each also listed in the design notes):
 *   leaf width      : 64 by default, parameter LW.
 *   in-leaf order   : SEQ  = ascending acc = fma(a_k, b_k, acc) from +0.0f;
 *                     LANE = 8 groups of LW/8 contiguous elements, each summed
 *                            SEQ from +0.0f, then ((s0+s1)+(s2+s3))+((s4+s5)+(s6+s7)).
 *                     A bf16*bf16 product is exact in binary32 (8+8 <= 24
 *                     significand bits), so fma(a,b,acc) == acc + a*b except
 *                     when the product under/overflows; fmaf() is the definition.
 *   midpoint split  : left child takes floor(n/2) leaves.
 *   node            : rne_bf16( (float)left + (float)right ).
 *   output          : rne_bf16(root); K == 0 gives +0.
 *   NaN             : rounds to the quiet NaN 0x7FC0 (sign kept); tests treat
 *                     every NaN encoding as one class.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------ */
/* Element rounding                                                          */
/* ------------------------------------------------------------------------ */

static inline uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static inline float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* binary32 -> bfloat16, round to nearest, ties to even.  Overflow goes to
 * +-Inf through the carry into the exponent; subnormals are kept. */
uint16_t or_rne_bf16(float v)
{
    uint32_t u = f2u(v);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7fc0u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* bfloat16 -> binary32: exact widening. */
float or_bf16_f32(uint16_t b) { return u2f((uint32_t)b << 16); }

/* binary32 -> binary16, round to nearest, ties to even, with subnormals. */
uint16_t or_rne_f16(float v)
{
    uint32_t u = f2u(v);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);
    if (a == 0x7f800000u) return (uint16_t)(sign | 0x7c00u);
    int e = (int)(a >> 23);
    if (e == 0) return sign; /* binary32 subnormals are < 2^-126, far below half the least fp16 subnormal */
    uint32_t m = (a & 0x7fffffu) | 0x800000u; /* value = m * 2^(x-23) */
    int x = e - 127;
    int ulp_exp = (x >= -14) ? (x - 10) : -24; /* exponent of one unit in the last place of the result */
    int shift = ulp_exp - (x - 23);            /* low bits of m that fall below that unit (>= 13) */
    uint32_t q;
    if (shift >= 32) {
        q = 0;
    } else {
        q = m >> shift;
        uint32_t rem = m & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        if (rem > half || (rem == half && (q & 1u))) q++;
    }
    if (x >= -14) {
        int E = x + 15;
        if (q == 0x800u) { q = 0x400u; E++; }
        if (E >= 31) return (uint16_t)(sign | 0x7c00u);
        return (uint16_t)(sign | ((uint32_t)E << 10) | (q & 0x3ffu));
    }
    return (uint16_t)(sign | q); /* q == 0x400 encodes the least normal number */
}

/* binary16 -> binary32: exact widening. */
float or_f16_f32(uint16_t h)
{
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t E = (h >> 10) & 0x1fu, m = h & 0x3ffu;
    if (E == 0x1f) return u2f(sign | 0x7f800000u | (m << 13));
    if (E == 0) {
        float v = (float)m * 0x1p-24f; /* exact: m < 2^10 */
        return sign ? -v : v;
    }
    return u2f(sign | ((E + 112u) << 23) | (m << 13));
}

void or_cvt_f32_bf16(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = or_rne_bf16(in[i]);
}
void or_cvt_f32_f16(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = or_rne_f16(in[i]);
}
void or_cvt_f16_f32(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = or_f16_f32(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Leaves and the canonical tree                                             */
/* ------------------------------------------------------------------------ */

enum { OR_SEQ = 0, OR_LANE = 1 };

/* One leaf: a partial dot product over len <= lw contiguous K positions,
 * a[k*sa] * b[k*sb].  Missing positions of a partial leaf contribute nothing. */
float or_leaf(const uint16_t *a, int64_t sa, const uint16_t *b, int64_t sb,
              int64_t len, int lw, int order)
{
    if (order == OR_SEQ) {
        float acc = 0.0f;
        for (int64_t k = 0; k < len; k++)
            acc = fmaf(or_bf16_f32(a[k * sa]), or_bf16_f32(b[k * sb]), acc);
        return acc;
    }
    /* LANE: eight groups of lw/8 contiguous positions. */
    int gw = lw / 8;
    float s[8];
    for (int g = 0; g < 8; g++) {
        float acc = 0.0f;
        for (int e = 0; e < gw; e++) {
            int64_t k = (int64_t)g * gw + e;
            if (k < len)
                acc = fmaf(or_bf16_f32(a[k * sa]), or_bf16_f32(b[k * sb]), acc);
        }
        s[g] = acc;
    }
    float p01 = s[0] + s[1], p23 = s[2] + s[3], p45 = s[4] + s[5], p67 = s[6] + s[7];
    float q0 = p01 + p23, q1 = p45 + p67;
    return q0 + q1;
}

/* Node value over leaves [lo, hi): an FP32 leaf when it is a single leaf,
 * otherwise the BF16 node rne_bf16(left + right), returned widened. */
static float tree_rec(const float *lv, int64_t lo, int64_t hi)
{
    if (hi - lo == 1) return lv[lo];
    int64_t mid = lo + (hi - lo) / 2;
    float l = tree_rec(lv, lo, mid);
    float r = tree_rec(lv, mid, hi);
    return or_bf16_f32(or_rne_bf16(l + r));
}

/* Output element from L leaves: rne_bf16(root); L == 0 gives +0. */
uint16_t or_tree_from_leaves(const float *lv, int64_t L)
{
    if (L <= 0) return 0;
    return or_rne_bf16(tree_rec(lv, 0, L));
}

/* Root of the subtree over leaves [lo, hi) as a raw float (no output rounding). */
float or_tree_node(const float *lv, int64_t lo, int64_t hi) { return tree_rec(lv, lo, hi); }

static int64_t n_leaves(int64_t K, int lw) { return (K + lw - 1) / lw; }

static void leaves_of(const uint16_t *a, int64_t sa, const uint16_t *b, int64_t sb,
                      int64_t K, int lw, int order, float *lv)
{
    int64_t L = n_leaves(K, lw);
    for (int64_t j = 0; j < L; j++) {
        int64_t k0 = j * lw;
        int64_t len = (K - k0 < lw) ? (K - k0) : lw;
        lv[j] = or_leaf(a + k0 * sa, sa, b + k0 * sb, sb, len, lw, order);
    }
}

/* ------------------------------------------------------------------------ */
/* Tree GEMM: C[r, c] = T_K( A[r, :], B[c, :] ) with arbitrary strides.       */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *A; int64_t a_rs, a_ks;
    const uint16_t *B; int64_t b_rs, b_ks;
    int64_t R, C, K;
    uint16_t *out; int64_t o_rs, o_cs;
    float *leaves_out; /* optional [R, C, L] */
    int lw, order;
    int64_t r0, r1;
} gemm_job;

static void *gemm_worker(void *p)
{
    gemm_job *j = (gemm_job *)p;
    int64_t L = n_leaves(j->K, j->lw);
    float *lv = (float *)malloc((size_t)(L > 0 ? L : 1) * sizeof(float));
    for (int64_t r = j->r0; r < j->r1; r++) {
        for (int64_t c = 0; c < j->C; c++) {
            leaves_of(j->A + r * j->a_rs, j->a_ks, j->B + c * j->b_rs, j->b_ks,
                      j->K, j->lw, j->order, lv);
            if (j->out) j->out[r * j->o_rs + c * j->o_cs] = or_tree_from_leaves(lv, L);
            if (j->leaves_out)
                memcpy(j->leaves_out + (r * j->C + c) * L, lv, (size_t)L * sizeof(float));
        }
    }
    free(lv);
    return NULL;
}

static int pick_threads(int nthreads, int64_t rows)
{
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > rows) nthreads = (int)(rows > 0 ? rows : 1);
    return nthreads;
}

void or_tree_gemm(const uint16_t *A, int64_t a_rs, int64_t a_ks,
                  const uint16_t *B, int64_t b_rs, int64_t b_ks,
                  int64_t R, int64_t C, int64_t K,
                  uint16_t *out, int64_t o_rs, int64_t o_cs,
                  float *leaves_out, int lw, int order, int nthreads)
{
    int nt = pick_threads(nthreads, R);
    pthread_t th[256];
    gemm_job jobs[256];
    for (int t = 0; t < nt; t++) {
        gemm_job j = {A, a_rs, a_ks, B, b_rs, b_ks, R, C, K, out, o_rs, o_cs,
                      leaves_out, lw, order, R * t / nt, R * (t + 1) / nt};
        jobs[t] = j;
    }
    if (nt == 1) { gemm_worker(&jobs[0]); return; }
    for (int t = 0; t < nt; t++) pthread_create(&th[t], NULL, gemm_worker, &jobs[t]);
    for (int t = 0; t < nt; t++) pthread_join(th[t], NULL);
}

/* Replays the tree over n_elem independent rows of L leaves each. */
void or_tree_replay(const float *leaves, int64_t n_elem, int64_t L, uint16_t *out)
{
    for (int64_t e = 0; e < n_elem; e++) out[e] = or_tree_from_leaves(leaves + e * L, L);
}

/* ------------------------------------------------------------------------ */
/* SiLU and its derivative as functions of the 16-bit gate value.            */
/* ------------------------------------------------------------------------ */

/* Double-double arithmetic (value = hi + lo, |lo| <= ulp(hi)/2), used so that
 * the SiLU tables are the correctly rounded values of the real functions:
 * a binary64 evaluation misses near-ties (e.g. dsilu at tiny g, where the
 * rounding is decided by an O(g^3) term). */
typedef struct { double hi, lo; } dd;

static dd dd_two_sum(double a, double b)
{
    double s = a + b, bb = s - a;
    dd r = {s, (a - (s - bb)) + (b - bb)};
    return r;
}
static dd dd_fast(double a, double b)
{
    double s = a + b;
    dd r = {s, b - (s - a)};
    return r;
}
static dd dd_d(double a) { dd r = {a, 0.0}; return r; }
static dd dd_add(dd a, dd b)
{
    dd s = dd_two_sum(a.hi, b.hi), t = dd_two_sum(a.lo, b.lo);
    s.lo += t.hi;
    s = dd_fast(s.hi, s.lo);
    s.lo += t.lo;
    return dd_fast(s.hi, s.lo);
}
static dd dd_neg(dd a) { dd r = {-a.hi, -a.lo}; return r; }
static dd dd_mul(dd a, dd b)
{
    double p = a.hi * b.hi;
    double e = fma(a.hi, b.hi, -p);
    e += a.hi * b.lo;
    e += a.lo * b.hi;
    return dd_fast(p, e);
}
static dd dd_div(dd a, dd b)
{
    double q1 = a.hi / b.hi;
    dd r = dd_add(a, dd_neg(dd_mul(b, dd_d(q1))));
    double q2 = r.hi / b.hi;
    r = dd_add(r, dd_neg(dd_mul(b, dd_d(q2))));
    double q3 = r.hi / b.hi;
    return dd_add(dd_fast(q1, q2), dd_d(q3));
}
static dd dd_ldexp(dd a, int k) { dd r = {ldexp(a.hi, k), ldexp(a.lo, k)}; return r; }

/* e^x for a finite double x with -740 < x < 700: x = k*ln2 + r, r scaled by
 * 2^-10, Taylor series of e^r - 1, then ten squarings of (1 + p). */
static dd dd_exp(double x)
{
    static const dd LN2 = {0x1.62e42fefa39efp-1, 0x1.abc9e3b39803fp-56};
    double k = nearbyint(x / LN2.hi);
    dd r = dd_add(dd_d(x), dd_neg(dd_mul(LN2, dd_d(k))));
    r = dd_ldexp(r, -10);
    dd p = dd_d(0.0);
    /* Horner form of e^r - 1 = r*(1 + r/2*(1 + r/3*(1 + ... r/14))). */
    for (int n = 14; n >= 1; n--) {
        p = dd_mul(dd_add(p, dd_d(1.0)), r);
        p = dd_div(p, dd_d((double)n));
    }
    for (int i = 0; i < 10; i++) p = dd_add(dd_add(p, p), dd_mul(p, p)); /* (1+p)^2 - 1 */
    return dd_ldexp(dd_add(dd_d(1.0), p), (int)k);
}

/* Correct rounding of a double-double to binary32 (ties to even). */
static float dd_to_f32(dd v)
{
    float f = (float)v.hi;
    double diff = v.hi - (double)f; /* exact */
    if (diff != 0.0 && v.lo != 0.0 && (diff > 0) == (v.lo > 0)) {
        float nb = nextafterf(f, diff > 0 ? INFINITY : -INFINITY);
        double half = ((double)nb - (double)f) / 2.0;
        if (diff == half) f = nb; /* hi sat exactly on the midpoint; lo breaks the tie */
    }
    return f;
}

/* silu[g]  = rne_bf16( RN_f32( g * sigma(g) ) )
 * dsilu[g] = RN_f32( sigma(g) * (1 + g * (1 - sigma(g))) ), the derivative of
 * g*sigma(g); both are correctly rounded values of the real functions.
 * Infinite gates take the limits: silu(+inf)=+inf, d=1; silu(-inf)=-0, d=0.
 * Below g = -200 both values are far under half the least binary32 subnormal
 * and round to -0; above g = 200, sigma(g) rounds to 1 in double-double. */
void or_silu_tables(uint16_t *silu, float *dsilu)
{
    for (uint32_t i = 0; i < 65536u; i++) {
        float gf = or_bf16_f32((uint16_t)i);
        double g = (double)gf;
        if (isnan(g)) {
            silu[i] = or_rne_bf16(gf);
            dsilu[i] = gf;
        } else if (g > 200.0) {
            silu[i] = or_rne_bf16(gf);
            dsilu[i] = 1.0f;
        } else if (g < -200.0) {
            silu[i] = 0x8000;
            dsilu[i] = -0.0f;
        } else {
            dd t = dd_exp(-g);                     /* e^-g */
            dd den = dd_add(dd_d(1.0), t);
            dd s = dd_div(dd_d(1.0), den);         /* sigma(g) */
            dd oms = dd_div(t, den);               /* 1 - sigma(g), without cancellation */
            dd y = dd_mul(dd_d(g), s);
            dd d = dd_mul(s, dd_add(dd_d(1.0), dd_mul(dd_d(g), oms)));
            silu[i] = (g == 0.0) ? (uint16_t)i : or_rne_bf16(dd_to_f32(y));
            dsilu[i] = dd_to_f32(d);
        }
    }
}

static uint16_t g_silu[65536];
static float g_dsilu[65536];
static int g_tables_ready = 0;
static pthread_mutex_t g_tab_mu = PTHREAD_MUTEX_INITIALIZER;

static void tables(void)
{
    pthread_mutex_lock(&g_tab_mu);
    if (!g_tables_ready) { or_silu_tables(g_silu, g_dsilu); g_tables_ready = 1; }
    pthread_mutex_unlock(&g_tab_mu);
}

/* Forward stage boundary: a = silu_bf16(g); h = rne_bf16(a * u) (the product
 * of two bf16 values is exact in binary32, so this is one rounding). */
void or_silu_mul(const uint16_t *gate, const uint16_t *up, int64_t n, uint16_t *h)
{
    tables();
    for (int64_t i = 0; i < n; i++) {
        float a = or_bf16_f32(g_silu[gate[i]]);
        h[i] = or_rne_bf16(a * or_bf16_f32(up[i]));
    }
}

/* Backward stage boundary:
 *   dU = rne_bf16(dh * a), dA = rne_bf16(dh * u),
 *   dG = rne_bf16( rne_f32( dA * dsilu(g) ) ). */
void or_silu_bwd(const uint16_t *dh, const uint16_t *gate, const uint16_t *up, int64_t n,
                 uint16_t *dU, uint16_t *dA, uint16_t *dG)
{
    tables();
    for (int64_t i = 0; i < n; i++) {
        float d = or_bf16_f32(dh[i]);
        float a = or_bf16_f32(g_silu[gate[i]]);
        float u = or_bf16_f32(up[i]);
        uint16_t du = or_rne_bf16(d * a);
        uint16_t da = or_rne_bf16(d * u);
        float dg32 = or_bf16_f32(da) * g_dsilu[gate[i]];
        if (dU) dU[i] = du;
        if (dA) dA[i] = da;
        if (dG) dG[i] = or_rne_bf16(dg32);
    }
}

/* dX = rne_bf16(cg + cu): the gate contribution first, then the up one. */
void or_add_bf16(const uint16_t *a, const uint16_t *b, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = or_rne_bf16(or_bf16_f32(a[i]) + or_bf16_f32(b[i]));
}

/* ------------------------------------------------------------------------ */
/* Rank tree: ((b0 + b1) + (b2 + b3)) + ..., rounded in the buffer dtype.     */
/* ------------------------------------------------------------------------ */

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };

static float load_elem(const void *p, int64_t i, int dtype)
{
    if (dtype == OR_F32) return ((const float *)p)[i];
    if (dtype == OR_F16) return or_f16_f32(((const uint16_t *)p)[i]);
    return or_bf16_f32(((const uint16_t *)p)[i]);
}

static float round_to(float v, int dtype)
{
    if (dtype == OR_F32) return v;
    if (dtype == OR_F16) return or_f16_f32(or_rne_f16(v));
    return or_bf16_f32(or_rne_bf16(v));
}

static float rank_rec(const void *const *in, int lo, int hi, int64_t i, int dtype)
{
    if (hi - lo == 1) return load_elem(in[lo], i, dtype);
    int mid = lo + (hi - lo) / 2;
    float l = rank_rec(in, lo, mid, i, dtype);
    float r = rank_rec(in, mid, hi, i, dtype);
    return round_to(l + r, dtype);
}

/* n in {1, 2, 4, 8}; returns 0 on success, -1 for an unsupported n or dtype. */
int or_rank_tree(const void *const *in, int n, int64_t count, int dtype, void *out)
{
    if (!(n == 1 || n == 2 || n == 4 || n == 8)) return -1;
    if (dtype < 0 || dtype > 2) return -1;
    for (int64_t i = 0; i < count; i++) {
        float v = rank_rec(in, 0, n, i, dtype);
        if (dtype == OR_F32) ((float *)out)[i] = v;
        else if (dtype == OR_F16) ((uint16_t *)out)[i] = or_rne_f16(v);
        else ((uint16_t *)out)[i] = or_rne_bf16(v);
    }
    return 0;
}
