/*
 * kdt_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU restatement of DDTree tree-verify
 * MLA-absorb attention with visibility masking, in double precision. Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg load it; the
 * library's CUDA path never does, and this file shares no code, header, table or
 * helper with it.
 *
 * Sources (page titles of the method's write-up):
 *  - "The Verify-Attn Kernel: A Single File Write ..." -- section "The Design
 *    Journey: From Concept to CUDA": a score adds two dot products, the absorbed
 *    query against the latent row and the rope query against the rope key; a query
 *    sees only the shared prefix and its own ancestors; softmax with max
 *    subtraction; output is the latent (w_vc stays outside), section "Design
 *    Decisions and Trade-Offs"; the per-row
 *    log-sum-exp feeds the prefix/tail merge described there.
 *  - same page, section "Assumptions and the Path Forward": every query sees at
 *    least its own position.
 *  - "The Moment of Truth: Validating a Custom CUDA Attention Kernel ..." --
 *    section "Context": the visibility mask comes from the draft tree.
 *
 * Readings where the pages are silent:
 *  - tree node t of sequence b sits at cache row prefix_len[b] + t; the root is
 *    tree query 0 (parent -1); kv_len = prefix_len + T;
 *  - lse is the natural log of the sum of exp over the SCALED scores of the
 *    visible keys;
 *  - a row with no visible key (only possible with caller-supplied bits that
 *    lack the self bit and prefix 0) returns o = 0 and lse = -inf.
 *
 * Every function computes the plain definition: for each (b, i, h)
 *   V(b,i) = {0 .. prefix_len[b]-1} U {prefix_len[b] + t : t in anc*(i)}
 *   s_j    = scale * (sum_d<512 qn[d] c_kv[j,d] + sum_d<64 qp[d] k_pe[j,d])
 *   m = max_j s_j,  l = sum_j exp(s_j - m),  o = sum_j exp(s_j - m) c_kv[j,:] / l,
 *   lse = m + ln l
 * over j in V(b,i), everything in double, rounded to float32 at the end.
 * Visibility by explicit ancestor walk (not by any recurrence over words).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define DC 512
#define DR 64

/* ---- element access: exact widening of stored inputs to double ---------------- */

static double ld(const void *base, int dtype, size_t idx) {
    if (dtype == 0) {
        return (double)((const float *)base)[idx];
    } else {
        /* bf16 bit pattern: the top 16 bits of a float32 */
        uint32_t u = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
}

/* ---- visibility by ancestor walk -------------------------------------------- */

/* Returns 0, or 1 + (b*T + i) for the first entry (row-major) violating
 * -1 <= parent[b,i] < i. On success fills vis[B,T,W] (W = ceil(T/32)):
 * bit t of word t/32 (LSB first) of vis[b,i] is set iff tree node t is i or an
 * ancestor of i. Bits >= T are zero. */
int kdt_ref_build_visibility(const int32_t *parent, int B, int T, uint32_t *vis) {
    int W = (T + 31) / 32;
    for (long long k = 0; k < (long long)B * T; ++k) {
        int i = (int)(k % T);
        int p = parent[k];
        if (p < -1 || p >= i) return (int)(k + 1);
    }
    memset(vis, 0, sizeof(uint32_t) * (size_t)B * T * W);
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < T; ++i) {
            uint32_t *w = vis + ((size_t)b * T + i) * W;
            int j = i;
            while (j >= 0) {                       /* i itself, then each ancestor */
                w[j / 32] |= (uint32_t)1u << (j % 32);
                j = parent[(size_t)b * T + j];
            }
        }
    }
    return 0;
}

/* ---- attention ---------------------------------------------------------------- */

typedef struct {
    int B, T, H, dtype;
    const void *q_nope, *q_pe, *c_kv, *k_pe;
    long long L;
    const int32_t *prefix_len;
    const int32_t *parent;   /* [B,T] or NULL */
    const uint32_t *vis;     /* [B,T,W] or NULL */
    double scale;
} ref_args;

/* visible[j] for j < kv_len of (b, i). */
static void visible_set(const ref_args *a, int b, int i, unsigned char *visible, long long kv_len) {
    long long P = a->prefix_len[b];
    memset(visible, 0, (size_t)kv_len);
    for (long long j = 0; j < P; ++j) visible[j] = 1;          /* shared prefix */
    if (a->parent) {
        int j = i;
        while (j >= 0) {                                       /* self + ancestors */
            visible[P + j] = 1;
            j = a->parent[(size_t)b * a->T + j];
        }
    } else {
        int W = (a->T + 31) / 32;
        const uint32_t *w = a->vis + ((size_t)b * a->T + i) * W;
        for (int t = 0; t < a->T; ++t)
            if ((w[t / 32] >> (t % 32)) & 1u) visible[P + t] = 1;
    }
}

/* One row (b, i, h) in double. s is scratch of kv_len doubles. p_out, if not NULL,
 * receives the softmax weight of every j < L (0 for keys not in V). */
static void ref_row(const ref_args *a, int b, int i, int h, const unsigned char *visible,
                    double *s, double *o, double *lse, double *p_out) {
    long long kv_len = (long long)a->prefix_len[b] + a->T;
    size_t qrow = ((size_t)b * a->T + i) * a->H + h;
    double m = -INFINITY;
    for (long long j = 0; j < kv_len; ++j) {
        if (!visible[j]) continue;
        size_t krow = (size_t)b * a->L + j;
        double dot = 0.0;
        for (int d = 0; d < DC; ++d)
            dot += ld(a->q_nope, a->dtype, qrow * DC + d) * ld(a->c_kv, a->dtype, krow * DC + d);
        for (int d = 0; d < DR; ++d)
            dot += ld(a->q_pe, a->dtype, qrow * DR + d) * ld(a->k_pe, a->dtype, krow * DR + d);
        s[j] = a->scale * dot;
        if (s[j] > m) m = s[j];
    }
    for (int d = 0; d < DC; ++d) o[d] = 0.0;
    if (p_out)
        for (long long j = 0; j < a->L; ++j) p_out[j] = 0.0;
    if (m == -INFINITY) {            /* no visible key: o = 0, lse = -inf */
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (long long j = 0; j < kv_len; ++j)
        if (visible[j]) l += exp(s[j] - m);
    for (long long j = 0; j < kv_len; ++j) {
        if (!visible[j]) continue;
        double p = exp(s[j] - m) / l;
        size_t krow = (size_t)b * a->L + j;
        for (int d = 0; d < DC; ++d) o[d] += p * ld(a->c_kv, a->dtype, krow * DC + d);
        if (p_out) p_out[j] = p;
    }
    *lse = m + log(l);
}

static int check_args(const ref_args *a) {
    if (a->B < 0 || a->T < 1 || a->H < 1) return -2;
    if (!a->q_nope || !a->q_pe || !a->c_kv || !a->k_pe || !a->prefix_len) return -1;
    if ((a->parent == NULL) == (a->vis == NULL)) return -1;
    for (int b = 0; b < a->B; ++b)
        if (a->prefix_len[b] < 0 || (long long)a->prefix_len[b] + a->T > a->L) return -2;
    if (a->parent) {
        for (long long k = 0; k < (long long)a->B * a->T; ++k) {
            int i = (int)(k % a->T), p = a->parent[k];
            if (p < -1 || p >= i) return (int)(k + 1);
        }
    }
    return 0;
}

/* Rows given as flat indices r = (b*T + i)*H + h. Writes double outputs
 * (out64 [n,512], lse64 [n]) and/or float32 ones rounded to nearest (out32, lse32);
 * any of the four may be NULL. Returns 0, -1 (null/both-or-neither mask inputs),
 * -2 (bad shape) or 1 + first bad parent index. */
static int run_rows(const ref_args *a, const long long *rows, long long n,
                    double *out64, double *lse64, float *out32, float *lse32, int nthreads) {
    int rc = check_args(a);
    if (rc) return rc;
    long long maxkv = 0;
    for (int b = 0; b < a->B; ++b)
        if ((long long)a->prefix_len[b] + a->T > maxkv) maxkv = (long long)a->prefix_len[b] + a->T;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(maxkv > 0 ? maxkv : 1));
        unsigned char *vis = (unsigned char *)malloc((size_t)(maxkv > 0 ? maxkv : 1));
        double o[DC];
#pragma omp for schedule(dynamic, 1)
        for (long long k = 0; k < n; ++k) {
            long long r = rows ? rows[k] : k;
            int h = (int)(r % a->H);
            int i = (int)((r / a->H) % a->T);
            int b = (int)(r / ((long long)a->H * a->T));
            double lse;
            visible_set(a, b, i, vis, (long long)a->prefix_len[b] + a->T);
            ref_row(a, b, i, h, vis, s, o, &lse, NULL);
            for (int d = 0; d < DC; ++d) {
                if (out64) out64[(size_t)k * DC + d] = o[d];
                if (out32) out32[(size_t)k * DC + d] = (float)o[d];
            }
            if (lse64) lse64[k] = lse;
            if (lse32) lse32[k] = (float)lse;
        }
        free(s);
        free(vis);
    }
    return 0;
}

#define REF_ARGS_INIT                                                                  \
    ref_args a = {B, T, H, dtype, q_nope, q_pe, c_kv, k_pe, L, prefix_len, parent, vis, scale}

/* Full problem: out [B,T,H,512] float32, lse [B,T,H] float32 (lse may be NULL). */
int kdt_ref_verify_attn(int B, int T, int H, int dtype, const void *q_nope, const void *q_pe,
                        const void *c_kv, const void *k_pe, long long L, const int32_t *prefix_len,
                        const int32_t *parent, const uint32_t *vis, double scale, float *out,
                        float *lse, int nthreads) {
    REF_ARGS_INIT;
    if (!out) return -1;
    return run_rows(&a, NULL, (long long)B * T * H, NULL, NULL, out, lse, nthreads);
}

/* Selected rows only, float32 and/or double outputs. */
int kdt_ref_verify_attn_rows(int B, int T, int H, int dtype, const void *q_nope, const void *q_pe,
                             const void *c_kv, const void *k_pe, long long L,
                             const int32_t *prefix_len, const int32_t *parent, const uint32_t *vis,
                             double scale, const long long *rows, long long n, float *out32,
                             float *lse32, double *out64, double *lse64, int nthreads) {
    REF_ARGS_INIT;
    return run_rows(&a, rows, n, out64, lse64, out32, lse32, nthreads);
}

/* Softmax weights of one row over all cache rows j < L (0 where not visible). */
int kdt_ref_attn_weights(int B, int T, int H, int dtype, const void *q_nope, const void *q_pe,
                         const void *c_kv, const void *k_pe, long long L, const int32_t *prefix_len,
                         const int32_t *parent, const uint32_t *vis, double scale, long long row,
                         double *p_out) {
    REF_ARGS_INIT;
    int rc = check_args(&a);
    if (rc) return rc;
    int h = (int)(row % H), i = (int)((row / H) % T), b = (int)(row / ((long long)H * T));
    long long kv_len = (long long)prefix_len[b] + T;
    double *s = (double *)malloc(sizeof(double) * (size_t)kv_len);
    unsigned char *v = (unsigned char *)malloc((size_t)kv_len);
    double o[DC], lse;
    visible_set(&a, b, i, v, kv_len);
    ref_row(&a, b, i, h, v, s, o, &lse, p_out);
    free(s);
    free(v);
    return 0;
}

/* Merge two attention states over disjoint key sets by log-sum-exp:
 *   M = max(lse_a, lse_b), w_x = exp(lse_x - M),
 *   o = (w_a o_a + w_b o_b) / (w_a + w_b),  lse = M + ln(w_a + w_b),
 * with both -inf giving o = 0, lse = -inf. Double in, double out. This is the
 * prefix/tail combination the verify-attn page describes for long prefixes. */
void kdt_ref_merge_states(long long n, int D, const double *o_a, const double *lse_a,
                          const double *o_b, const double *lse_b, double *o, double *lse) {
    for (long long r = 0; r < n; ++r) {
        double la = lse_a[r], lb = lse_b[r];
        double M = la > lb ? la : lb;
        if (M == -INFINITY) {
            for (int d = 0; d < D; ++d) o[(size_t)r * D + d] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        double wa = exp(la - M), wb = exp(lb - M);
        for (int d = 0; d < D; ++d)
            o[(size_t)r * D + d] = (wa * o_a[(size_t)r * D + d] + wb * o_b[(size_t)r * D + d]) / (wa + wb);
        lse[r] = M + log(wa + wb);
    }
}

int kdt_ref_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
