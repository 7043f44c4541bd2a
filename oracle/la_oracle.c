/*
 * Plain fp64 CPU oracle for causal feature-map linear attention with the
 * BASED second-order Taylor feature map.  TEST INFRASTRUCTURE ONLY: the
 * library's GPU path never links, loads or calls this file; only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg do.
 *
 * Everything here is the textbook recurrence written out with plain loops,
 * in double precision, one (batch, head) pair at a time, with OpenMP over
 * the pairs only.  No blocking, fusion or reordering of the sums beyond what
 * the definitions below state.
 *
 * Sources (page title, section / equation):
 *  - "BASED: Simple linear attention language models balance the
 *    recall-throughput tradeoff" (reading notes), sec. 2.2 "from attention
 *    sums to a fixed-size state", Eqs. (1)-(3): the s/z recurrence and
 *    y_i = s_i^T phi(q_i) / z_i^T phi(q_i).
 *  - same page, sec. 2.3, Eq. (4) and the scaled form below it: the Taylor
 *    map phi(x) = [1, xbar, vec(xbar xbar^T)/sqrt(2)], xbar = x / d'^(1/4).
 *  - same page, sec. 2.5: the chunked (blockwise) form
 *    U_b = (M_b o Phi_Qb Phi_Kb^T) V_b + Phi_Qb S_<b  (oracle_prefill_chunked).
 *  - "Just read twice: closing the recall gap for recurrent language models"
 *    (reading notes), sec. 2.6, Eqs. (3)-(4): prefix linear attention, a
 *    non-causal state s_E, z_E over the first M positions of a second K/V
 *    set, added to the causal state for every output position.
 *  - same page, sec. 2.7 (inference with prompts shorter than M: left-pad to M
 *    and mask the padding in the prefix linear attention) and sec. 4.7 (the
 *    padding must be kept out of the linear-attention state): the padded
 *    variants below drop the first p_b positions of row b from every sum.
 *  - "Understanding and Improving Length Generalization in Recurrent Models"
 *    (reading notes), sec. 2.5 "non-zero initial state", Eq. (4): with the
 *    identity transition the initial state simply adds to the running sum.
 *  - same page, sec. 2.1, Eq. (1): the general recurrence h_t = A_t h_{t-1}
 *    + B_t x_t.  The decayed variants below take A_t = gamma_h I, a fixed
 *    per-head decay (BASED page, sec. 2.4: fixed per-head decay rates in some
 *    of its runs): s_t = gamma s_{t-1} + phi(k_t) v_t^T, z likewise, so the
 *    initial state reaches token t (0-based) as gamma^(t+1) s0 (sec. 2.5).
 *
 * Layouts (all dense, row-major, double):
 *   q, k   [B][H][N][dk]      v, y  [B][H][N][dv]
 *   ke     [B][H][M][dk]      ve    [B][H][M][dv]
 *   s      [B][H][D][dv]      z     [B][H][D]        D = 1 + dk + dk*dk
 * Feature index: 0 = constant, 1 + a = linear, 1 + dk + a*dk + b = quadratic.
 * s0 / z0 may be NULL (zero initial state); s_out / z_out may be NULL.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

long oracle_feature_dim(long dk) { return 1 + dk + dk * dk; }

/* phi(x) with xbar = x / dk^(1/4)  (BASED page, sec. 2.3). */
void oracle_phi(const double *x, long dk, double *phi) {
    const double scale = 1.0 / pow((double)dk, 0.25);
    const double inv_sqrt2 = 1.0 / sqrt(2.0);
    double xb[256];
    for (long a = 0; a < dk; ++a) xb[a] = x[a] * scale;
    phi[0] = 1.0;
    for (long a = 0; a < dk; ++a) phi[1 + a] = xb[a];
    for (long a = 0; a < dk; ++a)
        for (long b = 0; b < dk; ++b)
            phi[1 + dk + a * dk + b] = xb[a] * xb[b] * inv_sqrt2;
}

static double dot(const double *a, const double *b, long n) {
    double acc = 0.0;
    for (long i = 0; i < n; ++i) acc += a[i] * b[i];
    return acc;
}

/* One recurrent step on one head: s += phi(k) v^T, z += phi(k), then
 * y = phi(q)^T s / (phi(q)^T z + eps).  The state includes the current token
 * before it is read (BASED page, Eq. (2): y_i uses s_i, not s_{i-1}). */
static void step_decay(const double *q, const double *k, const double *v, double *s,
                       double *z, double *y, long dk, long dv, double eps,
                       double *phq, double *phk, double gamma, int decay) {
    const long D = oracle_feature_dim(dk);
    oracle_phi(k, dk, phk);
    oracle_phi(q, dk, phq);
    for (long f = 0; f < D; ++f) {
        if (decay) {
            for (long c = 0; c < dv; ++c) s[f * dv + c] = gamma * s[f * dv + c] + phk[f] * v[c];
            z[f] = gamma * z[f] + phk[f];
        } else {
            for (long c = 0; c < dv; ++c) s[f * dv + c] += phk[f] * v[c];
            z[f] += phk[f];
        }
    }
    const double den = dot(phq, z, D) + eps;
    for (long c = 0; c < dv; ++c) {
        double num = 0.0;
        for (long f = 0; f < D; ++f) num += phq[f] * s[f * dv + c];
        y[c] = num / den;
    }
}

static void step(const double *q, const double *k, const double *v, double *s,
                 double *z, double *y, long dk, long dv, double eps,
                 double *phq, double *phk) {
    step_decay(q, k, v, s, z, y, dk, dv, eps, phq, phk, 1.0, 0);
}

static void load_state(const double *s0, const double *z0, long bh, long D,
                       long dv, double *s, double *z) {
    if (s0) memcpy(s, s0 + bh * D * dv, sizeof(double) * D * dv);
    else memset(s, 0, sizeof(double) * D * dv);
    if (z0) memcpy(z, z0 + bh * D, sizeof(double) * D);
    else memset(z, 0, sizeof(double) * D);
}

static void store_state(double *s_out, double *z_out, long bh, long D, long dv,
                        const double *s, const double *z) {
    if (s_out) memcpy(s_out + bh * D * dv, s, sizeof(double) * D * dv);
    if (z_out) memcpy(z_out + bh * D, z, sizeof(double) * D);
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Prefix linear attention (Just read twice page, sec. 2.6):
 *   s_E = sum_{j<=M} phi(ke_j) ve_j^T,   z_E = sum_{j<=M} phi(ke_j),
 *   y_i = phi(q_i)(s0 + s_E + s_{D,i}) / phi(q_i)(z0 + z_E + z_{D,i}).
 * M = 0 (or ke == NULL) is plain causal linear attention from (s0, z0).
 * The returned state is s0 + s_E + s_{D,N} (the merge of Eq. (4)).
 *
 * Left padding (same page, sec. 2.7 and 4.7): with left_pad != NULL, row b's
 * first p = left_pad[b] positions (0 <= p <= N) are padding.  Prefix
 * positions j < min(p, M) and causal positions i < p are left out of every
 * sum, and y_i = 0 for i < p.  left_pad == NULL means no padding. */
int oracle_prefix_prefill_padded(const double *q, const double *k, const double *v,
                                 const double *ke, const double *ve, long M,
                                 const double *s0, const double *z0, const long *left_pad,
                                 double *y, double *s_out, double *z_out, long B, long H,
                                 long N, long dk, long dv, double eps, int nthreads) {
    if (dk < 1 || dk > 256 || dv < 1 || B < 0 || H < 0 || N < 0 || M < 0)
        return 1;
    for (long b = 0; left_pad && b < B; ++b)
        if (left_pad[b] < 0 || left_pad[b] > N) return 1;
    const long D = oracle_feature_dim(dk);
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *s = malloc(sizeof(double) * D * dv);
        double *z = malloc(sizeof(double) * D);
        double *phq = malloc(sizeof(double) * D);
        double *phk = malloc(sizeof(double) * D);
        if (!s || !z || !phq || !phk) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long bh = 0; bh < B * H; ++bh) {
                const long pad = left_pad ? left_pad[bh / H] : 0;
                load_state(s0, z0, bh, D, dv, s, z);
                /* non-causal prefix state over the second K/V set */
                for (long j = pad < M ? pad : M; ke && j < M; ++j) {
                    oracle_phi(ke + (bh * M + j) * dk, dk, phk);
                    const double *vj = ve + (bh * M + j) * dv;
                    for (long f = 0; f < D; ++f) {
                        for (long c = 0; c < dv; ++c) s[f * dv + c] += phk[f] * vj[c];
                        z[f] += phk[f];
                    }
                }
                /* causal path over all N positions (padding: y = 0, no state change) */
                for (long i = 0; i < N; ++i) {
                    const long t = bh * N + i;
                    if (i < pad) {
                        for (long c = 0; c < dv; ++c) y[t * dv + c] = 0.0;
                        continue;
                    }
                    step(q + t * dk, k + t * dk, v + t * dv, s, z, y + t * dv,
                         dk, dv, eps, phq, phk);
                }
                store_state(s_out, z_out, bh, D, dv, s, z);
            }
        }
        free(s); free(z); free(phq); free(phk);
    }
    return err;
}

int oracle_prefix_prefill(const double *q, const double *k, const double *v,
                          const double *ke, const double *ve, long M,
                          const double *s0, const double *z0, double *y,
                          double *s_out, double *z_out, long B, long H, long N,
                          long dk, long dv, double eps, int nthreads) {
    return oracle_prefix_prefill_padded(q, k, v, ke, ve, M, s0, z0, NULL, y, s_out, z_out,
                                        B, H, N, dk, dv, eps, nthreads);
}

/* Causal prefill from an optional initial state (BASED page Eqs. (1)-(3);
 * length-generalization page, Eq. (4) with A_t = I). */
int oracle_prefill(const double *q, const double *k, const double *v,
                   const double *s0, const double *z0, double *y, double *s_out,
                   double *z_out, long B, long H, long N, long dk, long dv,
                   double eps, int nthreads) {
    return oracle_prefix_prefill(q, k, v, NULL, NULL, 0, s0, z0, y, s_out, z_out,
                                 B, H, N, dk, dv, eps, nthreads);
}

/* Causal prefill with a fixed per-head decay gamma[h] (0 <= gamma <= 1):
 *   s_i = gamma s_{i-1} + phi(k_i) v_i^T,  z_i = gamma z_{i-1} + phi(k_i),
 *   y_i = phi(q_i)^T s_i / (phi(q_i)^T z_i + eps),  s_{-1} = s0, z_{-1} = z0
 * (length-generalization page, Eq. (1) with A_t = gamma I; Eq. (4)). */
int oracle_prefill_decay(const double *q, const double *k, const double *v,
                         const double *s0, const double *z0, const double *gamma,
                         double *y, double *s_out, double *z_out, long B, long H, long N,
                         long dk, long dv, double eps, int nthreads) {
    if (dk < 1 || dk > 256 || dv < 1 || B < 0 || H < 0 || N < 0 || !gamma) return 1;
    for (long h = 0; h < H; ++h)
        if (!(gamma[h] >= 0.0 && gamma[h] <= 1.0)) return 1;
    const long D = oracle_feature_dim(dk);
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *s = malloc(sizeof(double) * D * dv);
        double *z = malloc(sizeof(double) * D);
        double *phq = malloc(sizeof(double) * D);
        double *phk = malloc(sizeof(double) * D);
        if (!s || !z || !phq || !phk) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long bh = 0; bh < B * H; ++bh) {
                load_state(s0, z0, bh, D, dv, s, z);
                for (long i = 0; i < N; ++i) {
                    const long t = bh * N + i;
                    step_decay(q + t * dk, k + t * dk, v + t * dv, s, z, y + t * dv, dk, dv,
                               eps, phq, phk, gamma[bh % H], 1);
                }
                store_state(s_out, z_out, bh, D, dv, s, z);
            }
        }
        free(s); free(z); free(phq); free(phk);
    }
    return err;
}

/* One decode step per (b, h): the same recurrence for a single token.
 * q, k [B][H][dk], v, y [B][H][dv]; s_out may equal s_in (in place). */
int oracle_decode_step_decay(const double *q, const double *k, const double *v,
                             const double *gamma, const double *s_in, const double *z_in,
                             double *s_out, double *z_out, double *y, long B, long H,
                             long dk, long dv, double eps, int nthreads) {
    if (dk < 1 || dk > 256 || dv < 1 || B < 0 || H < 0) return 1;
    for (long h = 0; gamma && h < H; ++h)
        if (!(gamma[h] >= 0.0 && gamma[h] <= 1.0)) return 1;
    const long D = oracle_feature_dim(dk);
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *s = malloc(sizeof(double) * D * dv);
        double *z = malloc(sizeof(double) * D);
        double *phq = malloc(sizeof(double) * D);
        double *phk = malloc(sizeof(double) * D);
        if (!s || !z || !phq || !phk) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(static)
            for (long bh = 0; bh < B * H; ++bh) {
                load_state(s_in, z_in, bh, D, dv, s, z);
                step_decay(q + bh * dk, k + bh * dk, v + bh * dv, s, z, y + bh * dv, dk,
                           dv, eps, phq, phk, gamma ? gamma[bh % H] : 1.0, gamma != NULL);
                store_state(s_out, z_out, bh, D, dv, s, z);
            }
        }
        free(s); free(z); free(phq); free(phk);
    }
    return err;
}

int oracle_decode_step(const double *q, const double *k, const double *v,
                       const double *s_in, const double *z_in, double *s_out,
                       double *z_out, double *y, long B, long H, long dk,
                       long dv, double eps, int nthreads) {
    return oracle_decode_step_decay(q, k, v, NULL, s_in, z_in, s_out, z_out, y, B, H, dk, dv,
                                    eps, nthreads);
}

/* The blockwise form of the same prefill (BASED page, sec. 2.5):
 *   num_b = (M_b o Phi_Qb Phi_Kb^T) V_b + Phi_Qb S_<b
 *   den_b = (M_b o Phi_Qb Phi_Kb^T) 1   + Phi_Qb z_<b
 *   S_<b+1 = S_<b + Phi_Kb^T V_b,  z_<b+1 = z_<b + Phi_Kb^T 1
 * with M_b the causal mask j <= i inside the block.  The last block may be
 * short.  Used only to check that chunking is an exact re-association. */
int oracle_prefill_chunked(const double *q, const double *k, const double *v,
                           const double *s0, const double *z0, double *y,
                           double *s_out, double *z_out, long B, long H, long N,
                           long dk, long dv, long C, double eps, int nthreads) {
    if (dk < 1 || dk > 256 || dv < 1 || C < 1 || B < 0 || H < 0 || N < 0) return 1;
    const long D = oracle_feature_dim(dk);
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *s = malloc(sizeof(double) * D * dv);
        double *z = malloc(sizeof(double) * D);
        double *PQ = malloc(sizeof(double) * C * D);
        double *PK = malloc(sizeof(double) * C * D);
        double *A = malloc(sizeof(double) * C * C);
        if (!s || !z || !PQ || !PK || !A) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long bh = 0; bh < B * H; ++bh) {
                load_state(s0, z0, bh, D, dv, s, z);
                for (long c0 = 0; c0 < N; c0 += C) {
                    const long L = (N - c0 < C) ? (N - c0) : C;
                    for (long i = 0; i < L; ++i) {
                        const long t = bh * N + c0 + i;
                        oracle_phi(q + t * dk, dk, PQ + i * D);
                        oracle_phi(k + t * dk, dk, PK + i * D);
                    }
                    /* intra-block kernel matrix, causally masked */
                    for (long i = 0; i < L; ++i)
                        for (long j = 0; j < L; ++j)
                            A[i * C + j] = (j <= i) ? dot(PQ + i * D, PK + j * D, D) : 0.0;
                    for (long i = 0; i < L; ++i) {
                        const long t = bh * N + c0 + i;
                        double den = dot(PQ + i * D, z, D);
                        for (long j = 0; j < L; ++j) den += A[i * C + j];
                        for (long c = 0; c < dv; ++c) {
                            double num = 0.0;
                            for (long f = 0; f < D; ++f) num += PQ[i * D + f] * s[f * dv + c];
                            for (long j = 0; j < L; ++j)
                                num += A[i * C + j] * v[(bh * N + c0 + j) * dv + c];
                            y[t * dv + c] = num / (den + eps);
                        }
                    }
                    /* carry the state past this block */
                    for (long j = 0; j < L; ++j) {
                        const double *vj = v + (bh * N + c0 + j) * dv;
                        for (long f = 0; f < D; ++f) {
                            for (long c = 0; c < dv; ++c) s[f * dv + c] += PK[j * D + f] * vj[c];
                            z[f] += PK[j * D + f];
                        }
                    }
                }
                store_state(s_out, z_out, bh, D, dv, s, z);
            }
        }
        free(s); free(z); free(PQ); free(PK); free(A);
    }
    return err;
}
