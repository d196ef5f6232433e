/*
 * oracle.c -- plain fp64 CPU oracle for the linear-attention segment scan and
 * state composition of position-independent caching (HYPIC).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The GPU library shares
 * no code, header, helper or constant with it, and neither includes the other.
 *
 * Sources (web pages about HYPIC):
 *   [xix-fr] xix.ai/fr "Xiaohongshu, l'Université de Pékin ... dévoilent HYPIC",
 *            paragraph on linear layers ("opérateurs de transition"): the
 *            segment operator T_C is the product of all per-token transition
 *            matrices of the segment; S(C|0) is the final state from a zero
 *            start; S(C1.C2) = T(C2).S(C1) + S(C2); the families are decay,
 *            gating and delta-erasure variants (RetNet, Mamba2, GLA, DeltaNet,
 *            GDN).
 *   [remio-ja] remio.ai/ja "HYPIC ...", section "how HYPIC composes states":
 *            the cached transition is applied to the running state and the
 *            zero-start contribution is added.
 *
 * The pages print no per-token rule.  This file takes the plainest reading:
 *   S_t = T_t S_{t-1} + beta_t k_t v_t^T,   S in R^{dk x dv}, fp64,
 *     scalar : T_t = alpha_t I                      (RetNet / Mamba2)
 *     diag   : T_t = diag(alpha_t), alpha_t in R^dk (GLA, gates the key axis)
 *     dense  : T_t = alpha_t (I - beta_t k_t k_t^T) (gated delta rule)
 *     kda    : T_t = diag(alpha_t) (I - beta_t k_t k_t^T), alpha_t in R^dk
 *              (the pages name KDA among the delta-erasure variants and give no
 *              rule; this is the gated delta rule with its scalar gate made
 *              per channel)
 *   beta_t defaults to 1 when no beta is given.
 *   T_C = T_L ... T_1 ;  S(C|0) = S_L from S_0 = 0 ;  o_t = S_t^T q_t.
 * T_C is returned as (lambda, M) with T_C = exp(lambda) * M:
 *   scalar: lambda = sum log alpha_t, M == 1 (not stored);
 *   diag  : lambda_i = sum log alpha_{t,i}, M == I (not stored);
 *   dense : M = prod (I - beta_t k_t k_t^T) scaled to max|M| = 1,
 *           lambda = sum log alpha_t + log(scale).  If M is exactly zero it is
 *           left at zero and lambda keeps sum log alpha_t.
 *   kda   : the per-channel gates do not factor out, so M = prod T_t itself,
 *           scaled to max|M| = 1, and lambda = log(scale) only.
 * Everything here is token by token, one (layer, segment, head) at a time,
 * in the order the recurrence states it.  No blocking, no chunking.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_SCALAR = 0, OR_DIAG = 1, OR_DENSE = 2, OR_KDA = 3 };
/* families whose operator is exp(lambda) * M with a matrix M */
#define HAS_M(fam) ((fam) == OR_DENSE || (fam) == OR_KDA)

/* Scale M by an exact power of two whenever its largest entry leaves
 * [2^-256, 2^256]; the factor goes into *lam.  Exact in binary floating point,
 * so it changes no digit of exp(lam) * M. */
static void keep_in_range(double *M, int n, double *lam)
{
    double mx = 0.0;
    for (int i = 0; i < n; ++i) {
        double a = fabs(M[i]);
        if (a > mx) mx = a;
    }
    if (mx == 0.0) return;
    if (mx < 0x1p-256 || mx > 0x1p256) {
        int e;
        frexp(mx, &e);
        for (int i = 0; i < n; ++i) M[i] = ldexp(M[i], -e);
        *lam += (double)e * log(2.0);
    }
}

/* Final normalisation: max|M| = 1, factor moved into lambda. */
static void normalise_maxabs(double *M, int n, double *lam)
{
    double mx = 0.0;
    for (int i = 0; i < n; ++i) {
        double a = fabs(M[i]);
        if (a > mx) mx = a;
    }
    if (mx == 0.0) return;
    for (int i = 0; i < n; ++i) M[i] /= mx;
    *lam += log(mx);
}

/*
 * Segment scan.  Layouts (row-major, innermost last):
 *   q, k  [n_layers, N, H, dk]    v [n_layers, N, H, dv]
 *   alpha [n_layers, N, H] (scalar, dense) or [n_layers, N, H, dk] (diag, kda)
 *   beta  [n_layers, N, H] or NULL (=> 1)
 *   seg_offsets [n_seg + 1], ascending, seg_offsets[0] = 0, last = N
 *   lam_out [n_layers, n_seg, H] or [n_layers, n_seg, H, dk] (diag)
 *   M_out   [n_layers, n_seg, H, dk, dk] (dense, kda; may be NULL)
 *   S_out   [n_layers, n_seg, H, dk, dv]
 *   o_out   [n_layers, N, H, dv] or NULL; needs q.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_segment_scan(int fam, int n_layers, int n_seg, int64_t N, int H,
                        int dk, int dv, const int64_t *seg_offsets,
                        const double *q, const double *k, const double *v,
                        const double *alpha, const double *beta,
                        double *lam_out, double *M_out, double *S_out,
                        double *o_out, int n_threads)
{
    if (fam < 0 || fam > 3 || n_layers < 0 || n_seg < 0 || N < 0 || H <= 0 ||
        dk <= 0 || dv <= 0 || !seg_offsets || !k || !v || !alpha || !lam_out ||
        !S_out || (o_out && !q))
        return -1;
    if (seg_offsets[0] != 0 || seg_offsets[n_seg] != N) return -1;
    for (int s = 0; s < n_seg; ++s)
        if (seg_offsets[s + 1] < seg_offsets[s]) return -1;

    const int64_t units = (int64_t)n_layers * n_seg * H;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        const int h = (int)(u % H);
        const int seg = (int)((u / H) % n_seg);
        const int l = (int)(u / ((int64_t)H * n_seg));
        double *S = calloc((size_t)dk * dv, sizeof(double));
        const int has_M = fam == OR_DENSE || fam == OR_KDA;
        double *M = has_M ? calloc((size_t)dk * dk, sizeof(double)) : NULL;
        double *kS = malloc(sizeof(double) * (size_t)(dv > dk ? dv : dk));
        double *lam = calloc((size_t)dk, sizeof(double));
        if (has_M)
            for (int i = 0; i < dk; ++i) M[(size_t)i * dk + i] = 1.0;

        for (int64_t t = seg_offsets[seg]; t < seg_offsets[seg + 1]; ++t) {
            const int64_t row = ((int64_t)l * N + t) * H + h;   /* token-head row */
            const double *kt = k + row * dk;
            const double *vt = v + row * dv;
            const double b = beta ? beta[row] : 1.0;
            if (fam == OR_SCALAR) {
                const double a = alpha[row];
                /* S <- a S + b k v^T */
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)i * dv + j] = a * S[(size_t)i * dv + j] + b * kt[i] * vt[j];
                lam[0] += log(a);
            } else if (fam == OR_DIAG) {
                const double *at = alpha + row * dk;
                /* S <- diag(a) S + b k v^T */
                for (int i = 0; i < dk; ++i) {
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)i * dv + j] = at[i] * S[(size_t)i * dv + j] + b * kt[i] * vt[j];
                    lam[i] += log(at[i]);
                }
            } else if (fam == OR_DENSE) {
                const double a = alpha[row];
                /* S <- a (S - b k (k^T S)) + b k v^T */
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i) acc += kt[i] * S[(size_t)i * dv + j];
                    kS[j] = acc;
                }
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)i * dv + j] =
                            a * (S[(size_t)i * dv + j] - b * kt[i] * kS[j]) + b * kt[i] * vt[j];
                /* T <- a (I - b k k^T) T, kept as exp(lam) * M */
                for (int j = 0; j < dk; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i) acc += kt[i] * M[(size_t)i * dk + j];
                    kS[j] = acc;
                }
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dk; ++j)
                        M[(size_t)i * dk + j] -= b * kt[i] * kS[j];
                lam[0] += log(a);
                keep_in_range(M, dk * dk, &lam[0]);
            } else {
                const double *at = alpha + row * dk;
                /* S <- diag(a) (S - b k (k^T S)) + b k v^T */
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i) acc += kt[i] * S[(size_t)i * dv + j];
                    kS[j] = acc;
                }
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)i * dv + j] =
                            at[i] * (S[(size_t)i * dv + j] - b * kt[i] * kS[j]) + b * kt[i] * vt[j];
                /* T <- diag(a) (I - b k k^T) T: the gates stay inside M */
                for (int j = 0; j < dk; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i) acc += kt[i] * M[(size_t)i * dk + j];
                    kS[j] = acc;
                }
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dk; ++j)
                        M[(size_t)i * dk + j] = at[i] * (M[(size_t)i * dk + j] - b * kt[i] * kS[j]);
                keep_in_range(M, dk * dk, &lam[0]);
            }
            if (o_out) {
                /* o_t = S_t^T q_t */
                const double *qt = q + row * dk;
                double *ot = o_out + row * dv;
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * qt[i];
                    ot[j] = acc;
                }
            }
        }
        const int64_t unit = ((int64_t)l * n_seg + seg) * H + h;
        memcpy(S_out + unit * dk * dv, S, sizeof(double) * (size_t)dk * dv);
        if (fam == OR_DIAG) {
            memcpy(lam_out + unit * dk, lam, sizeof(double) * (size_t)dk);
        } else if (fam == OR_SCALAR) {
            lam_out[unit] = lam[0];
        } else {
            normalise_maxabs(M, dk * dk, &lam[0]);
            lam_out[unit] = lam[0];
            if (M_out) memcpy(M_out + unit * dk * dk, M, sizeof(double) * (size_t)dk * dk);
        }
        free(S);
        free(M);
        free(kS);
        free(lam);
    }
    return 0;
}

/*
 * One composition step for one head, literally S = T(C2) S(C1) + S(C2) with
 * T(C2) = exp(lam) M:
 *   scalar: S = exp(lam) S_prev + S_C
 *   diag  : S[i,:] = exp(lam_i) S_prev[i,:] + S_C[i,:]
 *   dense : S = exp(lam) (M S_prev) + S_C
 */
static void compose_one(int fam, int dk, int dv, const double *lam, const double *M,
                        const double *S_prev, const double *S_C, double *S_out)
{
    double *tmp = malloc(sizeof(double) * (size_t)dk * dv);
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) {
            double acc;
            if (!S_prev) {
                acc = 0.0;
            } else if (fam == OR_SCALAR) {
                acc = exp(lam[0]) * S_prev[(size_t)i * dv + j];
            } else if (fam == OR_DIAG) {
                acc = exp(lam[i]) * S_prev[(size_t)i * dv + j];
            } else {
                double mm = 0.0;
                for (int r = 0; r < dk; ++r) mm += M[(size_t)i * dk + r] * S_prev[(size_t)r * dv + j];
                acc = exp(lam[0]) * mm;
            }
            tmp[(size_t)i * dv + j] = acc + S_C[(size_t)i * dv + j];
        }
    memcpy(S_out, tmp, sizeof(double) * (size_t)dk * dv);
    free(tmp);
}

/*
 * Batched composition over n items x H heads:
 *   lam [n,H] or [n,H,dk] (diag);  M [n,H,dk,dk] (dense, kda);
 *   S_prev [n,H,dk,dv] or NULL (=> 0);  S_C, S_out [n,H,dk,dv].
 * Optional operator composition T(C1.C2) = T(C2) T(C1):
 *   lam_out = lam + lam_prev;  dense, kda: M_out = M M_prev, max-abs normalised.
 * lam_prev/lam_out (and M_prev/M_out for dense, kda) are both given or both NULL.
 */
int oracle_compose(int fam, int n, int H, int dk, int dv, const double *lam,
                   const double *M, const double *S_prev, const double *S_C,
                   double *S_out, const double *lam_prev, const double *M_prev,
                   double *lam_out, double *M_out)
{
    if (fam < 0 || fam > 3 || n < 0 || H <= 0 || dk <= 0 || dv <= 0 || !lam ||
        !S_C || !S_out || (HAS_M(fam) && !M) || (!lam_prev) != (!lam_out))
        return -1;
    if (HAS_M(fam) && lam_out && ((!M_prev) || (!M_out))) return -1;
    const int nl = fam == OR_DIAG ? dk : 1;
    for (int64_t u = 0; u < (int64_t)n * H; ++u) {
        const double *Mu = HAS_M(fam) ? M + u * dk * dk : NULL;
        compose_one(fam, dk, dv, lam + u * nl, Mu, S_prev ? S_prev + u * dk * dv : NULL,
                    S_C + u * dk * dv, S_out + u * dk * dv);
        if (lam_out) {
            for (int i = 0; i < nl; ++i) lam_out[u * nl + i] = lam[u * nl + i] + lam_prev[u * nl + i];
            if (HAS_M(fam)) {
                const double *Mp = M_prev + u * dk * dk;
                double *P = malloc(sizeof(double) * (size_t)dk * dk);
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dk; ++j) {
                        double acc = 0.0;
                        for (int r = 0; r < dk; ++r) acc += Mu[(size_t)i * dk + r] * Mp[(size_t)r * dk + j];
                        P[(size_t)i * dk + j] = acc;
                    }
                normalise_maxabs(P, dk * dk, &lam_out[u]);
                memcpy(M_out + u * dk * dk, P, sizeof(double) * (size_t)dk * dk);
                free(P);
            }
        }
    }
    return 0;
}

/*
 * Chained composition ([remio-ja] "cold requests become parallel": the
 * combine step folds every segment's cached pair into the request's running
 * state; [xix-fr]: reuse under any prefix).  For each request r, layer l and
 * head h, starting from S_init (or 0):
 *   for j = 0 .. chain_len[r]-1:  p = seg_idx[r, j];  S = T_p S + S_p.
 * Layouts: seg_idx [R, max_chain]; pool_lam [P, Lyr, H] or [P, Lyr, H, dk];
 * pool_M [P, Lyr, H, dk, dk] (dense, kda); pool_S [P, Lyr, H, dk, dv];
 * S_init, S_out [R, Lyr, H, dk, dv].  Returns -2 on an index out of range.
 */
int oracle_compose_chain(int fam, int R, int Lyr, int H, int dk, int dv, int max_chain,
                         const int32_t *chain_len, const int32_t *seg_idx, int P,
                         const double *pool_lam, const double *pool_M,
                         const double *pool_S, const double *S_init, double *S_out,
                         int n_threads)
{
    if (fam < 0 || fam > 3 || R < 0 || Lyr < 0 || H <= 0 || dk <= 0 || dv <= 0 ||
        max_chain < 0 || !chain_len || (max_chain > 0 && !seg_idx) || P < 0 ||
        !pool_lam || !pool_S || (HAS_M(fam) && !pool_M) || !S_out)
        return -1;
    for (int r = 0; r < R; ++r) {
        if (chain_len[r] < 0 || chain_len[r] > max_chain) return -1;
        for (int j = 0; j < chain_len[r]; ++j)
            if (seg_idx[(int64_t)r * max_chain + j] < 0 || seg_idx[(int64_t)r * max_chain + j] >= P)
                return -2;
    }
    const int nl = fam == OR_DIAG ? dk : 1;
    const int64_t units = (int64_t)R * Lyr * H;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        const int64_t r = u / ((int64_t)Lyr * H);
        const int64_t lh = u % ((int64_t)Lyr * H);     /* layer * H + head */
        double *S = S_out + u * dk * dv;
        if (S_init)
            memcpy(S, S_init + u * dk * dv, sizeof(double) * (size_t)dk * dv);
        else
            memset(S, 0, sizeof(double) * (size_t)dk * dv);
        for (int j = 0; j < chain_len[r]; ++j) {
            const int64_t p = seg_idx[r * max_chain + j];
            const int64_t e = p * Lyr * H + lh;       /* pool entry for this layer, head */
            compose_one(fam, dk, dv, pool_lam + e * nl,
                        HAS_M(fam) ? pool_M + e * dk * dk : NULL, S,
                        pool_S + e * dk * dv, S);
        }
    }
    return 0;
}

/*
 * Composed prefix ([xix-fr]: T(C1.C2) = T(C2) T(C1) makes compositions
 * chainable, so a popular ordered group of cached segments can itself be
 * cached as one pair).  For each request r, layer l and head h, the pair of
 * the concatenation of pool entries seg_idx[r, 0 .. chain_len[r]-1]:
 *   T = T_{p_n} ... T_{p_1}   (lambda summed; dense / kda: M product, max-abs normalised)
 *   S = S(C_{p_1} ... C_{p_n} | 0)   (the chain from a zero state)
 * Layouts as oracle_compose_chain; lam_out [R, Lyr, H] or [R, Lyr, H, dk] (diag),
 * M_out [R, Lyr, H, dk, dk] (dense, kda), S_out [R, Lyr, H, dk, dv].
 */
int oracle_compose_prefix(int fam, int R, int Lyr, int H, int dk, int dv, int max_chain,
                          const int32_t *chain_len, const int32_t *seg_idx, int P,
                          const double *pool_lam, const double *pool_M,
                          const double *pool_S, double *lam_out, double *M_out,
                          double *S_out)
{
    if (!lam_out || (HAS_M(fam) && !M_out)) return -1;
    const int rc = oracle_compose_chain(fam, R, Lyr, H, dk, dv, max_chain, chain_len, seg_idx, P,
                                        pool_lam, pool_M, pool_S, NULL, S_out, 0);
    if (rc != 0) return rc;
    const int nl = fam == OR_DIAG ? dk : 1;
    double *P2 = malloc(sizeof(double) * (size_t)dk * dk);
    for (int64_t u = 0; u < (int64_t)R * Lyr * H; ++u) {
        const int64_t r = u / ((int64_t)Lyr * H);
        const int64_t lh = u % ((int64_t)Lyr * H);
        double *lam = lam_out + u * nl;
        for (int i = 0; i < nl; ++i) lam[i] = 0.0;
        double *Mo = HAS_M(fam) ? M_out + u * dk * dk : NULL;
        if (Mo) {
            memset(Mo, 0, sizeof(double) * (size_t)dk * dk);
            for (int i = 0; i < dk; ++i) Mo[(size_t)i * dk + i] = 1.0;
        }
        for (int j = 0; j < chain_len[r]; ++j) {
            const int64_t e = (int64_t)seg_idx[r * max_chain + j] * Lyr * H + lh;
            for (int i = 0; i < nl; ++i) lam[i] += pool_lam[e * nl + i];
            if (Mo) {   /* M <- M_p M */
                const double *Mp = pool_M + e * dk * dk;
                for (int i = 0; i < dk; ++i)
                    for (int c = 0; c < dk; ++c) {
                        double acc = 0.0;
                        for (int x = 0; x < dk; ++x) acc += Mp[(size_t)i * dk + x] * Mo[(size_t)x * dk + c];
                        P2[(size_t)i * dk + c] = acc;
                    }
                memcpy(Mo, P2, sizeof(double) * (size_t)dk * dk);
                keep_in_range(Mo, dk * dk, &lam[0]);
            }
        }
        if (Mo) normalise_maxabs(Mo, dk * dk, &lam[0]);
    }
    free(P2);
    return 0;
}

/*
 * Seam-window advance with composition ([xix-fr], paragraph on full-attention
 * layers, "fenetres de jonction"): the first w tokens of every reused segment
 * are left out of its cache and recomputed at reuse under the full prefix; the
 * linear layers advance the running state through them, hand each seam
 * token's output to the layer above, and the rest of the segment enters by
 * its cached pair.  Per item i and head h, token by token in fp64:
 *   S = S_prev (or 0);
 *   for t = 0 .. w-1:  S = T_t S + beta_t k_t v_t^T;  o_t = S^T q_t;
 *   S_out = T_body S + S_body      (T_body = exp(lam) M, as in compose_one).
 * Layouts: q, k [n, w, H, dk], v [n, w, H, dv], alpha [n, w, H] or
 * [n, w, H, dk] (diag, kda), beta [n, w, H] or NULL (=> 1); lam [n, H] or
 * [n, H, dk] (diag); M [n, H, dk, dk] (dense, kda); S_prev (or NULL), S_C,
 * S_out [n, H, dk, dv];
 * o_out [n, w, H, dv] or NULL.
 */
int oracle_seam_compose(int fam, int n, int w, int H, int dk, int dv,
                        const double *q, const double *k, const double *v,
                        const double *alpha, const double *beta,
                        const double *lam, const double *M, const double *S_prev,
                        const double *S_C, double *S_out, double *o_out)
{
    if (fam < 0 || fam > 3 || n < 0 || w < 0 || H <= 0 || dk <= 0 || dv <= 0 ||
        (w > 0 && (!k || !v || !alpha)) || (o_out && w > 0 && !q) || !lam || !S_C ||
        !S_out || (HAS_M(fam) && !M))
        return -1;
    const int nl = fam == OR_DIAG ? dk : 1;
    double *S = malloc(sizeof(double) * (size_t)dk * dv);
    double *kS = malloc(sizeof(double) * (size_t)dv);
    for (int64_t u = 0; u < (int64_t)n * H; ++u) {
        const int64_t i = u / H, h = u % H;
        if (S_prev)
            memcpy(S, S_prev + u * dk * dv, sizeof(double) * (size_t)dk * dv);
        else
            memset(S, 0, sizeof(double) * (size_t)dk * dv);
        for (int t = 0; t < w; ++t) {
            const int64_t row = (i * w + t) * H + h;   /* seam token-head row */
            const double *kt = k + row * dk;
            const double *vt = v + row * dv;
            const double b = beta ? beta[row] : 1.0;
            if (fam == OR_SCALAR) {
                const double a = alpha[row];
                for (int r = 0; r < dk; ++r)
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)r * dv + j] = a * S[(size_t)r * dv + j] + b * kt[r] * vt[j];
            } else if (fam == OR_DIAG) {
                const double *at = alpha + row * dk;
                for (int r = 0; r < dk; ++r)
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)r * dv + j] = at[r] * S[(size_t)r * dv + j] + b * kt[r] * vt[j];
            } else {
                /* gated delta rule (one gate) or KDA (a gate per channel) */
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int r = 0; r < dk; ++r) acc += kt[r] * S[(size_t)r * dv + j];
                    kS[j] = acc;
                }
                for (int r = 0; r < dk; ++r) {
                    const double a = fam == OR_KDA ? alpha[row * dk + r] : alpha[row];
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)r * dv + j] =
                            a * (S[(size_t)r * dv + j] - b * kt[r] * kS[j]) + b * kt[r] * vt[j];
                }
            }
            if (o_out) {
                const double *qt = q + row * dk;
                double *ot = o_out + row * dv;
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int r = 0; r < dk; ++r) acc += S[(size_t)r * dv + j] * qt[r];
                    ot[j] = acc;
                }
            }
        }
        compose_one(fam, dk, dv, lam + u * nl, HAS_M(fam) ? M + u * dk * dk : NULL, S,
                    S_C + u * dk * dv, S_out + u * dk * dv);
    }
    free(S);
    free(kS);
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
