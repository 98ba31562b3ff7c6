/*
 * attn_fp64.c -- plain fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path (the CUDA library,
 * its Python binding) may call, link or load this file.  Only the tests, the
 * package's smoke check and the benchmark's CPU-baseline leg use it.
 *
 * It is the *definition* of attention, written out with no tiling, no online
 * softmax and no recomputation trick, so that a reader can check it by eye:
 *
 *   "FlashAttention" (notes.yuuk.io wiki), section 定義 (Definition): the
 *   method is exact attention, not an approximation; the N x N score matrix is
 *   what a standard implementation materialises.  "FlashAttention：GPU
 *   ハードウェア階層を考慮した高速・省メモリな厳密アテンション"
 *   (singularity-lens.com), paragraph on the online softmax: the tiled result
 *   is identical to standard attention.  So the oracle is standard attention:
 *
 *     S_ij = scale * <q_i, k_g(j)>        (g = h / (H/Hkv), grouped heads)
 *     S_ij = -inf  if causal and j > pos(i)
 *     P_ij = exp(S_ij - m_i) / sum_j' exp(S_ij' - m_i),   m_i = max_j S_ij
 *     O_i  = sum_j P_ij v_j
 *     LSE_i = m_i + log sum_j exp(S_ij - m_i)       (natural log)
 *
 * The backward pass is the textbook gradient of the scalar L = sum(O * dO)
 * (the pages print no backward equations; the same wiki's 定義 item (2)
 * and the explainer's recomputation paragraph only say that P is recomputed):
 *
 *     dV_j  = sum_i P_ij dO_i
 *     dP_ij = <dO_i, v_j>
 *     D_i   = sum_j P_ij dP_ij
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale * sum_j dS_ij k_j
 *     dK_j  = scale * sum_i dS_ij q_i
 *   with dK/dV of a shared (grouped) K/V head summed over its query heads.
 *
 * Layouts (all fp64, row-major, contiguous):
 *   q, o, dout, dq : [B][H][Nq][d]      k, v, dk, dv : [B][Hkv][Nk][d]
 *   lse            : [B][H][Nq]
 * Causal masking: query row i sits at position pos(i) and sees keys 0..pos(i).
 * With Nq = Nk, pos(i) = i.  With Nq != Nk the plain reading for a block of
 * queries that follows earlier keys (a KV cache) is bottom-right alignment,
 * pos(i) = i + (Nk - Nq): the last query sees every key.  A row whose pos is
 * negative sees no key; its O is 0 and its LSE -inf (no gradient flows).
 *
 * Return value: 0 on success, -1 on an invalid argument, -2 on out-of-memory.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int check_args(int B, int H, int Hkv, int Nq, int Nk, int d)
{
    if (B < 0 || H < 1 || Hkv < 1 || Nq < 0 || Nk < 0 || d < 1) return -1;
    if (H % Hkv != 0) return -1;
    return 0;
}

static double dot(const double* a, const double* b, int d)
{
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

/* Number of OpenMP threads the oracle would use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Forward.  qpos (may be NULL) gives the absolute position of each of the Nq
 * query rows, for the causal mask only; NULL means positions 0..Nq-1.  This
 * lets a caller evaluate a subset of rows of a long sequence exactly. */
int oracle_attn_fwd(const double* q, const double* k, const double* v,
                    double* o, double* lse,
                    int B, int H, int Hkv, int Nq, int Nk, int d,
                    int causal, double scale, const long long* qpos)
{
    if (check_args(B, H, Hkv, Nq, Nk, d)) return -1;
    const int group = H / Hkv;
    const long long rows = (long long)B * H * Nq;
    int oom = 0;

#pragma omp parallel
    {
        double* srow = (double*)malloc(sizeof(double) * (Nk > 0 ? Nk : 1));
        if (!srow) {
#pragma omp atomic write
            oom = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long long r = 0; r < rows; ++r) {
            if (!srow) continue;
            const long long bh = r / Nq;          /* b*H + h */
            const int i = (int)(r % Nq);
            const int b = (int)(bh / H), h = (int)(bh % H);
            const int g = h / group;
            const double* qi = q + r * d;
            const double* K = k + ((long long)b * Hkv + g) * Nk * d;
            const double* V = v + ((long long)b * Hkv + g) * Nk * d;
            double* oi = o + r * d;
            const long long pos = qpos ? qpos[i] : i;

            /* the full score row S_i. (materialised) and its max */
            double m = -INFINITY;
            for (int j = 0; j < Nk; ++j) {
                double s = (causal && j > pos) ? -INFINITY : scale * dot(qi, K + (long long)j * d, d);
                srow[j] = s;
                if (s > m) m = s;
            }
            for (int c = 0; c < d; ++c) oi[c] = 0.0;
            if (m == -INFINITY) {             /* no visible key: O = 0, LSE = -inf */
                lse[r] = -INFINITY;
                continue;
            }
            double l = 0.0;
            for (int j = 0; j < Nk; ++j) {
                srow[j] = exp(srow[j] - m);   /* unnormalised probabilities */
                l += srow[j];
            }
            for (int j = 0; j < Nk; ++j) {
                const double p = srow[j] / l; /* P_ij */
                if (p == 0.0) continue;
                const double* vj = V + (long long)j * d;
                for (int c = 0; c < d; ++c) oi[c] += p * vj[c];
            }
            lse[r] = m + log(l);
        }
        free(srow);
    }
    return oom ? -2 : 0;
}

/* Backward.  Query row i sits at position i + qoff (see the causal note in the
 * header), keys at 0..Nk-1.  Two plain passes, both straight from the formulas
 * in the header:
 *  pass 1 (one query row at a time): P_i., dP_i., D_i, dS_i., dQ_i, and LSE_i;
 *  pass 2 (one key row j of a K/V head at a time): the column sums
 *         dV_j = sum_{h in group, i} P_ij dO_i and dK_j = scale sum dS_ij q_i,
 *         with P_ij = exp(S_ij - LSE_i) (the softmax written with its
 *         normaliser) and dS_ij formed exactly as in pass 1. */
int oracle_attn_bwd_off(const double* q, const double* k, const double* v,
                        const double* dout, double* dq, double* dk, double* dv,
                        int B, int H, int Hkv, int Nq, int Nk, int d,
                        int causal, double scale, long long qoff)
{
    if (check_args(B, H, Hkv, Nq, Nk, d)) return -1;
    const int group = H / Hkv;
    const long long rows = (long long)B * H * Nq;
    double* lse = (double*)malloc(sizeof(double) * (rows > 0 ? rows : 1));
    double* Dv = (double*)malloc(sizeof(double) * (rows > 0 ? rows : 1));
    if (!lse || !Dv) { free(lse); free(Dv); return -2; }
    int oom = 0;

#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (Nk > 0 ? Nk : 1));
        double* dp = (double*)malloc(sizeof(double) * (Nk > 0 ? Nk : 1));
        if (!p || !dp) {
#pragma omp atomic write
            oom = 1;
        }
        /* pass 1: per query row */
#pragma omp for schedule(dynamic, 16)
        for (long long r = 0; r < rows; ++r) {
            if (!p || !dp) continue;
            const long long bh = r / Nq;
            const int i = (int)(r % Nq);
            const int b = (int)(bh / H), h = (int)(bh % H);
            const int g = h / group;
            const double* qi = q + r * d;
            const double* doi = dout + r * d;
            const double* K = k + ((long long)b * Hkv + g) * Nk * d;
            const double* V = v + ((long long)b * Hkv + g) * Nk * d;
            double* dqi = dq + r * d;
            for (int c = 0; c < d; ++c) dqi[c] = 0.0;

            double m = -INFINITY;
            for (int j = 0; j < Nk; ++j) {
                double s = (causal && j > i + qoff) ? -INFINITY : scale * dot(qi, K + (long long)j * d, d);
                p[j] = s;
                if (s > m) m = s;
            }
            if (m == -INFINITY) { lse[r] = -INFINITY; Dv[r] = 0.0; continue; }
            double l = 0.0;
            for (int j = 0; j < Nk; ++j) { p[j] = exp(p[j] - m); l += p[j]; }
            for (int j = 0; j < Nk; ++j) p[j] /= l;              /* P_ij */
            double D = 0.0;
            for (int j = 0; j < Nk; ++j) {
                dp[j] = dot(doi, V + (long long)j * d, d);       /* dP_ij */
                D += p[j] * dp[j];
            }
            for (int j = 0; j < Nk; ++j) {
                const double ds = p[j] * (dp[j] - D);           /* dS_ij */
                if (ds == 0.0) continue;
                const double* kj = K + (long long)j * d;
                for (int c = 0; c < d; ++c) dqi[c] += scale * ds * kj[c];
            }
            lse[r] = m + log(l);
            Dv[r] = D;
        }
        /* implicit barrier: lse and D are complete */

        /* pass 2: per key row of each K/V head */
        const long long krows = (long long)B * Hkv * Nk;
#pragma omp for schedule(dynamic, 16)
        for (long long r = 0; r < krows; ++r) {
            const long long bg = r / Nk;
            const int j = (int)(r % Nk);
            const int b = (int)(bg / Hkv), g = (int)(bg % Hkv);
            const double* kj = k + r * d;
            const double* vj = v + r * d;
            double* dkj = dk + r * d;
            double* dvj = dv + r * d;
            for (int c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
            for (int hh = 0; hh < group; ++hh) {
                const int h = g * group + hh;
                const long long base = ((long long)b * H + h) * Nq;
                for (int i = 0; i < Nq; ++i) {
                    if (causal && j > i + qoff) continue;
                    const long long ri = base + i;
                    if (lse[ri] == -INFINITY) continue;
                    const double* qi = q + ri * d;
                    const double* doi = dout + ri * d;
                    const double pij = exp(scale * dot(qi, kj, d) - lse[ri]);
                    const double dpij = dot(doi, vj, d);
                    const double ds = pij * (dpij - Dv[ri]);
                    for (int c = 0; c < d; ++c) {
                        dvj[c] += pij * doi[c];
                        dkj[c] += scale * ds * qi[c];
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    free(lse);
    free(Dv);
    return oom ? -2 : 0;
}

/* Backward with the positions of the Nq = Nk case (qoff = 0). */
int oracle_attn_bwd(const double* q, const double* k, const double* v,
                    const double* dout, double* dq, double* dk, double* dv,
                    int B, int H, int Hkv, int Nq, int Nk, int d,
                    int causal, double scale)
{
    return oracle_attn_bwd_off(q, k, v, dout, dq, dk, dv, B, H, Hkv, Nq, Nk, d, causal, scale, 0);
}
