/*
 * band_oracle.c -- plain fp64 CPU oracle for sliding-window ("diagonal",
 * banded) attention, as used by Longformer.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark load this file.  It shares no code, header, table or
 * helper with the CUDA library, and the CUDA library never calls it.
 *
 * What it follows (page titles and the post / item on them):
 *  - "Developing a faster schedule for Longformer's kernel" (TVM forum)
 *      post 1: the kernel is a banded matrix product that evaluates only
 *              some diagonals of the output matrix;
 *      post 3: dilation is the number of skipped positions between two
 *              attended positions (key stride dilation+1);
 *      posts 5-6: the parameters b, n, h, w (window on one side), w_upper
 *              (window to the right: w, or 0 for the autoregressive case),
 *              padding (a constant stored where the key falls outside the
 *              sequence), t3d3 = 2w+1 diagonals in the forward product and
 *              the two backward products selected by transpose_t1.
 *  - "[WIP] Improve LongformerAttention performance" (ONNX Runtime issue),
 *      item (1): one global-token index of length S, shared by every
 *      sequence of the batch.
 *  - "HuggingFace BertForMaskedLM - Log Softmax Fusion with Autocast has bad
 *      perf" (nvFuser issue), fusion 1: scores divided by 8 = sqrt(64), then
 *      row max, exp(x - max), row sum and division, in fp32 (fp64 here).
 *
 * Conventions (the readings where the pages are silent):
 *  - s = dilation + 1;  D = w + w_upper + 1 band slots per query row;
 *    slot t in [0, D) holds key j = i + (t - w) * s  (slot w is the
 *    diagonal; slots ascend with the key position);
 *  - a slot is valid iff 0 <= j < n; invalid slots of a score tensor hold
 *    `padding`; every consumer ignores invalid slots whatever they hold;
 *  - global tokens G (sorted, unique, shared by all b*h slices): a row
 *    i not in G attends to its valid band keys that are not in G, plus all
 *    of G; a row i in G attends to every key.  Band slots whose key is in G
 *    are excluded for local rows (the key is counted once, through G).
 *  - tensors: dense [BH][n][hd]; band [BH][n][D]; global columns
 *    [BH][n][G] (value of row i at key G[g]); global rows [BH][G][n]
 *    (dense row of query G[g]); lse [BH][n].
 *
 * Every function returns 0 on success and a negative code on bad arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int check_geom(int BH, int n, int hd, int w, int wu, int dil) {
    if (BH < 0 || n < 0 || hd < 1 || w < 0 || wu < 0 || dil < 0) return -1;
    return 0;
}

/* Build a membership mask of the global index; -2 if an index is out of
 * range, repeated or out of order. */
static int build_gmask(int n, int G, const int *gidx, unsigned char **mask_out,
                       int **pos_out) {
    *mask_out = NULL;
    *pos_out = NULL;
    if (G < 0) return -2;
    unsigned char *mask = (unsigned char *)calloc((size_t)(n > 0 ? n : 1), 1);
    int *pos = (int *)malloc(sizeof(int) * (size_t)(n > 0 ? n : 1));
    if (!mask || !pos) { free(mask); free(pos); return -3; }
    for (int j = 0; j < n; ++j) pos[j] = -1;
    for (int g = 0; g < G; ++g) {
        int j = gidx[g];
        if (j < 0 || j >= n || (g > 0 && gidx[g - 1] >= j)) {
            free(mask); free(pos); return -2;
        }
        mask[j] = 1;
        pos[j] = g;
    }
    *mask_out = mask;
    *pos_out = pos;
    return 0;
}

static double dot(const double *a, const double *b, int hd) {
    double acc = 0.0;
    for (int c = 0; c < hd; ++c) acc += a[c] * b[c];
    return acc;
}

/* Slot t of row i is used by attention: its key is inside the sequence and,
 * when global tokens are present, the key is not global. */
static int slot_used(long long i, int t, int w, int s, int n,
                     const unsigned char *gmask) {
    long long j = i + (long long)(t - w) * s;
    if (j < 0 || j >= n) return 0;
    if (gmask && gmask[j]) return 0;
    return 1;
}

/* ---------------------------------------------------------------------
 * Banded product, forward mode (TVM forum, posts 5-6: dense x dense^T
 * restricted to t3d3 = w + w_upper + 1 diagonals):
 *   S[i,t] = alpha * sum_c A[i,c] * B[j,c],  j = i + (t-w)*s, if 0<=j<n
 *          = padding                          otherwise.
 * With G > 0 also the dense global pieces
 *   Sg[i,g] = alpha * A[i] . B[G[g]]   and   Sr[g,j] = alpha * A[G[g]] . B[j].
 * --------------------------------------------------------------------- */
int orc_band_qk(int BH, int n, int hd, int w, int wu, int dil, double alpha,
                double padding, const double *A, const double *B, double *S,
                int G, const int *gidx, double *Sg, double *Sr) {
    if (check_geom(BH, n, hd, w, wu, dil)) return -1;
    const int D = w + wu + 1, s = dil + 1;
    unsigned char *gm; int *gp;
    int rc = build_gmask(n, G, gidx, &gm, &gp);
    if (rc) return rc;
    free(gm); free(gp);
#pragma omp parallel for collapse(2) schedule(static)
    for (int bh = 0; bh < BH; ++bh) {
        for (int i = 0; i < n; ++i) {
            const double *a = A + ((size_t)bh * n + i) * hd;
            double *srow = S + ((size_t)bh * n + i) * D;
            for (int t = 0; t < D; ++t) {
                long long j = (long long)i + (long long)(t - w) * s;
                if (j < 0 || j >= n) {
                    srow[t] = padding;
                } else {
                    srow[t] = alpha * dot(a, B + ((size_t)bh * n + j) * hd, hd);
                }
            }
            for (int g = 0; g < G; ++g) {
                Sg[((size_t)bh * n + i) * G + g] =
                    alpha * dot(a, B + ((size_t)bh * n + gidx[g]) * hd, hd);
            }
        }
    }
    if (G > 0) {
#pragma omp parallel for collapse(2) schedule(static)
        for (int bh = 0; bh < BH; ++bh) {
            for (int g = 0; g < G; ++g) {
                const double *a = A + ((size_t)bh * n + gidx[g]) * hd;
                for (int j = 0; j < n; ++j)
                    Sr[((size_t)bh * G + g) * n + j] =
                        alpha * dot(a, B + ((size_t)bh * n + j) * hd, hd);
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------
 * Masked row softmax over the band (nvFuser issue, fusion 1: max, exp of the
 * difference, sum, divide), extended with the global columns / rows.
 *   local row i : m = max over used slots and Sg[i,:];  Z = sum exp(x - m)
 *                 P[i,t] = exp(S[i,t]-m)/Z on used slots, 0 elsewhere
 *                 Pg[i,g] = exp(Sg[i,g]-m)/Z
 *   global row i = G[g] : softmax of the dense row Sr[g,:] -> Pr[g,:];
 *                 P[i,:] = 0, Pg[i,:] = 0
 *   lse[i] = m + log Z.
 * With a key bias, kbias[bh, j] is added to every score of key j first: the
 * band slots, the global columns (j = G[g]) and the dense global rows.
 * --------------------------------------------------------------------- */
static double drop_factor(uint64_t seed, int drop_t, int bh, int i, int j, int s);

int orc_band_softmax(int BH, int n, int w, int wu, int dil, const double *S,
                     double *P, double *lse, int G, const int *gidx,
                     const double *Sg, const double *Sr, double *Pg, double *Pr,
                     const double *kbias, uint64_t seed, int drop_t, double *Pd) {
    if (check_geom(BH, n, 1, w, wu, dil)) return -1;
    if (drop_t < 0 || drop_t > 255 || (drop_t > 0 && (G > 0 || !Pd))) return -4;
    const int D = w + wu + 1, s = dil + 1;
    unsigned char *gm; int *gp;
    int rc = build_gmask(n, G, gidx, &gm, &gp);
    if (rc) return rc;
    const unsigned char *gmask = G > 0 ? gm : NULL;
#pragma omp parallel
    {
    /* the row's scores plus the key bias of each slot's key (nvFuser issue,
     * fusion 1: the additive mask term is added to the scaled score) */
    double *xb = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for collapse(2) schedule(static)
    for (int bh = 0; bh < BH; ++bh) {
        for (int i = 0; i < n; ++i) {
            const double *srow0 = S + ((size_t)bh * n + i) * D;
            for (int t = 0; t < D; ++t) {
                const long long j = (long long)i + (long long)(t - w) * s;
                xb[t] = srow0[t] + ((kbias && j >= 0 && j < n) ? kbias[(size_t)bh * n + j] : 0.0);
            }
            const double *srow = xb;
            double *prow = P + ((size_t)bh * n + i) * D;
            if (gmask && gmask[i]) {
                /* the dense row, plus the key bias of every key */
                const int g = gp[i];
                const double *x0 = Sr + ((size_t)bh * G + g) * n;
                double *p = Pr + ((size_t)bh * G + g) * n;
#define XR(j) (x0[j] + (kbias ? kbias[(size_t)bh * n + (j)] : 0.0))
                double m = -INFINITY, z = 0.0;
                for (int j = 0; j < n; ++j) m = fmax(m, XR(j));
                for (int j = 0; j < n; ++j) z += exp(XR(j) - m);
                for (int j = 0; j < n; ++j) p[j] = exp(XR(j) - m) / z;
#undef XR
                for (int t = 0; t < D; ++t) prow[t] = 0.0;
                for (int q = 0; q < G; ++q) Pg[((size_t)bh * n + i) * G + q] = 0.0;
                if (lse) lse[(size_t)bh * n + i] = m + log(z);
                continue;
            }
            /* the global columns, plus the key bias of each global key */
#define XG(q) (Sg[((size_t)bh * n + i) * G + (q)] + (kbias ? kbias[(size_t)bh * n + gidx[q]] : 0.0))
            double m = -INFINITY, z = 0.0;
            for (int t = 0; t < D; ++t)
                if (slot_used(i, t, w, s, n, gmask)) m = fmax(m, srow[t]);
            for (int q = 0; q < G; ++q) m = fmax(m, XG(q));
            for (int t = 0; t < D; ++t)
                if (slot_used(i, t, w, s, n, gmask)) z += exp(srow[t] - m);
            for (int q = 0; q < G; ++q) z += exp(XG(q) - m);
            for (int t = 0; t < D; ++t)
                prow[t] = slot_used(i, t, w, s, n, gmask) ? exp(srow[t] - m) / z : 0.0;
            /* dropped probabilities: the keep-and-scale factor of the slot's key */
            if (Pd) {
                double *drow = Pd + ((size_t)bh * n + i) * D;
                for (int t = 0; t < D; ++t)
                    drow[t] = slot_used(i, t, w, s, n, gmask)
                                  ? drop_factor(seed, drop_t, bh, i, i + (t - w) * s, s) * prow[t]
                                  : 0.0;
            }
            for (int q = 0; q < G; ++q) Pg[((size_t)bh * n + i) * G + q] = exp(XG(q) - m) / z;
#undef XG
            if (lse) lse[(size_t)bh * n + i] = m + log(z);
        }
    }
    free(xb);
    }
    free(gm); free(gp);
    return 0;
}

/* ---------------------------------------------------------------------
 * Band x dense product (TVM forum, post 6: transpose_t1 = 0, t1d3 = 2w+1):
 *   O[i,c] = alpha * sum over used slots t of P[i,t] * V[j(i,t), c]
 *          (+ alpha * sum_g Pg[i,g] * V[G[g], c] for local rows)
 *   global row i = G[g]: O[i,c] = alpha * sum_j Pr[g,j] * V[j,c].
 * Forward: P.V (alpha = 1).  Backward: dQ = alpha * dS.K.
 * --------------------------------------------------------------------- */
int orc_band_pv(int BH, int n, int hd, int w, int wu, int dil, double alpha,
                const double *P, const double *V, double *O, int G,
                const int *gidx, const double *Pg, const double *Pr) {
    if (check_geom(BH, n, hd, w, wu, dil)) return -1;
    const int D = w + wu + 1, s = dil + 1;
    unsigned char *gm; int *gp;
    int rc = build_gmask(n, G, gidx, &gm, &gp);
    if (rc) return rc;
    const unsigned char *gmask = G > 0 ? gm : NULL;
#pragma omp parallel for collapse(2) schedule(static)
    for (int bh = 0; bh < BH; ++bh) {
        for (int i = 0; i < n; ++i) {
            double *o = O + ((size_t)bh * n + i) * hd;
            for (int c = 0; c < hd; ++c) o[c] = 0.0;
            if (gmask && gmask[i]) {
                const double *p = Pr + ((size_t)bh * G + gp[i]) * n;
                for (int j = 0; j < n; ++j) {
                    const double *v = V + ((size_t)bh * n + j) * hd;
                    for (int c = 0; c < hd; ++c) o[c] += p[j] * v[c];
                }
            } else {
                const double *p = P + ((size_t)bh * n + i) * D;
                for (int t = 0; t < D; ++t) {
                    if (!slot_used(i, t, w, s, n, gmask)) continue;
                    long long j = (long long)i + (long long)(t - w) * s;
                    const double *v = V + ((size_t)bh * n + j) * hd;
                    for (int c = 0; c < hd; ++c) o[c] += p[t] * v[c];
                }
                for (int q = 0; q < G; ++q) {
                    const double pg = Pg[((size_t)bh * n + i) * G + q];
                    const double *v = V + ((size_t)bh * n + gidx[q]) * hd;
                    for (int c = 0; c < hd; ++c) o[c] += pg * v[c];
                }
            }
            for (int c = 0; c < hd; ++c) o[c] *= alpha;
        }
    }
    free(gm); free(gp);
    return 0;
}

/* ---------------------------------------------------------------------
 * Transposed band x dense product (TVM forum, post 6: transpose_t1 = 1),
 * written as a SCATTER over (query row, used slot) so that it shares no
 * indexing with the gather form a GPU kernel uses:
 *   for every local row i and used slot t:  X[j(i,t)] += alpha*Bd[i,t]*Y[i]
 *   for every local row i and g:            X[G[g]]   += alpha*Bg[i,g]*Y[i]
 *   for every global row i = G[g], all j:   X[j]      += alpha*Br[g,j]*Y[i]
 * Backward: dK = alpha * dS^T.Q, dV = P^T.dO.
 * Parallel over (slice, channel) so every output element has one writer.
 * --------------------------------------------------------------------- */
int orc_band_t(int BH, int n, int hd, int w, int wu, int dil, double alpha,
               const double *Bd, const double *Y, double *X, int G,
               const int *gidx, const double *Bg, const double *Br) {
    if (check_geom(BH, n, hd, w, wu, dil)) return -1;
    const int D = w + wu + 1, s = dil + 1;
    unsigned char *gm; int *gp;
    int rc = build_gmask(n, G, gidx, &gm, &gp);
    if (rc) return rc;
    const unsigned char *gmask = G > 0 ? gm : NULL;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int bh = 0; bh < BH; ++bh) {
        for (int c = 0; c < hd; ++c) {
            double *x = X + (size_t)bh * n * hd;
            const double *y = Y + (size_t)bh * n * hd;
            for (int j = 0; j < n; ++j) x[(size_t)j * hd + c] = 0.0;
            for (int i = 0; i < n; ++i) {
                const double yi = y[(size_t)i * hd + c];
                if (gmask && gmask[i]) {
                    const double *br = Br + ((size_t)bh * G + gp[i]) * n;
                    for (int j = 0; j < n; ++j) x[(size_t)j * hd + c] += alpha * br[j] * yi;
                    continue;
                }
                const double *b = Bd + ((size_t)bh * n + i) * D;
                for (int t = 0; t < D; ++t) {
                    if (!slot_used(i, t, w, s, n, gmask)) continue;
                    long long j = (long long)i + (long long)(t - w) * s;
                    x[(size_t)j * hd + c] += alpha * b[t] * yi;
                }
                for (int q = 0; q < G; ++q)
                    x[(size_t)gidx[q] * hd + c] +=
                        alpha * Bg[((size_t)bh * n + i) * G + q] * yi;
            }
        }
    }
    free(gm); free(gp);
    return 0;
}

/* ---------------------------------------------------------------------
 * Softmax backward on the band (the derivative of the row softmax above):
 *   local row i:  delta = sum_used P*dP + sum_g Pg*dPg
 *                 dS = P*(dP - delta) on used slots, 0 elsewhere
 *                 dSg = Pg*(dPg - delta)
 *   global row i = G[g]: delta = sum_j Pr*dPr;  dSr = Pr*(dPr - delta);
 *                 dS[i,:] = 0, dSg[i,:] = 0.
 * --------------------------------------------------------------------- */
int orc_band_softmax_bwd(int BH, int n, int w, int wu, int dil, const double *P,
                         const double *dP, double *dS, int G, const int *gidx,
                         const double *Pg, const double *dPg, double *dSg,
                         const double *Pr, const double *dPr, double *dSr,
                         uint64_t seed, int drop_t) {
    if (check_geom(BH, n, 1, w, wu, dil)) return -1;
    if (drop_t < 0 || drop_t > 255 || (drop_t > 0 && G > 0)) return -4;
    const int D = w + wu + 1, s = dil + 1;
    unsigned char *gm; int *gp;
    int rc = build_gmask(n, G, gidx, &gm, &gp);
    if (rc) return rc;
    const unsigned char *gmask = G > 0 ? gm : NULL;
#pragma omp parallel for collapse(2) schedule(static)
    for (int bh = 0; bh < BH; ++bh) {
        for (int i = 0; i < n; ++i) {
            const size_t r = (size_t)bh * n + i;
            if (gmask && gmask[i]) {
                const size_t k = ((size_t)bh * G + gp[i]) * n;
                double delta = 0.0;
                for (int j = 0; j < n; ++j) delta += Pr[k + j] * dPr[k + j];
                for (int j = 0; j < n; ++j) dSr[k + j] = Pr[k + j] * (dPr[k + j] - delta);
                for (int t = 0; t < D; ++t) dS[r * D + t] = 0.0;
                for (int q = 0; q < G; ++q) dSg[r * G + q] = 0.0;
                continue;
            }
            /* with dropout the forward's output is f*P and dP is its gradient:
             * the gradient reaching P is f*dP (f the slot key's keep-and-scale
             * factor, 1 without dropout) */
            double delta = 0.0;
            for (int t = 0; t < D; ++t)
                if (slot_used(i, t, w, s, n, gmask))
                    delta += P[r * D + t] * drop_factor(seed, drop_t, bh, i, i + (t - w) * s, s) *
                             dP[r * D + t];
            for (int q = 0; q < G; ++q) delta += Pg[r * G + q] * dPg[r * G + q];
            for (int t = 0; t < D; ++t)
                dS[r * D + t] = slot_used(i, t, w, s, n, gmask)
                                    ? P[r * D + t] * (drop_factor(seed, drop_t, bh, i, i + (t - w) * s, s) *
                                                      dP[r * D + t] - delta)
                                    : 0.0;
            for (int q = 0; q < G; ++q)
                dSg[r * G + q] = Pg[r * G + q] * (dPg[r * G + q] - delta);
        }
    }
    free(gm); free(gp);
    return 0;
}

/* ---------------------------------------------------------------------
 * Attention by its definition, on explicit key sets (no band slots):
 *   A(i) = { i + k*s : k in [-w, w_upper], 0 <= key < n, key not in G } u G
 *          for i not in G;   A(i) = [0, n) for i in G.
 *   p_ij = exp(scale*q_i.k_j - m_i) / Z_i over j in A(i);  O_i = sum p_ij v_j
 *   lse_i = m_i + log Z_i.
 * The key sets are kept in CSR form (row offsets + key lists).
 * --------------------------------------------------------------------- */
typedef struct {
    long long *off;  /* n*BH + 1 */
    int *key;
} keysets;

/* ---------------------------------------------------------------------
 * Dropout mask from the counter-based generator Philox4x64-10 (Salmon,
 * Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 * SC'11): ten rounds of two 64x64->128 multiplies with the published
 * multipliers, the key bumped by the published Weyl constants between
 * rounds.  Element (slice bh, query i, key j) with b = floor(j / s) reads byte
 * (b mod 32) of the block at counter (floor(b / 32), i, bh, 0) and key
 * (seed, 0), bytes taken little-endian from the four output words; it is
 * kept when that byte is >= drop_t (keep probability 1 - drop_t/256) and
 * then scaled by 256 / (256 - drop_t) (nvFuser issue, fusion 1: dropout with
 * 1/(1-p) scaling).
 * --------------------------------------------------------------------- */
static void mulhilo64(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo) {
    const uint64_t a0 = a & 0xffffffffu, a1 = a >> 32, b0 = b & 0xffffffffu, b1 = b >> 32;
    const uint64_t p00 = a0 * b0, p01 = a0 * b1, p10 = a1 * b0, p11 = a1 * b1;
    const uint64_t mid = (p00 >> 32) + (p01 & 0xffffffffu) + (p10 & 0xffffffffu);
    *lo = a * b;
    *hi = p11 + (p01 >> 32) + (p10 >> 32) + (mid >> 32);
}

int orc_philox4x64(const uint64_t *ctr, const uint64_t *key, uint64_t *out) {
    uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3], k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B97F4A7C15ull;
            k1 += 0xBB67AE8584CAA73Bull;
        }
        uint64_t hi0, lo0, hi1, lo1;
        mulhilo64(0xD2E7470EE14C6C93ull, c0, &hi0, &lo0);
        mulhilo64(0xCA5A826395121157ull, c2, &hi1, &lo1);
        const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
    return 0;
}

/* keep-and-scale factor of element (bh, i, j): 0 or 256 / (256 - drop_t) */
static double drop_factor(uint64_t seed, int drop_t, int bh, int i, int j, int s) {
    if (drop_t <= 0) return 1.0;
    const uint64_t b = (uint64_t)(j / s);
    const uint64_t ctr[4] = {b / 32, (uint64_t)i, (uint64_t)bh, 0};
    const uint64_t key[2] = {seed, 0};
    uint64_t out[4];
    orc_philox4x64(ctr, key, out);
    const int k = (int)(b % 32);
    const int byte = (int)((out[k / 8] >> (8 * (k % 8))) & 0xffu);
    return byte >= drop_t ? 256.0 / (256.0 - drop_t) : 0.0;
}

int orc_dropout_factor(uint64_t seed, int drop_t, int bh, int i, int j, int s, double *out) {
    if (drop_t < 0 || drop_t > 255 || s < 1) return -1;
    *out = drop_factor(seed, drop_t, bh, i, j, s);
    return 0;
}

static int build_keysets(int n, int w, int wu, int dil, int G, const int *gidx,
                         const unsigned char *gmask, keysets *ks) {
    const int s = dil + 1;
    ks->off = (long long *)malloc(sizeof(long long) * ((size_t)n + 1));
    if (!ks->off) return -3;
    ks->off[0] = 0;
    for (int i = 0; i < n; ++i) {
        long long cnt = 0;
        if (gmask && gmask[i]) {
            cnt = n;
        } else {
            for (int k = -w; k <= wu; ++k) {
                long long j = (long long)i + (long long)k * s;
                if (j >= 0 && j < n && !(gmask && gmask[j])) ++cnt;
            }
            cnt += G;
        }
        ks->off[i + 1] = ks->off[i] + cnt;
    }
    ks->key = (int *)malloc(sizeof(int) * (size_t)(ks->off[n] > 0 ? ks->off[n] : 1));
    if (!ks->key) { free(ks->off); return -3; }
    for (int i = 0; i < n; ++i) {
        long long p = ks->off[i];
        if (gmask && gmask[i]) {
            for (int j = 0; j < n; ++j) ks->key[p++] = j;
        } else {
            for (int k = -w; k <= wu; ++k) {
                long long j = (long long)i + (long long)k * s;
                if (j >= 0 && j < n && !(gmask && gmask[j])) ks->key[p++] = (int)j;
            }
            for (int g = 0; g < G; ++g) ks->key[p++] = gidx[g];
        }
    }
    return 0;
}

int orc_attention_fwd(int BH, int n, int hd, int w, int wu, int dil, double scale,
                      const double *Q, const double *K, const double *V, double *O,
                      double *lse, int G, const int *gidx, const double *kbias, uint64_t seed,
                      int drop_t) {
    if (check_geom(BH, n, hd, w, wu, dil)) return -1;
    if (drop_t < 0 || drop_t > 255 || (G > 0 && drop_t > 0)) return -4;
    const int s_ = dil + 1;
    unsigned char *gm; int *gp;
    int rc = build_gmask(n, G, gidx, &gm, &gp);
    if (rc) return rc;
    keysets ks;
    rc = build_keysets(n, w, wu, dil, G, gidx, G > 0 ? gm : NULL, &ks);
    if (rc) { free(gm); free(gp); return rc; }
#pragma omp parallel
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
#pragma omp for collapse(2) schedule(static)
        for (int bh = 0; bh < BH; ++bh) {
            for (int i = 0; i < n; ++i) {
                const double *q = Q + ((size_t)bh * n + i) * hd;
                const long long b0 = ks.off[i], cnt = ks.off[i + 1] - b0;
                double m = -INFINITY, z = 0.0;
                for (long long u = 0; u < cnt; ++u) {
                    x[u] = scale * dot(q, K + ((size_t)bh * n + ks.key[b0 + u]) * hd, hd) +
                           (kbias ? kbias[(size_t)bh * n + ks.key[b0 + u]] : 0.0);
                    m = fmax(m, x[u]);
                }
                for (long long u = 0; u < cnt; ++u) z += exp(x[u] - m);
                double *o = O + ((size_t)bh * n + i) * hd;
                for (int c = 0; c < hd; ++c) o[c] = 0.0;
                for (long long u = 0; u < cnt; ++u) {
                    const double p = exp(x[u] - m) / z *
                                     drop_factor(seed, drop_t, bh, i, ks.key[b0 + u], s_);
                    const double *v = V + ((size_t)bh * n + ks.key[b0 + u]) * hd;
                    for (int c = 0; c < hd; ++c) o[c] += p * v[c];
                }
                if (lse) lse[(size_t)bh * n + i] = m + log(z);
            }
        }
        free(x);
    }
    free(ks.off); free(ks.key); free(gm); free(gp);
    return 0;
}

/* Backward of the definition above, by scatter over (i, j in A(i)):
 *   dp_ij = dO_i . v_j;  ds_ij = p_ij (dp_ij - sum_j' p_ij' dp_ij')
 *   dQ_i = scale sum_j ds_ij k_j;  dK_j += scale ds_ij q_i;  dV_j += p_ij dO_i.
 * Phase 1 (parallel over rows) stores p and ds per (i, j in A(i)); phase 2
 * (parallel over slice and channel) scatters dK and dV with one writer per
 * element. */
int orc_attention_bwd(int BH, int n, int hd, int w, int wu, int dil, double scale,
                      const double *Q, const double *K, const double *V,
                      const double *dO, double *dQ, double *dK, double *dV, int G,
                      const int *gidx, const double *kbias, uint64_t seed, int drop_t) {
    if (check_geom(BH, n, hd, w, wu, dil)) return -1;
    if (drop_t < 0 || drop_t > 255 || (G > 0 && drop_t > 0)) return -4;
    const int s_ = dil + 1;
    unsigned char *gm; int *gp;
    int rc = build_gmask(n, G, gidx, &gm, &gp);
    if (rc) return rc;
    keysets ks;
    rc = build_keysets(n, w, wu, dil, G, gidx, G > 0 ? gm : NULL, &ks);
    if (rc) { free(gm); free(gp); return rc; }
    const long long nnz = ks.off[n];
    double *pbuf = (double *)malloc(sizeof(double) * (size_t)(BH * nnz > 0 ? BH * nnz : 1));
    double *sbuf = (double *)malloc(sizeof(double) * (size_t)(BH * nnz > 0 ? BH * nnz : 1));
    if (!pbuf || !sbuf) {
        free(pbuf); free(sbuf); free(ks.off); free(ks.key); free(gm); free(gp);
        return -3;
    }
#pragma omp parallel
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
#pragma omp for collapse(2) schedule(static)
        for (int bh = 0; bh < BH; ++bh) {
            for (int i = 0; i < n; ++i) {
                const double *q = Q + ((size_t)bh * n + i) * hd;
                const double *go = dO + ((size_t)bh * n + i) * hd;
                const long long b0 = ks.off[i], cnt = ks.off[i + 1] - b0;
                double *p = pbuf + (size_t)bh * nnz + b0;
                double *ds = sbuf + (size_t)bh * nnz + b0;
                double m = -INFINITY, z = 0.0, delta = 0.0;
                for (long long u = 0; u < cnt; ++u) {
                    x[u] = scale * dot(q, K + ((size_t)bh * n + ks.key[b0 + u]) * hd, hd) +
                           (kbias ? kbias[(size_t)bh * n + ks.key[b0 + u]] : 0.0);
                    m = fmax(m, x[u]);
                }
                for (long long u = 0; u < cnt; ++u) z += exp(x[u] - m);
                /* with dropout the product uses p * f (f the keep-and-scale
                 * factor): dP~ = f dP, delta = sum p f dP = dO . O, and
                 * dS = p (f dP - delta); dV takes p f */
                for (long long u = 0; u < cnt; ++u) {
                    const double f = drop_factor(seed, drop_t, bh, i, ks.key[b0 + u], s_);
                    p[u] = exp(x[u] - m) / z;
                    ds[u] = f * dot(go, V + ((size_t)bh * n + ks.key[b0 + u]) * hd, hd);
                    delta += p[u] * ds[u];
                }
                double *gq = dQ + ((size_t)bh * n + i) * hd;
                for (int c = 0; c < hd; ++c) gq[c] = 0.0;
                for (long long u = 0; u < cnt; ++u) {
                    ds[u] = p[u] * (ds[u] - delta);
                    p[u] *= drop_factor(seed, drop_t, bh, i, ks.key[b0 + u], s_);
                    const double *k = K + ((size_t)bh * n + ks.key[b0 + u]) * hd;
                    for (int c = 0; c < hd; ++c) gq[c] += scale * ds[u] * k[c];
                }
            }
        }
        free(x);
#pragma omp for collapse(2) schedule(dynamic)
        for (int bh = 0; bh < BH; ++bh) {
            for (int c = 0; c < hd; ++c) {
                for (int j = 0; j < n; ++j) {
                    dK[((size_t)bh * n + j) * hd + c] = 0.0;
                    dV[((size_t)bh * n + j) * hd + c] = 0.0;
                }
                for (int i = 0; i < n; ++i) {
                    const double qi = Q[((size_t)bh * n + i) * hd + c];
                    const double gi = dO[((size_t)bh * n + i) * hd + c];
                    for (long long u = ks.off[i]; u < ks.off[i + 1]; ++u) {
                        const size_t j = (size_t)ks.key[u];
                        dK[((size_t)bh * n + j) * hd + c] += scale * sbuf[(size_t)bh * nnz + u] * qi;
                        dV[((size_t)bh * n + j) * hd + c] += pbuf[(size_t)bh * nnz + u] * gi;
                    }
                }
            }
        }
    }
    free(pbuf); free(sbuf); free(ks.off); free(ks.key); free(gm); free(gp);
    return 0;
}

/* ---------------------------------------------------------------------
 * AddBiasTranspose (ONNX Runtime issue "[WIP] Improve LongformerAttention
 * performance", item (2): bias add and transpose after the merged
 * projection): X holds rows of [b, n, M, h, hd] (M projections side by
 * side), bias is [M, h, hd] (or NULL), Y is [M, b, h, n, hd]:
 *   Y[m][bb][hh][i][c] = X[bb][i][m][hh][c] + bias[m][hh][c].
 * --------------------------------------------------------------------- */
int orc_add_bias_transpose(int b, int n, int M, int h, int hd, const double *X,
                           const double *bias, double *Y) {
    if (b < 1 || n < 1 || M < 1 || h < 1 || hd < 1) return -1;
    for (int m = 0; m < M; ++m)
        for (int bb = 0; bb < b; ++bb)
            for (int hh = 0; hh < h; ++hh)
                for (int i = 0; i < n; ++i)
                    for (int c = 0; c < hd; ++c) {
                        const size_t src = ((((size_t)bb * n + i) * M + m) * h + hh) * hd + c;
                        const size_t dst = ((((size_t)m * b + bb) * h + hh) * n + i) * hd + c;
                        Y[dst] = X[src] + (bias ? bias[((size_t)m * h + hh) * hd + c] : 0.0);
                    }
    return 0;
}

/* ---------------------------------------------------------------------
 * Global queries with their own projections (ONNX Runtime issue, item (3):
 * the global_q projection computed only for the global tokens, i.e. a
 * compact Qg; separate global key / value projections Kg, Vg over every
 * position).  Per slice bh and global query g:
 *   p_gj = exp(scale * Qg[g].Kg[j] - m_g) / Z_g over all j in [0, n)
 *   Og[g] = sum_j p_gj Vg[j],   lseg[g] = m_g + log Z_g.
 * Backward (dOg given): delta_g = dOg[g].Og[g],
 *   ds_gj = p_gj (dOg[g].Vg[j] - delta_g),
 *   dQg[g] = scale sum_j ds_gj Kg[j],  dKg[j] = scale sum_g ds_gj Qg[g],
 *   dVg[j] = sum_g p_gj dOg[g].
 * --------------------------------------------------------------------- */
int orc_global_attention_fwd(int BH, int G, int n, int hd, double scale, const double *Qg,
                             const double *Kg, const double *Vg, double *Og, double *lseg) {
    if (BH < 1 || G < 1 || n < 1 || hd < 1) return -1;
#pragma omp parallel for collapse(2) schedule(static)
    for (int bh = 0; bh < BH; ++bh) {
        for (int g = 0; g < G; ++g) {
            const double *q = Qg + ((size_t)bh * G + g) * hd;
            const double *K = Kg + (size_t)bh * n * hd, *V = Vg + (size_t)bh * n * hd;
            double *o = Og + ((size_t)bh * G + g) * hd;
            double m = -INFINITY, z = 0.0;
            for (int j = 0; j < n; ++j) m = fmax(m, scale * dot(q, K + (size_t)j * hd, hd));
            for (int c = 0; c < hd; ++c) o[c] = 0.0;
            for (int j = 0; j < n; ++j) {
                const double e = exp(scale * dot(q, K + (size_t)j * hd, hd) - m);
                z += e;
                for (int c = 0; c < hd; ++c) o[c] += e * V[(size_t)j * hd + c];
            }
            for (int c = 0; c < hd; ++c) o[c] /= z;
            lseg[(size_t)bh * G + g] = m + log(z);
        }
    }
    return 0;
}

int orc_global_attention_bwd(int BH, int G, int n, int hd, double scale, const double *Qg,
                             const double *Kg, const double *Vg, const double *dOg, double *dQg,
                             double *dKg, double *dVg) {
    if (BH < 1 || G < 1 || n < 1 || hd < 1) return -1;
#pragma omp parallel for schedule(static)
    for (int bh = 0; bh < BH; ++bh) {
        const double *K = Kg + (size_t)bh * n * hd, *V = Vg + (size_t)bh * n * hd;
        double *dK = dKg + (size_t)bh * n * hd, *dV = dVg + (size_t)bh * n * hd;
        for (size_t e = 0; e < (size_t)n * hd; ++e) dK[e] = dV[e] = 0.0;
        double *p = (double *)malloc(sizeof(double) * (size_t)n);
        double *o = (double *)malloc(sizeof(double) * (size_t)hd);
        for (int g = 0; g < G; ++g) {
            const double *q = Qg + ((size_t)bh * G + g) * hd;
            const double *dO = dOg + ((size_t)bh * G + g) * hd;
            double *dq = dQg + ((size_t)bh * G + g) * hd;
            /* the probabilities of this global query and its output */
            double m = -INFINITY, z = 0.0;
            for (int j = 0; j < n; ++j) {
                p[j] = scale * dot(q, K + (size_t)j * hd, hd);
                m = fmax(m, p[j]);
            }
            for (int j = 0; j < n; ++j) {
                p[j] = exp(p[j] - m);
                z += p[j];
            }
            for (int c = 0; c < hd; ++c) o[c] = 0.0;
            for (int j = 0; j < n; ++j) {
                p[j] /= z;
                for (int c = 0; c < hd; ++c) o[c] += p[j] * V[(size_t)j * hd + c];
            }
            const double delta = dot(dO, o, hd);
            for (int c = 0; c < hd; ++c) dq[c] = 0.0;
            for (int j = 0; j < n; ++j) {
                const double ds = p[j] * (dot(dO, V + (size_t)j * hd, hd) - delta);
                for (int c = 0; c < hd; ++c) {
                    dq[c] += scale * ds * K[(size_t)j * hd + c];
                    dK[(size_t)j * hd + c] += scale * ds * q[c];
                    dV[(size_t)j * hd + c] += p[j] * dO[c];
                }
            }
        }
        free(p); free(o);
    }
    return 0;
}
