/*
 * Exact-attention oracle: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may call this file. The GPU library never links or calls it, and it shares no code,
 * header, table or constant with the GPU library.
 *
 * What is computed is the plain definition of attention, written out with every N x N
 * matrix materialised per head, in the order the pages state it:
 *
 *   S = scale * Q K^T            "Standard attention", FlashAttention-2 reading notes,
 *                                eq. (2); the 1/sqrt(d) scale from the FlashAttention post
 *                                (bluuewhale), section "How Attention Is Computed".
 *   S_ij = -inf where masked     causal: key j > query i (FlashAttention-2 reading notes,
 *                                section on causal masking); block-sparse: mask entry
 *                                M[i/128][j/128] == 0 (FlashAttention post, section
 *                                "Block-Sparse FlashAttention").
 *   P = softmax(S) by the three-pass safe softmax: pass 1 row max, pass 2 sum of
 *                                exp(S - max), pass 3 normalise ("Flash Attention v1",
 *                                languisher.top, sections "Naive Attention" and
 *                                "Online Softmax", the three-pass description).
 *   O = P V                      FlashAttention-2 reading notes, eq. (4).
 *   LSE_i = m_i + ln(l_i)        FlashAttention-2 reading notes, eq. (15).
 *
 * Backward (analytic gradient of L = sum(O o dO)):
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,  dS = P o (dP - D),
 *   dQ = scale * dS K,  dK = scale * dS^T Q
 *   (FlashAttention-2 reading notes, Algorithm 2 and the softmax-Jacobian identity eq. (17);
 *   D here is the definition <p, dp>; the identity D = rowsum(dO o O) from the FlashAttention
 *   paper-detail page, "Technique 2 (Recomputation)", is checked separately by the tests.)
 *
 * Readings where the pages are silent: a row with every score masked has O = 0, LSE = -inf
 * and zero gradients; the block mask is shared by every (batch, head) and indexed with ceil
 * for ragged tails.
 *
 * Parallelism: OpenMP over rows inside each matrix product of one head; heads one at a time.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static int masked(long i, long j, int causal, const uint8_t *mask, int tiles, int block) {
    if (causal && j > i) return 1;
    if (mask && !mask[(i / block) * (long)tiles + (j / block)]) return 1;
    return 0;
}

/* Tiles per side of the block mask: ceil(max(Nq, Nk) / block). */
static int mask_tiles(long Nq, long Nk, int block) {
    long n = Nq > Nk ? Nq : Nk;
    return (int)((n + block - 1) / block);
}

/* S = scale * Q K^T with masked entries set to -inf. q: [Nq][d], k: [Nk][d]; S: [Nq][Nk]. */
static void scores(long Nq, long Nk, long d, const double *q, const double *k, double scale,
                   int causal, const uint8_t *mask, int block, double *S) {
    int tiles = mask_tiles(Nq, Nk, block);
#pragma omp parallel for schedule(static)
    for (long i = 0; i < Nq; ++i) {
        for (long j = 0; j < Nk; ++j) {
            double acc = 0.0;
            for (long c = 0; c < d; ++c) acc += q[i * d + c] * k[j * d + c];
            S[i * Nk + j] = masked(i, j, causal, mask, tiles, block) ? -INFINITY : scale * acc;
        }
    }
}

/* Three-pass safe softmax of every row of S into P; m and l receive the row max and sum. */
static void softmax_rows(long Nq, long Nk, const double *S, double *P, double *m, double *l) {
#pragma omp parallel for schedule(static)
    for (long i = 0; i < Nq; ++i) {
        const double *s = S + i * Nk;
        double *p = P + i * Nk;
        double mx = -INFINITY;
        for (long j = 0; j < Nk; ++j)           /* pass 1: max */
            if (s[j] > mx) mx = s[j];
        if (mx == -INFINITY) {                  /* every entry masked */
            for (long j = 0; j < Nk; ++j) p[j] = 0.0;
            m[i] = -INFINITY;
            l[i] = 0.0;
            continue;
        }
        double sum = 0.0;
        for (long j = 0; j < Nk; ++j)           /* pass 2: normaliser */
            sum += exp(s[j] - mx);
        for (long j = 0; j < Nk; ++j)           /* pass 3: probabilities */
            p[j] = exp(s[j] - mx) / sum;
        m[i] = mx;
        l[i] = sum;
    }
}

/* C[R][d] = A[R][K] B[K][d] */
static void mm_nn(long R, long K, long d, const double *A, const double *B, double *C) {
#pragma omp parallel for schedule(static)
    for (long i = 0; i < R; ++i) {
        double *c = C + i * d;
        for (long x = 0; x < d; ++x) c[x] = 0.0;
        for (long j = 0; j < K; ++j) {
            double a = A[i * K + j];
            const double *b = B + j * d;
            for (long x = 0; x < d; ++x) c[x] += a * b[x];
        }
    }
}

/* C[K][d] = A[R][K]^T B[R][d] */
static void mm_tn(long R, long K, long d, const double *A, const double *B, double *C) {
#pragma omp parallel for schedule(static)
    for (long j = 0; j < K; ++j) {
        double *c = C + j * d;
        for (long x = 0; x < d; ++x) c[x] = 0.0;
        for (long i = 0; i < R; ++i) {
            double a = A[i * K + j];
            const double *b = B + i * d;
            for (long x = 0; x < d; ++x) c[x] += a * b[x];
        }
    }
}

/* C[R][K] = A[R][d] B[K][d]^T */
static void mm_nt(long R, long K, long d, const double *A, const double *B, double *C) {
#pragma omp parallel for schedule(static)
    for (long i = 0; i < R; ++i)
        for (long j = 0; j < K; ++j) {
            double acc = 0.0;
            for (long x = 0; x < d; ++x) acc += A[i * d + x] * B[j * d + x];
            C[i * K + j] = acc;
        }
}

/* Scores of one head (for the tests' bound and sum checks). S: [Nq][Nk]. */
int oracle_scores(long Nq, long Nk, long d, const double *q, const double *k, double scale,
                  int causal, const uint8_t *mask, int block, double *S) {
    if (Nq < 1 || Nk < 1 || d < 1 || block < 1) return -1;
    scores(Nq, Nk, d, q, k, scale, causal, mask, block, S);
    return 0;
}

/* Probabilities of one head: P = softmax(S), [Nq][Nk]. */
int oracle_probabilities(long Nq, long Nk, long d, const double *q, const double *k,
                         double scale, int causal, const uint8_t *mask, int block, double *P) {
    if (Nq < 1 || Nk < 1 || d < 1 || block < 1) return -1;
    double *S = (double *)malloc(sizeof(double) * Nq * Nk);
    double *m = (double *)malloc(sizeof(double) * Nq);
    double *l = (double *)malloc(sizeof(double) * Nq);
    if (!S || !m || !l) { free(S); free(m); free(l); return -2; }
    scores(Nq, Nk, d, q, k, scale, causal, mask, block, S);
    softmax_rows(Nq, Nk, S, P, m, l);
    free(S); free(m); free(l);
    return 0;
}

/*
 * Full forward (and, when dout != NULL, backward) over BH heads.
 * q, o, dout, dq: [BH][Nq][d]; k, v, dk, dv: [BH][Nk][d]; lse, delta: [BH][Nq]; fp64.
 * Backward outputs dq, dk, dv (and delta when non-NULL) are written only when dout != NULL.
 * Causal masking compares absolute indices (query i sees keys j <= i).
 */
int oracle_attention(long BH, long Nq, long Nk, long d, const double *q, const double *k,
                     const double *v, const double *dout, double scale, int causal,
                     const uint8_t *mask, int block, double *o, double *lse, double *dq,
                     double *dk, double *dv, double *delta) {
    if (BH < 1 || Nq < 1 || Nk < 1 || d < 1 || block < 1) return -1;
    double *S = (double *)malloc(sizeof(double) * Nq * Nk);
    double *P = (double *)malloc(sizeof(double) * Nq * Nk);
    double *m = (double *)malloc(sizeof(double) * Nq);
    double *l = (double *)malloc(sizeof(double) * Nq);
    double *D = (double *)malloc(sizeof(double) * Nq);
    if (!S || !P || !m || !l || !D) { free(S); free(P); free(m); free(l); free(D); return -2; }
    for (long h = 0; h < BH; ++h) {
        const double *qh = q + h * Nq * d, *kh = k + h * Nk * d, *vh = v + h * Nk * d;
        double *oh = o + h * Nq * d;
        scores(Nq, Nk, d, qh, kh, scale, causal, mask, block, S);
        softmax_rows(Nq, Nk, S, P, m, l);
        mm_nn(Nq, Nk, d, P, vh, oh);                         /* O = P V */
        for (long i = 0; i < Nq; ++i)
            lse[h * Nq + i] = (m[i] == -INFINITY) ? -INFINITY : m[i] + log(l[i]);
        if (!dout) continue;
        const double *doh = dout + h * Nq * d;
        double *dP = S; /* S is no longer needed: reuse it for dP, then dS */
        mm_tn(Nq, Nk, d, P, doh, dv + h * Nk * d);           /* dV = P^T dO */
        mm_nt(Nq, Nk, d, doh, vh, dP);                       /* dP = dO V^T */
#pragma omp parallel for schedule(static)
        for (long i = 0; i < Nq; ++i) {                      /* D_i = <P_i, dP_i> */
            double acc = 0.0;
            for (long j = 0; j < Nk; ++j) acc += P[i * Nk + j] * dP[i * Nk + j];
            D[i] = acc;
        }
#pragma omp parallel for schedule(static)
        for (long i = 0; i < Nq; ++i)                        /* dS = P o (dP - D) */
            for (long j = 0; j < Nk; ++j)
                dP[i * Nk + j] = P[i * Nk + j] * (dP[i * Nk + j] - D[i]);
        double *dqh = dq + h * Nq * d, *dkh = dk + h * Nk * d;
        mm_nn(Nq, Nk, d, dP, kh, dqh);                       /* dQ = dS K */
        mm_tn(Nq, Nk, d, dP, qh, dkh);                       /* dK = dS^T Q */
        for (long x = 0; x < Nq * d; ++x) dqh[x] *= scale;
        for (long x = 0; x < Nk * d; ++x) dkh[x] *= scale;
        if (delta)
            for (long i = 0; i < Nq; ++i) delta[h * Nq + i] = D[i];
    }
    free(S); free(P); free(m); free(l); free(D);
    return 0;
}

/*
 * Forward for selected query rows of ONE head (softmax is row-wise, so a row's result needs
 * only that row of S). q: [Nq][d]; k, v: [Nk][d]; rows: nrows indices in [0, Nq);
 * o_rows: [nrows][d]; lse_rows: [nrows].
 */
int oracle_forward_rows(long Nq, long Nk, long d, const double *q, const double *k,
                        const double *v, double scale, int causal, const uint8_t *mask, int block,
                        long nrows, const long *rows, double *o_rows, double *lse_rows) {
    if (Nq < 1 || Nk < 1 || d < 1 || block < 1 || nrows < 0) return -1;
    int tiles = mask_tiles(Nq, Nk, block);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (long r = 0; r < nrows; ++r) {
        long i = rows[r];
        if (i < 0 || i >= Nq) { bad = 1; continue; }
        double *s = (double *)malloc(sizeof(double) * Nk);
        if (!s) { bad = 1; continue; }
        for (long j = 0; j < Nk; ++j) {
            double acc = 0.0;
            for (long c = 0; c < d; ++c) acc += q[i * d + c] * k[j * d + c];
            s[j] = masked(i, j, causal, mask, tiles, block) ? -INFINITY : scale * acc;
        }
        double mx = -INFINITY;
        for (long j = 0; j < Nk; ++j) if (s[j] > mx) mx = s[j];
        double *orow = o_rows + r * d;
        for (long c = 0; c < d; ++c) orow[c] = 0.0;
        if (mx == -INFINITY) { lse_rows[r] = -INFINITY; free(s); continue; }
        double sum = 0.0;
        for (long j = 0; j < Nk; ++j) sum += exp(s[j] - mx);
        for (long j = 0; j < Nk; ++j) {
            double p = exp(s[j] - mx) / sum;
            for (long c = 0; c < d; ++c) orow[c] += p * v[j * d + c];
        }
        lse_rows[r] = mx + log(sum);
        free(s);
    }
    return bad ? -1 : 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
