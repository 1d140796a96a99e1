/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for the
 * contractions of the hot path and for IKBO attention.  TEST
 * INFRASTRUCTURE ONLY: the product path (the CUDA library) never links,
 * loads or calls this file; only the tests,
 * the smoke check and the benchmark's CPU-baseline leg do.
 *
 * Everything is accumulated in IEEE double.  bf16 inputs (passed as their
 * raw 16-bit patterns) are widened exactly: a bf16 value is the top half of
 * an fp32 value, and every fp32 value is exactly a double.
 *
 * Sources (web pages on Meta's TLX):
 *   [P1] "How We Built TLX: A Hardware-Native GPU Compiler for Production ML
 *        at Scale" (engineering.fb.com).
 *   [P3] "TLX in production" commentary (yuxiaoba.github.io).
 *
 *   gemm      -- [P1] "Introducing TLX": the tiled matmul keeps an fp32
 *                accumulator and adds dot(a_tile, b_tile) over K; the
 *                blocked loop computes C[m][n] = sum_k A[m][k] * B[k][n].
 *                Written here as that definition, one k at a time.
 *   epilogue  -- [P1] "Five key areas" (model-aware fusion) names fusing
 *                elementwise work into the matmul; the bias + activation
 *                forms add the bias first, then SiLU(x) = x / (1 + exp(-x))
 *                or GELU(x) = x * Phi(x) (the exact erf form; "other
 *                activations" of the norm-fusion companion work).
 *   grouped   -- [P1] "TLX in Production" / "Case Study 3: Distributed
 *                Grouped GEMM for LLM Pretraining": one GEMM per expert over
 *                that expert's rows; written as a loop of plain GEMMs.
 *   ikbo      -- [P1] "Case Study 2: In-Kernel Broadcast Optimization for
 *                RecSys": user features are the same for every candidate of
 *                a user; the reference form MATERIALISES the broadcast
 *                (one copy of the user's features per candidate), then does
 *                the dense linear compression Y[c] = W . concat(U[u], C[c]).
 *   ikbo_decomposed -- the same section's "matmul decomposition": W split
 *                column-wise into the user part and the candidate part,
 *                Y[c] = W_u . U[u] + W_c . C[c].  A second, independent
 *                coding used only to cross-check the materialised form.
 *   ikbo_attention -- [P1] "Case Study 2" names an IKBO form of
 *                FlashAttention in which the candidates of one user share
 *                the reads of that user's keys and values.  The pages print
 *                no formula; the reading used: every query row of candidate
 *                c attends over the
 *                context (keys, values) of its user u = user(c), per head,
 *                o = sum_j softmax_j(scale * q . k_j) v_j, no mask.  The
 *                reference form materialises the broadcast: one copy of the
 *                user's K and V per candidate.
 *   ikbo_attention_grouped -- a second coding of the same result: per user
 *                and head, the query rows of all of the user's candidates
 *                stacked into one matrix, S = Q K^T, row softmax, O = P V
 *                (the IKBO form), with no per-candidate copy.
 *
 * Threading: OpenMP over independent output rows / candidates only; each
 * output element is one sequential k-ordered sum, so the thread count does
 * not change any result.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern. */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* SiLU(x) = x * sigmoid(x) = x / (1 + e^-x). */
static double silu(double x)
{
    return x / (1.0 + exp(-x));
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* GELU(x) = x * Phi(x), Phi(x) = erfc(-x / sqrt(2)) / 2 the standard normal
 * distribution function (the exact, erf form of GELU). */
static double gelu(double x)
{
    return 0.5 * x * erfc(-x / sqrt(2.0));
}

/* Epilogue codes: 0 none, 1 + bias[n], 2 + bias[n] then SiLU, 3 + bias[n]
 * then GELU. */
static double apply_epilogue(double acc, int epi, const uint16_t *bias_row, int n)
{
    if (epi >= 1) acc += bf16_to_double(bias_row[n]);
    if (epi == 2) acc = silu(acc);
    if (epi == 3) acc = gelu(acc);
    return acc;
}

/*
 * Batched dense GEMM, C[b][m][n] = epi( sum_k A[b][m][k] * B[b][n][k] ).
 *   A: bf16, element (b,m,k) at A[b*sA + m*lda + k]      (row-major M x K)
 *   B: bf16, element (b,n,k) at B[b*sB + n*ldb + k]      (N x K, K contiguous:
 *      the column-major K x N operand)
 *   bias: bf16, element (b,n) at bias[b*sBias + n]; may be NULL when epi == 0
 *   C: double, element (b,m,n) at C[b*sC + m*ldc + n]
 *   rows: if non-NULL, only the listed m (nrows of them) are computed, for
 *         every b; other rows of C are not touched.
 */
void oracle_gemm(int batch, int M, int N, int K,
                 const uint16_t *A, long lda, long sA,
                 const uint16_t *B, long ldb, long sB,
                 const uint16_t *bias, long sBias, int epi,
                 double *C, long ldc, long sC,
                 const int *rows, int nrows)
{
    long nr = rows ? nrows : M;
    long total = (long)batch * nr;
    #pragma omp parallel for schedule(dynamic, 1)
    for (long idx = 0; idx < total; ++idx) {
        int b = (int)(idx / nr);
        int m = rows ? rows[idx % nr] : (int)(idx % nr);
        const uint16_t *a = A + (long)b * sA + (long)m * lda;
        const uint16_t *bias_row = bias ? bias + (long)b * sBias : 0;
        double *c = C + (long)b * sC + (long)m * ldc;
        for (int n = 0; n < N; ++n) {
            const uint16_t *bn = B + (long)b * sB + (long)n * ldb;
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += bf16_to_double(a[k]) * bf16_to_double(bn[k]);
            c[n] = apply_epilogue(acc, epi, bias_row, n);
        }
    }
}

/*
 * GEMM on RMS-normalised rows of A (norm fused into the GEMM; any learned
 * per-feature scale is taken as already folded into B):
 *   r[b][m]    = 1 / sqrt( (1/K) sum_k A[b][m][k]^2 + eps )
 *   C[b][m][n] = epi( r[b][m] * sum_k A[b][m][k] * B[b][n][k] (+ bias[b][n]) )
 * Same argument conventions as oracle_gemm, plus eps.  The pages only name
 * "norm fusion into GEMM" (a companion post of "How We Built TLX: A
 * Hardware-Native GPU Compiler for Production ML at Scale"); this is the
 * plainest RMSNorm reading.
 */
void oracle_gemm_rmsnorm(int batch, int M, int N, int K,
                         const uint16_t *A, long lda, long sA,
                         const uint16_t *B, long ldb, long sB, double eps,
                         const uint16_t *bias, long sBias, int epi,
                         double *C, long ldc, long sC,
                         const int *rows, int nrows)
{
    long nr = rows ? nrows : M;
    long total = (long)batch * nr;
    #pragma omp parallel for schedule(dynamic, 1)
    for (long idx = 0; idx < total; ++idx) {
        int b = (int)(idx / nr);
        int m = rows ? rows[idx % nr] : (int)(idx % nr);
        const uint16_t *a = A + (long)b * sA + (long)m * lda;
        const uint16_t *bias_row = bias ? bias + (long)b * sBias : 0;
        double *c = C + (long)b * sC + (long)m * ldc;
        double ss = 0.0;
        for (int k = 0; k < K; ++k) {
            double x = bf16_to_double(a[k]);
            ss += x * x;
        }
        double r = 1.0 / sqrt(ss / (double)K + eps);
        for (int n = 0; n < N; ++n) {
            const uint16_t *bn = B + (long)b * sB + (long)n * ldb;
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += bf16_to_double(a[k]) * bf16_to_double(bn[k]);
            c[n] = apply_epilogue(r * acc, epi, bias_row, n);
        }
    }
}

/*
 * GEMM on LayerNorm-normalised rows of A (same conventions as
 * oracle_gemm_rmsnorm).  For each row: mu = (1/K) sum_k a[k],
 * var = (1/K) sum_k (a[k] - mu)^2 (two passes), xhat[k] = (a[k] - mu) /
 * sqrt(var + eps), then C[n] = epi(sum_k xhat[k] * B[n][k] (+ bias[n])): the
 * norm's learned scale folded into B and its shift into the bias.
 */
void oracle_gemm_layernorm(int batch, int M, int N, int K,
                           const uint16_t *A, long lda, long sA,
                           const uint16_t *B, long ldb, long sB, double eps,
                           const uint16_t *bias, long sBias, int epi,
                           double *C, long ldc, long sC,
                           const int *rows, int nrows)
{
    long nr = rows ? nrows : M;
    long total = (long)batch * nr;
    #pragma omp parallel
    {
        double *xh = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        #pragma omp for schedule(dynamic, 1)
        for (long idx = 0; idx < total; ++idx) {
            int b = (int)(idx / nr);
            int m = rows ? rows[idx % nr] : (int)(idx % nr);
            const uint16_t *a = A + (long)b * sA + (long)m * lda;
            const uint16_t *bias_row = bias ? bias + (long)b * sBias : 0;
            double *c = C + (long)b * sC + (long)m * ldc;
            if (!xh) { for (int n = 0; n < N; ++n) c[n] = NAN; continue; }
            double mu = 0.0;
            for (int k = 0; k < K; ++k) mu += bf16_to_double(a[k]);
            mu /= (double)K;
            double var = 0.0;
            for (int k = 0; k < K; ++k) {
                double d = bf16_to_double(a[k]) - mu;
                var += d * d;
            }
            var /= (double)K;
            double r = 1.0 / sqrt(var + eps);
            for (int k = 0; k < K; ++k) xh[k] = (bf16_to_double(a[k]) - mu) * r;
            for (int n = 0; n < N; ++n) {
                const uint16_t *bn = B + (long)b * sB + (long)n * ldb;
                double acc = 0.0;
                for (int k = 0; k < K; ++k)
                    acc += xh[k] * bf16_to_double(bn[k]);
                c[n] = apply_epilogue(acc, epi, bias_row, n);
            }
        }
        free(xh);
    }
}

/*
 * Grouped GEMM: group g owns rows [off[g], off[g+1]) of A and C and uses
 * weight matrix B[g] (N x K, K contiguous, at B + g*sBg).  Empty groups
 * contribute nothing.  bias (if epi > 0) is per group: bias + g*sBias.
 * off is a HOST array of G+1 ints.  Returns 0, or -1 if off is not a
 * non-decreasing sequence from 0 to M_total.
 */
int oracle_grouped(int G, int M_total, int N, int K,
                   const uint16_t *A, long lda,
                   const uint16_t *B, long ldb, long sBg,
                   const int *off,
                   const uint16_t *bias, long sBias, int epi,
                   double *C, long ldc)
{
    if (off[0] != 0 || off[G] != M_total) return -1;
    for (int g = 0; g < G; ++g)
        if (off[g + 1] < off[g]) return -1;
    for (int g = 0; g < G; ++g) {
        int Mg = off[g + 1] - off[g];
        if (Mg == 0) continue;
        oracle_gemm(1, Mg, N, K,
                    A + (long)off[g] * lda, lda, 0,
                    B + (long)g * sBg, ldb, 0,
                    bias ? bias + (long)g * sBias : 0, 0, epi,
                    C + (long)off[g] * ldc, ldc, 0, 0, 0);
    }
    return 0;
}

/* Owner of candidate c under the contiguous per-user candidate blocks. */
static int user_of(int num_users, const int *uoff, int c)
{
    int u = 0;
    while (u < num_users && uoff[u + 1] <= c) ++u;
    return u;
}

/*
 * IKBO linear compression, materialised reference form.
 *   U : bf16 [num_users][Du][D]     user features
 *   Cf: bf16 [num_cand][Dc][D]      candidate features
 *   W : bf16 [O][Du+Dc]             compression weights (U part first)
 *   uoff: host int[num_users+1], candidates of user u are [uoff[u], uoff[u+1])
 *   Y : double [num_cand][O][D]
 *   cands: if non-NULL, only the listed candidates (ncands) are computed.
 * For each candidate the user's features are copied out (the broadcast the
 * in-kernel method avoids), stacked above the candidate's rows, and W is
 * applied to the stacked [Du+Dc][D] matrix.  Returns -1 on bad offsets.
 */
int oracle_ikbo(int num_users, int num_cand, int Du, int Dc, int D, int O,
                const uint16_t *U, const uint16_t *Cf, const uint16_t *W,
                const int *uoff, double *Y, const int *cands, int ncands)
{
    if (uoff[0] != 0 || uoff[num_users] != num_cand) return -1;
    for (int u = 0; u < num_users; ++u)
        if (uoff[u + 1] < uoff[u]) return -1;
    int F = Du + Dc;
    long n = cands ? ncands : num_cand;
    int bad = 0;
    #pragma omp parallel
    {
        /* Per-thread buffer for one materialised X[c] = [F][D]. */
        double *X = (double *)malloc(sizeof(double) * (size_t)F * (size_t)D);
        if (!X) bad = 1;
        #pragma omp for schedule(dynamic, 4)
        for (long i = 0; i < n; ++i) {
            int c = cands ? cands[i] : (int)i;
            if (!X || c < 0 || c >= num_cand) { bad = 1; continue; }
            int u = user_of(num_users, uoff, c);
            /* The broadcast: copy user u's rows, then candidate c's rows. */
            for (int f = 0; f < Du; ++f)
                for (int d = 0; d < D; ++d)
                    X[(long)f * D + d] = bf16_to_double(U[((long)u * Du + f) * D + d]);
            for (int f = 0; f < Dc; ++f)
                for (int d = 0; d < D; ++d)
                    X[(long)(Du + f) * D + d] = bf16_to_double(Cf[((long)c * Dc + f) * D + d]);
            /* Dense linear compression Y[c] = W . X[c]. */
            double *y = Y + (long)c * O * D;
            for (int o = 0; o < O; ++o)
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int f = 0; f < F; ++f)
                        acc += bf16_to_double(W[(long)o * F + f]) * X[(long)f * D + d];
                    y[(long)o * D + d] = acc;
                }
        }
        free(X);
    }
    return bad ? -2 : 0;
}

/*
 * IKBO by matmul decomposition: P[u] = W[:, :Du] . U[u] once per user, then
 * Y[c] = W[:, Du:] . Cf[c] + P[user(c)].  Same argument conventions as
 * oracle_ikbo; P is caller scratch of num_users*O*D doubles.
 */
int oracle_ikbo_decomposed(int num_users, int num_cand, int Du, int Dc, int D, int O,
                           const uint16_t *U, const uint16_t *Cf, const uint16_t *W,
                           const int *uoff, double *Y, double *P)
{
    if (uoff[0] != 0 || uoff[num_users] != num_cand) return -1;
    for (int u = 0; u < num_users; ++u)
        if (uoff[u + 1] < uoff[u]) return -1;
    int F = Du + Dc;
    #pragma omp parallel for
    for (int u = 0; u < num_users; ++u)
        for (int o = 0; o < O; ++o)
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int f = 0; f < Du; ++f)
                    acc += bf16_to_double(W[(long)o * F + f]) *
                           bf16_to_double(U[((long)u * Du + f) * D + d]);
                P[((long)u * O + o) * D + d] = acc;
            }
    #pragma omp parallel for schedule(dynamic, 4)
    for (int c = 0; c < num_cand; ++c) {
        int u = user_of(num_users, uoff, c);
        for (int o = 0; o < O; ++o)
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int f = 0; f < Dc; ++f)
                    acc += bf16_to_double(W[(long)o * F + Du + f]) *
                           bf16_to_double(Cf[((long)c * Dc + f) * D + d]);
                Y[((long)c * O + o) * D + d] = acc + P[((long)u * O + o) * D + d];
            }
    }
    return 0;
}

/*
 * IKBO attention, materialised reference form.
 *   Q : bf16 [num_cand*Lq][H][Dh]      query rows; candidate c owns rows
 *                                      [c*Lq, (c+1)*Lq)
 *   K, V: bf16 [num_users][Lkv][H][Dh] each user's context
 *   uoff: host int[num_users+1], candidates of user u are [uoff[u], uoff[u+1])
 *   scale: logit scale
 *   Out : double [num_cand*Lq][H][Dh]
 *   cands: if non-NULL, only the listed candidates (ncands) are computed.
 * For each candidate and head the user's keys and values are copied out (the
 * broadcast the in-kernel method avoids); each query row q of the candidate
 * then takes s_j = scale * q . k_j over the copy, p_j = exp(s_j - max s) /
 * sum_i exp(s_i - max s), and o = sum_j p_j v_j.  Returns -1 on bad offsets,
 * -2 on a bad candidate index or allocation failure.
 */
int oracle_ikbo_attention(int num_users, int num_cand, int Lq, int H, int Dh, int Lkv,
                          const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                          const int *uoff, double scale, double *Out,
                          const int *cands, int ncands)
{
    if (uoff[0] != 0 || uoff[num_users] != num_cand) return -1;
    for (int u = 0; u < num_users; ++u)
        if (uoff[u + 1] < uoff[u]) return -1;
    long n = cands ? ncands : num_cand;
    int bad = 0;
    #pragma omp parallel
    {
        double *Kc = (double *)malloc(sizeof(double) * (size_t)Lkv * (size_t)Dh);
        double *Vc = (double *)malloc(sizeof(double) * (size_t)Lkv * (size_t)Dh);
        double *sc = (double *)malloc(sizeof(double) * (size_t)Lkv);
        if (!Kc || !Vc || !sc) bad = 1;
        #pragma omp for schedule(dynamic, 1) collapse(2)
        for (long i = 0; i < n; ++i)
            for (int h = 0; h < H; ++h) {
                int c = cands ? cands[i] : (int)i;
                if (!Kc || !Vc || !sc || c < 0 || c >= num_cand) { bad = 1; continue; }
                int u = user_of(num_users, uoff, c);
                /* The broadcast: this candidate's own copy of K[u], V[u] (head h). */
                for (int j = 0; j < Lkv; ++j)
                    for (int d = 0; d < Dh; ++d) {
                        long src = (((long)u * Lkv + j) * H + h) * Dh + d;
                        Kc[(long)j * Dh + d] = bf16_to_double(K[src]);
                        Vc[(long)j * Dh + d] = bf16_to_double(V[src]);
                    }
                for (int r = 0; r < Lq; ++r) {
                    long row = (long)c * Lq + r;
                    const uint16_t *q = Q + (row * H + h) * Dh;
                    double mx = -INFINITY;
                    for (int j = 0; j < Lkv; ++j) {
                        double acc = 0.0;
                        for (int d = 0; d < Dh; ++d)
                            acc += bf16_to_double(q[d]) * Kc[(long)j * Dh + d];
                        sc[j] = scale * acc;
                        if (sc[j] > mx) mx = sc[j];
                    }
                    double sum = 0.0;
                    for (int j = 0; j < Lkv; ++j) {
                        sc[j] = exp(sc[j] - mx);
                        sum += sc[j];
                    }
                    double *o = Out + (row * H + h) * Dh;
                    for (int d = 0; d < Dh; ++d) {
                        double acc = 0.0;
                        for (int j = 0; j < Lkv; ++j)
                            acc += sc[j] * Vc[(long)j * Dh + d];
                        o[d] = acc / sum;
                    }
                }
            }
        free(Kc);
        free(Vc);
        free(sc);
    }
    return bad ? -2 : 0;
}

/*
 * IKBO attention, second coding: per user u and head h, the rows of all of
 * u's candidates form one matrix Qs [nq][Dh]; S = scale * Qs K[u]^T, each row
 * of S is normalised (P = exp(S - rowmax) / rowsum), and O = P V[u].  Same
 * conventions as oracle_ikbo_attention (all candidates).
 */
int oracle_ikbo_attention_grouped(int num_users, int num_cand, int Lq, int H, int Dh, int Lkv,
                                  const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                  const int *uoff, double scale, double *Out)
{
    if (uoff[0] != 0 || uoff[num_users] != num_cand) return -1;
    for (int u = 0; u < num_users; ++u)
        if (uoff[u + 1] < uoff[u]) return -1;
    int bad = 0;
    #pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int u = 0; u < num_users; ++u)
        for (int h = 0; h < H; ++h) {
            long r0 = (long)uoff[u] * Lq, nq = (long)(uoff[u + 1] - uoff[u]) * Lq;
            if (nq == 0) continue;
            double *P = (double *)malloc(sizeof(double) * (size_t)nq * (size_t)Lkv);
            if (!P) { bad = 1; continue; }
            for (long r = 0; r < nq; ++r) {
                double mx = -INFINITY;
                for (int j = 0; j < Lkv; ++j) {
                    double acc = 0.0;
                    for (int d = 0; d < Dh; ++d)
                        acc += bf16_to_double(Q[((r0 + r) * H + h) * Dh + d]) *
                               bf16_to_double(K[(((long)u * Lkv + j) * H + h) * Dh + d]);
                    P[r * Lkv + j] = scale * acc;
                    if (P[r * Lkv + j] > mx) mx = P[r * Lkv + j];
                }
                double sum = 0.0;
                for (int j = 0; j < Lkv; ++j) {
                    P[r * Lkv + j] = exp(P[r * Lkv + j] - mx);
                    sum += P[r * Lkv + j];
                }
                for (int j = 0; j < Lkv; ++j) P[r * Lkv + j] /= sum;
            }
            for (long r = 0; r < nq; ++r)
                for (int d = 0; d < Dh; ++d) {
                    double acc = 0.0;
                    for (int j = 0; j < Lkv; ++j)
                        acc += P[r * Lkv + j] *
                               bf16_to_double(V[(((long)u * Lkv + j) * H + h) * Dh + d]);
                    Out[((r0 + r) * H + h) * Dh + d] = acc;
                }
            free(P);
        }
    return bad ? -2 : 0;
}
