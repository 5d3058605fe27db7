/*
 * flare_oracle.c -- plain fp64 CPU oracle for the FLARE / FLARE++ token mixer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file; only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header or constant with the CUDA
 * library and is deliberately slow: every quantity is formed from its
 * definition, in double precision, without blocking, fusion or reordering.
 *
 * Source: "FLARE++: Low-rank attention with dynamic attention routing",
 * appendix on context parallelism (the arXiv 2608.11519 HTML page). Its display
 * equations were lost in extraction; the forms below are the plain readings of
 * the surrounding prose, written out:
 *
 *   encoder, eq. 18 ("global encoder"): for latent row m of head h, batch b,
 *       S_mn = s * <Q_m, K_n>           over the valid (unpadded) tokens n,
 *       L_m  = log sum_n exp(S_mn)       (row log-normaliser, natural log),
 *       Z_m  = sum_n exp(S_mn - L_m) V_n (softmax(S) V),         s = D^-1/2.
 *     A row with no valid key returns L = -inf and Z = 0 (empty-row rule of
 *     the cross-rank log-sum-exp paragraph).
 *   per-shard encoder (the paragraph before eq. 23): the same definition over
 *     one shard's tokens, giving O_r and L_r.
 *   merge, eq. 23 and the cross-rank log-sum-exp paragraph:
 *       L_max = max_r L_r, a = sum_r exp(L_r - L_max),
 *       U = sum_r exp(L_r - L_max) O_r, Z = U / a, L = L_max + log a.
 *   decode (FLARE decode paragraph): each token's own key is its query against
 *     the replicated latents: T_nm = s * <K_n, Q_m>, Y_n = sum_m softmax_m(T_n) Z_m.
 *   decode backward (chain rule of the decode; the pages name the decoder's
 *     contribution to the gradients of the latents, the formula is stripped):
 *       A_nm = softmax_m(T_n), g_nm = <dY_n, Z_m>, r_n = sum_m A_nm g_nm,
 *       dT_nm = A_nm (g_nm - r_n), dZ_m = sum_n A_nm dY_n,
 *       dK_n = s sum_m dT_nm Q_m, dQ_m = s sum_n dT_nm K_n.
 *   encoder backward (the backward paragraphs): with the global Z, L,
 *       P_mn = exp(S_mn - L_m), c_m = <dZ_m, Z_m>,
 *       dV_n = sum_m P_mn dZ_m, dS_mn = P_mn (<dZ_m, V_n> - c_m),
 *       dK_n = s sum_m dS_mn Q_m, dQ_m = s sum_n dS_mn K_n.
 *
 * Layouts (row-major): token tensors [B, N, H, D]; latent tensors [B, H, M, D]
 * (a query with batch stride 0 is one [H, M, D] tensor shared by all b);
 * row statistics [B, H, M]; masks uint8 [B, N], 1 = valid, NULL = all valid.
 *
 * Input element codes: 0 = double, 1 = float, 2 = bfloat16 bit pattern
 * (uint16). Converting any of them to double is exact, so the oracle always
 * computes on the very values a device run consumed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { T_F64 = 0, T_F32 = 1, T_BF16 = 2 };

static double load(const void *p, int t, size_t i) {
    if (t == T_F64) return ((const double *)p)[i];
    if (t == T_F32) return (double)((const float *)p)[i];
    /* bfloat16: the upper half of an IEEE binary32 */
    uint32_t bits = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static size_t tok_index(long b, long n, long h, long N, long H, long D) {
    return (((size_t)b * N + n) * H + h) * D;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Encoder over the token range [n0, n1) (the whole sequence for eq. 18, one
 * shard for the per-shard O_r, L_r). rows: optional list of flat row indices
 * (b*H + h)*M + m to evaluate (NULL = every row); rows not listed are left
 * untouched in Z [B,H,M,D] and L [B,H,M].
 */
void oracle_encode(int B, int H, int M, int N, int D, double scale, long q_bstride,
                   const void *Q, int qt, const void *K, const void *V, int kvt,
                   const uint8_t *mask, long n0, long n1,
                   const int64_t *rows, long nrows, double *Z, double *L) {
    long total = rows ? nrows : (long)B * H * M;
#pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < total; ++i) {
        long row = rows ? (long)rows[i] : i;
        long m = row % M, h = (row / M) % H, b = row / ((long)M * H);
        size_t qoff = (size_t)b * q_bstride + ((size_t)h * M + m) * D;
        long len = n1 - n0;
        double *S = (double *)malloc(sizeof(double) * (len > 0 ? len : 1));
        double mx = -INFINITY;
        long nvalid = 0;
        for (long n = n0; n < n1; ++n) {
            if (mask && !mask[(size_t)b * N + n]) continue;
            size_t ko = tok_index(b, n, h, N, H, D);
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += load(Q, qt, qoff + d) * load(K, kvt, ko + d);
            S[n - n0] = scale * dot;
            if (S[n - n0] > mx) mx = S[n - n0];
            ++nvalid;
        }
        double *z = Z + (size_t)row * D;
        for (int d = 0; d < D; ++d) z[d] = 0.0;
        if (nvalid == 0) {            /* empty row: L = -inf, Z = 0 */
            L[row] = -INFINITY;
            free(S);
            continue;
        }
        double sum = 0.0;
        for (long n = n0; n < n1; ++n) {
            if (mask && !mask[(size_t)b * N + n]) continue;
            sum += exp(S[n - n0] - mx);
        }
        double lse = mx + log(sum);
        L[row] = lse;
        for (long n = n0; n < n1; ++n) {
            if (mask && !mask[(size_t)b * N + n]) continue;
            double p = exp(S[n - n0] - lse);
            size_t vo = tok_index(b, n, h, N, H, D);
            for (int d = 0; d < D; ++d) z[d] += p * load(V, kvt, vo + d);
        }
        free(S);
    }
}

/*
 * Elementwise log-sum-exp merge of R per-shard results (eq. 23 with the
 * cross-rank maximum): O_r [R, rows, D], L_r [R, rows] -> Z [rows, D], L [rows].
 * Shards whose L_r is -inf carry no mass; if every shard is empty for a row
 * the row is empty: L = -inf, Z = 0.
 */
void oracle_lse_merge(int R, long rows, int D, const double *O_r, const double *L_r,
                      double *Z, double *L) {
#pragma omp parallel for schedule(static)
    for (long i = 0; i < rows; ++i) {
        double lmax = -INFINITY;
        for (int r = 0; r < R; ++r)
            if (L_r[(size_t)r * rows + i] > lmax) lmax = L_r[(size_t)r * rows + i];
        double *z = Z + (size_t)i * D;
        for (int d = 0; d < D; ++d) z[d] = 0.0;
        if (lmax == -INFINITY) {
            L[i] = -INFINITY;
            continue;
        }
        double a = 0.0;
        for (int r = 0; r < R; ++r) {
            double lr = L_r[(size_t)r * rows + i];
            if (lr == -INFINITY) continue;
            double w = exp(lr - lmax);
            a += w;
            const double *o = O_r + ((size_t)r * rows + i) * D;
            for (int d = 0; d < D; ++d) z[d] += w * o[d];   /* U */
        }
        for (int d = 0; d < D; ++d) z[d] /= a;             /* Z = U / a */
        L[i] = lmax + log(a);
    }
}

/*
 * Local decode for the listed token slots (flat b*N + n; NULL = every slot).
 * Q: query latents (batch stride q_bstride), Z [B,H,M,D] double, K token keys.
 * Y: [ntok, H, D] in list order (or [B,N,H,D] when tokens is NULL).
 * The decode has no mask: its softmax runs over the M latents, never empty.
 */
void oracle_decode(int B, int H, int M, int N, int D, double scale, long q_bstride,
                   const void *Q, int qt, const double *Z, const void *K, int kt,
                   const int64_t *tokens, long ntok, double *Y) {
    long total = tokens ? ntok : (long)B * N;
#pragma omp parallel for schedule(dynamic, 64)
    for (long i = 0; i < total; ++i) {
        long slot = tokens ? (long)tokens[i] : i;
        long b = slot / N, n = slot % N;
        double *T = (double *)malloc(sizeof(double) * M);
        for (int h = 0; h < H; ++h) {
            size_t ko = tok_index(b, n, h, N, H, D);
            double mx = -INFINITY;
            for (int m = 0; m < M; ++m) {
                size_t qoff = (size_t)b * q_bstride + ((size_t)h * M + m) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += load(K, kt, ko + d) * load(Q, qt, qoff + d);
                T[m] = scale * dot;
                if (T[m] > mx) mx = T[m];
            }
            double sum = 0.0;
            for (int m = 0; m < M; ++m) sum += exp(T[m] - mx);
            double *y = Y + ((size_t)i * H + h) * D;
            for (int d = 0; d < D; ++d) y[d] = 0.0;
            for (int m = 0; m < M; ++m) {
                double p = exp(T[m] - mx) / sum;
                const double *z = Z + (((size_t)b * H + h) * M + m) * D;
                for (int d = 0; d < D; ++d) y[d] += p * z[d];
            }
        }
        free(T);
    }
}

/*
 * Encoder backward with the global forward statistics (Z, L [B,H,M]) and the
 * summed output gradient dZ [B,H,M,D] (all double). Outputs: dQ [B,H,M,D]
 * (one per batch element, also for a replicated query), dK and dV [B,N,H,D].
 * Masked tokens get dK = dV = 0; rows with L = -inf carry P = 0.
 */
void oracle_encode_bwd(int B, int H, int M, int N, int D, double scale, long q_bstride,
                       const void *Q, int qt, const void *K, const void *V, int kvt,
                       const uint8_t *mask, const double *Z, const double *L,
                       const double *dZ, double *dQ, double *dK, double *dV) {
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        long b = bh / H, h = bh % H;
        const double *Lb = L + (size_t)bh * M;
        double *c = (double *)malloc(sizeof(double) * M);
        double *Qd = (double *)malloc(sizeof(double) * (size_t)M * D);
        for (int m = 0; m < M; ++m) {
            const double *dz = dZ + ((size_t)bh * M + m) * D;
            const double *z = Z + ((size_t)bh * M + m) * D;
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += dz[d] * z[d];
            c[m] = acc;
            size_t qoff = (size_t)b * q_bstride + ((size_t)h * M + m) * D;
            for (int d = 0; d < D; ++d) Qd[(size_t)m * D + d] = load(Q, qt, qoff + d);
        }
        double *dq = dQ + (size_t)bh * M * D;
        for (size_t j = 0; j < (size_t)M * D; ++j) dq[j] = 0.0;
        for (long n = 0; n < N; ++n) {
            size_t to = tok_index(b, n, h, N, H, D);
            double *dk = dK + to, *dv = dV + to;
            for (int d = 0; d < D; ++d) { dk[d] = 0.0; dv[d] = 0.0; }
            if (mask && !mask[(size_t)b * N + n]) continue;
            for (int m = 0; m < M; ++m) {
                if (Lb[m] == -INFINITY) continue;
                const double *q = Qd + (size_t)m * D;
                const double *dz = dZ + ((size_t)bh * M + m) * D;
                double sdot = 0.0, dp = 0.0;
                for (int d = 0; d < D; ++d) {
                    sdot += q[d] * load(K, kvt, to + d);
                    dp += dz[d] * load(V, kvt, to + d);
                }
                double P = exp(scale * sdot - Lb[m]);
                double dS = P * (dp - c[m]);
                for (int d = 0; d < D; ++d) {
                    dv[d] += P * dz[d];
                    dk[d] += scale * dS * q[d];
                    dq[(size_t)m * D + d] += scale * dS * load(K, kvt, to + d);
                }
            }
        }
        free(c);
        free(Qd);
    }
}

/*
 * Decode backward: the gradients of the local decode for an output gradient
 * dY [B,N,H,D] (element code yt). Z [B,H,M,D] double. Outputs (double):
 * dQ [B,H,M,D] (one per batch element, also for a replicated query),
 * dZ [B,H,M,D] and dK [B,N,H,D]. Every token slot contributes (the decode has
 * no mask).
 */
void oracle_decode_bwd(int B, int H, int M, int N, int D, double scale, long q_bstride,
                       const void *Q, int qt, const double *Z, const void *K, int kt,
                       const void *dY, int yt, double *dQ, double *dZ, double *dK) {
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        long b = bh / H, h = bh % H;
        double *Qd = (double *)malloc(sizeof(double) * (size_t)M * D);
        double *A = (double *)malloc(sizeof(double) * M);
        double *g = (double *)malloc(sizeof(double) * M);
        for (int m = 0; m < M; ++m) {
            size_t qoff = (size_t)b * q_bstride + ((size_t)h * M + m) * D;
            for (int d = 0; d < D; ++d) Qd[(size_t)m * D + d] = load(Q, qt, qoff + d);
        }
        const double *Zb = Z + (size_t)bh * M * D;
        double *dq = dQ + (size_t)bh * M * D, *dz = dZ + (size_t)bh * M * D;
        for (size_t j = 0; j < (size_t)M * D; ++j) dq[j] = dz[j] = 0.0;
        for (long n = 0; n < N; ++n) {
            size_t to = tok_index(b, n, h, N, H, D);
            /* A = softmax over the latents of T_nm = s <K_n, Q_m> */
            double mx = -INFINITY;
            for (int m = 0; m < M; ++m) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += load(K, kt, to + d) * Qd[(size_t)m * D + d];
                A[m] = scale * dot;
                if (A[m] > mx) mx = A[m];
            }
            double sum = 0.0;
            for (int m = 0; m < M; ++m) sum += exp(A[m] - mx);
            double r = 0.0;
            for (int m = 0; m < M; ++m) {
                A[m] = exp(A[m] - mx) / sum;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += load(dY, yt, to + d) * Zb[(size_t)m * D + d];
                g[m] = dot;
                r += A[m] * g[m];
            }
            double *dk = dK + to;
            for (int d = 0; d < D; ++d) dk[d] = 0.0;
            for (int m = 0; m < M; ++m) {
                double dT = A[m] * (g[m] - r);
                for (int d = 0; d < D; ++d) {
                    dk[d] += scale * dT * Qd[(size_t)m * D + d];
                    dq[(size_t)m * D + d] += scale * dT * load(K, kt, to + d);
                    dz[(size_t)m * D + d] += A[m] * load(dY, yt, to + d);
                }
            }
        }
        free(Qd);
        free(A);
        free(g);
    }
}
