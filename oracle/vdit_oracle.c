/*
 * vdit oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the frame-window + reference-frame
 * block-sparse attention computes. Only the tests, the package smoke check and
 * the benchmark's CPU-baseline leg may load it; the library never does. It
 * shares no code, header, table or helper with the CUDA sources.
 *
 * Source: "HeyGen x Google Cloud: Bringing Avatar IV to TPUs"
 *   - "Deleting the Mask" (+ Fig. 3): a query attends to the frames within W of
 *     its own frame and to one fixed reference frame; blocks whose size divides
 *     the frame's token span are entirely live or entirely dead.
 *   - "Unchaining the Softmax" (+ Fig. 4): mean-centred keys, the
 *     Cauchy-Schwarz row bound |q|*max|k - mean|, per-head eligibility.
 *
 * Everything here is the plain definition, written out with an explicit
 * token-level mask and an ordinary max-subtracted softmax:
 *   J(i)  = { j : |f(i) - f(j)| <= W } U { j : f(j) = ref },  f(x) = floor(x / T)
 *   s_ij  = scale * q_i . k_j
 *   O_i   = sum_{j in J(i)} exp(s_ij - m_i) v_j / sum_{j in J(i)} exp(s_ij - m_i),
 *           m_i = max_{j in J(i)} s_ij
 *   LSE_i = m_i + ln sum_{j in J(i)} exp(s_ij - m_i)
 *
 * Tensor arguments are [B, H, N, D] with the last dimension contiguous and
 * element strides (sb, sh, sn) for the first three. Element type: 0 = bf16
 * bit patterns (uint16), 1 = float64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double elem(const void *p, int64_t idx, int dtype)
{
    if (dtype == 1)
        return ((const double *)p)[idx];
    uint32_t u = ((uint32_t)((const uint16_t *)p)[idx]) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int vo_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* The token-level mask ("Deleting the Mask"): query token i sees key token j
 * when their frames are at most W apart, or when j lies in the reference
 * frame. ref < 0 means no reference frame. */
int vo_mask(int64_t T, int32_t W, int32_t ref, int64_t i, int64_t j)
{
    int64_t fi = i / T, fj = j / T;
    int64_t d = fi > fj ? fi - fj : fj - fi;
    if (d <= (int64_t)W)
        return 1;
    if (ref >= 0 && fj == (int64_t)ref)
        return 1;
    return 0;
}

/* Block census for square bs x bs blocks over an N x N token grid (last block
 * ragged when bs does not divide N). Every token pair of every block is tested
 * through vo_mask. Counts blocks that are fully live, partially live and dead. */
void vo_block_census(int32_t F, int32_t T, int32_t W, int32_t ref, int32_t bs,
                     int64_t *full, int64_t *partial, int64_t *dead)
{
    int64_t N = (int64_t)F * T, nb = (N + bs - 1) / bs;
    int64_t nf = 0, np = 0, nd = 0;
#pragma omp parallel for schedule(dynamic) reduction(+ : nf, np, nd)
    for (int64_t qb = 0; qb < nb; ++qb) {
        int64_t i0 = qb * bs, i1 = i0 + bs < N ? i0 + bs : N;
        for (int64_t kb = 0; kb < nb; ++kb) {
            int64_t j0 = kb * bs, j1 = j0 + bs < N ? j0 + bs : N;
            int64_t live = 0;
            for (int64_t i = i0; i < i1; ++i)
                for (int64_t j = j0; j < j1; ++j)
                    live += vo_mask(T, W, ref, i, j);
            int64_t area = (i1 - i0) * (j1 - j0);
            if (live == area)
                nf++;
            else if (live == 0)
                nd++;
            else
                np++;
        }
    }
    *full = nf;
    *partial = np;
    *dead = nd;
}

/* Block schedule (Fig. 3): CSR over bs x bs blocks of the live (query block,
 * key block) pairs, key blocks ascending; for every query frame its maximal
 * ascending runs of live key tokens [lo, hi) (at most two are stored: runs[4f
 * .. 4f+3] = lo0, hi0, lo1, hi1, with (0, 0) for an absent second run); and
 * the total count of live token pairs.
 * Returns 0 on success, -1 if some block is partially live, -2 if col_idx
 * capacity is too small, -3 if some frame has more than two runs.
 * row_ptr must hold ceil(N/bs)+1 entries. */
int vo_schedule(int32_t F, int32_t T, int32_t W, int32_t ref, int32_t bs,
                int32_t *row_ptr, int32_t *col_idx, int64_t cap, int64_t *nnz_out,
                int32_t *runs, int64_t *live_pairs_out)
{
    int64_t N = (int64_t)F * T, nb = (N + bs - 1) / bs;
    int64_t *rowlen = (int64_t *)calloc((size_t)nb, sizeof(int64_t));
    uint8_t *live = (uint8_t *)calloc((size_t)(nb * nb), 1);
    int bad = 0;
    int64_t pairs = 0;
#pragma omp parallel for schedule(dynamic) reduction(+ : pairs) reduction(| : bad)
    for (int64_t qb = 0; qb < nb; ++qb) {
        int64_t i0 = qb * bs, i1 = i0 + bs < N ? i0 + bs : N;
        for (int64_t kb = 0; kb < nb; ++kb) {
            int64_t j0 = kb * bs, j1 = j0 + bs < N ? j0 + bs : N;
            int64_t cnt = 0;
            for (int64_t i = i0; i < i1; ++i)
                for (int64_t j = j0; j < j1; ++j)
                    cnt += vo_mask(T, W, ref, i, j);
            pairs += cnt;
            if (cnt == (i1 - i0) * (j1 - j0)) {
                live[qb * nb + kb] = 1;
                rowlen[qb]++;
            } else if (cnt != 0) {
                bad = 1;
            }
        }
    }
    int rc = 0;
    if (bad)
        rc = -1;
    int64_t nnz = 0;
    row_ptr[0] = 0;
    for (int64_t qb = 0; qb < nb; ++qb) {
        for (int64_t kb = 0; kb < nb; ++kb) {
            if (!live[qb * nb + kb])
                continue;
            if (nnz < cap)
                col_idx[nnz] = (int32_t)kb;
            nnz++;
        }
        row_ptr[qb + 1] = (int32_t)nnz;
    }
    if (rc == 0 && nnz > cap)
        rc = -2;
    *nnz_out = nnz;
    *live_pairs_out = pairs;

    for (int32_t f = 0; f < F; ++f) {
        int64_t i = (int64_t)f * T; /* the frame's first query token */
        int nr = 0;
        int64_t lo[3] = {0, 0, 0}, hi[3] = {0, 0, 0};
        int64_t j = 0;
        while (j < N) {
            if (!vo_mask(T, W, ref, i, j)) {
                j++;
                continue;
            }
            int64_t a = j;
            while (j < N && vo_mask(T, W, ref, i, j))
                j++;
            if (nr < 3) {
                lo[nr] = a;
                hi[nr] = j;
            }
            nr++;
        }
        if (nr > 2 && rc == 0)
            rc = -3;
        runs[4 * f + 0] = (int32_t)lo[0];
        runs[4 * f + 1] = (int32_t)hi[0];
        runs[4 * f + 2] = nr > 1 ? (int32_t)lo[1] : 0;
        runs[4 * f + 3] = nr > 1 ? (int32_t)hi[1] : 0;
    }
    free(rowlen);
    free(live);
    return rc;
}

/* Per-head key statistics ("Unchaining the Softmax"):
 *   c_h    = (1/N) sum_j k_j                     (the key mean)
 *   R_h    = max_j |k_j - c_h|_2                 (largest centred key norm)
 *   Qmax_h = max_i |q_i|_2
 *   G_h    = 2 * scale * Qmax_h * R_h            (widest possible gap between a
 *                                                row's bound and its true max)
 *   elig_h = G_h <= tau, decided in fp32 (the kernel's precision).
 * c is [B*H*D], the rest [B*H]. */
void vo_key_stats(const void *q, const void *k, int dtype, int32_t B, int32_t H, int64_t N,
                  int32_t D, const int64_t *qs, const int64_t *ks, double scale, double tau,
                  double *c, double *R, double *qmax, double *G, uint8_t *elig)
{
#pragma omp parallel for schedule(dynamic)
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        int64_t b = bh / H, h = bh % H;
        int64_t kb = b * ks[0] + h * ks[1], qb = b * qs[0] + h * qs[1];
        double *cc = c + bh * D;
        for (int32_t d = 0; d < D; ++d)
            cc[d] = 0.0;
        for (int64_t j = 0; j < N; ++j)
            for (int32_t d = 0; d < D; ++d)
                cc[d] += elem(k, kb + j * ks[2] + d, dtype);
        for (int32_t d = 0; d < D; ++d)
            cc[d] /= (double)N;
        double r2 = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int32_t d = 0; d < D; ++d) {
                double x = elem(k, kb + j * ks[2] + d, dtype) - cc[d];
                acc += x * x;
            }
            if (acc > r2)
                r2 = acc;
        }
        double q2 = 0.0;
        for (int64_t i = 0; i < N; ++i) {
            double acc = 0.0;
            for (int32_t d = 0; d < D; ++d) {
                double x = elem(q, qb + i * qs[2] + d, dtype);
                acc += x * x;
            }
            if (acc > q2)
                q2 = acc;
        }
        R[bh] = sqrt(r2);
        qmax[bh] = sqrt(q2);
        G[bh] = 2.0 * scale * qmax[bh] * R[bh];
        elig[bh] = ((float)G[bh] <= (float)tau) ? 1 : 0;
    }
}

/* Row bound ("Unchaining the Softmax"): for query row i of head h,
 *   m_i = scale * (q_i . c_h + |q_i|_2 * R_h).
 * By Cauchy-Schwarz, scale*q_i.k_j = scale*q_i.(k_j - c_h) + scale*q_i.c_h
 * <= m_i for every key j of the head, whatever slice of keys the row sees.
 * rows[r] = (b*H + h)*N + i. */
void vo_row_bounds(const void *q, int dtype, int32_t H, int64_t N, int32_t D, const int64_t *qs,
                   const double *c, const double *R, double scale, int64_t nrows,
                   const int64_t *rows, double *m)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t bh = rows[r] / N, i = rows[r] % N;
        int64_t b = bh / H, h = bh % H;
        int64_t qo = b * qs[0] + h * qs[1] + i * qs[2];
        double dot = 0.0, nn = 0.0;
        for (int32_t d = 0; d < D; ++d) {
            double x = elem(q, qo + d, dtype);
            dot += x * c[bh * D + d];
            nn += x * x;
        }
        m[r] = scale * (dot + sqrt(nn) * R[bh]);
    }
}

/* Masked attention for a list of query rows, plain fp64:
 * every key j of the head is tested through vo_mask; the softmax subtracts the
 * true row max. Also returns each row's max logit (mx, may be NULL).
 * rows[r] = (b*H + h)*N + i; o is [nrows, D]; lse and mx are [nrows]. */
void vo_attention_rows(const void *q, const void *k, const void *v, int dtype, int32_t H,
                       int64_t N, int32_t D, const int64_t *qs, const int64_t *ks,
                       const int64_t *vs, int32_t T, int32_t W, int32_t ref, double scale,
                       int64_t nrows, const int64_t *rows, double *o, double *lse, double *mx)
{
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)N * sizeof(double));
        double *qrow = (double *)malloc((size_t)D * sizeof(double));
#pragma omp for schedule(dynamic)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t bh = rows[r] / N, i = rows[r] % N;
            int64_t b = bh / H, h = bh % H;
            int64_t qo = b * qs[0] + h * qs[1] + i * qs[2];
            int64_t kb = b * ks[0] + h * ks[1], vb = b * vs[0] + h * vs[1];
            for (int32_t d = 0; d < D; ++d)
                qrow[d] = elem(q, qo + d, dtype);
            double m = -INFINITY;
            for (int64_t j = 0; j < N; ++j) {
                if (!vo_mask(T, W, ref, i, j))
                    continue;
                double acc = 0.0;
                for (int32_t d = 0; d < D; ++d)
                    acc += qrow[d] * elem(k, kb + j * ks[2] + d, dtype);
                s[j] = scale * acc;
                if (s[j] > m)
                    m = s[j];
            }
            double l = 0.0;
            double *out = o + r * D;
            for (int32_t d = 0; d < D; ++d)
                out[d] = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                if (!vo_mask(T, W, ref, i, j))
                    continue;
                double p = exp(s[j] - m);
                l += p;
                for (int32_t d = 0; d < D; ++d)
                    out[d] += p * elem(v, vb + j * vs[2] + d, dtype);
            }
            for (int32_t d = 0; d < D; ++d)
                out[d] /= l;
            lse[r] = m + log(l);
            if (mx)
                mx[r] = m;
        }
        free(s);
        free(qrow);
    }
}

/* Per-query-frame key statistics ("Unchaining the Softmax": the bound stays
 * valid under windowed masks, where rows of different frames attend to
 * different subsets of the keys). For query frame f of head (b, h), with c the
 * key mean over all N keys of the head and J(f) = { j : mask(f*T, j) } the
 * keys that frame's queries see (tested token by token through vo_mask):
 *   R_f    = max_{j in J(f)} |k_j - c|_2
 *   Qmax_f = max_{i in frame f} |q_i|_2
 *   G_f    = 2 * scale * Qmax_f * R_f,  elig_f = G_f <= tau (decided in fp32)
 * Outputs are [B*H*F]. */
void vo_frame_stats(const void *q, const void *k, int dtype, int32_t B, int32_t H, int64_t N,
                    int32_t D, const int64_t *qs, const int64_t *ks, int32_t T, int32_t W,
                    int32_t ref, double scale, double tau, double *Rf, double *qmaxf, double *Gf,
                    uint8_t *eligf)
{
    const int64_t F = N / T;
#pragma omp parallel for schedule(dynamic)
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        int64_t b = bh / H, h = bh % H;
        int64_t kb = b * ks[0] + h * ks[1], qb = b * qs[0] + h * qs[1];
        double *c = (double *)calloc((size_t)D, sizeof(double));
        double *kn = (double *)malloc((size_t)N * sizeof(double));
        for (int64_t j = 0; j < N; ++j)
            for (int32_t d = 0; d < D; ++d)
                c[d] += elem(k, kb + j * ks[2] + d, dtype);
        for (int32_t d = 0; d < D; ++d)
            c[d] /= (double)N;
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int32_t d = 0; d < D; ++d) {
                double x = elem(k, kb + j * ks[2] + d, dtype) - c[d];
                acc += x * x;
            }
            kn[j] = sqrt(acc);
        }
        for (int64_t f = 0; f < F; ++f) {
            double r = 0.0, qm = 0.0;
            for (int64_t j = 0; j < N; ++j)
                if (vo_mask(T, W, ref, f * T, j) && kn[j] > r)
                    r = kn[j];
            for (int64_t i = f * T; i < (f + 1) * T; ++i) {
                double acc = 0.0;
                for (int32_t d = 0; d < D; ++d) {
                    double x = elem(q, qb + i * qs[2] + d, dtype);
                    acc += x * x;
                }
                if (sqrt(acc) > qm)
                    qm = sqrt(acc);
            }
            int64_t o = bh * F + f;
            Rf[o] = r;
            qmaxf[o] = qm;
            Gf[o] = 2.0 * scale * qm * r;
            eligf[o] = ((float)Gf[o] <= (float)tau) ? 1 : 0;
        }
        free(c);
        free(kn);
    }
}

/* Row bound with the per-query-frame R: m_i = scale * (q_i . c_h + |q_i| R_{f(i)}),
 * Rf indexed [bh * F + i / T]. */
void vo_row_bounds_frames(const void *q, int dtype, int32_t H, int64_t N, int32_t D,
                          const int64_t *qs, const double *c, const double *Rf, int32_t T,
                          double scale, int64_t nrows, const int64_t *rows, double *m)
{
    const int64_t F = N / T;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t bh = rows[r] / N, i = rows[r] % N;
        int64_t b = bh / H, h = bh % H;
        int64_t qo = b * qs[0] + h * qs[1] + i * qs[2];
        double dot = 0.0, nn = 0.0;
        for (int32_t d = 0; d < D; ++d) {
            double x = elem(q, qo + d, dtype);
            dot += x * c[bh * D + d];
            nn += x * x;
        }
        m[r] = scale * (dot + sqrt(nn) * Rf[bh * F + i / T]);
    }
}

/* Fused pre-attention chain ("Layout Is the ABI", Fig. 5: normalisation,
 * projections, rotary embeddings and head packing, written straight into the
 * layout attention reads). For each listed token row (b, n) of x [B, N, C]:
 *   y_c   = x_c * gamma_c / sqrt(mean_c x_c^2 + eps)                  (RMSNorm)
 *   z_o   = sum_c y_c * w[o, c],  o in [0, 3*H*D)                      (QKV projection,
 *           w is [3*H*D, C]: rows 0..HD-1 give q, then k, then v, head-major)
 *   rotary embedding on q and k of every head, position n, pairs (i, i + D/2):
 *           t_i = base^(-2i/D), a = n * t_i,
 *           (u, w) -> (u cos a - w sin a, u sin a + w cos a)
 * Outputs are [nrows, H, D] each (q, k, v). x and w element type: 0 = bf16, 1 = f64.
 * x strides (elements) for (b, n); the channel dimension is contiguous.
 * rows[r] = b * N + n. */
void vo_qkv_prologue(const void *x, const void *w, int dtype, int32_t B, int64_t N, int32_t C,
                     const int64_t *xs, const double *gamma, int32_t H, int32_t D, double eps,
                     double base, int64_t nrows, const int64_t *rows, double *q_out,
                     double *k_out, double *v_out)
{
    const int64_t HD = (int64_t)H * D;
    (void)B;
#pragma omp parallel
    {
        double *y = (double *)malloc((size_t)C * sizeof(double));
        double *z = (double *)malloc((size_t)(3 * HD) * sizeof(double));
#pragma omp for schedule(dynamic)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t b = rows[r] / N, n = rows[r] % N;
            const int64_t xo = b * xs[0] + n * xs[1];
            double ss = 0.0;
            for (int32_t c = 0; c < C; ++c) {
                double v = elem(x, xo + c, dtype);
                ss += v * v;
            }
            const double inv = 1.0 / sqrt(ss / (double)C + eps);
            for (int32_t c = 0; c < C; ++c)
                y[c] = elem(x, xo + c, dtype) * inv * gamma[c];
            for (int64_t o = 0; o < 3 * HD; ++o) {
                double acc = 0.0;
                for (int32_t c = 0; c < C; ++c)
                    acc += y[c] * elem(w, o * C + c, dtype);
                z[o] = acc;
            }
            for (int part = 0; part < 2; ++part) {           /* q, k: rotary embedding */
                for (int32_t h = 0; h < H; ++h) {
                    double *zh = z + part * HD + (int64_t)h * D;
                    for (int32_t i = 0; i < D / 2; ++i) {
                        const double t = pow(base, -2.0 * i / (double)D);
                        const double a = (double)n * t;
                        const double u = zh[i], wv = zh[i + D / 2];
                        zh[i] = u * cos(a) - wv * sin(a);
                        zh[i + D / 2] = u * sin(a) + wv * cos(a);
                    }
                }
            }
            for (int64_t o = 0; o < HD; ++o) {
                q_out[r * HD + o] = z[o];
                k_out[r * HD + o] = z[HD + o];
                v_out[r * HD + o] = z[2 * HD + o];
            }
        }
        free(y);
        free(z);
    }
}
