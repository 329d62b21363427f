/*
 * Oracle for the anchor-attention forward of AnchorFormer (arXiv 2505.16463).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark may load this file's library; the GPU product never calls it.  It shares
 * no code with the CUDA path.
 *
 * What it computes (pith.science verdict on 2505.16463, "core_discovery",
 * "key_machinery" and the referee summary; the referee's Eq. 11/12):
 *   A  in R^{n x m}, A[i][j] = softmax over anchors j of  scale * q_i . u_j
 *        (the token->anchor attention matrix; rows sum to one)
 *   Delta = diag of the column sums of A   (the "anchor degrees")
 *   H  = A Delta^{-1} A^T V, evaluated as A (Delta^{-1} (A^T V)) so that no n x n matrix
 *        is formed (the reordering B^T V -> Delta^{-1}(B^T V) -> B(Delta^{-1} B^T V) of the
 *        referee summary; B there is the same matrix as A).
 *
 * Plain definition, double precision, single thread, no blocking or reordering.  Every
 * sum runs in ascending index order.  The softmax subtracts the row maximum first; that is
 * the same function mathematically and keeps exp() in range.
 *
 * Backward (the anchors are learned by gradient descent: "core_discovery"; the arXiv abstract,
 * where the anchors are weights of a trainable layer): for an upstream gradient dH of H, the gradients of
 * the loss with respect to Q, U and V follow by the chain rule through the same steps, taken
 * in reverse:
 *   dW' = A^T dH,  dW = Delta^{-1} dW',  dDelta_j = -sum_k dW'[j][k] W'[j][k] / Delta_j,
 *   G = dH W'^T + V dW^T + 1 dDelta^T   (dL/dA through H, through W and through Delta),
 *   dS[i][j] = A[i][j] (G[i][j] - sum_l A[i][l] G[i][l])   (the softmax's Jacobian),
 *   dQ = scale dS U,  dV = A dW,  dU = scale dS^T Q, summed over the batch entries that share
 *   the head's anchors.
 *
 * Readings where the pages are silent:
 *   - Delta_j == 0 (every A[i][j] underflowed): W'_j := 0.  Its contribution A[i][j] W'_j
 *     vanishes in the limit because every A[i][j] is 0.
 *   - Layout: Q, V, H are [B][heads][n][d] row-major; U is [heads][m][d] and is shared by
 *     every batch entry (one set of learnable anchors per head).
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>

/* Status codes: 0 ok, 1 bad argument, 2 out of memory. */

/* Steps 1-2: A[i][j] for one slice (softmax of scaled scores over the anchors). */
static void token_anchor_matrix(const double *Q, const double *U, long n, long m, long d,
                                double scale, double *A)
{
    for (long i = 0; i < n; ++i) {
        double *a = A + i * m;
        double mx = -INFINITY;
        for (long j = 0; j < m; ++j) {
            double s = 0.0;
            for (long k = 0; k < d; ++k) s += Q[i * d + k] * U[j * d + k];
            a[j] = scale * s;
            if (a[j] > mx) mx = a[j];
        }
        double z = 0.0;
        for (long j = 0; j < m; ++j) {
            a[j] = exp(a[j] - mx);
            z += a[j];
        }
        for (long j = 0; j < m; ++j) a[j] /= z;
    }
}

/* Step 3: Delta_j = sum_i A[i][j].  Steps 4-5: W'[j][k] = (sum_i A[i][j] V[i][k]) / Delta_j. */
static void anchor_summaries(const double *A, const double *V, long n, long m, long d,
                             double *delta, double *W, double *Wp)
{
    for (long j = 0; j < m; ++j) {
        double s = 0.0;
        for (long i = 0; i < n; ++i) s += A[i * m + j];
        delta[j] = s;
    }
    for (long j = 0; j < m; ++j) {
        for (long k = 0; k < d; ++k) {
            double s = 0.0;
            for (long i = 0; i < n; ++i) s += A[i * m + j] * V[i * d + k];
            W[j * d + k] = s;
            Wp[j * d + k] = delta[j] != 0.0 ? s / delta[j] : 0.0;
        }
    }
}

/* Step 6 for one token row: H[i][k] = sum_j A[i][j] W'[j][k]. */
static void apply_row(const double *a, const double *Wp, long m, long d, double *h)
{
    for (long k = 0; k < d; ++k) {
        double s = 0.0;
        for (long j = 0; j < m; ++j) s += a[j] * Wp[j * d + k];
        h[k] = s;
    }
}

static int bad_shape(long n, long m, long d) { return n < 0 || m < 1 || d < 1; }

/*
 * One (batch, head) slice with its intermediates.  Q, V: [n][d]; U: [m][d].
 * Outputs (each may be NULL): A [n][m], delta [m], W [m][d] (= A^T V), Wp [m][d]
 * (= Delta^{-1} A^T V), H [n][d].
 */
int oracle_anchor_slice(const double *Q, const double *U, const double *V, long n, long m,
                        long d, double scale, double *A_out, double *delta_out, double *W_out,
                        double *Wp_out, double *H)
{
    if (bad_shape(n, m, d)) return 1;
    double *A = malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)m);
    double *delta = malloc(sizeof(double) * (size_t)m);
    double *W = malloc(sizeof(double) * (size_t)m * (size_t)d);
    double *Wp = malloc(sizeof(double) * (size_t)m * (size_t)d);
    if (!A || !delta || !W || !Wp) {
        free(A); free(delta); free(W); free(Wp);
        return 2;
    }
    token_anchor_matrix(Q, U, n, m, d, scale, A);
    anchor_summaries(A, V, n, m, d, delta, W, Wp);
    if (H)
        for (long i = 0; i < n; ++i) apply_row(A + i * m, Wp, m, d, H + i * d);
    for (long i = 0; A_out && i < n * m; ++i) A_out[i] = A[i];
    for (long j = 0; delta_out && j < m; ++j) delta_out[j] = delta[j];
    for (long i = 0; W_out && i < m * d; ++i) W_out[i] = W[i];
    for (long i = 0; Wp_out && i < m * d; ++i) Wp_out[i] = Wp[i];
    free(A); free(delta); free(W); free(Wp);
    return 0;
}

/*
 * H rows of one slice for the listed token indices only (the anchor summaries still need
 * every token of the slice).  Hrows: [nrows][d].
 */
int oracle_anchor_slice_rows(const double *Q, const double *U, const double *V, long n, long m,
                             long d, double scale, const long *rows, long nrows, double *Hrows)
{
    if (bad_shape(n, m, d) || nrows < 0) return 1;
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= n) return 1;
    double *A = malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)m);
    double *delta = malloc(sizeof(double) * (size_t)m);
    double *W = malloc(sizeof(double) * (size_t)m * (size_t)d);
    double *Wp = malloc(sizeof(double) * (size_t)m * (size_t)d);
    if (!A || !delta || !W || !Wp) {
        free(A); free(delta); free(W); free(Wp);
        return 2;
    }
    token_anchor_matrix(Q, U, n, m, d, scale, A);
    anchor_summaries(A, V, n, m, d, delta, W, Wp);
    for (long r = 0; r < nrows; ++r) apply_row(A + rows[r] * m, Wp, m, d, Hrows + r * d);
    free(A); free(delta); free(W); free(Wp);
    return 0;
}

/*
 * Backward of one slice: dQ, dV [n][d] are written, dU [m][d] is ADDED to (the caller sums the
 * batch entries of a head).  dH: [n][d].  An anchor with Delta_j == 0 (the reading above: its
 * W'_j is 0) gets dW_j = 0 and dDelta_j = 0.
 */
int oracle_anchor_slice_backward(const double *Q, const double *U, const double *V, const double *dH,
                                 long n, long m, long d, double scale, double *dQ, double *dU, double *dV)
{
    if (bad_shape(n, m, d)) return 1;
    double *A = malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)m);
    double *delta = malloc(sizeof(double) * (size_t)m);
    double *W = malloc(sizeof(double) * (size_t)m * (size_t)d);
    double *Wp = malloc(sizeof(double) * (size_t)m * (size_t)d);
    double *dWp = malloc(sizeof(double) * (size_t)m * (size_t)d);
    double *dW = malloc(sizeof(double) * (size_t)m * (size_t)d);
    double *ddelta = malloc(sizeof(double) * (size_t)m);
    double *G = malloc(sizeof(double) * (size_t)m);
    if (!A || !delta || !W || !Wp || !dWp || !dW || !ddelta || !G) {
        free(A); free(delta); free(W); free(Wp); free(dWp); free(dW); free(ddelta); free(G);
        return 2;
    }
    /* the forward's intermediates */
    token_anchor_matrix(Q, U, n, m, d, scale, A);
    anchor_summaries(A, V, n, m, d, delta, W, Wp);
    /* dW' = A^T dH */
    for (long j = 0; j < m; ++j)
        for (long k = 0; k < d; ++k) {
            double s = 0.0;
            for (long i = 0; i < n; ++i) s += A[i * m + j] * dH[i * d + k];
            dWp[j * d + k] = s;
        }
    /* W' = W / Delta: dW = dW' / Delta and dDelta_j = -sum_k dW'_jk W_jk / Delta_j^2 */
    for (long j = 0; j < m; ++j) {
        double s = 0.0;
        for (long k = 0; k < d; ++k) {
            dW[j * d + k] = delta[j] != 0.0 ? dWp[j * d + k] / delta[j] : 0.0;
            s += dWp[j * d + k] * W[j * d + k];
        }
        ddelta[j] = delta[j] != 0.0 ? -s / (delta[j] * delta[j]) : 0.0;
    }
    for (long i = 0; i < n; ++i) {
        const double *a = A + i * m;
        /* G_j = dL/dA_ij: through H = A W', through W = A^T V and through Delta = A^T 1 */
        for (long j = 0; j < m; ++j) {
            double g = ddelta[j];
            for (long k = 0; k < d; ++k) g += dH[i * d + k] * Wp[j * d + k] + V[i * d + k] * dW[j * d + k];
            G[j] = g;
        }
        /* softmax: dS_ij = A_ij (G_j - sum_l A_il G_l) */
        double ag = 0.0;
        for (long j = 0; j < m; ++j) ag += a[j] * G[j];
        for (long j = 0; j < m; ++j) G[j] = a[j] * (G[j] - ag);  /* G now holds dS_i */
        /* S = scale Q U^T: dQ_i = scale sum_j dS_ij U_j; dU_j += scale dS_ij Q_i */
        for (long k = 0; k < d; ++k) {
            double s = 0.0;
            for (long j = 0; j < m; ++j) s += G[j] * U[j * d + k];
            dQ[i * d + k] = scale * s;
        }
        for (long j = 0; j < m; ++j)
            for (long k = 0; k < d; ++k) dU[j * d + k] += scale * G[j] * Q[i * d + k];
        /* W = A^T V: dV_i = sum_j A_ij dW_j */
        for (long k = 0; k < d; ++k) {
            double s = 0.0;
            for (long j = 0; j < m; ++j) s += a[j] * dW[j * d + k];
            dV[i * d + k] = s;
        }
    }
    free(A); free(delta); free(W); free(Wp); free(dWp); free(dW); free(ddelta); free(G);
    return 0;
}

/*
 * Whole backward.  Q, V, dH, dQ, dV: [B][heads][n][d]; U, dU: [heads][m][d] (dU is the sum
 * over the batch entries of each head; it is overwritten).
 */
int oracle_anchor_backward(const double *Q, const double *U, const double *V, const double *dH, double *dQ,
                           double *dU, double *dV, long B, long heads, long n, long m, long d, double scale)
{
    if (B < 0 || heads < 0 || bad_shape(n, m, d)) return 1;
    for (long i = 0; i < heads * m * d; ++i) dU[i] = 0.0;
    for (long b = 0; b < B; ++b) {
        for (long h = 0; h < heads; ++h) {
            size_t off = ((size_t)b * (size_t)heads + (size_t)h) * (size_t)n * (size_t)d;
            size_t uoff = (size_t)h * (size_t)m * (size_t)d;
            int rc = oracle_anchor_slice_backward(Q + off, U + uoff, V + off, dH + off, n, m, d, scale,
                                                  dQ + off, dU + uoff, dV + off);
            if (rc) return rc;
        }
    }
    return 0;
}

/*
 * Masked (causal) variant: the anchors' summaries seen by token i include only tokens j <= i,
 * so that no token draws on a later one (one of the pith.science verdict's inferences: A
 * can be masked against later tokens without giving up the O(mn) cost):
 *   Delta^(i)_l = sum_{j<=i} A[j][l],  W^(i)_l = sum_{j<=i} A[j][l] v_j,
 *   H[i] = sum_l A[i][l] W^(i)_l / Delta^(i)_l   (0 for an anchor with Delta^(i)_l = 0).
 * Each row of the masked S_t still sums to one.  One slice, prefixes in token order.
 */
int oracle_anchor_causal_slice(const double *Q, const double *U, const double *V, long n, long m, long d,
                               double scale, double *H)
{
    if (bad_shape(n, m, d)) return 1;
    double *A = malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)m);
    double *delta = calloc((size_t)m, sizeof(double));
    double *W = calloc((size_t)m * (size_t)d, sizeof(double));
    if (!A || !delta || !W) {
        free(A); free(delta); free(W);
        return 2;
    }
    token_anchor_matrix(Q, U, n, m, d, scale, A);
    for (long i = 0; i < n; ++i) {
        const double *a = A + i * m;
        for (long l = 0; l < m; ++l) {
            delta[l] += a[l];
            for (long k = 0; k < d; ++k) W[l * d + k] += a[l] * V[i * d + k];
        }
        for (long k = 0; k < d; ++k) {
            double s = 0.0;
            for (long l = 0; l < m; ++l)
                if (delta[l] != 0.0) s += a[l] * W[l * d + k] / delta[l];
            H[i * d + k] = s;
        }
    }
    free(A); free(delta); free(W);
    return 0;
}

int oracle_anchor_causal(const double *Q, const double *U, const double *V, double *H, long B, long heads, long n,
                         long m, long d, double scale)
{
    if (B < 0 || heads < 0 || bad_shape(n, m, d)) return 1;
    for (long b = 0; b < B; ++b)
        for (long h = 0; h < heads; ++h) {
            size_t off = ((size_t)b * (size_t)heads + (size_t)h) * (size_t)n * (size_t)d;
            const size_t uoff = (size_t)h * (size_t)m * (size_t)d;
            int rc = oracle_anchor_causal_slice(Q + off, U + uoff, V + off, n, m, d, scale, H + off);
            if (rc) return rc;
        }
    return 0;
}

/*
 * Full softmax attention, the quadratic construction the anchors approximate (the skeptic's
 * concrete test in the pith.science verdict: compare H with softmax(Q K^T / sqrt(d)) V when
 * the anchors come from rows of K).  One slice: Q, V [n][d], K [nk][d]:
 *   H[i] = sum_j softmax over j of (scale q_i . k_j) v_j    (max subtracted first).
 */
int oracle_full_attention_slice(const double *Q, const double *K, const double *V, long n, long nk, long d,
                                double scale, double *H)
{
    if (n < 0 || nk < 1 || d < 1) return 1;
    double *p = malloc(sizeof(double) * (size_t)nk);
    if (!p) return 2;
    for (long i = 0; i < n; ++i) {
        double mx = -INFINITY;
        for (long j = 0; j < nk; ++j) {
            double s = 0.0;
            for (long k = 0; k < d; ++k) s += Q[i * d + k] * K[j * d + k];
            p[j] = scale * s;
            if (p[j] > mx) mx = p[j];
        }
        double z = 0.0;
        for (long j = 0; j < nk; ++j) {
            p[j] = exp(p[j] - mx);
            z += p[j];
        }
        for (long k = 0; k < d; ++k) {
            double s = 0.0;
            for (long j = 0; j < nk; ++j) s += p[j] * V[j * d + k];
            H[i * d + k] = s / z;
        }
    }
    free(p);
    return 0;
}

/* Full attention of every slice: Q, V, H [B][heads][n][d]; K [heads][n][d], one key matrix
 * per head shared by the batch (as the anchors are). */
int oracle_full_attention(const double *Q, const double *K, const double *V, double *H, long B, long heads,
                          long n, long d, double scale)
{
    if (B < 0 || heads < 0 || n < 1 || d < 1) return 1;
    for (long b = 0; b < B; ++b)
        for (long h = 0; h < heads; ++h) {
            size_t off = ((size_t)b * (size_t)heads + (size_t)h) * (size_t)n * (size_t)d;
            int rc = oracle_full_attention_slice(Q + off, K + (size_t)h * (size_t)n * (size_t)d, V + off, n, n, d,
                                                 scale, H + off);
            if (rc) return rc;
        }
    return 0;
}

/*
 * Whole forward.  Q, V, H: [B][heads][n][d]; U: [heads][m][d] shared across the batch.
 * Each (b, h) slice is independent (the construction is per attention head).
 */
int oracle_anchor_forward(const double *Q, const double *U, const double *V, double *H, long B,
                          long heads, long n, long m, long d, double scale)
{
    if (B < 0 || heads < 0 || bad_shape(n, m, d)) return 1;
    for (long b = 0; b < B; ++b) {
        for (long h = 0; h < heads; ++h) {
            size_t off = ((size_t)b * (size_t)heads + (size_t)h) * (size_t)n * (size_t)d;
            int rc = oracle_anchor_slice(Q + off, U + (size_t)h * (size_t)m * (size_t)d, V + off,
                                         n, m, d, scale, NULL, NULL, NULL, NULL, H + off);
            if (rc) return rc;
        }
    }
    return 0;
}

/*
 * Block front end: in an AnchorFormer layer the anchor attention takes the place of a ViT
 * block's self-attention, so its per-head queries and values are linear projections of the
 * token embeddings X (no bias: the pages give none):
 *   Q[i][k] = sum_c X[i][c] Wq[k][c],   V[i][k] = sum_c X[i][c] Wv[k][c],
 * followed by the forward above on (Q, U, V).  One slice: X [n][dm] (the batch entry's
 * tokens), Wq, Wv [d][dm] (the head's rows of the projection matrices), U [m][d], H [n][d].
 */
int oracle_anchor_block_slice(const double *X, const double *Wq, const double *Wv, const double *U, long n,
                              long m, long d, long dm, double scale, double *H)
{
    if (bad_shape(n, m, d) || dm < 1) return 1;
    double *Qp = malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)d);
    double *Vp = malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)d);
    if (!Qp || !Vp) {
        free(Qp); free(Vp);
        return 2;
    }
    for (long i = 0; i < n; ++i)
        for (long k = 0; k < d; ++k) {
            double sq = 0.0, sv = 0.0;
            for (long c = 0; c < dm; ++c) {
                sq += X[i * dm + c] * Wq[k * dm + c];
                sv += X[i * dm + c] * Wv[k * dm + c];
            }
            Qp[i * d + k] = sq;
            Vp[i * d + k] = sv;
        }
    int rc = oracle_anchor_slice(Qp, U, Vp, n, m, d, scale, NULL, NULL, NULL, NULL, H);
    free(Qp); free(Vp);
    return rc;
}

/* Every slice: X [B][n][dm]; Wq, Wv [heads][d][dm]; U [heads][m][d]; H [B][heads][n][d]. */
int oracle_anchor_block(const double *X, const double *Wq, const double *Wv, const double *U, double *H, long B,
                        long heads, long n, long m, long d, long dm, double scale)
{
    if (B < 0 || heads < 0 || bad_shape(n, m, d) || dm < 1) return 1;
    for (long b = 0; b < B; ++b)
        for (long h = 0; h < heads; ++h) {
            const size_t xoff = (size_t)b * (size_t)n * (size_t)dm;
            const size_t woff = (size_t)h * (size_t)d * (size_t)dm;
            const size_t hoff = ((size_t)b * (size_t)heads + (size_t)h) * (size_t)n * (size_t)d;
            const size_t uoff = (size_t)h * (size_t)m * (size_t)d;
            int rc = oracle_anchor_block_slice(X + xoff, Wq + woff, Wv + woff, U + uoff, n, m, d, dm, scale,
                                               H + hoff);
            if (rc) return rc;
        }
    return 0;
}
