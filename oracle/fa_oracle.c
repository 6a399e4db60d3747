/*
 * fa_oracle.c -- fp64 CPU oracle for exact scaled dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  The product library never links, calls or
 * imports this file; only the test-suite, the package smoke check and the
 * CPU-baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * It is the plain definition written out, slowly, with every intermediate
 * materialised in fp64:
 *
 *   forward   S = scale * Q K^T, masked entries set to -inf,
 *             P = row-softmax(S) by the three-pass safe softmax,
 *             O = P V,  LSE_i = m_i + ln(l_i)
 *   backward  with the loss L = sum(O o dO):
 *             dV = P^T dO,  dP = dO V^T,  D_i = sum_k dO_ik O_ik,
 *             dS = P o (dP - D 1^T),  dQ = scale dS K,  dK = scale dS^T Q
 *
 * Sources (page title, section):
 *  - "FlashAttention: Mathematical Foundations, IO-Aware Tiling, Online
 *    Softmax, and Recomputation Dynamics", section "The GPU Memory Hierarchy
 *    and the Attention Memory Wall": O = softmax(Q K^T / sqrt(d)) V with Q, K,
 *    V of shape (N, d), computed as scores -> probabilities -> output.
 *  - same page, section "Online Softmax: The Mathematical Core": the safe
 *    softmax m = max_j x_j, l = sum_j exp(x_j - m), y_i = exp(x_i - m) / l,
 *    taken in three passes over the row.
 *  - same page, section "Backward Pass and Activation Recomputation": the
 *    backward needs O and the per-row statistics m, l.  Here the two are
 *    stored folded into one number, LSE = m + ln l.
 *  - The backward formulas are the chain rule through O = P V and the row
 *    softmax (the softmax Jacobian diag(p) - p p^T applied to dP); the pages
 *    state no backward equations.  S = scale * Q K^T, so dQ and dK carry the
 *    factor `scale`.
 *  - Masks.  The pages state none for causal or key padding; the readings
 *    here are: causal keeps key j for query i iff j <= i (square, top-left
 *    aligned); key padding keeps key j iff j < key_len[b] and masks no query;
 *    block sparsity ("Attention" chapter, block-sparse paragraph: blocks a
 *    block mask zeroes are skipped) keeps (i, j) iff
 *    block_mask[(i / mask_block) * nb + j / mask_block] != 0, nb =
 *    ceil(N / mask_block), one mask shared by every (b, h).
 *  - A query row with no visible key has O = 0, LSE = -inf, a zero P row and
 *    contributes no gradient (the pages are silent; this is the reading).
 *
 * Decode shapes (oracle_decode): Nq query rows against Nk cached keys per
 * (b, h).  Key j is visible to query i iff j < kv_len[b] (all Nk when kv_len
 * is NULL) and, with the causal flag, j <= kv_len[b] - Nq + i: the queries
 * are the last Nq positions of the sequence (bottom-right alignment; equal
 * to the square causal mask when Nq = Nk = kv_len).  The pages describe the
 * decode kernel only as the same IO-aware framing applied to one new token
 * per step ("Attention" chapter, decoding paragraph); this is the plain
 * definition of that step.
 *
 * Layout: every tensor is contiguous [B, H, N, d] (d fastest); LSE is
 * [B, H, N]; P (optional) is [B, H, N, N].  All functions return 0 on
 * success and a negative number on a bad argument or allocation failure.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX(bh, i, N) ((int64_t)(bh) * (int64_t)(N) + (int64_t)(i))

/* Is key j visible to query i of batch b? (the element mask) */
static int visible(int b, int i, int j, int N, int causal, const int32_t *key_len,
                   const uint8_t *block_mask, int mask_block)
{
    if (i < 0 || j < 0 || i >= N || j >= N) return 0;
    if (causal && j > i) return 0;
    if (key_len && j >= key_len[b]) return 0;
    if (block_mask) {
        int nb = (N + mask_block - 1) / mask_block;
        if (block_mask[(int64_t)(i / mask_block) * nb + j / mask_block] == 0) return 0;
    }
    return 1;
}

static int check_args(int B, int H, int N, int d, const uint8_t *block_mask, int mask_block)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0) return -1;
    if (block_mask && mask_block <= 0) return -1;
    return 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * One score row: s[j] = scale * <q_i, k_j>, or -inf where masked.
 */
static void score_row(const double *Qh, const double *Kh, int b, int i, int N, int d,
                      double scale, int causal, const int32_t *key_len,
                      const uint8_t *block_mask, int mask_block, double *s)
{
    const double *q = Qh + (int64_t)i * d;
    for (int j = 0; j < N; j++) {
        if (!visible(b, i, j, N, causal, key_len, block_mask, mask_block)) {
            s[j] = -INFINITY;
            continue;
        }
        const double *k = Kh + (int64_t)j * d;
        double acc = 0.0;
        for (int t = 0; t < d; t++) acc += q[t] * k[t];
        s[j] = scale * acc;
    }
}

/*
 * Three-pass safe softmax of one row, in place: s becomes p.
 * Pass 1 the maximum, pass 2 the normaliser, pass 3 the division.
 * Returns LSE = m + ln(l), or -inf for a row with no visible entry.
 */
static double safe_softmax_row(double *s, int N)
{
    double m = -INFINITY;
    for (int j = 0; j < N; j++)
        if (s[j] > m) m = s[j];
    if (m == -INFINITY) {
        for (int j = 0; j < N; j++) s[j] = 0.0;
        return -INFINITY;
    }
    double l = 0.0;
    for (int j = 0; j < N; j++) l += exp(s[j] - m);
    for (int j = 0; j < N; j++) s[j] = exp(s[j] - m) / l;
    return m + log(l);
}

/*
 * Forward for one (b, h): materialise S (N x N), then P, then O = P V.
 */
static int fwd_head(const double *Qh, const double *Kh, const double *Vh, int b, int N, int d,
                    double scale, int causal, const int32_t *key_len,
                    const uint8_t *block_mask, int mask_block,
                    double *Oh, double *LSEh, double *Ph /* N*N, caller-owned scratch */)
{
    /* S = scale * Q K^T (masked) */
#pragma omp parallel for schedule(static)
    for (int i = 0; i < N; i++)
        score_row(Qh, Kh, b, i, N, d, scale, causal, key_len, block_mask, mask_block,
                  Ph + (int64_t)i * N);
    /* P = softmax(S), row by row; LSE from the same passes */
#pragma omp parallel for schedule(static)
    for (int i = 0; i < N; i++)
        LSEh[i] = safe_softmax_row(Ph + (int64_t)i * N, N);
    /* O = P V */
#pragma omp parallel for schedule(static)
    for (int i = 0; i < N; i++) {
        double *o = Oh + (int64_t)i * d;
        for (int t = 0; t < d; t++) o[t] = 0.0;
        const double *p = Ph + (int64_t)i * N;
        for (int j = 0; j < N; j++) {
            if (p[j] == 0.0) continue;
            const double *v = Vh + (int64_t)j * d;
            for (int t = 0; t < d; t++) o[t] += p[j] * v[t];
        }
    }
    return 0;
}

int oracle_fwd(const double *Q, const double *K, const double *V, int B, int H, int N, int d,
               double scale, int causal, const int32_t *key_len, const uint8_t *block_mask,
               int mask_block, double *O, double *LSE, double *P_out)
{
    if (check_args(B, H, N, d, block_mask, mask_block)) return -1;
    if (N == 0 || B == 0 || H == 0) return 0;
    double *P = P_out ? NULL : (double *)malloc(sizeof(double) * (size_t)N * (size_t)N);
    if (!P_out && !P) return -2;
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++) {
            int64_t bh = (int64_t)b * H + h;
            double *Ph = P_out ? P_out + bh * (int64_t)N * N : P;
            fwd_head(Q + IDX(bh, 0, N) * d, K + IDX(bh, 0, N) * d, V + IDX(bh, 0, N) * d, b, N, d,
                     scale, causal, key_len, block_mask, mask_block, O + IDX(bh, 0, N) * d,
                     LSE + IDX(bh, 0, N), Ph);
        }
    free(P);
    return 0;
}

/*
 * Forward and backward together.  O and LSE are written too (they are the
 * forward's outputs and D needs O).
 */
int oracle_bwd(const double *Q, const double *K, const double *V, const double *dO, int B, int H,
               int N, int d, double scale, int causal, const int32_t *key_len,
               const uint8_t *block_mask, int mask_block, double *O, double *LSE, double *dQ,
               double *dK, double *dV)
{
    if (check_args(B, H, N, d, block_mask, mask_block)) return -1;
    if (N == 0 || B == 0 || H == 0) return 0;
    size_t nn = (size_t)N * (size_t)N;
    double *P = (double *)malloc(sizeof(double) * nn);
    double *dS = (double *)malloc(sizeof(double) * nn);
    double *Dv = (double *)malloc(sizeof(double) * (size_t)N);
    if (!P || !dS || !Dv) {
        free(P); free(dS); free(Dv);
        return -2;
    }
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++) {
            int64_t bh = (int64_t)b * H + h;
            const double *Qh = Q + IDX(bh, 0, N) * d, *Kh = K + IDX(bh, 0, N) * d;
            const double *Vh = V + IDX(bh, 0, N) * d, *dOh = dO + IDX(bh, 0, N) * d;
            double *Oh = O + IDX(bh, 0, N) * d, *LSEh = LSE + IDX(bh, 0, N);
            double *dQh = dQ + IDX(bh, 0, N) * d, *dKh = dK + IDX(bh, 0, N) * d;
            double *dVh = dV + IDX(bh, 0, N) * d;
            fwd_head(Qh, Kh, Vh, b, N, d, scale, causal, key_len, block_mask, mask_block, Oh, LSEh, P);

            /* D_i = sum_k dO_ik O_ik */
#pragma omp parallel for schedule(static)
            for (int i = 0; i < N; i++) {
                double acc = 0.0;
                for (int t = 0; t < d; t++) acc += dOh[(int64_t)i * d + t] * Oh[(int64_t)i * d + t];
                Dv[i] = acc;
            }
            /* dP_ij = <dO_i, V_j>;  dS_ij = P_ij (dP_ij - D_i) */
#pragma omp parallel for schedule(static)
            for (int i = 0; i < N; i++) {
                for (int j = 0; j < N; j++) {
                    double p = P[(int64_t)i * N + j];
                    double dp = 0.0;
                    for (int t = 0; t < d; t++) dp += dOh[(int64_t)i * d + t] * Vh[(int64_t)j * d + t];
                    dS[(int64_t)i * N + j] = p * (dp - Dv[i]);
                }
            }
            /* dQ = scale * dS K */
#pragma omp parallel for schedule(static)
            for (int i = 0; i < N; i++) {
                for (int t = 0; t < d; t++) {
                    double acc = 0.0;
                    for (int j = 0; j < N; j++) acc += dS[(int64_t)i * N + j] * Kh[(int64_t)j * d + t];
                    dQh[(int64_t)i * d + t] = scale * acc;
                }
            }
            /* dK = scale * dS^T Q;  dV = P^T dO */
#pragma omp parallel for schedule(static)
            for (int j = 0; j < N; j++) {
                for (int t = 0; t < d; t++) {
                    double ak = 0.0, av = 0.0;
                    for (int i = 0; i < N; i++) {
                        ak += dS[(int64_t)i * N + j] * Qh[(int64_t)i * d + t];
                        av += P[(int64_t)i * N + j] * dOh[(int64_t)i * d + t];
                    }
                    dKh[(int64_t)j * d + t] = scale * ak;
                    dVh[(int64_t)j * d + t] = av;
                }
            }
        }
    free(P);
    free(dS);
    free(Dv);
    return 0;
}

/*
 * The same definition restricted to chosen query rows, for checks at sizes
 * where the full N x N matrices do not fit: rows[r] = (b * H + h) * N + i.
 * Writes O, LSE and (when dO and dQ_rows are given) dQ for those rows.
 * Each row needs only its own score row: D_i = <dO_i, O_i> uses the row's
 * own O, and dQ_i = scale * sum_j P_ij (dP_ij - D_i) K_j.
 */
int oracle_query_rows(const double *Q, const double *K, const double *V, const double *dO, int B,
                      int H, int N, int d, double scale, int causal, const int32_t *key_len,
                      const uint8_t *block_mask, int mask_block, int n_rows, const int64_t *rows,
                      double *O_rows, double *LSE_rows, double *dQ_rows)
{
    if (check_args(B, H, N, d, block_mask, mask_block)) return -1;
    for (int r = 0; r < n_rows; r++)
        if (rows[r] < 0 || rows[r] >= (int64_t)B * H * N) return -1;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int r = 0; r < n_rows; r++) {
        int64_t bh = rows[r] / N;
        int i = (int)(rows[r] % N);
        int b = (int)(bh / H);
        double *p = (double *)malloc(sizeof(double) * (size_t)N);
        if (!p) { err |= 1; continue; }
        const double *Kh = K + IDX(bh, 0, N) * d, *Vh = V + IDX(bh, 0, N) * d;
        score_row(Q + IDX(bh, 0, N) * d, Kh, b, i, N, d, scale, causal, key_len, block_mask,
                  mask_block, p);
        LSE_rows[r] = safe_softmax_row(p, N);
        double *o = O_rows + (int64_t)r * d;
        for (int t = 0; t < d; t++) o[t] = 0.0;
        for (int j = 0; j < N; j++)
            if (p[j] != 0.0)
                for (int t = 0; t < d; t++) o[t] += p[j] * Vh[(int64_t)j * d + t];
        if (dO && dQ_rows) {
            const double *g = dO + IDX(bh, i, N) * d;
            double Di = 0.0;
            for (int t = 0; t < d; t++) Di += g[t] * o[t];
            double *dq = dQ_rows + (int64_t)r * d;
            for (int t = 0; t < d; t++) dq[t] = 0.0;
            for (int j = 0; j < N; j++) {
                if (p[j] == 0.0) continue;
                double dp = 0.0;
                for (int t = 0; t < d; t++) dp += g[t] * Vh[(int64_t)j * d + t];
                double ds = p[j] * (dp - Di);
                for (int t = 0; t < d; t++) dq[t] += ds * Kh[(int64_t)j * d + t];
            }
            for (int t = 0; t < d; t++) dq[t] *= scale;
        }
        free(p);
    }
    return err ? -2 : 0;
}

/*
 * dK and dV restricted to chosen key rows: keys[r] = (b * H + h) * N + j.
 * dV_j = sum_i P_ij dO_i and dK_j = scale * sum_i dS_ij Q_i need, for every
 * query row i of the head, that row's full softmax and D_i, so every row of
 * each head that owns a chosen key is recomputed here.
 */
int oracle_key_rows(const double *Q, const double *K, const double *V, const double *dO, int B,
                    int H, int N, int d, double scale, int causal, const int32_t *key_len,
                    const uint8_t *block_mask, int mask_block, int n_keys, const int64_t *keys,
                    double *dK_rows, double *dV_rows)
{
    if (check_args(B, H, N, d, block_mask, mask_block)) return -1;
    for (int r = 0; r < n_keys; r++)
        if (keys[r] < 0 || keys[r] >= (int64_t)B * H * N) return -1;
    memset(dK_rows, 0, sizeof(double) * (size_t)n_keys * d);
    memset(dV_rows, 0, sizeof(double) * (size_t)n_keys * d);
    int err = 0;
    for (int64_t bh = 0; bh < (int64_t)B * H; bh++) {
        int nsel = 0;
        for (int r = 0; r < n_keys; r++)
            if (keys[r] / N == bh) nsel++;
        if (!nsel) continue;
        int b = (int)(bh / H);
        const double *Qh = Q + IDX(bh, 0, N) * d, *Kh = K + IDX(bh, 0, N) * d;
        const double *Vh = V + IDX(bh, 0, N) * d, *dOh = dO + IDX(bh, 0, N) * d;
#pragma omp parallel reduction(| : err)
        {
            double *p = (double *)malloc(sizeof(double) * (size_t)N);
            double *o = (double *)malloc(sizeof(double) * (size_t)d);
            double *accK = (double *)calloc((size_t)n_keys * d, sizeof(double));
            double *accV = (double *)calloc((size_t)n_keys * d, sizeof(double));
            int ok = p && o && accK && accV;
            if (!ok) err |= 1;
            {
#pragma omp for schedule(static)
                for (int i = 0; i < N; i++) {
                    if (!ok) continue;
                    score_row(Qh, Kh, b, i, N, d, scale, causal, key_len, block_mask, mask_block, p);
                    safe_softmax_row(p, N);
                    for (int t = 0; t < d; t++) o[t] = 0.0;
                    for (int j = 0; j < N; j++)
                        if (p[j] != 0.0)
                            for (int t = 0; t < d; t++) o[t] += p[j] * Vh[(int64_t)j * d + t];
                    const double *g = dOh + (int64_t)i * d;
                    double Di = 0.0;
                    for (int t = 0; t < d; t++) Di += g[t] * o[t];
                    for (int r = 0; r < n_keys; r++) {
                        if (keys[r] / N != bh) continue;
                        int j = (int)(keys[r] % N);
                        if (p[j] == 0.0) continue;
                        double dp = 0.0;
                        for (int t = 0; t < d; t++) dp += g[t] * Vh[(int64_t)j * d + t];
                        double ds = p[j] * (dp - Di);
                        for (int t = 0; t < d; t++) {
                            accV[(int64_t)r * d + t] += p[j] * g[t];
                            accK[(int64_t)r * d + t] += ds * Qh[(int64_t)i * d + t];
                        }
                    }
                }
#pragma omp critical
                if (ok) {
                    for (int r = 0; r < n_keys; r++) {
                        if (keys[r] / N != bh) continue;
                        for (int t = 0; t < d; t++) {
                            dK_rows[(int64_t)r * d + t] += scale * accK[(int64_t)r * d + t];
                            dV_rows[(int64_t)r * d + t] += accV[(int64_t)r * d + t];
                        }
                    }
                }
            }
            free(p); free(o); free(accK); free(accV);
        }
    }
    return err ? -2 : 0;
}

/*
 * Tile plan by brute force over elements: for every batch b and every
 * (query tile, key tile) pair of tile_q x tile_k elements, look at each
 * element (i, j) with i < N inside the tile and key index j anywhere in the
 * tile's key range (j >= N counts as masked), and classify the tile
 *   0 = skip     (every element masked),
 *   1 = full     (no element masked),
 *   2 = partial  (some masked, some not).
 * plan is [B][ceil(N/tile_q)][ceil(N/tile_k)].
 */
int oracle_tile_plan(int B, int N, int causal, const int32_t *key_len, const uint8_t *block_mask,
                     int mask_block, int tile_q, int tile_k, uint8_t *plan)
{
    if (B < 0 || N < 0 || tile_q <= 0 || tile_k <= 0) return -1;
    if (block_mask && mask_block <= 0) return -1;
    int Tq = (N + tile_q - 1) / tile_q, Tk = (N + tile_k - 1) / tile_k;
    for (int b = 0; b < B; b++)
        for (int ti = 0; ti < Tq; ti++)
            for (int tj = 0; tj < Tk; tj++) {
                int64_t n_vis = 0, n_all = 0;
                for (int i = ti * tile_q; i < (ti + 1) * tile_q && i < N; i++)
                    for (int j = tj * tile_k; j < (tj + 1) * tile_k; j++) {
                        n_all++;
                        n_vis += visible(b, i, j, N, causal, key_len, block_mask, mask_block);
                    }
                uint8_t c = n_vis == 0 ? 0 : (n_vis == n_all ? 1 : 2);
                plan[((int64_t)b * Tq + ti) * Tk + tj] = c;
            }
    return 0;
}

/*
 * Decode: Q [B, H, Nq, d], K and V [B, H, Nk, d] -> O [B, H, Nq, d] and
 * LSE [B, H, Nq].  Each query row: masked scores, three-pass safe softmax,
 * O = P V, LSE = m + ln l.
 */
int oracle_decode(const double *Q, const double *K, const double *V, int B, int H, int Nq, int Nk,
                  int d, double scale, int causal, const int32_t *kv_len, double *O, double *LSE)
{
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0) return -1;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t r = 0; r < (int64_t)B * H * Nq; r++) {
        const int64_t bh = r / Nq;
        const int i = (int)(r % Nq);
        const int b = (int)(bh / H);
        const int len = kv_len ? kv_len[b] : Nk;
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        if (!s) { err |= 1; continue; }
        const double *q = Q + r * d;
        const double *Kh = K + bh * (int64_t)Nk * d, *Vh = V + bh * (int64_t)Nk * d;
        for (int j = 0; j < Nk; j++) {
            int vis = j < len;
            if (causal && j > len - Nq + i) vis = 0;
            if (!vis) { s[j] = -INFINITY; continue; }
            double acc = 0.0;
            for (int t = 0; t < d; t++) acc += q[t] * Kh[(int64_t)j * d + t];
            s[j] = scale * acc;
        }
        LSE[r] = safe_softmax_row(s, Nk);
        double *o = O + r * d;
        for (int t = 0; t < d; t++) o[t] = 0.0;
        for (int j = 0; j < Nk; j++)
            if (s[j] != 0.0)
                for (int t = 0; t < d; t++) o[t] += s[j] * Vh[(int64_t)j * d + t];
        free(s);
    }
    return err ? -2 : 0;
}

/*
 * Backward of decode-shaped attention: per (b, h), Nq query rows that are the
 * last Nq positions of a sequence of Nk keys.  Key j is visible to query i
 * iff j < Nk and, with the causal flag, j <= i + (Nk - Nq) (bottom-right
 * alignment, as in oracle_decode without kv_len; Nq = Nk gives the square
 * causal mask).  This is one sequence of a ragged batch ("Attention"
 * chapter, serving paragraph: ragged layouts); the pages give no backward
 * formulas, so they are the chain rule of the file header:
 *   S = scale Q K^T (masked), P = row-softmax(S) (three passes), O = P V,
 *   D_i = sum_t dO_it O_it,  dS = P o (dO V^T - D 1^T),
 *   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
 * Q, dO, O, dQ: [BH][Nq][d]; K, V, dK, dV: [BH][Nk][d]; LSE: [BH][Nq].
 * A query row with no visible key has O = 0, LSE = -inf and a zero gradient.
 */
int oracle_bwd_rect(const double *Q, const double *K, const double *V, const double *dO, int BH, int Nq,
                    int Nk, int d, double scale, int causal, double *O, double *LSE, double *dQ, double *dK,
                    double *dV)
{
    if (BH < 0 || Nq < 0 || Nk < 0 || d <= 0) return -1;
    const size_t nqk = (size_t)(Nq > 0 ? Nq : 1) * (size_t)(Nk > 0 ? Nk : 1);
    double *P = (double *)malloc(sizeof(double) * nqk);
    double *dS = (double *)malloc(sizeof(double) * nqk);
    double *Dv = (double *)malloc(sizeof(double) * (size_t)(Nq > 0 ? Nq : 1));
    if (!P || !dS || !Dv) {
        free(P); free(dS); free(Dv);
        return -2;
    }
    for (int64_t bh = 0; bh < BH; bh++) {
        const double *Qh = Q + bh * (int64_t)Nq * d, *dOh = dO + bh * (int64_t)Nq * d;
        const double *Kh = K + bh * (int64_t)Nk * d, *Vh = V + bh * (int64_t)Nk * d;
        double *Oh = O + bh * (int64_t)Nq * d, *LSEh = LSE + bh * (int64_t)Nq;
        double *dQh = dQ + bh * (int64_t)Nq * d;
        double *dKh = dK + bh * (int64_t)Nk * d, *dVh = dV + bh * (int64_t)Nk * d;
        /* S = scale Q K^T, masked; P = softmax(S) row by row; O = P V */
#pragma omp parallel for schedule(static)
        for (int i = 0; i < Nq; i++) {
            double *p = P + (int64_t)i * Nk;
            for (int j = 0; j < Nk; j++) {
                if (causal && j > i + (Nk - Nq)) {
                    p[j] = -INFINITY;
                    continue;
                }
                double acc = 0.0;
                for (int t = 0; t < d; t++) acc += Qh[(int64_t)i * d + t] * Kh[(int64_t)j * d + t];
                p[j] = scale * acc;
            }
            LSEh[i] = safe_softmax_row(p, Nk);
            double *o = Oh + (int64_t)i * d;
            for (int t = 0; t < d; t++) o[t] = 0.0;
            for (int j = 0; j < Nk; j++)
                if (p[j] != 0.0)
                    for (int t = 0; t < d; t++) o[t] += p[j] * Vh[(int64_t)j * d + t];
            /* D_i = sum_t dO_it O_it */
            double Di = 0.0;
            for (int t = 0; t < d; t++) Di += dOh[(int64_t)i * d + t] * o[t];
            Dv[i] = Di;
        }
        /* dS_ij = P_ij (<dO_i, V_j> - D_i) */
#pragma omp parallel for schedule(static)
        for (int i = 0; i < Nq; i++)
            for (int j = 0; j < Nk; j++) {
                double dp = 0.0;
                for (int t = 0; t < d; t++) dp += dOh[(int64_t)i * d + t] * Vh[(int64_t)j * d + t];
                dS[(int64_t)i * Nk + j] = P[(int64_t)i * Nk + j] * (dp - Dv[i]);
            }
        /* dQ = scale dS K */
#pragma omp parallel for schedule(static)
        for (int i = 0; i < Nq; i++)
            for (int t = 0; t < d; t++) {
                double acc = 0.0;
                for (int j = 0; j < Nk; j++) acc += dS[(int64_t)i * Nk + j] * Kh[(int64_t)j * d + t];
                dQh[(int64_t)i * d + t] = scale * acc;
            }
        /* dK = scale dS^T Q;  dV = P^T dO */
#pragma omp parallel for schedule(static)
        for (int j = 0; j < Nk; j++)
            for (int t = 0; t < d; t++) {
                double ak = 0.0, av = 0.0;
                for (int i = 0; i < Nq; i++) {
                    ak += dS[(int64_t)i * Nk + j] * Qh[(int64_t)i * d + t];
                    av += P[(int64_t)i * Nk + j] * dOh[(int64_t)i * d + t];
                }
                dKh[(int64_t)j * d + t] = scale * ak;
                dVh[(int64_t)j * d + t] = av;
            }
    }
    free(P);
    free(dS);
    free(Dv);
    return 0;
}

/*
 * FP8 block quantisation.  "FlashAttention: Mathematical Foundations ...",
 * section "Architectural Evolution" (FlashAttention-3 paragraph): the FP8
 * matmuls are block-quantised with dynamic scaling; "Attention" chapter
 * (learn-kernels.com), FlashAttention-3 paragraph: block quantisation on the
 * hardware FP8 format.  The pages fix no format details.  Readings:
 *   - element format e4m3 without infinities: 1 sign bit, 4 exponent bits
 *     with bias 7, 3 mantissa bits; exponent field 0 holds the subnormals
 *     m/8 * 2^-6; the largest finite magnitude is 1.75 * 2^8 = 448 and the
 *     pattern S.1111.111 is NaN.  Conversion rounds to nearest, ties to
 *     even, keeps the sign of values that round to zero and saturates
 *     magnitudes above 448 to 448;
 *   - a block is 128 consecutive rows (tokens) x all d columns of one
 *     (b, h); "dynamic" scaling takes its scale from the data: amax / 448 in
 *     fp32.  An all-zero block has no range to scale: its scale is 0 and its
 *     codes are 0 (so it never inflates a maximum taken over block scales);
 *   - code = e4m3(x / scale), the division in fp32; the codes stand for the
 *     values code * scale.
 */
unsigned char oracle_e4m3_encode(float xf)
{
    if (isnan(xf)) return 0x7F;
    const unsigned char sign = signbit(xf) ? 0x80 : 0x00;
    double a = fabs((double)xf);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7E;
    /* binade of a: a = f * 2^E, f in [0.5, 1), so 2^(E-1) <= a < 2^E;
     * below 2^-6 every value shares the subnormal spacing 2^-9 */
    int E;
    frexp(a, &E);
    int e = E - 1;
    if (e < -6) e = -6;
    const double ulp = ldexp(1.0, e - 3);          /* 3 mantissa bits */
    const double q = a / ulp;                       /* exact: ulp is a power of two */
    double r = floor(q);
    const double frac = q - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    double v = r * ulp;
    if (v > 448.0) v = 448.0;
    if (v == 0.0) return sign;
    /* encode the representable magnitude v */
    int E2;
    frexp(v, &E2);
    const int field = (E2 - 1) + 7;
    unsigned mag;
    if (field <= 0) {
        mag = (unsigned)(v / ldexp(1.0, -9));       /* subnormal: m * 2^-9 */
    } else {
        const double m = (v / ldexp(1.0, E2 - 1) - 1.0) * 8.0;
        mag = ((unsigned)field << 3) | (unsigned)m;
    }
    return (unsigned char)(sign | mag);
}

double oracle_e4m3_decode(unsigned char c)
{
    const int field = (c >> 3) & 0xF, m = c & 7;
    if (field == 15 && m == 7) return NAN;
    const double mag = field == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, field - 7);
    return (c & 0x80) ? -mag : mag;
}

/*
 * X: fp32 [BH][N][d] (the bf16 inputs, exactly).  Writes the codes to
 * codes ([BH][N][d], or with transpose [BH][d][Np], Np = ceil(N / 16) * 16,
 * code 0 in the columns N..Np-1) and one scale per (bh, 128-row block) to
 * scales [BH][ceil(N / 128)].
 */
int oracle_quantize_fp8(const float *X, int BH, int N, int d, int transpose, unsigned char *codes,
                        float *scales)
{
    if (BH < 0 || N < 0 || d <= 0) return -1;
    const int T = (N + 127) / 128;
    const int Np = (N + 15) / 16 * 16;
    if (transpose)
        memset(codes, 0, (size_t)BH * d * Np);
#pragma omp parallel for schedule(static)
    for (int64_t blk = 0; blk < (int64_t)BH * T; blk++) {
        const int64_t bh = blk / T;
        const int t = (int)(blk % T);
        const int r0 = 128 * t, r1 = r0 + 128 < N ? r0 + 128 : N;
        float amax = 0.0f;
        for (int r = r0; r < r1; r++)
            for (int c = 0; c < d; c++) {
                const float v = fabsf(X[(bh * N + r) * d + c]);
                if (v > amax) amax = v;
            }
        const float scale = amax > 0.0f ? amax / 448.0f : 0.0f;
        scales[blk] = scale;
        for (int r = r0; r < r1; r++)
            for (int c = 0; c < d; c++) {
                const unsigned char code = scale > 0.0f ? oracle_e4m3_encode(X[(bh * N + r) * d + c] / scale) : 0;
                if (transpose)
                    codes[(bh * d + c) * Np + r] = code;
                else
                    codes[(bh * N + r) * d + c] = code;
            }
    }
    return 0;
}
