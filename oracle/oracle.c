/*
 * oracle.c - plain, slow, fp64 CPU oracle for the delta-rule memory scans.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA library never
 * links, includes or calls anything here, and nothing here is shared with it.
 *
 * Every function is a direct, sequential, per-token restatement of the
 * recurrences on the pages, in fp64, with no blocking, fusion or reordering:
 *
 *   oracle_address   - product-key addressing (Sparse Delta Memory deck,
 *                      "Product keys select addresses without scoring every
 *                      slot", Secs. 2 / 3.1).
 *   oracle_address_backward - the gradient of the selected weights with
 *                      respect to the two score halves (softmax over the
 *                      selected sums; the selection itself is piecewise
 *                      constant).
 *   oracle_sdm_scan  - selective decay, delta write, read after write (same
 *                      deck, "Selected slots decay and update; other slots
 *                      persist", Eqs. 3-5, and "A v1 inconsistency matters for
 *                      reproducing the update", Fig. 2 shared residual).
 *   oracle_sdm_scan_backward - the gradients of oracle_sdm_scan, walking the
 *                      tokens backwards and undoing each token's writes from
 *                      the rows the forward logged (same deck, "Training
 *                      parallelizes within chunks and recurs across chunks"
 *                      and "Backup: undoing writes avoids repeated full-table
 *                      snapshots", App. A.3).
 *   oracle_gdn_scan  - dense Gated DeltaNet / KDA (Linear Attention
 *                      Architectures deck, "GDN and KDA change the granularity
 *                      of forgetting", Eqs. 15-20).
 *   oracle_gdn2_scan - GDN2 (same deck, "GDN2 separates key-side erase and
 *                      value-side write", Eqs. 21-24).
 *   oracle_sse_scan  - Sparse State Expansion (SSE deck, "One gate controls
 *                      both writes and reads", Eqs. 9-14, with the always-active
 *                      shared partition of "SSE routes tokens into
 *                      shared-parameter state partitions").
 *
 * Precision: all state and value arithmetic is fp64.  Only the selection
 * arithmetic is fp32 on purpose: a slot's score is the fp32 sum of two fp32
 * halves, and every comparison that picks an index compares fp32 values, so
 * the chosen index sets are a property of the fp32 inputs.  Ties are broken
 * towards the lower index at every stage.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC.
 * No function here is threaded; the callers parallelise over independent
 * sequences if they want to.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_VERSION 1

int oracle_version(void) { return ORACLE_VERSION; }

/* bf16 bit pattern -> exact value. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One scored candidate: fp32 score, integer id. */
typedef struct {
    float score;
    int id;
} cand_t;

/* Order: score descending, then id ascending. */
static int cand_cmp(const void *pa, const void *pb)
{
    const cand_t *a = (const cand_t *)pa, *b = (const cand_t *)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

/* Indices of the k largest entries of x[0..n), by (value desc, index asc),
 * written in rank order. */
static void topk_f32(const float *x, int n, int k, int *out, cand_t *work)
{
    for (int i = 0; i < n; ++i) {
        work[i].score = x[i];
        work[i].id = i;
    }
    qsort(work, (size_t)n, sizeof(cand_t), cand_cmp);
    for (int i = 0; i < k; ++i) out[i] = work[i].id;
}

/*
 * Product-key addressing for one token-head (SDM deck, "Product keys select
 * addresses without scoring every slot"):
 *   1. keep each half's top-k (by value, ties to the lower index);
 *   2. form only the k*k candidate scores s_{a,b} = s1[a] + s2[b] (an outer
 *      SUM, one fp32 addition each), slot id i = a*sqrtN + b;
 *   3. keep the top-W candidates by (score desc, id asc);
 *   4. weights = softmax over the W selected scores (no temperature, max
 *      subtracted), in fp64.
 * idx[W] comes out in rank order.
 */
static void address_one(const float *s1, const float *s2, int sqrtN, int k, int W,
                        int32_t *idx, double *w, cand_t *work, int *ta, int *tb)
{
    topk_f32(s1, sqrtN, k, ta, work);
    topk_f32(s2, sqrtN, k, tb, work);
    int nc = 0;
    for (int x = 0; x < k; ++x) {
        for (int y = 0; y < k; ++y) {
            float s = s1[ta[x]] + s2[tb[y]]; /* fp32 sum, round to nearest */
            work[nc].score = s;
            work[nc].id = ta[x] * sqrtN + tb[y];
            ++nc;
        }
    }
    qsort(work, (size_t)nc, sizeof(cand_t), cand_cmp);
    double mx = (double)work[0].score;
    double z = 0.0;
    for (int j = 0; j < W; ++j) z += exp((double)work[j].score - mx);
    for (int j = 0; j < W; ++j) {
        idx[j] = work[j].id;
        w[j] = exp((double)work[j].score - mx) / z;
    }
}

/*
 * s1, s2: fp32 [B,T,H,sqrtN].  idx_out: int32 [B,T,H,W]; w_out: fp64
 * [B,T,H,W].  Requires 1 <= k <= sqrtN and 1 <= W <= k*k.  Returns 0, or -1
 * on bad sizes.
 */
int oracle_address(const float *s1, const float *s2, int B, int T, int H, int sqrtN, int k, int W,
                   int32_t *idx_out, double *w_out)
{
    if (B < 0 || T < 0 || H < 0 || sqrtN < 1 || k < 1 || k > sqrtN || W < 1 || W > k * k) return -1;
    int ncand = k * k > sqrtN ? k * k : sqrtN;
    cand_t *work = (cand_t *)malloc(sizeof(cand_t) * (size_t)ncand);
    int *ta = (int *)malloc(sizeof(int) * (size_t)k);
    int *tb = (int *)malloc(sizeof(int) * (size_t)k);
    if (!work || !ta || !tb) {
        free(work); free(ta); free(tb);
        return -1;
    }
    long rows = (long)B * T * H;
    for (long r = 0; r < rows; ++r)
        address_one(s1 + r * sqrtN, s2 + r * sqrtN, sqrtN, k, W, idx_out + r * W, w_out + r * W, work, ta,
                    tb);
    free(work); free(ta); free(tb);
    return 0;
}

/*
 * Backward of the addressing weights (SDM deck, Secs. 2 / 3.1): with
 * w = softmax(s) over the W selected sums s_i = s1[a_i] + s2[b_i],
 * i = a_i sqrtN + b_i, the loss gradient dw gives
 *   ds_i = w_i (dw_i - sum_j w_j dw_j),   ds1[a_i] += ds_i,   ds2[b_i] += ds_i,
 * and zero for every score outside the selection.
 *
 * idx, w, dw : [rows][W] (int32, fp64, fp64).  ds1, ds2 : fp64 [rows][sqrtN] out.
 */
int oracle_address_backward(const int32_t *idx, const double *w, const double *dw, long rows, int sqrtN, int W,
                            double *ds1, double *ds2)
{
    if (rows < 0 || sqrtN < 1 || W < 1) return -1;
    for (long r = 0; r < rows; ++r) {
        const int32_t *ix = idx + r * W;
        const double *wr = w + r * W, *dwr = dw + r * W;
        double *d1 = ds1 + r * sqrtN, *d2 = ds2 + r * sqrtN;
        for (int a = 0; a < sqrtN; ++a) d1[a] = d2[a] = 0.0;
        double dot = 0.0;
        for (int j = 0; j < W; ++j) dot += wr[j] * dwr[j];
        for (int j = 0; j < W; ++j) {
            if (ix[j] < 0 || ix[j] >= sqrtN * sqrtN) return -2;
            double ds = wr[j] * (dwr[j] - dot);
            d1[ix[j] / sqrtN] += ds;
            d2[ix[j] % sqrtN] += ds;
        }
    }
    return 0;
}

/* Residual modes of the sparse write. */
#define ORACLE_RESID_SHARED 0   /* Fig. 2: one shared prediction v_hat       */
#define ORACLE_RESID_PERSLOT 1  /* printed Eq. 4: each slot's own residual    */
#define ORACLE_RESID_ADDITIVE 2 /* additive write (no residual), SSE-style    */

/*
 * Sparse delta-rule memory scan (SDM deck, Eqs. 3-5 and Fig. 2).
 *
 * state : fp64 [B,H,N,dv], updated in place (M_0 in, M_T out).
 * v     : fp64 [B,T,H,dv]  (callers widen fp32 or bf16 exactly).
 * alpha, beta : fp64 [B,T,H]  (per-head forget and input gates).
 * idx_w, w_w  : int32 / fp64 [B,T,H,W]  write slots I^w and weights k^(i).
 * idx_r, w_r  : int32 / fp64 [B,T,H,R]  read slots I^r and weights q^(i).
 * y     : fp64 [B,T,H,dv].
 * undo  : optional fp64 [B,T,H,W,dv] (NULL: not kept): the rows of I^w as
 *         they were before token t's decay, the log the backward undoes.
 *
 * For each (b,h), tokens in order:
 *   M~[i]  = alpha * M[i]                          for i in I^w only
 *   shared   : v_hat = sum_j w_j M~[j];  M[i] = M~[i] + beta w_i (v - v_hat)
 *   per-slot : M[i] = M~[i] + beta w_i (v - M~[i])
 *   additive : M[i] = M~[i] + beta w_i v
 *   rows not in I^w are left as they are;
 *   y = sum_{i in I^r} r_i M[i], read after the write.
 * Returns 0, -1 on bad sizes, -2 on an out-of-range or repeated write slot.
 */
int oracle_sdm_scan(double *state, const double *v, const double *alpha, const double *beta,
                    const int32_t *idx_w, const double *w_w, int W, const int32_t *idx_r, const double *w_r,
                    int R, int B, int T, int H, int N, int dv, int mode, double *y, double *undo)
{
    if (B < 0 || T < 0 || H < 0 || N < 1 || dv < 1 || W < 1 || R < 1) return -1;
    if (mode != ORACLE_RESID_SHARED && mode != ORACLE_RESID_PERSLOT && mode != ORACLE_RESID_ADDITIVE)
        return -1;
    double *mt = (double *)malloc(sizeof(double) * (size_t)W * dv);
    double *vhat = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!mt || !vhat) {
        free(mt); free(vhat);
        return -1;
    }
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        for (int h = 0; h < H && rc == 0; ++h) {
            double *M = state + ((size_t)b * H + h) * (size_t)N * dv;
            for (int t = 0; t < T; ++t) {
                size_t tok = ((size_t)b * T + t) * H + h;
                const int32_t *iw = idx_w + tok * W;
                const int32_t *ir = idx_r + tok * R;
                const double *ww = w_w + tok * W;
                const double *wr = w_r + tok * R;
                const double *vt = v + tok * dv;
                double a = alpha[tok], be = beta[tok];
                for (int j = 0; j < W; ++j) {
                    if (iw[j] < 0 || iw[j] >= N) { rc = -2; goto done; }
                    for (int jj = 0; jj < j; ++jj)
                        if (iw[jj] == iw[j]) { rc = -2; goto done; }
                }
                for (int j = 0; j < R; ++j)
                    if (ir[j] < 0 || ir[j] >= N) { rc = -2; goto done; }
                if (undo)
                    for (int j = 0; j < W; ++j)
                        memcpy(undo + (tok * W + j) * (size_t)dv, M + (size_t)iw[j] * dv, sizeof(double) * dv);
                /* selective decay of the written rows only */
                for (int j = 0; j < W; ++j)
                    for (int c = 0; c < dv; ++c) mt[(size_t)j * dv + c] = a * M[(size_t)iw[j] * dv + c];
                /* shared prediction from the decayed rows (Fig. 2) */
                for (int c = 0; c < dv; ++c) {
                    double s = 0.0;
                    for (int j = 0; j < W; ++j) s += ww[j] * mt[(size_t)j * dv + c];
                    vhat[c] = s;
                }
                /* delta write into the selected rows */
                for (int j = 0; j < W; ++j) {
                    double *row = M + (size_t)iw[j] * dv;
                    for (int c = 0; c < dv; ++c) {
                        double m = mt[(size_t)j * dv + c];
                        double resid;
                        if (mode == ORACLE_RESID_SHARED) resid = vt[c] - vhat[c];
                        else if (mode == ORACLE_RESID_PERSLOT) resid = vt[c] - m;
                        else resid = vt[c];
                        row[c] = m + be * ww[j] * resid;
                    }
                }
                /* read after the write */
                double *yt = y + tok * dv;
                for (int c = 0; c < dv; ++c) {
                    double s = 0.0;
                    for (int j = 0; j < R; ++j) s += wr[j] * M[(size_t)ir[j] * dv + c];
                    yt[c] = s;
                }
            }
        }
    }
done:
    free(mt); free(vhat);
    return rc;
}

/*
 * Backward of oracle_sdm_scan, undoing the writes (SDM deck, App. A.3: the
 * forward keeps only the sparse update log, the backward walks the tokens in
 * reverse and restores each token's written rows from it).
 *
 * state  : fp64 [B,H,N,dv]  M_T in; M_0 out (every written row restored).
 * dstate : fp64 [B,H,N,dv]  dL/dM_T in; dL/dM_0 out.
 * v, alpha, beta, idx_w, w_w, idx_r, w_r, mode : as in oracle_sdm_scan.
 * undo   : fp64 [B,T,H,W,dv]  the forward's log (rows of I^w before decay).
 * dy     : fp64 [B,T,H,dv]    dL/dy.
 * dv     : fp64 [B,T,H,dv] out.   dalpha, dbeta : fp64 [B,T,H] out.
 * dw_w   : fp64 [B,T,H,W] out.    dw_r : fp64 [B,T,H,R] out.
 *
 * For token t (last to first), with M = M_t and G = dL/dM_t:
 *   read   y = sum_i r_i M[i]:       dr_i = <dy, M[i]>,  G[i] += r_i dy
 *   write  M[i_j] = m_j + beta w_j rho_j,  m_j = alpha undo_j, with
 *            shared   rho_j = v - sum_k w_k m_k
 *            per-slot rho_j = v - m_j
 *            additive rho_j = v
 *          and G_j = G[i_j]:
 *            dbeta   = sum_j w_j <G_j, rho_j>
 *            dw_j    = beta <G_j, rho_j>  (- <g, m_j> for shared)
 *            dv      = g = beta sum_j w_j G_j
 *            dm_j    = G_j - w_j g (shared), G_j (1 - beta w_j) (per-slot), G_j (additive)
 *            dalpha  = sum_j <dm_j, undo_j>
 *          then G[i_j] = alpha dm_j and M[i_j] = undo_j.
 * Rows outside I^w pass their gradient through unchanged.
 */
int oracle_sdm_scan_backward(double *state, double *dstate, const double *v, const double *alpha,
                             const double *beta, const int32_t *idx_w, const double *w_w, int W,
                             const int32_t *idx_r, const double *w_r, int R, int B, int T, int H, int N, int dv,
                             int mode, const double *undo, const double *dy, double *dvo, double *dalpha,
                             double *dbeta, double *dw_w, double *dw_r)
{
    if (B < 0 || T < 0 || H < 0 || N < 1 || dv < 1 || W < 1 || R < 1) return -1;
    if (mode != ORACLE_RESID_SHARED && mode != ORACLE_RESID_PERSLOT && mode != ORACLE_RESID_ADDITIVE)
        return -1;
    double *m = (double *)malloc(sizeof(double) * (size_t)W * dv);
    double *G = (double *)malloc(sizeof(double) * (size_t)W * dv);
    double *res = (double *)malloc(sizeof(double) * (size_t)W * dv);
    double *g = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!m || !G || !res || !g) {
        free(m); free(G); free(res); free(g);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double *M = state + ((size_t)b * H + h) * (size_t)N * dv;
            double *dM = dstate + ((size_t)b * H + h) * (size_t)N * dv;
            for (int t = T - 1; t >= 0; --t) {
                size_t tok = ((size_t)b * T + t) * H + h;
                const int32_t *iw = idx_w + tok * W, *ir = idx_r + tok * R;
                const double *ww = w_w + tok * W, *wr = w_r + tok * R;
                const double *vt = v + tok * dv, *dyt = dy + tok * dv;
                const double *un = undo + tok * (size_t)W * dv;
                double a = alpha[tok], be = beta[tok];
                /* read after the write */
                for (int i = 0; i < R; ++i) {
                    double *row = M + (size_t)ir[i] * dv, *drow = dM + (size_t)ir[i] * dv;
                    double s = 0.0;
                    for (int c = 0; c < dv; ++c) s += dyt[c] * row[c];
                    dw_r[tok * R + i] = s;
                    for (int c = 0; c < dv; ++c) drow[c] += wr[i] * dyt[c];
                }
                /* the write: decayed rows, residuals, incoming gradients */
                for (int j = 0; j < W; ++j)
                    for (int c = 0; c < dv; ++c) {
                        m[(size_t)j * dv + c] = a * un[(size_t)j * dv + c];
                        G[(size_t)j * dv + c] = dM[(size_t)iw[j] * dv + c];
                    }
                for (int c = 0; c < dv; ++c) {
                    double vh = 0.0;
                    if (mode == ORACLE_RESID_SHARED)
                        for (int j = 0; j < W; ++j) vh += ww[j] * m[(size_t)j * dv + c];
                    for (int j = 0; j < W; ++j)
                        res[(size_t)j * dv + c] = mode == ORACLE_RESID_SHARED    ? vt[c] - vh
                                                  : mode == ORACLE_RESID_PERSLOT ? vt[c] - m[(size_t)j * dv + c]
                                                                                 : vt[c];
                    double s = 0.0;
                    for (int j = 0; j < W; ++j) s += ww[j] * G[(size_t)j * dv + c];
                    g[c] = be * s;
                    dvo[tok * dv + c] = g[c];
                }
                double db = 0.0, da = 0.0;
                for (int j = 0; j < W; ++j) {
                    double gr = 0.0, gm = 0.0;
                    for (int c = 0; c < dv; ++c) {
                        gr += G[(size_t)j * dv + c] * res[(size_t)j * dv + c];
                        gm += g[c] * m[(size_t)j * dv + c];
                    }
                    db += ww[j] * gr;
                    dw_w[tok * W + j] = be * gr - (mode == ORACLE_RESID_SHARED ? gm : 0.0);
                    double *drow = dM + (size_t)iw[j] * dv, *row = M + (size_t)iw[j] * dv;
                    for (int c = 0; c < dv; ++c) {
                        double Gc = G[(size_t)j * dv + c];
                        double dm = mode == ORACLE_RESID_SHARED    ? Gc - ww[j] * g[c]
                                    : mode == ORACLE_RESID_PERSLOT ? Gc * (1.0 - be * ww[j])
                                                                   : Gc;
                        da += dm * un[(size_t)j * dv + c];
                        drow[c] = a * dm;
                        row[c] = un[(size_t)j * dv + c];
                    }
                }
                dbeta[tok] = db;
                dalpha[tok] = da;
            }
        }
    }
    free(m); free(G); free(res); free(g);
    return 0;
}

/*
 * Dense Gated DeltaNet / KDA scan (Linear Attention Architectures deck,
 * Eqs. 15-20), with the state stored key-major: S = W^T, S in R^{dk x dv}.
 *
 * state : fp64 [B,H,dk,dv] in place.   q, k : fp64 [B,T,H,dk].  v : [B,T,H,dv].
 * alpha : fp64 [B,T,H] (GDN, per_channel = 0) or [B,T,H,dk] (KDA).
 * beta  : fp64 [B,T,H].  y : fp64 [B,T,H,dv].
 *
 * Per token:  S~ = D_alpha S            (row r scaled by alpha_r; GDN: alpha)
 *             pred = S~^T k             (decay-adjusted prediction, W D_a k)
 *             S = S~ + beta k (v - pred)^T
 *             y = S^T q                 (unnormalised read of the new state)
 */
int oracle_gdn_scan(double *state, const double *q, const double *k, const double *v, const double *alpha,
                    int per_channel, const double *beta, int B, int T, int H, int dk, int dv, double *y)
{
    if (B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1) return -1;
    double *pred = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!pred) return -1;
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double *S = state + ((size_t)b * H + h) * (size_t)dk * dv;
            for (int t = 0; t < T; ++t) {
                size_t tok = ((size_t)b * T + t) * H + h;
                const double *qt = q + tok * dk, *kt = k + tok * dk, *vt = v + tok * dv;
                double be = beta[tok];
                for (int r = 0; r < dk; ++r) {
                    double a = per_channel ? alpha[tok * dk + r] : alpha[tok];
                    for (int c = 0; c < dv; ++c) S[(size_t)r * dv + c] *= a;
                }
                for (int c = 0; c < dv; ++c) {
                    double s = 0.0;
                    for (int r = 0; r < dk; ++r) s += S[(size_t)r * dv + c] * kt[r];
                    pred[c] = s;
                }
                for (int r = 0; r < dk; ++r)
                    for (int c = 0; c < dv; ++c) S[(size_t)r * dv + c] += be * kt[r] * (vt[c] - pred[c]);
                double *yt = y + tok * dv;
                for (int c = 0; c < dv; ++c) {
                    double s = 0.0;
                    for (int r = 0; r < dk; ++r) s += S[(size_t)r * dv + c] * qt[r];
                    yt[c] = s;
                }
            }
        }
    }
    free(pred);
    return 0;
}

/*
 * GDN2 (Linear Attention Architectures deck, "GDN2 separates key-side erase
 * and value-side write", Eqs. 21-24), with the state stored key-major
 * (S = W^T, so W D_alpha is D_alpha S):
 *
 * state  : fp64 [B,H,dk,dv] in place.   q, k : fp64 [B,T,H,dk].  v : [B,T,H,dv].
 * alpha  : fp64 [B,T,H,dk] per-key-channel decay.
 * berase : fp64 [B,T,H,dk] erase gate b.   wwrite : fp64 [B,T,H,dv] write gate w.
 * y      : fp64 [B,T,H,dv].
 *
 * Per token:  S~ = D_alpha S
 *             e = b (.) k,   z = w (.) v
 *             r = z - S~^T e             (the residual at the erase key)
 *             S = S~ + k r^T             (the outer product takes k, not e)
 *             y = S^T q
 */
int oracle_gdn2_scan(double *state, const double *q, const double *k, const double *v, const double *alpha,
                     const double *berase, const double *wwrite, int B, int T, int H, int dk, int dv, double *y)
{
    if (B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1) return -1;
    double *r = (double *)malloc(sizeof(double) * (size_t)dv);
    double *e = (double *)malloc(sizeof(double) * (size_t)dk);
    if (!r || !e) { free(r); free(e); return -1; }
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double *S = state + ((size_t)b * H + h) * (size_t)dk * dv;
            for (int t = 0; t < T; ++t) {
                size_t tok = ((size_t)b * T + t) * H + h;
                const double *qt = q + tok * dk, *kt = k + tok * dk, *vt = v + tok * dv;
                for (int i = 0; i < dk; ++i) {
                    double a = alpha[tok * dk + i];
                    for (int c = 0; c < dv; ++c) S[(size_t)i * dv + c] *= a;
                    e[i] = berase[tok * dk + i] * kt[i];
                }
                for (int c = 0; c < dv; ++c) {
                    double s = 0.0;
                    for (int i = 0; i < dk; ++i) s += S[(size_t)i * dv + c] * e[i];
                    r[c] = wwrite[tok * dv + c] * vt[c] - s;
                }
                for (int i = 0; i < dk; ++i)
                    for (int c = 0; c < dv; ++c) S[(size_t)i * dv + c] += kt[i] * r[c];
                double *yt = y + tok * dv;
                for (int c = 0; c < dv; ++c) {
                    double s = 0.0;
                    for (int i = 0; i < dk; ++i) s += S[(size_t)i * dv + c] * qt[i];
                    yt[c] = s;
                }
            }
        }
    }
    free(r);
    free(e);
    return 0;
}

/*
 * Sparse State Expansion scan (SSE deck, Eqs. 9-14) with one always-active
 * shared partition.
 *
 * state  : fp64 [B,H,N+1,c,d] in place; partition N is the shared one.
 * route  : fp32 [B,T,H,N] router logits x W_e.
 * klog   : fp32 [B,T,H,c] key logits x W_k.
 * q      : fp64 [B,T,H,c].  v : fp64 [B,T,H,d].
 * alpha  : fp64 [B,T,H,c]  per-row (GLA-style) decay Lambda_t = diag(alpha_t).
 * y      : fp64 [B,T,H,d].  sel : int32 [B,T,H,topk] selected partitions (rank order).
 * mode   : 0 additive write (the deck's SSE), 1 delta write: the write
 *          residual of every visited partition is shared by its rows,
 *          v - vhat_p with vhat_p = sum_j kk_j alpha_j S^p[j,:] (the decayed
 *          prediction of the partition, as the Sparse Delta Memory deck's
 *          shared residual of Fig. 2 with weights kk and strength g).
 *
 * Per token:  e = softmax(route) over all N (not renormalised after top-k);
 *             T_t = top-k of the fp32 logits (ties to the lower index);
 *             kk = softmax(klog) over the c rows;
 *             for p in T_t (gate g = e_p) and the shared partition (g = 1):
 *                 S^p[j,:] = alpha_j S^p[j,:] + g kk_j v      (j < c)
 *             partitions not visited keep their state (and their decay clock);
 *             y = sum_p g_p sum_j q_j S^p[j,:]   (read of the updated states).
 */
int oracle_sse_scan(double *state, const float *route, int topk, const float *klog, const double *q,
                    const double *v, const double *alpha, int B, int T, int H, int N, int c, int d, double *y,
                    int32_t *sel, int mode)
{
    if (B < 0 || T < 0 || H < 0 || N < 1 || topk < 1 || topk > N || c < 1 || d < 1) return -1;
    if (mode != 0 && mode != 1) return -1;
    cand_t *work = (cand_t *)malloc(sizeof(cand_t) * (size_t)N);
    int *tsel = (int *)malloc(sizeof(int) * (size_t)(topk + 1));
    double *e = (double *)malloc(sizeof(double) * (size_t)N);
    double *kk = (double *)malloc(sizeof(double) * (size_t)c);
    double *g = (double *)malloc(sizeof(double) * (size_t)(topk + 1));
    double *res = (double *)malloc(sizeof(double) * (size_t)d);
    if (!work || !tsel || !e || !kk || !g || !res) {
        free(work); free(tsel); free(e); free(kk); free(g); free(res);
        return -1;
    }
    size_t part = (size_t)c * d;
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double *S = state + ((size_t)b * H + h) * (size_t)(N + 1) * part;
            for (int t = 0; t < T; ++t) {
                size_t tok = ((size_t)b * T + t) * H + h;
                const float *lt = route + tok * N;
                const float *kl = klog + tok * c;
                const double *qt = q + tok * c, *vt = v + tok * d, *at = alpha + tok * c;
                /* e_t = softmax(x W_e) over all N partitions */
                double mx = (double)lt[0];
                for (int p = 1; p < N; ++p) if ((double)lt[p] > mx) mx = (double)lt[p];
                double z = 0.0;
                for (int p = 0; p < N; ++p) z += exp((double)lt[p] - mx);
                for (int p = 0; p < N; ++p) e[p] = exp((double)lt[p] - mx) / z;
                /* T_t = TopKIndices(e_t, k) */
                topk_f32(lt, N, topk, tsel, work);
                for (int j = 0; j < topk; ++j) {
                    sel[tok * topk + j] = tsel[j];
                    g[j] = e[tsel[j]];
                }
                tsel[topk] = N; /* shared partition */
                g[topk] = 1.0;
                /* k_t = softmax(x W_k) over the c rows */
                double km = (double)kl[0];
                for (int j = 1; j < c; ++j) if ((double)kl[j] > km) km = (double)kl[j];
                double kz = 0.0;
                for (int j = 0; j < c; ++j) kz += exp((double)kl[j] - km);
                for (int j = 0; j < c; ++j) kk[j] = exp((double)kl[j] - km) / kz;
                /* update the visited partitions */
                for (int s = 0; s <= topk; ++s) {
                    double *Sp = S + (size_t)tsel[s] * part;
                    for (int col = 0; col < d; ++col) {
                        double vhat = 0.0;
                        if (mode == 1)
                            for (int j = 0; j < c; ++j) vhat += kk[j] * at[j] * Sp[(size_t)j * d + col];
                        res[col] = vt[col] - vhat;
                    }
                    for (int j = 0; j < c; ++j)
                        for (int col = 0; col < d; ++col)
                            Sp[(size_t)j * d + col] = at[j] * Sp[(size_t)j * d + col] + g[s] * kk[j] * res[col];
                }
                /* read the updated visited partitions */
                double *yt = y + tok * d;
                for (int col = 0; col < d; ++col) {
                    double acc = 0.0;
                    for (int s = 0; s <= topk; ++s) {
                        const double *Sp = S + (size_t)tsel[s] * part;
                        double inner = 0.0;
                        for (int j = 0; j < c; ++j) inner += qt[j] * Sp[(size_t)j * d + col];
                        acc += g[s] * inner;
                    }
                    yt[col] = acc;
                }
            }
        }
    }
    free(work); free(tsel); free(e); free(kk); free(g); free(res);
    return 0;
}

/* bf16 bits -> fp64, for callers that hand the oracle bf16 inputs. */
void oracle_widen_bf16(const uint16_t *src, double *dst, long n)
{
    for (long i = 0; i < n; ++i) dst[i] = bf16_value(src[i]);
}
