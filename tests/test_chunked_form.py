"""The chunked form of the sparse scan (Sparse Delta Memory deck, "Training
parallelizes within chunks and recurs across chunks" and "Backup: sparse
interactions drive the triangular solve", App. A.1-A.2, Eq. 7) written out in
numpy, checked against the sequential fp64 oracle: the algebra the chunked
GPU kernel implements, independent of it.

Within a chunk, D_i(s) is the product of the decays of the tokens j <= i that
write slot s, u_i = v_i - vhat_i is token i's shared residual, and
    (I + A diag(beta)) u = v - p,     p_i = sum_n k_in D_i(s_in) M0[s_in],
    A[i,j] = sum_{n,m: s_in = s_jm} k_in k_jm D_i(s) / D_j(s)     (j < i),
    y_i = sum_m r_im D_i(rho_im) M0[rho_im] + sum_{j<=i} beta_j Qr[i,j] u_j,
    Qr[i,j] = sum_{m,n: rho_im = s_jn} r_im k_jn D_i(rho) / D_j(rho),
    M_C[s] = D_C(s) M0[s] + sum_{j writes s} beta_j k_j(s) D_C(s) / D_j(s) u_j.
(The additive write has u = v.)"""
import numpy as np
import pytest

import oracle


def chunked_scan(M0, v, alpha, beta, iw, ww, ir, wr, C, additive=False):
    """One (b, h) sequence: M0 [N, dv]; v [T, dv]; alpha, beta [T]; iw, ww
    [T, W]; ir, wr [T, R].  Returns (M_T, y [T, dv])."""
    M = M0.astype(np.float64).copy()
    T, dv = v.shape
    y = np.zeros((T, dv))
    for c0 in range(0, T, C):
        toks = range(c0, min(T, c0 + C))
        L = len(toks)
        Dw = np.zeros((L, iw.shape[1]))          # D_i(s_in) of every write pair
        Dr = np.ones((L, ir.shape[1]))           # D_i(rho_im) of every read pair
        cum = {}                                 # slot -> its decay so far in the chunk
        hist = {}                                # slot -> [(token, pair, D)] writes in the chunk
        for i, t in enumerate(toks):
            for n, s in enumerate(iw[t]):
                cum[s] = cum.get(s, 1.0) * alpha[t]
                Dw[i, n] = cum[s]
                hist.setdefault(s, []).append((i, n, cum[s]))
            for m, s in enumerate(ir[t]):
                Dr[i, m] = cum.get(s, 1.0)
        A = np.zeros((L, L))
        Qr = np.zeros((L, L))
        for s, lst in hist.items():
            for a_i, (i, n, di) in enumerate(lst):
                for (j, m, dj) in lst[:a_i]:
                    A[i, j] += ww[toks[i], n] * ww[toks[j], m] * di / dj
        for i, t in enumerate(toks):
            for m, s in enumerate(ir[t]):
                for (j, n, dj) in hist.get(s, []):
                    if j <= i:
                        Qr[i, j] += wr[t, m] * ww[toks[j], n] * Dr[i, m] / dj
        tt = np.array(list(toks))
        p = np.stack([(ww[t, :, None] * Dw[i, :, None] * M[iw[t]]).sum(0) for i, t in enumerate(toks)])
        if additive:
            u = v[tt].astype(np.float64)
        else:
            u = np.linalg.solve(np.eye(L) + A * beta[tt][None, :], v[tt] - p)
        y[tt] = np.stack([(wr[t, :, None] * Dr[i, :, None] * M[ir[t]]).sum(0) for i, t in enumerate(toks)])
        y[tt] += (Qr * beta[tt][None, :]) @ u
        newM = {}
        for s, lst in hist.items():
            dC = lst[-1][2]
            row = dC * M[s]
            for (j, n, dj) in lst:
                row = row + beta[toks[j]] * ww[toks[j], n] * dC / dj * u[j]
            newM[s] = row
        for s, row in newM.items():
            M[s] = row
    return M, y


@pytest.mark.parametrize("additive", [False, True])
@pytest.mark.parametrize("N,C", [(12, 4), (40, 8), (40, 16)])
def test_chunked_form_equals_the_sequential_scan(N, C, additive):
    """Small N makes rows repeat within chunks (write-write and read-write
    interactions) and T = 37 leaves a ragged last chunk."""
    rng = np.random.default_rng(N + C)
    T, dv, W, R = 37, 5, 3, 4
    iw = np.stack([rng.permutation(N)[:W] for _ in range(T)]).astype(np.int32)
    ir = np.stack([rng.permutation(N)[:R] for _ in range(T)]).astype(np.int32)
    ww = rng.uniform(0.05, 0.6, (T, W))
    wr = rng.uniform(-1, 1, (T, R))
    v = rng.standard_normal((T, dv))
    alpha = rng.uniform(0.5, 1.0, T)
    beta = rng.uniform(0.1, 0.9, T)
    M0 = rng.standard_normal((N, dv))
    mode = oracle.RESID_ADDITIVE if additive else oracle.RESID_SHARED
    Mr, yr = oracle.sdm_scan(M0[None, None], v[None, :, None], alpha[None, :, None], beta[None, :, None],
                             iw[None, :, None], ww[None, :, None], ir[None, :, None], wr[None, :, None], mode)
    Mc, yc = chunked_scan(M0, v, alpha, beta, iw, ww, ir, wr, C, additive)
    np.testing.assert_allclose(Mc, Mr[0, 0], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(yc, yr[0, :, 0], rtol=1e-10, atol=1e-10)
