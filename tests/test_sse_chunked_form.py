"""The SSE prefill by varlen grouping (SSE deck, "Varlen groups tokens while
preserving causal order"; "One gate controls both writes and reads", Eqs.
9-14) in chunked form, written out in numpy and checked against the
sequential fp64 oracle: the algebra the chunked GPU kernels implement,
independent of them.

Per (batch, head) the tokens that visit a partition are gathered into one
subsequence (time order kept); the shared partition's subsequence is the whole
sequence.  Along a subsequence the partition follows a GLA recurrence,
S_i = diag(alpha_i) S_{i-1} + g_i kk_i^T v_i, read as o_i = g_i q_i S_i.
Within a chunk of C tokens (decay products over the chunk's tokens only):
    O    = Qt S0 + A V,           Qt_i = g_i q_i * prod_{t<=i} alpha_t
    A_ij = g_i g_j sum_r q_ir kk_jr prod_{t=j+1..i} alpha_tr      (j <= i)
    S_C  = diag(gamma) S0 + Kh^T V,  Kh_j = g_j kk_j * prod_{t>j} alpha_t,
    gamma = prod_t alpha_t.
Every decay factor is a product of alphas over a token range (never a
quotient), so nothing overflows; A's blocks of 16 tokens are formed with the
block boundaries as reference points (product within the later block up to i,
products of whole blocks between, product within the earlier block after j),
and each token's output is the sum of its visits' partial outputs."""
import numpy as np
import pytest

import oracle

SUB = 16  # tokens per block of A


def route(rt, topk):
    """top-k by (logit desc, index asc) and the softmax gates over all N."""
    order = sorted(range(len(rt)), key=lambda p: (-float(rt[p]), p))[:topk]
    e = np.exp(rt.astype(np.float64) - rt.max())
    return order, e[order] / e.sum()


def group(rt, topk):
    """per routed partition: the time-ordered (token, rank, gate) visits."""
    T, N = rt.shape
    lists = [[] for _ in range(N)]
    for t in range(T):
        sel, g = route(rt[t], topk)
        for r, (p, gp) in enumerate(zip(sel, g)):
            lists[p].append((t, r, gp))
    return lists


def chunk_operands(q, kk, al, g):
    """q, kk, al [L, c] (L <= C, padded by the caller), g [L].
    Returns Qt, Kh [L, c], A [L, L], gamma [c], built from block-local
    products as the GPU preparation forms them."""
    L, c = q.shape
    nb = (L + SUB - 1) // SUB
    F = np.ones((L, c))      # product within i's block, up to and including i
    R = np.ones((L, c))      # product within j's block, after j
    P = np.ones((nb, c))     # product over a whole block
    for J in range(nb):
        s, e = J * SUB, min(L, J * SUB + SUB)
        run = np.ones(c)
        for i in range(s, e):
            run = run * al[i]
            F[i] = run
        P[J] = run
        run = np.ones(c)
        for j in range(e - 1, s - 1, -1):
            R[j] = run
            run = run * al[j]
    pre = np.ones((nb, c))   # product of the blocks before J
    suf = np.ones((nb, c))   # product of the blocks after J
    for J in range(1, nb):
        pre[J] = pre[J - 1] * P[J - 1]
    for J in range(nb - 2, -1, -1):
        suf[J] = suf[J + 1] * P[J + 1]
    blk = np.arange(L) // SUB
    Qt = g[:, None] * q * F * pre[blk]
    Kh = g[:, None] * kk * R * suf[blk]
    A = np.zeros((L, L))
    for i in range(L):
        for j in range(i + 1):
            I, J = blk[i], blk[j]
            if I == J:
                f = np.ones(c)
                for t in range(j + 1, i + 1):
                    f = f * al[t]
            else:
                mid = np.ones(c)
                for K in range(J + 1, I):
                    mid = mid * P[K]
                f = F[i] * mid * R[j]
            A[i, j] = g[i] * g[j] * np.sum(q[i] * kk[j] * f)
    gamma = pre[nb - 1] * P[nb - 1]
    return Qt, Kh, A, gamma


def chunked_partition(S0, toks, gates, q, kk, al, v, C):
    """One partition's subsequence: toks (time order), gates.  Returns the
    final state and the partial output of every visit [len(toks), d]."""
    S = S0.copy()
    out = np.zeros((len(toks), v.shape[1]))
    for c0 in range(0, len(toks), C):
        sl = slice(c0, min(len(toks), c0 + C))
        tt = np.array(toks[sl])
        g = np.array(gates[sl])
        Qt, Kh, A, gamma = chunk_operands(q[tt], kk[tt], al[tt], g)
        out[sl] = Qt @ S + A @ v[tt]
        S = gamma[:, None] * S + Kh.T @ v[tt]
    return S, out


def sse_varlen(S0, rt, topk, klog, q, v, al, C):
    """One (batch, head): S0 [N+1, c, d]; returns (state, y)."""
    T, N = rt.shape
    kk = np.exp(klog - klog.max(1, keepdims=True))
    kk = kk / kk.sum(1, keepdims=True)
    S = S0.copy()
    part = np.zeros((T, topk + 1, v.shape[1]))
    for p, lst in enumerate(group(rt, topk)):
        if lst:
            toks, ranks, gates = zip(*lst)
            S[p], o = chunked_partition(S0[p], list(toks), list(gates), q, kk, al, v, C)
            part[list(toks), list(ranks)] = o
    S[N], part[:, topk] = chunked_partition(S0[N], list(range(T)), [1.0] * T, q, kk, al, v, C)
    return S, part.sum(1)


@pytest.mark.parametrize("C", [16, 32, 64])
@pytest.mark.parametrize("N,topk", [(4, 1), (8, 2), (5, 3)])
def test_varlen_chunked_form_equals_the_sequential_scan(N, topk, C):
    """T = 53 leaves ragged chunks in every subsequence; strong decays
    (alpha down to 0.02) would overflow a single-reference form (a quotient of
    products over 64 tokens) but not the block-referenced one."""
    rng = np.random.default_rng(10 * N + C + topk)
    T, c, d = 53, 24, 6
    rt = rng.standard_normal((T, N)).astype(np.float32)
    klog = rng.standard_normal((T, c)).astype(np.float32)
    q = rng.standard_normal((T, c))
    v = rng.standard_normal((T, d))
    al = rng.uniform(0.02, 1.0, (T, c))
    S0 = rng.standard_normal((N + 1, c, d))
    Sr, yr, _ = oracle.sse_scan(S0[None, None], rt[None, :, None], topk, klog[None, :, None], q[None, :, None],
                                v[None, :, None], al[None, :, None])
    Sc, yc = sse_varlen(S0, rt, topk, klog.astype(np.float64), q, v, al, C)
    np.testing.assert_allclose(Sc, Sr[0, 0], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(yc, yr[0, :, 0], rtol=1e-10, atol=1e-10)


def test_block_referenced_factors_stay_finite_under_strong_decay():
    """alpha = 1e-3 on every channel: the products over 64 tokens underflow
    to 0, and a quotient form b_i / b_j would be 0/0; the block-referenced
    operands stay finite and A equals its definition."""
    rng = np.random.default_rng(3)
    L, c = 64, 8
    q = rng.standard_normal((L, c))
    kk = rng.uniform(0.0, 1.0, (L, c))
    al = np.full((L, c), 1e-3)
    g = rng.uniform(0.1, 1.0, L)
    with np.errstate(under="ignore"):
        Qt, Kh, A, gamma = chunk_operands(q, kk, al, g)
    assert np.all(np.isfinite(Qt)) and np.all(np.isfinite(Kh)) and np.all(np.isfinite(A))
    for i in range(L):
        for j in (i, i - 1):
            if j >= 0:
                want = g[i] * g[j] * np.sum(q[i] * kk[j]) * 1e-3 ** (i - j)
                assert A[i, j] == pytest.approx(want, rel=1e-12, abs=1e-300)


def offdiag_blocks_by_stacked_product(q, kk, al, g):
    """The blocks of A below the diagonal (I > J) as products of two
    block-referenced operands, the form a tensor-core preparation would use:
        X_I           = rows of block I of  g q F          (F: product in i's block up to i)
        Z_J^(s)       = rows of block J of  g kk R * prod_{K=J+1}^{J+s-1} P_K
        A_IJ          = X_I (Z_J^(I-J))^T
    so all of them come out of one product X [L, c] times the stacked
    [Z^(1); Z^(2); Z^(3)]^T [c, 3L], with no quotient of decay products."""
    L, c = q.shape
    nb = (L + SUB - 1) // SUB
    F = np.ones((L, c))
    R = np.ones((L, c))
    P = np.ones((nb, c))
    for J in range(nb):
        s, e = J * SUB, min(L, J * SUB + SUB)
        run = np.ones(c)
        for i in range(s, e):
            run = run * al[i]
            F[i] = run
        P[J] = run
        run = np.ones(c)
        for j in range(e - 1, s - 1, -1):
            R[j] = run
            run = run * al[j]
    blk = np.arange(L) // SUB
    X = g[:, None] * q * F
    Y = g[:, None] * kk * R
    Zs = []
    for span in range(1, nb):        # span = I - J
        mid = np.ones((L, c))
        for j in range(L):
            for K in range(blk[j] + 1, min(nb, blk[j] + span)):
                mid[j] = mid[j] * P[K]
        Zs.append(Y * mid)
    G = X @ np.concatenate(Zs, axis=0).T if Zs else np.zeros((L, 0))   # [L, (nb-1) L]
    A = np.zeros((L, L))
    for i in range(L):
        for j in range(L):
            span = blk[i] - blk[j]
            if span >= 1:
                A[i, j] = G[i, (span - 1) * L + j]
    return A


@pytest.mark.parametrize("L,lo", [(64, 0.05), (53, 0.02), (64, 1e-3)])
def test_offdiagonal_blocks_as_one_stacked_product(L, lo):
    """The stacked-product form of A's blocks below the diagonal equals the
    definition, for full and ragged chunks and under decays strong enough
    that products over the chunk underflow (every factor stays finite)."""
    rng = np.random.default_rng(int(L + 1000 * lo))
    c = 16
    q = rng.standard_normal((L, c))
    kk = rng.uniform(0.0, 1.0, (L, c))
    al = rng.uniform(lo, 1.0, (L, c))
    g = rng.uniform(0.1, 1.0, L)
    with np.errstate(under="ignore"):
        _, _, A, _ = chunk_operands(q, kk, al, g)
        B = offdiag_blocks_by_stacked_product(q, kk, al, g)
    blk = np.arange(L) // SUB
    below = blk[:, None] > blk[None, :]
    assert np.all(np.isfinite(B))
    # the same products summed in another order: rounding only (entries that
    # nearly cancel get an absolute bound scaled to the matrix)
    np.testing.assert_allclose(B[below], A[below], rtol=1e-10, atol=1e-13 * np.abs(A).max())
    assert not np.any(B[~below])
