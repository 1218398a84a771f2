"""The chunk forms that the tensor-core preparation and chain
kernels implement (dense GDN, and the per-channel-decay form of KDA: Linear
Attention Architectures deck, "GDN and KDA
change the granularity of forgetting", Eqs. 18-20; GDN2: "GDN2 separates
key-side erase and value-side write", Eqs. 21-24; the SSE delta write on each
partition's visit subsequence), written out in numpy and checked against the
sequential fp64 oracle, independent of the kernels.

Within a chunk of C = 64 tokens, with lambda_t = sum_{s<=t} log alpha_s per
key channel (the chunk's own tokens only), every pair sum needs its own decay
sum_r x_ir y_jr prod_{t=j+1..i} alpha_tr.  The preparation forms it in two
ways: pairs inside a block of 4 tokens from running products of alpha; every
other pair split at the highest bit in which i and j differ (half size h),
i in the right half and j in the left half of a segment of 2h tokens whose
left half ends at token b, as (x_i e^{lambda_i - lambda_b}) . (y_j
e^{lambda_b - lambda_j}) - two decay ratios of at most 1.  Then
    A_ij = beta_i (k_i . k_j)~ (j < i)   [GDN2: (e_i . k_j)~, no beta]
    Mq_ij = (q_i . k_j)~ (j <= i)
    T = (I + A)^-1 diag(beta)            [GDN2: (I + A)^-1]
    W = T (k e^lambda)                   [GDN2: T (e e^lambda)]
    Ut = T V                             [GDN2: T (w v)]
and the chain runs U = Ut - W S0, Y = (q e^lambda) S0 + Mq U,
S_C = diag(e^{lambda_C}) S0 + (k e^{lambda_C - lambda})^T U."""
import numpy as np
import pytest

import oracle

C = 64


def pair_sums(lam, al, x, y, strict):
    """P_ij = sum_r x_ir y_jr prod_{t=j+1..i} al_tr for j < i (strict) or
    j <= i, as the preparation forms them (see the module docstring).  Also
    checks that no decay factor used exceeds 1."""
    L, c = x.shape
    P = np.zeros((L, L))
    for i in range(L):
        for j in range(i if strict else i + 1):
            if (i >> 2) == (j >> 2):  # inside a block of 4: running product of alpha
                pr = np.prod(al[j + 1:i + 1], axis=0) if i > j else np.ones(c)
                P[i, j] = np.sum(x[i] * y[j] * pr)
            else:
                p = (i ^ j).bit_length() - 1  # highest differing bit: half size h = 2^p
                h = 1 << p
                b = 2 * h * (i >> (p + 1)) + h - 1
                assert j <= b < i
                fi, fj = np.exp(lam[i] - lam[b]), np.exp(lam[b] - lam[j])
                assert fi.max() <= 1.0 + 1e-12 and fj.max() <= 1.0 + 1e-12
                P[i, j] = np.sum((x[i] * fi) * (y[j] * fj))
    return P


def chunk_step(S0, q, k, v, al, beta, e=None, w=None, gate=None):
    """One chunk (rows padded to C by the caller: k = q = v = 0, alpha = 1,
    beta = 0).  e, w: GDN2's erase rows e = b (.) k and write gates; gate:
    the SSE read scale of each row.  Returns (S_C, Y)."""
    lam = np.cumsum(np.log(al), axis=0)
    g2 = e is not None
    A = pair_sums(lam, al, e if g2 else k, k, strict=True)
    if not g2:
        A = beta[:, None] * A
    Mq = pair_sums(lam, al, q, k, strict=False)
    Linv = np.linalg.inv(np.eye(C) + A)
    T = Linv if g2 else Linv * beta[None, :]
    W = T @ ((e if g2 else k) * np.exp(lam))
    Ut = T @ (w * v if g2 else v)
    U = Ut - W @ S0
    Y = (q * np.exp(lam)) @ S0 + Mq @ U
    if gate is not None:
        Y = gate[:, None] * Y
    S = np.exp(lam[-1])[:, None] * S0 + (k * np.exp(lam[-1] - lam)).T @ U
    return S, Y


def pad(x, L, fill):
    out = np.full((C,) + x.shape[1:], fill, np.float64)
    out[:L] = x
    return out


def run_chunked(S0, q, k, v, al, beta, e=None, w=None, gate=None):
    """The whole sequence chunk by chunk (one (batch, head))."""
    S = np.array(S0, np.float64)
    T = q.shape[0]
    Y = np.zeros((T, v.shape[1]))
    for t0 in range(0, T, C):
        L = min(C, T - t0)
        sl = slice(t0, t0 + L)
        S, Yc = chunk_step(S, pad(q[sl], L, 0), pad(k[sl], L, 0), pad(v[sl], L, 0), pad(al[sl], L, 1),
                           pad(beta[sl], L, 0), None if e is None else pad(e[sl], L, 0),
                           None if w is None else pad(w[sl], L, 0), None if gate is None else pad(gate[sl], L, 0))
        Y[sl] = Yc[:L]
    return S, Y


def inputs(T, dk, dv, seed, strong=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, dk)) / np.sqrt(dk)
    k = rng.standard_normal((T, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv))
    x = rng.standard_normal((T, dk))
    al = np.exp(-(6.0 if strong else 0.3) * np.log1p(np.exp(x)))  # exp(-s softplus(N(0,1)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    S0 = 0.3 * rng.standard_normal((dk, dv))
    return S0, q, k, v, al, beta


def close(got, want, tol=1e-9):
    scale = max(1.0, float(np.max(np.abs(want))))
    assert np.max(np.abs(got - want)) <= tol * scale


@pytest.mark.parametrize("T", [1, 63, 64, 150])
@pytest.mark.parametrize("strong", [False, True], ids=["mild", "strong"])
def test_kda_chunk_form_matches_the_oracle(T, strong):
    dk, dv = 16, 12
    S0, q, k, v, al, beta = inputs(T, dk, dv, seed=T + 7 * strong, strong=strong)
    S, Y = run_chunked(S0, q, k, v, al, beta)
    Sr, Yr = oracle.gdn_scan(S0[None, None], q[None, :, None], k[None, :, None], v[None, :, None],
                             al[None, :, None], beta[None, :, None], True)
    close(Y, Yr[0, :, 0])
    close(S, Sr[0, 0])


@pytest.mark.parametrize("T", [5, 64, 150])
def test_gdn2_chunk_form_matches_the_oracle(T):
    dk, dv = 16, 12
    S0, q, k, v, al, _ = inputs(T, dk, dv, seed=40 + T)
    rng = np.random.default_rng(T)
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, dk))))
    w = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, dv))))
    S, Y = run_chunked(S0, q, k, v, al, np.zeros(T), e=b * k, w=w)
    Sr, Yr = oracle.gdn2_scan(S0[None, None], q[None, :, None], k[None, :, None], v[None, :, None],
                              al[None, :, None], b[None, :, None], w[None, :, None])
    close(Y, Yr[0, :, 0])
    close(S, Sr[0, 0])


def test_level_split_reaches_every_pair_once():
    """Every pair j < i of a chunk falls in exactly one place: a block of 4,
    or one level's segment with i in the right half and j in the left."""
    seen = np.zeros((C, C), int)
    for i in range(C):
        for j in range(i):
            if (i >> 2) == (j >> 2):
                seen[i, j] += 1
                continue
            for lvl in range(4):  # levels 0-3: half sizes 32, 16, 8, 4
                h = 32 >> lvl
                seg_i, seg_j = i // (2 * h), j // (2 * h)
                if seg_i == seg_j and (i % (2 * h)) >= h > (j % (2 * h)):
                    seen[i, j] += 1
    assert np.all(seen[np.tril_indices(C, -1)] == 1)


@pytest.mark.parametrize("T,N,topk", [(100, 4, 2), (150, 3, 1)])
def test_sse_delta_chunk_form_matches_the_oracle(T, N, topk):
    """The SSE delta write per partition: keys kk = softmax of the key logits,
    write strength = the visit's gate (1 on the shared partition), every read
    scaled by the gate; each token's output is the sum of its visits'."""
    c, d = 8, 6
    rng = np.random.default_rng(T + N)
    route = rng.standard_normal((T, N)).astype(np.float32)
    klog = rng.standard_normal((T, c)).astype(np.float32)
    q = rng.standard_normal((T, c))
    v = rng.standard_normal((T, d))
    al = 1.0 / (1.0 + np.exp(-(3.0 + rng.standard_normal((T, c)))))
    S0 = 0.5 * rng.standard_normal((N + 1, c, d))
    kl = klog.astype(np.float64)
    kk = np.exp(kl - kl.max(axis=1, keepdims=True))
    kk /= kk.sum(axis=1, keepdims=True)
    visits = [[] for _ in range(N + 1)]  # per partition: (token, gate)
    for t in range(T):
        lt = route[t].astype(np.float64)
        order = sorted(range(N), key=lambda p: (-float(route[t, p]), p))[:topk]
        ep = np.exp(lt - lt.max())
        ep /= ep.sum()
        for p in order:
            visits[p].append((t, ep[p]))
        visits[N].append((t, 1.0))
    Y = np.zeros((T, d))
    S = np.zeros_like(S0)
    for p in range(N + 1):
        if not visits[p]:
            S[p] = S0[p]
            continue
        ts = np.array([t for t, _ in visits[p]])
        g = np.array([gp for _, gp in visits[p]])
        S[p], Yp = run_chunked(S0[p], q[ts], kk[ts], v[ts], al[ts], g, gate=g)
        Y[ts] += Yp
    Sr, Yr, _ = oracle.sse_scan(S0[None, None], route[None, :, None], topk, klog[None, :, None], q[None, :, None],
                                v[None, :, None], al[None, :, None], oracle.SSE_WRITE_DELTA)
    close(Y, Yr[0, :, 0])
    close(S, Sr[0, 0])


def gdn_chunk_step(S0, q, k, v, al, beta):
    """The dense GDN chunk (a scalar decay per token; SDM deck App. A.1-A.2,
    Eq. 7, dense case) as the GDN preparation and chain form it: with
    gamma_i = e^{lambda_i}, A_ij = beta_i e^{lambda_i - lambda_j} k_i . k_j
    (j < i), T = (I + A)^-1 diag(beta), W = T diag(gamma) K, Ut = T V,
    U = Ut - W S0, Y = diag(gamma) Q S0 + Mq U (Mq_ij = e^{lambda_i -
    lambda_j} q_i . k_j, j <= i), S_C = gamma_C S0 + Khat^T U (Khat_j =
    e^{lambda_C - lambda_j} k_j)."""
    lam = np.cumsum(np.log(al))
    dec = np.exp(lam[:, None] - lam[None, :])
    A = np.tril(beta[:, None] * dec * (k @ k.T), -1)
    Mq = np.tril(dec * (q @ k.T))
    T = np.linalg.inv(np.eye(C) + A) * beta[None, :]
    gam = np.exp(lam)
    W = T @ (gam[:, None] * k)
    U = T @ v - W @ S0
    Y = gam[:, None] * (q @ S0) + Mq @ U
    S = gam[-1] * S0 + (np.exp(lam[-1] - lam)[:, None] * k).T @ U
    return S, Y


@pytest.mark.parametrize("T", [1, 64, 150])
def test_gdn_chunk_form_matches_the_oracle(T):
    dk, dv = 16, 12
    S0, q, k, v, al, beta = inputs(T, dk, dv, seed=90 + T)
    a = al[:, 0]  # one decay per token
    S = np.array(S0)
    Y = np.zeros((T, dv))
    for t0 in range(0, T, C):
        L = min(C, T - t0)
        sl = slice(t0, t0 + L)
        S, Yc = gdn_chunk_step(S, pad(q[sl], L, 0), pad(k[sl], L, 0), pad(v[sl], L, 0), pad(a[sl], L, 1),
                               pad(beta[sl], L, 0))
        Y[sl] = Yc[:L]
    Sr, Yr = oracle.gdn_scan(S0[None, None], q[None, :, None], k[None, :, None], v[None, :, None],
                             a[None, :, None], beta[None, :, None], False)
    close(Y, Yr[0, :, 0])
    close(S, Sr[0, 0])
