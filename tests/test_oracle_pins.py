"""Pins for the fp64 CPU oracle (no GPU).

The oracle is checked against things other than itself: values printed on
the pages (``tests/golden``), closed forms, special cases that reduce to a
different formulation, invariants, and brute force on tiny inputs.  Each test
names the passage it follows.
"""
import numpy as np
import pytest

import oracle
import synth

RNG = np.random.default_rng(1234)


def _one_token(arr):
    return np.asarray(arr, dtype=np.float64).reshape(1, 1, 1, -1)


# ---------------------------------------------------------------------------
# Sparse delta write: the two-slot worked example (SDM deck, backup frame
# "two slots expose the update discrepancy"; Eq. 4 vs Fig. 2).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode,key", [(oracle.RESID_PERSLOT, "per_slot"), (oracle.RESID_SHARED, "shared")])
def test_two_slot_worked_example(golden, mode, key):
    g = golden("two_slot_update.txt")
    M0 = np.array(g["m_prev"]).reshape(1, 1, 2, 1)
    v = np.array(g["v"]).reshape(1, 1, 1, 1)
    a = np.array(g["alpha"]).reshape(1, 1, 1)
    b = np.array(g["beta"]).reshape(1, 1, 1)
    idx = np.array([0, 1], np.int32).reshape(1, 1, 1, 2)
    w = np.array(g["k"]).reshape(1, 1, 1, 2)
    r = np.array([0.25, 0.75]).reshape(1, 1, 1, 2)
    M, y = oracle.sdm_scan(M0, v, a, b, idx, w, idx, r, mode)
    np.testing.assert_allclose(M.ravel(), g[key], rtol=0, atol=1e-12)
    np.testing.assert_allclose(y.ravel(), [0.25 * g[key][0] + 0.75 * g[key][1]], atol=1e-12)
    # the decayed rows the page prints, recovered from the additive mode with v = 0
    Md, _ = oracle.sdm_scan(M0, np.zeros_like(v), a, b, idx, w, idx, r, oracle.RESID_ADDITIVE)
    np.testing.assert_allclose(Md.ravel(), g["m_decayed"], atol=1e-12)


def test_shared_prediction_of_two_slot_example(golden):
    """v_hat = sum_j k_j M~[j] = 3: with beta*k = 1 on a single-slot write the
    new row equals v - v_hat + M~[i] ... checked instead through the read:
    shared mode with v = v_hat leaves every written row at its decayed value."""
    g = golden("two_slot_update.txt")
    M0 = np.array(g["m_prev"]).reshape(1, 1, 2, 1)
    idx = np.array([0, 1], np.int32).reshape(1, 1, 1, 2)
    w = np.array(g["k"]).reshape(1, 1, 1, 2)
    v = np.array(g["v_hat"]).reshape(1, 1, 1, 1)
    M, _ = oracle.sdm_scan(M0, v, np.full((1, 1, 1), g["alpha"][0]), np.full((1, 1, 1), g["beta"][0]),
                           idx, w, idx, w, oracle.RESID_SHARED)
    np.testing.assert_allclose(M.ravel(), g["m_decayed"], atol=1e-12)


def test_single_slot_write_makes_modes_identical():
    """With W = 1 the softmax weight is exactly 1, so the shared prediction is
    the slot itself and Fig. 2 and Eq. 4 coincide."""
    shape = synth.SDM_TINY.with_(T=32, W=1, R=3)
    inp = synth.sdm_inputs(shape, seed=7)
    idx_w, w_w = oracle.address(inp["s1w"], inp["s2w"], shape.k, 1)
    assert np.all(w_w == 1.0)
    idx_r, w_r = oracle.address(inp["s1r"], inp["s2r"], shape.k, 3)
    M0 = synth.random_state((1, 1, shape.N, shape.d_v), seed=3)
    a = oracle.sdm_scan(M0, inp["v"], inp["alpha"], inp["beta"], idx_w, w_w, idx_r, w_r, oracle.RESID_SHARED)
    b = oracle.sdm_scan(M0, inp["v"], inp["alpha"], inp["beta"], idx_w, w_w, idx_r, w_r, oracle.RESID_PERSLOT)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_modes_differ_for_multislot_writes():
    shape = synth.SDM_TINY.with_(T=16)
    inp = synth.sdm_inputs(shape, seed=8)
    M0 = synth.random_state((1, 1, shape.N, shape.d_v), seed=4)
    sh = oracle.sdm_forward(inp, shape.k, shape.W, shape.R, state=M0, mode=oracle.RESID_SHARED)
    ps = oracle.sdm_forward(inp, shape.k, shape.W, shape.R, state=M0, mode=oracle.RESID_PERSLOT)
    assert np.max(np.abs(sh["y"] - ps["y"])) > 1e-3


# ---------------------------------------------------------------------------
# DeltaNet teaching example and the gradient-step identities (Linear
# Attention Architectures deck, Eq. 14 and the backup "delta rule is a local
# gradient step").
# ---------------------------------------------------------------------------
def test_deltanet_teaching_example_dense(golden):
    g = golden("deltanet_teaching.txt")
    dk, dv = 6, 4
    S0 = synth.random_state((1, 1, dk, dv), seed=11).astype(np.float64)
    S0[0, 0, 2, :] = g["prediction"][0]          # prediction 2 at the unit key e_2
    k = np.zeros(dk); k[2] = 1.0
    S, y = oracle.gdn_scan(S0, _one_token(k), _one_token(k), _one_token(np.full(dv, g["target"][0])),
                           np.ones((1, 1, 1)), np.full((1, 1, 1), g["beta"][0]), per_channel=False)
    np.testing.assert_allclose(y.ravel(), g["new_prediction"][0], atol=1e-12)
    # only the row of the key moved
    keep = [r for r in range(dk) if r != 2]
    np.testing.assert_array_equal(S[0, 0, keep], S0[0, 0, keep])


@pytest.mark.parametrize("mode", [oracle.RESID_SHARED, oracle.RESID_PERSLOT])
def test_deltanet_teaching_example_sparse(golden, mode):
    g = golden("deltanet_teaching.txt")
    N, dv = 9, 3
    M0 = synth.random_state((1, 1, N, dv), seed=12).astype(np.float64)
    M0[0, 0, 5] = g["prediction"][0]
    idx = np.array([5], np.int32).reshape(1, 1, 1, 1)
    one = np.ones((1, 1, 1, 1))
    M, y = oracle.sdm_scan(M0, np.full((1, 1, 1, dv), g["target"][0]), np.ones((1, 1, 1)),
                           np.full((1, 1, 1), g["beta"][0]), idx, one, idx, one, mode)
    np.testing.assert_allclose(y.ravel(), g["new_prediction"][0], atol=1e-12)
    np.testing.assert_allclose(M[0, 0, 5], g["new_prediction"][0], atol=1e-12)


def test_gradient_step_identities():
    dk, dv = 16, 8
    S0 = RNG.standard_normal((1, 1, dk, dv))
    kap = RNG.standard_normal(dk); kap /= np.linalg.norm(kap)
    v = RNG.standard_normal(dv)
    u = RNG.standard_normal(dk)
    beta = 0.37
    S, _ = oracle.gdn_scan(S0, _one_token(kap), _one_token(kap), _one_token(v), np.ones((1, 1, 1)),
                           np.full((1, 1, 1), beta), per_channel=False)
    Wold, Wnew = S0[0, 0].T, S[0, 0].T         # W = S^T in R^{dv x dk}
    np.testing.assert_allclose(Wnew @ kap, (1 - beta) * (Wold @ kap) + beta * v, atol=1e-12)
    np.testing.assert_allclose((Wnew - Wold) @ u, beta * (v - Wold @ kap) * (kap @ u), atol=1e-12)


def test_gated_prediction_uses_decayed_state():
    """GDN residual is v - alpha W_old k (decay-adjusted): for a unit key the new
    prediction is (1-beta) alpha W_old k + beta v."""
    dk, dv = 12, 5
    S0 = RNG.standard_normal((1, 1, dk, dv))
    kap = RNG.standard_normal(dk); kap /= np.linalg.norm(kap)
    v = RNG.standard_normal(dv)
    alpha, beta = 0.83, 0.61
    S, y = oracle.gdn_scan(S0, _one_token(kap), _one_token(kap), _one_token(v), np.full((1, 1, 1), alpha),
                           np.full((1, 1, 1), beta), per_channel=False)
    np.testing.assert_allclose(y.ravel(), (1 - beta) * alpha * (S0[0, 0].T @ kap) + beta * v, atol=1e-12)


def test_gdn_closed_form_first_token():
    """From a zero state: S_1 = beta k v^T and y_1 = beta (k . q) v."""
    dk, dv = 10, 7
    k, q, v = RNG.standard_normal(dk), RNG.standard_normal(dk), RNG.standard_normal(dv)
    beta = 0.45
    S, y = oracle.gdn_scan(np.zeros((1, 1, dk, dv)), _one_token(q), _one_token(k), _one_token(v),
                           np.full((1, 1, 1), 0.7), np.full((1, 1, 1), beta), per_channel=False)
    np.testing.assert_allclose(S[0, 0], beta * np.outer(k, v), atol=1e-12)
    np.testing.assert_allclose(y.ravel(), beta * (k @ q) * v, atol=1e-12)


# ---------------------------------------------------------------------------
# KDA (Linear Attention Architectures deck, Eqs. 18-20): per-key-channel
# decay on the right of W, i.e. on the rows of S = W^T.
# ---------------------------------------------------------------------------
def test_kda_channel_decay_scales_rows():
    T, dk, dv = 9, 8, 5
    S0 = RNG.standard_normal((1, 1, dk, dv))
    a = RNG.uniform(0.5, 1.0, (1, T, 1, dk))
    q = RNG.standard_normal((1, T, 1, dk))
    S, y = oracle.gdn_scan(S0, q, RNG.standard_normal((1, T, 1, dk)), RNG.standard_normal((1, T, 1, dv)), a,
                           np.zeros((1, T, 1)), per_channel=True)
    np.testing.assert_allclose(S[0, 0], np.prod(a[0, :, 0, :], axis=0)[:, None] * S0[0, 0], rtol=1e-13)
    cum = np.cumprod(a[0, :, 0, :], axis=0)
    for t in range(T):
        np.testing.assert_allclose(y[0, t, 0], (cum[t][:, None] * S0[0, 0]).T @ q[0, t, 0], rtol=1e-12,
                                   atol=1e-12)


def test_kda_constant_vector_is_gdn():
    shape = synth.GDN_DENSE.with_(B=1, T=24, H=2, dk=16, dv=8)
    inp = synth.gdn_inputs(shape, seed=5)
    a_vec = np.repeat(inp["alpha_gdn"][..., None], shape.dk, axis=-1)
    S0 = synth.random_state((1, 2, 16, 8), seed=6)
    g = oracle.gdn_scan(S0, inp["q"], inp["k"], inp["v"], inp["alpha_gdn"], inp["beta"], per_channel=False)
    kd = oracle.gdn_scan(S0, inp["q"], inp["k"], inp["v"], a_vec, inp["beta"], per_channel=True)
    np.testing.assert_array_equal(g[0], kd[0])
    np.testing.assert_array_equal(g[1], kd[1])


@pytest.mark.parametrize("per_channel", [False, True])
def test_gdn_value_columns_evolve_independently(per_channel):
    """The prediction S~^T k and the read S^T q mix the key rows of the state
    only, never its value columns (Linear Attention Architectures deck, GDN
    and KDA updates): a scan over any subset of value columns reproduces
    those columns of the full scan exactly.  A transposed state or operand
    anywhere in the recurrence breaks this."""
    T, dk, dv = 12, 6, 7
    S0 = RNG.standard_normal((1, 1, dk, dv))
    q, k = RNG.standard_normal((1, T, 1, dk)), RNG.standard_normal((1, T, 1, dk))
    v = RNG.standard_normal((1, T, 1, dv))
    a = RNG.uniform(0.5, 1.0, (1, T, 1, dk) if per_channel else (1, T, 1))
    b = RNG.uniform(0.1, 0.9, (1, T, 1))
    S, y = oracle.gdn_scan(S0, q, k, v, a, b, per_channel=per_channel)
    cols = [1, 4, 6]
    Ss, ys = oracle.gdn_scan(np.ascontiguousarray(S0[..., cols]), q, k, np.ascontiguousarray(v[..., cols]), a, b,
                             per_channel=per_channel)
    np.testing.assert_array_equal(Ss, S[..., cols])
    np.testing.assert_array_equal(ys, y[..., cols])


# ---------------------------------------------------------------------------
# GDN2 (Linear Attention Architectures deck, "GDN2 separates key-side erase and
# value-side write", Eqs. 21-24): erase gate b on the key side, write gate w on
# the value side, outer product with the key itself.
# ---------------------------------------------------------------------------
def _gdn2_one(S0, k, q, v, alpha, b, w):
    return oracle.gdn2_scan(S0, _one_token(q), _one_token(k), _one_token(v), _one_token(alpha), _one_token(b),
                            _one_token(w))


def test_gdn2_gates_equal_to_beta_are_kda():
    """b = w = beta 1 recovers KDA (the deck's stated special case)."""
    shape = synth.GDN_DENSE.with_(B=2, T=30, H=2, dk=16, dv=8)
    inp = synth.gdn_inputs(shape, seed=21)
    S0 = synth.random_state((2, 2, 16, 8), seed=22)
    bb = np.repeat(inp["beta"][..., None], 16, axis=-1)
    ww = np.repeat(inp["beta"][..., None], 8, axis=-1)
    S2, y2 = oracle.gdn2_scan(S0, inp["q"], inp["k"], inp["v"], inp["alpha_kda"], bb, ww)
    Sk, yk = oracle.gdn_scan(S0, inp["q"], inp["k"], inp["v"], inp["alpha_kda"], inp["beta"], per_channel=True)
    np.testing.assert_allclose(S2, Sk, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(y2, yk, rtol=1e-12, atol=1e-13)


def test_gdn2_teaching_example(golden):
    """Prediction 2 at a unit key, target 5, b = w = 0.5: the DeltaNet teaching
    value 3.5; with the write gate opened to w = 1 (erase still 0.5) the
    prediction becomes 2 + (5 - 0.5 * 2) = 6: erase and write act separately."""
    g = golden("deltanet_teaching.txt")
    dk, dv = 5, 3
    S0 = synth.random_state((1, 1, dk, dv), seed=23).astype(np.float64)
    S0[0, 0, 1, :] = g["prediction"][0]
    k = np.zeros(dk); k[1] = 1.0
    v = np.full(dv, g["target"][0])
    half = g["beta"][0]
    S, y = _gdn2_one(S0, k, k, v, np.ones(dk), np.full(dk, half), np.full(dv, half))
    np.testing.assert_allclose(y.ravel(), g["new_prediction"][0], atol=1e-12)
    S, y = _gdn2_one(S0, k, k, v, np.ones(dk), np.full(dk, half), np.ones(dv))
    np.testing.assert_allclose(y.ravel(), 6.0, atol=1e-12)
    keep = [r for r in range(dk) if r != 1]
    np.testing.assert_array_equal(S[0, 0, keep], S0[0, 0, keep])


def test_gdn2_update_is_along_the_key_not_the_erase_vector():
    """W_new - W~ = r k^T: directions orthogonal to k see no change even when
    they are not orthogonal to e = b (.) k."""
    dk, dv = 12, 6
    S0 = RNG.standard_normal((1, 1, dk, dv))
    k = RNG.standard_normal(dk)
    b = RNG.uniform(0.05, 0.95, dk)
    S, _ = _gdn2_one(S0, k, RNG.standard_normal(dk), RNG.standard_normal(dv), np.ones(dk), b,
                     RNG.uniform(0.05, 0.95, dv))
    dS = S[0, 0] - S0[0, 0]                     # alpha = 1: S~ = S0
    u = RNG.standard_normal(dk); u -= (u @ k) / (k @ k) * k          # u orthogonal to k
    np.testing.assert_allclose(u @ dS, 0.0, atol=1e-12)
    e = b * k
    assert abs(u @ e) > 1e-3                    # ... yet not orthogonal to e
    assert np.linalg.norm(dS) > 1e-3


def test_gdn2_zero_erase_is_an_additive_write():
    """b = 0 and alpha = 1: S_T = S_0 + sum_t k_t (w_t (.) v_t)^T = S_0 + K^T (W (.) V)."""
    T, dk, dv = 7, 9, 4
    S0 = RNG.standard_normal((1, 1, dk, dv))
    k = RNG.standard_normal((1, T, 1, dk))
    v = RNG.standard_normal((1, T, 1, dv))
    w = RNG.uniform(0.1, 0.9, (1, T, 1, dv))
    S, _ = oracle.gdn2_scan(S0, RNG.standard_normal((1, T, 1, dk)), k, v, np.ones((1, T, 1, dk)),
                            np.zeros((1, T, 1, dk)), w)
    np.testing.assert_allclose(S[0, 0], S0[0, 0] + k[0, :, 0].T @ (w * v)[0, :, 0], rtol=1e-12, atol=1e-12)


def test_gdn2_full_gates_at_a_unit_key_reach_the_target():
    """b = w = 1, alpha = 1, unit-norm key: the new prediction at k is v."""
    dk, dv = 10, 5
    S0 = RNG.standard_normal((1, 1, dk, dv))
    k = RNG.standard_normal(dk); k /= np.linalg.norm(k)
    v = RNG.standard_normal(dv)
    S, y = _gdn2_one(S0, k, k, v, np.ones(dk), np.ones(dk), np.ones(dv))
    np.testing.assert_allclose(y.ravel(), v, atol=1e-12)


# ---------------------------------------------------------------------------
# Sparse <-> dense: with every row selected, weights k_t (write) and q_t (read)
# and the shared residual, the sparse table update is Gated DeltaNet (SDM deck,
# "A v1 inconsistency ...": only the shared residual gives the GDN limit).
# ---------------------------------------------------------------------------
def test_sparse_all_rows_selected_is_dense_gdn():
    B, T, H, dk, dv = 1, 20, 2, 8, 6
    shape = synth.GDN_DENSE.with_(B=B, T=T, H=H, dk=dk, dv=dv)
    inp = synth.gdn_inputs(shape, seed=9)
    S0 = synth.random_state((B, H, dk, dv), seed=10)
    Sg, yg = oracle.gdn_scan(S0, inp["q"], inp["k"], inp["v"], inp["alpha_gdn"], inp["beta"], per_channel=False)
    perm = RNG.permutation(dk).astype(np.int32)
    idx = np.broadcast_to(perm, (B, T, H, dk)).copy()
    kk, qq = oracle.widen(inp["k"]), oracle.widen(inp["q"])
    Ms, ys = oracle.sdm_scan(S0, inp["v"], inp["alpha_gdn"], inp["beta"], idx, kk[..., perm], idx, qq[..., perm],
                             oracle.RESID_SHARED)
    np.testing.assert_allclose(Ms, Sg, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ys, yg, rtol=1e-12, atol=1e-12)
    Mp, yp = oracle.sdm_scan(S0, inp["v"], inp["alpha_gdn"], inp["beta"], idx, kk[..., perm], idx, qq[..., perm],
                             oracle.RESID_PERSLOT)
    assert np.max(np.abs(yp - yg)) > 1e-3


# ---------------------------------------------------------------------------
# Persistence and closed forms of the sparse scan (SDM deck, Eqs. 3-5).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode", [oracle.RESID_SHARED, oracle.RESID_PERSLOT, oracle.RESID_ADDITIVE])
def test_untouched_rows_bit_unchanged(mode):
    shape = synth.SDM_TINY.with_(T=8)
    inp = synth.sdm_inputs(shape, seed=0)
    M0 = synth.random_state((1, 1, shape.N, shape.d_v), seed=1)
    out = oracle.sdm_forward(inp, shape.k, shape.W, shape.R, state=M0, mode=mode)
    written = np.unique(out["idx_w"])
    untouched = np.setdiff1d(np.arange(shape.N), written)
    assert untouched.size > 0
    np.testing.assert_array_equal(out["state"][0, 0, untouched], M0[0, 0, untouched].astype(np.float64))
    # read-only rows are read without decay: a row read but never written
    # contributes its initial value.
    assert np.setdiff1d(np.unique(out["idx_r"]), written).size > 0


@pytest.mark.parametrize("mode", [oracle.RESID_SHARED, oracle.RESID_PERSLOT, oracle.RESID_ADDITIVE])
def test_first_token_closed_form(mode):
    """From a zero table: M[i] = beta w_i v for i in I^w, and the read after the
    write gives y = beta (sum over I^w & I^r of r_i w_i) v."""
    N, dv = 20, 7
    iw = np.array([3, 11, 0, 17], np.int32)
    ir = np.array([11, 5, 17, 2, 9], np.int32)
    ww = RNG.dirichlet(np.ones(4))
    wr = RNG.dirichlet(np.ones(5))
    v = RNG.standard_normal(dv)
    beta = 0.66
    M, y = oracle.sdm_scan(np.zeros((1, 1, N, dv)), _one_token(v), np.full((1, 1, 1), 0.9),
                           np.full((1, 1, 1), beta), iw.reshape(1, 1, 1, 4), _one_token(ww), ir.reshape(1, 1, 1, 5),
                           _one_token(wr), mode)
    exp_M = np.zeros((N, dv))
    for j, i in enumerate(iw):
        exp_M[i] = beta * ww[j] * v
    np.testing.assert_allclose(M[0, 0], exp_M, atol=1e-14)
    coef = beta * (wr[0] * ww[1] + wr[2] * ww[3])
    np.testing.assert_allclose(y.ravel(), coef * v, atol=1e-14)


def test_rejects_repeated_or_out_of_range_slots():
    z = np.zeros((1, 1, 4, 2))
    one = np.ones((1, 1, 1))
    with pytest.raises(ValueError):
        oracle.sdm_scan(z, np.zeros((1, 1, 1, 2)), one, one, np.array([1, 1], np.int32).reshape(1, 1, 1, 2),
                        np.ones((1, 1, 1, 2)), np.array([0], np.int32).reshape(1, 1, 1, 1), np.ones((1, 1, 1, 1)))
    with pytest.raises(ValueError):
        oracle.sdm_scan(z, np.zeros((1, 1, 1, 2)), one, one, np.array([4], np.int32).reshape(1, 1, 1, 1),
                        np.ones((1, 1, 1, 1)), np.array([0], np.int32).reshape(1, 1, 1, 1), np.ones((1, 1, 1, 1)))


# ---------------------------------------------------------------------------
# Product-key addressing (SDM deck, "Product keys select addresses without
# scoring every slot"): top-W over the k^2 candidates equals brute force over
# all N outer sums when k >= W and no fp32 rounding tie can occur.
# ---------------------------------------------------------------------------
def _brute_force_topw(s1, s2, W):
    sq = s1.shape[-1]
    sums = (s1[:, None].astype(np.float32) + s2[None, :].astype(np.float32)).astype(np.float32).ravel()
    ids = np.arange(sq * sq)
    order = np.lexsort((ids, -sums.astype(np.float64)))
    return order[:W], sums


@pytest.mark.parametrize("sq,k,W,seed", [(8, 4, 4, 0), (16, 6, 5, 1), (12, 12, 12, 2), (8, 8, 1, 3)])
def test_address_matches_brute_force_dyadic(sq, k, W, seed):
    s1 = synth.dyadic_scores((2, 40, 3, sq), seed)
    s2 = synth.dyadic_scores((2, 40, 3, sq), seed + 100)
    idx, w = oracle.address(s1, s2, k, W)
    for r in np.ndindex(2, 40, 3):
        bf, _ = _brute_force_topw(s1[r], s2[r], W)
        np.testing.assert_array_equal(idx[r], bf)


def test_address_ties_broken_by_lower_index():
    """Integer scores in a tiny range: massive exact ties; the order must be
    (sum desc, flat id asc) and the per-half cut must prefer lower indices."""
    g = np.random.default_rng(5)
    s1 = g.integers(-2, 3, (1, 50, 2, 8)).astype(np.float32)
    s2 = g.integers(-2, 3, (1, 50, 2, 8)).astype(np.float32)
    idx, _ = oracle.address(s1, s2, 5, 5)
    for r in np.ndindex(1, 50, 2):
        bf, _ = _brute_force_topw(s1[r], s2[r], 5)
        np.testing.assert_array_equal(idx[r], bf)


def test_address_matches_brute_force_gaussian_without_ties():
    shape = synth.SDM_TINY.with_(T=200, H=2, sqrtN=16, k=8, W=8)
    inp = synth.sdm_inputs(shape, seed=3)
    idx, _ = oracle.address(inp["s1w"], inp["s2w"], shape.k, shape.W)
    checked = 0
    for r in np.ndindex(1, 200, 2):
        bf, sums = _brute_force_topw(inp["s1w"][r], inp["s2w"][r], shape.W + 1)
        top = sums[bf]
        if len(np.unique(top)) < len(top):
            continue                      # a rounding tie near the cut: skip
        np.testing.assert_array_equal(idx[r], bf[: shape.W])
        checked += 1
    assert checked > 350


def test_address_weights_are_softmax_of_selected_sums():
    shape = synth.SDM_TINY.with_(T=64)
    inp = synth.sdm_inputs(shape, seed=4)
    idx, w = oracle.address(inp["s1r"], inp["s2r"], shape.k, shape.R)
    np.testing.assert_allclose(w.sum(-1), 1.0, atol=1e-14)
    a, b = idx // shape.sqrtN, idx % shape.sqrtN
    s = (np.take_along_axis(inp["s1r"], a, -1) + np.take_along_axis(inp["s2r"], b, -1)).astype(np.float32)
    assert np.all(np.diff(s.astype(np.float64), axis=-1) <= 0)      # rank order
    ratio = w / w[..., :1]
    np.testing.assert_allclose(ratio, np.exp(s.astype(np.float64) - s[..., :1].astype(np.float64)), rtol=1e-13)


# ---------------------------------------------------------------------------
# Sparse State Expansion (SSE deck, Eqs. 9-14).
# ---------------------------------------------------------------------------
def test_sse_local_clock(golden):
    """A partition written once then visited 10 times in 100 tokens with v = 0
    keeps alpha^10 of its content; the always-active shared partition decays
    every token (alpha^100)."""
    g = golden("sse_local_clock.txt")
    a, T, visits = g["decay"][0], int(g["tokens"][0]), int(g["visits"][0])
    N, c, d = 4, 6, 3
    route = np.full((1, T, 1, N), -5.0, np.float32)
    visit_t = np.linspace(0, T - 1, visits).astype(int)
    route[0, :, 0, 1] = 3.0
    route[0, visit_t, 0, 0] = 4.0
    S0 = synth.random_state((1, 1, N + 1, c, d), seed=21) + 2.0
    S, y, sel = oracle.sse_scan(S0, route, 1, np.zeros((1, T, 1, c), np.float32), np.zeros((1, T, 1, c)),
                                np.zeros((1, T, 1, d)), np.full((1, T, 1, c), a))
    assert np.sum(sel == 0) == visits
    ratio0 = S[0, 0, 0] / S0[0, 0, 0]
    np.testing.assert_allclose(ratio0, a ** visits, rtol=1e-13)
    np.testing.assert_allclose(ratio0, g["sparse_retained"][0], atol=5e-4)
    np.testing.assert_allclose(S[0, 0, N] / S0[0, 0, N], g["dense_retained"][0], atol=5e-4)
    np.testing.assert_allclose(S[0, 0, 1] / S0[0, 0, 1], a ** (T - visits), rtol=1e-13)
    for p in (2, 3):                           # never visited: bit-unchanged
        np.testing.assert_array_equal(S[0, 0, p], S0[0, 0, p].astype(np.float64))


def test_sse_unit_decay_retains_exactly():
    N, c, d, T = 3, 4, 2, 57
    route = np.zeros((1, T, 1, N), np.float32)
    route[0, :, 0, 2] = 1.0
    S0 = synth.random_state((1, 1, N + 1, c, d), seed=22)
    S, _, _ = oracle.sse_scan(S0, route, 1, np.zeros((1, T, 1, c), np.float32), np.zeros((1, T, 1, c)),
                              np.zeros((1, T, 1, d)), np.ones((1, T, 1, c)))
    np.testing.assert_array_equal(S, S0.astype(np.float64))


def _softmax(x):
    x = np.asarray(x, np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


def test_sse_first_token_closed_form_and_gate_mass():
    """From zero state: o = (1 + sum_{p in T} e_p^2) (sum_j q_j kk_j) v, with e
    the softmax over ALL N logits (not renormalised) and kk the row softmax;
    the selected gate mass sum_{p in T} e_p is at most 1."""
    shape = synth.SSE_PART.with_(B=2, T=1, H=3, c=16, d=5)
    inp = synth.sse_inputs(shape, seed=2)
    S, y, sel = oracle.sse_scan(np.zeros((2, 3, shape.N + 1, 16, 5)), inp["route"], shape.topk, inp["klog"],
                                inp["q"], inp["v"], inp["alpha"])
    qf, vf = oracle.widen(inp["q"]), oracle.widen(inp["v"])
    for b, h in np.ndindex(2, 3):
        logit = inp["route"][b, 0, h]
        order = np.lexsort((np.arange(shape.N), -logit.astype(np.float64)))[: shape.topk]
        np.testing.assert_array_equal(sel[b, 0, h], order)
        e = _softmax(logit)
        assert e[order].sum() <= 1.0
        kk = _softmax(inp["klog"][b, 0, h])
        np.testing.assert_allclose(kk.sum(), 1.0, atol=1e-15)
        expect = (1.0 + np.sum(e[order] ** 2)) * (qf[b, 0, h] @ kk) * vf[b, 0, h]
        np.testing.assert_allclose(y[b, 0, h], expect, rtol=1e-12, atol=1e-14)


def test_sse_unvisited_partitions_bit_unchanged():
    shape = synth.SSE_PART.with_(B=1, T=40, H=2, N=8, c=8, d=4)
    inp = synth.sse_inputs(shape, seed=3)
    S0 = synth.random_state((1, 2, 9, 8, 4), seed=4)
    route = inp["route"].copy()
    route[..., 6:] = -50.0                  # partitions 6 and 7 never selected
    S, _, sel = oracle.sse_scan(S0, route, shape.topk, inp["klog"], inp["q"], inp["v"], inp["alpha"])
    assert not np.isin(sel, [6, 7]).any()
    np.testing.assert_array_equal(S[:, :, 6:8], S0[:, :, 6:8].astype(np.float64))


# ---------------------------------------------------------------------------
# Table sizes (SDM deck, Eq. 6 and the learned-state column of its table).
# ---------------------------------------------------------------------------
# ---------------------------------------------------------------------------
# SSE with a delta write: the partition's rows share one residual, the
# Sparse Delta Memory deck's shared residual (Fig. 2) with row weights kk and
# strength g.
# ---------------------------------------------------------------------------
def _one_hot_logits(c, row):
    kl = np.full(c, -1e30, np.float32)
    kl[row] = 0.0
    return kl


def test_sse_delta_teaching_example(golden):
    """Two routed partitions with equal logits (gates 1/2), top-1 picks the
    lower one; a one-hot key on row 0 holding prediction 2, target 5: the
    routed row becomes 2 + 0.5 (5 - 2) = 3.5 (the DeltaNet teaching value)
    and the shared partition (gate 1) reaches the target 5."""
    g = golden("deltanet_teaching.txt")
    N, c, d = 2, 4, 3
    S0 = synth.random_state((1, 1, N + 1, c, d), seed=41).astype(np.float64)
    S0[0, 0, 0, 0] = g["prediction"][0]
    S0[0, 0, N, 0] = g["prediction"][0]
    route = np.zeros((1, 1, 1, N), np.float32)
    klog = _one_hot_logits(c, 0).reshape(1, 1, 1, c)
    v = np.full((1, 1, 1, d), g["target"][0])
    S, _, sel = oracle.sse_scan(S0, route, 1, klog, np.zeros((1, 1, 1, c)), v, np.ones((1, 1, 1, c)),
                                oracle.SSE_WRITE_DELTA)
    assert sel.ravel().tolist() == [0]
    np.testing.assert_allclose(S[0, 0, 0, 0], g["new_prediction"][0], atol=1e-12)
    np.testing.assert_allclose(S[0, 0, N, 0], g["target"][0], atol=1e-12)
    np.testing.assert_array_equal(S[0, 0, 0, 1:], S0[0, 0, 0, 1:])     # rows with weight 0 keep their bits
    np.testing.assert_array_equal(S[0, 0, 1], S0[0, 0, 1])             # unvisited partition untouched


def test_sse_delta_is_the_sdm_shared_residual():
    """One routed partition (gate 1) and the shared one, decay equal across
    rows: each partition evolves exactly as the sparse scan with every row
    written (weights kk, beta = 1, shared residual) and read with weights q, so
    y is twice the sparse scan's read."""
    T, N, c, d = 12, 1, 6, 5
    rng = np.random.default_rng(42)
    S0p = rng.standard_normal((c, d))
    S0 = np.broadcast_to(S0p, (1, 1, N + 1, c, d)).copy()
    klog = rng.standard_normal((1, T, 1, c)).astype(np.float32)
    q = rng.standard_normal((1, T, 1, c))
    v = rng.standard_normal((1, T, 1, d))
    a_tok = rng.uniform(0.6, 1.0, (1, T, 1))
    alpha = np.repeat(a_tok[..., None], c, axis=-1)
    S, y, _ = oracle.sse_scan(S0, np.zeros((1, T, 1, N), np.float32), 1, klog, q, v, alpha, oracle.SSE_WRITE_DELTA)
    kl64 = klog.astype(np.float64)
    kk = np.exp(kl64 - kl64.max(axis=-1, keepdims=True))
    kk /= kk.sum(axis=-1, keepdims=True)
    idx = np.broadcast_to(np.arange(c, dtype=np.int32), (1, T, 1, c)).copy()
    M, ys = oracle.sdm_scan(S0p.reshape(1, 1, c, d), v, a_tok, np.ones((1, T, 1)), idx, kk, idx, q,
                            oracle.RESID_SHARED)
    np.testing.assert_allclose(S[0, 0, 0], M[0, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S[0, 0, N], M[0, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y, 2 * ys, rtol=1e-12, atol=1e-12)


def test_sse_delta_from_zero_state_first_token_is_additive():
    shape = synth.SSE_PART.with_(B=1, T=3, H=2, N=4, topk=2, c=16, d=8)
    inp = synth.sse_inputs(shape, seed=43)
    S0 = np.zeros((1, 2, 5, 16, 8))
    first = {k: v[:, :1] for k, v in inp.items()}
    Sa, ya, _ = oracle.sse_scan(S0, first["route"], 2, first["klog"], first["q"], first["v"], first["alpha"],
                                oracle.SSE_WRITE_ADDITIVE)
    Sd, yd, _ = oracle.sse_scan(S0, first["route"], 2, first["klog"], first["q"], first["v"], first["alpha"],
                                oracle.SSE_WRITE_DELTA)
    np.testing.assert_array_equal(Sa, Sd)
    np.testing.assert_array_equal(ya, yd)
    Sa, _, _ = oracle.sse_scan(S0, inp["route"], 2, inp["klog"], inp["q"], inp["v"], inp["alpha"],
                               oracle.SSE_WRITE_ADDITIVE)
    Sd, _, _ = oracle.sse_scan(S0, inp["route"], 2, inp["klog"], inp["q"], inp["v"], inp["alpha"],
                               oracle.SSE_WRITE_DELTA)
    assert np.max(np.abs(Sa - Sd)) > 1e-6           # later tokens see a nonzero prediction


def test_state_sizes(golden):
    g = golden("sdm_state_sizes.txt")
    for d, H, n_slots, layers, total, unit in g["rows"]:
        s = synth.sdm_layer_sizes(int(d), int(H))
        assert s["N"] == n_slots
        assert s["elements"] == d ** 3 / (16 * H * H)
        assert abs(s["elements"] * layers - total) <= unit / 2
    assert synth.SDM_14B_LAYER.N == 57600 and synth.SDM_14B_LAYER.d_v == 960
    for H, (n, dv) in {2: (57600, 960), 4: (14400, 480), 8: (3600, 240)}.items():
        sh = synth.sdm_sweep_shape(H)
        assert (sh.N, sh.d_v) == (n, dv)
        assert sh.H * sh.d_v == 1920


def test_tiny_config_runs_and_is_stable():
    shape = synth.SDM_TINY
    inp = synth.sdm_inputs(shape, seed=0)
    out = oracle.sdm_forward(inp, shape.k, shape.W, shape.R)
    assert np.all(np.isfinite(out["y"]))
    # the shared-residual transition alpha (I - beta w w^T) has eigenvalues in
    # [alpha (1 - beta |w|^2), alpha] for |w|_2 <= 1, so the table stays bounded
    assert np.max(np.abs(out["state"])) <= 10 * np.max(np.abs(inp["v"]))
