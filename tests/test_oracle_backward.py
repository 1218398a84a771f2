"""Pins of the backward oracle of the sparse scan (undoing the writes, Sparse
Delta Memory deck, "Backup: undoing writes avoids repeated full-table
snapshots", App. A.3) against central finite differences of the forward
oracle, on tiny inputs, in all three residual modes; and the exact
restoration of the initial table from the forward's log."""
import numpy as np
import pytest

import oracle

MODES = [oracle.RESID_SHARED, oracle.RESID_PERSLOT, oracle.RESID_ADDITIVE]


def _case(seed, used=10):
    """B=1, H=2, T=6 tokens over N=10 rows (slots drawn from the first `used`),
    W=3 written and R=2 read slots per token: rows are rewritten by later
    tokens, and at t = 2 a token reads a row it writes."""
    rng = np.random.default_rng(seed)
    B, T, H, N, dv, W, R = 1, 6, 2, 10, 3, 3, 2
    iw = np.stack([rng.permutation(used)[:W] for _ in range(B * T * H)]).reshape(B, T, H, W).astype(np.int32)
    ir = np.stack([rng.permutation(used)[:R] for _ in range(B * T * H)]).reshape(B, T, H, R).astype(np.int32)
    ir[0, 2, :, 0] = iw[0, 2, :, 1]
    return {
        "M0": rng.standard_normal((B, H, N, dv)),
        "v": rng.standard_normal((B, T, H, dv)),
        "alpha": rng.uniform(0.5, 1.0, (B, T, H)),
        "beta": rng.uniform(0.2, 0.9, (B, T, H)),
        "w_w": rng.uniform(0.1, 0.6, (B, T, H, W)),
        "w_r": rng.uniform(-1.0, 1.0, (B, T, H, R)),
        "iw": iw, "ir": ir,
        "dy": rng.standard_normal((B, T, H, dv)),
        "dMT": rng.standard_normal((B, H, N, dv)),
    }


def _loss(c, mode, **over):
    x = dict(c, **over)
    M, y = oracle.sdm_scan(x["M0"], x["v"], x["alpha"], x["beta"], x["iw"], x["w_w"], x["ir"], x["w_r"], mode)
    return float((c["dy"] * y).sum() + (c["dMT"] * M).sum())


def _fd(c, mode, name, eps=1e-6):
    base = c[name]
    g = np.zeros_like(base)
    it = np.nditer(base, flags=["multi_index"])
    for _ in it:
        ix = it.multi_index
        up, dn = base.copy(), base.copy()
        up[ix] += eps
        dn[ix] -= eps
        g[ix] = (_loss(c, mode, **{name: up}) - _loss(c, mode, **{name: dn})) / (2 * eps)
    return g


@pytest.mark.parametrize("mode", MODES)
def test_backward_matches_finite_differences(mode):
    c = _case(7 + mode)
    MT, _, undo = oracle.sdm_scan(c["M0"], c["v"], c["alpha"], c["beta"], c["iw"], c["w_w"], c["ir"], c["w_r"], mode,
                                  keep_undo=True)
    M0, dM0, dv, da, db, dww, dwr = oracle.sdm_scan_backward(MT, c["dMT"], c["v"], c["alpha"], c["beta"], c["iw"],
                                                             c["w_w"], c["ir"], c["w_r"], mode, undo, c["dy"])
    for name, got in (("M0", dM0), ("v", dv), ("alpha", da), ("beta", db), ("w_w", dww), ("w_r", dwr)):
        np.testing.assert_allclose(got, _fd(c, mode, name), rtol=1e-6, atol=1e-7, err_msg=f"d{name}")


@pytest.mark.parametrize("mode", MODES)
def test_undo_restores_the_initial_table_exactly(mode):
    c = _case(20 + mode)
    MT, _, undo = oracle.sdm_scan(c["M0"], c["v"], c["alpha"], c["beta"], c["iw"], c["w_w"], c["ir"], c["w_r"], mode,
                                  keep_undo=True)
    M0, *_ = oracle.sdm_scan_backward(MT, c["dMT"], c["v"], c["alpha"], c["beta"], c["iw"], c["w_w"], c["ir"],
                                      c["w_r"], mode, undo, c["dy"])
    np.testing.assert_array_equal(M0, c["M0"])


def test_unwritten_rows_pass_their_gradient_through():
    """Row 9, which no token writes or reads: dL/dM_0 = dL/dM_T there."""
    c = _case(31, used=9)
    MT, _, undo = oracle.sdm_scan(c["M0"], c["v"], c["alpha"], c["beta"], c["iw"], c["w_w"], c["ir"], c["w_r"],
                                  oracle.RESID_SHARED, keep_undo=True)
    _, dM0, *_ = oracle.sdm_scan_backward(MT, c["dMT"], c["v"], c["alpha"], c["beta"], c["iw"], c["w_w"], c["ir"],
                                          c["w_r"], oracle.RESID_SHARED, undo, c["dy"])
    np.testing.assert_array_equal(dM0[:, :, 9], c["dMT"][:, :, 9])
    assert np.max(np.abs(dM0[:, :, :9] - c["dMT"][:, :, :9])) > 1e-3   # the touched rows do change


def test_address_backward_matches_finite_differences():
    """Scores drawn so that no k-th or W-th value is within 1e-3 of the next:
    small perturbations keep the selection, and d(sum dw * w) / d(scores)
    is the softmax backward scattered to the two halves."""
    rng = np.random.default_rng(77)
    sq, k, W = 8, 4, 6
    s1 = (rng.permutation(sq) * 0.37 + rng.uniform(0, 0.01, sq)).astype(np.float32).reshape(1, 1, 1, sq)
    s2 = (rng.permutation(sq) * 0.53 + rng.uniform(0, 0.01, sq)).astype(np.float32).reshape(1, 1, 1, sq)
    dw = rng.standard_normal((1, 1, 1, W))
    idx, w = oracle.address(s1, s2, k, W)
    ds1, ds2 = oracle.address_backward(idx, w, dw, sq)
    eps = 1e-3                                   # fp32 scores: a coarse but exact-enough step
    for which, base in (("s1", s1), ("s2", s2)):
        for a in range(sq):
            up, dn = base.copy(), base.copy()
            up[..., a] += eps
            dn[..., a] -= eps
            args_up = (up, s2) if which == "s1" else (s1, up)
            args_dn = (dn, s2) if which == "s1" else (s1, dn)
            iu, wu = oracle.address(*args_up, k, W)
            idn, wd = oracle.address(*args_dn, k, W)
            assert (iu == idx).all() and (idn == idx).all()
            fd = ((wu - wd) * dw).sum() / (float(up[..., a].item()) - float(dn[..., a].item()))
            got = (ds1 if which == "s1" else ds2)[0, 0, 0, a]
            np.testing.assert_allclose(got, fd, rtol=1e-4, atol=1e-6)


def test_address_backward_is_zero_outside_the_selection():
    rng = np.random.default_rng(78)
    shape = (2, 3, 2, 16)
    s1 = rng.standard_normal(shape).astype(np.float32)
    s2 = rng.standard_normal(shape).astype(np.float32)
    idx, w = oracle.address(s1, s2, 4, 5)
    ds1, ds2 = oracle.address_backward(idx, w, rng.standard_normal(idx.shape), 16)
    sel_a = np.zeros(shape, bool)
    sel_b = np.zeros(shape, bool)
    for ix in np.ndindex(idx.shape[:-1]):
        sel_a[ix][idx[ix] // 16] = True
        sel_b[ix][idx[ix] % 16] = True
    assert np.all(ds1[~sel_a] == 0) and np.all(ds2[~sel_b] == 0)
    # softmax weights sum to one: a constant shift of all dw changes nothing
    d1b, d2b = oracle.address_backward(idx, w, rng.standard_normal(idx.shape) * 0 + 3.0, 16)
    np.testing.assert_allclose(d1b, 0.0, atol=1e-12)
    np.testing.assert_allclose(d2b, 0.0, atol=1e-12)
