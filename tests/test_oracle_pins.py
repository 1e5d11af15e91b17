"""Pins for the fp64 oracle, checked against things other than itself:
textbook values, hand-worked examples, the pages' shard identity, finite
differences and a brute-force loop.  No GPU needed."""
import math

import numpy as np
import pytest

from oracle import mlp as O


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def _problem(seed=0, T=3, h=4, f=8, ln=True, bias=True, wscale=0.7):
    rng = np.random.default_rng(seed)
    p = dict(X=_rand(rng, T, h), A=_rand(rng, h, f, scale=wscale),
             B=_rand(rng, f, h, scale=wscale), dZ=_rand(rng, T, h))
    p["b1"] = _rand(rng, f) if bias else None
    p["b2"] = _rand(rng, h) if bias else None
    if ln:
        p["gamma"] = 1.0 + 0.3 * _rand(rng, h)
        p["beta"] = 0.3 * _rand(rng, h)
    else:
        p["gamma"] = p["beta"] = None
    return p


# -------------------------------------------------------------- GeLU ----

def test_gelu_matches_normal_table(golden):
    """GeLU(x) = x Phi(x), GeLU'(x) = Phi(x) + x phi(x), at tabulated x."""
    for x, cdf, pdf in golden("normal_cdf.txt"):
        assert abs(float(O.gelu(x)) - x * cdf) <= 1e-15 * max(1, abs(x)) + 1e-16
        assert abs(float(O.gelu_grad(x)) - (cdf + x * pdf)) <= 2e-15


def test_gelu_special_values():
    assert O.gelu(0.0) == 0.0
    assert O.gelu_grad(0.0) == 0.5
    big = np.array([40.0, 100.0])
    assert np.all(O.gelu(big) == big)            # GeLU(x) -> x for x >> 0
    assert np.all(O.gelu(-big) == 0.0)           # GeLU(x) -> 0 for x << 0
    assert np.all(O.gelu_grad(big) == 1.0)
    for mode in ("erf", "tanh"):
        assert O.gelu(0.0, mode) == 0.0
        assert abs(O.gelu_grad(0.0, mode) - 0.5) < 1e-15


def test_gelu_tanh_is_close_to_exact():
    """The tanh form approximates x Phi(x) to a few 1e-4 everywhere."""
    x = np.linspace(-8, 8, 20001)
    err = np.abs(O.gelu(x, "tanh") - O.gelu(x, "erf"))
    assert err.max() < 1e-3
    assert err.max() > 1e-6                      # it is a different function


@pytest.mark.parametrize("mode", ["erf", "tanh"])
def test_gelu_grad_finite_difference(mode):
    x = np.linspace(-6, 6, 241)
    eps = 1e-6
    fd = (O.gelu(x + eps, mode) - O.gelu(x - eps, mode)) / (2 * eps)
    np.testing.assert_allclose(O.gelu_grad(x, mode), fd, rtol=1e-8, atol=1e-9)


# --------------------------------------------------------- LayerNorm ----

def test_layernorm_hand_example(golden):
    rows = golden("layernorm_example.txt")
    x = np.array([[r[0] for r in rows]])
    want = np.array([[r[1] for r in rows]])
    h = x.shape[1]
    xn, mean, rstd = O.layernorm_forward(x, np.ones(h), np.zeros(h), eps=0.0)
    np.testing.assert_allclose(xn, want, rtol=0, atol=1e-15)
    assert mean[0] == 2.5
    assert abs(rstd[0] - 2 / math.sqrt(5)) < 1e-15


def test_layernorm_constant_rows_give_beta():
    h = 16
    beta = np.linspace(-1, 1, h)
    gamma = np.linspace(0.5, 2, h)
    x = np.full((3, h), 7.25)
    xn, _, _ = O.layernorm_forward(x, gamma, beta, eps=1e-5)
    np.testing.assert_array_equal(xn, np.broadcast_to(beta, xn.shape))


def test_layernorm_output_moments():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 64)) * 3 + 11
    xn, _, _ = O.layernorm_forward(x, np.ones(64), np.zeros(64), eps=0.0)
    np.testing.assert_allclose(xn.mean(axis=1), 0, atol=1e-13)
    np.testing.assert_allclose((xn ** 2).mean(axis=1), 1, atol=1e-13)


# ------------------------------------------------ brute force forward ----

def _brute_forward(X, A, B, b1, b2, gamma, beta, eps, mode, residual=False):
    """Per-element loops with math.erf / math.tanh; no numpy, no helpers
    from the oracle."""
    T, h = len(X), len(X[0])
    f = len(A[0])
    Z = [[0.0] * h for _ in range(T)]
    for r in range(T):
        row = list(X[r])
        if gamma is not None:
            mu = sum(row) / h
            var = sum((v - mu) ** 2 for v in row) / h
            s = 1.0 / math.sqrt(var + eps)
            row = [(row[c] - mu) * s * gamma[c] + beta[c] for c in range(h)]
        for j in range(f):
            acc = 0.0
            for c in range(h):
                acc += row[c] * A[c][j]
            if b1 is not None:
                acc += b1[j]
            if mode == "erf":
                y = acc * 0.5 * (1.0 + math.erf(acc / math.sqrt(2.0)))
            else:
                u = math.sqrt(2.0 / math.pi) * (acc + 0.044715 * acc ** 3)
                y = 0.5 * acc * (1.0 + math.tanh(u))
            for c in range(h):
                Z[r][c] += y * B[j][c]
        if b2 is not None:
            for c in range(h):
                Z[r][c] += b2[c]
        if residual:
            for c in range(h):
                Z[r][c] += X[r][c]
    return np.array(Z)


@pytest.mark.parametrize("ln,bias,mode,res", [(False, False, "erf", False),
                                              (True, True, "erf", False),
                                              (True, False, "tanh", False),
                                              (False, True, "tanh", False),
                                              (True, True, "erf", True),
                                              (False, False, "tanh", True)])
def test_forward_matches_brute_force(ln, bias, mode, res):
    p = _problem(seed=3, T=3, h=5, f=7, ln=ln, bias=bias)
    got = O.forward(p["X"], p["A"], p["B"], p["b1"], p["b2"], p["gamma"],
                    p["beta"], eps=1e-5, mode=mode, residual=res)["Z"]
    want = _brute_forward(p["X"].tolist(), p["A"].tolist(), p["B"].tolist(),
                          None if p["b1"] is None else p["b1"].tolist(),
                          None if p["b2"] is None else p["b2"].tolist(),
                          None if p["gamma"] is None else p["gamma"].tolist(),
                          None if p["beta"] is None else p["beta"].tolist(),
                          1e-5, mode, res)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-14)


# ------------------------------------------- gradients: finite diffs ----

def _loss(p, mode, res=False):
    z = O.forward(p["X"], p["A"], p["B"], p["b1"], p["b2"], p["gamma"],
                  p["beta"], eps=1e-5, mode=mode, residual=res)["Z"]
    return float((z * p["dZ"]).sum())


@pytest.mark.parametrize("mode,res", [("erf", False), ("tanh", False),
                                      ("erf", True)])
@pytest.mark.parametrize("ln", [False, True])
def test_backward_matches_central_differences(mode, ln, res):
    """Every gradient entry of L = sum(Z * dZ) against central differences."""
    p = _problem(seed=5, T=3, h=4, f=8, ln=ln, bias=True)
    fwd = O.forward(p["X"], p["A"], p["B"], p["b1"], p["b2"], p["gamma"],
                    p["beta"], eps=1e-5, mode=mode, residual=res)
    g = O.backward(p["dZ"], p["X"], p["A"], p["B"], fwd, p["gamma"], mode,
                   residual=res)
    names = {"X": "dX", "A": "dA", "B": "dB", "b1": "db1", "b2": "db2"}
    if ln:
        names.update(gamma="dgamma", beta="dbeta")
    for pname, gname in names.items():
        base = p[pname]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            step = 1e-5 * max(1.0, abs(base[idx]))
            keep = base[idx]
            base[idx] = keep + step
            lp = _loss(p, mode, res)
            base[idx] = keep - step
            lm = _loss(p, mode, res)
            base[idx] = keep
            fd[idx] = (lp - lm) / (2 * step)
        scale = max(1.0, np.abs(fd).max())
        np.testing.assert_allclose(g[gname], fd, rtol=0, atol=2e-8 * scale,
                                   err_msg=pname)


# ------------------------------------ the pages' shard identity (f/g) ----

@pytest.mark.parametrize("t", [1, 2, 4, 8])
@pytest.mark.parametrize("ln,bias,res", [(False, False, False), (True, True, False),
                                         (True, True, True)])
def test_shard_identity_forward_and_backward(t, ln, bias, res):
    """sum_i GeLU(X A_i) B_i = GeLU(X A) B, and the f/g backward (dZ to
    every shard, dX = sum_i dX_i) gives the unsharded gradients."""
    p = _problem(seed=11, T=6, h=8, f=32, ln=ln, bias=bias)
    args = (p["X"], p["A"], p["B"])
    full = O.forward(*args, b1=p["b1"], b2=p["b2"], gamma=p["gamma"],
                     beta=p["beta"], residual=res)
    sh = O.forward_sharded(*args, t, b1=p["b1"], b2=p["b2"], gamma=p["gamma"],
                           beta=p["beta"], residual=res)
    assert len(sh["Z_parts"]) == t
    np.testing.assert_allclose(sh["Z"], full["Z"], rtol=1e-12, atol=1e-13)
    gf = O.backward(p["dZ"], *args, full, p["gamma"], residual=res)
    gs = O.backward_sharded(p["dZ"], *args, t, sh, p["gamma"], residual=res)
    assert len(gs["dXn_parts"]) == t
    for k in ("dX", "dA", "dB", "db1", "db2") + (("dgamma", "dbeta") if ln else ()):
        np.testing.assert_allclose(gs[k], gf[k], rtol=1e-12, atol=1e-13, err_msg=k)


def test_single_shard_partial_is_the_whole_output():
    """t = 1: the one partial product is already the output (no reduction)."""
    p = _problem(seed=2, T=4, h=8, f=16, ln=False, bias=False)
    sh = O.forward_sharded(p["X"], p["A"], p["B"], 1)
    np.testing.assert_array_equal(sh["Z_parts"][0], sh["Z"])


def test_row_split_of_first_gemm_is_not_equivalent():
    """Splitting A by rows would need a sync before GeLU:
    GeLU(X1 A1 + X2 A2) != GeLU(X1 A1) + GeLU(X2 A2)."""
    p = _problem(seed=4, T=5, h=8, f=16, ln=False, bias=False, wscale=1.0)
    X, A = p["X"], p["A"]
    X1, X2, A1, A2 = X[:, :4], X[:, 4:], A[:4], A[4:]
    joint = O.gelu(X1 @ A1 + X2 @ A2)
    split = O.gelu(X1 @ A1) + O.gelu(X2 @ A2)
    np.testing.assert_allclose(joint, O.gelu(X @ A), rtol=1e-13, atol=1e-14)
    assert np.abs(joint - split).max() > 0.1


# ---------------------------------------------------- special cases ----

def test_zero_first_weight():
    """A = 0 (no b1): H = 0, Y = GeLU(0) = 0, so Z = b2, dB = 0, dX = 0 and
    dA = GeLU'(0) Xn^T dZ B^T = 0.5 Xn^T dZ B^T."""
    p = _problem(seed=6, T=5, h=4, f=8, ln=False, bias=True)
    A0 = np.zeros_like(p["A"])
    fwd = O.forward(p["X"], A0, p["B"], None, p["b2"])
    np.testing.assert_array_equal(fwd["Z"], np.broadcast_to(p["b2"], fwd["Z"].shape))
    g = O.backward(p["dZ"], p["X"], A0, p["B"], fwd)
    assert np.all(g["dX"] == 0) and np.all(g["dB"] == 0)
    np.testing.assert_allclose(g["dA"], 0.5 * p["X"].T @ p["dZ"] @ p["B"].T,
                               rtol=1e-14, atol=1e-15)


def test_zero_first_weight_with_residual_is_identity_plus_bias():
    """Residual sub-block with A = 0 (no b1): Z = X + b2 and dX = dZ."""
    p = _problem(seed=7, T=4, h=4, f=8, ln=True, bias=True)
    A0 = np.zeros_like(p["A"])
    fwd = O.forward(p["X"], A0, p["B"], None, p["b2"], p["gamma"], p["beta"],
                    residual=True)
    np.testing.assert_array_equal(fwd["Z"], p["X"] + p["b2"][None, :])
    g = O.backward(p["dZ"], p["X"], A0, p["B"], fwd, p["gamma"], residual=True)
    np.testing.assert_array_equal(g["dX"], p["dZ"])


def test_empty_token_set():
    h, f = 4, 8
    X = np.zeros((0, h))
    A = np.ones((h, f))
    B = np.ones((f, h))
    fwd = O.forward(X, A, B)
    assert fwd["Z"].shape == (0, h)
    g = O.backward(np.zeros((0, h)), X, A, B, fwd)
    assert np.all(g["dA"] == 0) and np.all(g["dB"] == 0) and np.all(g["db2"] == 0)


# ------------------------- sampled evaluators equal the full definition ----

@pytest.mark.parametrize("ln", [False, True])
def test_sampled_evaluators_match_full(ln):
    p = _problem(seed=9, T=20, h=16, f=48, ln=ln, bias=True)
    kw = dict(b1=p["b1"], gamma=p["gamma"], beta=p["beta"])
    fwd = O.forward(p["X"], p["A"], p["B"], p["b1"], p["b2"], p["gamma"], p["beta"])
    g = O.backward(p["dZ"], p["X"], p["A"], p["B"], fwd, p["gamma"])
    rows = np.array([0, 7, 19])
    cols = np.array([1, 30, 47])
    np.testing.assert_allclose(
        O.forward_rows(p["X"], p["A"], p["B"], rows, b2=p["b2"], **kw),
        fwd["Z"][rows], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(
        O.dxn_rows(p["dZ"], p["X"], p["A"], p["B"], rows, **kw),
        g["dXn"][rows], rtol=1e-13, atol=1e-13)
    dac, db1c = O.dA_cols(p["dZ"], p["X"], p["A"], p["B"], cols, **kw)
    np.testing.assert_allclose(dac, g["dA"][:, cols], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(db1c, g["db1"][cols], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(
        O.dB_rows(p["dZ"], p["X"], p["A"], cols, **kw), g["dB"][cols],
        rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(O.db2(p["dZ"]), g["db2"], rtol=1e-14, atol=1e-14)
