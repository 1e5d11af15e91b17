"""fp64 CPU oracle for the Megatron-LM tensor-parallel transformer MLP block.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library.

What it computes, and where each piece comes from:

* "Megatron-LM" explainer (azimuth.plus/paper/megatron-lm), section "The core
  idea: slicing the feed-forward network across units": the MLP computes
  Y = GeLU(X A) and Z = Dropout(Y B).  A is split by columns,
  A = [A_1 ... A_t], so every shard applies GeLU to X A_i on its own; B is
  split by rows so the partial products need a single all-reduce at the end.
  The Megatron-LM paper notes (notes.yuuk.io), section "MLP block split",
  state the same split and the single all-reduce per direction.
* Same explainer, section "The f and g operators: two lines of code": f is
  the identity going forward and an all-reduce of gradients going backward;
  g is an all-reduce of partial outputs going forward and the identity going
  backward.
* Same explainer, section "Fixing BERT: reordering layer normalisation for
  scaling", and the notes' section "Changing the placement of layer
  normalisation (BERT scaling)": LayerNorm is applied to the input of the
  sub-block (pre-LN) and the residual path carries the raw input, added
  linearly: the whole sub-block is X + MLP(LN(X)) (``residual=True``).

Readings where the pages are silent (each is listed in the design notes):

* "GeLU" is the exact x * Phi(x) by default; the tanh approximation of
  Hendrycks & Gimpel (2016) is available as ``mode="tanh"``.
* Biases: b1 [f] (split by columns with A) is added before GeLU; b2 [h] is
  added once, after the sum over shards.  Both are optional.
* Dropout (``dropout=(p, seed, offset)``, training only) acts on the MLP's
  output Y B + b2 before the residual add, outside the parallel region, so
  its mask must not depend on the shard count (the notes' "Implementation
  features": dropout seeds differ inside and outside the model-parallel
  region).  Mask: element (r, c) is kept when word c % 4 of
  Philox4x32-10(counter = (c // 4, r, offset_lo, offset_hi),
  key = (seed_lo, seed_hi)) is >= floor(p 2^32); kept values are scaled by
  1 / (1 - p).  No workload uses it (p = 0).
* LayerNorm uses the biased variance over h and eps inside the square root.

The method is an exact re-association of the unsharded block, so the
reference result is the unsharded block written out in fp64
(``forward``/``backward``).  ``forward_sharded``/``backward_sharded`` follow
the pages' f/g decomposition literally; the tests check that the two agree.
Library primitives used as steps: numpy matmul (BLAS dgemm) and
``scipy.special.erf``.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf

from .philox import philox4x32_10

_SQRT1_2 = 1.0 / math.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)
_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
_TANH_C = 0.044715


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor -> fp64 numpy (widening only)
        return a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------- GeLU ----

def gelu(x, mode: str = "erf"):
    """GeLU(x) = x * Phi(x) (exact) or its tanh approximation."""
    x = np.asarray(x, dtype=np.float64)
    if mode == "erf":
        return 0.5 * x * (1.0 + _erf(x * _SQRT1_2))
    if mode == "tanh":
        u = _SQRT_2_OVER_PI * (x + _TANH_C * x ** 3)
        return 0.5 * x * (1.0 + np.tanh(u))
    raise ValueError(mode)


def gelu_grad(x, mode: str = "erf"):
    """d GeLU / dx.  Exact: Phi(x) + x * phi(x)."""
    x = np.asarray(x, dtype=np.float64)
    if mode == "erf":
        cdf = 0.5 * (1.0 + _erf(x * _SQRT1_2))
        pdf = _INV_SQRT_2PI * np.exp(-0.5 * x * x)
        return cdf + x * pdf
    if mode == "tanh":
        u = _SQRT_2_OVER_PI * (x + _TANH_C * x ** 3)
        th = np.tanh(u)
        du = _SQRT_2_OVER_PI * (1.0 + 3.0 * _TANH_C * x * x)
        return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * du
    raise ValueError(mode)


# ----------------------------------------------------------- LayerNorm ----

def layernorm_forward(X, gamma, beta, eps: float = 1e-5):
    """Per-token LayerNorm over the hidden axis.

    Returns (Xn, mean, rstd) with Xn = (X - mean) * rstd * gamma + beta,
    mean and the biased variance taken over h, rstd = 1/sqrt(var + eps).
    """
    X = _f64(X)
    mean = X.mean(axis=1)
    var = ((X - mean[:, None]) ** 2).mean(axis=1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (X - mean[:, None]) * rstd[:, None]
    return xhat * _f64(gamma)[None, :] + _f64(beta)[None, :], mean, rstd


def layernorm_backward(dXn, X, mean, rstd, gamma):
    """Gradients of LayerNorm: returns (dX, dgamma, dbeta).

    With xhat = (x - mean) * rstd and g = gamma * dXn (per row of h values):
    dX = rstd * (g - mean(g) - xhat * mean(g * xhat)),
    dgamma = sum over tokens of dXn * xhat, dbeta = sum over tokens of dXn.
    """
    dXn, X = _f64(dXn), _f64(X)
    xhat = (X - mean[:, None]) * rstd[:, None]
    g = dXn * _f64(gamma)[None, :]
    c_g = g.mean(axis=1)
    c_gx = (g * xhat).mean(axis=1)
    dX = rstd[:, None] * (g - c_g[:, None] - xhat * c_gx[:, None])
    return dX, (dXn * xhat).sum(axis=0), dXn.sum(axis=0)


# ------------------------------------------------------------- dropout ----

def dropout_threshold(p: float) -> int:
    """Keep an element when its 32-bit draw is >= floor(p * 2^32)."""
    return min(int(p * 4294967296.0), 0xFFFFFFFF)


def dropout_mask(rows, cols, p, seed, offset=0):
    """Boolean keep-mask for token rows `rows` (array) and `cols` columns."""
    rows = np.asarray(rows, dtype=np.uint64)
    c = np.arange(cols, dtype=np.uint64)
    R, C = np.meshgrid(rows, c, indexing="ij")
    words = philox4x32_10(C // np.uint64(4), R, offset & 0xFFFFFFFF,
                          offset >> 32, seed & 0xFFFFFFFF, seed >> 32)
    w = np.choose((C % np.uint64(4)).astype(np.int64), words)
    return w >= np.uint32(dropout_threshold(p))


def _apply_dropout(Zpre, dropout, rows=None):
    p, seed, offset = dropout
    rows = np.arange(Zpre.shape[0]) if rows is None else rows
    mask = dropout_mask(rows, Zpre.shape[1], p, seed, offset)
    return np.where(mask, Zpre / (1.0 - p), 0.0), mask


# ------------------------------------------------- unsharded MLP block ----

def forward(X, A, B, b1=None, b2=None, gamma=None, beta=None, eps=1e-5,
            mode="erf", residual=False, dropout=None):
    """Unsharded block: Xn = LN(X) or X; H = Xn A + b1; Y = GeLU(H);
    Z = Dropout(Y B + b2) (+ X with the residual connection).  Returns a dict
    with Xn, mean, rstd, H, Y, Z (fp64) and the dropout mask (or None)."""
    X, A, B = _f64(X), _f64(A), _f64(B)
    mean = rstd = None
    if gamma is not None:
        Xn, mean, rstd = layernorm_forward(X, gamma, beta, eps)
    else:
        Xn = X
    H = Xn @ A
    if b1 is not None:
        H = H + _f64(b1)[None, :]
    Y = gelu(H, mode)
    Z = Y @ B
    if b2 is not None:
        Z = Z + _f64(b2)[None, :]
    mask = None
    if dropout is not None:
        Z, mask = _apply_dropout(Z, dropout)
    if residual:
        Z = Z + X
    return dict(Xn=Xn, mean=mean, rstd=rstd, H=H, Y=Y, Z=Z, mask=mask,
                dropout=dropout)


def backward(dZ, X, A, B, fwd, gamma=None, mode="erf", residual=False):
    """Analytic gradients of the unsharded block given dZ = dL/dZ.

    db2 = sum_T dZ; dB = Y^T dZ; dY = dZ B^T; dH = dY * GeLU'(H);
    db1 = sum_T dH; dA = Xn^T dH; dXn = dH A^T; dX = LN-backward(dXn) (or
    dXn without LayerNorm), with dgamma and dbeta; the residual connection
    adds dZ to dX.
    """
    dZ, X, A, B = _f64(dZ), _f64(X), _f64(A), _f64(B)
    dZr = dZ                                    # residual path: unmasked
    if fwd.get("dropout") is not None:
        dZ = np.where(fwd["mask"], dZ / (1.0 - fwd["dropout"][0]), 0.0)
    db2 = dZ.sum(axis=0)
    dB = fwd["Y"].T @ dZ
    dY = dZ @ B.T
    dH = dY * gelu_grad(fwd["H"], mode)
    db1 = dH.sum(axis=0)
    dA = fwd["Xn"].T @ dH
    dXn = dH @ A.T
    dgamma = dbeta = None
    if gamma is not None:
        dX, dgamma, dbeta = layernorm_backward(dXn, X, fwd["mean"],
                                               fwd["rstd"], gamma)
    else:
        dX = dXn
    if residual:
        dX = dX + dZr
    return dict(dX=dX, dA=dA, dB=dB, db1=db1, db2=db2, dgamma=dgamma,
                dbeta=dbeta, dH=dH, dXn=dXn)


# ------------------------------- the pages' sharded form (f / g) ----------

def _f_forward(x):
    return x                                    # f: identity going forward


def _g_forward(partials):
    out = np.zeros_like(partials[0])            # g: all-reduce going forward
    for p in partials:
        out = out + p
    return out


def _f_backward(partials):
    return _g_forward(partials)                 # f: all-reduce going back


def forward_sharded(X, A, B, t, b1=None, b2=None, gamma=None, beta=None,
                    eps=1e-5, mode="erf", residual=False, dropout=None):
    """The block as t column/row shards joined by f and g.

    Shard i owns columns [i f/t, (i+1) f/t) of A (and of b1) and the same
    rows of B: Y_i = GeLU(f(Xn) A_i + b1_i), Z_i = Y_i B_i, Z = g(Z_i) + b2.
    """
    X, A, B = _f64(X), _f64(A), _f64(B)
    f = A.shape[1]
    if f % t:
        raise ValueError("ffn must be divisible by the shard count")
    ft = f // t
    if gamma is not None:
        Xn, mean, rstd = layernorm_forward(X, gamma, beta, eps)
    else:
        Xn, mean, rstd = X, None, None
    x = _f_forward(Xn)
    Hs, Ys, Zs = [], [], []
    for i in range(t):
        cols = slice(i * ft, (i + 1) * ft)
        Hi = x @ A[:, cols]
        if b1 is not None:
            Hi = Hi + _f64(b1)[cols][None, :]
        Yi = gelu(Hi, mode)
        Hs.append(Hi)
        Ys.append(Yi)
        Zs.append(Yi @ B[cols, :])
    Z = _g_forward(Zs)
    if b2 is not None:
        Z = Z + _f64(b2)[None, :]
    mask = None
    if dropout is not None:                     # outside the parallel region
        Z, mask = _apply_dropout(Z, dropout)
    if residual:
        Z = Z + X                               # outside the parallel region
    return dict(Xn=Xn, mean=mean, rstd=rstd, H=Hs, Y=Ys, Z_parts=Zs, Z=Z,
                mask=mask, dropout=dropout)


def backward_sharded(dZ, X, A, B, t, fwd_sh, gamma=None, mode="erf",
                     residual=False):
    """Backward of ``forward_sharded``: g passes dZ unchanged to every shard;
    each shard forms its own dA_i, dB_i, db1_i and dXn_i; f sums the dXn_i."""
    dZ, X, A, B = _f64(dZ), _f64(X), _f64(A), _f64(B)
    ft = A.shape[1] // t
    dZr = dZ
    if fwd_sh.get("dropout") is not None:
        dZ = np.where(fwd_sh["mask"], dZ / (1.0 - fwd_sh["dropout"][0]), 0.0)
    dz = dZ                                     # g: identity going backward
    dA_parts, dB_parts, db1_parts, dXn_parts = [], [], [], []
    for i in range(t):
        cols = slice(i * ft, (i + 1) * ft)
        dYi = dz @ B[cols, :].T
        dHi = dYi * gelu_grad(fwd_sh["H"][i], mode)
        dA_parts.append(fwd_sh["Xn"].T @ dHi)
        dB_parts.append(fwd_sh["Y"][i].T @ dz)
        db1_parts.append(dHi.sum(axis=0))
        dXn_parts.append(dHi @ A[:, cols].T)
    dXn = _f_backward(dXn_parts)
    dgamma = dbeta = None
    if gamma is not None:
        dX, dgamma, dbeta = layernorm_backward(dXn, X, fwd_sh["mean"],
                                               fwd_sh["rstd"], gamma)
    else:
        dX = dXn
    if residual:
        dX = dX + dZr
    return dict(dX=dX, dA=np.concatenate(dA_parts, axis=1),
                dB=np.concatenate(dB_parts, axis=0),
                db1=np.concatenate(db1_parts), db2=dZ.sum(axis=0),
                dgamma=dgamma, dbeta=dbeta, dXn_parts=dXn_parts)


# ------------------------- sampled outputs for the full-size workloads ----
# Each function below evaluates a subset of the unsharded definition's
# outputs exactly (one token row or one weight column at a time).

def _normalized(X, gamma, beta, eps, rows=None):
    X = _f64(X) if rows is None else _f64(X)[rows]
    if gamma is None:
        return X
    return layernorm_forward(X, gamma, beta, eps)[0]


def forward_rows(X, A, B, rows, b1=None, b2=None, gamma=None, beta=None,
                 eps=1e-5, mode="erf", residual=False, dropout=None):
    """Z[rows, :] (each token row depends only on its own input row)."""
    Xn = _normalized(X, gamma, beta, eps, rows)
    H = Xn @ _f64(A)
    if b1 is not None:
        H = H + _f64(b1)[None, :]
    Z = gelu(H, mode) @ _f64(B)
    if b2 is not None:
        Z = Z + _f64(b2)[None, :]
    if dropout is not None:
        Z, _ = _apply_dropout(Z, dropout, rows)
    if residual:
        Z = Z + _f64(X)[rows]
    return Z


def dxn_rows(dZ, X, A, B, rows, b1=None, gamma=None, beta=None, eps=1e-5,
             mode="erf"):
    """dXn[rows, :] = (dZ B^T * GeLU'(H))[rows] A^T; without LayerNorm this
    is dX[rows]."""
    A = _f64(A)
    Xn = _normalized(X, gamma, beta, eps, rows)
    H = Xn @ A
    if b1 is not None:
        H = H + _f64(b1)[None, :]
    dH = (_f64(dZ)[rows] @ _f64(B).T) * gelu_grad(H, mode)
    return dH @ A.T


def dA_cols(dZ, X, A, B, cols, b1=None, gamma=None, beta=None, eps=1e-5,
            mode="erf"):
    """(dA[:, cols], db1[cols]) from H[:, cols] and dY[:, cols] over all T."""
    Xn = _normalized(X, gamma, beta, eps)
    Hc = Xn @ _f64(A)[:, cols]
    if b1 is not None:
        Hc = Hc + _f64(b1)[cols][None, :]
    dHc = (_f64(dZ) @ _f64(B)[cols, :].T) * gelu_grad(Hc, mode)
    return Xn.T @ dHc, dHc.sum(axis=0)


def dB_rows(dZ, X, A, rows, b1=None, gamma=None, beta=None, eps=1e-5,
            mode="erf"):
    """dB[rows, :] = Y[:, rows]^T dZ."""
    Xn = _normalized(X, gamma, beta, eps)
    Hr = Xn @ _f64(A)[:, rows]
    if b1 is not None:
        Hr = Hr + _f64(b1)[rows][None, :]
    return gelu(Hr, mode).T @ _f64(dZ)


def db2(dZ):
    """db2 = sum over tokens of dZ."""
    return _f64(dZ).sum(axis=0)
