"""The attention block's backward in fp64 with bf16 rounding applied at
chosen storage points: the error budget behind the attention gradient bar.

The attention kernels store or stage these tensors as bf16 (the rest is fp32
arithmetic, close to exact here):
  xn    the LayerNorm output (the projection's A operand; with LayerNorm only)
  qkv   the projection output Q, K, V (read by both core kernels)
  p     the probabilities, as the MMA operand of P V (forward) and of
        P^T dO (backward)
  ctx   the context rows (the forward's output; the output projection and
        dW_o read them)
  dctx  dO = dZ W_o^T (read by both backward core kernels)
  ds    dS = P (dP - delta) / sqrt(d), the MMA operand of dQ and dK
  dqkv  the core's output dQ, dK, dV (read by dW_qkv and dX)
`backward_rounded(points=...)` evaluates the block's unsharded definition
(the oracle's, written out below with the same primitives) with rounding at
the named points only, so that comparing it with the exact result measures
each point's share of the error.  Test infrastructure; nothing here is on
the product path or shares code with it.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import attention as A
from oracle import mlp as M

POINTS = ("xn", "qkv", "p", "ctx", "dctx", "ds", "dqkv")


def bf16(x):
    """Round fp64 values to bf16 (nearest even, through fp32) and widen back."""
    return torch.from_numpy(np.ascontiguousarray(x)).float().bfloat16() \
        .double().numpy()


def backward_rounded(inp, heads, seq_len, shards, causal, residual,
                     points=()):
    """Forward and backward of the attention block in fp64, rounding to bf16
    at `points`.  Returns the oracle's gradient dict keys dX, dQKV, dWqkv,
    dWo (and the forward's Z)."""
    r = (lambda name, x: bf16(x) if name in points else x)
    X = M._f64(inp["X"])
    Wqkv, Wo = M._f64(inp["Wqkv"]), M._f64(inp["Wo"])
    bqkv = None if inp["bqkv"] is None else M._f64(inp["bqkv"])
    bo = None if inp["bo"] is None else M._f64(inp["bo"])
    gamma = None if inp["gamma"] is None else M._f64(inp["gamma"])
    beta = None if inp["beta"] is None else M._f64(inp["beta"])
    dZ = M._f64(inp["dZ"])
    T = X.shape[0]
    if gamma is not None:
        Xn, mean, rstd = M.layernorm_forward(X, gamma, beta)
        Xn = r("xn", Xn)
    else:
        Xn = X
    qkv = Xn @ Wqkv + (0 if bqkv is None else bqkv[None, :])
    qkv = r("qkv", qkv)
    q, k, v = A._split(qkv, heads, shards)
    d = q.shape[2]
    scale = 1.0 / math.sqrt(d)
    allowed = A._mask(seq_len, causal)
    o = np.zeros_like(q)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    probs = []
    for b in range(T // seq_len):
        rows = slice(b * seq_len, (b + 1) * seq_len)
        for j in range(heads):
            s = np.where(allowed, (q[rows, j] @ k[rows, j].T) * scale, -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            p = e / e.sum(axis=1, keepdims=True)
            probs.append(p)
            o[rows, j] = r("p", p) @ v[rows, j]
    ctx = r("ctx", o.reshape(T, -1))
    Z = ctx @ Wo + (0 if bo is None else bo[None, :])
    if residual:
        Z = Z + X
    dWo = ctx.T @ dZ
    do = r("dctx", dZ @ Wo.T).reshape(T, heads, d)
    idx = 0
    for b in range(T // seq_len):
        rows = slice(b * seq_len, (b + 1) * seq_len)
        for j in range(heads):
            p = probs[idx]
            idx += 1
            dv[rows, j] = r("p", p).T @ do[rows, j]
            dp = do[rows, j] @ v[rows, j].T
            ds = r("ds", p * (dp - (dp * p).sum(axis=1, keepdims=True)) * scale)
            dq[rows, j] = ds @ k[rows, j]
            dk[rows, j] = ds.T @ q[rows, j]
    dqkv = r("dqkv", A._merge(dq, dk, dv, shards))
    dWqkv = Xn.T @ dqkv
    dXn = dqkv @ Wqkv.T
    if gamma is not None:
        dX = M.layernorm_backward(dXn, X, mean, rstd, gamma)[0]
    else:
        dX = dXn
    if residual:
        dX = dX + dZ
    return dict(Z=Z, dX=dX, dQKV=dqkv, dWqkv=dWqkv, dWo=dWo)


def rel_fro(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def budget(inp, heads, seq_len, shards, causal, residual,
           keys=("dQKV", "dX")):
    """Relative Frobenius error of `keys` against the exact block for every
    single rounding point and for all of them together:
    {point or "all": {key: error}}."""
    exact = backward_rounded(inp, heads, seq_len, shards, causal, residual)
    out = {}
    for pts in [(p,) for p in POINTS] + [POINTS]:
        got = backward_rounded(inp, heads, seq_len, shards, causal, residual,
                               pts)
        out["all" if len(pts) > 1 else pts[0]] = {
            k: rel_fro(got[k], exact[k]) for k in keys}
    return out
