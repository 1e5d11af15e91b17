"""fp64 CPU oracle for the head-parallel self-attention block.

TEST INFRASTRUCTURE ONLY (never on the product path).

What it computes (Megatron-LM explainer, azimuth.plus, section "Attention: a
design that parallelises naturally"; Megatron-LM notes, notes.yuuk.io,
section "Self-attention block split"): the attention heads are independent,
so the Q, K and V projection GEMMs are split by columns head by head, every
shard computes the attention of its own heads with no communication, and the
output projection O is split by rows, exactly like B in the MLP, with one
all-reduce after it (the same f / g operators).

Readings where the pages are silent (listed in the design notes):

* Scaled dot-product attention softmax(Q K^T / sqrt(d)) V per head, causal
  (GPT-style: query i sees keys j <= i inside its own sequence) unless
  ``causal=False``; tokens are ``batch * seq_len`` rows, sequence-major.
* Fused projection W_qkv [h, 3h] with columns grouped by shard: shard i owns
  columns [3 i h / t, 3 (i+1) h / t) = [Q_i | K_i | V_i], each h / t wide,
  i.e. heads i H/t .. (i+1) H/t - 1 of Q, K and V in order; b_qkv [3h]
  likewise.  The context Ctx [T, h] holds head j in columns [j d, (j+1) d),
  so W_o [h, h] row block i belongs to shard i; b_o [h] is added once after
  the sum.
* Optional pre-LayerNorm on X and residual X + Attn(LN(X)), as for the MLP.
* No attention dropout.
"""
from __future__ import annotations

import math

import numpy as np

from .mlp import _f64, layernorm_backward, layernorm_forward


def _split(qkv, heads, shards):
    """Views of Q, K, V [T, heads, d] from the shard-grouped projection."""
    T, three_h = qkv.shape
    h = three_h // 3
    d = h // heads
    hs = h // shards
    q = np.empty((T, heads, d))
    k = np.empty((T, heads, d))
    v = np.empty((T, heads, d))
    hp = heads // shards
    for i in range(shards):
        base = 3 * hs * i
        q[:, i * hp:(i + 1) * hp] = qkv[:, base:base + hs].reshape(T, hp, d)
        k[:, i * hp:(i + 1) * hp] = qkv[:, base + hs:base + 2 * hs].reshape(T, hp, d)
        v[:, i * hp:(i + 1) * hp] = qkv[:, base + 2 * hs:base + 3 * hs].reshape(T, hp, d)
    return q, k, v


def _merge(dq, dk, dv, shards):
    """Inverse of _split for gradients: [T, heads, d] x 3 -> [T, 3h]."""
    T, heads, d = dq.shape
    h = heads * d
    hs = h // shards
    hp = heads // shards
    out = np.empty((T, 3 * h))
    for i in range(shards):
        base = 3 * hs * i
        out[:, base:base + hs] = dq[:, i * hp:(i + 1) * hp].reshape(T, hs)
        out[:, base + hs:base + 2 * hs] = dk[:, i * hp:(i + 1) * hp].reshape(T, hs)
        out[:, base + 2 * hs:base + 3 * hs] = dv[:, i * hp:(i + 1) * hp].reshape(T, hs)
    return out


def _mask(seq_len, causal):
    if not causal:
        return np.ones((seq_len, seq_len), dtype=bool)
    return np.tril(np.ones((seq_len, seq_len), dtype=bool))


def attention_core(q, k, v, seq_len, causal=True):
    """Per sequence and head: P = softmax(q k^T / sqrt(d) masked), O = P v.
    q, k, v: [T, heads, d].  Returns (O [T, heads, d], P list, lse [T, heads])."""
    T, heads, d = q.shape
    nb = T // seq_len
    scale = 1.0 / math.sqrt(d)
    allowed = _mask(seq_len, causal)
    o = np.zeros_like(q)
    lse = np.zeros((T, heads))
    probs = []
    for b in range(nb):
        rows = slice(b * seq_len, (b + 1) * seq_len)
        for j in range(heads):
            s = (q[rows, j] @ k[rows, j].T) * scale
            s = np.where(allowed, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            l = e.sum(axis=1, keepdims=True)
            p = e / l
            o[rows, j] = p @ v[rows, j]
            lse[rows, j] = (m + np.log(l))[:, 0]
            probs.append(p)
    return o, probs, lse


def core_backward(q, k, v, do, probs, seq_len):
    """Per sequence and head, given P from attention_core (same order):
    dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dP * P)),
    dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d).  All [T, heads, d]."""
    T, heads, d = q.shape
    scale = 1.0 / math.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    idx = 0
    for b in range(T // seq_len):
        rows = slice(b * seq_len, (b + 1) * seq_len)
        for j in range(heads):
            p = probs[idx]
            idx += 1
            dv[rows, j] = p.T @ do[rows, j]
            dp = do[rows, j] @ v[rows, j].T
            ds = p * (dp - (dp * p).sum(axis=1, keepdims=True))
            dq[rows, j] = (ds @ k[rows, j]) * scale
            dk[rows, j] = (ds.T @ q[rows, j]) * scale
    return dq, dk, dv


def forward(X, Wqkv, Wo, heads, seq_len, shards=1, bqkv=None, bo=None,
            gamma=None, beta=None, eps=1e-5, causal=True, residual=False):
    """Unsharded attention block.  Returns a dict with Xn, mean, rstd, QKV,
    Ctx, P (per sequence and head), Z."""
    X, Wqkv, Wo = _f64(X), _f64(Wqkv), _f64(Wo)
    mean = rstd = None
    if gamma is not None:
        Xn, mean, rstd = layernorm_forward(X, gamma, beta, eps)
    else:
        Xn = X
    qkv = Xn @ Wqkv
    if bqkv is not None:
        qkv = qkv + _f64(bqkv)[None, :]
    q, k, v = _split(qkv, heads, shards)
    o, probs, lse = attention_core(q, k, v, seq_len, causal)
    ctx = o.reshape(X.shape[0], -1)
    Z = ctx @ Wo
    if bo is not None:
        Z = Z + _f64(bo)[None, :]
    if residual:
        Z = Z + X
    return dict(Xn=Xn, mean=mean, rstd=rstd, QKV=qkv, Ctx=ctx, P=probs,
                lse=lse, Z=Z)


def backward(dZ, X, Wqkv, Wo, fwd, heads, seq_len, shards=1, gamma=None,
             causal=True, residual=False):
    """Analytic gradients: dbo = sum_T dZ, dWo = Ctx^T dZ, dCtx = dZ Wo^T;
    per sequence and head dV = P^T dO, dP = dO V^T,
    dS = P * (dP - rowsum(dP * P)), dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d);
    dWqkv = Xn^T dQKV, dbqkv = sum_T dQKV, dXn = dQKV Wqkv^T, then LayerNorm
    backward and the residual."""
    dZ, X, Wqkv, Wo = _f64(dZ), _f64(X), _f64(Wqkv), _f64(Wo)
    T = X.shape[0]
    dbo = dZ.sum(axis=0)
    dWo = fwd["Ctx"].T @ dZ
    dctx = dZ @ Wo.T
    q, k, v = _split(fwd["QKV"], heads, shards)
    d = q.shape[2]
    do = dctx.reshape(T, heads, d)
    dq, dk, dv = core_backward(q, k, v, do, fwd["P"], seq_len)
    dqkv = _merge(dq, dk, dv, shards)
    dWqkv = fwd["Xn"].T @ dqkv
    dbqkv = dqkv.sum(axis=0)
    dXn = dqkv @ Wqkv.T
    dgamma = dbeta = None
    if gamma is not None:
        dX, dgamma, dbeta = layernorm_backward(dXn, X, fwd["mean"], fwd["rstd"],
                                               gamma)
    else:
        dX = dXn
    if residual:
        dX = dX + dZ
    return dict(dX=dX, dWqkv=dWqkv, dbqkv=dbqkv, dWo=dWo, dbo=dbo,
                dgamma=dgamma, dbeta=dbeta, dQKV=dqkv, dCtx=dctx)


def forward_sharded(X, Wqkv, Wo, heads, seq_len, shards, bqkv=None, bo=None,
                    gamma=None, beta=None, eps=1e-5, causal=True,
                    residual=False):
    """The pages' decomposition: f (identity) hands the full input to every
    shard; shard i projects with its column block of W_qkv, runs attention
    on its own heads and multiplies by its row block of W_o; g sums the
    shards' partial outputs; b_o is added once."""
    X, Wqkv, Wo = _f64(X), _f64(Wqkv), _f64(Wo)
    h = X.shape[1]
    hs = h // shards
    hp = heads // shards
    if gamma is not None:
        Xn, _, _ = layernorm_forward(X, gamma, beta, eps)
    else:
        Xn = X
    partials = []
    for i in range(shards):
        cols = slice(3 * hs * i, 3 * hs * (i + 1))
        qkv_i = Xn @ Wqkv[:, cols]
        if bqkv is not None:
            qkv_i = qkv_i + _f64(bqkv)[cols][None, :]
        q_i, k_i, v_i = _split(qkv_i, hp, 1)
        o_i, _, _ = attention_core(q_i, k_i, v_i, seq_len, causal)
        ctx_i = o_i.reshape(X.shape[0], hs)
        partials.append(ctx_i @ Wo[i * hs:(i + 1) * hs, :])
    Z = np.zeros_like(partials[0])
    for p in partials:                          # g: sum of the partials
        Z = Z + p
    if bo is not None:
        Z = Z + _f64(bo)[None, :]
    if residual:
        Z = Z + X
    return dict(Z=Z, Z_parts=partials)
