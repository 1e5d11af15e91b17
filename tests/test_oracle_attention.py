"""Pins for the fp64 attention-block oracle: brute-force loops, softmax
properties, closed-form special cases, the pages' head-shard identity and
central finite differences for every gradient.  No GPU."""
import math

import numpy as np
import pytest

from oracle import attention as A


def _problem(seed=0, nb=2, s=3, h=8, heads=2, ln=False, bias=True):
    rng = np.random.default_rng(seed)
    T = nb * s
    p = dict(X=rng.standard_normal((T, h)),
             Wqkv=rng.standard_normal((h, 3 * h)) * 0.5,
             Wo=rng.standard_normal((h, h)) * 0.5,
             dZ=rng.standard_normal((T, h)),
             bqkv=rng.standard_normal(3 * h) * 0.3 if bias else None,
             bo=rng.standard_normal(h) * 0.3 if bias else None,
             gamma=(1 + 0.3 * rng.standard_normal(h)) if ln else None,
             beta=(0.3 * rng.standard_normal(h)) if ln else None)
    return p, dict(heads=heads, seq_len=s)


def _brute(X, Wqkv, Wo, bqkv, bo, heads, s, shards, causal):
    """Per-element loops, math.exp, the shard-grouped W_qkv column layout
    written out index by index."""
    T, h = len(X), len(X[0])
    d = h // heads
    hs = h // shards
    hp = heads // shards
    qkv = [[sum(X[r][c] * Wqkv[c][n] for c in range(h)) + (bqkv[n] if bqkv is not None else 0.0)
            for n in range(3 * h)] for r in range(T)]

    def col(kind, head, e):          # kind 0 = Q, 1 = K, 2 = V
        i, jj = divmod(head, hp)
        return 3 * hs * i + kind * hs + jj * d + e

    ctx = [[0.0] * h for _ in range(T)]
    for b in range(T // s):
        for head in range(heads):
            for i in range(s):
                r = b * s + i
                keys = [j for j in range(s) if (j <= i or not causal)]
                sc = [sum(qkv[r][col(0, head, e)] * qkv[b * s + j][col(1, head, e)]
                          for e in range(d)) / math.sqrt(d) for j in keys]
                m = max(sc)
                w = [math.exp(x - m) for x in sc]
                tot = sum(w)
                for e in range(d):
                    ctx[r][head * d + e] = sum(
                        w[n] / tot * qkv[b * s + j][col(2, head, e)]
                        for n, j in enumerate(keys))
    return np.array([[sum(ctx[r][c] * Wo[c][o] for c in range(h)) + (bo[o] if bo is not None else 0.0)
                      for o in range(h)] for r in range(T)])


@pytest.mark.parametrize("causal,shards,h,heads", [
    (True, 1, 8, 2), (True, 2, 8, 2), (False, 2, 8, 2),
    # a head dim that is not a power of two (d = 3, as 96 = 3 * 32): the
    # 1 / sqrt(d) scale and the head columns at multiples of d
    (True, 2, 12, 4), (False, 1, 12, 4)])
def test_forward_matches_brute_force(causal, shards, h, heads):
    p, c = _problem(seed=1, h=h, heads=heads)
    got = A.forward(p["X"], p["Wqkv"], p["Wo"], c["heads"], c["seq_len"], shards,
                    bqkv=p["bqkv"], bo=p["bo"], causal=causal)["Z"]
    want = _brute(p["X"].tolist(), p["Wqkv"].tolist(), p["Wo"].tolist(),
                  p["bqkv"].tolist(), p["bo"].tolist(), c["heads"], c["seq_len"],
                  shards, causal)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_softmax_rows_and_causal_mask():
    p, c = _problem(seed=2, nb=1, s=5)
    f = A.forward(p["X"], p["Wqkv"], p["Wo"], c["heads"], c["seq_len"])
    for P in f["P"]:
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert np.all(P[np.triu_indices(5, 1)] == 0.0)
        assert np.all(P[np.tril_indices(5)] > 0.0)


@pytest.mark.parametrize("causal", [True, False])
def test_zero_query_key_projection_gives_prefix_means(causal):
    """W_q = W_k = 0 (no bias): every score is 0, so each query averages the
    values of the keys it may see: running means (causal) or the sequence
    mean."""
    p, c = _problem(seed=3, nb=2, s=4, h=4, heads=2, bias=False)
    W = p["Wqkv"].copy()
    hs = 4
    W[:, 0:2 * hs] = 0.0                      # one shard: [Q | K | V]
    f = A.forward(p["X"], W, np.eye(4), c["heads"], c["seq_len"], causal=causal)
    v = p["X"] @ W[:, 2 * hs:3 * hs]
    for b in range(2):
        vb = v[b * 4:(b + 1) * 4]
        want = (np.cumsum(vb, axis=0) / np.arange(1, 5)[:, None]) if causal \
            else np.broadcast_to(vb.mean(axis=0), vb.shape)
        np.testing.assert_allclose(f["Ctx"][b * 4:(b + 1) * 4], want, rtol=1e-13,
                                   atol=1e-14)


def test_length_one_sequences_return_values():
    p, c = _problem(seed=4, nb=5, s=1)
    f = A.forward(p["X"], p["Wqkv"], p["Wo"], c["heads"], 1, bqkv=p["bqkv"])
    q, k, v = A._split(f["QKV"], c["heads"], 1)
    np.testing.assert_allclose(f["Ctx"], v.reshape(5, -1), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("shards", [1, 2, 4])
@pytest.mark.parametrize("ln,res", [(False, False), (True, True)])
def test_head_shard_identity(shards, ln, res):
    """sum_i Attn_i(X) Wo_i over head groups equals the unsharded block."""
    p, c = _problem(seed=5, nb=2, s=4, h=16, heads=4, ln=ln)
    kw = dict(bqkv=p["bqkv"], bo=p["bo"], gamma=p["gamma"], beta=p["beta"],
              residual=res)
    full = A.forward(p["X"], p["Wqkv"], p["Wo"], 4, 4, shards, **kw)
    sh = A.forward_sharded(p["X"], p["Wqkv"], p["Wo"], 4, 4, shards, **kw)
    assert len(sh["Z_parts"]) == shards
    np.testing.assert_allclose(sh["Z"], full["Z"], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal,ln,res,shards", [(True, False, False, 1),
                                                  (True, True, True, 2),
                                                  (False, True, False, 2)])
def test_backward_matches_central_differences(causal, ln, res, shards):
    p, c = _problem(seed=6, nb=2, s=3, h=8, heads=2, ln=ln)
    heads, s = c["heads"], c["seq_len"]

    def fwd():
        return A.forward(p["X"], p["Wqkv"], p["Wo"], heads, s, shards,
                         bqkv=p["bqkv"], bo=p["bo"], gamma=p["gamma"],
                         beta=p["beta"], causal=causal, residual=res)

    f = fwd()
    g = A.backward(p["dZ"], p["X"], p["Wqkv"], p["Wo"], f, heads, s, shards,
                   gamma=p["gamma"], causal=causal, residual=res)
    names = {"X": "dX", "Wqkv": "dWqkv", "bqkv": "dbqkv", "Wo": "dWo", "bo": "dbo"}
    if ln:
        names.update(gamma="dgamma", beta="dbeta")
    for pname, gname in names.items():
        base = p[pname]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            step = 1e-5 * max(1.0, abs(base[idx]))
            keep = base[idx]
            base[idx] = keep + step
            lp = float((fwd()["Z"] * p["dZ"]).sum())
            base[idx] = keep - step
            lm = float((fwd()["Z"] * p["dZ"]).sum())
            base[idx] = keep
            fd[idx] = (lp - lm) / (2 * step)
        np.testing.assert_allclose(g[gname], fd, rtol=0,
                                   atol=3e-8 * max(1.0, np.abs(fd).max()),
                                   err_msg=pname)
