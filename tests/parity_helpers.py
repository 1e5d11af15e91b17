"""Shared helpers for the GPU parity tests: run the CUDA path through the
binding and compare with the fp64 oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

from oracle import mlp as O
from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP

# Tolerances (the block's stated bars): bf16 inputs with fp32 accumulation:
# relative Frobenius error <= 5e-3 and max |err| <= 3e-2 max |ref|;
# the fp32 configuration: <= 1e-5 relative for both.
TOL_BF16 = (5e-3, 3e-2)
TOL_FP32 = (1e-5, 1e-5)


def f64(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.astype(np.float64, copy=False)
    return t.detach().to("cpu").double().numpy()


def errors(got, ref):
    got, ref = f64(got), f64(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = got - ref
    nref = np.linalg.norm(ref)
    mref = np.abs(ref).max() if ref.size else 0.0
    rel_fro = np.linalg.norm(err) / nref if nref > 0 else np.linalg.norm(err)
    max_rel = np.abs(err).max() / mref if mref > 0 else (np.abs(err).max() if err.size else 0.0)
    return float(rel_fro), float(max_rel)


def assert_close(name, got, ref, fp32=False):
    tol = TOL_FP32 if fp32 else TOL_BF16
    rel_fro, max_rel = errors(got, ref)
    assert np.all(np.isfinite(f64(got))), f"{name}: non-finite values"
    assert rel_fro <= tol[0] and max_rel <= tol[1], (
        f"{name}: rel_fro={rel_fro:.3e} (tol {tol[0]}), "
        f"max_rel={max_rel:.3e} (tol {tol[1]})")
    return rel_fro, max_rel


def to_dev(x):
    return None if x is None else x.cuda().contiguous()


def run_cuda(w, inp, backward=True, training=True, gelu="erf", repeat=1,
             residual=False, dropout=None):
    """Forward (+ backward) on cuda:0 through the binding.  Returns a dict of
    CPU tensors; with repeat > 1 a list of such dicts (same inputs)."""
    p, seed, offset = dropout if dropout is not None else (0.0, 0, 0)
    m = TensorParallelMLP(w.hidden, w.ffn, w.shards, max(w.tokens, 1),
                          dtype=w.dtype, layernorm=w.layernorm, gelu=gelu,
                          residual=residual, dropout_p=p, dropout_seed=seed,
                          dropout_offset=offset)
    d = {k: to_dev(v) for k, v in inp.items()}
    outs = []
    for _ in range(repeat):
        Z = m.forward(d["X"], d["A"], d["B"], d["b1"], d["b2"], d["gamma"],
                      d["beta"], training=training or backward)
        res = {"Z": Z}
        if backward:
            res.update(m.backward(d["dZ"], d["X"], d["A"], d["B"], d["gamma"],
                                  bias_grads=True))
        rc = m.check()
        assert rc == 0, f"device status {rc}"
        torch.cuda.synchronize()
        outs.append({k: v.cpu() for k, v in res.items()})
    m.close()
    return outs if repeat > 1 else outs[0]


def oracle_full(inp, mode="erf", backward=True, residual=False, dropout=None):
    X, A, B = f64(inp["X"]), f64(inp["A"]), f64(inp["B"])
    fwd = O.forward(X, A, B, f64(inp["b1"]), f64(inp["b2"]), f64(inp["gamma"]),
                    f64(inp["beta"]), mode=mode, residual=residual,
                    dropout=dropout)
    out = {"Z": fwd["Z"]}
    if fwd.get("mask") is not None:
        out["_mask"] = fwd["mask"]
    if backward:
        g = O.backward(f64(inp["dZ"]), X, A, B, fwd, f64(inp["gamma"]), mode,
                       residual=residual)
        out.update(dX=g["dX"], dA=g["dA"], dB=g["dB"], db1=g["db1"],
                   db2=g["db2"])
        if inp["gamma"] is not None:
            out.update(dgamma=g["dgamma"], dbeta=g["dbeta"])
    return out


def compare_full(got, ref, fp32=False):
    report = {}
    for k, v in ref.items():
        if k.startswith("_"):
            continue
        report[k] = assert_close(k, got[k], v, fp32=fp32)
    return report
