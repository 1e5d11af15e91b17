"""Pins for the attention error-budget emulation (tests/attention_rounding.py)
on the CPU: its bf16 rounding is round-to-nearest-even with the format's
spacing, with no rounding point it is the oracle's block, and each point only
adds error."""
import numpy as np
import pytest
import torch

import attention_rounding as R
from oracle import attention as A
from tensor_transformer_mlp_tcgen05_gb300 import workloads as W


def test_bf16_rounding_is_nearest_even():
    u = 2.0 ** -7        # bf16 spacing on [1, 2)
    x = np.array([1.0, 1 + u / 2, 1 + 3 * u / 2, 1 + u / 2 + 2.0 ** -20,
                  -(1 + 3 * u / 2), 3.0e38])
    got = R.bf16(x)
    assert got[0] == 1.0
    assert got[1] == 1.0                 # tie -> even mantissa
    assert got[2] == 1 + 2 * u           # tie -> even mantissa
    assert got[3] == 1 + u               # above the tie
    assert got[4] == -(1 + 2 * u)
    assert np.isfinite(got[5])           # below bf16's largest value


def _case(base, over, ln, seed=3):
    w = W.ATTN_WORKLOADS[base].with_(batch=1, seq=128, **over)
    inp = W.make_attn_inputs(w, seed=seed, with_bias=True)
    if ln:
        g = torch.Generator().manual_seed(5)
        inp["gamma"] = 1 + 0.2 * torch.randn(w.hidden, generator=g)
        inp["beta"] = 0.2 * torch.randn(w.hidden, generator=g)
    return w, inp


@pytest.mark.parametrize("ln,res,causal", [(False, False, True),
                                           (True, True, False)])
def test_no_rounding_point_is_the_oracle(ln, res, causal):
    w, inp = _case("attn_tiny_d64", dict(causal=causal, layernorm=ln), ln)
    f64 = {k: (None if v is None else v.double().numpy()) for k, v in inp.items()}
    fwd = A.forward(f64["X"], f64["Wqkv"], f64["Wo"], w.heads, w.seq, w.shards,
                    bqkv=f64["bqkv"], bo=f64["bo"], gamma=f64["gamma"],
                    beta=f64["beta"], causal=causal, residual=res)
    g = A.backward(f64["dZ"], f64["X"], f64["Wqkv"], f64["Wo"], fwd, w.heads,
                   w.seq, w.shards, gamma=f64["gamma"], causal=causal,
                   residual=res)
    emu = R.backward_rounded(inp, w.heads, w.seq, w.shards, causal, res)
    for k, ref in (("Z", fwd["Z"]), ("dX", g["dX"]), ("dQKV", g["dQKV"]),
                   ("dWqkv", g["dWqkv"]), ("dWo", g["dWo"])):
        np.testing.assert_allclose(emu[k], ref, rtol=1e-11,
                                   atol=1e-12 * np.abs(ref).max(), err_msg=k)


def test_budget_points_add_error():
    w, inp = _case("attn_tiny_d96", dict(layernorm=True), True)
    b = R.budget(inp, w.heads, w.seq, w.shards, w.causal, False)
    assert set(b) == set(R.POINTS) | {"all"}
    # "ctx" feeds only the output projection and dW_o, not dQKV or dX
    assert b["ctx"]["dQKV"] == 0.0 and b["ctx"]["dX"] == 0.0
    for p in R.POINTS:
        if p != "ctx":
            assert 1e-4 < b[p]["dQKV"] < 1e-2, (p, b[p])
        assert b[p]["dQKV"] <= b["all"]["dQKV"] * 1.05, (p, b[p], b["all"])
    # independent roundings add roughly in quadrature
    quad = np.sqrt(sum(b[p]["dQKV"] ** 2 for p in R.POINTS))
    assert 0.6 * quad < b["all"]["dQKV"] < 1.4 * quad, (quad, b["all"])


def test_layernorm_output_point_needs_layernorm():
    w, inp = _case("attn_tiny_d64", {}, False)
    b = R.budget(inp, w.heads, w.seq, w.shards, w.causal, False)
    assert b["xn"]["dQKV"] == 0.0
