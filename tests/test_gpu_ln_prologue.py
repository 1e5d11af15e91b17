"""The fused pre-LayerNorm prologue of the bf16 forward (pre-LN placement:
Megatron-LM explainer, "Fixing BERT: reordering layer normalisation for
scaling"), against the stand-alone LayerNorm launch it replaces.

With the prologue the first GEMM's epilogue warps normalise the token rows
(rows claimed from a grid-wide counter) and the producers load each 128-row
block of the A operand once its rows are published; without it a separate
LayerNorm kernel runs first.  One device function normalises a row on both
paths, so every output of the forward and the backward (which reads the
saved Xn, mean and rstd) must be bitwise equal between the two, over ragged
token counts, every row length class (vector counts 1, 3, 5 (the run-time
length path), 12, 24 (the largest fused row)), shards 1-4 and the residual.
The fused path is also checked against the fp64 oracle, with few CTA pairs
(so that warps normalise many rows while producers wait), and at the full
Megatron-8.3B layer; shapes outside the fused range fall back to the
stand-alone kernel."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from oracle import mlp as O
from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
from fingerprint import MLP_KERNEL, MLP_ORDER, assert_bitwise
from parity_helpers import assert_close, f64

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _inputs(T, h, f, t, seed):
    w = W.Workload("lnp", T, h, f, t, "bf16", True, True, w_std=0.05)
    inp = W.make_inputs(w, seed=seed, with_bias=True)
    g = torch.Generator().manual_seed(seed + 1)
    inp["gamma"] = 1 + 0.2 * torch.randn(h, generator=g)
    inp["beta"] = 0.2 * torch.randn(h, generator=g)
    return inp


def _run(inp, T, h, f, t, residual, fused):
    from tensor_transformer_mlp_tcgen05_gb300 import binding as B
    from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP
    m = TensorParallelMLP(h, f, t, T, layernorm=True, residual=residual,
                          ln_prologue=fused)
    d = {k: (None if v is None else v.cuda().contiguous())
         for k, v in inp.items()}
    B.tp_mlp_set_timing(m.handle, True)
    Z = m.forward(d["X"], d["A"], d["B"], d["b1"], d["b2"], d["gamma"],
                  d["beta"])
    n_fwd = B.tp_mlp_launch_count(m.handle)
    g = m.backward(d["dZ"], d["X"], d["A"], d["B"], d["gamma"])
    rc = m.check()
    assert rc == 0, (rc, B.tp_mlp_last_detail())
    names = [n for n, _, _ in B.tp_mlp_timing_get(m.handle)]
    out = {"Z": Z, **g}
    torch.cuda.synchronize()
    out = {k: v.cpu() for k, v in out.items()}
    m.close()
    return out, n_fwd, names


CASES = [
    # tokens, hidden, ffn, shards, residual
    (1, 256, 512, 2, False),
    (127, 768, 1536, 3, True),
    (300, 1280, 2560, 4, False),
    (513, 3072, 3072, 2, True),
    (1000, 6144, 1024, 1, False),
    (2048, 1024, 4096, 4, True),
]


@pytest.mark.parametrize("T,h,f,t,res", CASES)
def test_fused_prologue_is_bitwise_the_standalone_layernorm(T, h, f, t, res):
    inp = _inputs(T, h, f, t, seed=T + h)
    a, n_a, names_a = _run(inp, T, h, f, t, res, fused=True)
    b, n_b, names_b = _run(inp, T, h, f, t, res, fused=False)
    assert n_a == 2 and "gemm1_ln_gelu" in names_a and \
        "layernorm_fwd" not in names_a
    assert n_b == 3 and "layernorm_fwd" in names_b
    assert_bitwise(a, b, MLP_ORDER, MLP_KERNEL)
    for v in a.values():
        assert torch.isfinite(v.float()).all()


def test_fused_prologue_against_the_oracle():
    T, h, f, t = 777, 1280, 2560, 4
    inp = _inputs(T, h, f, t, seed=5)
    got, _, _ = _run(inp, T, h, f, t, True, fused=True)
    fwd = O.forward(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]),
                    f64(inp["b1"]), f64(inp["b2"]), f64(inp["gamma"]),
                    f64(inp["beta"]), residual=True)
    ref = O.backward(f64(inp["dZ"]), f64(inp["X"]), f64(inp["A"]),
                     f64(inp["B"]), fwd, f64(inp["gamma"]), residual=True)
    assert_close("Z", got["Z"], fwd["Z"])
    for k in ("dX", "dA", "dB", "db1", "db2", "dgamma", "dbeta"):
        assert_close(k, got[k], ref[k])


@pytest.mark.parametrize("h", [6400, 320])
def test_shapes_outside_the_fused_range_use_the_standalone_kernel(h):
    T, f, t = 200, 1024, 2
    inp = _inputs(T, h, f, t, seed=h)
    a, n_a, names_a = _run(inp, T, h, f, t, False, fused=True)
    assert n_a == 3 and "layernorm_fwd" in names_a
    b, _, _ = _run(inp, T, h, f, t, False, fused=False)
    assert_bitwise(a, b, MLP_ORDER, MLP_KERNEL)


_CHILD = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np, torch
import test_gpu_ln_prologue as L
out = {{}}
for i, (T, h, f, t) in enumerate([(4000, 1024, 2048, 2), (1100, 3072, 1024, 1)]):
    inp = L._inputs(T, h, f, t, seed=40 + i)
    for fused in (True, False):
        r, n, _ = L._run(inp, T, h, f, t, True, fused)
        assert n == (2 if fused else 3), n
        for k, v in r.items():
            out["c%d_%d_%s" % (i, fused, k)] = v.float().numpy()
np.savez({path!r}, **out)
print("child ok")
"""


def test_few_pairs_normalise_every_row(tmp_path):
    """One or two CTA pairs per launch (TPMLP_GEMM_MAX_PAIRS=2): 16 or 32
    warps normalise thousands of rows while the producers wait on the
    blocks; results equal the stand-alone path bit for bit."""
    path = str(tmp_path / "few.npz")
    env = dict(os.environ, TPMLP_GEMM_MAX_PAIRS="2")
    script = _CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"),
                           path=path)
    r = subprocess.run([sys.executable, "-c", script], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    z = dict(np.load(path))
    keys = [k for k in z if k.split("_")[1] == "1"]
    assert len(keys) >= 16
    for k in keys:
        k0 = k.replace("_1_", "_0_", 1)
        np.testing.assert_array_equal(z[k], z[k0], err_msg=k)


def test_megatron_8p3b_fused_equals_standalone():
    """The full 8.3B pre-LN layer (8192 tokens, h = 3072, f = 12288, t = 8),
    in the configuration the benchmark times: both paths bit for bit."""
    w = W.WORKLOADS["megatron_8p3b"]
    inp = W.make_inputs(w, seed=0, with_bias=True)
    a, n_a, names_a = _run(inp, w.tokens, w.hidden, w.ffn, w.shards, False,
                           True)
    b, n_b, _ = _run(inp, w.tokens, w.hidden, w.ffn, w.shards, False, False)
    # (GEMM2's tail split adds its combine launch on both paths)
    assert n_b == n_a + 1 and "layernorm_fwd" not in names_a
    assert_bitwise(a, b, MLP_ORDER, MLP_KERNEL)


def _run_attn(w, inp, fused):
    from tensor_transformer_mlp_tcgen05_gb300 import binding as B
    from tensor_transformer_mlp_tcgen05_gb300.attention import \
        TensorParallelAttention
    m = TensorParallelAttention(w.hidden, w.heads, w.shards, w.tokens, w.seq,
                                causal=w.causal, layernorm=True,
                                residual=True, ln_prologue=fused)
    d = {k: (None if v is None else v.cuda().contiguous())
         for k, v in inp.items()}
    B.tp_attn_set_timing(m.handle, True)
    Z = m.forward(d["X"], d["Wqkv"], d["Wo"], d["bqkv"], d["bo"], d["gamma"],
                  d["beta"])
    n_fwd = B.tp_attn_launch_count(m.handle)
    g = m.backward(d["dZ"], d["X"], d["Wqkv"], d["Wo"], d["gamma"])
    rc = m.check()
    assert rc == 0, (rc, B.tp_mlp_last_detail())
    names = [n for n, _, _ in B.tp_attn_timing_get(m.handle)]
    out = {"Z": Z, **g}
    torch.cuda.synchronize()
    out = {k: v.cpu() for k, v in out.items()}
    m.close()
    return out, n_fwd, names


@pytest.mark.parametrize("name,over", [
    ("attn_tiny_d64", {}),
    ("attn_tiny_d96", dict(causal=False, shards=4)),
    ("attn_tiny_d128", dict(batch=3)),
    ("attn_megatron_8p3b", {}),
])
def test_attention_fused_prologue_is_bitwise_the_standalone_layernorm(name,
                                                                     over):
    """The attention block's QKV projection with the same prologue (pre-LN
    sub-block with the residual): every output bitwise equal to the
    stand-alone LayerNorm path, one launch fewer in the forward."""
    from fingerprint import ATTN_KERNEL, ATTN_ORDER
    w = W.ATTN_WORKLOADS[name].with_(layernorm=True, **over)
    inp = W.make_attn_inputs(w, seed=17, with_bias=True)
    g = torch.Generator().manual_seed(18)
    inp["gamma"] = 1 + 0.2 * torch.randn(w.hidden, generator=g)
    inp["beta"] = 0.2 * torch.randn(w.hidden, generator=g)
    a, n_a, names_a = _run_attn(w, inp, True)
    b, n_b, names_b = _run_attn(w, inp, False)
    assert n_b == n_a + 1, (n_a, n_b)
    assert "gemm_ln_qkv" in names_a and "layernorm_fwd" not in names_a
    assert "layernorm_fwd" in names_b
    assert_bitwise(a, b, ATTN_ORDER, ATTN_KERNEL)
