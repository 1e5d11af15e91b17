"""The pair GEMM's tail split on the GPU.

With TPMLP_GEMM_MAX_PAIRS=4 (two groups of two CTA pairs) a GEMM with three
super-tiles runs a last round with one group idle; the split cuts that
super-tile into two pieces (shard segments for the shard sums, k-blocks for
the fp32 weight gradients) whose partials a second kernel combines.  The
same seeded steps run in child processes with the split on and off
(TPMLP_TAIL_SPLIT=2 forces the split at these short K; =0 turns it off):
the shard-sum outputs Z and dX (bias, dropout and
residual applied after the combine, LayerNorm's fp32 dXn) must be bitwise
equal, the k-split fp32 dB within fp32 rounding, and everything within the
bf16 bar against the oracle."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from oracle import fp8 as F
from tensor_transformer_mlp_tcgen05_gb300 import workloads as W

from parity_helpers import assert_close, compare_full, f64, oracle_full

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

DROP = (0.1, 7, 3)
# tokens, hidden, ffn, shards, layernorm, residual, dropout
CASES = [(1536, 256, 1536, 3, False, True, DROP),
         (1536, 256, 1024, 4, True, False, None)]
FP8 = (1536, 256, 1024, 4)

_CHILD = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np, torch
from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
from tensor_transformer_mlp_tcgen05_gb300 import binding as B
from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP
from parity_helpers import run_cuda
from test_gpu_tail_split import CASES, FP8, inputs, fp8_inputs
out = {{}}
for i, (T, h, f, t, ln, res, drop) in enumerate(CASES):
    w, inp = inputs(T, h, f, t, ln)
    got = run_cuda(w, inp, residual=res, dropout=drop)
    for k, v in got.items():
        out["c%d_%s" % (i, k)] = v.float().numpy()
T, h, f, t = FP8
inp = fp8_inputs(T, h, f, t)
m = TensorParallelMLP(h, f, t, T)
d = {{k: (None if v is None else v.cuda()) for k, v in inp.items()}}
packed = m.pack_fp8_weights(d["A"], d["B"])
Z = m.forward_fp8(d["X"], packed, d["b1"], d["b2"], train=True)
g = m.backward_fp8(d["dZ"], d["X"], packed)
assert m.check() == 0
torch.cuda.synchronize()
out["f8_Z"] = Z.float().cpu().numpy()
for k, v in g.items():
    out["f8_" + k] = v.float().cpu().numpy()
out["launches"] = np.array([B.tp_mlp_launch_count(m.handle)])
np.savez({path!r}, **out)
print("child ok")
"""


def inputs(T, h, f, t, ln):
    w = W.Workload("tail", T, h, f, t, "bf16", ln, True, w_std=0.05)
    inp = W.make_inputs(w, seed=T + t, with_bias=True)
    if ln:
        g = torch.Generator().manual_seed(5)
        inp["gamma"] = 1 + 0.2 * torch.randn(h, generator=g)
        inp["beta"] = 0.2 * torch.randn(h, generator=g)
    return w, inp


def fp8_inputs(T, h, f, t):
    w = W.Workload("tail_fp8", T, h, f, t, "bf16", False, True, w_std=0.05)
    return W.make_inputs(w, seed=11, with_bias=True)


def _run(tmp_path, split):
    path = str(tmp_path / ("split.npz" if split else "whole.npz"))
    env = dict(os.environ, TPMLP_GEMM_MAX_PAIRS="4",
               TPMLP_TAIL_SPLIT="2" if split else "0")
    script = _CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"),
                           path=path)
    r = subprocess.run([sys.executable, "-c", script], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return dict(np.load(path))


def test_tail_split_matches_unsplit_and_oracle(tmp_path):
    split, whole = _run(tmp_path, True), _run(tmp_path, False)
    assert split.keys() == whole.keys()
    # the FP8 step's GEMM2 and dX each added a combine launch
    assert split.pop("launches")[0] == whole.pop("launches")[0] + 2
    for k in split:
        name = k.split("_", 1)[1]
        if name in ("dB", "dA"):
            # fp32 weight gradients: the k-split adds two partial sums
            np.testing.assert_allclose(split[k], whole[k], rtol=1e-5,
                                       atol=1e-5 * np.abs(whole[k]).max(),
                                       err_msg=k)
        else:
            np.testing.assert_array_equal(split[k], whole[k], err_msg=k)
    for i, (T, h, f, t, ln, res, drop) in enumerate(CASES):
        w, inp = inputs(T, h, f, t, ln)
        ref = oracle_full(inp, residual=res, dropout=drop)
        got = {k[3:]: torch.from_numpy(v) for k, v in split.items()
               if k.startswith("c%d_" % i)}
        compare_full(got, ref)
    T, h, f, t = FP8
    inp = fp8_inputs(T, h, f, t)
    fwd = F.forward(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]),
                    f64(inp["b1"]), f64(inp["b2"]))
    ref = F.backward(f64(inp["dZ"]), f64(inp["X"]), fwd)
    assert_close("fp8 Z", split["f8_Z"], fwd["Z"])
    for k in ("dX", "dA", "dB", "db1", "db2"):
        assert_close("fp8 " + k, split["f8_" + k], ref[k])
