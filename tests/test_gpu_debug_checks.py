"""The debug build (-DTPMLP_CHECKS, libtpmlp_checks.so) on the GPU.

Its kernels verify, before every TMA copy and every computed store, the
conditions the hardware does not check (the innermost tile coordinate on a
16-byte boundary, store addresses and index ranges) and would report
TPMLP_ERR_CHECK instead of making the access.  On valid inputs no check may
fire and the arithmetic must not change: child processes run the same steps
through the debug build and the release build (TPMLP_LIB selects the
library) and the outputs must be bitwise equal, with the device status OK.
Cases: ragged bf16 blocks (LayerNorm, biases, residual, several shard
counts), the FP8 training step, and the attention block at head dims 64, 96
and 128."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np, torch
from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
from tensor_transformer_mlp_tcgen05_gb300 import binding as B
from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP
from tensor_transformer_mlp_tcgen05_gb300.attention import TensorParallelAttention
assert B.LIB_PATH == {lib!r}, B.LIB_PATH
out = {{}}
def cuda(inp):
    return {{k: (None if v is None else v.cuda().contiguous()) for k, v in inp.items()}}
def put(prefix, d):
    for k, v in d.items():
        out[prefix + k] = v.detach().float().cpu().numpy()
for i, (T, h, f, t, ln, res) in enumerate([(300, 256, 1024, 4, True, True),
                                            (513, 192, 768, 3, False, False),
                                            (129, 320, 1280, 2, True, False)]):
    w = W.Workload("chk", T, h, f, t, "bf16", ln, True, w_std=0.05)
    d = cuda(W.make_inputs(w, seed=80 + i, with_bias=True))
    m = TensorParallelMLP(h, f, t, T, layernorm=ln, residual=res)
    Z = m.forward(d["X"], d["A"], d["B"], d["b1"], d["b2"], d["gamma"], d["beta"])
    g = m.backward(d["dZ"], d["X"], d["A"], d["B"], d["gamma"])
    rc = m.check()
    assert rc == 0, (rc, B.tp_mlp_last_detail())
    g["Z"] = Z
    put("c%d_" % i, g)
    m.close()
T, h, f, t = 300, 256, 1024, 4
w = W.Workload("chk_fp8", T, h, f, t, "bf16", False, True, w_std=0.05)
d = cuda(W.make_inputs(w, seed=90, with_bias=True))
m = TensorParallelMLP(h, f, t, T)
packed = m.pack_fp8_weights(d["A"], d["B"])
Z = m.forward_fp8(d["X"], packed, d["b1"], d["b2"], train=True)
g = m.backward_fp8(d["dZ"], d["X"], packed)
rc = m.check()
assert rc == 0, (rc, B.tp_mlp_last_detail())
g["Z"] = Z
put("f8_", g)
m.close()
for name in ("attn_tiny_d64", "attn_tiny_d96", "attn_tiny_d128"):
    aw = W.ATTN_WORKLOADS[name]
    d = cuda(W.make_attn_inputs(aw, seed=91, with_bias=True))
    m = TensorParallelAttention(aw.hidden, aw.heads, aw.shards, aw.tokens,
                                aw.seq, causal=aw.causal)
    Z = m.forward(d["X"], d["Wqkv"], d["Wo"], d["bqkv"], d["bo"])
    g = m.backward(d["dZ"], d["X"], d["Wqkv"], d["Wo"])
    rc = m.check()
    assert rc == 0, (rc, B.tp_mlp_last_detail())
    g["Z"] = Z
    put(name + "_", g)
    m.close()
np.savez({path!r}, **out)
print("child ok")
"""


def _run(tmp_path, lib, tag):
    path = str(tmp_path / f"{tag}.npz")
    env = dict(os.environ, TPMLP_LIB=lib)
    script = _CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"),
                           path=path, lib=lib)
    r = subprocess.run([sys.executable, "-c", script], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return dict(np.load(path))


def test_debug_build_changes_nothing_on_valid_inputs(tmp_path):
    from tensor_transformer_mlp_tcgen05_gb300 import build
    checked = build.build(checks=True)
    release = build.build()
    a = _run(tmp_path, checked, "checked")
    b = _run(tmp_path, release, "release")
    assert a.keys() == b.keys() and len(a) >= 30
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
