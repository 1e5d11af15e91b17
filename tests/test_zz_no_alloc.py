"""The allocation-free bias-gradient entry point, for callers that cannot
allocate device memory (an engine that owns the whole device memory pool, or
a tool that must keep the process's device footprint fixed) and so cannot
hand tp_mlp_backward a workspace.  Its output must equal, bit for bit, the
db2 the regular entry point computes (both run the same fixed-order column
sums), agree with the oracle's db2 within the bf16 tolerance, and do so on
two calls in a row that share the library's static scratch (the second call
finds the first call's partial sums there).  Kept in its own file, collected
last."""
import pytest
import torch

from tensor_transformer_mlp_tcgen05_gb300 import binding as B
from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP

from oracle import mlp as O
from parity_helpers import assert_close, f64, to_dev

pytestmark = pytest.mark.gpu


def test_noalloc_bias_grad_matches_backward_twice():
    w = W.Workload("noalloc", 1000, 256, 1024, 4, "bf16", False, True)
    inp = W.make_inputs(w, seed=21, with_bias=True)
    d = {k: to_dev(v) for k, v in inp.items()}
    m = TensorParallelMLP(w.hidden, w.ffn, w.shards, w.tokens)
    m.forward(d["X"], d["A"], d["B"], d["b1"], d["b2"])
    ref = m.backward(d["dZ"], d["X"], d["A"], d["B"])["db2"]
    assert m.check() == 0
    outs = []
    for _ in range(2):
        out = torch.full((w.hidden,), float("nan"), dtype=torch.float32,
                         device="cuda")
        B.tp_mlp_bias_grad_noalloc(w.tokens, w.hidden, B.TPMLP_BF16, d["dZ"],
                                   out)
        outs.append(out)
    torch.cuda.synchronize()
    oracle_db2 = O.db2(f64(inp["dZ"]))
    for out in outs:
        assert torch.equal(out, ref), "no-alloc db2 differs from the backward's"
        assert_close("db2 (no-alloc) vs oracle", out.cpu(), oracle_db2)
    assert torch.equal(outs[0], outs[1])
    m.close()


def test_noalloc_bias_grad_rejects_oversize():
    cols = 4096
    tokens = (B.TPMLP_NOALLOC_SCRATCH_FLOATS // cols) * 256 + 1
    out = torch.empty(cols, dtype=torch.float32, device="cuda")
    with pytest.raises(B.TPMLPError) as e:
        B.tp_mlp_bias_grad_noalloc(tokens, cols, B.TPMLP_BF16, 1 << 20, out)
    assert e.value.code == B.TPMLP_ERR_SHAPE
    assert "static scratch" in str(e.value)
