"""Bounded-wait failure reporting on the GPU.

The timeout test makes every bounded wait inside the GEMM kernels give up at
once (a 1 ns budget): the kernels must return on their own, report
TPMLP_ERR_TIMEOUT through the status word, and leave the CUDA context usable
(a normal call afterwards still matches the oracle).  Nothing here faults,
traps or hangs the GPU: every wait, including the teardown ones, is bounded.
"""
import os
import subprocess
import sys

import pytest
import torch

from tensor_transformer_mlp_tcgen05_gb300 import binding as B
from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP

from parity_helpers import assert_close, oracle_full, to_dev

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_wait_timeout_is_reported_and_context_survives():
    w = W.Workload("timeout", 1024, 256, 2048, 2, "bf16", False, True)
    inp = W.make_inputs(w, seed=31)
    d = {k: to_dev(v) for k, v in inp.items()}
    m = TensorParallelMLP(w.hidden, w.ffn, w.shards, w.tokens)
    B.tp_mlp_set_wait_budget(m.handle, 1)
    m.forward(d["X"], d["A"], d["B"])
    rc = m.check()
    assert rc == B.TPMLP_ERR_TIMEOUT, (rc, B.tp_mlp_last_detail())
    assert "role" in B.tp_mlp_last_detail()
    # The status word is cleared by the check; with the default budget the
    # same handle and context compute the right answer again.
    B.tp_mlp_set_wait_budget(m.handle, 2_000_000_000)
    Z = m.forward(d["X"], d["A"], d["B"])
    assert m.check() == B.TPMLP_OK
    assert_close("Z after timeout", Z.cpu(), oracle_full(inp, backward=False)["Z"])
    m.close()


def test_layernorm_prologue_wait_timeout_is_reported_and_context_survives():
    """The same with the LayerNorm inside GEMM1's launch: the producers' waits
    for the normalised row blocks give up with the rest, and afterwards the
    same handle computes the block (LayerNorm included) correctly."""
    w = W.Workload("timeout_ln", 1000, 512, 2048, 2, "bf16", True, True)
    inp = W.make_inputs(w, seed=33, with_bias=True)
    d = {k: to_dev(v) for k, v in inp.items()}
    m = TensorParallelMLP(w.hidden, w.ffn, w.shards, w.tokens, layernorm=True)
    B.tp_mlp_set_wait_budget(m.handle, 1)
    m.forward(d["X"], d["A"], d["B"], d["b1"], d["b2"], d["gamma"], d["beta"])
    rc = m.check()
    assert rc == B.TPMLP_ERR_TIMEOUT, (rc, B.tp_mlp_last_detail())
    B.tp_mlp_set_wait_budget(m.handle, 2_000_000_000)
    Z = m.forward(d["X"], d["A"], d["B"], d["b1"], d["b2"], d["gamma"],
                  d["beta"])
    assert m.check() == B.TPMLP_OK
    assert_close("Z after timeout", Z.cpu(), oracle_full(inp, backward=False)["Z"])
    m.close()


def test_attention_wait_timeout_is_reported_and_context_survives():
    """The same for the attention block: every bounded wait in the attention
    forward and backward kernels (and their GEMMs) gives up at once, the
    calls report TPMLP_ERR_TIMEOUT, and the context then computes the block
    correctly."""
    from oracle import attention as OA
    from tensor_transformer_mlp_tcgen05_gb300.attention import \
        TensorParallelAttention
    from parity_helpers import f64
    # 40 sequences: 320 query-block items, more than the persistent forward
    # has CTAs, so CTAs that give up leave items of theirs unwalked
    w = W.ATTN_WORKLOADS["attn_tiny_d64"].with_(batch=40)
    inp = W.make_attn_inputs(w, seed=32, with_bias=True)
    d = {k: to_dev(v) for k, v in inp.items()}
    m = TensorParallelAttention(w.hidden, w.heads, w.shards, w.tokens, w.seq)
    B.tp_attn_set_wait_budget(m.handle, 1)
    m.forward(d["X"], d["Wqkv"], d["Wo"], d["bqkv"], d["bo"])
    rc = m.check()
    assert rc == B.TPMLP_ERR_TIMEOUT, (rc, B.tp_mlp_last_detail())
    m.backward(d["dZ"], d["X"], d["Wqkv"], d["Wo"])
    rc = m.check()
    assert rc == B.TPMLP_ERR_TIMEOUT, (rc, B.tp_mlp_last_detail())
    B.tp_attn_set_wait_budget(m.handle, 2_000_000_000)
    Z = m.forward(d["X"], d["Wqkv"], d["Wo"], d["bqkv"], d["bo"])
    assert m.check() == B.TPMLP_OK
    ref = OA.forward(f64(inp["X"]), f64(inp["Wqkv"]), f64(inp["Wo"]), w.heads,
                     w.seq, w.shards, bqkv=f64(inp["bqkv"]), bo=f64(inp["bo"]))
    assert_close("attention Z after timeout", Z.cpu(), ref["Z"])
    m.close()


def test_nvtx_ranges_change_nothing():
    """NVTX ranges around the launches (no tool attached): the same kernels,
    the same launch count and bitwise the same results."""
    w = W.Workload("nvtx", 300, 256, 1024, 4, "bf16", True, True)
    inp = W.make_inputs(w, seed=33, with_bias=True)
    d = {k: to_dev(v) for k, v in inp.items()}
    outs = []
    for enable in (False, True):
        m = TensorParallelMLP(w.hidden, w.ffn, w.shards, w.tokens,
                              layernorm=True)
        B.tp_mlp_set_nvtx(m.handle, enable)
        Z = m.forward(d["X"], d["A"], d["B"], d["b1"], d["b2"], d["gamma"],
                      d["beta"])
        g = m.backward(d["dZ"], d["X"], d["A"], d["B"], d["gamma"])
        assert m.check() == B.TPMLP_OK
        g["Z"] = Z
        outs.append(({k: v.cpu() for k, v in g.items()},
                     B.tp_mlp_launch_count(m.handle)))
        m.close()
    assert outs[0][1] == outs[1][1]
    for k in outs[0][0]:
        assert torch.equal(outs[0][0][k], outs[1][0][k]), k
