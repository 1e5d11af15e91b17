"""CUDA path against the fp64 oracle, element by element, on seeded inputs.

Small cases span several 128 x 256 tiles with ragged tails in every GEMM
dimension; the full-size workloads are compared in full where the oracle
finishes in seconds, otherwise on seeded samples of rows and columns that the
oracle computes exactly one by one."""
import numpy as np
import pytest
import torch

from oracle import mlp as O
from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP

from fingerprint import assert_bitwise
from parity_helpers import (assert_close, compare_full, f64, oracle_full,
                            run_cuda, to_dev)

pytestmark = pytest.mark.gpu


def small(T, h, f, t, ln=False, dtype="bf16"):
    return W.Workload("small", T, h, f, t, dtype, ln, True)


# ---------------------------------------------------------------- tiny ----

@pytest.mark.parametrize("with_bias", [False, True])
def test_tiny_fp32_block_full(with_bias):
    w = W.WORKLOADS["tiny_fp32"]
    inp = W.make_inputs(w, seed=0, with_bias=with_bias)
    got = run_cuda(w, inp)
    compare_full(got, oracle_full(inp), fp32=True)


# ------------------------------------------------ small bf16, ragged ----

CASES = [
    # T, h, f, t, ln, bias, gelu
    (300, 256, 1024, 1, False, False, "erf"),
    (300, 256, 1024, 2, False, True, "erf"),
    (300, 256, 1024, 4, True, True, "erf"),
    (129, 320, 1280, 2, True, False, "tanh"),
    (1, 256, 512, 2, False, True, "erf"),
    (1000, 384, 1536, 3, True, True, "erf"),
    (513, 192, 768, 4, False, False, "tanh"),
]


@pytest.mark.parametrize("T,h,f,t,ln,bias,gelu", CASES)
def test_small_bf16_block_full(T, h, f, t, ln, bias, gelu):
    w = small(T, h, f, t, ln)
    inp = W.make_inputs(w, seed=1, with_bias=bias)
    got = run_cuda(w, inp, gelu=gelu)
    compare_full(got, oracle_full(inp, mode=gelu))


# LayerNorm paths with gamma, beta away from (1, 0): the kernels that hold
# the row in registers (h = 3072, forward and backward) and the generic
# row-per-warp loops (h = 192, with lanes idle in the last round of vectors;
# h = 4352 and 8448); the 8-column parameter sums on every case.
@pytest.mark.parametrize("T,h,t,res", [(77, 192, 2, False), (301, 3072, 1, True),
                                       (45, 4352, 2, False), (37, 8448, 1, True)])
def test_layernorm_paths_full(T, h, t, res):
    w = small(T, h, 256 * t, t, ln=True)
    inp = W.make_inputs(w, seed=17, with_bias=True)
    g = torch.Generator().manual_seed(19)
    inp["gamma"] = 1 + 0.3 * torch.randn(h, generator=g)
    inp["beta"] = 0.3 * torch.randn(h, generator=g)
    got = run_cuda(w, inp, residual=res)
    compare_full(got, oracle_full(inp, residual=res))


RESIDUAL_CASES = [
    # T, h, f, t, ln, bias  (the pre-LN sub-block X + MLP(LN(X)) and the
    # plain block with a residual)
    (300, 256, 1024, 4, True, True),
    (300, 256, 1024, 1, False, True),
    (129, 320, 1280, 2, False, False),
    (1000, 384, 1536, 3, True, False),
]


@pytest.mark.parametrize("T,h,f,t,ln,bias", RESIDUAL_CASES)
def test_small_bf16_residual_subblock_full(T, h, f, t, ln, bias):
    w = small(T, h, f, t, ln)
    inp = W.make_inputs(w, seed=9, with_bias=bias)
    got = run_cuda(w, inp, residual=True)
    compare_full(got, oracle_full(inp, residual=True))


def test_tiny_fp32_residual_block_full():
    w = W.WORKLOADS["tiny_fp32"]
    inp = W.make_inputs(w, seed=0, with_bias=True)
    got = run_cuda(w, inp, residual=True)
    compare_full(got, oracle_full(inp, residual=True), fp32=True)


# ------------------------------------------------------------- dropout ----

DROP = (0.1, 0x5EED1234ABCD, 3)


def test_dropout_mask_is_bit_exact():
    """Every keep/drop decision equals the oracle's Philox mask (integer
    decisions: compared exactly, not within a tolerance)."""
    w = small(300, 256, 1024, 4)
    inp = W.make_inputs(w, seed=12)
    got = run_cuda(w, inp, backward=False, dropout=DROP)
    ref = oracle_full(inp, backward=False, dropout=DROP)
    mask = ref["_mask"]
    pre = oracle_full(inp, backward=False)["Z"]
    decided = np.abs(pre) > 1e-3           # a kept value cannot round to 0
    gz = f64(got["Z"]) != 0
    assert np.array_equal(gz[decided], mask[decided])
    assert 0.85 < mask.mean() < 0.95
    assert_close("Z", got["Z"], ref["Z"])


@pytest.mark.parametrize("T,h,f,t,ln,res", [(300, 256, 1024, 4, True, True),
                                            (513, 192, 768, 2, False, False),
                                            (129, 320, 1280, 1, False, True)])
def test_dropout_block_full(T, h, f, t, ln, res):
    w = small(T, h, f, t, ln)
    inp = W.make_inputs(w, seed=13, with_bias=True)
    got = run_cuda(w, inp, residual=res, dropout=DROP)
    compare_full(got, oracle_full(inp, residual=res, dropout=DROP))


def test_tiny_fp32_dropout_block_full():
    w = W.WORKLOADS["tiny_fp32"]
    inp = W.make_inputs(w, seed=0, with_bias=True)
    got = run_cuda(w, inp, residual=True, dropout=(0.25, 77, 0))
    compare_full(got, oracle_full(inp, residual=True, dropout=(0.25, 77, 0)),
                 fp32=True)


def test_dropout_mask_does_not_depend_on_shards_and_is_deterministic():
    base = small(256, 256, 2048, 1)
    inp = W.make_inputs(base, seed=14)
    z1 = run_cuda(base, inp, backward=False, dropout=DROP)["Z"]
    z8a, z8b = run_cuda(base.with_(shards=8), inp, backward=False,
                        dropout=DROP, repeat=2)
    assert_bitwise(z8a, z8b)
    assert torch.equal(z1 == 0, z8a["Z"] == 0)


def test_dropout_only_in_training_calls():
    w = small(256, 256, 1024, 2)
    inp = W.make_inputs(w, seed=15)
    a = run_cuda(w, inp, backward=False, training=False, dropout=DROP)
    b = run_cuda(w, inp, backward=False, training=False)
    assert torch.equal(a["Z"], b["Z"])


def test_small_fp32_layernorm_block_full():
    w = small(200, 128, 512, 4, ln=True, dtype="fp32")
    inp = W.make_inputs(w, seed=2, with_bias=True)
    got = run_cuda(w, inp)
    compare_full(got, oracle_full(inp), fp32=True)


def test_inference_forward_equals_training_forward():
    w = small(300, 256, 1024, 4)
    inp = W.make_inputs(w, seed=3)
    a = run_cuda(w, inp, backward=False, training=False)
    b = run_cuda(w, inp, backward=False, training=True)
    assert torch.equal(a["Z"], b["Z"])


@pytest.mark.parametrize("t", [1, 2, 8])
def test_two_runs_bitwise_identical_small(t):
    w = small(700, 256, 2048, t, ln=True)
    inp = W.make_inputs(w, seed=4, with_bias=True)
    r1, r2 = run_cuda(w, inp, repeat=2)
    assert_bitwise(r1, r2)


def test_shard_count_changes_only_rounding():
    """Different t give the same block up to fp32 summation order."""
    base = small(256, 256, 1024, 1)
    inp = W.make_inputs(base, seed=5)
    z1 = run_cuda(base, inp, backward=False)["Z"]
    z8 = run_cuda(base.with_(shards=8), inp, backward=False)["Z"]
    rel, mx = [float(v) for v in (
        (f64(z8) - f64(z1)).__abs__().max() / np.abs(f64(z1)).max(),
        np.linalg.norm(f64(z8) - f64(z1)) / np.linalg.norm(f64(z1)))]
    assert rel < 1e-2 and mx < 5e-3


# ---------------------------------------------------------- edge cases --

def test_empty_token_set():
    w = small(0, 128, 512, 2, ln=True)
    m = TensorParallelMLP(128, 512, 2, 16, layernorm=True)
    inp = W.make_inputs(w.with_(tokens=4), seed=6)
    d = {k: to_dev(v) for k, v in inp.items()}
    X0 = d["X"][:0]
    Z = m.forward(X0, d["A"], d["B"], None, None, d["gamma"], d["beta"])
    assert Z.shape == (0, 128)
    g = m.backward(d["dZ"][:0], X0, d["A"], d["B"], d["gamma"])
    assert m.check() == 0
    for k in ("dA", "dB", "db1", "db2", "dgamma", "dbeta"):
        assert torch.count_nonzero(g[k]) == 0, k
    m.close()


def test_max_tokens_and_oversize_rejected():
    from tensor_transformer_mlp_tcgen05_gb300.binding import TPMLPError
    w = small(384, 128, 256, 2)
    inp = W.make_inputs(w, seed=7)
    m = TensorParallelMLP(128, 256, 2, 384)
    d = {k: to_dev(v) for k, v in inp.items()}
    Z = m.forward(d["X"], d["A"], d["B"])
    assert m.check() == 0
    assert_close("Z", Z.cpu(), oracle_full(inp, backward=False)["Z"])
    big = torch.zeros((385, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TPMLPError):
        m.forward(big, d["A"], d["B"])
    m.close()


def test_launch_counts_are_fixed():
    """One reduction per direction: forward is exactly two GEMM launches
    (the shard sum lives in the second GEMM's epilogue; with LayerNorm the
    normalisation is the first GEMM's prologue), backward a fixed list of
    kernels (db1's first stage lives in the dH GEMM's epilogue)."""
    from tensor_transformer_mlp_tcgen05_gb300 import binding as B
    for ln, fwd_n, bwd_n in ((False, 2, 7), (True, 2, 11)):
        w = small(256, 256, 1024, 4, ln=ln)
        inp = W.make_inputs(w, seed=8, with_bias=True)
        m = TensorParallelMLP(256, 1024, 4, 256, layernorm=ln)
        d = {k: to_dev(v) for k, v in inp.items()}
        B.tp_mlp_set_timing(m.handle, True)
        m.forward(d["X"], d["A"], d["B"], d["b1"], d["b2"], d["gamma"], d["beta"])
        assert B.tp_mlp_launch_count(m.handle) == fwd_n
        m.backward(d["dZ"], d["X"], d["A"], d["B"], d["gamma"])
        assert B.tp_mlp_launch_count(m.handle) == fwd_n + bwd_n
        assert m.check() == 0
        names = [n for n, _, _ in B.tp_mlp_timing_get(m.handle)]
        assert "gemm2_shardsum" in names and "gemm_dx_shardsum" in names
        m.close()


# --------------------------------------------------- full-size workloads --

@pytest.mark.parametrize("t", [1, 4])
def test_gpt2_medium_forward_full(t):
    w = W.WORKLOADS["gpt2_medium"].with_(shards=t)
    inp = W.make_inputs(w, seed=0)
    got = run_cuda(w, inp, backward=False)
    compare_full(got, oracle_full(inp, backward=False))


def test_megatron_8p3b_block_full():
    """Pre-LN, t = 8: every output against the full fp64 oracle."""
    w = W.WORKLOADS["megatron_8p3b"]
    inp = W.make_inputs(w, seed=0)
    got = run_cuda(w, inp)
    compare_full(got, oracle_full(inp))


def test_megatron_8p3b_pre_ln_subblock_full():
    """The whole pre-LN sub-block X + MLP(LN(X)) at the 8.3B shape, in full,
    and bitwise identical over two runs."""
    w = W.WORKLOADS["megatron_8p3b"]
    inp = W.make_inputs(w, seed=0)
    r1, r2 = run_cuda(w, inp, residual=True, repeat=2)
    assert_bitwise(r1, r2)
    compare_full(r1, oracle_full(inp, residual=True))


def _sampled_check(w, inp, got, nrows, ncols, seed):
    X, A, B = f64(inp["X"]), f64(inp["A"]), f64(inp["B"])
    dZ = f64(inp["dZ"])
    gamma, beta = f64(inp["gamma"]), f64(inp["beta"])
    kw = dict(b1=f64(inp["b1"]), gamma=gamma, beta=beta)
    rows = W.sample_indices(w.tokens, nrows, seed).numpy()
    fcols = W.sample_indices(w.ffn, ncols, seed + 1).numpy()
    assert_close("Z[rows]", got["Z"][rows],
                 O.forward_rows(X, A, B, rows, b2=f64(inp["b2"]), **kw))
    dxn = O.dxn_rows(dZ, X, A, B, rows, **kw)
    if gamma is not None:
        Xr = X[rows]
        _, mean, rstd = O.layernorm_forward(Xr, gamma, beta)
        dxn = O.layernorm_backward(dxn, Xr, mean, rstd, gamma)[0]
    assert_close("dX[rows]", got["dX"][rows], dxn)
    dac, db1c = O.dA_cols(dZ, X, A, B, fcols, **kw)
    assert_close("dA[:,cols]", got["dA"][:, fcols], dac)
    assert_close("db1[cols]", got["db1"][fcols], db1c)
    assert_close("dB[rows]", got["dB"][fcols], O.dB_rows(dZ, X, A, fcols, **kw))
    assert_close("db2", got["db2"], O.db2(dZ))


def test_gpt3_13b_sampled_and_bitwise_identical():
    w = W.WORKLOADS["gpt3_13b"]
    inp = W.make_inputs(w, seed=0)
    r1, r2 = run_cuda(w, inp, repeat=2)
    assert_bitwise(r1, r2)
    _sampled_check(w, inp, r1, nrows=256, ncols=256, seed=11)
