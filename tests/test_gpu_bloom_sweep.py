"""The BLOOM-176B-shaped layer (h = 14336, f = 57344, weights N(0, 0.006^2))
across its token x shard sweep, against the fp64 oracle on samples.

The BLOOM-176B engineering page splits this layer over tensor-parallel ranks;
the sweep covers the ends of the token range (512 tokens: two 256-row tile
rows, so most of the GPU's pairs get a single tile or none and the weight
gradients' K = T loop is 8 k-blocks; 16384 tokens: about 1.9 GB per H, Y and
dH buffer, 3.3 GB per fp32 weight gradient) and the middle point, each with
several shard counts.  Every point runs the backward step twice in the launch
configuration the benchmark uses and requires bit-identical results (on the
device, before anything is copied back), then checks, from the original
inputs: 256 sampled token rows of Z and dX, 256 sampled ffn columns of dA and
db1, 256 sampled ffn rows of dB, and all of db2."""
import gc

import pytest
import torch

from oracle import mlp as O
from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP

from fingerprint import assert_bitwise
from parity_helpers import assert_close, f64, to_dev

pytestmark = pytest.mark.gpu

NSAMPLE = 256
POINTS = [(512, 1), (512, 2), (512, 8), (4096, 4), (16384, 1), (16384, 2),
          (16384, 8)]


def _run_twice(w, d):
    """Forward + backward twice on the device, separate outputs each time."""
    m = TensorParallelMLP(w.hidden, w.ffn, w.shards, w.tokens)
    outs = []
    for _ in range(2):
        Z = m.forward(d["X"], d["A"], d["B"], training=True)
        g = m.backward(d["dZ"], d["X"], d["A"], d["B"], bias_grads=True)
        assert m.check() == 0
        g["Z"] = Z
        outs.append(g)
    torch.cuda.synchronize()
    m.close()
    return outs


@pytest.mark.parametrize("T,t", POINTS)
def test_bloom_sweep_sampled_and_bitwise(T, t):
    assert T in W.BLOOM_SWEEP_TOKENS and t in W.BLOOM_SWEEP_SHARDS
    w = W.WORKLOADS["bloom_176b"].with_(tokens=T, shards=t)
    inp = W.make_inputs(w, seed=0)
    d = {k: to_dev(v) for k, v in inp.items()}
    r1, r2 = _run_twice(w, d)
    assert_bitwise(r1, r2)
    del r2, d
    gc.collect()
    torch.cuda.empty_cache()

    rows = W.sample_indices(T, NSAMPLE, 100 + T + t)
    fcols = W.sample_indices(w.ffn, NSAMPLE, 200 + T + t)
    got = {
        "Z": r1["Z"][rows.cuda()].cpu(),
        "dX": r1["dX"][rows.cuda()].cpu(),
        "dA": r1["dA"][:, fcols.cuda()].cpu(),
        "db1": r1["db1"][fcols.cuda()].cpu(),
        "dB": r1["dB"][fcols.cuda()].cpu(),
        "db2": r1["db2"].cpu(),
    }
    del r1
    gc.collect()
    torch.cuda.empty_cache()
    rows, fcols = rows.numpy(), fcols.numpy()
    X, A, B, dZ = f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), f64(inp["dZ"])
    del inp
    assert_close("Z[rows]", got["Z"], O.forward_rows(X, A, B, rows))
    assert_close("dX[rows]", got["dX"], O.dxn_rows(dZ, X, A, B, rows))
    dac, db1c = O.dA_cols(dZ, X, A, B, fcols)
    assert_close("dA[:, cols]", got["dA"], dac)
    assert_close("db1[cols]", got["db1"], db1c)
    assert_close("dB[rows]", got["dB"], O.dB_rows(dZ, X, A, fcols))
    assert_close("db2", got["db2"], O.db2(dZ))
