"""GPU parity of the FP8 (E4M3) forward (tp_mlp_fp8_pack_weights and
tp_mlp_forward_fp8 through the binding) against ``oracle/fp8.py``.

The quantization decisions are integers, taken by both sides from the same
fp32 values with the same fp32 division, so the weight codes, their scales
and (without LayerNorm) the activation codes and scale must agree bit for
bit.  Y is produced by an fp32 GEMM on the GPU and an fp64 one in the
oracle, so its bf16 values (and hence some Y codes at E4M3 rounding
boundaries) may differ by one step; Z must meet the bf16 bar."""
import numpy as np
import pytest
import torch

from oracle import fp8 as F
from tensor_transformer_mlp_tcgen05_gb300 import workloads as W

from fingerprint import assert_bitwise
from parity_helpers import assert_close, f64

pytestmark = pytest.mark.gpu


def _mlp(w, residual=False):
    from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP
    return TensorParallelMLP(w.hidden, w.ffn, w.shards, max(w.tokens, 1),
                             dtype="bf16", layernorm=w.layernorm,
                             residual=residual)


def run_fp8(w, inp, residual=False, repeat=1):
    m = _mlp(w, residual)
    d = {k: (None if v is None else v.cuda().contiguous()) for k, v in inp.items()}
    packed = m.pack_fp8_weights(d["A"], d["B"])
    outs = []
    for _ in range(repeat):
        Z = m.forward_fp8(d["X"], packed, d["b1"], d["b2"], d["gamma"],
                          d["beta"])
        assert m.check() == 0
        torch.cuda.synchronize()
        T = w.tokens
        outs.append({
            "Z": Z.cpu(),
            "xq": m.fp8_saved(T, "xq").cpu().numpy(),
            "y": m.fp8_saved(T, "y").cpu(),
            "yq": m.fp8_saved(T, "yq").cpu().numpy(),
            "scales": m.fp8_saved(T, "scales").cpu().numpy(),
            "aqt": m.fp8_saved(T, "aqt", packed).cpu().numpy(),
            "bqt": m.fp8_saved(T, "bqt", packed).cpu().numpy(),
            "wscales": m.fp8_saved(T, "wscales", packed).cpu().numpy()})
    m.close()
    return outs if repeat > 1 else outs[0]


def _f32(word):
    return np.array([word], dtype=np.int32).view(np.float32)[0]


def check(w, inp, got, residual=False):
    ref = F.forward(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]),
                    f64(inp["b1"]), f64(inp["b2"]), f64(inp["gamma"]),
                    f64(inp["beta"]), residual=residual)
    # weights: codes (stored transposed) and scales exactly
    np.testing.assert_array_equal(got["aqt"], ref["qa"].T)
    np.testing.assert_array_equal(got["bqt"], ref["qb"].T)
    assert _f32(got["wscales"][2]) == ref["sa"]
    assert _f32(got["wscales"][3]) == ref["sb"]
    # activations
    if inp["gamma"] is None:
        np.testing.assert_array_equal(got["xq"], ref["qx"])
        assert _f32(got["scales"][2]) == ref["sx"]
    else:
        assert np.mean(got["xq"] == ref["qx"]) > 0.999
    assert_close("Y", got["y"], ref["Y"])
    assert np.mean(got["yq"] == ref["qy"]) > 0.99
    assert abs(_f32(got["scales"][3]) / ref["sy"] - 1) < 1e-2
    assert_close("Z", got["Z"], ref["Z"])


CASES = [  # tokens, hidden, ffn, shards, layernorm, bias, residual
    (300, 256, 1024, 2, False, True, False),
    (129, 256, 1024, 8, False, False, False),
    (1, 128, 512, 1, False, True, False),
    (513, 384, 1536, 4, True, True, True),
    (1000, 192, 768, 3, False, True, True),
]


@pytest.mark.parametrize("T,h,f,t,ln,bias,res", CASES)
def test_fp8_forward_parity(T, h, f, t, ln, bias, res):
    w = W.WORKLOADS["gpt3_13b"].with_(tokens=T, hidden=h, ffn=f, shards=t,
                                       layernorm=ln, w_std=0.05)
    inp = W.make_inputs(w, seed=T + t, with_bias=bias, need_grad_input=False)
    if ln:
        g = torch.Generator().manual_seed(9)
        inp["gamma"] = 1 + 0.2 * torch.randn(h, generator=g)
        inp["beta"] = 0.2 * torch.randn(h, generator=g)
    check(w, inp, run_fp8(w, inp, residual=res), residual=res)


def test_fp8_rejects_unsupported_configs():
    from tensor_transformer_mlp_tcgen05_gb300 import binding as B
    from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP
    m = TensorParallelMLP(256, 768, 3, 64)          # f / t = 256: fine
    assert B.tp_mlp_fp8_weights_bytes(m.handle) > 0
    m.close()
    m = TensorParallelMLP(256, 768, 4, 64)          # f / t = 192: not % 128
    assert B.tp_mlp_fp8_weights_bytes(m.handle) == 0
    m.close()
    m = TensorParallelMLP(64, 256, 2, 64, dtype="fp32")
    assert B.tp_mlp_fp8_weights_bytes(m.handle) == 0
    m.close()


def test_fp8_zero_tokens_and_zero_input():
    w = W.WORKLOADS["gpt3_13b"].with_(tokens=64, hidden=128, ffn=512,
                                       shards=2)
    inp = W.make_inputs(w, seed=1, need_grad_input=False)
    inp["X"] = torch.zeros_like(inp["X"])           # amax 0: scale 1, codes 0
    got = run_fp8(w, inp)
    assert not got["xq"].any()
    assert _f32(got["scales"][2]) == 1.0
    check(w, inp, got)
    m = _mlp(w)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    packed = m.pack_fp8_weights(d["A"], d["B"])
    Z = m.forward_fp8(d["X"][:0], packed)
    assert Z.shape == (0, 128) and m.check() == 0
    m.close()


def test_fp8_gpt3_13b_layer():
    """The GPT-3-13B-shaped layer (h = 5120, f = 20480, t = 8): 512 tokens
    against the oracle in full, and the benchmark's 8192 tokens twice,
    bit-identical."""
    w = W.WORKLOADS["gpt3_13b"].with_(tokens=512)
    inp = W.make_inputs(w, seed=0, need_grad_input=False)
    check(w, inp, run_fp8(w, inp))
    w = W.WORKLOADS["gpt3_13b"]
    inp = W.make_inputs(w, seed=0, need_grad_input=False)
    a, b = run_fp8(w, inp, repeat=2)
    assert_bitwise(a, b)
    assert np.isfinite(f64(a["Z"])).all()
