"""GPU parity of the FP8 (E4M3) training step (tp_mlp_forward_fp8_train and
tp_mlp_backward_fp8 through the binding) against ``oracle/fp8.py``.

dZ is an input, so its codes and scale are decided by both sides from the
same bf16 values with the same fp32 division: they must agree bit for bit,
as must the plain weight codes the backward reads.  H and dH come out of
fp32 GEMMs on the GPU and fp64 ones in the oracle, so their bf16 values
(and a few dH codes at E4M3 rounding boundaries) may differ by one step;
every gradient must meet the bf16 bar (relative Frobenius error <= 5e-3,
max |err| <= 3e-2 max |ref|).  The transposed code sections must be the
plain ones transposed, byte for byte."""
import numpy as np
import pytest
import torch

from oracle import fp8 as F
from tensor_transformer_mlp_tcgen05_gb300 import workloads as W

from fingerprint import assert_bitwise
from parity_helpers import assert_close, f64

pytestmark = pytest.mark.gpu

SECTIONS = ("xq", "yq", "h", "dh", "dzq", "dhq", "xqt", "yqt", "dzqt", "dhqt",
            "scales", "bscales")


def _mlp(w, residual=False, gelu="erf"):
    from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP
    return TensorParallelMLP(w.hidden, w.ffn, w.shards, max(w.tokens, 1),
                             dtype="bf16", layernorm=w.layernorm,
                             residual=residual, gelu=gelu)


def run_step(w, inp, residual=False, repeat=1, bias_grads=True, gelu="erf"):
    m = _mlp(w, residual, gelu)
    d = {k: (None if v is None else v.cuda().contiguous()) for k, v in inp.items()}
    packed = m.pack_fp8_weights(d["A"], d["B"])
    outs = []
    T = w.tokens
    for _ in range(repeat):
        Z = m.forward_fp8(d["X"], packed, d["b1"], d["b2"], d["gamma"],
                          d["beta"], train=True)
        g = m.backward_fp8(d["dZ"], d["X"], packed, d["gamma"],
                           bias_grads=bias_grads)
        assert m.check() == 0
        torch.cuda.synchronize()
        out = {"Z": Z.cpu()}
        out.update({k: v.cpu() for k, v in g.items()})
        for k in SECTIONS:
            v = m.fp8_saved(T, k).cpu()
            out[k] = v.numpy() if v.dtype in (torch.uint8, torch.int32) else v
        out["aq"] = m.fp8_saved(T, "aq", packed).cpu().numpy()
        out["bq"] = m.fp8_saved(T, "bq", packed).cpu().numpy()
        outs.append(out)
    m.close()
    return outs if repeat > 1 else outs[0]


def _f32(word):
    return np.array([word], dtype=np.int32).view(np.float32)[0]


def check(inp, got, residual=False, bias_grads=True, gelu="erf"):
    fwd = F.forward(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]),
                    f64(inp["b1"]), f64(inp["b2"]), f64(inp["gamma"]),
                    f64(inp["beta"]), mode=gelu, residual=residual)
    ref = F.backward(f64(inp["dZ"]), f64(inp["X"]), fwd, f64(inp["gamma"]),
                     mode=gelu, residual=residual)
    # the plain weight codes the backward reads: exactly the oracle's
    np.testing.assert_array_equal(got["aq"], fwd["qa"])
    np.testing.assert_array_equal(got["bq"], fwd["qb"])
    # dZ: codes and scale exactly
    np.testing.assert_array_equal(got["dzq"], ref["qdz"])
    assert _f32(got["bscales"][2]) == ref["sdz"]
    # every transposed section is its plain section transposed
    for plain, tr in (("xq", "xqt"), ("yq", "yqt"), ("dzq", "dzqt"),
                      ("dhq", "dhqt")):
        np.testing.assert_array_equal(got[tr], got[plain].T, err_msg=tr)
    assert_close("Z", got["Z"], fwd["Z"])
    assert_close("H", got["h"], F.to_bf16(fwd["H"]))
    assert_close("dH", got["dh"], ref["dH"])
    assert np.mean(got["dhq"] == ref["qdh"]) > 0.99
    assert abs(_f32(got["bscales"][3]) / ref["sdh"] - 1) < 1e-2
    assert_close("dX", got["dX"], ref["dX"])
    assert_close("dA", got["dA"], ref["dA"])
    assert_close("dB", got["dB"], ref["dB"])
    if bias_grads:
        assert_close("db1", got["db1"], ref["db1"])
        assert_close("db2", got["db2"], ref["db2"])
    if inp["gamma"] is not None:
        assert_close("dgamma", got["dgamma"], ref["dgamma"])
        assert_close("dbeta", got["dbeta"], ref["dbeta"])


CASES = [  # tokens, hidden, ffn, shards, layernorm, bias, residual, GeLU
    (300, 256, 1024, 2, False, True, False, "erf"),
    (129, 256, 1024, 8, False, False, True, "erf"),
    (1, 128, 512, 1, False, True, False, "erf"),
    (513, 384, 1536, 4, True, True, True, "erf"),
    (1000, 192, 768, 3, False, True, True, "erf"),
    (77, 256, 512, 2, True, False, False, "erf"),
    (640, 256, 1024, 4, True, True, True, "tanh"),
]


@pytest.mark.parametrize("T,h,f,t,ln,bias,res,gelu", CASES)
def test_fp8_training_step_parity(T, h, f, t, ln, bias, res, gelu):
    w = W.WORKLOADS["gpt3_13b"].with_(tokens=T, hidden=h, ffn=f, shards=t,
                                       layernorm=ln, w_std=0.05)
    inp = W.make_inputs(w, seed=3 * T + t, with_bias=bias,
                        need_grad_input=True)
    if ln:
        g = torch.Generator().manual_seed(11)
        inp["gamma"] = 1 + 0.2 * torch.randn(h, generator=g)
        inp["beta"] = 0.2 * torch.randn(h, generator=g)
    check(inp, run_step(w, inp, residual=res, bias_grads=bias, gelu=gelu),
          residual=res, bias_grads=bias, gelu=gelu)


def test_fp8_backward_zero_tokens_and_zero_gradient():
    w = W.WORKLOADS["gpt3_13b"].with_(tokens=64, hidden=128, ffn=512,
                                       shards=2)
    inp = W.make_inputs(w, seed=5, with_bias=True, need_grad_input=True)
    inp["dZ"] = torch.zeros_like(inp["dZ"])   # amax 0: scale 1, all codes 0
    got = run_step(w, inp)
    # zeros: dH = 0 * GeLU'(H) is -0 where GeLU'(H) < 0, code 0x80 (the
    # oracle's encoding keeps the sign bit as well)
    assert not (got["dzq"] & 0x7F).any() and not (got["dhq"] & 0x7F).any()
    assert _f32(got["bscales"][2]) == 1.0 and _f32(got["bscales"][3]) == 1.0
    for k in ("dX", "dA", "dB", "db1", "db2"):
        assert not got[k].any(), k
    m = _mlp(w)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    packed = m.pack_fp8_weights(d["A"], d["B"])
    m.forward_fp8(d["X"][:0], packed, train=True)
    g = {k: torch.full(s, 7.0, device="cuda") for k, s in
         (("dA", (128, 512)), ("dB", (512, 128)), ("db1", (512,)),
          ("db2", (128,)))}
    g["dX"] = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    g = m.backward_fp8(d["dZ"][:0], d["X"][:0], packed, grads=g)
    assert m.check() == 0
    for k in ("dA", "dB", "db1", "db2"):
        assert not g[k].any(), k
    m.close()


def test_fp8_backward_rejects_a_short_workspace():
    from tensor_transformer_mlp_tcgen05_gb300 import binding as B
    w = W.WORKLOADS["gpt3_13b"].with_(tokens=64, hidden=128, ffn=512,
                                       shards=2)
    m = _mlp(w)
    fwd = B.tp_mlp_fp8_workspace_bytes(m.handle, 64)
    train = B.tp_mlp_fp8_train_workspace_bytes(m.handle, 64)
    assert 0 < fwd < train
    ws = torch.empty(train - 1, dtype=torch.uint8, device="cuda")
    inp = W.make_inputs(w, seed=2, need_grad_input=True)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    packed = m.pack_fp8_weights(d["A"], d["B"])
    Z = torch.empty_like(d["X"])
    with pytest.raises(B.TPMLPError, match="workspace"):
        B.tp_mlp_forward_fp8_train(m.handle, 64, d["X"], packed, None, None,
                                   None, None, Z, ws, ws.numel())
    dA = torch.empty((128, 512), device="cuda")
    dB = torch.empty((512, 128), device="cuda")
    with pytest.raises(B.TPMLPError, match="workspace"):
        B.tp_mlp_backward_fp8(m.handle, 64, d["dZ"], d["X"], packed, None, ws,
                              ws.numel(), torch.empty_like(d["X"]), dA, dB,
                              None, None, None, None)
    m.close()


def test_fp8_training_step_gpt3_13b_layer():
    """The GPT-3-13B-shaped layer (h = 5120, f = 20480, t = 8): 256 tokens
    against the oracle in full, and the benchmark's 8192 tokens twice,
    bit-identical."""
    w = W.WORKLOADS["gpt3_13b"].with_(tokens=256)
    inp = W.make_inputs(w, seed=0, with_bias=True, need_grad_input=True)
    check(inp, run_step(w, inp))
    w = W.WORKLOADS["gpt3_13b"]
    inp = W.make_inputs(w, seed=0, with_bias=True, need_grad_input=True)
    a, b = run_step(w, inp, repeat=2)
    assert_bitwise(a, b)
    for k in ("dX", "dA", "dB", "db1", "db2"):
        assert torch.isfinite(a[k].float()).all(), k


def _all_bf16_up_to(v, n):
    """Every finite bf16 value with |x| <= v (both signs, zeros, the
    subnormals), then v itself, zero-padded to n entries."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= v)]
    out = np.zeros(n, dtype=np.float32)
    out[:vals.size] = vals
    out[-1] = v
    return torch.from_numpy(out).to(torch.bfloat16)


# amax values: 448 (s = 1: every midpoint exact, ties to even), 1344
# (s = 3), powers of two, a spread of bf16 values with many mantissa bits,
# and amax so small that 1 / s overflows (1e-37) or s is an fp32 denormal
AMAXES = [448.0, 1344.0, 1.0, 2.0 ** -20, 0.0302734375, 0.71484375, 3.140625,
          5.15625, 11.8125, 97.5, 1000.0, 3.3e4, 6.5e5, 1.17e-7, 2.3e-3,
          0.1796875, 7.90625, 250.0, 1.1e9, 1.9e-30, 1.0e-37, 1.0e-39]


@pytest.mark.parametrize("amax", AMAXES)
def test_fp8_quantizers_on_every_bf16_value(amax):
    """Every finite bf16 value below a scale's amax, through the weight
    quantizer (plain and transposed codes) and the activation quantizer,
    bit for bit against the oracle's fp32 division and E4M3 rounding."""
    from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP
    v = float(torch.tensor(amax).to(torch.bfloat16))
    A = _all_bf16_up_to(v, 128 * 512).reshape(128, 512)
    qa, sa = F.quantize(f64(A))
    m = TensorParallelMLP(128, 512, 1, 128, dtype="bf16")
    B = torch.zeros((512, 128), dtype=torch.bfloat16)
    packed = m.pack_fp8_weights(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(m.fp8_saved(128, "aq", packed).cpu().numpy(), qa)
    np.testing.assert_array_equal(m.fp8_saved(128, "aqt", packed).cpu().numpy(),
                                  qa.T)
    assert _f32(m.fp8_saved(128, "wscales", packed).cpu().numpy()[2]) == sa
    m.close()
    # the activation quantizer (plain and, in a training forward, transposed)
    X = _all_bf16_up_to(v, 128 * 512).reshape(128, 512)
    qx, sx = F.quantize(f64(X))
    m = TensorParallelMLP(512, 512, 1, 128, dtype="bf16")
    Aw = torch.zeros((512, 512), dtype=torch.bfloat16, device="cuda")
    packed = m.pack_fp8_weights(Aw, Aw)
    for train in (False, True):
        m.forward_fp8(X.cuda(), packed, train=train)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(m.fp8_saved(128, "xq").cpu().numpy(), qx)
        assert _f32(m.fp8_saved(128, "scales").cpu().numpy()[2]) == sx
        if train:
            np.testing.assert_array_equal(
                m.fp8_saved(128, "xqt").cpu().numpy(), qx.T)
    m.close()
