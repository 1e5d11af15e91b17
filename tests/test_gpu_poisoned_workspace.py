"""Reads of unwritten memory, found without a sanitizer.

Every byte of the caller-owned workspace (including the GEMM tail split's
partial-sum section and the column-sum partials), of the packed FP8 weight
buffer and of every output is set to 0xFF before the calls that write them:
as fp32 or bf16 that is a NaN, so any element a kernel reads before some
kernel has written it turns into a NaN in an output.  The same steps then
run on zero-filled buffers, and the two runs must give finite, bitwise-equal
outputs.  The steps run in child processes with the tail split forced at
every size (TPMLP_TAIL_SPLIT=2) and at most four CTA pairs per GEMM launch
(TPMLP_GEMM_MAX_PAIRS=4), so the small ragged shapes below reach the split,
its partial slots and its combine kernel; they cover the bf16 block (ragged
token counts, LayerNorm, biases, residual, dropout), the FP8 training step
and the attention block.  The allocation-free bias gradient is run after a
call that leaves NaN partial sums in its static scratch, and must still equal
the backward's db2 bit for bit."""
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

FILL = {fill}
out = {{}}
dev = "cuda"


def filled(shape, dtype):
    t = torch.empty(shape, dtype=dtype, device=dev)
    t.view(torch.uint8).fill_(FILL) if t.numel() else None
    return t


def put(prefix, d):
    for k, v in d.items():
        out[prefix + k] = v.detach().float().cpu().numpy()


def cuda(inp):
    return {{k: (None if v is None else v.cuda().contiguous())
            for k, v in inp.items()}}


# bf16 block: tokens, hidden, ffn, shards, layernorm, residual, dropout
CASES = [(1536, 256, 1536, 3, False, True, (0.1, 7, 3)),
         (1000, 192, 768, 4, True, False, None),
         (513, 256, 1024, 2, True, True, None)]
for i, (T, h, f, t, ln, res, drop) in enumerate(CASES):
    w = W.Workload("poison", T, h, f, t, "bf16", ln, True, w_std=0.05)
    inp = W.make_inputs(w, seed=60 + i, with_bias=True)
    if ln:
        g = torch.Generator().manual_seed(9)
        inp["gamma"] = 1 + 0.2 * torch.randn(h, generator=g)
        inp["beta"] = 0.2 * torch.randn(h, generator=g)
    d = cuda(inp)
    p, seed, offset = drop if drop else (0.0, 0, 0)
    m = TensorParallelMLP(h, f, t, T, layernorm=ln, residual=res,
                          dropout_p=p, dropout_seed=seed,
                          dropout_offset=offset)
    m.workspace(T, True).fill_(FILL)
    Z = filled((T, h), torch.bfloat16)
    m.forward(d["X"], d["A"], d["B"], d["b1"], d["b2"], d["gamma"],
              d["beta"], training=True, out=Z)
    g = {{"dX": filled((T, h), torch.bfloat16),
         "dA": filled((h, f), torch.float32),
         "dB": filled((f, h), torch.float32),
         "db1": filled((f,), torch.float32),
         "db2": filled((h,), torch.float32)}}
    if ln:
        g["dgamma"] = filled((h,), torch.float32)
        g["dbeta"] = filled((h,), torch.float32)
    m.backward(d["dZ"], d["X"], d["A"], d["B"], d["gamma"], out=g)
    assert m.check() == 0
    g["Z"] = Z
    put("c%d_" % i, g)
    if i == 2:
        # the allocation-free bias gradient, after a call that leaves NaN
        # partial sums in its static scratch (a case without dropout, where
        # db2 is the plain column sum of dZ)
        nan_grad = torch.full((T, h), float("nan"), dtype=torch.bfloat16,
                              device=dev)
        junk = torch.empty(h, dtype=torch.float32, device=dev)
        B.tp_mlp_bias_grad_noalloc(T, h, B.TPMLP_BF16, nan_grad, junk)
        db2 = filled((h,), torch.float32)
        B.tp_mlp_bias_grad_noalloc(T, h, B.TPMLP_BF16, d["dZ"], db2)
        torch.cuda.synchronize()
        assert torch.isnan(junk).all()
        assert torch.equal(db2, g["db2"]), "no-alloc db2 after NaN scratch"
        out["noalloc_db2"] = db2.cpu().numpy()
    m.close()

# FP8 training step
T, h, f, t = 1536, 256, 1024, 4
w = W.Workload("poison_fp8", T, h, f, t, "bf16", False, True, w_std=0.05)
d = cuda(W.make_inputs(w, seed=70, with_bias=True))
m = TensorParallelMLP(h, f, t, T)
packed = torch.empty(B.tp_mlp_fp8_weights_bytes(m.handle), dtype=torch.uint8,
                     device=dev).fill_(FILL)
B.tp_mlp_fp8_pack_weights(m.handle, d["A"], d["B"], packed, packed.numel(),
                          None)
need = B.tp_mlp_fp8_train_workspace_bytes(m.handle, T)
m._ws = torch.empty(need, dtype=torch.uint8, device=dev).fill_(FILL)
Z = filled((T, h), torch.bfloat16)
m.forward_fp8(d["X"], packed, d["b1"], d["b2"], out=Z, train=True)
g = {{"dX": filled((T, h), torch.bfloat16), "dA": filled((h, f), torch.float32),
     "dB": filled((f, h), torch.float32), "db1": filled((f,), torch.float32),
     "db2": filled((h,), torch.float32)}}
m.backward_fp8(d["dZ"], d["X"], packed, grads=g)
assert m.check() == 0
g["Z"] = Z
put("f8_", g)
m.close()

# attention block (LayerNorm, residual, biases)
aw = W.ATTN_WORKLOADS["attn_tiny_d64"].with_(layernorm=True)
inp = W.make_attn_inputs(aw, seed=71, with_bias=True)
g0 = torch.Generator().manual_seed(9)
inp["gamma"] = 1 + 0.2 * torch.randn(aw.hidden, generator=g0)
inp["beta"] = 0.2 * torch.randn(aw.hidden, generator=g0)
d = cuda(inp)
T, h = aw.tokens, aw.hidden
m = TensorParallelAttention(h, aw.heads, aw.shards, T, aw.seq, causal=True,
                            layernorm=True, residual=True)
m.workspace(T, True).fill_(FILL)
Z = filled((T, h), torch.bfloat16)
m.forward(d["X"], d["Wqkv"], d["Wo"], d["bqkv"], d["bo"], d["gamma"],
          d["beta"], training=True, out=Z)
g = {{"dX": filled((T, h), torch.bfloat16),
     "dWqkv": filled((h, 3 * h), torch.float32),
     "dWo": filled((h, h), torch.float32),
     "dbqkv": filled((3 * h,), torch.float32),
     "dbo": filled((h,), torch.float32),
     "dgamma": filled((h,), torch.float32),
     "dbeta": filled((h,), torch.float32)}}
m.backward(d["dZ"], d["X"], d["Wqkv"], d["Wo"], d["gamma"], out=g)
assert m.check() == 0
g["Z"] = Z
put("at_", g)
m.close()
np.savez({path!r}, **out)
print("child ok")
"""


def _run(tmp_path, fill):
    path = str(tmp_path / f"fill{fill}.npz")
    env = dict(os.environ, TPMLP_GEMM_MAX_PAIRS="4", TPMLP_TAIL_SPLIT="2")
    script = _CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"),
                           path=path, fill=fill)
    r = subprocess.run([sys.executable, "-c", script], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return dict(np.load(path))


def test_poisoned_buffers_change_nothing(tmp_path):
    nan_run = _run(tmp_path, 0xFF)
    zero_run = _run(tmp_path, 0x00)
    assert nan_run.keys() == zero_run.keys()
    assert len(nan_run) >= 30
    for k, v in nan_run.items():
        assert np.isfinite(v).all(), f"{k}: non-finite values on NaN-filled buffers"
        np.testing.assert_array_equal(v, zero_run[k], err_msg=k)
