"""GPU parity of the head-parallel attention block (tp_attn_* through the
binding) against the fp64 oracle in ``oracle/attention.py``.

Element-by-element comparisons on seeded inputs at sizes the oracle finishes
in seconds (several 128-row blocks per sequence, two to forty sequences
(more query blocks than the persistent forward has CTAs), shards 1-4,
head dims 64, 96 and 128, causal and not, with and without LayerNorm, biases and
the residual), plus bitwise repeatability and the empty call."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from tensor_transformer_mlp_tcgen05_gb300 import workloads as W

import attention_rounding as R
from fingerprint import ATTN_KERNEL, ATTN_ORDER, assert_bitwise
from parity_helpers import assert_close, errors, f64

pytestmark = pytest.mark.gpu

LOG2E = 1.0 / math.log(2.0)

# Tolerances.  Forward outputs (QKV, Ctx, the log-sum-exp, Z) keep the
# block's bf16 bar: relative Frobenius error <= 5e-3, max |err| <= 3e-2
# max |ref|.  The gradients are bounded by the bf16 storage of the block's
# intermediates: the fp64 block with bf16 rounding at the kernels' seven
# storage points (tests/attention_rounding.py: LayerNorm output, Q/K/V, the
# staged P, Ctx, dCtx, the staged dS, dQ/dK/dV) has, against the exact
# block, the same errors the kernels show (e.g. dQKV 5.61e-3 emulated and
# 5.61e-3 measured for the full-attention, LayerNorm, residual case; Q/K/V
# alone 3-3.6e-3, the LayerNorm output alone ~3e-3).  The gradient bar is
# set just above the measured worst case, 6.4e-3 (dK of the 8.3B layer's
# sampled heads), with the max |err| bar unchanged.  In addition the
# gradients must agree with that emulation within TOL_EMU (measured <=
# 2.5e-3: the forward stages P before its normalisation and the query
# kernel stages dS before its row correction, so those two roundings fall
# on different values).  Exact sums (db_o = sum_T dZ) land near 1e-8.
FWD_KEYS = ("Z", "QKV", "Ctx", "lse")
TOL_GRAD = (7e-3, 3e-2)
TOL_EMU = (4e-3, 3e-2)


def run_attn(w, inp, backward=True, residual=False, repeat=1):
    from tensor_transformer_mlp_tcgen05_gb300.attention import \
        TensorParallelAttention
    m = TensorParallelAttention(w.hidden, w.heads, w.shards, w.tokens,
                                w.seq, causal=w.causal,
                                layernorm=w.layernorm, residual=residual)
    d = {k: (None if v is None else v.cuda().contiguous())
         for k, v in inp.items()}
    outs = []
    for _ in range(repeat):
        Z = m.forward(d["X"], d["Wqkv"], d["Wo"], d["bqkv"], d["bo"],
                      d["gamma"], d["beta"], training=True)
        res = {"Z": Z,
               "QKV": m.saved(w.tokens, "qkv").clone(),
               "Ctx": m.saved(w.tokens, "ctx").clone(),
               "lse2": m.saved(w.tokens, "lse2").clone()}
        if backward:
            res.update(m.backward(d["dZ"], d["X"], d["Wqkv"], d["Wo"],
                                  d["gamma"]))
            res["dQKV"] = m.saved(w.tokens, "dqkv").clone()
        rc = m.check()
        assert rc == 0, f"device status {rc}"
        torch.cuda.synchronize()
        outs.append({k: v.cpu() for k, v in res.items()})
    m.close()
    return outs if repeat > 1 else outs[0]


def oracle(w, inp, backward=True, residual=False):
    kw = dict(bqkv=f64(inp["bqkv"]), bo=f64(inp["bo"]), gamma=f64(inp["gamma"]),
              beta=f64(inp["beta"]), causal=w.causal, residual=residual)
    fwd = A.forward(f64(inp["X"]), f64(inp["Wqkv"]), f64(inp["Wo"]), w.heads,
                    w.seq, w.shards, **kw)
    out = {"Z": fwd["Z"], "QKV": fwd["QKV"], "Ctx": fwd["Ctx"],
           "lse": fwd["lse"]}
    if backward:
        g = A.backward(f64(inp["dZ"]), f64(inp["X"]), f64(inp["Wqkv"]),
                       f64(inp["Wo"]), fwd, w.heads, w.seq, w.shards,
                       gamma=f64(inp["gamma"]), causal=w.causal,
                       residual=residual)
        out.update({k: g[k] for k in ("dX", "dWqkv", "dWo", "dbqkv", "dbo",
                                      "dQKV")})
        if inp["gamma"] is not None:
            out.update(dgamma=g["dgamma"], dbeta=g["dbeta"])
    return out


def compare(got, ref):
    report = {}
    for k, v in ref.items():
        if k == "lse":
            # the kernel keeps log2-sum-exp of log2(e)-scaled scores
            report[k] = assert_close(k, f64(got["lse2"]).T / LOG2E, v)
        elif k in FWD_KEYS:
            report[k] = assert_close(k, got[k], v)
        else:
            rel_fro, max_rel = errors(got[k], v)
            assert np.all(np.isfinite(f64(got[k]))), k
            assert rel_fro <= TOL_GRAD[0] and max_rel <= TOL_GRAD[1], (
                f"{k}: rel_fro={rel_fro:.3e} (tol {TOL_GRAD[0]}), "
                f"max_rel={max_rel:.3e} (tol {TOL_GRAD[1]})")
            report[k] = (rel_fro, max_rel)
    return report


CASES = [
    # name, overrides, bias, residual
    ("d64_causal_t2", {}, True, False),
    ("d64_causal_t1", dict(shards=1), False, False),
    ("d64_full_t4", dict(causal=False, shards=4), True, False),
    ("d128_causal_t2", {}, True, False),
    ("d128_full_t1_ln_res", dict(causal=False, shards=1, layernorm=True), True,
     True),
    ("d128_causal_t4_ln", dict(shards=4, layernorm=True), False, False),
    # exact +-4 projections (see make_attn_sign_inputs): score std 16, so
    # the running row max keeps rising by more than the forward kernel's
    # rescale threshold across key blocks
    ("d64_causal_peaked", dict(seq=512, batch=1), "sign", False),
    ("d128_full_peaked", dict(causal=False), "sign", False),
    # head dim 96, the 8.3B model's 3072 / 32
    ("d96_causal_t2", {}, True, False),
    ("d96_full_t1", dict(causal=False, shards=1), False, False),
    ("d96_causal_t4_ln_res", dict(shards=4, layernorm=True), True, True),
    ("d96_full_t2_ln", dict(causal=False, layernorm=True), True, False),
    ("d96_causal_peaked", dict(seq=384, batch=1), "sign", False),
    # more (sequence, head, query block) items than the persistent forward
    # has CTAs (two per SM): a CTA walks several items, in rounds
    ("d64_causal_items320", dict(batch=40), True, False),
    ("d96_full_t4_items320", dict(batch=20, causal=False, shards=4), False,
     False),
]


def _workload(name, over):
    base = {"d64": "attn_tiny_d64", "d96": "attn_tiny_d96",
            "d128": "attn_tiny_d128"}[name.split("_")[0]]
    return W.ATTN_WORKLOADS[base].with_(**over)


@pytest.mark.parametrize("name,over,bias,res", CASES, ids=[c[0] for c in CASES])
def test_attention_forward_backward_parity(name, over, bias, res):
    w = _workload(name, over)
    if bias == "sign":
        inp = W.make_attn_sign_inputs(w, seed=11)
    else:
        inp = W.make_attn_inputs(w, seed=11, with_bias=bias)
    if w.layernorm:   # exercise gamma and beta away from (1, 0)
        g = torch.Generator().manual_seed(5)
        inp["gamma"] = 1 + 0.2 * torch.randn(w.hidden, generator=g)
        inp["beta"] = 0.2 * torch.randn(w.hidden, generator=g)
    got = run_attn(w, inp, residual=res)
    ref = oracle(w, inp, residual=res)
    report = compare(got, ref)
    print(name, " ".join(f"{k}={v[0]:.2e}/{v[1]:.2e}"
                         for k, v in sorted(report.items())))
    emu = R.backward_rounded(inp, w.heads, w.seq, w.shards, w.causal, res,
                             R.POINTS)
    emu["dX"] = R.bf16(emu["dX"])          # the output's own dtype
    for k in ("dQKV", "dX", "dWqkv", "dWo"):
        rel_fro, max_rel = errors(got[k], emu[k])
        print(name, "vs emulated", k, f"{rel_fro:.2e}/{max_rel:.2e}")
        assert rel_fro <= TOL_EMU[0] and max_rel <= TOL_EMU[1], (
            k, rel_fro, max_rel)


def test_attention_bitwise_repeatable():
    w = W.ATTN_WORKLOADS["attn_tiny_d128"]
    inp = W.make_attn_inputs(w, seed=3, with_bias=True)
    a, b = run_attn(w, inp, repeat=2)
    assert_bitwise(a, b, ATTN_ORDER, ATTN_KERNEL)


def test_attention_zero_tokens():
    from tensor_transformer_mlp_tcgen05_gb300.attention import \
        TensorParallelAttention
    w = W.ATTN_WORKLOADS["attn_tiny_d64"]
    m = TensorParallelAttention(w.hidden, w.heads, w.shards, w.tokens, w.seq)
    h = w.hidden
    dev = "cuda"
    X = torch.empty((0, h), dtype=torch.bfloat16, device=dev)
    Wqkv = torch.zeros((h, 3 * h), dtype=torch.bfloat16, device=dev)
    Wo = torch.zeros((h, h), dtype=torch.bfloat16, device=dev)
    Z = m.forward(X, Wqkv, Wo)
    assert Z.shape == (0, h)
    g = {k: torch.full(s, 7.0, device=dev)
         for k, s in (("dWqkv", (h, 3 * h)), ("dWo", (h, h)),
                      ("dbqkv", (3 * h,)), ("dbo", (h,)))}
    g = m.backward(torch.empty((0, h), dtype=torch.bfloat16, device=dev), X,
                   Wqkv, Wo, out=g)
    assert m.check() == 0
    for k in ("dWqkv", "dWo", "dbqkv", "dbo"):
        assert torch.count_nonzero(g[k]) == 0, k
    m.close()


def _head_cols(w, j):
    """Columns of head j's q, k, v inside the shard-grouped projection."""
    hs, hp, d = w.hidden // w.shards, w.heads // w.shards, w.head_dim
    i, jj = divmod(j, hp)
    base = 3 * hs * i + jj * d
    return (slice(base, base + d), slice(base + hs, base + hs + d),
            slice(base + 2 * hs, base + 2 * hs + d))


@pytest.mark.parametrize("name,samples", [
    ("attn_gpt3_13b", ((0, 0), (1, 17), (3, 39))),
    ("attn_gpt2_medium", ((0, 0), (5, 9), (7, 15))),
    ("attn_megatron_8p3b", ((0, 0), (3, 13), (7, 31))),
])
def test_attention_full_size_sampled_invariants_and_bitwise(name, samples):
    """The GPT-3-13B-shaped layer (4 x 2048 tokens, h = 5120, 40 heads of
    128, 8 shards, causal), the GPT-2-medium-shaped one (8 x 1024 tokens,
    h = 1024, 16 heads of 64, 4 shards) and the Megatron-8.3B one (8 x 1024
    tokens, h = 3072, 32 heads of 96, 8 shards, pre-LN) at full size, in the launch
    configuration the benchmark times.  Checked against the oracle from the original inputs:
    Ctx, the log-sum-exp and dQKV of sampled (sequence, head) pairs; Z on
    every sequence's first 128 rows (causal rows there see keys 0..127
    only); and over every sequence and head the exact identities
    sum_keys dK = 0 (each row of dS sums to zero) and sum_keys dV =
    sum_queries dO.  Two runs are bit-identical."""
    w = W.ATTN_WORKLOADS[name]
    inp = W.make_attn_inputs(w, seed=0, with_bias=True)
    a, b = run_attn(w, inp, repeat=2)
    assert_bitwise(a, b, ATTN_ORDER, ATTN_KERNEL)
    del b
    S, h, d, H = w.seq, w.hidden, w.head_dim, w.heads
    X, Wqkv, Wo = f64(inp["X"]), f64(inp["Wqkv"]), f64(inp["Wo"])
    bqkv, bo, dZ = f64(inp["bqkv"]), f64(inp["bo"]), f64(inp["dZ"])
    if w.layernorm:   # the projections see LN(X) (gamma = 1, beta = 0)
        X = A.layernorm_forward(X, f64(inp["gamma"]), f64(inp["beta"]))[0]
    ctx, dqkv = f64(a["Ctx"]), f64(a["dQKV"])
    lse2 = f64(a["lse2"])
    # sampled heads: forward core and its backward, from the inputs
    for seq, j in samples:
        rows = slice(seq * S, (seq + 1) * S)
        cq, ck, cv = _head_cols(w, j)
        x = X[rows]
        q = x @ Wqkv[:, cq] + bqkv[cq]
        k = x @ Wqkv[:, ck] + bqkv[ck]
        v = x @ Wqkv[:, cv] + bqkv[cv]
        o, probs, lse = A.attention_core(q[:, None], k[:, None], v[:, None], S,
                                         causal=True)
        assert_close(f"Ctx[{seq},{j}]", ctx[rows, j * d:(j + 1) * d], o[:, 0])
        assert_close(f"lse[{seq},{j}]", lse2[j, rows] / LOG2E, lse[:, 0])
        do = dZ[rows] @ Wo[j * d:(j + 1) * d, :].T
        dq, dk, dv = A.core_backward(q[:, None], k[:, None], v[:, None],
                                     do[:, None], probs, S)
        for nm, cols, ref in (("dQ", cq, dq), ("dK", ck, dk), ("dV", cv, dv)):
            rel_fro, max_rel = errors(dqkv[rows, cols], ref[:, 0])
            print(name, nm, seq, j, f"{rel_fro:.2e}/{max_rel:.2e}")
            assert rel_fro <= TOL_GRAD[0] and max_rel <= TOL_GRAD[1], (
                nm, seq, j, rel_fro, max_rel)
    # Z on the first 128 rows of every sequence
    for seq in range(w.batch):
        rows = slice(seq * S, seq * S + 128)
        qkv = X[rows] @ Wqkv + bqkv
        q, k, v = A._split(qkv, H, w.shards)
        o, _, _ = A.attention_core(q, k, v, 128, causal=True)
        Z = o.reshape(128, h) @ Wo + bo
        assert_close(f"Z[{seq}][:128]", a["Z"][rows], Z)
    # identities over every sequence and head
    sum_dO = np.stack([dZ[s * S:(s + 1) * S].sum(axis=0) @ Wo.T
                       for s in range(w.batch)])          # [batch, h]
    dk_sum, dk_scale, dv_sum = [], [], []
    for s in range(w.batch):
        blk = dqkv[s * S:(s + 1) * S]
        for j in range(H):
            _, ck, cv = _head_cols(w, j)
            dk_sum.append(blk[:, ck].sum(axis=0))
            dk_scale.append(np.sqrt(S) * np.sqrt((blk[:, ck] ** 2).mean(axis=0)))
            dv_sum.append(blk[:, cv].sum(axis=0))
    dk_sum, dk_scale = np.array(dk_sum), np.array(dk_scale)
    # with no cancellation the sum of S terms has the size sqrt(S) rms
    assert np.linalg.norm(dk_sum) <= 0.05 * np.linalg.norm(dk_scale)
    dv_sum = np.array(dv_sum).reshape(w.batch, H * d)
    rel = np.linalg.norm(dv_sum - sum_dO) / np.linalg.norm(sum_dO)
    assert rel <= TOL_GRAD[0], rel
    # db_o is the column sum of dZ
    assert_close("dbo", a["dbo"], dZ.sum(axis=0))
