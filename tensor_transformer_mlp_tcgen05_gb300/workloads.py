"""Seeded synthetic inputs for the tensor-parallel MLP and attention blocks.

This module only draws random numbers and names shapes. It holds none of the
block's arithmetic, so both the CUDA path (through the Python binding) and the
fp64 oracle under ``oracle/`` can take their inputs from it without sharing
any computation.

Shapes follow the layers the Megatron-LM explainer and the BLOOM article
discuss (GPT-2 medium, the 8.3B GPT-2 with hidden 3072, a GPT-3-13B-like
layer, BLOOM-176B).  Recipe, for every workload:

* ``torch.Generator('cpu').manual_seed(seed)`` (seed 0 unless stated);
* draw order X, A, B, then b1 and b2 (only when ``with_bias``), then dZ;
* every tensor is drawn as fp32 standard normals in blocks of ``ROW_BLOCK``
  leading-dimension rows (so peak host memory stays bounded for the
  BLOOM-sized weights), scaled by its standard deviation, then cast to the
  storage dtype (bf16, or fp32 for the tiny workload);
* LayerNorm gamma = 1, beta = 0 (not drawn).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

ROW_BLOCK = 1024


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tokens: int          # T = batch * seq
    hidden: int          # h
    ffn: int             # f = 4h
    shards: int          # t, the number of column/row shards
    dtype: str           # "bf16" or "fp32"
    layernorm: bool      # pre-LayerNorm before the first GEMM
    backward: bool       # whether the workload runs the backward pass
    x_std: float = 1.0
    w_std: float = 0.02
    dz_std: float = 1.0
    batch: int = 0
    seq: int = 0

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def flops_fwd(self, tokens: Optional[int] = None) -> float:
        T = self.tokens if tokens is None else tokens
        return 4.0 * T * self.hidden * self.ffn

    def flops_fwd_bwd(self, tokens: Optional[int] = None) -> float:
        T = self.tokens if tokens is None else tokens
        return 12.0 * T * self.hidden * self.ffn

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 32, 64, 256, 2, "fp32", False, True,
                          batch=2, seq=16),
    "gpt2_medium": Workload("gpt2_medium", 8192, 1024, 4096, 4, "bf16", False,
                            False, batch=8, seq=1024),
    "megatron_8p3b": Workload("megatron_8p3b", 8192, 3072, 12288, 8, "bf16",
                              True, True, batch=8, seq=1024),
    "gpt3_13b": Workload("gpt3_13b", 8192, 5120, 20480, 8, "bf16", False, True,
                         batch=4, seq=2048),
    "bloom_176b": Workload("bloom_176b", 4096, 14336, 57344, 4, "bf16", False,
                           True, w_std=0.006, batch=2, seq=2048),
}

# Token sweep for the BLOOM-shaped layer, and its shard counts.
BLOOM_SWEEP_TOKENS = (512, 1024, 2048, 4096, 8192, 16384)
BLOOM_SWEEP_SHARDS = (1, 2, 4, 8)


def _normal(gen: torch.Generator, rows: int, cols: int, std: float,
            dtype: torch.dtype) -> torch.Tensor:
    out = torch.empty((rows, cols), dtype=dtype)
    for r0 in range(0, rows, ROW_BLOCK):
        r1 = min(rows, r0 + ROW_BLOCK)
        blk = torch.randn((r1 - r0, cols), generator=gen, dtype=torch.float32)
        if std != 1.0:
            blk.mul_(std)
        out[r0:r1] = blk.to(dtype)
    return out


def make_inputs(w: Workload, seed: int = 0, with_bias: bool = False,
                bias_std: float = 1.0, need_grad_input: Optional[bool] = None):
    """Return a dict of CPU tensors for workload ``w``.

    Keys: X [T,h], A [h,f], B [f,h] in the storage dtype; b1 [f], b2 [h]
    (fp32, or None); gamma, beta [h] fp32 (or None without LayerNorm);
    dZ [T,h] in the storage dtype (or None for forward-only workloads).
    """
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    dt = w.torch_dtype
    T, h, f = w.tokens, w.hidden, w.ffn
    X = _normal(g, T, h, w.x_std, dt)
    A = _normal(g, h, f, w.w_std, dt)
    B = _normal(g, f, h, w.w_std, dt)
    b1 = b2 = None
    if with_bias:
        b1 = _normal(g, 1, f, bias_std, torch.float32).reshape(f)
        b2 = _normal(g, 1, h, bias_std, torch.float32).reshape(h)
    want_dz = w.backward if need_grad_input is None else need_grad_input
    dZ = _normal(g, T, h, w.dz_std, dt) if want_dz else None
    gamma = beta = None
    if w.layernorm:
        gamma = torch.ones(h, dtype=torch.float32)
        beta = torch.zeros(h, dtype=torch.float32)
    return dict(X=X, A=A, B=B, b1=b1, b2=b2, gamma=gamma, beta=beta, dZ=dZ)


def sample_indices(n: int, k: int, seed: int) -> torch.Tensor:
    """k distinct sorted indices in [0, n), seeded; always includes n-1."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    if k >= n:
        return torch.arange(n)
    idx = torch.randperm(n, generator=g)[: k - 1]
    idx = torch.unique(torch.cat([idx, torch.tensor([n - 1])]))
    return idx


# ------------------------------------------------------------- attention --

@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    """Head-parallel self-attention block: T = batch * seq tokens,
    sequence-major; d = hidden / heads."""
    name: str
    batch: int
    seq: int
    hidden: int
    heads: int
    shards: int
    causal: bool = True
    layernorm: bool = False
    x_std: float = 1.0
    w_std: float = 0.02
    dz_std: float = 1.0

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    @property
    def head_dim(self) -> int:
        return self.hidden // self.heads

    def score_pairs(self) -> int:
        """(query, key) pairs the softmax sees, over all sequences and heads."""
        per = self.seq * (self.seq + 1) // 2 if self.causal else self.seq ** 2
        return self.batch * self.heads * per

    def flops_fwd(self) -> float:
        """Projections 2 T h (3h + h) plus Q K^T and P V over the unmasked
        pairs (2 d each)."""
        T, h = self.tokens, self.hidden
        return 8.0 * T * h * h + 4.0 * self.head_dim * self.score_pairs()

    def flops_fwd_bwd(self) -> float:
        """Forward plus backward: each projection twice more (input and
        weight gradients), and dV, dP, dQ, dK over the unmasked pairs."""
        T, h = self.tokens, self.hidden
        return 24.0 * T * h * h + 12.0 * self.head_dim * self.score_pairs()

    def with_(self, **kw) -> "AttnWorkload":
        return dataclasses.replace(self, **kw)


ATTN_WORKLOADS = {
    # small cases the oracle finishes in seconds (several 128-row blocks)
    "attn_tiny_d64": AttnWorkload("attn_tiny_d64", 2, 256, 256, 4, 2,
                                  w_std=0.0625),
    "attn_tiny_d128": AttnWorkload("attn_tiny_d128", 2, 384, 512, 4, 2,
                                   w_std=0.044),
    "attn_tiny_d96": AttnWorkload("attn_tiny_d96", 2, 256, 768, 8, 2,
                                  w_std=0.036),
    # GPT-2-medium-shaped and GPT-3-13B-shaped layers (as the MLP workloads)
    "attn_gpt2_medium": AttnWorkload("attn_gpt2_medium", 8, 1024, 1024, 16, 4),
    "attn_gpt3_13b": AttnWorkload("attn_gpt3_13b", 4, 2048, 5120, 40, 8),
    # the 8.3B GPT-2 of the scaling study: h = 3072, 32 heads of 96, pre-LN
    "attn_megatron_8p3b": AttnWorkload("attn_megatron_8p3b", 8, 1024, 3072,
                                       32, 8, layernorm=True),
}


def make_attn_inputs(w: AttnWorkload, seed: int = 0, with_bias: bool = False,
                     bias_std: float = 0.5):
    """CPU tensors for attention workload ``w``: draw order X [T,h],
    W_qkv [h,3h], W_o [h,h], then b_qkv [3h] and b_o [h] (fp32, only with
    ``with_bias``), then dZ [T,h]; bf16 storage, LayerNorm gamma = 1,
    beta = 0 when ``w.layernorm``."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    bf = torch.bfloat16
    T, h = w.tokens, w.hidden
    X = _normal(g, T, h, w.x_std, bf)
    Wqkv = _normal(g, h, 3 * h, w.w_std, bf)
    Wo = _normal(g, h, h, w.w_std, bf)
    bqkv = bo = None
    if with_bias:
        bqkv = _normal(g, 1, 3 * h, bias_std, torch.float32).reshape(3 * h)
        bo = _normal(g, 1, h, bias_std, torch.float32).reshape(h)
    dZ = _normal(g, T, h, w.dz_std, bf)
    gamma = beta = None
    if w.layernorm:
        gamma = torch.ones(h, dtype=torch.float32)
        beta = torch.zeros(h, dtype=torch.float32)
    return dict(X=X, Wqkv=Wqkv, Wo=Wo, bqkv=bqkv, bo=bo, gamma=gamma,
                beta=beta, dZ=dZ)


def make_attn_sign_inputs(w: AttnWorkload, seed: int = 0, c: float = 4.0):
    """Attention inputs whose projection is exact in bf16: X has random
    +-1 entries and every column of W_qkv holds a single +-c (random row
    and sign), so Q, K and V are exactly +-c and each score is an integer
    multiple of c^2 / sqrt(d) (score std c^2 in natural units: peaked
    softmax rows with a running maximum that keeps rising across key
    blocks).  W_o ~ N(0, w_std^2), dZ ~ N(0, 1), no biases, no LayerNorm.
    Draw order: X signs, W_qkv rows, W_qkv signs, W_o, dZ."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    bf = torch.bfloat16
    T, h = w.tokens, w.hidden
    X = (torch.randint(0, 2, (T, h), generator=g) * 2 - 1).to(bf)
    rows = torch.randint(0, h, (3 * h,), generator=g)
    signs = (torch.randint(0, 2, (3 * h,), generator=g) * 2 - 1).float()
    Wqkv = torch.zeros((h, 3 * h), dtype=torch.float32)
    Wqkv[rows, torch.arange(3 * h)] = c * signs
    Wo = _normal(g, h, h, w.w_std, bf)
    dZ = _normal(g, T, h, w.dz_std, bf)
    return dict(X=X, Wqkv=Wqkv.to(bf), Wo=Wo, bqkv=None, bo=None, gamma=None,
                beta=None, dZ=dZ)
