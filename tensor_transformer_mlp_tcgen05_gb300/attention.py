"""A small object wrapper over the attention block's C ABI (tp_attn_*):
owns a handle and a workspace tensor, checks shapes, dtypes and devices, and
calls tp_attn_forward / tp_attn_backward.  All arithmetic happens in
libtpmlp's kernels; PyTorch only provides device memory and the stream."""
from __future__ import annotations

import torch

from . import binding as B_


class TensorParallelAttention:
    """Head-parallel self-attention block with t logical shards: W_qkv split
    by columns head group by head group ([Q_i | K_i | V_i] per shard), W_o by
    rows, the shard partials summed in a fixed order.  Optionally the whole
    pre-LN sub-block X + Attn(LN(X))."""

    def __init__(self, hidden: int, heads: int, shards: int, max_tokens: int,
                 seq_len: int, causal: bool = True, layernorm: bool = False,
                 ln_eps: float = 1e-5, residual: bool = False, device=None,
                 ln_prologue: bool = True):
        self.cfg = B_.tp_attn_config(
            hidden=hidden, heads=heads, shards=shards, max_tokens=max_tokens,
            seq_len=seq_len, causal=1 if causal else 0,
            use_layernorm=1 if layernorm else 0, ln_eps=ln_eps,
            use_residual=1 if residual else 0)
        self.handle = B_.tp_attn_create(self.cfg)
        if not ln_prologue:   # the LayerNorm as its own launch before QKV
            B_.tp_attn_set_ln_prologue(self.handle, False)
        self.hidden, self.heads, self.shards = hidden, heads, shards
        self.seq_len = seq_len
        self.layernorm = layernorm
        self.device = torch.device(device or "cuda")
        self._ws = None

    def close(self):
        if self.handle:
            B_.tp_attn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace(self, tokens: int, training: bool = True) -> torch.Tensor:
        need = B_.tp_attn_workspace_bytes(self.handle, tokens,
                                          1 if training else 0)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8,
                                   device=self.device)
        return self._ws

    def saved(self, tokens: int, which: str, training: bool = True):
        """A view of an intermediate kept in the workspace: "qkv" [T, 3h]
        bf16, "ctx" [T, h] bf16, "lse2" [H, T] fp32 (base-2 log-sum-exp of
        the scores scaled by log2(e)/sqrt(d)) or "dqkv" [T, 3h] bf16."""
        code = {"qkv": B_.TPATTN_WS_QKV, "ctx": B_.TPATTN_WS_CTX,
                "lse2": B_.TPATTN_WS_LSE, "dqkv": B_.TPATTN_WS_DQKV}[which]
        off = B_.tp_attn_workspace_offset(self.handle, tokens,
                                          1 if training else 0, code)
        if off < 0 or self._ws is None:
            raise ValueError(f"{which} is not in this workspace")
        h, H = self.hidden, self.heads
        shape, dt = {"qkv": ((tokens, 3 * h), torch.bfloat16),
                     "ctx": ((tokens, h), torch.bfloat16),
                     "lse2": ((H, tokens), torch.float32),
                     "dqkv": ((tokens, 3 * h), torch.bfloat16)}[which]
        n = shape[0] * shape[1] * (2 if dt == torch.bfloat16 else 4)
        return self._ws[off:off + n].view(dt).view(*shape)

    @staticmethod
    def _chk(name, t, shape, dtype):
        if t is None:
            return
        if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
            raise ValueError(f"{name}: expected {tuple(shape)} {dtype}, got "
                             f"{tuple(t.shape)} {t.dtype}")
        if not t.is_contiguous() or t.device.type != "cuda":
            raise ValueError(f"{name} must be a contiguous CUDA tensor")

    def forward(self, X, Wqkv, Wo, bqkv=None, bo=None, gamma=None, beta=None,
                training: bool = True, out=None, stream=None):
        T = X.shape[0]
        h = self.hidden
        bf = torch.bfloat16
        self._chk("X", X, (T, h), bf)
        self._chk("Wqkv", Wqkv, (h, 3 * h), bf)
        self._chk("Wo", Wo, (h, h), bf)
        self._chk("bqkv", bqkv, (3 * h,), torch.float32)
        self._chk("bo", bo, (h,), torch.float32)
        self._chk("gamma", gamma, (h,), torch.float32)
        self._chk("beta", beta, (h,), torch.float32)
        Z = out if out is not None else torch.empty((T, h), dtype=bf,
                                                   device=X.device)
        self._chk("Z", Z, (T, h), bf)
        ws = self.workspace(T, training)
        B_.tp_attn_forward(self.handle, T, X, Wqkv, Wo, bqkv, bo, gamma, beta,
                           Z, ws, ws.numel(), 1 if training else 0, stream)
        return Z

    def backward(self, dZ, X, Wqkv, Wo, gamma=None, bias_grads: bool = True,
                 out=None, stream=None):
        """Gradients after a training forward on the same workspace: a dict
        with dX, dWqkv, dWo and (optionally) dbqkv, dbo, dgamma, dbeta."""
        T = dZ.shape[0]
        h = self.hidden
        self._chk("dZ", dZ, (T, h), torch.bfloat16)
        dev = dZ.device
        f32 = torch.float32
        g = out if out is not None else {}
        g.setdefault("dX", torch.empty((T, h), dtype=torch.bfloat16, device=dev))
        g.setdefault("dWqkv", torch.empty((h, 3 * h), dtype=f32, device=dev))
        g.setdefault("dWo", torch.empty((h, h), dtype=f32, device=dev))
        if bias_grads:
            g.setdefault("dbqkv", torch.empty(3 * h, dtype=f32, device=dev))
            g.setdefault("dbo", torch.empty(h, dtype=f32, device=dev))
        if self.layernorm:
            g.setdefault("dgamma", torch.empty(h, dtype=f32, device=dev))
            g.setdefault("dbeta", torch.empty(h, dtype=f32, device=dev))
        ws = self.workspace(T, True)
        B_.tp_attn_backward(self.handle, T, dZ, X, Wqkv, Wo, gamma, ws,
                            ws.numel(), g["dX"], g["dWqkv"], g["dWo"],
                            g.get("dbqkv"), g.get("dbo"), g.get("dgamma"),
                            g.get("dbeta"), stream)
        return g

    def check(self, stream=None) -> int:
        """Synchronise and return the device status (TPMLP_OK or an error)."""
        if self._ws is None:
            return B_.TPMLP_OK
        return B_.tp_attn_check(self.handle, self._ws, stream)
