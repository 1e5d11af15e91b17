"""A small object wrapper over the C ABI: owns a handle and a workspace
tensor, checks tensor shapes/dtypes/devices, and calls tp_mlp_forward /
tp_mlp_backward.  All arithmetic happens in libtpmlp's kernels; PyTorch only
provides device memory and the stream."""
from __future__ import annotations

import torch

from . import binding as B_


class TensorParallelMLP:
    """Megatron-style column/row-split MLP block with t logical shards
    (optionally the whole pre-LN sub-block X + MLP(LN(X)) with
    ``layernorm=True, residual=True``)."""

    def __init__(self, hidden: int, ffn: int, shards: int, max_tokens: int,
                 dtype: str = "bf16", layernorm: bool = False,
                 ln_eps: float = 1e-5, gelu: str = "erf", residual: bool = False,
                 dropout_p: float = 0.0, dropout_seed: int = 0,
                 dropout_offset: int = 0, device=None,
                 ln_prologue: bool = True):
        self.cfg = B_.tp_mlp_config(
            hidden=hidden, ffn=ffn, shards=shards, max_tokens=max_tokens,
            dtype=B_.TPMLP_BF16 if dtype == "bf16" else B_.TPMLP_FP32,
            use_layernorm=1 if layernorm else 0, ln_eps=ln_eps,
            gelu_mode=B_.TPMLP_GELU_ERF if gelu == "erf" else B_.TPMLP_GELU_TANH,
            use_residual=1 if residual else 0, dropout_p=dropout_p)
        if dtype not in ("bf16", "fp32") or gelu not in ("erf", "tanh"):
            raise ValueError("dtype must be bf16|fp32 and gelu erf|tanh")
        self.handle = B_.tp_mlp_create(self.cfg)
        if dropout_p > 0:
            B_.tp_mlp_set_dropout_seed(self.handle, dropout_seed, dropout_offset)
        if not ln_prologue:   # the LayerNorm as its own launch before GEMM1
            B_.tp_mlp_set_ln_prologue(self.handle, False)
        self.hidden, self.ffn, self.shards = hidden, ffn, shards
        self.max_tokens = max_tokens
        self.layernorm = layernorm
        self.dtype = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.device = torch.device(device or "cuda")
        self._ws = None
        self._ws_tokens = None

    def close(self):
        if self.handle:
            B_.tp_mlp_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---------------------------------------------------------------- ---
    def workspace(self, tokens: int, training: bool = True) -> torch.Tensor:
        need = B_.tp_mlp_workspace_bytes(self.handle, tokens, 1 if training else 0)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8,
                                   device=self.device)
        return self._ws

    def _chk(self, name, t, shape, dtype):
        if t is None:
            return
        if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
            raise ValueError(f"{name}: expected {tuple(shape)} {dtype}, got "
                             f"{tuple(t.shape)} {t.dtype}")
        if not t.is_contiguous() or t.device.type != "cuda":
            raise ValueError(f"{name} must be a contiguous CUDA tensor")

    def forward(self, X, A, B, b1=None, b2=None, gamma=None, beta=None,
                training: bool = True, out=None, stream=None):
        T = X.shape[0]
        h, f = self.hidden, self.ffn
        self._chk("X", X, (T, h), self.dtype)
        self._chk("A", A, (h, f), self.dtype)
        self._chk("B", B, (f, h), self.dtype)
        self._chk("b1", b1, (f,), torch.float32)
        self._chk("b2", b2, (h,), torch.float32)
        self._chk("gamma", gamma, (h,), torch.float32)
        self._chk("beta", beta, (h,), torch.float32)
        Z = out if out is not None else torch.empty((T, h), dtype=self.dtype,
                                                   device=X.device)
        self._chk("Z", Z, (T, h), self.dtype)
        ws = self.workspace(T, training)
        B_.tp_mlp_forward(self.handle, T, X, A, B, b1, b2, gamma, beta, Z, ws,
                          ws.numel(), 1 if training else 0, stream)
        return Z

    def backward(self, dZ, X, A, B, gamma=None, bias_grads: bool = True,
                 out=None, stream=None):
        """Gradients after a training forward on the same workspace.
        Returns a dict with dX, dA, dB and (optionally) db1, db2, dgamma,
        dbeta."""
        T = dZ.shape[0]
        h, f = self.hidden, self.ffn
        self._chk("dZ", dZ, (T, h), self.dtype)
        dev = dZ.device
        g = out if out is not None else {}
        g.setdefault("dX", torch.empty((T, h), dtype=self.dtype, device=dev))
        g.setdefault("dA", torch.empty((h, f), dtype=torch.float32, device=dev))
        g.setdefault("dB", torch.empty((f, h), dtype=torch.float32, device=dev))
        if bias_grads:
            g.setdefault("db1", torch.empty(f, dtype=torch.float32, device=dev))
            g.setdefault("db2", torch.empty(h, dtype=torch.float32, device=dev))
        if self.layernorm:
            g.setdefault("dgamma", torch.empty(h, dtype=torch.float32, device=dev))
            g.setdefault("dbeta", torch.empty(h, dtype=torch.float32, device=dev))
        ws = self.workspace(T, True)
        B_.tp_mlp_backward(self.handle, T, dZ, X, A, B, gamma, ws, ws.numel(),
                           g["dX"], g["dA"], g["dB"], g.get("db1"), g.get("db2"),
                           g.get("dgamma"), g.get("dbeta"), stream)
        return g

    def check(self, stream=None) -> int:
        """Synchronise and return the device status (TPMLP_OK or an error)."""
        if self._ws is None:
            return B_.TPMLP_OK
        return B_.tp_mlp_check(self.handle, self._ws, stream)

    # ------------------------------------------------------------- fp8 --
    def pack_fp8_weights(self, A, B, stream=None) -> torch.Tensor:
        """Quantize A and B to E4M3 (per-tensor scales) into a new packed
        buffer for forward_fp8 (see tp_mlp_fp8_pack_weights)."""
        h, f = self.hidden, self.ffn
        self._chk("A", A, (h, f), torch.bfloat16)
        self._chk("B", B, (f, h), torch.bfloat16)
        n = B_.tp_mlp_fp8_weights_bytes(self.handle)
        if n == 0:
            raise ValueError("the FP8 variant needs a bf16 handle without "
                             "dropout and ffn / shards a multiple of 128")
        packed = torch.empty(n, dtype=torch.uint8, device=A.device)
        B_.tp_mlp_fp8_pack_weights(self.handle, A, B, packed, n, stream)
        return packed

    def forward_fp8(self, X, packed, b1=None, b2=None, gamma=None, beta=None,
                    out=None, stream=None, train=False):
        """FP8 (E4M3) forward with weights from pack_fp8_weights; with
        train=True it keeps what backward_fp8 needs in the workspace
        (tp_mlp_forward_fp8_train)."""
        T = X.shape[0]
        h, f = self.hidden, self.ffn
        self._chk("X", X, (T, h), torch.bfloat16)
        self._chk("b1", b1, (f,), torch.float32)
        self._chk("b2", b2, (h,), torch.float32)
        self._chk("gamma", gamma, (h,), torch.float32)
        self._chk("beta", beta, (h,), torch.float32)
        Z = out if out is not None else torch.empty((T, h), dtype=torch.bfloat16,
                                                   device=X.device)
        self._chk("Z", Z, (T, h), torch.bfloat16)
        need = (B_.tp_mlp_fp8_train_workspace_bytes if train
                else B_.tp_mlp_fp8_workspace_bytes)(self.handle, T)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8,
                                   device=self.device)
        fwd = B_.tp_mlp_forward_fp8_train if train else B_.tp_mlp_forward_fp8
        fwd(self.handle, T, X, packed, b1, b2, gamma, beta, Z, self._ws,
            self._ws.numel(), stream)
        return Z

    def backward_fp8(self, dZ, X, packed, gamma=None, bias_grads=True,
                     grads=None, stream=None):
        """FP8 backward after forward_fp8(..., train=True) on the same X and
        packed weights (tp_mlp_backward_fp8): returns dX (bf16), dA, dB and
        the bias / LayerNorm-parameter gradients (fp32)."""
        T = X.shape[0]
        h, f = self.hidden, self.ffn
        self._chk("dZ", dZ, (T, h), torch.bfloat16)
        self._chk("X", X, (T, h), torch.bfloat16)
        self._chk("gamma", gamma, (h,), torch.float32)
        need = B_.tp_mlp_fp8_train_workspace_bytes(self.handle, T)
        if self._ws is None or self._ws.numel() < need:
            raise RuntimeError("backward_fp8 needs the workspace of "
                               "forward_fp8(..., train=True)")
        dev = X.device
        g = dict(grads or {})
        g.setdefault("dX", torch.empty((T, h), dtype=torch.bfloat16, device=dev))
        g.setdefault("dA", torch.empty((h, f), dtype=torch.float32, device=dev))
        g.setdefault("dB", torch.empty((f, h), dtype=torch.float32, device=dev))
        if bias_grads:
            g.setdefault("db1", torch.empty(f, dtype=torch.float32, device=dev))
            g.setdefault("db2", torch.empty(h, dtype=torch.float32, device=dev))
        if self.layernorm:
            g.setdefault("dgamma", torch.empty(h, dtype=torch.float32, device=dev))
            g.setdefault("dbeta", torch.empty(h, dtype=torch.float32, device=dev))
        B_.tp_mlp_backward_fp8(self.handle, T, dZ, X, packed, gamma, self._ws,
                               self._ws.numel(), g["dX"], g["dA"], g["dB"],
                               g.get("db1"), g.get("db2"), g.get("dgamma"),
                               g.get("dbeta"), stream)
        return g

    def fp8_saved(self, tokens: int, which: str, packed=None):
        """Views of the FP8 path's intermediates: "xq" [T,h] / "yq" [T,f]
        uint8 codes, "y" [T,f] bf16, "scales" (4 words: amax_x, amax_y as
        fp32 bits, s_x, s_y) in the workspace; "aqt" [f,h], "bqt" [h,f],
        "aq" [h,f], "bq" [f,h] codes and "wscales" (amax_a, amax_b, s_a,
        s_b) in `packed`; after a training step also "h" [T,f] and "dh"
        [T,f] bf16, "dzq" [T,h] / "dhq" [T,f] codes, the transposed codes
        "xqt" [h,T], "yqt" [f,T], "dzqt" [h,T], "dhqt" [f,T] (strided views:
        rows are T rounded up to 16 bytes apart) and "bscales" (amax_dz,
        amax_dh, s_dz, s_dh)."""
        h, f = self.hidden, self.ffn
        tp = (tokens + 15) // 16 * 16
        transposed = {"xqt": (B_.TPMLP_FP8_WS_XQT, h),
                      "yqt": (B_.TPMLP_FP8_WS_YQT, f),
                      "dzqt": (B_.TPMLP_FP8_WS_DZQT, h),
                      "dhqt": (B_.TPMLP_FP8_WS_DHQT, f)}
        if which in transposed:
            code, rows = transposed[which]
            off = B_.tp_mlp_fp8_offset(self.handle, tokens, code)
            return self._ws[off:off + rows * tp].view(rows, tp)[:, :tokens]
        spec = {"xq": (B_.TPMLP_FP8_WS_XQ, (tokens, h), torch.uint8, False),
                "h": (B_.TPMLP_FP8_WS_H, (tokens, f), torch.bfloat16, False),
                "dh": (B_.TPMLP_FP8_WS_DH, (tokens, f), torch.bfloat16, False),
                "dzq": (B_.TPMLP_FP8_WS_DZQ, (tokens, h), torch.uint8, False),
                "dhq": (B_.TPMLP_FP8_WS_DHQ, (tokens, f), torch.uint8, False),
                "bscales": (B_.TPMLP_FP8_WS_BSCALES, (4,), torch.int32, False),
                "aq": (B_.TPMLP_FP8_PACK_AQ, (h, f), torch.uint8, True),
                "bq": (B_.TPMLP_FP8_PACK_BQ, (f, h), torch.uint8, True),
                "y": (B_.TPMLP_FP8_WS_Y, (tokens, f), torch.bfloat16, False),
                "yq": (B_.TPMLP_FP8_WS_YQ, (tokens, f), torch.uint8, False),
                "scales": (B_.TPMLP_FP8_WS_SCALES, (4,), torch.int32, False),
                "aqt": (B_.TPMLP_FP8_PACK_AQT, (f, h), torch.uint8, True),
                "bqt": (B_.TPMLP_FP8_PACK_BQT, (h, f), torch.uint8, True),
                "wscales": (B_.TPMLP_FP8_PACK_SCALES, (4,), torch.int32, True)}
        code, shape, dt, in_pack = spec[which]
        buf = packed if in_pack else self._ws
        off = B_.tp_mlp_fp8_offset(self.handle, tokens, code)
        n = 1
        for d in shape:
            n *= d
        n *= torch.tensor([], dtype=dt).element_size()
        return buf[off:off + n].view(dt).view(*shape)
