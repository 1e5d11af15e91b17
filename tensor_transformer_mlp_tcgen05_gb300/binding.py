"""ctypes binding of libtpmlp, with the C ABI's names (argument marshalling
only: every step of the block runs in the library's CUDA kernels).

Tensor arguments may be torch tensors (their ``data_ptr()`` is passed), raw
integer device addresses, or None for the C ABI's nullable pointers.  Status
codes other than TPMLP_OK raise :class:`TPMLPError`, except from
``tp_mlp_check`` and the plain queries, which return the code.  There is no
fallback: if the shared library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

# TPMLP_LIB selects another build of the library (e.g. the debug variant
# libtpmlp_checks.so); by default the in-tree libtpmlp.so.
LIB_PATH = os.environ.get("TPMLP_LIB") or _build.LIB_PATH

TPMLP_OK = 0
TPMLP_ERR_ARG = -1
TPMLP_ERR_SHAPE = -2
TPMLP_ERR_ALIGN = -3
TPMLP_ERR_ARCH = -4
TPMLP_ERR_CUDA = -5
TPMLP_ERR_TIMEOUT = -6
TPMLP_ERR_WORKSPACE = -7
TPMLP_ERR_CHECK = -8

TPMLP_BF16 = 0
TPMLP_FP32 = 1
TPMLP_GELU_ERF = 0
TPMLP_GELU_TANH = 1

# Every function the header declares, for the export check.
EXPORTED = (
    "tp_mlp_create", "tp_mlp_destroy", "tp_mlp_workspace_bytes",
    "tp_mlp_forward", "tp_mlp_backward", "tp_mlp_check",
    "tp_mlp_status_string", "tp_mlp_last_detail", "tp_mlp_launch_count",
    "tp_mlp_set_timing", "tp_mlp_timing_get", "tp_mlp_timing_reset",
    "tp_mlp_set_wait_budget", "tp_mlp_set_nvtx", "tp_mlp_set_ln_prologue",
    "tp_mlp_bias_grad_noalloc",
    "tp_mlp_set_dropout_seed",
    "tp_mlp_fp8_weights_bytes", "tp_mlp_fp8_pack_weights",
    "tp_mlp_fp8_workspace_bytes", "tp_mlp_forward_fp8", "tp_mlp_fp8_offset",
    "tp_mlp_fp8_train_workspace_bytes", "tp_mlp_forward_fp8_train",
    "tp_mlp_backward_fp8",
    "tp_mlp_probe_mma_cycles",
    "tp_mlp_probe_gelu",
    "tp_attn_create", "tp_attn_destroy", "tp_attn_workspace_bytes",
    "tp_attn_forward", "tp_attn_backward", "tp_attn_check",
    "tp_attn_launch_count", "tp_attn_set_timing", "tp_attn_timing_get",
    "tp_attn_timing_reset", "tp_attn_set_wait_budget", "tp_attn_set_nvtx",
    "tp_attn_set_ln_prologue",
    "tp_attn_workspace_offset",
)

TPMLP_FP8_PACK_SCALES = 0
TPMLP_FP8_PACK_AQT = 1
TPMLP_FP8_PACK_BQT = 2
TPMLP_FP8_WS_SCALES = 3
TPMLP_FP8_WS_XQ = 4
TPMLP_FP8_WS_Y = 5
TPMLP_FP8_WS_YQ = 6
TPMLP_FP8_PACK_AQ = 7
TPMLP_FP8_PACK_BQ = 8
TPMLP_FP8_WS_H = 9
TPMLP_FP8_WS_XQT = 10
TPMLP_FP8_WS_YQT = 11
TPMLP_FP8_WS_BSCALES = 12
TPMLP_FP8_WS_DZQ = 13
TPMLP_FP8_WS_DZQT = 14
TPMLP_FP8_WS_DH = 15
TPMLP_FP8_WS_DHQ = 16
TPMLP_FP8_WS_DHQT = 17

TPATTN_WS_QKV = 0
TPATTN_WS_CTX = 1
TPATTN_WS_LSE = 2
TPATTN_WS_DQKV = 3

TPMLP_NOALLOC_SCRATCH_FLOATS = 1 << 20


class tp_mlp_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("ffn", ctypes.c_int),
                ("shards", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("dtype", ctypes.c_int), ("use_layernorm", ctypes.c_int),
                ("ln_eps", ctypes.c_float), ("gelu_mode", ctypes.c_int),
                ("use_residual", ctypes.c_int), ("dropout_p", ctypes.c_float)]


class tp_attn_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("heads", ctypes.c_int),
                ("shards", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("seq_len", ctypes.c_int), ("causal", ctypes.c_int),
                ("use_layernorm", ctypes.c_int), ("ln_eps", ctypes.c_float),
                ("use_residual", ctypes.c_int)]


class TPMLPError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(message)
        self.code = code


_lib = None
_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t


def lib(path: str | None = None) -> ctypes.CDLL:
    """Load libtpmlp.so (once) and declare its signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is missing: build it with "
            "tensor_transformer_mlp_tcgen05_gb300.build.build() (nvcc, sm_103a)")
    L = ctypes.CDLL(p)
    L.tp_mlp_create.argtypes = [ctypes.POINTER(tp_mlp_config),
                                ctypes.POINTER(_vp)]
    L.tp_mlp_create.restype = _i
    L.tp_mlp_destroy.argtypes = [_vp]
    L.tp_mlp_destroy.restype = _i
    L.tp_mlp_workspace_bytes.argtypes = [_vp, _i, _i]
    L.tp_mlp_workspace_bytes.restype = _sz
    L.tp_mlp_forward.argtypes = [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                 _vp, _vp, _sz, _i, _vp]
    L.tp_mlp_forward.restype = _i
    L.tp_mlp_backward.argtypes = [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                  _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    L.tp_mlp_backward.restype = _i
    L.tp_mlp_check.argtypes = [_vp, _vp, _vp]
    L.tp_mlp_check.restype = _i
    L.tp_mlp_status_string.argtypes = [_i]
    L.tp_mlp_status_string.restype = ctypes.c_char_p
    L.tp_mlp_last_detail.argtypes = []
    L.tp_mlp_last_detail.restype = ctypes.c_char_p
    L.tp_mlp_launch_count.argtypes = [_vp]
    L.tp_mlp_launch_count.restype = ctypes.c_longlong
    L.tp_mlp_set_timing.argtypes = [_vp, _i]
    L.tp_mlp_set_timing.restype = _i
    L.tp_mlp_timing_get.argtypes = [_vp, _i, ctypes.POINTER(ctypes.c_char_p),
                                    ctypes.POINTER(ctypes.c_longlong),
                                    ctypes.POINTER(ctypes.c_double)]
    L.tp_mlp_timing_get.restype = _i
    L.tp_mlp_timing_reset.argtypes = [_vp]
    L.tp_mlp_timing_reset.restype = _i
    L.tp_mlp_set_wait_budget.argtypes = [_vp, ctypes.c_ulonglong]
    L.tp_mlp_set_wait_budget.restype = _i
    L.tp_mlp_set_nvtx.argtypes = [_vp, _i]
    L.tp_mlp_set_nvtx.restype = _i
    L.tp_mlp_set_ln_prologue.argtypes = [_vp, _i]
    L.tp_mlp_set_ln_prologue.restype = _i
    L.tp_mlp_set_dropout_seed.argtypes = [_vp, ctypes.c_ulonglong,
                                          ctypes.c_ulonglong]
    L.tp_mlp_set_dropout_seed.restype = _i
    L.tp_mlp_bias_grad_noalloc.argtypes = [_i, _i, _i, _vp, _vp, _vp]
    L.tp_mlp_bias_grad_noalloc.restype = _i
    L.tp_mlp_fp8_weights_bytes.argtypes = [_vp]
    L.tp_mlp_fp8_weights_bytes.restype = _sz
    L.tp_mlp_fp8_pack_weights.argtypes = [_vp, _vp, _vp, _vp, _sz, _vp]
    L.tp_mlp_fp8_pack_weights.restype = _i
    L.tp_mlp_fp8_workspace_bytes.argtypes = [_vp, _i]
    L.tp_mlp_fp8_workspace_bytes.restype = _sz
    L.tp_mlp_forward_fp8.argtypes = [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp,
                                     _vp, _vp, _sz, _vp]
    L.tp_mlp_forward_fp8.restype = _i
    L.tp_mlp_fp8_train_workspace_bytes.argtypes = [_vp, _i]
    L.tp_mlp_fp8_train_workspace_bytes.restype = _sz
    L.tp_mlp_forward_fp8_train.argtypes = [_vp, _i, _vp, _vp, _vp, _vp, _vp,
                                           _vp, _vp, _vp, _sz, _vp]
    L.tp_mlp_forward_fp8_train.restype = _i
    L.tp_mlp_backward_fp8.argtypes = [_vp, _i, _vp, _vp, _vp, _vp, _vp, _sz,
                                      _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    L.tp_mlp_backward_fp8.restype = _i
    L.tp_mlp_fp8_offset.argtypes = [_vp, _i, _i]
    L.tp_mlp_fp8_offset.restype = ctypes.c_longlong
    L.tp_mlp_probe_mma_cycles.argtypes = [_i, _i, _i, _vp, _vp, _vp]
    L.tp_mlp_probe_mma_cycles.restype = _i
    L.tp_mlp_probe_gelu.argtypes = [_vp, _vp, _vp, _i, _i, _vp]
    L.tp_mlp_probe_gelu.restype = _i
    L.tp_attn_create.argtypes = [ctypes.POINTER(tp_attn_config),
                                 ctypes.POINTER(_vp)]
    L.tp_attn_create.restype = _i
    L.tp_attn_destroy.argtypes = [_vp]
    L.tp_attn_destroy.restype = _i
    L.tp_attn_workspace_bytes.argtypes = [_vp, _i, _i]
    L.tp_attn_workspace_bytes.restype = _sz
    L.tp_attn_workspace_offset.argtypes = [_vp, _i, _i, _i]
    L.tp_attn_workspace_offset.restype = ctypes.c_longlong
    L.tp_attn_forward.argtypes = [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                  _vp, _vp, _sz, _i, _vp]
    L.tp_attn_forward.restype = _i
    L.tp_attn_backward.argtypes = [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                   _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    L.tp_attn_backward.restype = _i
    L.tp_attn_check.argtypes = [_vp, _vp, _vp]
    L.tp_attn_check.restype = _i
    L.tp_attn_launch_count.argtypes = [_vp]
    L.tp_attn_launch_count.restype = ctypes.c_longlong
    L.tp_attn_set_timing.argtypes = [_vp, _i]
    L.tp_attn_set_timing.restype = _i
    L.tp_attn_timing_get.argtypes = [_vp, _i, ctypes.POINTER(ctypes.c_char_p),
                                     ctypes.POINTER(ctypes.c_longlong),
                                     ctypes.POINTER(ctypes.c_double)]
    L.tp_attn_timing_get.restype = _i
    L.tp_attn_timing_reset.argtypes = [_vp]
    L.tp_attn_timing_reset.restype = _i
    L.tp_attn_set_nvtx.argtypes = [_vp, _i]
    L.tp_attn_set_nvtx.restype = _i
    L.tp_attn_set_ln_prologue.argtypes = [_vp, _i]
    L.tp_attn_set_ln_prologue.restype = _i
    L.tp_attn_set_wait_budget.argtypes = [_vp, ctypes.c_ulonglong]
    L.tp_attn_set_wait_budget.restype = _i
    if path is None:
        _lib = L
    return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def tp_mlp_status_string(code: int) -> str:
    return lib().tp_mlp_status_string(code).decode()


def tp_mlp_last_detail() -> str:
    return lib().tp_mlp_last_detail().decode()


def _check(code: int, what: str):
    if code != TPMLP_OK:
        raise TPMLPError(code, f"{what}: {tp_mlp_status_string(code)} "
                               f"[{tp_mlp_last_detail()}]")


def tp_mlp_create(config: tp_mlp_config) -> int:
    h = _vp()
    _check(lib().tp_mlp_create(ctypes.byref(config), ctypes.byref(h)),
           "tp_mlp_create")
    return h.value


def tp_mlp_destroy(handle: int) -> None:
    _check(lib().tp_mlp_destroy(handle), "tp_mlp_destroy")


def tp_mlp_workspace_bytes(handle: int, tokens: int, training: int) -> int:
    return int(lib().tp_mlp_workspace_bytes(handle, tokens, training))


def tp_mlp_forward(handle, tokens, X, A, B, bias1, bias2, ln_gamma, ln_beta,
                   Z, workspace, workspace_bytes, training, stream=None):
    _check(lib().tp_mlp_forward(
        handle, tokens, _ptr(X), _ptr(A), _ptr(B), _ptr(bias1), _ptr(bias2),
        _ptr(ln_gamma), _ptr(ln_beta), _ptr(Z), _ptr(workspace),
        workspace_bytes, training, _stream(stream)), "tp_mlp_forward")


def tp_mlp_backward(handle, tokens, dZ, X, A, B, ln_gamma, workspace,
                    workspace_bytes, dX, dA, dB, dbias1, dbias2, dgamma, dbeta,
                    stream=None):
    _check(lib().tp_mlp_backward(
        handle, tokens, _ptr(dZ), _ptr(X), _ptr(A), _ptr(B), _ptr(ln_gamma),
        _ptr(workspace), workspace_bytes, _ptr(dX), _ptr(dA), _ptr(dB),
        _ptr(dbias1), _ptr(dbias2), _ptr(dgamma), _ptr(dbeta),
        _stream(stream)), "tp_mlp_backward")


def tp_mlp_check(handle, workspace, stream=None) -> int:
    return int(lib().tp_mlp_check(handle, _ptr(workspace), _stream(stream)))


def tp_mlp_launch_count(handle) -> int:
    return int(lib().tp_mlp_launch_count(handle))


def tp_mlp_set_timing(handle, enable: bool) -> None:
    _check(lib().tp_mlp_set_timing(handle, 1 if enable else 0),
           "tp_mlp_set_timing")


def tp_mlp_timing_get(handle):
    """All per-kernel totals: list of (name, launches, total_ms)."""
    out = []
    i = 0
    while True:
        name = ctypes.c_char_p()
        n = ctypes.c_longlong()
        ms = ctypes.c_double()
        rc = lib().tp_mlp_timing_get(handle, i, ctypes.byref(name),
                                     ctypes.byref(n), ctypes.byref(ms))
        if rc == TPMLP_ERR_ARG:
            break
        _check(rc, "tp_mlp_timing_get")
        out.append((name.value.decode(), n.value, ms.value))
        i += 1
    return out


def tp_mlp_timing_reset(handle) -> None:
    _check(lib().tp_mlp_timing_reset(handle), "tp_mlp_timing_reset")


def tp_mlp_set_dropout_seed(handle, seed: int, offset: int = 0) -> None:
    _check(lib().tp_mlp_set_dropout_seed(handle, seed, offset),
           "tp_mlp_set_dropout_seed")


def tp_mlp_set_wait_budget(handle, ns: int) -> None:
    _check(lib().tp_mlp_set_wait_budget(handle, ns), "tp_mlp_set_wait_budget")


def tp_mlp_set_nvtx(handle, enable: bool) -> None:
    _check(lib().tp_mlp_set_nvtx(handle, 1 if enable else 0), "tp_mlp_set_nvtx")


def tp_mlp_set_ln_prologue(handle, enable: bool) -> None:
    _check(lib().tp_mlp_set_ln_prologue(handle, 1 if enable else 0),
           "tp_mlp_set_ln_prologue")


def tp_mlp_bias_grad_noalloc(tokens, cols, dtype, grad, dbias, stream=None):
    """Column sums of a [tokens, cols] gradient into dbias, with the partial
    sums in the library's static device scratch instead of a workspace (for
    callers that cannot allocate device memory)."""
    _check(lib().tp_mlp_bias_grad_noalloc(tokens, cols, dtype, _ptr(grad),
                                          _ptr(dbias), _stream(stream)),
           "tp_mlp_bias_grad_noalloc")


# ------------------------------------------------------------------ fp8 --

def tp_mlp_fp8_weights_bytes(handle) -> int:
    return int(lib().tp_mlp_fp8_weights_bytes(handle))


def tp_mlp_fp8_pack_weights(handle, A, B, packed, packed_bytes, stream=None):
    _check(lib().tp_mlp_fp8_pack_weights(handle, _ptr(A), _ptr(B),
                                         _ptr(packed), packed_bytes,
                                         _stream(stream)),
           "tp_mlp_fp8_pack_weights")


def tp_mlp_fp8_workspace_bytes(handle, tokens: int) -> int:
    return int(lib().tp_mlp_fp8_workspace_bytes(handle, tokens))


def tp_mlp_forward_fp8(handle, tokens, X, packed, bias1, bias2, ln_gamma,
                       ln_beta, Z, workspace, workspace_bytes, stream=None):
    _check(lib().tp_mlp_forward_fp8(
        handle, tokens, _ptr(X), _ptr(packed), _ptr(bias1), _ptr(bias2),
        _ptr(ln_gamma), _ptr(ln_beta), _ptr(Z), _ptr(workspace),
        workspace_bytes, _stream(stream)), "tp_mlp_forward_fp8")


def tp_mlp_fp8_train_workspace_bytes(handle, tokens: int) -> int:
    return int(lib().tp_mlp_fp8_train_workspace_bytes(handle, tokens))


def tp_mlp_forward_fp8_train(handle, tokens, X, packed, bias1, bias2,
                             ln_gamma, ln_beta, Z, workspace, workspace_bytes,
                             stream=None):
    _check(lib().tp_mlp_forward_fp8_train(
        handle, tokens, _ptr(X), _ptr(packed), _ptr(bias1), _ptr(bias2),
        _ptr(ln_gamma), _ptr(ln_beta), _ptr(Z), _ptr(workspace),
        workspace_bytes, _stream(stream)), "tp_mlp_forward_fp8_train")


def tp_mlp_backward_fp8(handle, tokens, dZ, X, packed, ln_gamma, workspace,
                        workspace_bytes, dX, dA, dB, dbias1, dbias2, dgamma,
                        dbeta, stream=None):
    _check(lib().tp_mlp_backward_fp8(
        handle, tokens, _ptr(dZ), _ptr(X), _ptr(packed), _ptr(ln_gamma),
        _ptr(workspace), workspace_bytes, _ptr(dX), _ptr(dA), _ptr(dB),
        _ptr(dbias1), _ptr(dbias2), _ptr(dgamma), _ptr(dbeta),
        _stream(stream)), "tp_mlp_backward_fp8")


def tp_mlp_fp8_offset(handle, tokens: int, which: int) -> int:
    return int(lib().tp_mlp_fp8_offset(handle, tokens, which))


def tp_mlp_probe_mma_cycles(n, ctas, n_mma, cycles, status, stream=None):
    _check(lib().tp_mlp_probe_mma_cycles(n, ctas, n_mma, _ptr(cycles),
                                         _ptr(status), _stream(stream)),
           "tp_mlp_probe_mma_cycles")


def tp_mlp_probe_gelu(x, y, dy, n, mode, stream=None):
    _check(lib().tp_mlp_probe_gelu(_ptr(x), _ptr(y), _ptr(dy), int(n),
                                   int(mode), _stream(stream)),
           "tp_mlp_probe_gelu")


def device_gelu(x, mode=None):
    """(GeLU(x), GeLU'(x)) as the library's GEMM epilogues compute them, for
    a contiguous fp32 CUDA tensor x."""
    import torch
    mode = TPMLP_GELU_ERF if mode is None else mode
    x = x.contiguous()
    y = torch.empty_like(x)
    dy = torch.empty_like(x)
    tp_mlp_probe_gelu(x, y, dy, x.numel(), mode)
    return y, dy


def mma_flops_per_cycle(n=256, n_mma=4096, device=None):
    """Measured per-SM dense bf16 tensor rate (flops per SM cycle), one CTA
    per SM, averaged over the SMs."""
    import torch
    dev = torch.device(device or "cuda")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cycles = torch.zeros(sms, dtype=torch.int64, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    tp_mlp_probe_mma_cycles(n, sms, n_mma, cycles, status)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise TPMLPError(int(status.item()), "mma probe: completion wait gave up")
    mean = float(cycles.double().mean().item())
    return 2.0 * 128 * n * 16 * n_mma / mean, sms


# ------------------------------------------------------------- attention --

def tp_attn_create(config: tp_attn_config) -> int:
    h = _vp()
    _check(lib().tp_attn_create(ctypes.byref(config), ctypes.byref(h)),
           "tp_attn_create")
    return h.value


def tp_attn_destroy(handle: int) -> None:
    _check(lib().tp_attn_destroy(handle), "tp_attn_destroy")


def tp_attn_workspace_bytes(handle: int, tokens: int, training: int) -> int:
    return int(lib().tp_attn_workspace_bytes(handle, tokens, training))


def tp_attn_workspace_offset(handle: int, tokens: int, training: int,
                             which: int) -> int:
    return int(lib().tp_attn_workspace_offset(handle, tokens, training, which))


def tp_attn_forward(handle, tokens, X, Wqkv, Wo, bqkv, bo, ln_gamma, ln_beta,
                    Z, workspace, workspace_bytes, training, stream=None):
    _check(lib().tp_attn_forward(
        handle, tokens, _ptr(X), _ptr(Wqkv), _ptr(Wo), _ptr(bqkv), _ptr(bo),
        _ptr(ln_gamma), _ptr(ln_beta), _ptr(Z), _ptr(workspace),
        workspace_bytes, training, _stream(stream)), "tp_attn_forward")


def tp_attn_backward(handle, tokens, dZ, X, Wqkv, Wo, ln_gamma, workspace,
                     workspace_bytes, dX, dWqkv, dWo, dbqkv, dbo, dgamma,
                     dbeta, stream=None):
    _check(lib().tp_attn_backward(
        handle, tokens, _ptr(dZ), _ptr(X), _ptr(Wqkv), _ptr(Wo),
        _ptr(ln_gamma), _ptr(workspace), workspace_bytes, _ptr(dX),
        _ptr(dWqkv), _ptr(dWo), _ptr(dbqkv), _ptr(dbo), _ptr(dgamma),
        _ptr(dbeta), _stream(stream)), "tp_attn_backward")


def tp_attn_check(handle, workspace, stream=None) -> int:
    return int(lib().tp_attn_check(handle, _ptr(workspace), _stream(stream)))


def tp_attn_launch_count(handle) -> int:
    return int(lib().tp_attn_launch_count(handle))


def tp_attn_set_timing(handle, enable: bool) -> None:
    _check(lib().tp_attn_set_timing(handle, 1 if enable else 0),
           "tp_attn_set_timing")


def tp_attn_timing_get(handle):
    """All per-kernel totals: list of (name, launches, total_ms)."""
    out = []
    i = 0
    while True:
        name = ctypes.c_char_p()
        n = ctypes.c_longlong()
        ms = ctypes.c_double()
        rc = lib().tp_attn_timing_get(handle, i, ctypes.byref(name),
                                      ctypes.byref(n), ctypes.byref(ms))
        if rc == TPMLP_ERR_ARG:
            break
        _check(rc, "tp_attn_timing_get")
        out.append((name.value.decode(), n.value, ms.value))
        i += 1
    return out


def tp_attn_timing_reset(handle) -> None:
    _check(lib().tp_attn_timing_reset(handle), "tp_attn_timing_reset")


def tp_attn_set_nvtx(handle, enable: bool) -> None:
    _check(lib().tp_attn_set_nvtx(handle, 1 if enable else 0), "tp_attn_set_nvtx")


def tp_attn_set_ln_prologue(handle, enable: bool) -> None:
    _check(lib().tp_attn_set_ln_prologue(handle, 1 if enable else 0),
           "tp_attn_set_ln_prologue")


def tp_attn_set_wait_budget(handle, ns: int) -> None:
    _check(lib().tp_attn_set_wait_budget(handle, ns), "tp_attn_set_wait_budget")
