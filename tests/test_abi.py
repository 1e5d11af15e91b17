"""The C-ABI library loads, exports every symbol the header declares, and
rejects invalid arguments on the host before touching a device.  No GPU."""
import ctypes
import os
import re

import pytest

from tensor_transformer_mlp_tcgen05_gb300 import binding as B
from tensor_transformer_mlp_tcgen05_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.lib()


def _declared_functions():
    names = set()
    for hdr in ("tp_mlp.h", "tp_attn.h"):
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(tp_(?:mlp|attn)_\w+)\s*\(", text))
    return sorted(names)


def _cfg(**kw):
    base = dict(hidden=128, ffn=512, shards=2, max_tokens=256,
                dtype=B.TPMLP_BF16, use_layernorm=0, ln_eps=1e-5,
                gelu_mode=B.TPMLP_GELU_ERF)
    base.update(kw)
    return B.tp_mlp_config(**base)


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert len(declared) >= 27
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(B.EXPORTED) == declared


def test_status_strings(lib):
    for code in range(-7, 1):
        assert B.tp_mlp_status_string(code) != "unknown status"
    assert B.tp_mlp_status_string(5) == "unknown status"


@pytest.mark.parametrize("kw,code", [
    (dict(hidden=100), B.TPMLP_ERR_SHAPE),          # h % 64
    (dict(ffn=500), B.TPMLP_ERR_SHAPE),             # f % t
    (dict(ffn=384, shards=4), B.TPMLP_ERR_SHAPE),   # f_t = 96, not % 64
    (dict(shards=0), B.TPMLP_ERR_SHAPE),
    (dict(max_tokens=-1), B.TPMLP_ERR_SHAPE),
    (dict(dtype=7), B.TPMLP_ERR_ARG),
    (dict(gelu_mode=3), B.TPMLP_ERR_ARG),
    (dict(use_layernorm=1, ln_eps=float("nan")), B.TPMLP_ERR_ARG),
])
def test_create_rejects_bad_configs(lib, kw, code):
    h = ctypes.c_void_p()
    assert lib.tp_mlp_create(ctypes.byref(_cfg(**kw)), ctypes.byref(h)) == code
    assert h.value is None


def test_create_destroy_and_workspace_sizes(lib):
    h = B.tp_mlp_create(_cfg(use_layernorm=1))
    try:
        inf = B.tp_mlp_workspace_bytes(h, 256, 0)
        trn = B.tp_mlp_workspace_bytes(h, 256, 1)
        # inference: status + Xn + mean + rstd + Y; training adds H, dH,
        # dXn (fp32) and the column-sum partials.
        assert inf >= 256 + 256 * 128 * 2 + 2 * 256 * 4 + 256 * 512 * 2
        assert trn >= inf + 2 * 256 * 512 * 2 + 256 * 128 * 4
        assert B.tp_mlp_workspace_bytes(h, -1, 1) == 0
        assert B.tp_mlp_workspace_bytes(None, 8, 1) == 0
        assert B.tp_mlp_launch_count(h) == 0
    finally:
        B.tp_mlp_destroy(h)
    assert lib.tp_mlp_destroy(None) == B.TPMLP_OK


def test_forward_backward_validate_before_device_work(lib):
    """Every failure here is decided on the host (no CUDA call is made)."""
    h = B.tp_mlp_create(_cfg())
    ws_need = B.tp_mlp_workspace_bytes(h, 64, 1)
    fake = 1 << 20  # 16-byte aligned stand-in addresses, never dereferenced
    try:
        f = lib.tp_mlp_forward
        args = [h, 64, fake, fake, fake, None, None, None, None, fake, fake,
                ws_need, 1, None]
        a = list(args); a[1] = 257                      # tokens > max_tokens
        assert f(*a) == B.TPMLP_ERR_SHAPE
        a = list(args); a[1] = -1
        assert f(*a) == B.TPMLP_ERR_SHAPE
        a = list(args); a[2] = None                     # X missing
        assert f(*a) == B.TPMLP_ERR_ARG
        a = list(args); a[3] = fake + 8                 # A misaligned
        assert f(*a) == B.TPMLP_ERR_ALIGN
        a = list(args); a[11] = ws_need - 1             # workspace short
        assert f(*a) == B.TPMLP_ERR_WORKSPACE
        assert f(None, *args[1:]) == B.TPMLP_ERR_ARG
        g = lib.tp_mlp_backward
        bargs = [h, 64, fake, fake, fake, fake, None, fake, ws_need, fake,
                 fake, fake, None, None, None, None, None]
        b = list(bargs); b[10] = None                   # dA missing
        assert g(*b) == B.TPMLP_ERR_ARG
        b = list(bargs); b[12] = fake + 4               # db1 misaligned
        assert g(*b) == B.TPMLP_ERR_ALIGN
        b = list(bargs); b[8] = 0
        assert g(*b) == B.TPMLP_ERR_WORKSPACE
    finally:
        B.tp_mlp_destroy(h)


def test_layernorm_config_requires_parameters(lib):
    h = B.tp_mlp_create(_cfg(use_layernorm=1))
    fake = 1 << 20
    try:
        ws = B.tp_mlp_workspace_bytes(h, 8, 1)
        rc = lib.tp_mlp_forward(h, 8, fake, fake, fake, None, None, None,
                                None, fake, fake, ws, 1, None)
        assert rc == B.TPMLP_ERR_ARG
    finally:
        B.tp_mlp_destroy(h)


# ------------------------------------------------------------- attention --

def _acfg(**kw):
    base = dict(hidden=256, heads=4, shards=2, max_tokens=512, seq_len=256,
                causal=1, use_layernorm=0, ln_eps=1e-5, use_residual=0)
    base.update(kw)
    return B.tp_attn_config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(heads=3), B.TPMLP_ERR_SHAPE),              # h % H
    (dict(heads=8), B.TPMLP_ERR_SHAPE),              # d = 32
    (dict(hidden=320, heads=4), B.TPMLP_ERR_SHAPE),  # d = 80
    (dict(heads=4, shards=3), B.TPMLP_ERR_SHAPE),    # H % t
    (dict(seq_len=200), B.TPMLP_ERR_SHAPE),          # seq % 128
    (dict(shards=0), B.TPMLP_ERR_SHAPE),
    (dict(max_tokens=-1), B.TPMLP_ERR_SHAPE),
    (dict(causal=2), B.TPMLP_ERR_ARG),
    (dict(use_residual=5), B.TPMLP_ERR_ARG),
    (dict(use_layernorm=1, ln_eps=float("inf")), B.TPMLP_ERR_ARG),
])
def test_attn_create_rejects_bad_configs(lib, kw, code):
    h = ctypes.c_void_p()
    assert lib.tp_attn_create(ctypes.byref(_acfg(**kw)), ctypes.byref(h)) == code
    assert h.value is None


@pytest.mark.parametrize("kw", [
    dict(hidden=128, heads=2, shards=2),     # h_t = 64, d = 64
    dict(hidden=5120, heads=40, shards=8),   # d = 128, 5 heads per shard
    dict(hidden=3072, heads=32, shards=8),   # d = 96, the 8.3B layer
    dict(causal=0, use_layernorm=1, use_residual=1, max_tokens=0),
])
def test_attn_create_accepts_valid_corners(lib, kw):
    h = B.tp_attn_create(_acfg(**kw))
    B.tp_attn_destroy(h)


def test_attn_workspace_layout(lib):
    h = B.tp_attn_create(_acfg(use_layernorm=1))
    try:
        T, hd, H = 512, 256, 4
        inf = B.tp_attn_workspace_bytes(h, T, 0)
        trn = B.tp_attn_workspace_bytes(h, T, 1)
        # inference: status, Xn, mean, rstd, QKV, Ctx, lse; training adds
        # dCtx, delta, dQKV, dXn (fp32) and column-sum partials.
        assert inf >= 256 + T * hd * 2 + 2 * T * 4 + T * 3 * hd * 2 + \
            T * hd * 2 + H * T * 4
        assert trn >= inf + T * hd * 2 + H * T * 4 + T * 3 * hd * 2 + T * hd * 4
        offs = [B.tp_attn_workspace_offset(h, T, 1, k) for k in range(4)]
        assert all(o % 256 == 0 for o in offs)
        assert offs == sorted(offs) and offs[-1] < trn
        assert B.tp_attn_workspace_offset(h, T, 0, B.TPATTN_WS_DQKV) == -1
        assert B.tp_attn_workspace_offset(h, T, 1, 9) == -1
        assert B.tp_attn_workspace_bytes(None, T, 1) == 0
        assert B.tp_attn_launch_count(h) == 0
    finally:
        B.tp_attn_destroy(h)


def test_attn_host_validation_before_device(lib):
    """Argument errors are reported without touching a device (there is
    none here): bad token counts, NULL weights, misaligned pointers, a small
    workspace."""
    h = B.tp_attn_create(_acfg())
    L = lib
    try:
        ws = 1 << 20
        # tokens not a multiple of seq_len, or above max_tokens
        assert L.tp_attn_forward(h, 100, 16, 16, 16, None, None, None, None,
                                 16, 16, ws, 1, None) == B.TPMLP_ERR_SHAPE
        assert L.tp_attn_forward(h, 768, 16, 16, 16, None, None, None, None,
                                 16, 16, ws, 1, None) == B.TPMLP_ERR_SHAPE
        # NULL weights
        assert L.tp_attn_forward(h, 256, 16, None, 16, None, None, None, None,
                                 16, 16, ws, 1, None) == B.TPMLP_ERR_ARG
        # misaligned
        assert L.tp_attn_forward(h, 256, 18, 16, 16, None, None, None, None,
                                 16, 16, ws, 1, None) == B.TPMLP_ERR_ALIGN
        # workspace too small
        assert L.tp_attn_forward(h, 256, 16, 16, 16, None, None, None, None,
                                 16, 16, 64, 1, None) == B.TPMLP_ERR_WORKSPACE
        assert L.tp_attn_backward(h, 256, 16, 16, 16, 16, None, 16, 64, 16,
                                  16, 16, None, None, None, None,
                                  None) == B.TPMLP_ERR_WORKSPACE
        assert L.tp_attn_backward(h, 256, 16, 16, 16, 16, None, 16, ws, 16,
                                  None, 16, None, None, None, None,
                                  None) == B.TPMLP_ERR_ARG
    finally:
        B.tp_attn_destroy(h)


def test_mma_probe_rejects_bad_arguments(lib):
    ok = ctypes.c_void_p(16)
    assert lib.tp_mlp_probe_mma_cycles(128, 4, 100, ok, None, None) == B.TPMLP_ERR_ARG
    assert lib.tp_mlp_probe_mma_cycles(128, 4, 102, ok, ok, None) == B.TPMLP_ERR_ARG
    assert lib.tp_mlp_probe_mma_cycles(128, 0, 100, ok, ok, None) == B.TPMLP_ERR_ARG
    assert lib.tp_mlp_probe_mma_cycles(96, 4, 100, ok, ok, None) == B.TPMLP_ERR_SHAPE


def test_gelu_probe_rejects_bad_arguments(lib):
    ok = ctypes.c_void_p(16)
    assert lib.tp_mlp_probe_gelu(ok, ok, ok, 4, 7, None) == B.TPMLP_ERR_ARG
    assert lib.tp_mlp_probe_gelu(None, ok, ok, 4, B.TPMLP_GELU_ERF,
                                 None) == B.TPMLP_ERR_ARG
    assert lib.tp_mlp_probe_gelu(ok, ok, ok, -1, B.TPMLP_GELU_ERF,
                                 None) == B.TPMLP_ERR_ARG
    assert lib.tp_mlp_probe_gelu(None, None, None, 0, B.TPMLP_GELU_ERF,
                                 None) == B.TPMLP_OK


def test_ln_prologue_switch_validates_arguments(lib):
    assert lib.tp_mlp_set_ln_prologue(None, 1) == B.TPMLP_ERR_ARG
    assert lib.tp_attn_set_ln_prologue(None, 1) == B.TPMLP_ERR_ARG
    h = B.tp_mlp_create(B.tp_mlp_config(hidden=256, ffn=1024, shards=4,
                                        max_tokens=64, dtype=B.TPMLP_BF16,
                                        use_layernorm=1, ln_eps=1e-5))
    try:
        assert lib.tp_mlp_set_ln_prologue(h, 2) == B.TPMLP_ERR_ARG
        assert lib.tp_mlp_set_ln_prologue(h, 0) == B.TPMLP_OK
        assert lib.tp_mlp_set_ln_prologue(h, 1) == B.TPMLP_OK
    finally:
        B.tp_mlp_destroy(h)


def test_workspace_holds_the_layernorm_row_counters(lib):
    """With bf16 LayerNorm the status section also holds the fused
    prologue's counters (1 + ceil(T / 128) words): the workspace grows with
    the token count by that much beyond the token-sized buffers."""
    cfg = dict(hidden=256, ffn=1024, shards=4, max_tokens=1 << 20,
               dtype=B.TPMLP_BF16, ln_eps=1e-5)
    with_ln = B.tp_mlp_create(B.tp_mlp_config(use_layernorm=1, **cfg))
    no_ln = B.tp_mlp_create(B.tp_mlp_config(use_layernorm=0, **cfg))
    try:
        for T in (1, 128, 129, 70000):
            a = B.tp_mlp_workspace_bytes(with_ln, T, 0)
            b = B.tp_mlp_workspace_bytes(no_ln, T, 0)
            # Xn (bf16), mean and rstd (fp32), each section 256-aligned,
            # and the counters beyond the plain 256-byte status section
            up = lambda x: (x + 255) // 256 * 256
            words = 1 + (T + 127) // 128
            assert a - b == (up(T * 256 * 2) + 2 * up(T * 4)
                             + up(16 + 4 * words) - 256), T
    finally:
        B.tp_mlp_destroy(with_ln)
        B.tp_mlp_destroy(no_ln)


def test_nvtx_switch_validates_arguments(lib):
    assert lib.tp_mlp_set_nvtx(None, 1) == B.TPMLP_ERR_ARG
    assert lib.tp_attn_set_nvtx(None, 0) == B.TPMLP_ERR_ARG
    h = ctypes.c_void_p()
    assert lib.tp_mlp_create(ctypes.byref(B.tp_mlp_config(
        hidden=128, ffn=256, shards=2, max_tokens=64, dtype=B.TPMLP_BF16,
        use_layernorm=0, ln_eps=1e-5, gelu_mode=B.TPMLP_GELU_ERF,
        use_residual=0, dropout_p=0.0)), ctypes.byref(h)) == B.TPMLP_OK
    assert lib.tp_mlp_set_nvtx(h, 2) == B.TPMLP_ERR_ARG
    assert lib.tp_mlp_set_nvtx(h, 1) == B.TPMLP_OK
    assert lib.tp_mlp_set_nvtx(h, 0) == B.TPMLP_OK
    assert lib.tp_mlp_destroy(h) == B.TPMLP_OK
