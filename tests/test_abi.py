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
    text = open(os.path.join(ROOT, "include", "tp_mlp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tp_mlp_\w+)\s*\(", text)))


def _cfg(**kw):
    base = dict(hidden=128, ffn=512, shards=2, max_tokens=256,
                dtype=B.TPMLP_BF16, use_layernorm=0, ln_eps=1e-5,
                gelu_mode=B.TPMLP_GELU_ERF)
    base.update(kw)
    return B.tp_mlp_config(**base)


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert len(declared) >= 13
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
