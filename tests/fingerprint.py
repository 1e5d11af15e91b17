"""Tensor fingerprints and a chunk-wise diff for the bitwise two-run checks.

The Megatron Core determinism article (news.hamidun.com, "NVIDIA extends
bitwise determinism in Megatron Core to 2432 GPUs", tensor fingerprinting and
progressive divergence tracing) locates a determinism failure by hashing
tensors and walking the computation in order until the first hash that
differs.  This is the same idea at the scale of one block: every output (and,
where a test has them, the saved intermediates) is cut into 128 x 256 tiles
of raw bits, one fingerprint per tile, and the tensors are visited in the
order the kernels that write them are launched.  The first tensor with a
differing tile names the kernel to look at; the tile names the rows and
columns.

A fingerprint is a weighted sum of the tile's raw bit patterns (as unsigned
integers) with fixed pseudo-random weights in [1, 2^16): any single changed
element changes it, and since the weights are below 2^16 and the patterns
below 2^32, no product or sum of a 32 768-element tile leaves int64.  Equal
fingerprints are not taken as proof of equality: `first_difference` confirms
with an exact comparison and reports the first tile whose elements differ.
"""
from __future__ import annotations

import numpy as np
import torch

TILE_M, TILE_N = 128, 256

# Launch order of the tensors each block writes, and the kernel that writes
# each one (MLP forward then backward; attention forward then backward).
MLP_ORDER = ["Xn", "H", "Y", "Z", "dH", "db2", "db1", "dB", "dA", "dX",
             "dgamma", "dbeta"]
MLP_KERNEL = {
    "Xn": "layernorm_fwd (fused: gemm1_ln_gelu's prologue)",
    "H": "gemm1_gelu / gemm1_ln_gelu", "Y": "gemm1_gelu / gemm1_ln_gelu",
    "Z": "gemm2_shardsum (tail: gemm_tail_combine)",
    "dH": "gemm_dh_gelu_bwd", "db2": "colsum_db2 + colsum_finalize",
    "db1": "gemm_dh_gelu_bwd partials + colsum_finalize",
    "dB": "gemm_wgrad_dB (tail: gemm_tail_combine)",
    "dA": "gemm_wgrad_dA (tail: gemm_tail_combine)",
    "dX": "gemm_dx_shardsum (with LayerNorm: layernorm_bwd)",
    "dgamma": "layernorm_param_partial + colsum_finalize",
    "dbeta": "layernorm_param_partial + colsum_finalize",
}
ATTN_ORDER = ["QKV", "Ctx", "lse", "Z", "dbo", "dWo", "dQKV", "dbqkv", "dWqkv",
              "dX", "dgamma", "dbeta"]
ATTN_KERNEL = {
    "QKV": "gemm_qkv / gemm_ln_qkv", "Ctx": "attn_fwd", "lse": "attn_fwd",
    "Z": "gemm_out_shardsum", "dbo": "colsum_dbo", "dWo": "gemm_wgrad_dWo",
    "dQKV": "attn_bwd_dq (dQ) / attn_bwd_dkdv (dK, dV)",
    "dbqkv": "attn_bwd_* partials + colsum_finalize",
    "dWqkv": "gemm_wgrad_dWqkv",
    "dX": "gemm_dx_shardsum (with LayerNorm: layernorm_bwd)",
    "dgamma": "layernorm_param_partial", "dbeta": "layernorm_param_partial",
}

_UNSIGNED = {1: (torch.uint8, 0xFF), 2: (torch.int16, 0xFFFF),
             4: (torch.int32, 0xFFFFFFFF)}
# 8-byte elements (fp64, int64) are split into two 32-bit words
_WIDE = 8


def raw_bits(t: torch.Tensor) -> torch.Tensor:
    """The tensor's bit patterns as non-negative int64, shaped 2-D (a 1-D
    tensor becomes one row).  numpy arrays are accepted too."""
    if not torch.is_tensor(t):
        t = torch.from_numpy(np.ascontiguousarray(t))
    t = t.detach().contiguous()
    if t.dim() == 0:
        t = t.reshape(1)
    if t.dim() == 1:
        t = t.reshape(1, -1)
    elif t.dim() > 2:
        t = t.reshape(-1, t.shape[-1])
    size = t.element_size()
    if size == _WIDE:
        t = t.view(torch.int32)
        size = 4
    if size not in _UNSIGNED:
        raise TypeError(f"no raw view for {t.dtype}")
    view_dtype, mask = _UNSIGNED[size]
    return t.view(view_dtype).to(torch.int64) & mask


def _weights(device) -> torch.Tensor:
    # fixed odd weights in [1, 2^16) from a 64-bit LCG (Knuth's MMIX
    # constants), the same on every device and run
    n = TILE_M * TILE_N
    w = []
    x = 0x9E3779B97F4A7C15
    for _ in range(n):
        x = (x * 6364136223846793005 + 1442695040888963407) & (2**64 - 1)
        w.append(((x >> 40) & 0xFFFF) | 1)
    return torch.tensor(w, dtype=torch.int64, device=device).view(TILE_M, TILE_N)


_W_CACHE: dict = {}


def tile_fingerprints(t: torch.Tensor) -> torch.Tensor:
    """int64 [ceil(rows / 128), ceil(cols / 256)]: one fingerprint per tile."""
    bits = raw_bits(t)
    rows, cols = bits.shape
    tm = (rows + TILE_M - 1) // TILE_M
    tn = (cols + TILE_N - 1) // TILE_N
    pad = torch.zeros((tm * TILE_M, tn * TILE_N), dtype=torch.int64,
                      device=bits.device)
    pad[:rows, :cols] = bits
    key = str(bits.device)
    if key not in _W_CACHE:
        _W_CACHE[key] = _weights(bits.device)
    w = _W_CACHE[key]
    tiles = pad.view(tm, TILE_M, tn, TILE_N).permute(0, 2, 1, 3)
    return (tiles * w).sum(dim=(2, 3))


def first_difference(name: str, a: torch.Tensor, b: torch.Tensor,
                     kernel: str | None = None) -> str | None:
    """None when a and b are bitwise equal; otherwise a one-line report of
    the first differing 128 x 256 tile (row-major tile order), how many tiles
    differ and which kernel writes the tensor."""
    if not torch.is_tensor(a):
        a = torch.from_numpy(np.ascontiguousarray(a))
    if not torch.is_tensor(b):
        b = torch.from_numpy(np.ascontiguousarray(b))
    if a.shape != b.shape or a.dtype != b.dtype:
        return f"{name}: shape/dtype {tuple(a.shape)} {a.dtype} vs {tuple(b.shape)} {b.dtype}"
    b = b.to(a.device)
    ba, bb = raw_bits(a), raw_bits(b)
    if torch.equal(ba, bb):
        return None
    fa, fb = tile_fingerprints(a), tile_fingerprints(b)
    rows, cols = ba.shape
    # exact per-tile comparison (fingerprints only rank the search)
    neq = ba != bb
    tm, tn = fa.shape
    pad = torch.zeros((tm * TILE_M, tn * TILE_N), dtype=torch.bool,
                      device=ba.device)
    pad[:rows, :cols] = neq
    per_tile = pad.view(tm, TILE_M, tn, TILE_N).any(dim=3).any(dim=1)
    idx = per_tile.flatten().nonzero()
    first = int(idx[0])
    i, j = divmod(first, tn)
    r0, c0 = i * TILE_M, j * TILE_N
    r1, c1 = min(r0 + TILE_M, rows), min(c0 + TILE_N, cols)
    cell = pad[r0:r0 + TILE_M, c0:c0 + TILE_N].nonzero()
    er, ec = int(cell[0, 0]) + r0, int(cell[0, 1]) + c0
    fp_note = "" if fa[i, j] != fb[i, j] else " (fingerprints collided)"
    where = f" (written by {kernel})" if kernel else ""
    return (f"{name}{where}: first differing tile ({i}, {j}) = rows "
            f"{r0}..{r1 - 1}, cols {c0}..{c1 - 1}, first element ({er}, {ec}); "
            f"{int(per_tile.sum())} of {tm * tn} tiles differ{fp_note}")


def trace_divergence(r1: dict, r2: dict, order=None, kernels=None) -> str | None:
    """Visit the tensors of two runs in launch order (names missing from
    `order` last, sorted) and report the first that differs, or None."""
    order = order or []
    names = [k for k in order if k in r1] + sorted(k for k in r1 if k not in order)
    for k in names:
        rep = first_difference(k, r1[k], r2[k], (kernels or {}).get(k))
        if rep is not None:
            return rep
    return None


def assert_bitwise(r1: dict, r2: dict, order=MLP_ORDER, kernels=MLP_KERNEL):
    """Assert two runs' tensors are bitwise identical; on failure the message
    names the first divergent tensor in launch order, its kernel and tile."""
    assert set(r1) == set(r2), (sorted(r1), sorted(r2))
    rep = trace_divergence(r1, r2, order, kernels)
    assert rep is None, "runs differ: " + rep
