"""FP8 (E4M3) forward of the tensor-parallel MLP block: the oracle.

TEST INFRASTRUCTURE ONLY (never on the product path).

The pages name low-precision formats only in passing (Megatron Core
determinism article, news.hamidun.com, introduction and "Validation across
parallelism configurations": MXFP8 / NVFP4 / FP8 runs are kept bitwise
deterministic too).  The reading taken here is the plainest FP8 GEMM:

* E4M3 numbers (OCP 8-bit floating point, "FN" variant): 1 sign bit, 4
  exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
  subnormals m * 2^-9; S.1111.111 is NaN, so the largest finite value is
  1.75 * 2^8 = 448 and there is no infinity.
* Conversion from a real value: round to nearest, ties to even mantissa,
  saturating to +-448 beyond the largest finite value (no NaN for finite
  inputs).
* Per-tensor scaling from the tensor's own current maximum magnitude:
  s = amax / 448 computed in fp32 (s = 1 for an all-zero tensor), element
  codes q = e4m3(x / s) with x / s an fp32 division; the tensor is then
  represented by q * s.  The weight matrices A and B are each scaled as a
  whole (not per shard), so the codes do not depend on the shard count.
* Forward: Xn = LN(X) (bf16) or X; H = (s_x s_a) (Xq . Aq) + b1 with the
  product s_x s_a rounded to fp32; Y = GeLU(H) rounded to bf16; Y is
  scaled and quantized like X; Z = (s_y s_b) (Yq . Bq) + b2 [+ X].  The
  dot products of codes are exact here (fp64 sums of exactly representable
  products); the GPU sums them in fp32.
"""
from __future__ import annotations

import numpy as np
import torch

from .mlp import gelu, gelu_grad, layernorm_backward, layernorm_forward

E4M3_MAX = 448.0
_MIN_NORMAL = 2.0 ** -6
_SUB_QUANTUM = 2.0 ** -9


def e4m3_decode(codes):
    """Values of E4M3 codes (uint8 array) as float64; NaN for S.1111.111."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * _SUB_QUANTUM,
                   (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return sign * val


def e4m3_encode(x):
    """Round float64 values to E4M3 codes: nearest, ties to even mantissa,
    saturating to +-448.  NaN inputs are not expected (not handled)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    sign = np.where(np.signbit(x), 0x80, 0x00)
    code = np.zeros(x.shape, dtype=np.int64)
    sat = a >= E4M3_MAX
    sub = a < _MIN_NORMAL
    # subnormal range: multiples of 2^-9 (m = 8 reaches the smallest normal)
    msub = np.rint(np.minimum(a, _MIN_NORMAL) / _SUB_QUANTUM).astype(np.int64)
    # normal range: 8 <= a / 2^(e-3) < 16 with e = floor(log2 a)
    _, ex = np.frexp(np.where(sub | sat, 1.0, a))     # a = f 2^ex, f in [.5,1)
    e = ex - 1
    mq = np.rint(np.where(sub | sat, 8.0, a) / np.exp2(e - 3.0)).astype(np.int64)
    carry = mq == 16
    e = np.where(carry, e + 1, e)
    mq = np.where(carry, 8, mq)
    normal_code = ((e + 7) << 3) | (mq - 8)
    code = np.where(sub, msub, normal_code)
    # a value that rounds up past 448 also saturates
    code = np.where(sat | (code > 0x7E), 0x7E, code)
    return (code | sign).astype(np.uint8)


def scale_of(x):
    """Per-tensor scale s = amax / 448 in fp32 (1 for an all-zero tensor)."""
    amax = np.float32(np.max(np.abs(np.asarray(x, dtype=np.float32)))) \
        if np.size(x) else np.float32(0)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax) / np.float32(E4M3_MAX)


def quantize(x):
    """(codes, s): codes = e4m3(fp32(x) / s), the division in fp32."""
    x32 = np.asarray(x, dtype=np.float32)
    s = scale_of(x32)
    with np.errstate(over="ignore"):
        y = (x32 / s).astype(np.float32)
    return e4m3_encode(y.astype(np.float64)), s


def quantized_matmul(qa, sa, qb, sb):
    """(s_a s_b) (decode(qa) @ decode(qb)), the scale product in fp32."""
    sc = np.float32(sa) * np.float32(sb)
    return float(sc) * (e4m3_decode(qa) @ e4m3_decode(qb))


def to_bf16(x):
    """Round to bf16 (nearest even) through fp32, as a bf16 store of an
    fp32 value does."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32).copy())
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def forward(X, A, B, b1=None, b2=None, gamma=None, beta=None, eps=1e-5,
            mode="erf", residual=False):
    """The FP8 forward above.  X, A, B hold the bf16 inputs' values.
    Returns the codes and scales of every quantized operand, Y (bf16
    values) and Z (before its final bf16 rounding)."""
    X = np.asarray(X, dtype=np.float64)
    mean = rstd = None
    if gamma is not None:
        Xn, mean, rstd = layernorm_forward(X, gamma, beta, eps)
        Xn = to_bf16(Xn)
    else:
        Xn = X
    qx, sx = quantize(Xn)
    qa, sa = quantize(A)
    qb, sb = quantize(B)
    H = quantized_matmul(qx, sx, qa, sa)
    if b1 is not None:
        H = H + np.asarray(b1, dtype=np.float64)[None, :]
    Y = to_bf16(gelu(H, mode))
    qy, sy = quantize(Y)
    Z = quantized_matmul(qy, sy, qb, sb)
    if b2 is not None:
        Z = Z + np.asarray(b2, dtype=np.float64)[None, :]
    if residual:
        Z = Z + X
    return dict(Xn=Xn, mean=mean, rstd=rstd, qx=qx, sx=sx, qa=qa, sa=sa,
                qb=qb, sb=sb, H=H, Y=Y, qy=qy, sy=sy, Z=Z)


def backward(dZ, X, fwd, gamma=None, mode="erf", residual=False):
    """The FP8 (E4M3) backward of ``forward``, every GEMM on codes with
    per-tensor current scaling as in the forward (E4M3 for the gradients
    too; the pages name no gradient format):

    * dZ is quantized (codes qdz, scale sdz); db2 = sum_T dZ;
    * dY = (sdz sb) (dZq . Bq^T); dH = dY * GeLU'(H) with H as stored
      (bf16), rounded to bf16; db1 = sum_T dH (of the bf16 values);
    * dH is quantized (qdh, sdh);
    * dXn = (sdh sa) (dHq . Aq^T), then LayerNorm's backward (with the
      forward's statistics) or dXn itself, plus dZ with the residual;
    * dA = (sx sdh) (Xq^T . dHq), dB = (sy sdz) (Yq^T . dZq), fp32 results.

    Each scale product is rounded to fp32, as in the forward.  Returns the
    gradients and the codes and scales of dZ and dH."""
    dZ = np.asarray(dZ, dtype=np.float64)
    X = np.asarray(X, dtype=np.float64)
    qdz, sdz = quantize(dZ)
    db2 = dZ.sum(axis=0)
    Hb = to_bf16(fwd["H"])
    dY = quantized_matmul(qdz, sdz, fwd["qb"].T, fwd["sb"])
    dH = to_bf16(dY * gelu_grad(Hb, mode))
    db1 = dH.sum(axis=0)
    qdh, sdh = quantize(dH)
    dXn = quantized_matmul(qdh, sdh, fwd["qa"].T, fwd["sa"])
    dA = quantized_matmul(fwd["qx"].T, fwd["sx"], qdh, sdh)
    dB = quantized_matmul(fwd["qy"].T, fwd["sy"], qdz, sdz)
    dgamma = dbeta = None
    if gamma is not None:
        dX, dgamma, dbeta = layernorm_backward(dXn, X, fwd["mean"],
                                               fwd["rstd"], gamma)
    else:
        dX = dXn
    if residual:
        dX = dX + dZ
    return dict(dX=dX, dXn=dXn, dA=dA, dB=dB, db1=db1, db2=db2, dH=dH,
                qdz=qdz, sdz=sdz, qdh=qdh, sdh=sdh, dgamma=dgamma,
                dbeta=dbeta)
