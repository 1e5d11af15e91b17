"""Pins for the FP8 (E4M3) oracle: the format's closed-form values, every
bf16 bit pattern against PyTorch's float8_e4m3fn conversion, saturation,
round trips, scale invariance, exactness on representable inputs, and the
plain block forward and backward when quantization loses nothing.  No GPU."""
import numpy as np
import pytest
import torch

from oracle import fp8 as F
from oracle import mlp as O


def test_closed_form_values():
    """E4M3: bias 7, 3 mantissa bits, subnormals m 2^-9, S.1111.111 NaN."""
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9,
             0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125, 0x40: 2.0,
             0x7E: 448.0, 0x7D: 416.0, 0x77: 240.0, 0xC0: -2.0,
             0x80: -0.0, 0xFE: -448.0}
    for code, val in cases.items():
        assert F.e4m3_decode(np.array([code]))[0] == val, hex(code)
    assert np.isnan(F.e4m3_decode(np.array([0x7F, 0xFF]))).all()


def test_every_bf16_value_matches_torch_float8_e4m3fn():
    """All 65536 bf16 bit patterns with |x| <= 448 (finite), converted by the
    oracle and by torch's float8_e4m3fn cast (round to nearest even)."""
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).to(torch.float32)
    keep = torch.isfinite(x) & (x.abs() <= 448)
    x = x[keep]
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.e4m3_encode(x.double().numpy())
    # -0.0 and +0.0 codes: torch keeps the sign of zero, as the oracle does
    np.testing.assert_array_equal(got, want)
    assert len(x) > 30000


def test_fp32_grid_near_ties_matches_torch():
    """Random fp32 values and exact midpoints between neighbouring codes."""
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-12, 9, 200000))
         ).astype(np.float32)
    x = x[np.abs(x) <= 448]
    codes = np.arange(0, 0x7E, dtype=np.uint8)
    vals = F.e4m3_decode(codes)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)   # exact in fp32
    allx = np.concatenate([x, mids, -mids])
    want = torch.from_numpy(allx).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(F.e4m3_encode(allx.astype(np.float64)), want)


def test_saturation_and_round_trip():
    np.testing.assert_array_equal(
        F.e4m3_encode(np.array([448.0, 460.0, 464.0, 500.0, 1e30, -449.0, -1e9])),
        [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE])
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    np.testing.assert_array_equal(F.e4m3_encode(F.e4m3_decode(codes)), codes)


def test_scale_and_quantize_properties():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((64, 96)) * 3).astype(np.float32)
    q, s = F.quantize(x)
    # the largest magnitude lands on +-448 exactly
    assert np.max(np.abs(F.e4m3_decode(q))) == 448.0
    assert s == np.float32(np.max(np.abs(x))) / np.float32(448)
    # a power-of-two rescale changes only the scale
    q2, s2 = F.quantize(x * np.float32(8))
    np.testing.assert_array_equal(q2, q)
    assert s2 == s * 8
    # relative error of q s against x: at most half an E4M3 step for the
    # normal range (2^-4), plus the subnormal quantum s 2^-10 absolute
    err = np.abs(F.e4m3_decode(q) * s - x)
    assert np.all(err <= np.abs(x) * 2.0 ** -4 + s * 2.0 ** -10 + 1e-30)
    # all zeros: scale 1, codes 0
    qz, sz = F.quantize(np.zeros((3, 4), np.float32))
    assert sz == 1.0 and not qz.any()


def test_quantized_matmul_is_exact_for_representable_operands():
    """Operands that are E4M3 values with amax 448 quantize losslessly
    (scale 1): the quantized product equals the plain product."""
    rng = np.random.default_rng(2)
    codes_a = rng.integers(0, 0x7E, (16, 48)).astype(np.uint8)
    codes_b = rng.integers(0, 0x7E, (48, 24)).astype(np.uint8)
    codes_a[0, 0] = 0x7E
    codes_b[0, 0] = 0xFE
    a, b = F.e4m3_decode(codes_a), F.e4m3_decode(codes_b)
    qa, sa = F.quantize(a)
    qb, sb = F.quantize(b)
    assert sa == 1.0 and sb == 1.0
    np.testing.assert_array_equal(F.e4m3_decode(qa), a)
    np.testing.assert_array_equal(F.quantized_matmul(qa, sa, qb, sb), a @ b)


def test_forward_reduces_to_the_block_when_quantization_is_lossless():
    """X, A, B exactly representable with amax 448: H equals the plain
    block's X A + b1, and Z equals the plain GEMM2 applied to the bf16 Y the
    forward quantized (here Y's own quantization is the only loss)."""
    rng = np.random.default_rng(3)
    X = F.e4m3_decode(rng.integers(0, 0x7E, (8, 32)).astype(np.uint8)) / 64
    A = F.e4m3_decode(rng.integers(0, 0x7E, (32, 64)).astype(np.uint8)) / 256
    B = F.e4m3_decode(rng.integers(0, 0x7E, (64, 32)).astype(np.uint8)) / 256
    X[0, 0], A[0, 0], B[0, 0] = 448 / 64, 448 / 256, 448 / 256
    b1 = rng.standard_normal(64)
    f = F.forward(X, A, B, b1=b1)
    np.testing.assert_allclose(f["H"], X @ A + b1, rtol=1e-6, atol=1e-12)
    plain = O.forward(X, A, B, b1=b1)
    np.testing.assert_allclose(f["Y"], F.to_bf16(plain["Y"]), rtol=1e-2,
                               atol=1e-3)
    Yd = F.e4m3_decode(f["qy"]) * f["sy"]
    np.testing.assert_allclose(f["Z"], Yd @ B, rtol=1e-12, atol=1e-12)
    # Y's quantization error is within half an E4M3 step of Y
    assert np.all(np.abs(Yd - f["Y"]) <= np.abs(f["Y"]) * 2.0 ** -4
                  + f["sy"] * 2.0 ** -10)


@pytest.mark.parametrize("ln,res", [(False, False), (True, True)])
def test_forward_close_to_the_unquantized_block(ln, res):
    """E4M3's 3 mantissa bits: the block output stays within ~10% of the
    unquantized fp64 block on Gaussian data."""
    rng = np.random.default_rng(4)
    X = rng.standard_normal((64, 128))
    A = rng.standard_normal((128, 512)) * 0.05
    B = rng.standard_normal((512, 128)) * 0.05
    g = (1 + 0.1 * rng.standard_normal(128)) if ln else None
    bt = (0.1 * rng.standard_normal(128)) if ln else None
    f = F.forward(X, A, B, gamma=g, beta=bt, residual=res)
    ref = O.forward(X, A, B, gamma=g, beta=bt, residual=res)["Z"]
    rel = np.linalg.norm(f["Z"] - ref) / np.linalg.norm(ref)
    assert rel < 0.1, rel


def _e4m3_values(rng, shape, lo=0, hi=0x7E):
    return F.e4m3_decode(rng.integers(lo, hi, shape).astype(np.uint8))


def test_backward_equals_the_plain_backward_when_quantization_is_lossless():
    """A construction where every quantization step loses nothing: X and A
    hold E4M3 values (scales 1/64 and 1/256), B holds E4M3 values with
    max |B| = 448 (scale 1), b1 = 20 makes H >= 20 so that GeLU'(H) = 1
    exactly in fp64, and each row of dZ is one-hot with 448 (scale 1).  Then
    dY = dZ B^T = 448 B[:, c(r)]^T, s_dh = 448 and dH / s_dh are B's own
    E4M3 values, so dXn, dA, db1 and db2 must equal the unquantized backward
    of the same block (up to fp64 rounding) — a swapped operand, a wrong
    transpose or a scale taken from the wrong tensor breaks the equality."""
    rng = np.random.default_rng(11)
    T, h, f = 16, 32, 64
    X = _e4m3_values(rng, (T, h)) / 64
    X[0, 0] = 448 / 64
    A = _e4m3_values(rng, (h, f)) / 256
    A[0, 0] = 448 / 256
    B = F.e4m3_decode(rng.integers(0, 0xFF, (f, h)).astype(np.uint8))
    B = np.where(np.isnan(B), 0.0, B)
    B[0, 0] = 448.0
    b1 = np.full(f, 20.0)
    dZ = np.zeros((T, h))
    cols = rng.integers(0, h, T)
    cols[0] = 0
    dZ[np.arange(T), cols] = 448.0
    fwd = F.forward(X, A, B, b1=b1)
    bwd = F.backward(dZ, X, fwd)
    assert bwd["sdz"] == 1.0
    plain = O.backward(dZ, X, A, B, O.forward(X, A, B, b1=b1))
    np.testing.assert_array_equal(O.gelu_grad(F.to_bf16(fwd["H"])), 1.0)
    # dH is representable in bf16 too (448 x E4M3 values), so rounding is exact
    np.testing.assert_allclose(bwd["dH"], plain["dH"], rtol=0, atol=0)
    np.testing.assert_array_equal(F.e4m3_decode(bwd["qdh"]) * bwd["sdh"],
                                  bwd["dH"])
    for k in ("dXn", "dA", "db1", "db2"):
        np.testing.assert_allclose(bwd[k], plain[k], rtol=1e-13, atol=1e-9,
                                   err_msg=k)


def test_backward_weight_gradient_dB_exact_when_Y_is_lossless():
    """dB = Yq^T dZq: with A = 0 (scale 1, codes 0), H = b1, chosen from the
    E4M3 values 16..28 (so that GeLU(H) = H to bf16 and Y / s_y = 16 b1 are
    E4M3 numbers), and dZ one-hot with 448, Y and dZ quantize losslessly and
    dB equals Y^T dZ of the plain block."""
    rng = np.random.default_rng(12)
    T, h, f = 24, 32, 48
    X = _e4m3_values(rng, (T, h)) / 64
    A = np.zeros((h, f))
    B = _e4m3_values(rng, (f, h)) / 256
    b1 = rng.choice([16.0, 18.0, 20.0, 22.0, 24.0, 26.0], f)
    b1[0] = 28.0
    dZ = np.zeros((T, h))
    dZ[np.arange(T), rng.integers(0, h, T)] = rng.choice([-448.0, 448.0], T)
    fwd = F.forward(X, A, B, b1=b1)
    np.testing.assert_array_equal(fwd["Y"], np.broadcast_to(b1, (T, f)))
    bwd = F.backward(dZ, X, fwd)
    plain = O.backward(dZ, X, A, B, O.forward(X, A, B, b1=b1))
    np.testing.assert_allclose(bwd["dB"], plain["dB"], rtol=1e-13, atol=1e-9)
    np.testing.assert_allclose(bwd["db2"], plain["db2"], rtol=0, atol=0)
    # A = 0: dXn is exactly zero on both sides
    np.testing.assert_array_equal(bwd["dXn"], 0.0)


@pytest.mark.parametrize("ln,res", [(False, False), (True, True)])
def test_backward_close_to_the_unquantized_block(ln, res):
    """E4M3 gradients: within ~15 % (relative Frobenius) of the fp64 block's
    gradients on Gaussian data, and the LayerNorm / residual paths wired
    like the plain backward's."""
    rng = np.random.default_rng(13)
    X = rng.standard_normal((64, 128))
    A = rng.standard_normal((128, 512)) * 0.05
    B = rng.standard_normal((512, 128)) * 0.05
    dZ = rng.standard_normal((64, 128))
    g = (1 + 0.1 * rng.standard_normal(128)) if ln else None
    bt = (0.1 * rng.standard_normal(128)) if ln else None
    fwd = F.forward(X, A, B, gamma=g, beta=bt, residual=res)
    bwd = F.backward(dZ, X, fwd, gamma=g, residual=res)
    pf = O.forward(X, A, B, gamma=g, beta=bt, residual=res)
    pb = O.backward(dZ, X, A, B, pf, gamma=g, residual=res)
    for k in ("dX", "dA", "dB", "db1", "db2") + (("dgamma", "dbeta") if ln else ()):
        rel = np.linalg.norm(bwd[k] - pb[k]) / np.linalg.norm(pb[k])
        assert rel < 0.15, (k, rel)


@pytest.mark.parametrize("amax", [448.0, 1.0, 3.140625, 97.5, 6.5e5, 1.9e-30,
                                  2.0 ** 100 * 1.5])
def test_codes_vanish_22_binades_below_amax(amax):
    """The GPU quantizers enumerate the codes of the 22 binades at and below
    amax's and take every smaller magnitude as code +-0: with s = amax / 448
    any |x| < 2^(e_amax - 21) has |x / s| < 448 * 2^-21 < 2^-10, half the
    smallest E4M3 subnormal.  Every bf16 value of those smaller binades
    (both signs) must quantize to a zero code; and the binade 18 below
    amax's, whose top exceeds amax 2^-18 >= 2^-10 s, must still give
    nonzero codes (the table's 22 binades leave a margin of three)."""
    v = float(torch.tensor(amax).to(torch.bfloat16))
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    e_amax = (np.array([v], dtype=np.float32).view(np.uint32)[0] >> 23) & 0xFF
    ebits = (vals.view(np.uint32) >> 23) & 0xFF
    below = np.isfinite(vals) & (ebits < e_amax - 21)
    x = np.append(vals[below], v).astype(np.float64)
    codes, s = F.quantize(x)
    assert s == np.float32(v) / np.float32(448.0)
    assert not (codes[:-1] & 0x7F).any()
    assert codes[-1] & 0x7F == 0x7E                      # amax itself: 448
    # the binade 18 below amax's still reaches the smallest subnormal
    near = np.isfinite(vals) & (ebits == e_amax - 18) & (vals > 0)
    c2, _ = F.quantize(np.append(vals[near], v).astype(np.float64))
    assert (c2[:-1] & 0x7F).max() >= 1
