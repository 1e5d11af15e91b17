"""Pins for the oracle's Philox4x32-10 generator and its dropout.

The generator is checked bit for bit against cuRAND's host-side Philox4_32_10
generator, an independent implementation of the same published algorithm:
its output block j (four 32-bit words) for seed s is Philox4x32-10 of the
counter (j div 65536, 0, j mod 65536, 0) under key (s low, s high), and a
generator offset past 2^32 blocks carries into the second counter word.  The
dropout built on it is checked by its keep rate, its independence from the
shard count, and finite differences with the mask fixed."""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest

from oracle import mlp as O
from oracle.philox import philox4x32_10

PHILOX4_32_10 = 161  # curandRngType_t value of CURAND_RNG_PSEUDO_PHILOX4_32_10


def _curand():
    for path in ("/usr/local/cuda/lib64/libcurand.so", ctypes.util.find_library("curand")):
        if path and os.path.exists(path):
            return ctypes.CDLL(path)
    return None


def _curand_words(lib, seed, offset_words, n):
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset_words)) == 0
        buf = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, buf.ctypes.data_as(ctypes.c_void_p),
                                  ctypes.c_size_t(n)) == 0
        return buf
    finally:
        lib.curandDestroyGenerator(gen)


@pytest.mark.parametrize("seed,first_block", [
    (0x0123456789ABCDEF, 0),
    (0xFEDCBA9876543210, 65536 * (1 << 32) + 3 * 65536 + 5),   # c1 = 1
    (7, 65536 * ((1 << 32) * 7 + 9) + 12345),                   # c1 = 7
])
def test_philox_matches_curand_host_generator(seed, first_block):
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not available")
    nblocks = 1 << 17 if first_block == 0 else 4096
    words = _curand_words(lib, seed, 4 * first_block, 4 * nblocks).reshape(-1, 4)
    j = np.uint64(first_block) + np.arange(nblocks, dtype=np.uint64)
    hi = j // np.uint64(65536)
    ref = np.stack(philox4x32_10(hi & np.uint64(0xFFFFFFFF), hi >> np.uint64(32),
                                 j % np.uint64(65536), 0,
                                 seed & 0xFFFFFFFF, seed >> 32), axis=1)
    np.testing.assert_array_equal(ref, words)


def test_philox_bits_look_uniform():
    w = np.concatenate(philox4x32_10(np.arange(1 << 16), 5, 0, 0, 1, 2))
    top = (w >> 28).astype(np.int64)
    counts = np.bincount(top, minlength=16)
    expected = len(w) / 16
    chi2 = ((counts - expected) ** 2 / expected).sum()
    assert chi2 < 60          # 15 degrees of freedom; p < 1e-6 beyond ~50
    bits = np.unpackbits(w.view(np.uint8))
    assert abs(bits.mean() - 0.5) < 0.002


def test_dropout_keep_rate_and_threshold():
    assert O.dropout_threshold(0.0) == 0
    assert O.dropout_threshold(0.5) == 1 << 31
    assert O.dropout_threshold(0.75) == 3 << 30
    assert O.dropout_threshold(1.0 - 1e-13) == 0xFFFFFFFF  # clamped to 32 bits
    m = O.dropout_mask(np.arange(512), 1024, 0.1, seed=1234, offset=7)
    n = m.size
    rate = m.mean()
    assert abs(rate - 0.9) < 5 * np.sqrt(0.09 / n)
    assert O.dropout_mask(np.arange(4), 64, 0.0, 1).all()


def test_dropout_mask_depends_on_seed_offset_row_column():
    a = O.dropout_mask(np.arange(64), 256, 0.5, seed=1, offset=0)
    assert (a != O.dropout_mask(np.arange(64), 256, 0.5, seed=2, offset=0)).mean() > 0.4
    assert (a != O.dropout_mask(np.arange(64), 256, 0.5, seed=1, offset=1)).mean() > 0.4
    rows = np.array([3, 17, 63])
    np.testing.assert_array_equal(O.dropout_mask(rows, 256, 0.5, 1, 0), a[rows])


def _problem(seed=0, T=4, h=8, f=16):
    rng = np.random.default_rng(seed)
    return dict(X=rng.standard_normal((T, h)), A=rng.standard_normal((h, f)) * 0.7,
                B=rng.standard_normal((f, h)) * 0.7, b1=rng.standard_normal(f),
                b2=rng.standard_normal(h), dZ=rng.standard_normal((T, h)),
                gamma=1 + 0.3 * rng.standard_normal(h), beta=0.3 * rng.standard_normal(h))


@pytest.mark.parametrize("t", [1, 2, 4])
def test_dropout_outside_the_parallel_region(t):
    """Sharded and unsharded blocks draw the same mask (it is keyed by token
    and column only), so the shard identity still holds with dropout."""
    p = _problem(seed=1)
    drop = (0.25, 99, 3)
    full = O.forward(p["X"], p["A"], p["B"], p["b1"], p["b2"], p["gamma"], p["beta"],
                     residual=True, dropout=drop)
    sh = O.forward_sharded(p["X"], p["A"], p["B"], t, p["b1"], p["b2"], p["gamma"],
                           p["beta"], residual=True, dropout=drop)
    np.testing.assert_allclose(sh["Z"], full["Z"], rtol=1e-12, atol=1e-13)
    gf = O.backward(p["dZ"], p["X"], p["A"], p["B"], full, p["gamma"], residual=True)
    gs = O.backward_sharded(p["dZ"], p["X"], p["A"], p["B"], t, sh, p["gamma"],
                            residual=True)
    for k in ("dX", "dA", "dB", "db1", "db2", "dgamma", "dbeta"):
        np.testing.assert_allclose(gs[k], gf[k], rtol=1e-12, atol=1e-13, err_msg=k)


def test_dropout_gradients_match_central_differences():
    """With the mask held fixed the block is differentiable: every gradient
    entry against central differences."""
    p = _problem(seed=2, T=3, h=4, f=8)
    drop = (0.3, 5, 0)

    def loss():
        z = O.forward(p["X"], p["A"], p["B"], p["b1"], p["b2"], p["gamma"],
                      p["beta"], residual=True, dropout=drop)["Z"]
        return float((z * p["dZ"]).sum())

    fwd = O.forward(p["X"], p["A"], p["B"], p["b1"], p["b2"], p["gamma"], p["beta"],
                    residual=True, dropout=drop)
    assert 0 < fwd["mask"].mean() < 1
    g = O.backward(p["dZ"], p["X"], p["A"], p["B"], fwd, p["gamma"], residual=True)
    for name, gname in (("X", "dX"), ("A", "dA"), ("B", "dB"), ("b1", "db1"),
                        ("b2", "db2"), ("gamma", "dgamma"), ("beta", "dbeta")):
        base = p[name]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            step = 1e-5 * max(1.0, abs(base[idx]))
            keep = base[idx]
            base[idx] = keep + step
            lp = loss()
            base[idx] = keep - step
            lm = loss()
            base[idx] = keep
            fd[idx] = (lp - lm) / (2 * step)
        np.testing.assert_allclose(g[gname], fd, rtol=0,
                                   atol=2e-8 * max(1.0, np.abs(fd).max()), err_msg=name)
