"""The determinism diagnostic (tests/fingerprint.py) on the CPU: a planted
one-bit difference is found in the right tile, element and tensor."""
import torch

from fingerprint import (MLP_KERNEL, MLP_ORDER, TILE_M, TILE_N, assert_bitwise,
                         first_difference, tile_fingerprints, trace_divergence)


def _flip_bit(t, r, c, bit):
    t = t.clone()
    view = t.view(torch.int16 if t.element_size() == 2 else torch.int32)
    view[r, c] ^= (1 << bit)
    return t


def test_identical_tensors_report_nothing():
    g = torch.Generator().manual_seed(0)
    a = torch.randn(300, 700, generator=g).to(torch.bfloat16)
    assert first_difference("Z", a, a.clone()) is None
    assert torch.equal(tile_fingerprints(a), tile_fingerprints(a.clone()))


def test_planted_bit_found_at_its_tile():
    g = torch.Generator().manual_seed(1)
    a = torch.randn(1000, 1300, generator=g).to(torch.bfloat16)
    for (r, c, bit) in [(0, 0, 0), (517, 1033, 3), (999, 1299, 15),
                        (128, 256, 7), (127, 255, 1)]:
        b = _flip_bit(a, r, c, bit)
        rep = first_difference("dX", a, b, "gemm_dx_shardsum")
        i, j = r // TILE_M, c // TILE_N
        assert f"first differing tile ({i}, {j})" in rep, rep
        assert f"first element ({r}, {c})" in rep, rep
        assert "1 of 48 tiles differ" in rep, rep
        assert "gemm_dx_shardsum" in rep
        assert "collided" not in rep
        fa, fb = tile_fingerprints(a), tile_fingerprints(b)
        diff = (fa != fb).nonzero().tolist()
        assert diff == [[i, j]], diff


def test_fp32_sign_bit_and_one_dimensional():
    g = torch.Generator().manual_seed(2)
    a = torch.randn(5120, generator=g)
    b = a.clone()
    b.view(torch.int32)[4097] ^= (1 << 31)
    rep = first_difference("db2", a, b)
    assert "first differing tile (0, 16)" in rep and "(0, 4097)" in rep, rep


def test_negative_zero_is_a_difference():
    a = torch.zeros(4, 4)
    b = a.clone()
    b[2, 3] = -0.0
    assert torch.equal(a, b)  # value-equal ...
    rep = first_difference("dA", a, b)  # ... but not bitwise equal
    assert rep is not None and "(2, 3)" in rep


def test_trace_names_the_first_kernel_in_launch_order():
    g = torch.Generator().manual_seed(3)
    r1 = {k: torch.randn(256, 512, generator=g) for k in
          ("Z", "dA", "dB", "dX", "db2")}
    r2 = {k: v.clone() for k, v in r1.items()}
    r2["dX"] = _flip_bit(r2["dX"], 5, 6, 2)   # launched last of these
    r2["dB"] = _flip_bit(r2["dB"], 300 % 256, 400, 9)  # launched before dA, dX
    rep = trace_divergence(r1, r2, MLP_ORDER, MLP_KERNEL)
    assert rep.startswith("dB (written by gemm_wgrad_dB"), rep
    try:
        assert_bitwise(r1, r2)
    except AssertionError as e:
        assert "dB" in str(e)
    else:
        raise AssertionError("assert_bitwise missed a difference")
    r2 = {k: v.clone() for k, v in r1.items()}
    assert_bitwise(r1, r2)


def test_every_single_bit_flip_changes_the_fingerprint():
    g = torch.Generator().manual_seed(4)
    a = torch.randn(TILE_M, TILE_N, generator=g)
    base = tile_fingerprints(a)
    idx = torch.randint(0, TILE_M * TILE_N, (64,), generator=g)
    for n, k in enumerate(idx.tolist()):
        r, c = divmod(k, TILE_N)
        b = _flip_bit(a, r, c, n % 32)
        assert tile_fingerprints(b)[0, 0] != base[0, 0]
