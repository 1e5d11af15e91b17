"""The tensor-core rate probe (tp_mlp_probe_mma_cycles): one thread per SM
issuing back-to-back 128 x N x 16 bf16 MMAs sustains the per-SM dense rate a
clock-based peak assumes (8192 flops per SM cycle, 64 cycles per
128 x 128 x 16 MMA), within a few percent, for N = 128 and 256."""
import pytest

from tensor_transformer_mlp_tcgen05_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [128, 256])
def test_mma_rate_matches_the_dense_rate(n):
    rate, sms = B.mma_flops_per_cycle(n, n_mma=2048)
    assert sms >= 100
    assert 0.9 * 8192 <= rate <= 1.02 * 8192, rate


def test_mma_probe_narrow_tile_is_operand_bound():
    """N = 64 reads 6 KB of operands per 128 x 64 x 16 MMA; at 128 bytes of
    shared memory per cycle that takes 48 cycles, i.e. 2/3 of the dense rate."""
    rate, _ = B.mma_flops_per_cycle(64, n_mma=2048)
    assert 0.6 * 8192 <= rate <= 0.75 * 8192, rate


def _gelu_inputs():
    import torch
    g = torch.Generator().manual_seed(3)
    grid = torch.linspace(-12.0, 12.0, 240001, dtype=torch.float64)
    rnd = torch.randn(100000, generator=g, dtype=torch.float64) * 3
    return torch.cat([grid, rnd, torch.tensor([0.0, -0.0, 1e-30, -1e-30])])


@pytest.mark.parametrize("mode", ["erf", "tanh"])
def test_epilogue_gelu_against_the_oracle_and_cuda(mode):
    """The GEMM epilogues' GeLU and GeLU' (exact form: Phi from Abramowitz &
    Stegun 7.1.26, |error| <= 7.5e-8 on Phi, with SFU reciprocal and
    exponential) against the fp64 oracle and against CUDA's own fp32 erf
    (torch.nn.functional.gelu): within 4e-7 (1 + |x|) of the oracle — the
    7.5e-8 of the published bound, the SFU exponential's ~2^-22.5 relative
    error on phi and fp32 rounding of Phi = 1 - Q near 1 — far inside the
    bf16 rounding (2^-9 relative) every GeLU output then goes through."""
    import numpy as np
    import torch
    import torch.nn.functional as F
    from oracle import mlp as O
    x64 = _gelu_inputs()
    x = x64.float().cuda()
    m = B.TPMLP_GELU_ERF if mode == "erf" else B.TPMLP_GELU_TANH
    y, dy = B.device_gelu(x, m)
    torch.cuda.synchronize()
    xd = x.double().cpu().numpy()
    ref = O.gelu(xd, mode)
    dref = O.gelu_grad(xd, mode)
    bound = 4e-7 * (1.0 + np.abs(xd))
    err = np.abs(y.double().cpu().numpy() - ref)
    derr = np.abs(dy.double().cpu().numpy() - dref)
    assert np.all(err <= bound + 1e-6 * np.abs(ref) * (mode == "tanh")), err.max()
    assert np.all(derr <= bound + 1e-6 * np.abs(dref) * (mode == "tanh")), derr.max()
    if mode == "erf":
        cuda = F.gelu(x).double().cpu().numpy()
        assert np.all(np.abs(y.double().cpu().numpy() - cuda) <= 2 * bound)
    # the kernel's odd/even structure: GeLU(x) - GeLU(-x) = x exactly in
    # exact arithmetic; here within the same bound
    yn, _ = B.device_gelu(-x, m)
    torch.cuda.synchronize()
    lhs = (y.double() - yn.double()).cpu().numpy()
    assert np.all(np.abs(lhs - xd) <= 2 * bound + 1e-6 * np.abs(xd) * (mode == "tanh"))

