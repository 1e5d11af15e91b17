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
