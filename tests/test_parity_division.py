"""The requantisation division of the fp8 GEMM1 epilogue (each element of a row group
divided by the group's scale max(amax, 1e-10) / 448, the G(128) quantisation of
"[vLLM] MoE Oracle & Prepare/Finalize") computes the quotient from the divisor's
correctly rounded reciprocal and one fma correction (Markstein's final division
step).  It must equal the IEEE division bit for bit: the self-test compares the two on
the device over pseudo-random pairs of that domain (dividends of both signs and zeros,
divisors over 80 binades with every mantissa)."""
import pytest
import torch

from mixture_experts_layer_tokens_gb300 import moe

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_row_division_matches_ieee_division(cuda_dev, seed):
    n = 1 << 26
    bad = moe.moe_selftest_row_division(n, seed)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    assert bad == 0, f"{bad} of {n} quotients differ from the IEEE division"


def test_row_division_rejects_bad_arguments(cuda_dev):
    with pytest.raises(moe.MoeError):
        moe.moe_selftest_row_division(-1, 0)
