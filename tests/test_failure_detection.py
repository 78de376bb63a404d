"""Failure detection without a GPU fault.

Every device-side wait of the library's kernels is bounded: when it runs out it
records MOE_ERR_TIMEOUT in a device status word and lets the kernel return, so
the context stays usable and the host learns of it through moe_device_status.
Here a wait is made to run out on purpose -- a barrier that nothing arrives on,
with a 1 ms limit -- and the status is checked; nothing faults, traps or hangs."""
import pytest
import torch

from mixture_experts_layer_tokens_gb300 import moe

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_clears(cuda_dev):
    moe.moe_device_status(clear=True)             # start from a clean word
    assert moe.moe_device_status(clear=False) == moe.MOE_OK
    moe.moe_selftest_wait_timeout(1_000_000)      # 1 ms, then the wait gives up
    assert moe.moe_device_status(clear=False) == moe.MOE_ERR_TIMEOUT
    assert moe.moe_device_status(clear=True) == moe.MOE_ERR_TIMEOUT   # read and clear
    assert moe.moe_device_status(clear=False) == moe.MOE_OK
    # the context is still usable: an ordinary call runs and leaves the word clear
    logits = torch.randn((64, 8), device=cuda_dev)
    ids = torch.empty((64, 2), dtype=torch.int32, device=cuda_dev)
    w = torch.empty((64, 2), dtype=torch.float32, device=cuda_dev)
    moe.moe_route(logits, 2, moe.MOE_SCORING_SOFTMAX_RENORM, ids, w)
    torch.cuda.synchronize()
    assert moe.moe_device_status(clear=False) == moe.MOE_OK
    assert torch.equal(ids[:, 0].long(), logits.argmax(dim=1))


def test_timeout_limit_is_checked_on_the_host(cuda_dev):
    with pytest.raises(moe.MoeError) as e:
        moe.moe_selftest_wait_timeout(10)          # below the 1 us floor: nothing is launched
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
