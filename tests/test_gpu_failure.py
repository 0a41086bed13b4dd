"""Failure detection without a GPU fault: a device wait on a flag that nothing
sets gives up after its limit and reports NVFP4_ERR_TIMEOUT through the
per-device error word; the context stays usable and the word is cleared."""
import pytest
import torch

from gpu_util import built_lib

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    nv.nvfp4_device_status()                                  # start from a clean word
    nv.nvfp4_selftest_bounded_wait(flag, 2_000_000)           # 2 ms
    with pytest.raises(nv.Nvfp4Error) as ei:
        nv.nvfp4_device_status()
    assert ei.value.status == 5                               # NVFP4_ERR_TIMEOUT
    nv.nvfp4_device_status()                                  # cleared after the report
    # the context still works
    assert torch.ones(4, device="cuda").sum().item() == 4.0


def test_bounded_wait_returns_when_flag_is_set():
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    flag = torch.ones(1, dtype=torch.int32, device="cuda")
    nv.nvfp4_selftest_bounded_wait(flag, 2_000_000_000)
    nv.nvfp4_device_status()
