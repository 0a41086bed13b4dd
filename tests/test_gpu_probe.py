"""The MMA issue-ceiling probe (nvfp4_mma_peak_probe) that bench.py reports next
to the GEMM rooflines: it runs on every SM pair, leaves the device error word
clear, and returns a rate and a clock in the plausible range of a GB300 (the
FP4 form's 128-cycle issue per 256x256x64 pair MMA at 1-2.1 GHz is 4.9-10.8
PFLOP/s; anything far outside means the probe measured something else)."""
import pytest

from gpu_util import built_lib

pytestmark = pytest.mark.gpu


def test_mma_peak_probe_rate_and_clock():
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    tf, mhz = nv.nvfp4_mma_peak_probe(4000)
    nv.nvfp4_device_status()
    assert 900.0 < mhz < 2300.0
    assert 3000.0 < tf < 13000.0
    # the rate follows the clock: 32768 FLOP per cycle per SM at most
    sms = __import__("torch").cuda.get_device_properties(0).multi_processor_count
    assert tf <= 32768 * sms * mhz * 1e6 / 1e12 * 1.02
