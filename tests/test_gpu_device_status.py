"""Device-side failure detection: the TMA-fed kernels give every wait for a
tile copy an iteration limit and, when it runs out, set a flag in device
memory instead of hanging the GPU.  fp4q_device_status makes that flag a
host-visible error.  No wait is made to run out here: the flag is set from
the host, as a timed-out wait would set it, and the status path is checked;
the GPU stays healthy throughout."""
import pytest
import torch

import block_scaled_fp4_quantize_gb300 as fq
from block_scaled_fp4_quantize_gb300 import _capi
from block_scaled_fp4_quantize_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()


def test_no_wait_ran_out_so_far():
    """Every GPU test collected before this one ran its tile kernels without
    a timed-out wait (the flags are per device and sticky until cleared)."""
    fq.device_status(clear=False)


def test_timeout_flag_reaches_the_host():
    lib = _capi.load()
    x = W.lognormal((512, 640), 71, sigma=2.0).cuda()
    q0 = fq.quantize(x, mode="outer_block", outer_block_size=64, rowwise=True, columnwise=True)
    fq.device_status()                                     # healthy: no error
    assert lib.fp4q_set_device_timeout_flag() == _capi.FP4Q_OK
    with pytest.raises(fq.FP4QError) as e:
        fq.device_status(clear=False)
    assert e.value.status == -10
    with pytest.raises(fq.FP4QError):                      # still set, cleared by this call
        fq.device_status(clear=True)
    fq.device_status()                                     # cleared
    # the context is still usable and the kernels give the same bits
    q1 = fq.quantize(x, mode="outer_block", outer_block_size=64, rowwise=True, columnwise=True)
    for k in ("row_codes", "row_scales", "row_outer", "col_codes", "col_scales", "col_outer"):
        assert torch.equal(getattr(q0, k), getattr(q1, k)), k
    fq.device_status()
    assert lib.fp4q_status_string(-10).startswith(b"FP4Q_ERR_TIMEOUT")
