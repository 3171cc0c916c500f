"""The device-side failure path on a GPU without a fault: a kernel's bounded
wait on an mbarrier that nothing arrives at runs out, the kernel records a
timeout in the device error word and returns; the host reads it as
CONV_ERR_TIMEOUT, the word is cleared, and the context keeps working."""
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, run_bf16_layer

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    sh = torch.cuda.current_stream().cuda_stream
    B.conv_sync_status(sh)  # nothing pending
    B.conv_selftest_wait_timeout(2000, sh)  # 2 ms limit
    with pytest.raises(B.GbconvError) as e:
        B.conv_sync_status(sh)
    assert e.value.status_name == "CONV_ERR_TIMEOUT"
    B.conv_sync_status(sh)  # the word was cleared
    # the context is still usable: a forward pass afterwards matches the oracle
    y, ref = run_bf16_layer(torch, 3, 2, 64, 14, 14, 256, 3, 3, 1, 1, act=1, seed=77)
    assert ol.normalized_max_error(y, ref) <= 1e-2
