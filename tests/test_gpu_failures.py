"""Failure handling on the GPU without faulting it: a bounded device-side wait
that runs out is reported through the status word, and the next call works."""
import os

import pytest

torch = pytest.importorskip("torch")

from forms import rel_err
from gpu_util import oracle_full, to_device
from mamba_ssd_chunked_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_gb300 import build
    build.build()


def test_state_wait_timeout_is_reported_and_recovered():
    import mamba_ssd_chunked_gb300 as pkg
    # many 128-token blocks per chain, so successors run while predecessors still work
    inp = make_inputs(1, 128 * 48, 16, 64, 1, 128, io_dtype="bf16", init="normal", seed=3)
    t = to_device(inp, "bf16")
    old = os.environ.get("SSD_DEVICE_WAIT_NS")
    os.environ["SSD_DEVICE_WAIT_NS"] = "1"   # a 1 ns limit on the chained-state wait
    try:
        pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"], chunk_len=256,
                    path="tc")
        st = pkg.ssd_device_status()
    finally:
        if old is None:
            del os.environ["SSD_DEVICE_WAIT_NS"]
        else:
            os.environ["SSD_DEVICE_WAIT_NS"] = old
    assert st == 4  # SSD_ERR_DEVICE_TIMEOUT
    # the status word was cleared and the next call is correct
    y, fs = pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                        chunk_len=256, path="tc")
    assert pkg.ssd_device_status() == 0
    y_ref, f_ref = oracle_full(inp)
    assert rel_err(y.float().cpu().numpy(), y_ref) < 2e-2 and rel_err(fs.cpu().numpy(), f_ref) < 2e-2


def test_invalid_arguments_rejected_before_launch():
    import mamba_ssd_chunked_gb300 as pkg
    inp = make_inputs(1, 64, 2, 64, 1, 128, io_dtype="bf16", seed=1)
    t = to_device(inp, "bf16")
    with pytest.raises(ValueError):
        pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"][:, :32].contiguous(), t["C"], t["D"], None)
    c0 = pkg.ssd_kernel_launches()
    with pytest.raises(pkg.SsdError):
        pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], None, chunk_len=0)
    assert pkg.ssd_kernel_launches() == c0
