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


# (path, b, L, h, g): shapes whose chained states cross between CTAs many times.
# The per-block path chains the state from block to block through ready flags;
# the chain path hands it from CTA to CTA (b=1, h=2: one head-pair chain of 16
# blocks spread over 16 CTAs, so every CTA but the first waits for a hand-off).
TIMEOUT_CASES = [("tc", 1, 128 * 48, 16, 1), ("chain", 1, 2000, 2, 1)]


@pytest.mark.parametrize("path,b,L,h,g", TIMEOUT_CASES)
def test_state_wait_timeout_is_reported_and_recovered(path, b, L, h, g):
    import mamba_ssd_chunked_gb300 as pkg
    if path == "chain":
        assert pkg.ssd_select_path(b, L, h, 64, g, 128, "bf16", 256) == "chain"
    inp = make_inputs(b, L, h, 64, g, 128, io_dtype="bf16", init="normal", seed=3)
    t = to_device(inp, "bf16")
    saved = {k: os.environ.get(k) for k in ("SSD_DEVICE_WAIT_NS", "SSD_CHAIN_WARMUP")}
    os.environ["SSD_DEVICE_WAIT_NS"] = "1"   # a 1 ns limit on the wait for another CTA's state
    os.environ["SSD_CHAIN_WARMUP"] = "0"     # chain path: always take the hand-off, never recompute it
    try:
        pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"], chunk_len=256,
                    path=path)
        st = pkg.ssd_device_status()
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    assert st == 4  # SSD_ERR_DEVICE_TIMEOUT
    # the status word was cleared and the next call is correct
    y, fs = pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                        chunk_len=256, path=path)
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
