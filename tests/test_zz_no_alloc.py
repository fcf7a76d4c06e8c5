"""ssd_fwd_noalloc: the forward for callers that must not allocate device
memory (a memory manager owns the device, or cudaMalloc's possible device
synchronisation is not allowed on their path). It runs the fused kernel on a
fixed scratch array inside the library. Checked through the C ABI against
ssd_fwd and against the fp64 oracle on two calls in a row (the second one
finds the array as the first left it). This file sorts last so that a failure
here comes after every other test has run."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from forms import rel_err
from gpu_util import TOL, oracle_full
from mamba_ssd_chunked_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_gb300 import build
    build.build()
    import mamba_ssd_chunked_gb300 as pkg
    lib = pkg.library()
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.ssd_fwd_noalloc.restype = i
    lib.ssd_fwd_noalloc.argtypes = [ctypes.POINTER(pkg.Dims), i, vp, vp, vp, vp, vp, vp, vp, vp, i, i, vp, vp, vp]
    return lib


def _device_inputs(inp):
    t = {}
    for k, v in inp.items():
        if v is None:
            t[k] = None
            continue
        x = torch.from_numpy(np.ascontiguousarray(v)).cuda()
        if k in ("x", "B", "C"):
            x = x.to(torch.bfloat16)
        t[k] = x.contiguous()
    return t


def _call(fn, dims, t, y, fs, chunk_len, stream):
    p = lambda v: None if v is None else v.data_ptr()
    return fn(ctypes.byref(dims), 1, p(t["x"]), p(t["dt"]), p(t["dt_bias"]), p(t["A"]), p(t["B"]), p(t["C"]),
              p(t["D"]), p(t["init_state"]), chunk_len, dims.ngroups, p(y), p(fs), stream)


def test_noalloc_matches_ssd_fwd_on_two_calls(lib):
    import mamba_ssd_chunked_gb300 as pkg
    b, L, h, p, g, n = 2, 700, 8, 64, 2, 128
    dims = pkg.Dims(b, L, h, p, g, n)
    stream = torch.cuda.current_stream().cuda_stream
    for seed in (101, 102):  # two calls in a row, different inputs
        inp = make_inputs(b, L, h, p, g, n, io_dtype="bf16", init="normal", seed=seed)
        t = _device_inputs(inp)
        y_ref = torch.empty_like(t["x"])
        f_ref = torch.empty((b, h, p, n), dtype=torch.float32, device="cuda")
        assert _call(lib.ssd_fwd, dims, t, y_ref, f_ref, 256, stream) == 0
        y = torch.full_like(t["x"], float("nan"))
        fs = torch.full((b, h, p, n), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(lib.ssd_fwd_noalloc, dims, t, y, fs, 256, stream) == 0
        assert lib.ssd_device_status(stream) == 0
        assert rel_err(y.float().cpu().numpy(), y_ref.float().cpu().numpy()) < TOL["bf16"]
        assert rel_err(fs.cpu().numpy(), f_ref.cpu().numpy()) < TOL["bf16"]
        # and against the fp64 oracle, so that a bias both GPU paths share would show
        y_o, f_o = oracle_full(inp)
        assert rel_err(y.float().cpu().numpy(), y_o) < TOL["bf16"]
        assert rel_err(fs.cpu().numpy(), f_o) < TOL["bf16"]


def test_noalloc_rejects_work_beyond_its_scratch(lib):
    import mamba_ssd_chunked_gb300 as pkg
    # 4 x 80 chains at dstate 128 need 20 MiB of scratch, more than the 16 MiB array
    dims = pkg.Dims(4, 256, 80, 64, 1, 128)
    assert pkg.ssd_fwd_workspace_bytes(4, 256, 80, 64, 1, 128, "bf16", 256, "tc") > SCRATCH_BYTES
    # real device buffers of the declared shapes: if the size check ever moved behind
    # the launch, this would show as a wrong return code or output, not as a fault
    b, L, h, p, g, n = 4, 256, 80, 64, 1, 128
    x = torch.zeros((b, L, h, p), dtype=torch.bfloat16, device="cuda")
    dt = torch.zeros((b, L, h), dtype=torch.float32, device="cuda")
    hv = torch.zeros((h,), dtype=torch.float32, device="cuda")
    A = -torch.ones((h,), dtype=torch.float32, device="cuda")
    B = torch.zeros((b, L, g, n), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((b, L, g, n), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros_like(x)
    torch.cuda.synchronize()
    c0 = pkg.ssd_kernel_launches()
    rc = lib.ssd_fwd_noalloc(ctypes.byref(dims), 1, x.data_ptr(), dt.data_ptr(), hv.data_ptr(), A.data_ptr(),
                             B.data_ptr(), C.data_ptr(), None, None, 256, 1, y.data_ptr(), None, None)
    assert rc == 5  # SSD_ERR_WORKSPACE, before any launch
    assert pkg.ssd_kernel_launches() == c0
