"""GPU parity of the dt_limit clamp (fla "mamba2.py", Mamba2.torch_forward: clamp of
softplus(dt + dt_bias) to time_step_limit) on every path against the fp64 oracle
run with the same limit, and the default limit (0, inf) leaving results
bit-identical. Tolerances as the forward: 1e-4 fp32 io, 2e-2 bf16 io.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from forms import rel_err
from gpu_util import TOL, to_device
from mamba_ssd_chunked_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

LIMITS = [(0.02, 0.3), (0.05, 0.05), (0.0, 0.01)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_gb300 import build
    build.build()


def _fwd(t, chunk_len, path, lim):
    import mamba_ssd_chunked_gb300 as pkg
    y, fs = pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                        chunk_len=chunk_len, path=path, dt_limit=lim)
    assert pkg.ssd_device_status() == 0
    return y, fs


# (shape b, L, h, p, g, n; io; chunk_len; path)
CASES = [
    ((2, 200, 4, 16, 2, 16), "f32", 64, "simt"),
    ((2, 333, 8, 64, 2, 128), "bf16", 256, "tc"),
    ((1, 700, 8, 64, 1, 256), "bf16", 128, "tc"),
    ((2, 333, 8, 64, 2, 128), "bf16", 256, "chain"),
]


@pytest.mark.parametrize("lim", LIMITS)
@pytest.mark.parametrize("shape,io,Q,path", CASES)
def test_forward_with_dt_limit_matches_oracle(shape, io, Q, path, lim):
    b, L, h, p, g, n = shape
    inp = make_inputs(b, L, h, p, g, n, io_dtype=io, init="normal", seed=sum(shape) + int(1000 * lim[0]))
    t = to_device(inp, io)
    y, fs = _fwd(t, Q, path, lim)
    y_ref, f_ref = oracle.recurrence(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["D"],
                                     inp["init_state"], dt_limit=lim)
    ey, ef = rel_err(y.float().cpu().numpy(), y_ref), rel_err(fs.cpu().numpy(), f_ref)
    assert ey <= TOL[io] and ef <= TOL[io], f"{shape} {path} {lim}: y {ey:.3e} final {ef:.3e}"
    # the clamp must have mattered: the unclamped oracle differs
    y0, f0 = oracle.recurrence(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["D"],
                               inp["init_state"])
    assert rel_err(y0, y_ref) > TOL[io] or rel_err(f0, f_ref) > TOL[io]


@pytest.mark.parametrize("shape,io,Q,path", CASES)
def test_default_dt_limit_is_bit_identical(shape, io, Q, path):
    import mamba_ssd_chunked_gb300 as pkg
    b, L, h, p, g, n = shape
    inp = make_inputs(b, L, h, p, g, n, io_dtype=io, init="normal", seed=11)
    t = to_device(inp, io)
    y1, f1 = _fwd(t, Q, path, (0.0, float("inf")))
    y0, f0 = pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                         chunk_len=Q, path=path)
    assert torch.equal(y0, y1) and torch.equal(f0, f1)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("n", [128, 64, 30])
@pytest.mark.parametrize("lim", LIMITS)
def test_decode_step_with_dt_limit_matches_oracle(io, n, lim):
    import mamba_ssd_chunked_gb300 as pkg
    b, h, p, g = 3, 8, 64, 2
    inp = make_inputs(b, 1, h, p, g, n, io_dtype=io, init="normal", seed=n + int(1000 * lim[0]))
    t = to_device(inp, io)
    state = t["init_state"].clone()
    y = pkg.ssd_step(t["x"][:, 0].contiguous(), t["dt"][:, 0].contiguous(), t["dt_bias"], t["A"],
                     t["B"][:, 0].contiguous(), t["C"][:, 0].contiguous(), t["D"], state, dt_limit=lim)
    y_ref, s_ref = oracle.step(inp["x"][:, 0], inp["dt"][:, 0], inp["dt_bias"], inp["A"], inp["B"][:, 0],
                               inp["C"][:, 0], inp["D"], inp["init_state"], dt_limit=lim)
    assert rel_err(y.float().cpu().numpy(), y_ref) <= TOL[io]
    assert rel_err(state.cpu().numpy(), s_ref) <= TOL[io]
