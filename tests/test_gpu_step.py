"""GPU parity of the decode step (ssd_step) against the fp64 oracle, and the
invariant that L decode steps reproduce the chunked forward over L tokens.

Tolerances: max|delta| / max|ref| <= 1e-4 for fp32 io and 2e-2 for bf16 io, on
y and on the updated state.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from forms import rel_err
from gpu_util import TOL, run_gpu, to_device
from mamba_ssd_chunked_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_gb300 import build
    build.build()


def _step_inputs(b, h, p, g, n, io, seed, with_D=True):
    inp = make_inputs(b, 1, h, p, g, n, io_dtype=io, init="normal", seed=seed, with_D=with_D)
    return {"x": inp["x"][:, 0], "dt": inp["dt"][:, 0], "dt_bias": inp["dt_bias"], "A": inp["A"],
            "B": inp["B"][:, 0], "C": inp["C"][:, 0], "D": inp["D"], "state": inp["init_state"]}


def _to_dev(s, io):
    tdt = torch.bfloat16 if io == "bf16" else torch.float32
    out = {}
    for k, v in s.items():
        if v is None:
            out[k] = None
            continue
        t = torch.from_numpy(np.ascontiguousarray(v)).cuda()
        out[k] = t.to(tdt) if k in ("x", "B", "C") else t
    return out


STEP_SHAPES = [
    # b, h, p, g, n
    (2, 4, 64, 2, 128),
    (3, 6, 16, 3, 16),
    (1, 8, 32, 1, 64),
    (2, 4, 64, 1, 100),   # n not a multiple of 4: the scalar kernel
    (1, 1, 1, 1, 1),
    (5, 80, 64, 1, 128),  # the Mamba2-2.7B layer's heads
]


@pytest.mark.parametrize("shape", STEP_SHAPES)
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_step_matches_oracle(shape, io):
    import mamba_ssd_chunked_gb300 as pkg
    b, h, p, g, n = shape
    s = _step_inputs(b, h, p, g, n, io, seed=sum(shape) + (7 if io == "bf16" else 0))
    d = _to_dev(s, io)
    y = pkg.ssd_step(d["x"], d["dt"], d["dt_bias"], d["A"], d["B"], d["C"], d["D"], d["state"])
    torch.cuda.synchronize()
    y_ref, s_ref = oracle.step(s["x"], s["dt"], s["dt_bias"], s["A"], s["B"], s["C"], s["D"], s["state"])
    assert rel_err(y.float().cpu().numpy(), y_ref) <= TOL[io]
    assert rel_err(d["state"].cpu().numpy(), s_ref) <= TOL[io]


def test_step_without_D():
    import mamba_ssd_chunked_gb300 as pkg
    s = _step_inputs(2, 4, 64, 2, 128, "f32", seed=3, with_D=False)
    d = _to_dev(s, "f32")
    y = pkg.ssd_step(d["x"], d["dt"], d["dt_bias"], d["A"], d["B"], d["C"], None, d["state"])
    y_ref, s_ref = oracle.step(s["x"], s["dt"], s["dt_bias"], s["A"], s["B"], s["C"], None, s["state"])
    assert rel_err(y.cpu().numpy(), y_ref) <= 1e-4 and rel_err(d["state"].cpu().numpy(), s_ref) <= 1e-4


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_decode_steps_reproduce_the_chunked_forward(io):
    """Feeding L tokens one ssd_step at a time from an initial state gives the
    same y and final state as one ssd_fwd call over the L tokens."""
    import mamba_ssd_chunked_gb300 as pkg
    b, L, h, p, g, n = 2, 40, 4, 64, 2, 128
    inp = make_inputs(b, L, h, p, g, n, io_dtype=io, init="normal", seed=61)
    t = to_device(inp, io)
    y_fwd, f_fwd = run_gpu(t, 256)
    state = t["init_state"].clone()
    ys = []
    for i in range(L):
        ys.append(pkg.ssd_step(t["x"][:, i].contiguous(), t["dt"][:, i].contiguous(), t["dt_bias"], t["A"],
                               t["B"][:, i].contiguous(), t["C"][:, i].contiguous(), t["D"], state))
    y_steps = torch.stack(ys, dim=1)
    torch.cuda.synchronize()
    tol = TOL[io]
    assert rel_err(y_steps.float().cpu().numpy(), y_fwd.float().cpu().numpy()) <= tol
    assert rel_err(state.cpu().numpy(), f_fwd.cpu().numpy()) <= tol


def test_step_counts_one_launch():
    import mamba_ssd_chunked_gb300 as pkg
    s = _step_inputs(1, 2, 16, 1, 16, "f32", seed=5)
    d = _to_dev(s, "f32")
    c0 = pkg.ssd_kernel_launches()
    pkg.ssd_step(d["x"], d["dt"], d["dt_bias"], d["A"], d["B"], d["C"], d["D"], d["state"])
    assert pkg.ssd_kernel_launches() - c0 == 1
