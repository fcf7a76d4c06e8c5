"""The input guard (ssd_check_inputs) on the GPU: per-input counts of
non-finite elements, checked against numpy's isfinite on the same values.

NaN and both infinities are planted at the first and last element and in the
middle of each input, at element offsets that leave the tensors off 16-byte
boundaries (the kernel's scalar head and tail), and in a tensor large enough
that every thread of the grid loops. Finite extremes (the largest finite
value, subnormals, -0) must not count. ssd_fwd(check_inputs=True) refuses
non-finite inputs before launching and leaves clean ones bit-identical.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from mamba_ssd_chunked_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

NAMES = ("x", "dt", "dt_bias", "A", "B", "C", "D", "init_state")
IO_NAMES = ("x", "B", "C")


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mamba_ssd_chunked_gb300 as p
    from mamba_ssd_chunked_gb300 import build
    build.build()
    return p


def place(arr: np.ndarray, io: str, name: str, offset: int):
    """The array on the GPU in its input dtype, `offset` elements into a larger buffer."""
    dt = torch.bfloat16 if (io == "bf16" and name in IO_NAMES) else torch.float32
    flat = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32).ravel()).to(dt)
    buf = torch.zeros(flat.numel() + offset + 5, dtype=dt, device="cuda")
    buf[offset:offset + flat.numel()] = flat.cuda()
    return buf[offset:offset + flat.numel()].view(arr.shape)


def expected(t) -> int:
    return int((~torch.isfinite(t.float())).sum().item()) if t is not None else 0


def run_guard(pkg, inp, io, offsets=None, drop=()):
    offsets = offsets or {}
    t = {k: (None if (inp[k] is None or k in drop) else place(inp[k], io, k, offsets.get(k, 0))) for k in NAMES}
    got = pkg.ssd_check_inputs(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"])
    return got, {k: expected(t[k]) for k in NAMES}


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_clean_inputs_count_zero(pkg, io):
    inp = make_inputs(2, 37, 4, 64, 2, 128, io_dtype=io, init="normal", seed=11)
    got, want = run_guard(pkg, inp, io)
    assert got == want == {k: 0 for k in NAMES}
    got, _ = run_guard(pkg, inp, io, drop=("D", "init_state"))
    assert got["D"] == 0 and got["init_state"] == 0


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("offset", [0, 1, 3])
def test_planted_values_counted_per_input(pkg, io, offset):
    rng = np.random.Generator(np.random.PCG64(100 + offset))
    inp = make_inputs(2, 37, 4, 64, 2, 128, io_dtype=io, init="normal", seed=12)
    specials = (np.nan, np.inf, -np.inf)
    for i, name in enumerate(NAMES):
        arr = np.array(inp[name], dtype=np.float32, copy=True)
        flat = arr.reshape(-1)
        picks = {0, flat.size - 1, flat.size // 2}
        picks |= {int(v) for v in rng.integers(0, flat.size, size=min(5, flat.size))}
        for j, pos in enumerate(sorted(picks)):
            flat[pos] = specials[(i + j) % 3]
        inp[name] = arr
    offsets = {k: offset for k in NAMES}
    got, want = run_guard(pkg, inp, io, offsets)
    for name in NAMES:
        assert want[name] > 0
    assert got == want


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_finite_extremes_do_not_count(pkg, io):
    inp = make_inputs(1, 40, 2, 64, 1, 128, io_dtype=io, init="normal", seed=13)
    big = float(torch.finfo(torch.bfloat16 if io == "bf16" else torch.float32).max)
    tiny = 1e-40  # subnormal in fp32 and bf16
    for name in NAMES:
        arr = np.array(inp[name], dtype=np.float32, copy=True)
        flat = arr.reshape(-1)
        flat[0] = big if name in IO_NAMES else np.finfo(np.float32).max
        flat[-1] = -tiny
        if flat.size > 2:
            flat[1] = -0.0
        inp[name] = arr
    got, want = run_guard(pkg, inp, io, {k: 1 for k in NAMES})
    assert got == want == {k: 0 for k in NAMES}


def test_large_input_every_thread_loops(pkg):
    # x of 2.1 M bf16 elements: more 16-byte loads than the guard's grid has threads
    inp = make_inputs(1, 4096, 8, 64, 1, 128, io_dtype="bf16", init="zero", seed=14)
    x = np.array(inp["x"], dtype=np.float32, copy=True).reshape(-1)
    pos = np.random.Generator(np.random.PCG64(15)).choice(x.size, size=1000, replace=False)
    x[pos] = np.nan
    x[-1] = np.inf
    inp["x"] = x.reshape(inp["x"].shape)
    got, want = run_guard(pkg, inp, "bf16", {"x": 1})
    assert got == want and got["x"] == len(set(pos.tolist()) | {x.size - 1})


def test_forward_refuses_non_finite_inputs(pkg):
    inp = make_inputs(1, 300, 4, 64, 2, 128, io_dtype="bf16", init="normal", seed=16)
    t = {k: place(inp[k], "bf16", k, 0) for k in NAMES}
    args = [t[k] for k in NAMES]
    y0, f0 = pkg.ssd_fwd(*args, chunk_len=256)
    y1, f1 = pkg.ssd_fwd(*args, chunk_len=256, check_inputs=True)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(f0, f1)
    launches = pkg.ssd_kernel_launches()
    t["dt"][0, 17, 3] = float("nan")
    with pytest.raises(ValueError, match="dt"):
        pkg.ssd_fwd(*[t[k] for k in NAMES], chunk_len=256, check_inputs=True)
    assert pkg.ssd_kernel_launches() == launches + 1  # the guard ran, the forward did not
    assert pkg.ssd_device_status() == 0
