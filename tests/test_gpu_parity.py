"""GPU parity: the CUDA paths against the fp64 oracle on seeded inputs.

Sizes span several 128-token tiles and ragged tails; edge cases cover a
single token, lengths one below/above a tile, every head its own group,
absent D / initial state / final state, and both chunk lengths of the
tensor-core path. Tolerances: max|dy|/max|y| and max|dfinal|/max|final| at
most 1e-4 for fp32 io and 2e-2 for bf16 io.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from forms import rel_err
from gpu_util import TOL, check_against_oracle, oracle_full, run_gpu, to_device
from mamba_ssd_chunked_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_gb300 import build
    build.build()


TC_SHAPES = [
    # b, L, h, p, g, n
    (1, 128, 1, 64, 1, 128),      # one tile
    (1, 1, 2, 64, 1, 128),        # a single token
    (2, 127, 4, 64, 2, 128),      # one below a tile
    (2, 129, 4, 64, 1, 128),      # one above a tile
    (2, 300, 4, 64, 2, 128),      # ragged, several tiles
    (1, 1000, 3, 64, 3, 128),     # ngroups == nheads
    (3, 513, 8, 64, 2, 128),
    (1, 640, 2, 64, 1, 256),      # dstate 256
    (2, 333, 4, 64, 4, 256),
]


@pytest.mark.parametrize("shape", TC_SHAPES)
@pytest.mark.parametrize("chunk_len", [128, 256])
def test_tensor_core_path_matches_oracle(shape, chunk_len):
    check_against_oracle(shape, "bf16", chunk_len, "tc", seed=sum(shape) + chunk_len)


@pytest.mark.parametrize("dt_shift,A_scale", [(3.0, 4.0), (-2.0, 0.25), (0.0, 1.0)])
def test_tensor_core_path_strong_and_weak_decay(dt_shift, A_scale):
    """Heads whose decay across 32 tokens is far above (strong) or below (weak)
    the range where the kernel stores the causal mask in factored form."""
    inp = make_inputs(2, 520, 8, 64, 2, 128, io_dtype="bf16", init="normal", seed=41)
    inp["dt"] = (inp["dt"] + dt_shift).astype(np.float32)
    inp["A"] = (inp["A"] * A_scale).astype(np.float32)
    t = to_device(inp, "bf16")
    y, fs = run_gpu(t, 256, "tc")
    y_ref, f_ref = oracle_full(inp)
    assert rel_err(y.float().cpu().numpy(), y_ref) < 2e-2
    assert rel_err(fs.cpu().numpy(), f_ref) < 2e-2


@pytest.mark.parametrize("init,with_D", [("zero", True), ("normal", False), ("zero", False)])
def test_tensor_core_path_optional_inputs(init, with_D):
    check_against_oracle((2, 400, 4, 64, 2, 128), "bf16", 256, "tc", init=init, with_D=with_D, seed=7)


SIMT_CASES = [
    # shape, io, chunk_len
    ((1, 256, 4, 16, 1, 16), "f32", 64),
    ((2, 77, 3, 8, 1, 4), "f32", 1),
    ((2, 77, 6, 8, 3, 4), "f32", 16),
    ((1, 300, 2, 32, 2, 64), "f32", 100),
    ((1, 513, 4, 64, 1, 128), "f32", 256),
    ((2, 300, 4, 64, 2, 128), "bf16", 64),
    ((1, 200, 2, 64, 1, 256), "bf16", 256),
    ((1, 1, 1, 1, 1, 1), "f32", 256),
]


@pytest.mark.parametrize("shape,io,chunk_len", SIMT_CASES)
def test_simt_path_matches_oracle(shape, io, chunk_len):
    check_against_oracle(shape, io, chunk_len, "simt", seed=3 + chunk_len)


def test_result_independent_of_chunk_length_fp32():
    inp = make_inputs(2, 700, 4, 16, 2, 32, io_dtype="f32", init="normal", seed=5)
    t = to_device(inp, "f32")
    ys, fss = [], []
    for Q in (16, 64, 128, 200, 256):
        y, fs = run_gpu(t, Q, "simt")
        ys.append(y.cpu().numpy())
        fss.append(fs.cpu().numpy())
    y_ref, f_ref = oracle_full(inp)
    for y, fs in zip(ys, fss):
        assert rel_err(y, y_ref) < 1e-4 and rel_err(fs, f_ref) < 1e-4
        assert rel_err(y, ys[0]) < 1e-4 and rel_err(fs, fss[0]) < 1e-4


def test_tensor_core_and_simt_paths_agree():
    inp = make_inputs(2, 600, 6, 64, 2, 128, io_dtype="bf16", init="normal", seed=9)
    t = to_device(inp, "bf16")
    y1, f1 = run_gpu(t, 256, "tc")
    y2, f2 = run_gpu(t, 256, "simt")
    assert rel_err(y1.float().cpu().numpy(), y2.float().cpu().numpy()) < 2e-2
    assert rel_err(f1.cpu().numpy(), f2.cpu().numpy()) < 2e-2


@pytest.mark.parametrize("path,io,split", [("tc", "bf16", 256), ("tc", "bf16", 200), ("simt", "f32", 131)])
def test_split_sequence_carries_state(path, io, split):
    """Running [0, s) then [s, L) from the carried final state reproduces the
    unsplit run (the Mamba2Cache hand-off of the final SSM state)."""
    L = 640
    inp = make_inputs(2, L, 4, 64, 2, 128, io_dtype=io, init="normal", seed=13)
    t = to_device(inp, io)
    y, fs = run_gpu(t, 256, path)
    first = {k: (v[:, :split].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in t.items()}
    second = {k: (v[:, split:].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in t.items()}
    y1, f1 = run_gpu(first, 256, path)
    second["init_state"] = f1
    y2, f2 = run_gpu(second, 256, path)
    y_cat = torch.cat([y1, y2], dim=1).float().cpu().numpy()
    tol = TOL[io]
    assert rel_err(y_cat, y.float().cpu().numpy()) < tol
    assert rel_err(f2.cpu().numpy(), fs.cpu().numpy()) < tol


@pytest.mark.parametrize("path", ["tc", "simt"])
def test_repeat_runs_are_bitwise_identical(path):
    inp = make_inputs(2, 900, 8, 64, 2, 128, io_dtype="bf16", init="normal", seed=17)
    t = to_device(inp, "bf16")
    y1, f1 = run_gpu(t, 256, path)
    y2, f2 = run_gpu(t, 256, path)
    assert torch.equal(y1, y2) and torch.equal(f1, f2)


def test_final_state_optional():
    inp = make_inputs(1, 300, 2, 64, 1, 128, io_dtype="bf16", init="normal", seed=19)
    t = to_device(inp, "bf16")
    y, fs = run_gpu(t, 256, "tc", return_final_state=False)
    assert fs is None
    y_ref, _ = oracle_full(inp)
    assert rel_err(y.float().cpu().numpy(), y_ref) < 2e-2


def test_caller_workspace_and_explicit_stream():
    import mamba_ssd_chunked_gb300 as pkg
    inp = make_inputs(2, 500, 4, 64, 1, 128, io_dtype="bf16", init="normal", seed=23)
    t = to_device(inp, "bf16")
    need = pkg.ssd_fwd_workspace_bytes(2, 500, 4, 64, 1, 128, "bf16", 256, "tc")
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y, fs = pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                            chunk_len=256, path="tc", workspace=ws, stream=s.cuda_stream)
    assert pkg.ssd_device_status(s.cuda_stream) == 0
    y_ref, f_ref = oracle_full(inp)
    assert rel_err(y.float().cpu().numpy(), y_ref) < 2e-2 and rel_err(fs.cpu().numpy(), f_ref) < 2e-2


# (shape b, L, h, p, g, n; io; init; with D; final state): the host entry point cuts
# the sequence into token slices of at least 512 tokens (cuts on multiples of 256)
# and passes the state from slice to slice: one slice (L < 1024), two with a ragged
# second one, four with a ragged last one, eight; with and without an initial and a
# final state, on the chain and the SIMT paths
HOST_CASES = [
    ((2, 300, 4, 64, 2, 128), "bf16", "normal", True, True),
    ((5, 200, 4, 64, 1, 128), "bf16", "normal", True, True),
    ((1, 129, 2, 64, 1, 128), "bf16", "zero", False, False),
    ((3, 150, 4, 16, 2, 16), "f32", "normal", True, True),
    ((2, 1100, 4, 64, 2, 128), "bf16", "normal", True, True),
    ((1, 2100, 2, 64, 1, 128), "bf16", "zero", True, True),
    ((2, 4096, 2, 64, 1, 128), "bf16", "normal", True, False),
    ((1, 1100, 4, 16, 2, 16), "f32", "normal", False, True),
]


@pytest.mark.parametrize("shape,io,init,with_D,final", HOST_CASES)
def test_host_buffer_entry_point(shape, io, init, with_D, final):
    import mamba_ssd_chunked_gb300 as pkg
    b, L, h_, p, g, n = shape
    inp = make_inputs(b, L, h_, p, g, n, io_dtype=io, init=init, seed=29 + b, with_D=with_D)
    h = {k: (None if v is None else torch.from_numpy(v)) for k, v in inp.items()}
    if io == "bf16":
        for k in ("x", "B", "C"):
            h[k] = h[k].to(torch.bfloat16)
    h = {k: (None if v is None else v.contiguous().pin_memory()) for k, v in h.items()}
    y, fs = pkg.ssd_fwd_host(h["x"], h["dt"], h["dt_bias"], h["A"], h["B"], h["C"], h["D"], h["init_state"],
                             chunk_len=256 if io == "bf16" else 64, return_final_state=final)
    y_ref, f_ref = oracle_full(inp)
    tol = TOL[io]
    assert rel_err(y.float().numpy(), y_ref) <= tol
    if final:
        assert rel_err(fs.numpy(), f_ref) <= tol
    else:
        assert fs is None


@pytest.mark.parametrize("slices,shape", [(16, (1, 8192, 2, 64, 1, 128)), (5, (2, 2600, 4, 64, 2, 128)),
                                          (3, (1, 1700, 4, 16, 2, 16))])
def test_host_entry_point_forced_slices(slices, shape, monkeypatch):
    # SSD_HOST_SLICES overrides the slice count the copy bytes give (small inputs
    # would get the minimum): the most slices the pipeline takes, an odd count
    # with a ragged last slice, and the SIMT path
    import mamba_ssd_chunked_gb300 as pkg
    b, L, h_, p, g, n = shape
    io = "bf16" if p == 64 else "f32"
    inp = make_inputs(b, L, h_, p, g, n, io_dtype=io, init="normal", seed=41 + slices)
    h = {k: torch.from_numpy(v) for k, v in inp.items()}
    if io == "bf16":
        for k in ("x", "B", "C"):
            h[k] = h[k].to(torch.bfloat16)
    h = {k: v.contiguous().pin_memory() for k, v in h.items()}
    monkeypatch.setenv("SSD_HOST_SLICES", str(slices))
    y, fs = pkg.ssd_fwd_host(h["x"], h["dt"], h["dt_bias"], h["A"], h["B"], h["C"], h["D"], h["init_state"],
                             chunk_len=256 if io == "bf16" else 64)
    y_ref, f_ref = oracle_full(inp)
    assert rel_err(y.float().numpy(), y_ref) <= TOL[io]
    assert rel_err(fs.numpy(), f_ref) <= TOL[io]


@pytest.mark.parametrize("path", ["chain", "tc", "simt"])
def test_kernel_timing_records_one_pair_per_forward(path):
    import mamba_ssd_chunked_gb300 as pkg
    inp = make_inputs(2, 300, 4, 64, 2, 128, io_dtype="bf16", init="normal", seed=3)
    t = to_device(inp, "bf16")
    pkg.ssd_kernel_timing_read()  # forget anything recorded before
    run_gpu(t, 256, path)
    assert pkg.ssd_kernel_timing_read() == (0.0, 0)  # off by default
    pkg.ssd_kernel_timing(True)
    try:
        for _ in range(3):
            run_gpu(t, 256, path)
    finally:
        pkg.ssd_kernel_timing(False)
    ms, n = pkg.ssd_kernel_timing_read()
    assert n == 3 and ms > 0.0
    assert pkg.ssd_kernel_timing_read() == (0.0, 0)


def test_launch_counter_counts_kernels():
    import mamba_ssd_chunked_gb300 as pkg
    inp = make_inputs(1, 256, 2, 64, 1, 128, io_dtype="bf16", init="zero", seed=1)
    t = to_device(inp, "bf16")
    c0 = pkg.ssd_kernel_launches()
    run_gpu(t, 256, "tc")
    c1 = pkg.ssd_kernel_launches()
    run_gpu(t, 256, "simt")
    c2 = pkg.ssd_kernel_launches()
    assert c1 - c0 == 1 and c2 - c1 == 3
