"""GPU parity of the operations around the scan (causal conv1d + SiLU, its
decode step, the gated RMSNorm) against the fp64 oracle in oracle/layer_ops.py.

Inputs are slices of a seeded in_proj output zxbcdt [b, L, 2 d_inner + 2 g n + h]
(xBC = channels [d_inner, 2 d_inner + 2 g n), gate z = channels [0, d_inner)),
read in place through the row stride. Tolerance: max|delta| / max|ref| <= 1e-4
for fp32 io and 2e-2 for bf16 io (the forward's bound), on every output.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from forms import rel_err
from gpu_util import TOL
from mamba_ssd_chunked_gb300.inputs import CONV_WORKLOAD, NORM_WORKLOAD, make_layer_inputs, round_to_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_gb300 import build
    build.build()


def _dev(a, io):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(torch.bfloat16) if io == "bf16" else t


def _np(t):
    return t.float().cpu().numpy()


# (b, L, d_inner, g, n, K): several 32-token runs with a ragged tail, L < K,
# a scalar-path shape (d_inner not a multiple of 8), other tap counts
CONV_SHAPES = [
    (2, 77, 64, 2, 16, 4),
    (1, 2, 64, 1, 16, 4),
    (3, 33, 60, 1, 12, 4),
    (2, 40, 32, 1, 8, 1),
    (2, 40, 32, 1, 8, 3),
    (1, 129, 128, 2, 32, 8),
]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", CONV_SHAPES)
@pytest.mark.parametrize("bias,act", [(True, True), (False, True), (True, False)])
def test_conv1d_matches_oracle(shape, io, bias, act):
    import mamba_ssd_chunked_gb300 as pkg
    b, L, di, g, n, K = shape
    nh = 4
    inp = make_layer_inputs(b, L, di, g, n, nh, kernel_size=K, io_dtype=io, seed=sum(shape) + K)
    cd = di + 2 * g * n
    z = _dev(inp["zxbcdt"], io)
    xbc = z[..., di:di + cd]                               # strided slice, read in place
    w = _dev(inp["conv_w"], "f32")
    bb = _dev(inp["conv_b"], "f32") if bias else None
    x, Bo, Co, st = pkg.ssd_conv1d_silu(xbc, w, bb, di, g, n, activation=act, return_state=True)
    rx, rB, rC, rst = oracle.conv1d_silu(inp["zxbcdt"][..., di:di + cd], inp["conv_w"],
                                         inp["conv_b"] if bias else None, di, g * n, activation=act)
    tol = TOL[io]
    for name, got, ref in (("x", x, rx), ("B", Bo.reshape(b, L, g * n), rB), ("C", Co.reshape(b, L, g * n), rC)):
        e = rel_err(_np(got), ref)
        assert e <= tol, f"{shape} {io} {name}: {e:.3e}"
    assert np.array_equal(_np(st), rst), "conv state must be the last K inputs exactly"


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv1d_decode_steps_reproduce_the_prefill(io):
    """Token-by-token ssd_conv1d_step from a zero conv state gives the prefill's
    outputs (to rounding) and, exactly, its conv state."""
    import mamba_ssd_chunked_gb300 as pkg
    b, L, di, g, n, K = 2, 21, 64, 1, 16, 4
    inp = make_layer_inputs(b, L, di, g, n, 4, kernel_size=K, io_dtype=io, seed=5)
    cd = di + 2 * g * n
    z = _dev(inp["zxbcdt"], io)
    w, bb = _dev(inp["conv_w"], "f32"), _dev(inp["conv_b"], "f32")
    x, Bo, Co, st = pkg.ssd_conv1d_silu(z[..., di:di + cd], w, bb, di, g, n, return_state=True)
    state = torch.zeros((b, cd, K), dtype=z.dtype, device="cuda")
    tol = TOL[io]
    for t in range(L):
        xs, bs, cs = pkg.ssd_conv1d_step(z[:, t, di:di + cd], state, w, bb, di, g, n)
        assert rel_err(_np(xs), _np(x[:, t])) <= tol
        assert rel_err(_np(bs).reshape(b, -1), _np(Bo[:, t]).reshape(b, -1)) <= tol
        assert rel_err(_np(cs).reshape(b, -1), _np(Co[:, t]).reshape(b, -1)) <= tol
    assert torch.equal(state, st)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv1d_step_matches_oracle(io):
    import mamba_ssd_chunked_gb300 as pkg
    b, di, g, n, K = 3, 96, 2, 16, 4
    inp = make_layer_inputs(b, K + 1, di, g, n, 4, kernel_size=K, io_dtype=io, seed=6)
    cd = di + 2 * g * n
    z = _dev(inp["zxbcdt"], io)
    # carried state = the first K tokens; the step consumes token K
    _, _, _, st = pkg.ssd_conv1d_silu(z[:, :K].contiguous()[..., di:di + cd], _dev(inp["conv_w"], "f32"), None,
                                      di, g, n, return_state=True)
    _, _, _, st0 = oracle.conv1d_silu(inp["zxbcdt"][:, :K, di:di + cd], inp["conv_w"], None, di, g * n)
    assert np.array_equal(_np(st), st0)
    xs, bs, cs = pkg.ssd_conv1d_step(z[:, K, di:di + cd], st, _dev(inp["conv_w"], "f32"),
                                     _dev(inp["conv_b"], "f32"), di, g, n)
    rx, rB, rC, rst = oracle.conv1d_step(inp["zxbcdt"][:, K, di:di + cd], st0, inp["conv_w"], inp["conv_b"], di,
                                         g * n)
    tol = TOL[io]
    assert rel_err(_np(xs), rx) <= tol
    assert rel_err(_np(bs).reshape(b, -1), rB) <= tol
    assert rel_err(_np(cs).reshape(b, -1), rC) <= tol
    assert np.array_equal(_np(st), rst)


def test_conv1d_full_size_sampled_channels():
    """The 2.7B-layer conv (b 4, L 4096, d_inner 5120, g 1, n 128, K 4, bf16) in the
    launch configuration the benchmark times; the oracle checks a sample of channels
    (each channel is an independent convolution) over every token."""
    import mamba_ssd_chunked_gb300 as pkg
    w = CONV_WORKLOAD
    b, L, di, g, n, h, K = w["batch"], w["seqlen"], w["d_inner"], w["ngroups"], w["dstate"], w["nheads"], \
        w["kernel_size"]
    inp = make_layer_inputs(b, L, di, g, n, h, kernel_size=K, io_dtype=w["io_dtype"], seed=w["seed"])
    cd = di + 2 * g * n
    z = _dev(inp["zxbcdt"], "bf16")
    x, Bo, Co, st = pkg.ssd_conv1d_silu(z[..., di:di + cd], _dev(inp["conv_w"], "f32"), _dev(inp["conv_b"], "f32"),
                                        di, g, n, return_state=True)
    full = torch.cat([x, Bo.reshape(b, L, -1), Co.reshape(b, L, -1)], dim=-1)
    rng = np.random.Generator(np.random.PCG64(7))
    chans = np.unique(np.concatenate([[0, di - 1, di, di + g * n, cd - 1], rng.integers(0, cd, 59)]))
    xs = inp["zxbcdt"][..., di:di + cd][..., chans]
    ref, _, _, _ = oracle.conv1d_silu(xs, inp["conv_w"][chans], inp["conv_b"][chans], len(chans), 0)
    got = _np(full[..., torch.from_numpy(chans).cuda()])
    assert rel_err(got, ref) <= TOL["bf16"]


# (rows, dim, group_size or None, with z, z strided)
NORM_SHAPES = [
    (37, 256, None, True, True),
    (16, 5120, None, True, True),
    (9, 5120, 640, True, False),
    (5, 96, None, False, False),
    (6, 9216, None, True, True),   # more than 8 vectors per thread: the re-reading pass
    (7, 100, 25, True, False),     # not a multiple of 8: scalar path
]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", NORM_SHAPES)
def test_gated_rmsnorm_matches_oracle(shape, io):
    import mamba_ssd_chunked_gb300 as pkg
    rows, dim, gs, with_z, strided = shape
    rng = np.random.Generator(np.random.PCG64(rows * dim))
    rnd = round_to_bf16 if io == "bf16" else (lambda a: a)
    y = rnd(rng.standard_normal((rows, dim)).astype(np.float32))
    wide = rnd(rng.standard_normal((rows, dim + (24 if strided else 0))).astype(np.float32))
    wgt = (1.0 + 0.1 * rng.standard_normal(dim)).astype(np.float32)
    yd, wd = _dev(y, io), _dev(wide, io)
    zd = wd[:, 8:8 + dim] if strided else wd[:, :dim]
    y_ref_in = y
    z_ref_in = (wide[:, 8:8 + dim] if strided else wide[:, :dim]) if with_z else None
    out = pkg.ssd_gated_rmsnorm(yd, zd if with_z else None, _dev(wgt, "f32"), eps=1e-5, group_size=gs)
    ref = oracle.gated_rmsnorm(y_ref_in, z_ref_in, wgt, 1e-5, group_size=gs)
    e = rel_err(_np(out), ref)
    assert e <= TOL[io], f"{shape} {io}: {e:.3e}"


def test_gated_rmsnorm_full_size_sampled_rows():
    """The 2.7B-layer norm (16384 rows of 5120, bf16, gate read in place from the
    in_proj output) in the benchmark's launch configuration; sampled rows checked."""
    import mamba_ssd_chunked_gb300 as pkg
    w = NORM_WORKLOAD
    b, L, di, g, n, h = w["batch"], w["seqlen"], w["d_inner"], w["ngroups"], w["dstate"], w["nheads"]
    inp = make_layer_inputs(b, L, di, g, n, h, io_dtype=w["io_dtype"], seed=w["seed"])
    z = _dev(inp["zxbcdt"], "bf16")[..., :di]
    y = _dev(inp["y"], "bf16")
    out = pkg.ssd_gated_rmsnorm(y, z, _dev(inp["norm_w"], "f32"), eps=w["eps"])
    rng = np.random.Generator(np.random.PCG64(8))
    rows = np.unique(np.concatenate([[0, b * L - 1], rng.integers(0, b * L, 126)]))
    yf = inp["y"].reshape(b * L, di)[rows]
    zf = inp["zxbcdt"].reshape(b * L, -1)[rows, :di]
    ref = oracle.gated_rmsnorm(yf, zf, inp["norm_w"], w["eps"])
    got = _np(out.reshape(b * L, di)[torch.from_numpy(rows).cuda()])
    assert rel_err(got, ref) <= TOL["bf16"]
