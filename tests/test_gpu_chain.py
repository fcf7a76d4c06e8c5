"""GPU parity of the chain-local tensor-core path (SSD_PATH_CHAIN) against the
fp64 oracle.

The cases cover: one tile, a single token, lengths one below / above a tile,
ragged lengths, head pairs of one or several groups, headdim 128 (a chain
per head); chains split across CTAs
(a hand-off at every block, and hand-offs in the middle of long chains);
blocks that run whole, blocks split into 64-, 32- and 16-token sub-blocks by
their decay, and 16-token sub-blocks whose decay is still too strong
("extreme", finished on the CUDA cores), mixed within one head pair; absent
D / initial state / final state; the rejection of odd heads per group; and
agreement with the per-block tensor-core path.
Tolerance: max|delta| / max|ref| <= 2e-2 on y and on the final state (bf16 io).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from forms import rel_err
from gpu_util import TOL, check_against_oracle, check_sampled, oracle_full, run_gpu, to_device
from mamba_ssd_chunked_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_gb300 import build
    build.build()


CHAIN_SHAPES = [
    # b, L, h, p, g, n
    (1, 128, 2, 64, 1, 128),      # one tile, one head pair
    (1, 1, 2, 64, 1, 128),        # a single token
    (2, 127, 4, 64, 2, 128),      # one below a tile
    (2, 129, 4, 64, 1, 128),      # one above a tile
    (2, 300, 4, 64, 2, 128),      # ragged, several tiles
    (1, 1000, 6, 64, 3, 128),     # three groups of one pair each
    (3, 513, 8, 64, 2, 128),
    (1, 2000, 2, 64, 1, 128),     # one chain spread over many CTAs: a hand-off at every block
    (2, 4100, 6, 64, 1, 128),     # long chains split across CTAs mid-chain
    # dstate 256: the state fills half of tensor memory (single-buffered H and Y)
    (1, 128, 2, 64, 1, 256),
    (2, 300, 4, 64, 2, 256),
    (1, 1000, 6, 64, 3, 256),
    (1, 2000, 2, 64, 1, 256),     # a hand-off at every block
    (2, 4100, 6, 64, 1, 256),
    # headdim 128: a chain is one head, its two 64-row halves in one MMA
    (1, 128, 1, 128, 1, 128),     # one tile, one head
    (2, 300, 3, 128, 3, 128),     # ragged; three groups of one head (odd heads per group)
    (1, 1000, 5, 128, 1, 128),
    (1, 2000, 1, 128, 1, 128),    # one chain over many CTAs: a hand-off at every block
    (2, 300, 4, 128, 2, 256),     # dstate 256
    (1, 2000, 2, 128, 1, 256),
]


@pytest.mark.parametrize("shape", CHAIN_SHAPES)
@pytest.mark.parametrize("chunk_len", [128, 256])
def test_chain_path_matches_oracle(shape, chunk_len):
    check_against_oracle(shape, "bf16", chunk_len, "chain", seed=sum(shape) + chunk_len + 1)


@pytest.mark.parametrize("n,p", [(128, 64), (256, 64), (128, 128)])
@pytest.mark.parametrize("dt_shift,A_scale", [(3.0, 4.0), (1.0, 2.0), (-2.0, 0.25), (0.0, 1.0)])
def test_chain_path_strong_and_weak_decay(dt_shift, A_scale, n, p):
    """Uniformly strong decay (most 16-token sub-blocks extreme), moderate
    (blocks split into sub-blocks), weak (whole blocks)."""
    inp = make_inputs(2, 1100, 8, p, 2, n, io_dtype="bf16", init="normal", seed=43)
    inp["dt"] = (inp["dt"] + dt_shift).astype(np.float32)
    inp["A"] = (inp["A"] * A_scale).astype(np.float32)
    t = to_device(inp, "bf16")
    y, fs = run_gpu(t, 256, "chain")
    y_ref, f_ref = oracle_full(inp)
    assert rel_err(y.float().cpu().numpy(), y_ref) < 2e-2
    assert rel_err(fs.cpu().numpy(), f_ref) < 2e-2


def test_chain_path_vanishing_dt():
    """Heads whose dt underflows (dt_bias -100, mixed with ordinary heads inside
    head pairs): their W factor falls below the bf16 range, so D x comes from x
    itself; with dt = 0 the state stays the initial one and y = C s_in + D x."""
    import oracle
    inp = make_inputs(2, 700, 8, 64, 2, 128, io_dtype="bf16", init="normal", seed=23)
    inp["dt_bias"] = inp["dt_bias"].copy()
    inp["dt_bias"][[1, 4, 6]] = -100.0
    t = to_device(inp, "bf16")
    y, fs = run_gpu(t, 256, "chain")
    y_ref, f_ref = oracle_full(inp)
    yg = y.float().cpu().numpy()
    for sel in ([1, 4, 6], [0, 2, 3, 5, 7]):
        assert rel_err(yg[:, :, sel], y_ref[:, :, sel]) < TOL["bf16"], sel
    assert rel_err(fs.cpu().numpy(), f_ref) < TOL["bf16"]
    # the D term is a large part of y on those heads: dropping it would fail
    y_nod, _ = oracle.recurrence(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                                 np.zeros_like(inp["D"]), inp["init_state"])
    assert rel_err(y_nod[:, :, [1, 4, 6]], y_ref[:, :, [1, 4, 6]]) > 0.1


def test_chain_path_mixed_modes_within_a_pair():
    """Heads of one pair decay at very different rates, and a head's blocks
    switch between whole, split and extreme along the chain (dt bursts)."""
    b, L, h = 2, 1500, 4
    inp = make_inputs(b, L, h, 64, 1, 128, io_dtype="bf16", init="normal", seed=47)
    inp["A"] = np.array([-0.5, -12.0, -2.0, -16.0], dtype=np.float32)
    dt = inp["dt"]
    dt[:, 300:420, :] += 3.0          # a burst: strong decay in a few blocks only
    dt[:, 900:1000, 0] += 4.0
    inp["dt"] = dt.astype(np.float32)
    t = to_device(inp, "bf16")
    y, fs = run_gpu(t, 256, "chain")
    y_ref, f_ref = oracle_full(inp)
    assert rel_err(y.float().cpu().numpy(), y_ref) < 2e-2
    assert rel_err(fs.cpu().numpy(), f_ref) < 2e-2


@pytest.mark.parametrize("init,with_D", [("zero", True), ("normal", False), ("zero", False)])
def test_chain_path_optional_inputs(init, with_D):
    check_against_oracle((2, 400, 4, 64, 2, 128), "bf16", 256, "chain", init=init, with_D=with_D, seed=8)


def test_chain_path_final_state_optional():
    inp = make_inputs(1, 300, 2, 64, 1, 128, io_dtype="bf16", init="normal", seed=20)
    t = to_device(inp, "bf16")
    y, fs = run_gpu(t, 256, "chain", return_final_state=False)
    assert fs is None
    y_ref, _ = oracle_full(inp)
    assert rel_err(y.float().cpu().numpy(), y_ref) < 2e-2


@pytest.mark.parametrize("split", [256, 200])
def test_chain_path_split_sequence_carries_state(split):
    L = 900
    inp = make_inputs(2, L, 4, 64, 2, 128, io_dtype="bf16", init="normal", seed=14)
    t = to_device(inp, "bf16")
    y, fs = run_gpu(t, 256, "chain")
    first = {k: (v[:, :split].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in t.items()}
    second = {k: (v[:, split:].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in t.items()}
    y1, f1 = run_gpu(first, 256, "chain")
    second["init_state"] = f1
    y2, f2 = run_gpu(second, 256, "chain")
    y_cat = torch.cat([y1, y2], dim=1).float().cpu().numpy()
    assert rel_err(y_cat, y.float().cpu().numpy()) < TOL["bf16"]
    assert rel_err(f2.cpu().numpy(), fs.cpu().numpy()) < TOL["bf16"]


def test_chain_path_repeat_runs_are_bitwise_identical():
    inp = make_inputs(2, 2900, 8, 64, 2, 128, io_dtype="bf16", init="normal", seed=18)
    t = to_device(inp, "bf16")
    y1, f1 = run_gpu(t, 256, "chain")
    y2, f2 = run_gpu(t, 256, "chain")
    assert torch.equal(y1, y2) and torch.equal(f1, f2)


def test_chain_and_per_block_paths_agree():
    inp = make_inputs(2, 1600, 8, 64, 2, 128, io_dtype="bf16", init="normal", seed=10)
    t = to_device(inp, "bf16")
    y1, f1 = run_gpu(t, 256, "chain")
    y2, f2 = run_gpu(t, 256, "tc")
    assert rel_err(y1.float().cpu().numpy(), y2.float().cpu().numpy()) < 2e-2
    assert rel_err(f1.cpu().numpy(), f2.cpu().numpy()) < 2e-2


def test_chain_path_headline_strongest_heads():
    """The Mamba2-2.7B layer shape, checked on the heads with the strongest and
    the weakest decay (exact mode in most blocks / reference mode throughout)."""
    from mamba_ssd_chunked_gb300.inputs import workload_inputs
    inp = workload_inputs("mamba2_2p7b_layer")
    t = to_device(inp, "bf16")
    y, fs = run_gpu(t, 256, "chain")
    dt = np.logaddexp(0.0, inp["dt"].astype(np.float64) + inp["dt_bias"])
    rate = (dt * -inp["A"]).mean(axis=(0, 1))
    order = np.argsort(rate)
    heads = [int(order[-1]), int(order[-2]), int(order[0])]
    chains = sorted({(bi, hi) for bi in (0, 3) for hi in heads})
    check_sampled(inp, y, fs, chains, "bf16")


@pytest.mark.parametrize("name", ["mamba2_130m_layer", "grouped_ragged"])
def test_chain_path_full_size_workloads(name):
    """Full-size workloads with dstate 128 through the chain path, on a seeded
    sample of (batch, head) chains plus the strongest-decay head."""
    from gpu_util import sampled_chains
    from mamba_ssd_chunked_gb300.inputs import WORKLOADS, workload_inputs
    w = WORKLOADS[name]
    inp = workload_inputs(name)
    t = to_device(inp, "bf16")
    y, fs = run_gpu(t, w.chunk_len, "chain")
    dt = np.logaddexp(0.0, inp["dt"].astype(np.float64) + inp["dt_bias"])
    strongest = int(np.argmax((dt * -inp["A"]).mean(axis=(0, 1))))
    chains = sorted(set(sampled_chains(w.batch, w.nheads, 8, seed=w.seed)) | {(0, strongest), (w.batch - 1, strongest)})
    check_sampled(inp, y, fs, chains, "bf16")
    assert torch.isfinite(y.float()).all() and torch.isfinite(fs).all()


def test_chain_path_consecutive_strong_reference_blocks():
    """Every block decays by about 120 nats (below the split threshold), so the
    rescaling from one block's scaled state to the next spans e^{-120}: the
    scale pass must not form that factor in one fp32 number (it underflows),
    or the state term of each block's first rows is lost."""
    b, L, h = 2, 1536, 4
    inp = make_inputs(b, L, h, 64, 1, 128, io_dtype="bf16", init="normal", seed=53)
    inp["A"] = np.array([-1.0, -1.0, -0.5, -2.0], dtype=np.float32)
    # softplus(dt_raw + dt_bias) close to 0.94 / |A|: block decay near 120
    target = 0.94 / -inp["A"]
    inp["dt_bias"] = (target + np.log(-np.expm1(-target))).astype(np.float32)
    inp["dt"] = (0.02 * inp["dt"]).astype(np.float32)
    t = to_device(inp, "bf16")
    y, fs = run_gpu(t, 256, "chain")
    y_ref, f_ref = oracle_full(inp)
    ey = rel_err(y.float().cpu().numpy(), y_ref)
    ef = rel_err(fs.cpu().numpy(), f_ref)
    assert ey < 2e-2 and ef < 2e-2, (ey, ef)
    # the first row of every block carries the state term: check it on its own
    first = y_ref[:, ::128]
    got = y.float().cpu().numpy()[:, ::128]
    assert rel_err(got, first) < 2e-2


@pytest.mark.parametrize("decay", [200.0, 400.0, 800.0, 3000.0])
def test_chain_path_each_split_level(decay):
    """A block decay of ~200 / 400 / 800 nats selects 64- / 32- / 16-token
    sub-blocks, ~3000 makes every 16-token sub-block extreme."""
    b, L, h = 1, 640, 2
    inp = make_inputs(b, L, h, 64, 1, 128, io_dtype="bf16", init="normal", seed=61)
    inp["A"] = np.array([-1.0, -0.5], dtype=np.float32)
    target = (decay / 128.0) / -inp["A"]
    inp["dt_bias"] = (target + np.log(-np.expm1(-target))).astype(np.float32)
    inp["dt"] = (0.02 * inp["dt"]).astype(np.float32)
    t = to_device(inp, "bf16")
    y, fs = run_gpu(t, 256, "chain")
    y_ref, f_ref = oracle_full(inp)
    assert rel_err(y.float().cpu().numpy(), y_ref) < 2e-2
    assert rel_err(fs.cpu().numpy(), f_ref) < 2e-2


def test_chain_path_rejects_odd_heads_per_group():
    import mamba_ssd_chunked_gb300 as pkg
    inp = make_inputs(1, 256, 3, 64, 3, 128, io_dtype="bf16", init="zero", seed=3)
    t = to_device(inp, "bf16")
    assert pkg.ssd_fwd_workspace_bytes(1, 256, 3, 64, 3, 128, "bf16", 256, "chain") == 0
    with pytest.raises(pkg.SsdError):
        run_gpu(t, 256, "chain")
