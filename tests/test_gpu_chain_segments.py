"""Chain path: chains whose blocks are spread over several CTAs, and the
pairing of heads by decay rate, against the fp64 oracle.

Where a CTA's range begins inside a chain, the CTA either waits for the
previous CTA's hand-off of the state or recomputes that state itself from the
blocks before its segment (a warm-up): from a zero state where both heads of
the pair decay by more than 32 nats over the warm-up, else from the chain's
initial state at block 0. SSD_CHAIN_WARMUP selects 0 (always the hand-off),
1 (the default: warm up where the hand-off would come late) or 2 (warm up
wherever possible). Every mode must give the oracle's result.

Heads are paired by their decay rate within each B/C group, so a pair is in
general not two neighbouring heads; the cases below put fast and slow heads
in scrambled order (and across groups) so that a wrong head map would show.
Tolerance: max|delta| / max|ref| <= 2e-2 on y and on the final state (bf16 io).
"""
import contextlib
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from forms import rel_err
from gpu_util import TOL, oracle_full, run_gpu, to_device
from mamba_ssd_chunked_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_gb300 import build
    build.build()


@contextlib.contextmanager
def warmup_mode(mode):
    old = os.environ.get("SSD_CHAIN_WARMUP")
    os.environ["SSD_CHAIN_WARMUP"] = str(mode)
    try:
        yield
    finally:
        if old is None:
            os.environ.pop("SSD_CHAIN_WARMUP", None)
        else:
            os.environ["SSD_CHAIN_WARMUP"] = old


def check(inp, chunk_len=256):
    t = to_device(inp, "bf16")
    y, fs = run_gpu(t, chunk_len, "chain")
    y_ref, f_ref = oracle_full(inp)
    ey, ef = rel_err(y.float().cpu().numpy(), y_ref), rel_err(fs.cpu().numpy(), f_ref)
    assert ey <= TOL["bf16"] and ef <= TOL["bf16"], (ey, ef)
    return y, fs


# (b, L, h, g, dt_shift, A_scale): jobs are (head pair, 128-token block); with fewer
# jobs than SMs every CTA takes one or two blocks, so chains cross CTAs at every block
SEGMENT_CASES = [
    (1, 2000, 2, 1, 0.0, 1.0),     # one chain, 16 CTAs of one block each
    (1, 2000, 2, 1, 2.0, 4.0),     # the same, strongly decaying: warm-ups start from zero
    (2, 4100, 6, 1, 0.0, 1.0),     # long chains, a few blocks per CTA
    (1, 3000, 4, 2, 1.5, 3.0),     # two groups, strong decay
    (2, 1500, 8, 2, -2.0, 0.1),    # weak decay: warm-ups reach back to the initial state
]


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("case", SEGMENT_CASES)
def test_segments_match_oracle_in_every_warmup_mode(case, mode):
    b, L, h, g, dt_shift, A_scale = case
    inp = make_inputs(b, L, h, 64, g, 128, io_dtype="bf16", init="normal", seed=b * 31 + L + h)
    inp["dt"] = (inp["dt"] + dt_shift).astype(np.float32)
    inp["A"] = (inp["A"] * A_scale).astype(np.float32)
    with warmup_mode(mode):
        check(inp)


def test_warmup_from_zero_state_is_exact_to_rounding():
    """Strong decay and a forced warm-up everywhere: most CTAs restart their
    chain from a zero state a few blocks early. The result must equal the
    hand-off result to within bf16 rounding of y, and both must equal the
    oracle."""
    inp = make_inputs(1, 4096, 4, 64, 1, 128, io_dtype="bf16", init="normal", seed=77)
    inp["dt"] = (inp["dt"] + 2.5).astype(np.float32)
    inp["A"] = (inp["A"] * 6.0).astype(np.float32)
    with warmup_mode(2):
        y2, f2 = check(inp)
    with warmup_mode(0):
        y0, f0 = check(inp)
    assert rel_err(y2.float().cpu().numpy(), y0.float().cpu().numpy()) <= 1e-2
    assert rel_err(f2.cpu().numpy(), f0.cpu().numpy()) <= 1e-3


@pytest.mark.parametrize("g", [1, 2, 4])
def test_decay_sorted_pairs_map_heads_back(g):
    """Decay rates in scrambled order: the chain kernel pairs heads 0..h-1 by
    rank within each group, and every head's y and final state must still land
    in its own slot."""
    b, L, h = 2, 900, 16
    inp = make_inputs(b, L, h, 64, g, 128, io_dtype="bf16", init="normal", seed=1000 + g)
    rng = np.random.Generator(np.random.PCG64(5 + g))
    inp["A"] = (-np.exp(rng.uniform(np.log(0.2), np.log(40.0), size=h))).astype(np.float32)
    inp["dt_bias"] = rng.permutation(inp["dt_bias"]).astype(np.float32)
    for mode in (0, 2):
        with warmup_mode(mode):
            check(inp)


@pytest.mark.parametrize("mode", [0, 2])
def test_headdim_128_segments_match_oracle(mode):
    """Headdim 128 (a chain per head, its two 64-row halves in one MMA): chains
    across many CTAs with hand-offs or warm-ups."""
    inp = make_inputs(1, 3000, 3, 128, 1, 128, io_dtype="bf16", init="normal", seed=91)
    inp["dt"] = (inp["dt"] + 1.5).astype(np.float32)
    inp["A"] = (inp["A"] * 3.0).astype(np.float32)
    with warmup_mode(mode):
        check(inp)
