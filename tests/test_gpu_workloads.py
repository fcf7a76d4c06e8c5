"""The five workloads at full size, through ssd_fwd exactly as bench.py calls
it, checked against the fp64 oracle.

Every (batch, head) chain is compared for tiny_fp32, mamba2_130m_layer,
mamba2_2p7b_layer and grouped_ragged: the chain kernel cuts chains between
CTAs at cost-balanced, data-dependent places, so every chain is checked, not a
sample. long_context (64 chains of 131072 tokens at dstate 256) is compared on
at least 16 chains: the heads with the strongest and the weakest decay, the
first and the last chain, and a seeded sample of the rest.

The tolerance is max|delta| / max|ref| over all compared chains, for y and
for the final state separately."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from gpu_util import TOL, to_device
from mamba_ssd_chunked_gb300.inputs import WORKLOADS, workload_inputs

pytestmark = pytest.mark.gpu

CHAINS_PER_ORACLE_CALL = 32  # bounds the fp64 copy of y the oracle returns at once
LONG_CONTEXT_CHAINS = 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_gb300 import build
    build.build()


def decay_ranked_heads(inp):
    """Heads ordered by their mean per-token log-decay rate softplus(dt_bias) * (-A)."""
    bias = inp["dt_bias"].astype(np.float64)
    rate = np.log1p(np.exp(bias)) * -inp["A"].astype(np.float64)
    return [int(h) for h in np.argsort(rate, kind="stable")]


def compared_chains(name, inp):
    w = WORKLOADS[name]
    if name != "long_context":
        return [(b, h) for b in range(w.batch) for h in range(w.nheads)]
    ranked = decay_ranked_heads(inp)
    chains = {(0, ranked[0]), (0, ranked[1]), (0, ranked[-1]), (0, ranked[-2]), (0, 0), (w.batch - 1, w.nheads - 1)}
    rng = np.random.Generator(np.random.PCG64(w.seed))
    while len(chains) < LONG_CONTEXT_CHAINS:
        chains.add((int(rng.integers(w.batch)), int(rng.integers(w.nheads))))
    return sorted(chains)


def compare_chains(inp, y, fs, chains):
    """max|delta| / max|ref| of y and of the final state over the given chains."""
    dy = ry = df = rf = 0.0
    for i in range(0, len(chains), CHAINS_PER_ORACLE_CALL):
        part = chains[i:i + CHAINS_PER_ORACLE_CALL]
        y_ref, f_ref = oracle.recurrence(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                                         inp["D"], inp["init_state"], chains=part)
        bi = torch.tensor([c[0] for c in part], device=y.device)
        hi = torch.tensor([c[1] for c in part], device=y.device)
        yg = y[bi, :, hi].float().cpu().numpy()   # [k, L, p]
        fg = fs[bi, hi].cpu().numpy()             # [k, p, n]
        dy = max(dy, float(np.max(np.abs(yg - y_ref))))
        ry = max(ry, float(np.max(np.abs(y_ref))))
        df = max(df, float(np.max(np.abs(fg - f_ref))))
        rf = max(rf, float(np.max(np.abs(f_ref))))
    return dy / ry, df / rf


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_workload_matches_oracle(name):
    import mamba_ssd_chunked_gb300 as pkg
    w = WORKLOADS[name]
    inp = workload_inputs(name)
    t = to_device(inp, w.io_dtype)
    y, fs = pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                        chunk_len=w.chunk_len)
    assert pkg.ssd_device_status() == 0
    if w.io_dtype == "f32":
        expect_path = "simt"
    elif w.dstate in (128, 256) and (w.nheads // w.ngroups) % 2 == 0:
        expect_path = "chain"
    else:
        expect_path = "tc"
    assert pkg.ssd_select_path(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.io_dtype,
                               w.chunk_len) == expect_path
    assert torch.isfinite(y.float()).all() and torch.isfinite(fs).all()
    chains = compared_chains(name, inp)
    assert len(chains) >= (LONG_CONTEXT_CHAINS if name == "long_context" else w.batch * w.nheads)
    ey, ef = compare_chains(inp, y, fs, chains)
    tol = TOL[w.io_dtype]
    assert ey <= tol and ef <= tol, f"{name}, {len(chains)} chains: y {ey:.3e} final {ef:.3e} (tol {tol})"
