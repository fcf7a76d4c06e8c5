"""The five workloads at full size, through ssd_fwd exactly as bench.py calls
it, checked against the fp64 oracle on whole (batch, head) chains: all chains
for the small workloads, a seeded sample (including the first and last chain)
for the large ones."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gpu_util import TOL, check_sampled, oracle_full, sampled_chains, to_device
from forms import rel_err
from mamba_ssd_chunked_gb300.inputs import WORKLOADS, workload_inputs

pytestmark = pytest.mark.gpu

SAMPLE = {"tiny_fp32": None, "mamba2_130m_layer": 12, "mamba2_2p7b_layer": 12, "grouped_ragged": 10,
          "long_context": 4}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_gb300 import build
    build.build()


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
    elif w.dstate == 128 and (w.nheads // w.ngroups) % 2 == 0:
        expect_path = "chain"
    else:
        expect_path = "tc"
    assert pkg.ssd_select_path(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.io_dtype,
                               w.chunk_len) == expect_path
    if SAMPLE[name] is None:
        y_ref, f_ref = oracle_full(inp)
        assert rel_err(y.float().cpu().numpy(), y_ref) <= TOL[w.io_dtype]
        assert rel_err(fs.cpu().numpy(), f_ref) <= TOL[w.io_dtype]
    else:
        chains = sampled_chains(w.batch, w.nheads, SAMPLE[name], seed=w.seed)
        check_sampled(inp, y, fs, chains, w.io_dtype)
    assert torch.isfinite(y.float()).all() and torch.isfinite(fs).all()
