"""GPU parity of packed sequences (seq_idx, ssd_fwd_ex) on every path against
the fp64 oracle.

Reading (fla "fla/layers/mamba2.py" passes seq_idx to the fused chunked scan):
wherever seq_idx changes between consecutive tokens of a row the state
restarts from zero; init_state is the state before the row's first token and
final_state the state after its last. The cases put boundaries at a block
start, inside blocks, several in one block, at token 1 and before the last
token (one-token sequences), let an id return to an earlier value, and check
that a constant seq_idx gives bit-identical results to none.
Tolerance: max|delta| / max|ref| <= 1e-4 (fp32 io) / 2e-2 (bf16 io) on y and
on the final state.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from forms import rel_err
from gpu_util import TOL, to_device
from mamba_ssd_chunked_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_gb300 import build
    build.build()


def ids_from_cuts(L, cuts):
    ids = np.zeros(L, np.int32)
    for c in sorted(cuts):
        ids[c:] += 1
    return ids


def run_case(inp, ids, io, chunk_len, path):
    import mamba_ssd_chunked_gb300 as pkg
    t = to_device(inp, io)
    seq = torch.from_numpy(np.ascontiguousarray(ids)).cuda()
    y, fs = pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                        chunk_len=chunk_len, path=path, seq_idx=seq)
    assert pkg.ssd_device_status() == 0
    y_ref, f_ref = oracle.recurrence(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["D"],
                                     inp["init_state"], seq_idx=ids)
    ey, ef = rel_err(y.float().cpu().numpy(), y_ref), rel_err(fs.cpu().numpy(), f_ref)
    assert ey <= TOL[io] and ef <= TOL[io], f"{path} {io}: y {ey:.3e} final {ef:.3e}"
    # the restarts matter: the oracle without them is far off
    y0, _ = oracle.recurrence(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["init_state"])
    assert rel_err(y0, y_ref) > 5 * TOL[io]
    return y, fs


# (path, io, chunk_len, b, L, h, p, g, n)
PATH_CASES = [
    ("chain", "bf16", 256, 2, 700, 4, 64, 2, 128),
    ("chain", "bf16", 128, 1, 1100, 6, 64, 1, 128),
    ("chain", "bf16", 256, 2, 900, 3, 128, 3, 128),     # headdim 128: a chain per head
    ("tc", "bf16", 256, 2, 700, 4, 64, 2, 128),
    ("tc", "bf16", 256, 1, 600, 8, 64, 1, 256),
    ("simt", "f32", 64, 2, 300, 3, 16, 1, 16),
    ("simt", "bf16", 100, 1, 450, 4, 32, 2, 64),
]


def row_ids(L, seed):
    """Packed rows: boundaries at a block start, mid-block, several in one block, at token 1 and
    before the last token, and (second row) ids that return to an earlier value."""
    cuts = {1, 128, 200, 205, 213, L // 2, L - 1}
    rng = np.random.Generator(np.random.PCG64(seed))
    cuts |= set(int(c) for c in rng.integers(2, L - 1, size=4))
    r0 = ids_from_cuts(L, [c for c in cuts if 0 < c < L])
    r1 = (np.arange(L) // 97 % 3).astype(np.int32)  # 0,1,2,0,1,2,... every 97 tokens
    return r0, r1


@pytest.mark.parametrize("case", PATH_CASES)
def test_packed_sequences_match_oracle(case):
    path, io, Q, b, L, h, p, g, n = case
    import mamba_ssd_chunked_gb300 as pkg
    if path != "simt":
        assert pkg.ssd_select_path(b, L, h, p, g, n, io, Q) in (path, "chain")
    inp = make_inputs(b, L, h, p, g, n, io_dtype=io, init="normal", seed=L + h + n)
    r0, r1 = row_ids(L, seed=L)
    ids = np.stack([r0, r1][:b]) if b > 1 else r0[None]
    run_case(inp, ids, io, Q, path)


@pytest.mark.parametrize("path,io,Q", [("chain", "bf16", 256), ("tc", "bf16", 256), ("simt", "f32", 64)])
def test_constant_seq_idx_is_bit_identical_to_none(path, io, Q):
    import mamba_ssd_chunked_gb300 as pkg
    inp = make_inputs(2, 500, 4, 64 if io == "bf16" else 16, 1, 128 if io == "bf16" else 16, io_dtype=io,
                      init="normal", seed=5)
    t = to_device(inp, io)
    args = (t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"])
    y0, f0 = pkg.ssd_fwd(*args, chunk_len=Q, path=path)
    seq = torch.full((2, 500), 3, dtype=torch.int32, device="cuda")
    y1, f1 = pkg.ssd_fwd(*args, chunk_len=Q, path=path, seq_idx=seq)
    assert pkg.ssd_device_status() == 0
    assert torch.equal(y0, y1) and torch.equal(f0, f1)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_chain_segments_with_packed_sequences(mode):
    """Chains spread over many CTAs, with the hand-off, the warm-up or both,
    across sequence boundaries (a warm-up horizon stops at a boundary)."""
    old = os.environ.get("SSD_CHAIN_WARMUP")
    os.environ["SSD_CHAIN_WARMUP"] = str(mode)
    try:
        inp = make_inputs(1, 2600, 2, 64, 1, 128, io_dtype="bf16", init="normal", seed=17)
        ids = ids_from_cuts(2600, [300, 301, 1024, 1500, 2599])[None]
        run_case(inp, ids, "bf16", 256, "chain")
    finally:
        if old is None:
            os.environ.pop("SSD_CHAIN_WARMUP", None)
        else:
            os.environ["SSD_CHAIN_WARMUP"] = old


def test_many_packed_sequences_at_scale():
    """A longer packed batch (2 rows of 8192 tokens, 16 heads in 2 groups, random
    sequence lengths from 1 to 1500 tokens), every chain compared."""
    b, L, h = 2, 8192, 16
    inp = make_inputs(b, L, h, 64, 2, 128, io_dtype="bf16", init="normal", seed=29)
    rng = np.random.Generator(np.random.PCG64(30))
    rows = []
    for _ in range(b):
        cuts, t = [], 0
        while True:
            t += int(rng.integers(1, 1500))
            if t >= L:
                break
            cuts.append(t)
        rows.append(ids_from_cuts(L, cuts))
    run_case(inp, np.stack(rows), "bf16", 256, "auto")
