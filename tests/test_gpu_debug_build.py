"""The index-checked build (libssd_debug.so, SSD_DEBUG) on the GPU: the small,
odd-shaped parity cases of every tensor-core path, run through it once. In
that build every index the kernels compute by hand (ring, X/W and table slots,
tensor-memory columns, TMA coordinates, global state rows, job positions) is
checked before use; a failed check skips the access and makes
ssd_device_status return SSD_ERR_DEBUG_CHECK. This is the stand-in for a
memory checker. Each case must pass every check and still match the oracle.
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


@pytest.fixture(scope="module")
def debug_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mamba_ssd_chunked_gb300 as pkg
    from mamba_ssd_chunked_gb300 import build
    build.build()
    path = build.build(debug=True)
    old = pkg.use_library(path)
    try:
        assert pkg.library().ssd_debug_build() == 1
        yield pkg
    finally:
        pkg.use_library(old)


# (path, b, L, h, g, n, chunk, warm-up mode, dt shift, A scale, seq cuts[, headdim (64)])
CASES = [
    ("chain", 1, 1, 2, 1, 128, 256, 1, 0.0, 1.0, ()),          # a single token
    ("chain", 2, 127, 4, 2, 128, 128, 1, 0.0, 1.0, ()),        # one below a tile
    ("chain", 2, 300, 4, 2, 128, 256, 1, 0.0, 1.0, ()),        # ragged, several tiles
    ("chain", 1, 2000, 2, 1, 128, 256, 0, 0.0, 1.0, ()),       # a hand-off at every block
    ("chain", 1, 2000, 2, 1, 128, 256, 2, 2.0, 4.0, ()),       # warm-ups, split and extreme sub-blocks
    ("chain", 2, 1100, 8, 2, 128, 256, 1, 3.0, 4.0, ()),       # mostly extreme sub-blocks
    ("chain", 1, 1000, 6, 3, 256, 256, 1, 0.0, 1.0, ()),       # dstate 256
    ("chain", 1, 2000, 2, 1, 256, 256, 2, 1.0, 2.0, ()),       # dstate 256, warm-ups, splits
    ("chain", 1, 2600, 2, 1, 128, 256, 1, 0.0, 1.0, (300, 301, 1024)),  # packed sequences
    ("chain", 2, 700, 3, 3, 128, 256, 2, 1.0, 2.0, (), 128),   # headdim 128, warm-ups, splits
    ("chain", 1, 2000, 1, 1, 256, 256, 0, 0.0, 1.0, (), 128),  # headdim 128, dstate 256, hand-offs
    ("tc", 2, 300, 4, 2, 128, 256, 1, 0.0, 1.0, ()),
    ("tc", 1, 600, 8, 1, 256, 256, 1, 0.0, 1.0, ()),
    ("tc", 2, 700, 4, 2, 128, 128, 1, 1.0, 3.0, (1, 200, 513)),
]


@pytest.mark.parametrize("case", CASES)
def test_debug_build_checks_pass_and_results_match(debug_lib, case):
    pkg = debug_lib
    path, b, L, h, g, n, Q, mode, dt_shift, A_scale, cuts = case[:11]
    p = case[11] if len(case) > 11 else 64
    inp = make_inputs(b, L, h, p, g, n, io_dtype="bf16", init="normal", seed=b + L + h + n)
    inp["dt"] = (inp["dt"] + dt_shift).astype(np.float32)
    inp["A"] = (inp["A"] * A_scale).astype(np.float32)
    ids = None
    if cuts:
        row = np.zeros(L, np.int32)
        for c in cuts:
            row[c:] += 1
        ids = np.stack([row] * b)
    t = to_device(inp, "bf16")
    old = os.environ.get("SSD_CHAIN_WARMUP")
    os.environ["SSD_CHAIN_WARMUP"] = str(mode)
    try:
        seq = None if ids is None else torch.from_numpy(ids).cuda()
        y, fs = pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                            chunk_len=Q, path=path, seq_idx=seq)
        line = pkg.library().ssd_debug_failed_line(torch.cuda.current_stream().cuda_stream)
        st = pkg.ssd_device_status()
    finally:
        if old is None:
            os.environ.pop("SSD_CHAIN_WARMUP", None)
        else:
            os.environ["SSD_CHAIN_WARMUP"] = old
    assert st == 0 and line == 0, f"status {st}, first failed check at line {line}"
    y_ref, f_ref = oracle.recurrence(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["D"],
                                     inp["init_state"], seq_idx=ids)
    assert rel_err(y.float().cpu().numpy(), y_ref) <= TOL["bf16"]
    assert rel_err(fs.cpu().numpy(), f_ref) <= TOL["bf16"]
