"""Pins of the oracle's packed-sequence input seq_idx (CPU only).

Reading (flash-linear-attention "fla/layers/mamba2.py" passes seq_idx to the
fused chunked scan and defines nothing more): tokens of one batch row whose
seq_idx differ belong to different sequences, so the state restarts from zero
wherever seq_idx changes between consecutive tokens; init_state is the state
before the row's first token and final_state the state after its last token.

Pinned by: separate oracle runs on every packed sub-sequence (the first with
the row's initial state, the others from zero), concatenated; the brute-force
semiseparable form with the same cut (tests/forms.py, independent code);
constant seq_idx changing nothing; and source mutants of the oracle that drop
or misplace the reset.
"""
import numpy as np
import pytest

import oracle
from forms import quadratic, rel_err
from mamba_ssd_chunked_gb300.inputs import make_inputs

TIGHT = 1e-12


def _run(inp, seq_idx=None, lib=None):
    return oracle.recurrence(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["D"],
                             inp["init_state"], seq_idx=seq_idx, lib=lib)


def _packed_ids(L, cuts):
    ids = np.zeros(L, np.int32)
    for c in cuts:
        ids[c:] += 1
    return ids


@pytest.mark.parametrize("cuts", [[1], [5], [3, 4, 9], [13], [2, 7, 8, 11]])
def test_seq_idx_equals_separate_runs_of_each_sequence(cuts):
    b, L, h, p, g, n = 2, 14, 4, 3, 2, 5
    inp = make_inputs(b, L, h, p, g, n, io_dtype="f32", init="normal", seed=61 + len(cuts))
    ids = np.stack([_packed_ids(L, cuts), _packed_ids(L, [c + 1 for c in cuts if c + 1 < L])])
    y, fs = _run(inp, ids)
    for bi in range(b):
        bounds = [0] + [t for t in range(1, L) if ids[bi, t] != ids[bi, t - 1]] + [L]
        for k in range(len(bounds) - 1):
            t0, t1 = bounds[k], bounds[k + 1]
            part = {key: (None if v is None else v) for key, v in inp.items()}
            for key in ("x", "dt", "B", "C"):
                part[key] = np.ascontiguousarray(inp[key][bi:bi + 1, t0:t1])
            part["init_state"] = (np.ascontiguousarray(inp["init_state"][bi:bi + 1]) if k == 0
                                  else np.zeros_like(inp["init_state"][bi:bi + 1]))
            yp, fp = _run(part)
            assert np.max(np.abs(y[bi, t0:t1] - yp[0])) <= TIGHT * max(1.0, np.max(np.abs(yp)))
            if k == len(bounds) - 2:
                assert np.max(np.abs(fs[bi] - fp[0])) <= TIGHT * max(1.0, np.max(np.abs(fp)))


@pytest.mark.parametrize("ids_row", [
    [0, 0, 0, 1, 1, 1, 1, 2, 2, 2, 2],   # three packed sequences
    [5, 5, 7, 7, 5, 5, 5, 9, 9, 9, 9],   # an id returns: a new sequence all the same
    [0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10],  # every token alone
    [3, 3, 3, 3, 3, 3, 3, 3, 3, 3, 4],   # a one-token sequence at the end
])
def test_seq_idx_matches_the_brute_force_form(ids_row):
    inp = make_inputs(2, 11, 4, 3, 2, 4, io_dtype="f32", init="normal", seed=71)
    ids = np.stack([np.array(ids_row, np.int32), np.array(ids_row[::-1], np.int32)])
    y, fs = _run(inp, ids)
    yq, fq = quadratic(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["D"],
                       inp["init_state"], seq_idx=ids)
    assert rel_err(y, yq) < TIGHT and rel_err(fs, fq) < TIGHT
    # the cut changes the result: without it the forms disagree
    y0, _ = _run(inp)
    assert rel_err(y0, yq) > 1e-3


def test_constant_seq_idx_changes_nothing():
    inp = make_inputs(2, 20, 3, 4, 1, 5, io_dtype="f32", init="normal", seed=72)
    y0, f0 = _run(inp)
    y1, f1 = _run(inp, np.full((2, 20), 7, np.int32))
    assert np.array_equal(y0, y1) and np.array_equal(f0, f1)


SEQ_MUTANTS = {
    "seq_reset_dropped": (
        "memset(s, 0, sizeof(double) * (size_t)(P * N)); /* a new sequence starts from zero */", ";"),
    "seq_reset_one_token_late": ("seq[t] != seq[t - 1]", "t > 1 && seq[t - 1] != seq[t - 2]"),
    "seq_reset_on_increase_only": ("seq[t] != seq[t - 1]", "seq[t] > seq[t - 1]"),
}


@pytest.mark.parametrize("name", sorted(SEQ_MUTANTS))
def test_seq_idx_pins_reject_planted_mistake(name, tmp_path):
    old, new = SEQ_MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation target for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    so = oracle.compile_oracle(str(mutated), str(tmp_path / "mutant.so"))
    inp = make_inputs(2, 11, 4, 3, 2, 4, io_dtype="f32", init="normal", seed=73)
    ids = np.stack([np.array([5, 5, 7, 7, 5, 5, 5, 9, 9, 9, 9], np.int32),
                    np.array([0, 0, 0, 1, 1, 1, 1, 2, 2, 2, 2], np.int32)])
    y, fs = _run(inp, ids, lib=oracle.library(so))
    yq, fq = quadratic(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["D"],
                       inp["init_state"], seq_idx=ids)
    assert rel_err(y, yq) > 1e-6 or rel_err(fs, fq) > 1e-6, f"pins missed mutant {name}"
