"""The seeded input generator: determinism, shapes, dtypes and distributions."""
import numpy as np
import pytest

from mamba_ssd_chunked_gb300.inputs import WORKLOADS, make_inputs, round_to_bf16


def test_same_seed_same_inputs():
    a = make_inputs(2, 33, 4, 8, 2, 16, io_dtype="bf16", init="normal", seed=5)
    b = make_inputs(2, 33, 4, 8, 2, 16, io_dtype="bf16", init="normal", seed=5)
    for k in a:
        assert (a[k] is None and b[k] is None) or np.array_equal(a[k], b[k])


def test_shapes_and_optional_tensors():
    i = make_inputs(3, 10, 6, 4, 3, 5, io_dtype="f32", init="zero", seed=1, with_D=False)
    assert i["x"].shape == (3, 10, 6, 4) and i["dt"].shape == (3, 10, 6)
    assert i["B"].shape == (3, 10, 3, 5) and i["C"].shape == (3, 10, 3, 5)
    assert i["D"] is None and i["init_state"] is None
    for k in ("x", "dt", "dt_bias", "A", "B", "C"):
        assert i[k].dtype == np.float32 and i[k].flags["C_CONTIGUOUS"]


def test_bf16_rounding_is_exact_and_nearest_even():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38, 1e-40], np.float32)
    r = round_to_bf16(v)
    assert np.array_equal(r, round_to_bf16(r))                    # idempotent
    assert r[1] == 1.0 and r[2] == 1.0 + 2 ** -6                   # ties to even
    assert np.all((r.view(np.uint32) & 0xFFFF) == 0)
    i = make_inputs(1, 64, 2, 8, 1, 8, io_dtype="bf16", seed=3)
    for k in ("x", "B", "C"):
        assert np.all((i[k].view(np.uint32) & 0xFFFF) == 0)


def test_parameter_distributions_follow_the_recipe():
    i = make_inputs(1, 4, 4096, 1, 1, 1, seed=2)
    assert np.all(i["A"] < 0) and np.all(i["A"] >= -16.0001) and np.all(i["A"] <= -0.9999)
    # softplus(dt_bias) lands in [1e-3, 1e-1]
    sp = np.log1p(np.exp(i["dt_bias"].astype(np.float64)))
    assert sp.min() >= 1e-3 * (1 - 1e-5) and sp.max() <= 1e-1 * (1 + 1e-5)
    assert abs(float(np.mean(np.log(sp))) - 0.5 * (np.log(1e-3) + np.log(1e-1))) < 0.1


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_workloads_are_well_formed(name):
    w = WORKLOADS[name]
    assert w.nheads % w.ngroups == 0
    assert w.io_dtype in ("f32", "bf16")
    assert w.chunk_len in (64, 128, 256)
