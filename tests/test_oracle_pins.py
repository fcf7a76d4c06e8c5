"""Pins for the fp64 oracle: checks against things other than itself.

Each check ties the C recurrence (oracle/ssd_oracle.c) to the mathematics the
pages fix: a hand-worked example, the brute-force semiseparable form, the
five-stage chunked form at many chunk lengths (chunk length 1 is the
recurrence itself and chunk length L is the quadratic form), closed forms,
the split-sequence invariant (the final state carried into the next call, as
the Mamba2Cache ssm_states hand-off does), linearity, the group expansion and
source-level mutants that each plant a plausible mistake and must be caught.
"""
import json
import math
import os
import numpy as np
import pytest

import oracle
from forms import chunked, quadratic, rel_err, softplus
from mamba_ssd_chunked_gb300.inputs import make_inputs

HERE = os.path.dirname(os.path.abspath(__file__))
TIGHT = 1e-12


def _run(inp, **kw):
    return oracle.recurrence(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                             inp["D"], inp["init_state"], **kw)


def _forms_args(inp):
    return (inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["D"], inp["init_state"])


SMALL_SHAPES = [
    # batch, seqlen, nheads, headdim, ngroups, dstate, io, init
    (1, 1, 1, 1, 1, 1, "f32", "zero"),
    (1, 9, 2, 3, 1, 4, "f32", "normal"),
    (2, 13, 4, 5, 2, 3, "bf16", "normal"),
    (1, 16, 6, 2, 3, 5, "f32", "zero"),
    (2, 7, 4, 4, 4, 2, "f32", "normal"),
]


def test_worked_example_from_golden():
    g = json.load(open(os.path.join(HERE, "golden", "worked_example.json")))
    i = {k: np.asarray(v, np.float32) for k, v in g["inputs"].items()}
    y, fs = oracle.recurrence(i["x"], i["dt"], i["dt_bias"], i["A"], i["B"], i["C"], i["D"], None)
    np.testing.assert_allclose(y, np.asarray(g["expected"]["y"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(fs, np.asarray(g["expected"]["final_state"]), rtol=0, atol=1e-15)


@pytest.mark.parametrize("shape", SMALL_SHAPES)
def test_matches_quadratic_form(shape):
    b, L, h, p, g, n, io, init = shape
    inp = make_inputs(b, L, h, p, g, n, io_dtype=io, init=init, seed=11 + L)
    y, fs = _run(inp)
    yq, fq = quadratic(*_forms_args(inp))
    assert rel_err(y, yq) < TIGHT
    assert rel_err(fs, fq) < TIGHT


@pytest.mark.parametrize("Q", [1, 2, 7, 16, 64, 50])
@pytest.mark.parametrize("L", [50, 64])
def test_matches_chunked_form_any_chunk_length(Q, L):
    inp = make_inputs(2, L, 4, 3, 2, 5, io_dtype="bf16", init="normal", seed=3 * L + Q)
    y, fs = _run(inp)
    yc, fc = chunked(*_forms_args(inp), chunk_len=Q)
    assert rel_err(y, yc) < TIGHT
    assert rel_err(fs, fc) < TIGHT


def test_chunked_form_spanning_whole_sequence_is_quadratic_form():
    inp = make_inputs(1, 11, 2, 2, 1, 3, io_dtype="f32", init="normal", seed=5)
    yc, fc = chunked(*_forms_args(inp), chunk_len=11)
    yq, fq = quadratic(*_forms_args(inp))
    assert rel_err(yc, yq) < TIGHT and rel_err(fc, fq) < TIGHT


@pytest.mark.parametrize("split", [1, 37, 64, 100, 127])
def test_split_sequence_reproduces_unsplit_run(split):
    L = 128
    inp = make_inputs(2, L, 4, 8, 2, 16, io_dtype="bf16", init="normal", seed=77)
    y, fs = _run(inp)
    first = {k: (v[:, :split] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    second = {k: (v[:, split:] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    y1, f1 = _run(first)
    second["init_state"] = f1.astype(np.float32)
    # carry the fp64 state exactly: rerun the tail from the fp64 state by
    # linearity (tail(s) = tail(s32) + tail_from_state(s - s32))
    y2, f2 = _run(second)
    resid = {**second, "x": np.zeros_like(second["x"]), "D": None,
             "init_state": (f1 - f1.astype(np.float32).astype(np.float64)).astype(np.float32)}
    y2r, f2r = _run(resid)
    y_cat = np.concatenate([y1, y2 + y2r], axis=1)
    assert rel_err(y_cat, y) < 1e-9
    assert rel_err(f2 + f2r, fs) < 1e-9


def test_single_token_closed_form():
    inp = make_inputs(2, 1, 3, 4, 1, 5, io_dtype="f32", init="normal", seed=9)
    y, fs = _run(inp)
    for bi in range(2):
        for hi in range(3):
            d = float(softplus(float(inp["dt"][bi, 0, hi]) + float(inp["dt_bias"][hi])))
            a = math.exp(d * float(inp["A"][hi]))
            x = inp["x"][bi, 0, hi].astype(np.float64)
            Bv = inp["B"][bi, 0, 0].astype(np.float64)
            Cv = inp["C"][bi, 0, 0].astype(np.float64)
            s = a * inp["init_state"][bi, hi].astype(np.float64) + d * np.outer(x, Bv)
            np.testing.assert_allclose(fs[bi, hi], s, rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(y[bi, 0, hi], s @ Cv + float(inp["D"][hi]) * x, rtol=1e-12, atol=1e-14)


def test_zero_B_leaves_only_decayed_initial_state():
    inp = make_inputs(1, 40, 2, 3, 1, 4, io_dtype="f32", init="normal", seed=21)
    inp["B"] = np.zeros_like(inp["B"])
    y, fs = _run(inp)
    delta = softplus(inp["dt"].astype(np.float64) + inp["dt_bias"][None, None, :])
    for hi in range(2):
        cum = np.cumsum(delta[0, :, hi]) * float(inp["A"][hi])
        s0 = inp["init_state"][0, hi].astype(np.float64)
        expect = np.exp(cum)[:, None] * (inp["C"][0, :, 0].astype(np.float64) @ s0.T) \
            + float(inp["D"][hi]) * inp["x"][0, :, hi].astype(np.float64)
        np.testing.assert_allclose(y[0, :, hi], expect, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(fs[0, hi], math.exp(cum[-1]) * s0, rtol=1e-11, atol=1e-300)


def test_constant_step_geometric_sum():
    # p = n = 1, B = C = x = 1, constant delta: s_t = a^(t+1) s0 + delta (1 - a^(t+1)) / (1 - a)
    L = 30
    dt_raw = 0.3
    x = np.ones((1, L, 1, 1), np.float32)
    ones = np.ones((1, L, 1, 1), np.float32)
    dt = np.full((1, L, 1), dt_raw, np.float32)
    bias = np.zeros(1, np.float32)
    A = np.array([-0.7], np.float32)
    s0 = np.array([[[[2.0]]]], np.float32)
    y, fs = oracle.recurrence(x, dt, bias, A, ones, ones, None, s0)
    d = float(softplus(np.float64(np.float32(dt_raw))))
    a = math.exp(d * float(np.float32(-0.7)))
    t = np.arange(L, dtype=np.float64)
    expect = a ** (t + 1) * 2.0 + d * (1 - a ** (t + 1)) / (1 - a)
    np.testing.assert_allclose(y[0, :, 0, 0], expect, rtol=1e-13)
    np.testing.assert_allclose(fs[0, 0, 0, 0], expect[-1], rtol=1e-13)


def test_vanishing_decay_is_a_prefix_sum():
    inp = make_inputs(1, 25, 2, 3, 1, 4, io_dtype="f32", init="normal", seed=4)
    inp["A"] = np.full(2, -1e-30, np.float32)
    y, fs = _run(inp)
    delta = softplus(inp["dt"].astype(np.float64) + inp["dt_bias"][None, None, :])
    for hi in range(2):
        x = inp["x"][0, :, hi].astype(np.float64)
        Bv = inp["B"][0, :, 0].astype(np.float64)
        outer = delta[0, :, hi][:, None, None] * x[:, :, None] * Bv[:, None, :]
        s = np.cumsum(outer, axis=0) + inp["init_state"][0, hi].astype(np.float64)[None]
        expect = np.einsum("tpn,tn->tp", s, inp["C"][0, :, 0].astype(np.float64)) + float(inp["D"][hi]) * x
        np.testing.assert_allclose(y[0, :, hi], expect, rtol=1e-10, atol=1e-12)


def test_linear_in_x_and_initial_state_jointly():
    a = make_inputs(1, 33, 3, 4, 1, 6, io_dtype="f32", init="normal", seed=1)
    b = make_inputs(1, 33, 3, 4, 1, 6, io_dtype="f32", init="normal", seed=2)
    # round x and the initial state to multiples of 1/16 so that the fp32
    # mixture below is exact
    for i in (a, b):
        for k in ("x", "init_state"):
            i[k] = (np.round(i[k] * 16.0) / 16.0).astype(np.float32)
    mix = dict(a)
    mix["x"] = (2.0 * a["x"] - 0.5 * b["x"]).astype(np.float32)
    mix["init_state"] = (2.0 * a["init_state"] - 0.5 * b["init_state"]).astype(np.float32)
    b_same = dict(a, x=b["x"], init_state=b["init_state"])
    ya, fa = _run(a)
    yb, fb = _run(b_same)
    ym, fm = _run(mix)
    # x, init combine exactly in fp32 here (scale by powers of two), so the
    # mixed run is an exact linear combination up to fp64 rounding
    assert rel_err(ym, 2.0 * ya - 0.5 * yb) < 1e-12
    assert rel_err(fm, 2.0 * fa - 0.5 * fb) < 1e-12


def test_group_expansion_equals_per_head_B_C():
    inp = make_inputs(2, 21, 6, 3, 2, 4, io_dtype="f32", init="normal", seed=8)
    y, fs = _run(inp)
    rep = dict(inp)
    rep["B"] = np.ascontiguousarray(np.repeat(inp["B"], 3, axis=2))
    rep["C"] = np.ascontiguousarray(np.repeat(inp["C"], 3, axis=2))
    y2, f2 = _run(rep)
    assert np.array_equal(y, y2) and np.array_equal(fs, f2)


def test_selected_chains_match_full_run():
    inp = make_inputs(2, 17, 5, 3, 1, 4, io_dtype="bf16", init="normal", seed=6)
    y, fs = _run(inp)
    sel = [(1, 4), (0, 0), (1, 2)]
    ys, fss = _run(inp, chains=sel)
    for k, (bi, hi) in enumerate(sel):
        assert np.array_equal(ys[k], y[bi, :, hi])
        assert np.array_equal(fss[k], fs[bi, hi])


def test_thread_count_does_not_change_results():
    inp = make_inputs(2, 40, 6, 4, 2, 8, io_dtype="bf16", init="normal", seed=12)
    y1, f1 = _run(inp, nthreads=1)
    y4, f4 = _run(inp, nthreads=4)
    assert np.array_equal(y1, y4) and np.array_equal(f1, f4)


# ---------------------------------------------------------------------------
# Mutants: each replaces one statement of the oracle's source with a plausible
# mistake; the pins above must reject every one of them.
MUTANTS = {
    "readout_before_update": (
        "sp[n] = decay * sp[n] + u * (double)Bt[n];\n                acc += sp[n] * (double)Ct[n];",
        "acc += sp[n] * (double)Ct[n];\n                sp[n] = decay * sp[n] + u * (double)Bt[n];"),
    "dropped_D_skip": ("acc + d_h * xp", "acc"),
    "wrong_group_index": ("const int64_t g = h / (H / G);", "const int64_t g = h % G;"),
    "B_in_readout": ("acc += sp[n] * (double)Ct[n];", "acc += sp[n] * (double)Bt[n];"),
    "decay_sign": ("exp(delta * a_h)", "exp(-delta * a_h)"),
    "no_delta_on_input": ("const double u = delta * xp;", "const double u = xp;"),
    "bias_dropped": ("+ bias_h)", ")"),
    "softplus_branch": ("? v + log1p(exp(-v))", "? log1p(exp(-v))"),
    "x_token_head_transposed": ("j->x + ((b * L + t) * H + h) * P", "j->x + ((b * H + h) * L + t) * P"),
    "init_ignored": ("s[i] = (double)s0[i];", "s[i] = 0.0 * s0[i];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation target for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    so = oracle.compile_oracle(str(mutated), str(tmp_path / "mutant.so"))
    lib = oracle.library(so)
    inp = make_inputs(2, 12, 4, 3, 2, 5, io_dtype="f32", init="normal", seed=31)
    # a softplus argument above zero is needed to reach the v > 0 branch
    inp["dt"] = (inp["dt"] + 2.5).astype(np.float32)
    y, fs = _run(inp, lib=lib)
    yq, fq = quadratic(*_forms_args(inp))
    assert rel_err(y, yq) > 1e-6 or rel_err(fs, fq) > 1e-6, f"pins missed mutant {name}"


def test_unmutated_source_passes_the_mutant_harness(tmp_path):
    so = oracle.compile_oracle(oracle.SOURCE, str(tmp_path / "same.so"))
    inp = make_inputs(2, 12, 4, 3, 2, 5, io_dtype="f32", init="normal", seed=31)
    inp["dt"] = (inp["dt"] + 2.5).astype(np.float32)
    y, fs = _run(inp, lib=oracle.library(so))
    yq, fq = quadratic(*_forms_args(inp))
    assert rel_err(y, yq) < TIGHT and rel_err(fs, fq) < TIGHT


def test_invalid_arguments_are_rejected():
    inp = make_inputs(1, 4, 3, 2, 1, 2, seed=0)
    bad = dict(inp)
    bad["B"] = np.zeros((1, 4, 2, 2), np.float32)  # 3 heads, 2 groups
    with pytest.raises(RuntimeError):
        _run(bad)


def test_decode_step_matches_its_closed_form():
    """oracle.step against the single-token update written out with numpy:
    s' = e^{dA} s + d x B^T, y = s' C + D x (d = softplus(dt + dt_bias))."""
    rng = np.random.Generator(np.random.PCG64(77))
    b, h, p, g, n = 2, 6, 5, 3, 7
    x = rng.standard_normal((b, h, p)).astype(np.float32)
    dt = rng.standard_normal((b, h)).astype(np.float32)
    dt_bias = rng.standard_normal(h).astype(np.float32)
    A = -np.exp(rng.uniform(0, 2, h)).astype(np.float32)
    B = rng.standard_normal((b, g, n)).astype(np.float32)
    C = rng.standard_normal((b, g, n)).astype(np.float32)
    D = rng.standard_normal(h).astype(np.float32)
    s0 = rng.standard_normal((b, h, p, n)).astype(np.float32)
    y, s1 = oracle.step(x, dt, dt_bias, A, B, C, D, s0)
    hg = np.arange(h) // (h // g)
    d = np.log1p(np.exp(dt.astype(np.float64) + dt_bias))
    decay = np.exp(d * A)[..., None, None]
    Bh = B.astype(np.float64)[:, hg]             # [b,h,n]
    Ch = C.astype(np.float64)[:, hg]
    s_ref = decay * s0 + (d[..., None] * x)[..., None] * Bh[:, :, None, :]
    y_ref = np.einsum("bhpn,bhn->bhp", s_ref, Ch) + D.astype(np.float64)[None, :, None] * x.astype(np.float64)
    assert np.max(np.abs(s1 - s_ref)) < 1e-12 * max(1.0, np.max(np.abs(s_ref)))
    assert np.max(np.abs(y - y_ref)) < 1e-12 * max(1.0, np.max(np.abs(y_ref)))


def test_decode_step_special_cases():
    """Two reductions of the single-token update (fla Mamba2.torch_forward,
    cached-decode branch): from a zero state the new state is the outer
    product d x B^T, so y = x (d <B, C> + D) per row; with x = 0 the state
    only decays, s' = e^{d A} s, and y = s' C. A dropped decay, a transposed
    outer product or a wrong group map fails one of them."""
    rng = np.random.Generator(np.random.PCG64(78))
    b, h, p, g, n = 3, 4, 6, 2, 9
    x = rng.standard_normal((b, h, p)).astype(np.float32)
    dt = rng.standard_normal((b, h)).astype(np.float32)
    dt_bias = rng.standard_normal(h).astype(np.float32)
    A = -np.exp(rng.uniform(0, 2, h)).astype(np.float32)
    B = rng.standard_normal((b, g, n)).astype(np.float32)
    C = rng.standard_normal((b, g, n)).astype(np.float32)
    D = rng.standard_normal(h).astype(np.float32)
    d = np.log1p(np.exp(dt.astype(np.float64) + dt_bias))       # [b, h]
    # zero state: y[b,h,p] = x (d <B_g, C_g> + D_h), g = h // (h / g)
    y, s1 = oracle.step(x, dt, dt_bias, A, B, C, D, np.zeros((b, h, p, n), np.float32))
    for bi in range(b):
        for hi in range(h):
            gi = hi // (h // g)
            bc = float(np.dot(B[bi, gi].astype(np.float64), C[bi, gi].astype(np.float64)))
            want = x[bi, hi].astype(np.float64) * (d[bi, hi] * bc + float(D[hi]))
            assert np.allclose(y[bi, hi], want, rtol=1e-12, atol=1e-12)
            assert np.allclose(s1[bi, hi], d[bi, hi] * np.outer(x[bi, hi].astype(np.float64), B[bi, gi].astype(np.float64)), rtol=1e-12, atol=1e-12)
    # x = 0: pure decay of the carried state
    s0 = rng.standard_normal((b, h, p, n)).astype(np.float32)
    y, s1 = oracle.step(np.zeros_like(x), dt, dt_bias, A, B, C, D, s0)
    for bi in range(b):
        for hi in range(h):
            gi = hi // (h // g)
            decayed = np.exp(d[bi, hi] * float(A[hi])) * s0[bi, hi].astype(np.float64)
            assert np.allclose(s1[bi, hi], decayed, rtol=1e-12, atol=1e-300)
            assert np.allclose(y[bi, hi], decayed @ C[bi, gi].astype(np.float64), rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------------------------- conv1d + SiLU, gated RMSNorm
def _silu_lib(v):
    """SiLU through scipy's logistic function (independent of the oracle's formula)."""
    from scipy.special import expit
    return v * expit(v)


def test_conv1d_matches_numpy_convolve():
    """The causal depthwise conv (fla Mamba2.__init__, nn.Conv1d with groups = conv_dim and
    padding K - 1, cropped to seq_len) equals numpy's full convolution of each channel with the
    reversed taps, first seq_len outputs; then bias and SiLU."""
    rng = np.random.Generator(np.random.PCG64(91))
    b, L, d_inner, gn, K = 2, 37, 12, 4, 4
    cd = d_inner + 2 * gn
    xbc = rng.standard_normal((b, L, cd))
    w = rng.standard_normal((cd, K))
    bias = rng.standard_normal(cd)
    x, Bo, Co, state = oracle.conv1d_silu(xbc, w, bias, d_inner, gn)
    full = np.concatenate([x, Bo, Co], axis=-1)
    for bi in range(b):
        for c in range(cd):
            pre = np.convolve(xbc[bi, :, c], w[c, ::-1])[:L] + bias[c]
            assert np.allclose(full[bi, :, c], _silu_lib(pre), rtol=1e-12, atol=1e-12)
    # the conv state is the last K inputs, channel-major
    assert np.array_equal(state, xbc[:, L - K:, :].transpose(0, 2, 1))


def test_conv1d_single_taps_and_short_sequences():
    """Only the last tap set: out = silu(x + bias) (no shift); only the first tap: the input delayed
    by K - 1 steps with zeros before the sequence; seq_len < K pads the conv state with zeros."""
    rng = np.random.Generator(np.random.PCG64(92))
    b, L, d_inner, gn, K = 1, 9, 4, 2, 4
    cd = d_inner + 2 * gn
    xbc = rng.standard_normal((b, L, cd))
    last = np.zeros((cd, K)); last[:, K - 1] = 1.0
    x, Bo, Co, _ = oracle.conv1d_silu(xbc, last, None, d_inner, gn)
    assert np.allclose(np.concatenate([x, Bo, Co], -1), _silu_lib(xbc), rtol=1e-13, atol=1e-15)
    first = np.zeros((cd, K)); first[:, 0] = 1.0
    x, Bo, Co, _ = oracle.conv1d_silu(xbc, first, None, d_inner, gn, activation=False)
    got = np.concatenate([x, Bo, Co], -1)
    assert np.array_equal(got[:, :K - 1], np.zeros((b, K - 1, cd)))
    assert np.array_equal(got[:, K - 1:], xbc[:, :L - K + 1])
    short = xbc[:, :2]
    _, _, _, st = oracle.conv1d_silu(short, last, None, d_inner, gn)
    assert np.array_equal(st[:, :, :K - 2], np.zeros((b, cd, K - 2)))
    assert np.array_equal(st[:, :, K - 2:], short.transpose(0, 2, 1))


def test_conv1d_decode_steps_reproduce_the_prefill():
    """The cached-decode branch (roll the conv state, append the token, dot with the taps), run
    token by token from a zero state, gives the prefill's outputs and its final conv state."""
    rng = np.random.Generator(np.random.PCG64(93))
    b, L, d_inner, gn, K = 2, 11, 6, 2, 4
    cd = d_inner + 2 * gn
    xbc = rng.standard_normal((b, L, cd))
    w = rng.standard_normal((cd, K))
    bias = rng.standard_normal(cd)
    x, Bo, Co, st = oracle.conv1d_silu(xbc, w, bias, d_inner, gn)
    state = np.zeros((b, cd, K))
    for t in range(L):
        xs, bs, cs, state = oracle.conv1d_step(xbc[:, t], state, w, bias, d_inner, gn)
        assert np.allclose(xs, x[:, t], rtol=1e-12, atol=1e-13)
        assert np.allclose(bs, Bo[:, t], rtol=1e-12, atol=1e-13)
        assert np.allclose(cs, Co[:, t], rtol=1e-12, atol=1e-13)
    assert np.array_equal(state, st)


def test_gated_rmsnorm_against_torch_rms_norm_and_closed_forms():
    """norm_before_gate=False: out = rms_norm(y * silu(z)) * w. Checked against torch's fp64
    rms_norm of the gated product, a constant row (c / sqrt(c^2 + eps)), a zero gate (output 0),
    and groups (each group normalised on its own)."""
    import torch
    rng = np.random.Generator(np.random.PCG64(94))
    rows, d, eps = 7, 48, 1e-5
    y = rng.standard_normal((rows, d))
    z = rng.standard_normal((rows, d))
    w = rng.standard_normal(d)
    got = oracle.gated_rmsnorm(y, z, w, eps)
    v = torch.from_numpy(y) * torch.nn.functional.silu(torch.from_numpy(z))
    ref = torch.nn.functional.rms_norm(v, (d,), torch.from_numpy(w), eps).numpy()
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)
    const = np.full((1, d), 0.3)
    out = oracle.gated_rmsnorm(const, None, np.ones(d), eps)
    assert np.allclose(out, 0.3 / np.sqrt(0.09 + eps), rtol=1e-14)
    assert np.array_equal(oracle.gated_rmsnorm(y, np.zeros_like(z), w, eps), np.zeros_like(y))
    gs = 16
    grouped = oracle.gated_rmsnorm(y, z, w, eps, group_size=gs)
    for gi in range(d // gs):
        sl = slice(gi * gs, (gi + 1) * gs)
        ref_g = torch.nn.functional.rms_norm(v[:, sl], (gs,), torch.from_numpy(w[sl]), eps).numpy()
        assert np.allclose(grouped[:, sl], ref_g, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------- dt_limit
def _inverse_softplus64(v):
    return v + np.log(-np.expm1(-v))


def test_dt_limit_equals_a_shifted_raw_dt():
    """clamp(softplus(dt + bias), lo, hi) (fla Mamba2.torch_forward, time_step_limit) is the same
    discretisation as an unclamped run on the raw dt that softplus maps onto the clamped value, so
    the clamped oracle must match the unclamped oracle on that raw dt (up to its fp32 rounding)."""
    inp = make_inputs(2, 40, 4, 3, 2, 5, io_dtype="f32", init="normal", seed=41)
    lo, hi = 0.02, 0.3
    y, fs = _run(inp, dt_limit=(lo, hi))
    delta = softplus(inp["dt"].astype(np.float64) + inp["dt_bias"].astype(np.float64))
    assert (delta < lo).any() and (delta > hi).any(), "the draw must hit both bounds"
    raw = (_inverse_softplus64(np.clip(delta, lo, hi)) - inp["dt_bias"].astype(np.float64)).astype(np.float32)
    shifted = dict(inp, dt=raw)
    y2, f2 = _run(shifted)
    assert rel_err(y, y2) < 1e-5 and rel_err(fs, f2) < 1e-5
    # and the brute-force form with the clip agrees to fp64 rounding
    yq, fq = quadratic(*_forms_args(inp), dt_limit=(lo, hi))
    assert rel_err(y, yq) < TIGHT and rel_err(fs, fq) < TIGHT


def test_default_dt_limit_is_no_clamp_and_a_point_limit_is_constant_dt():
    """(0, inf) leaves every result bit-identical; lo == hi == c makes every step dt = c, which
    the brute-force form reproduces with a constant delta."""
    inp = make_inputs(1, 17, 3, 2, 1, 4, io_dtype="f32", init="normal", seed=42)
    y0, f0 = _run(inp)
    y1, f1 = _run(inp, dt_limit=(0.0, float("inf")))
    assert np.array_equal(y0, y1) and np.array_equal(f0, f1)
    c = 0.05
    y, fs = _run(inp, dt_limit=(c, c))
    raw = np.full_like(inp["dt"], 0.0)
    bias = _inverse_softplus64(np.full(3, c)).astype(np.float64)
    yq, fq = quadratic(inp["x"], raw, bias, inp["A"], inp["B"], inp["C"], inp["D"], inp["init_state"])
    assert rel_err(y, yq) < 1e-12 and rel_err(fs, fq) < 1e-12


CLAMP_MUTANTS = {
    "clamp_lower_dropped": ("if (delta < j->dt_min) delta = j->dt_min;", ""),
    "clamp_upper_dropped": ("if (delta > j->dt_max) delta = j->dt_max;", ""),
    "clamp_before_softplus": (
        "double delta = softplus((double)j->dt[(b * L + t) * H + h] + bias_h);\n"
        "        if (delta < j->dt_min) delta = j->dt_min;\n"
        "        if (delta > j->dt_max) delta = j->dt_max;",
        "double delta = (double)j->dt[(b * L + t) * H + h] + bias_h;\n"
        "        if (delta < j->dt_min) delta = j->dt_min;\n"
        "        if (delta > j->dt_max) delta = j->dt_max;\n"
        "        delta = softplus(delta);"),
}


@pytest.mark.parametrize("name", sorted(CLAMP_MUTANTS))
def test_dt_limit_pins_reject_planted_mistake(name, tmp_path):
    old, new = CLAMP_MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation target for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    so = oracle.compile_oracle(str(mutated), str(tmp_path / "mutant.so"))
    inp = make_inputs(2, 12, 4, 3, 2, 5, io_dtype="f32", init="normal", seed=43)
    y, fs = _run(inp, lib=oracle.library(so), dt_limit=(0.02, 0.3))
    yq, fq = quadratic(*_forms_args(inp), dt_limit=(0.02, 0.3))
    assert rel_err(y, yq) > 1e-6 or rel_err(fs, fq) > 1e-6, f"pins missed mutant {name}"
