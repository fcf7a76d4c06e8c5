"""Helpers for the GPU tests: move seeded inputs to the device, call the C ABI
binding, and compare with the fp64 oracle (max|delta| / max|ref|)."""
import numpy as np

import oracle
from forms import rel_err
from mamba_ssd_chunked_gb300.inputs import make_inputs

TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_device(inp, io, device="cuda"):
    import torch
    tdt = torch.bfloat16 if io == "bf16" else torch.float32
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
            continue
        t = torch.from_numpy(np.ascontiguousarray(v)).to(device)
        if k in ("x", "B", "C"):
            t = t.to(tdt)
        out[k] = t.contiguous()
    return out


def run_gpu(t, chunk_len, path="auto", return_final_state=True, **kw):
    import mamba_ssd_chunked_gb300 as pkg
    y, fs = pkg.ssd_fwd(t["x"], t["dt"], t["dt_bias"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                        chunk_len=chunk_len, path=path, return_final_state=return_final_state, **kw)
    st = pkg.ssd_device_status()
    assert st == 0, f"device status {st}"
    return y, fs


def oracle_full(inp, nthreads=None):
    return oracle.recurrence(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["D"],
                             inp["init_state"], nthreads=nthreads)


def check_against_oracle(shape, io, chunk_len, path, init="normal", with_D=True, seed=0, tol=None):
    b, L, h, p, g, n = shape
    inp = make_inputs(b, L, h, p, g, n, io_dtype=io, init=init, seed=seed, with_D=with_D)
    t = to_device(inp, io)
    y, fs = run_gpu(t, chunk_len, path)
    y_ref, f_ref = oracle_full(inp)
    tol = TOL[io] if tol is None else tol
    ey = rel_err(y.float().cpu().numpy(), y_ref)
    ef = rel_err(fs.cpu().numpy(), f_ref)
    assert ey <= tol and ef <= tol, f"{shape} {io} Q={chunk_len} {path}: y {ey:.3e} final {ef:.3e} (tol {tol})"
    return ey, ef


def sampled_chains(batch, nheads, k, seed=0):
    rng = np.random.Generator(np.random.PCG64(seed))
    chains = {(0, 0), (batch - 1, nheads - 1)}
    while len(chains) < min(k, batch * nheads):
        chains.add((int(rng.integers(batch)), int(rng.integers(nheads))))
    return sorted(chains)


def check_sampled(inp, y, fs, chains, io, nthreads=None):
    """Compare the GPU outputs with the oracle on a sample of (b, h) chains.

    The relative error of each output is taken over the sampled slices.
    """
    y_ref, f_ref = oracle.recurrence(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                                     inp["D"], inp["init_state"], chains=chains, nthreads=nthreads)
    yg = np.stack([y[bi, :, hi].float().cpu().numpy() for bi, hi in chains])
    fg = np.stack([fs[bi, hi].cpu().numpy() for bi, hi in chains])
    ey, ef = rel_err(yg, y_ref), rel_err(fg, f_ref)
    tol = TOL[io]
    assert ey <= tol and ef <= tol, f"sampled {len(chains)} chains: y {ey:.3e} final {ef:.3e} (tol {tol})"
    return ey, ef
