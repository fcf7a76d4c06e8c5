"""fp64 CPU oracle for the Mamba-2 SSD forward (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. It shares no code with the CUDA path: the
arithmetic lives in ``ssd_oracle.c`` (token-by-token recurrence, fp64), built
with the host C compiler into ``libssd_oracle.so`` beside it.

``step`` (one decode step on a carried state) is the recurrence over one
token with that state as the initial state. ``layer_ops`` holds the causal
conv1d + SiLU before the scan, its decode step, and the gated RMSNorm after
it (fp64 numpy).

Parity status: pinned. The recurrence is checked (tests/test_oracle_pins.py)
against a brute-force semiseparable-matrix product, an independent fp64
five-stage chunked form at several chunk lengths, closed forms, the
split-sequence and linearity invariants, and source-level mutants of this
file that each plant a plausible mistake.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "ssd_oracle.c")
LIBRARY = os.path.join(_HERE, "libssd_oracle.so")

_lib = None


def compile_oracle(source: str = SOURCE, output: str = LIBRARY, extra_flags: Sequence[str] = ()) -> str:
    """Compile the C oracle with strict IEEE fp64 semantics (no fast-math)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           "-ffp-contract=off", *extra_flags, source, "-o", output, "-lm"]
    subprocess.run(cmd, check=True)
    return output


def _load(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    f = lib.ssd_oracle_recurrence
    f.restype = ctypes.c_int
    i64, fp = ctypes.c_int64, ctypes.c_void_p
    f.argtypes = [i64] * 6 + [fp] * 8 + [i64, fp, fp, fp, fp, ctypes.c_int, ctypes.c_double, ctypes.c_double, fp]
    return lib


def library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the oracle library, compiling it first if it is missing or stale."""
    global _lib
    if path is not None:
        return _load(path)
    if _lib is None:
        if (not os.path.exists(LIBRARY)) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE):
            compile_oracle()
        _lib = _load(LIBRARY)
    return _lib


def _ptr(a: Optional[np.ndarray]) -> Optional[int]:
    return None if a is None else a.ctypes.data


def _f32(a: Optional[np.ndarray]) -> Optional[np.ndarray]:
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def recurrence(
    x: np.ndarray,
    dt: np.ndarray,
    dt_bias: np.ndarray,
    A: np.ndarray,
    B: np.ndarray,
    C: np.ndarray,
    D: Optional[np.ndarray] = None,
    init_state: Optional[np.ndarray] = None,
    chains: Optional[Sequence[Tuple[int, int]]] = None,
    nthreads: Optional[int] = None,
    want_y: bool = True,
    lib: Optional[ctypes.CDLL] = None,
    dt_limit: Tuple[float, float] = (0.0, float("inf")),
    seq_idx: Optional[np.ndarray] = None,
) -> Tuple[Optional[np.ndarray], np.ndarray]:
    """Run the fp64 recurrence.

    ``dt_limit`` = (lo, hi) clamps softplus(dt + dt_bias) like torch.clamp
    (fla "mamba2.py", the time_step_limit clamp; (0, inf) is no clamp).

    ``seq_idx`` [b, L] (int32) packs several sequences into a row: the state
    restarts from zero wherever seq_idx changes between consecutive tokens
    (fla "mamba2.py" passes seq_idx to the fused chunked scan; reading of the
    packed-sequence case).

    Shapes: x [b,L,h,p], dt [b,L,h] (raw), dt_bias [h], A [h], B/C [b,L,g,n],
    D [h] or None, init_state [b,h,p,n] or None.

    With ``chains=None`` every (b, h) chain is computed and the results are
    y [b,L,h,p] and final [b,h,p,n] (fp64). With a list of (b, h) pairs only
    those chains run, and the results are y [k,L,p] and final [k,p,n].
    """
    x, dt, dt_bias, A, B, C = (_f32(v) for v in (x, dt, dt_bias, A, B, C))
    D, init_state = _f32(D), _f32(init_state)
    b, L, h, p = x.shape
    if seq_idx is not None:
        seq_idx = np.ascontiguousarray(seq_idx, dtype=np.int32)
        if seq_idx.shape != (b, L):
            raise ValueError(f"seq_idx must be [{b}, {L}], got {seq_idx.shape}")
    g, n = B.shape[2], B.shape[3]
    full = chains is None
    if full:
        chains = [(bi, hi) for bi in range(b) for hi in range(h)]
    sel_b = np.ascontiguousarray([c[0] for c in chains], dtype=np.int64)
    sel_h = np.ascontiguousarray([c[1] for c in chains], dtype=np.int64)
    k = len(chains)
    y_sel = np.empty((k, L, p), dtype=np.float64) if want_y else None
    final_sel = np.empty((k, p, n), dtype=np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = (lib or library()).ssd_oracle_recurrence(
        b, L, h, p, g, n,
        _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state),
        k, _ptr(sel_b), _ptr(sel_h), _ptr(y_sel), _ptr(final_sel), int(nthreads),
        float(dt_limit[0]), float(dt_limit[1]), _ptr(seq_idx))
    if rc != 0:
        raise RuntimeError(f"ssd_oracle_recurrence failed with code {rc}")
    if not full:
        return y_sel, final_sel
    y = None
    if want_y:
        y = y_sel.reshape(b, h, L, p).transpose(0, 2, 1, 3).copy()
    return y, final_sel.reshape(b, h, p, n)


def step(
    x: np.ndarray,
    dt: np.ndarray,
    dt_bias: np.ndarray,
    A: np.ndarray,
    B: np.ndarray,
    C: np.ndarray,
    D: Optional[np.ndarray],
    state: np.ndarray,
    nthreads: Optional[int] = None,
    dt_limit: Tuple[float, float] = (0.0, float("inf")),
) -> Tuple[np.ndarray, np.ndarray]:
    """One decode step on a carried state: the recurrence over a single token
    with the state as its initial state (fla "mamba2.py", Mamba2.torch_forward,
    cached-decode branch, computes exactly this step).

    Shapes: x [b,h,p], dt [b,h] (raw), B/C [b,g,n], state [b,h,p,n]. Returns
    y [b,h,p] and the new state [b,h,p,n] (fp64).
    """
    b, h, p = x.shape
    y, final = recurrence(x[:, None], dt[:, None], dt_bias, A, B[:, None], C[:, None], D, state, nthreads=nthreads,
                          dt_limit=dt_limit)
    return y[:, 0], final


# The per-token operations before and after the scan (causal conv1d + SiLU,
# its decode step, the gated RMSNorm), in fp64 numpy.
from .layer_ops import conv1d_silu, conv1d_step, gated_rmsnorm, silu  # noqa: E402,F401
