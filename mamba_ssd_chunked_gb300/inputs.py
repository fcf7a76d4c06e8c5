"""Seeded synthetic inputs for the Mamba-2 SSD chunked-scan forward.

This module is shared by the CUDA path's tests and benchmark and by the fp64
oracle's tests. It draws random numbers and rounds them to the storage dtype;
it holds none of the SSD arithmetic (no softplus, no decay, no scan).

Workloads are named by what they are. Shapes and distributions follow the
Mamba-2 layer configuration on the pages (flash-linear-attention
``fla/layers/mamba2.py``, ``Mamba2.__init__`` defaults: head_dim 64,
state_size 128, chunk_size 256) and the dt/A initialisation recipe of
``fla/models/mamba2/modeling_mamba2.py`` (``_init_weights``: dt drawn
log-uniform in [time_step_min, time_step_max] = [1e-3, 1e-1], stored through
the inverse of softplus as dt_bias).

Recipe (seed fixed per workload, one numpy PCG64 stream, tensors drawn in the
order x, dt_raw, dt_bias, A, B, C, D, init):
  x, B, C   ~ N(0, 1), rounded to bf16 for bf16 workloads (fp32 otherwise)
  dt_raw    ~ N(0, 1) fp32
  dt_bias   = inverse-softplus(exp(U[ln 1e-3, ln 1e-1])) fp32 (per head)
  A         = -exp(U[ln 1, ln 16]) fp32 (per head, strictly negative)
  D         ~ N(0, 1) fp32 (per head)
  init      = zeros, or ~ N(0, 0.1^2) fp32 [batch, nheads, headdim, dstate]
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    ngroups: int
    dstate: int
    chunk_len: int
    io_dtype: str          # "f32" or "bf16": dtype of x, B, C and y
    init: str              # "zero" or "normal"
    seed: int

    @property
    def d_inner(self) -> int:
        return self.nheads * self.headdim

    def as_dict(self) -> dict:
        return dataclasses.asdict(self)


# The five workloads, in order: the tiny fp32 parity case, the Mamba2-130M and
# Mamba2-2.7B layer shapes, grouped B/C with a ragged length, and long context.
WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_fp32", 1, 256, 4, 16, 1, 16, 64, "f32", "zero", 1234),
        Workload("mamba2_130m_layer", 8, 2048, 24, 64, 1, 128, 256, "bf16", "zero", 1235),
        Workload("mamba2_2p7b_layer", 4, 4096, 80, 64, 1, 128, 256, "bf16", "normal", 1236),
        Workload("grouped_ragged", 2, 16000, 128, 64, 8, 128, 256, "bf16", "normal", 1237),
        Workload("long_context", 1, 131072, 64, 64, 1, 256, 256, "bf16", "zero", 1238),
    ]
}

HEADLINE = "mamba2_2p7b_layer"


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returned as fp32.

    Storage-format conversion only: the result is exactly representable in
    bf16, so widening it back (on the GPU or in the oracle) is lossless.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (rounded.astype(np.uint32) << 16).view(np.float32).reshape(a.shape)


def _inverse_softplus(v: np.ndarray) -> np.ndarray:
    # Input recipe: dt_bias is stored so that softplus(dt_bias) = v.
    return v + np.log(-np.expm1(-v))


def make_inputs(
    batch: int,
    seqlen: int,
    nheads: int,
    headdim: int,
    ngroups: int,
    dstate: int,
    io_dtype: str = "bf16",
    init: str = "zero",
    seed: int = 0,
    with_D: bool = True,
) -> Dict[str, Optional[np.ndarray]]:
    """Draw one seeded input set. All arrays are C-contiguous float32.

    x [b,L,h,p], dt [b,L,h] (raw, before bias and softplus), dt_bias [h],
    A [h], B/C [b,L,g,n], D [h] or None, init_state [b,h,p,n] or None.
    For io_dtype "bf16", x/B/C hold bf16-representable values.
    """
    if io_dtype not in ("f32", "bf16"):
        raise ValueError(f"io_dtype must be 'f32' or 'bf16', got {io_dtype!r}")
    if init not in ("zero", "normal"):
        raise ValueError(f"init must be 'zero' or 'normal', got {init!r}")
    rng = np.random.Generator(np.random.PCG64(seed))
    f32 = np.float32
    x = rng.standard_normal((batch, seqlen, nheads, headdim), dtype=f32)
    dt = rng.standard_normal((batch, seqlen, nheads), dtype=f32)
    dt_floor = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), size=nheads))
    dt_bias = _inverse_softplus(dt_floor).astype(f32)
    A = (-np.exp(rng.uniform(np.log(1.0), np.log(16.0), size=nheads))).astype(f32)
    B = rng.standard_normal((batch, seqlen, ngroups, dstate), dtype=f32)
    C = rng.standard_normal((batch, seqlen, ngroups, dstate), dtype=f32)
    D = rng.standard_normal(nheads, dtype=f32)
    if init == "normal":
        init_state = (0.1 * rng.standard_normal((batch, nheads, headdim, dstate), dtype=f32)).astype(f32)
    else:
        init_state = None
    if io_dtype == "bf16":
        x, B, C = round_to_bf16(x), round_to_bf16(B), round_to_bf16(C)
    return {
        "x": x,
        "dt": dt,
        "dt_bias": dt_bias,
        "A": A,
        "B": B,
        "C": C,
        "D": D if with_D else None,
        "init_state": init_state,
    }


def workload_inputs(name: str) -> Dict[str, Optional[np.ndarray]]:
    w = WORKLOADS[name]
    return make_inputs(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate,
                       io_dtype=w.io_dtype, init=w.init, seed=w.seed)


# ----------------------------------------------------------------------------- around the scan
# Recipes for the operations before and after the scan (same rules: one PCG64
# stream per seed, values rounded to the io dtype where the tensor is io).
#   in_proj output zxbcdt [b, L, 2 d_inner + 2 g n + h] ~ N(0, 1) (io dtype); xBC
#       is its slice [d_inner, 2 d_inner + 2 g n) and the gate z its first d_inner
#       channels (fla "mamba2.py" split order: gate, xBC, dt when d_mlp = 0)
#   conv weight [conv_dim, K] and bias [conv_dim] ~ U(-1/sqrt(K), 1/sqrt(K)) fp32
#       (the bound of nn.Conv1d's default init for a depthwise kernel of K taps)
#   norm weight [d_inner] = 1 + N(0, 0.1^2) fp32 (RMSNorm weights start at one)
#   scan output y [b, L, d_inner] ~ N(0, 1) (io dtype) when the norm is tested alone

CONV_WORKLOAD = {"name": "mamba2_2p7b_conv", "batch": 4, "seqlen": 4096, "d_inner": 5120, "ngroups": 1,
                 "dstate": 128, "nheads": 80, "kernel_size": 4, "io_dtype": "bf16", "seed": 1241}
NORM_WORKLOAD = {"name": "mamba2_2p7b_gated_norm", "batch": 4, "seqlen": 4096, "d_inner": 5120, "ngroups": 1,
                 "dstate": 128, "nheads": 80, "io_dtype": "bf16", "eps": 1e-5, "seed": 1242}


def _io_round(a: np.ndarray, io_dtype: str) -> np.ndarray:
    if io_dtype not in ("f32", "bf16"):
        raise ValueError(f"io_dtype must be 'f32' or 'bf16', got {io_dtype!r}")
    return round_to_bf16(a) if io_dtype == "bf16" else np.ascontiguousarray(a, dtype=np.float32)


def make_layer_inputs(batch: int, seqlen: int, d_inner: int, ngroups: int, dstate: int, nheads: int,
                      kernel_size: int = 4, io_dtype: str = "bf16", seed: int = 0) -> Dict[str, np.ndarray]:
    """zxbcdt [b, L, 2 d_inner + 2 g n + h], conv weight [conv_dim, K], conv
    bias [conv_dim], norm weight [d_inner], y [b, L, d_inner] (all float32
    arrays; io tensors hold io-representable values)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    f32 = np.float32
    cd = d_inner + 2 * ngroups * dstate
    zxbcdt = _io_round(rng.standard_normal((batch, seqlen, d_inner + cd + nheads), dtype=f32), io_dtype)
    bound = 1.0 / np.sqrt(kernel_size)
    conv_w = rng.uniform(-bound, bound, size=(cd, kernel_size)).astype(f32)
    conv_b = rng.uniform(-bound, bound, size=cd).astype(f32)
    norm_w = (1.0 + 0.1 * rng.standard_normal(d_inner)).astype(f32)
    y = _io_round(rng.standard_normal((batch, seqlen, d_inner), dtype=f32), io_dtype)
    return {"zxbcdt": zxbcdt, "conv_w": conv_w, "conv_b": conv_b, "norm_w": norm_w, "y": y}
