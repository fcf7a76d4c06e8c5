"""fp64 oracle for the two per-token operations around the SSD scan
(test infrastructure only; same import rule as the rest of ``oracle/``).

* ``conv1d_silu`` -- the causal depthwise convolution plus SiLU that turns
  the in_proj slice xBC into x, B and C (fla "mamba2.py", ``Mamba2.__init__``:
  ``nn.Conv1d(conv_dim, conv_dim, kernel_size=conv_kernel, groups=conv_dim,
  padding=conv_kernel - 1)``; ``Mamba2.torch_forward`` step 2: conv over time,
  cropped to the first seq_len outputs, then ``self.act`` = SiLU, then the
  split into x / B / C). nn.Conv1d is a cross-correlation, so with K - 1
  zeros padded on the left output t is
      sum_k w[c, k] * xBC[t - (K - 1) + k, c]  (+ bias[c]).
  The returned conv state is what the same branch stores on cache init: the
  last K inputs of each channel, zero-padded on the left when seq_len < K.
* ``conv1d_step`` -- the cached-decode branch of step 2: the conv state
  shifts left by one, the new input enters at the right end, and the output
  is silu(sum_k state[c, k] w[c, k] + bias[c]).
* ``gated_rmsnorm`` -- ``RMSNormGated(d_inner, eps, norm_before_gate=False)``
  applied as ``norm(scan_output, gate)`` (fla "mamba2.py", step 3 of the
  fused branch). The pages name the module and its flag but do not print its
  body; the reading taken is the plain one the flag names: the gate is
  applied before the normalisation,
      v = y * silu(z);  out = v / sqrt(mean(v^2 over the group) + eps) * w,
  with the group the whole row unless a group size is given, and no bias.

Everything is computed in fp64 from the exactly widened inputs.

Parity status: pinned (tests/test_oracle_pins.py): the convolution against
numpy's ``np.convolve`` and single-tap kernels, the decode step against the
prefill on the same tokens, the norm against closed forms (constant rows,
scale invariance, per-group independence).
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np


def silu(v: np.ndarray) -> np.ndarray:
    """x * sigmoid(x) in fp64 (the activation the layer names "silu")."""
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def conv1d_silu(xbc: np.ndarray, weight: np.ndarray, bias: Optional[np.ndarray], d_inner: int,
                gn: int, activation: bool = True) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """Causal depthwise conv (+ SiLU) of xbc [b, L, conv_dim] with weight
    [conv_dim, K]; returns x [b, L, d_inner], B [b, L, gn], C [b, L, gn]
    and the conv state [b, conv_dim, K] (the last K inputs)."""
    xbc = np.asarray(xbc, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    b, L, cd = xbc.shape
    K = w.shape[1]
    assert w.shape[0] == cd and cd == d_inner + 2 * gn
    padded = np.concatenate([np.zeros((b, K - 1, cd)), xbc], axis=1)   # K - 1 zeros on the left
    out = np.zeros((b, L, cd))
    for k in range(K):
        out += w[None, None, :, k] * padded[:, k:k + L, :]
    if bias is not None:
        out += np.asarray(bias, dtype=np.float64)[None, None, :]
    if activation:
        out = silu(out)
    state = np.concatenate([np.zeros((b, max(K - L, 0), cd)), xbc[:, max(L - K, 0):, :]], axis=1)
    state = np.ascontiguousarray(state.transpose(0, 2, 1))              # [b, conv_dim, K]
    return out[..., :d_inner], out[..., d_inner:d_inner + gn], out[..., d_inner + gn:], state


def conv1d_step(xbc_t: np.ndarray, conv_state: np.ndarray, weight: np.ndarray, bias: Optional[np.ndarray],
                d_inner: int, gn: int, activation: bool = True):
    """One decode token: xbc_t [b, conv_dim], conv_state [b, conv_dim, K].
    Returns (x [b, d_inner], B [b, gn], C [b, gn], new conv state)."""
    s = np.asarray(conv_state, dtype=np.float64)
    new = np.concatenate([s[:, :, 1:], np.asarray(xbc_t, dtype=np.float64)[:, :, None]], axis=2)
    out = np.sum(new * np.asarray(weight, dtype=np.float64)[None], axis=-1)
    if bias is not None:
        out = out + np.asarray(bias, dtype=np.float64)[None]
    if activation:
        out = silu(out)
    return out[:, :d_inner], out[:, d_inner:d_inner + gn], out[:, d_inner + gn:], new


def gated_rmsnorm(y: np.ndarray, z: Optional[np.ndarray], weight: np.ndarray, eps: float,
                  group_size: Optional[int] = None) -> np.ndarray:
    """norm_before_gate=False gated RMSNorm over the last dimension of y
    (rows of length d, normalised in groups of group_size channels)."""
    y = np.asarray(y, dtype=np.float64)
    d = y.shape[-1]
    gs = d if group_size is None else group_size
    assert d % gs == 0
    v = y if z is None else y * silu(z)
    g = v.reshape(*v.shape[:-1], d // gs, gs)
    rstd = 1.0 / np.sqrt(np.mean(g * g, axis=-1, keepdims=True) + eps)
    return (g * rstd).reshape(v.shape) * np.asarray(weight, dtype=np.float64)
