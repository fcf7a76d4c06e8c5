"""Independent fp64 statements of the SSD forward, used only to pin the oracle.

Neither form shares code with the oracle (a C token recurrence) or with the
CUDA path. Both are written from the pages:

* ``quadratic``: the semiseparable-matrix ("attention-like") form. Output
  y_t = sum_{s<=t} (C_t . B_s) * delta_s * exp(sum_{k=s+1..t} delta_k A) * x_s
        + exp(sum_{k<=t} delta_k A) * (C_t . s_init) + D x_t.
  Source: burn-mamba ``Mamba2SsdInput`` rustdoc, "Minimal chunkwise SSD
  algorithm", Step 1 (Y_diag = (L o C B^T) X with the 1-semiseparable mask)
  and Step 4 (state-to-output); with a single chunk spanning the whole
  sequence this is the full quadratic form. Every decay exponent is summed
  token by token (no cumulative-sum differences), so it does not share the
  chunked form's arithmetic either.

* ``chunked``: the five-stage chunked decomposition, following the naive
  chunked SSD of flash-linear-attention ``fla/layers/mamba2.py``
  (Mamba2.torch_forward, "begin ssd naive implementation") and the k1..k5
  dataflow of burn-mamba ``mamba2/ssd/serial.rs`` (k1_ssd_chunk_cumsum,
  k2_ssd_bmm, k3_ssd_chunk_state, k4_ssd_state_passing, k5_ssd_chunk_scan):
  pad after discretisation, cumsum of dt*A within each chunk, C.B^T per
  chunk, the exp-segsum mask, chunk states, serial state passing, and the
  chunk scan with the D skip.
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np


def softplus(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    return np.where(v > 0, v + np.log1p(np.exp(-np.abs(v))), np.log1p(np.exp(np.minimum(v, 0))))


def _expand_groups(M: np.ndarray, nheads: int) -> np.ndarray:
    """[b,L,g,n] -> [b,L,h,n] with head h reading group h // (nheads/ngroups)."""
    g = M.shape[2]
    r = nheads // g
    return np.repeat(M, r, axis=2)


def quadratic(x, dt, dt_bias, A, B, C, D=None, init_state=None, dt_limit=None,
              seq_idx=None) -> Tuple[np.ndarray, np.ndarray]:
    """Brute-force semiseparable form in fp64 (O(L^2) per chain: tiny inputs only).
    dt_limit = (lo, hi) bounds the softplus output with np.clip. seq_idx [b, L]
    packs sequences into a row: token s reaches token t only if seq_idx does
    not change anywhere between them (no k in s+1..t with seq[k] != seq[k-1]),
    and the initial state only reaches tokens before the row's first change."""
    x = np.asarray(x, np.float64)
    b, L, h, p = x.shape
    n = B.shape[3]
    delta = softplus(np.asarray(dt, np.float64) + np.asarray(dt_bias, np.float64)[None, None, :])
    if dt_limit is not None:
        delta = np.clip(delta, dt_limit[0], dt_limit[1])
    Bh = _expand_groups(np.asarray(B, np.float64), h)
    Ch = _expand_groups(np.asarray(C, np.float64), h)
    A = np.asarray(A, np.float64)
    y = np.zeros((b, L, h, p))
    final = np.zeros((b, h, p, n))
    for bi in range(b):
        seq = None if seq_idx is None else np.asarray(seq_idx[bi])

        def cut(lo, hi_):  # a sequence boundary at some k in lo..hi_ (inclusive)
            return seq is not None and any(seq[k] != seq[k - 1] for k in range(max(lo, 1), hi_ + 1))

        for hi in range(h):
            dA = delta[bi, :, hi] * A[hi]
            s0 = np.zeros((p, n)) if init_state is None else np.asarray(init_state[bi, hi], np.float64)
            for t in range(L):
                acc = np.zeros(p)
                for s in range(t + 1):
                    if cut(s + 1, t):
                        continue
                    expo = 0.0
                    for k in range(s + 1, t + 1):
                        expo += dA[k]
                    w = float(Ch[bi, t, hi] @ Bh[bi, s, hi]) * delta[bi, s, hi] * np.exp(expo)
                    acc += w * x[bi, s, hi]
                expo0 = 0.0
                for k in range(0, t + 1):
                    expo0 += dA[k]
                if not cut(1, t):
                    acc += np.exp(expo0) * (s0 @ Ch[bi, t, hi])
                if D is not None:
                    acc += float(D[hi]) * x[bi, t, hi]
                y[bi, t, hi] = acc
            # final state: the same weights with t = L - 1, without the C readout
            fs = np.zeros((p, n))
            for s in range(L):
                if cut(s + 1, L - 1):
                    continue
                expo = 0.0
                for k in range(s + 1, L):
                    expo += dA[k]
                fs += delta[bi, s, hi] * np.exp(expo) * np.outer(x[bi, s, hi], Bh[bi, s, hi])
            expo0 = 0.0
            for k in range(L):
                expo0 += dA[k]
            final[bi, hi] = fs + (0.0 if cut(1, L - 1) else np.exp(expo0)) * s0
    return y, final


def _segsum(cs_chunk: np.ndarray) -> np.ndarray:
    """exp-segsum mask for one chunk: out[t, s] = cs[t] - cs[s] for s <= t, -inf above."""
    Q = cs_chunk.shape[-1]
    diff = cs_chunk[..., :, None] - cs_chunk[..., None, :]
    mask = np.tril(np.ones((Q, Q), dtype=bool))
    return np.where(mask, diff, -np.inf)


def chunked(x, dt, dt_bias, A, B, C, D=None, init_state=None, chunk_len: int = 64,
            ) -> Tuple[np.ndarray, np.ndarray]:
    """The five-stage chunked SSD in fp64 (numpy), for any chunk length >= 1."""
    x = np.asarray(x, np.float64)
    b, L, h, p = x.shape
    n = B.shape[3]
    Q = int(chunk_len)
    delta = softplus(np.asarray(dt, np.float64) + np.asarray(dt_bias, np.float64)[None, None, :])
    Bh = _expand_groups(np.asarray(B, np.float64), h)
    Ch = _expand_groups(np.asarray(C, np.float64), h)
    A = np.asarray(A, np.float64)

    # discretise, then pad the sequence with zeros up to a multiple of Q
    xdt = x * delta[..., None]
    dA = delta * A[None, None, :]
    pad = (-L) % Q
    Lp = L + pad
    c = Lp // Q

    def padded(a):
        widths = [(0, 0)] * a.ndim
        widths[1] = (0, pad)
        return np.pad(a, widths)

    xdt_c = padded(xdt).reshape(b, c, Q, h, p)
    x_c = padded(x).reshape(b, c, Q, h, p)
    dA_c = padded(dA).reshape(b, c, Q, h).transpose(0, 3, 1, 2)          # [b,h,c,Q]
    B_c = padded(Bh).reshape(b, c, Q, h, n)
    C_c = padded(Ch).reshape(b, c, Q, h, n)

    # k1: cumulative sum of dt*A within each chunk
    cs = np.cumsum(dA_c, axis=-1)                                           # [b,h,c,Q]
    # k2: C . B^T per chunk
    CB = np.einsum("bclhn,bcshn->bchls", C_c, B_c)                         # [b,c,h,Q,Q]
    # k5 (intra part): exp-segsum mask applied to CB, then to x*dt
    Lmask = np.exp(_segsum(cs)).transpose(0, 2, 1, 3, 4)                   # [b,c,h,Q,Q]
    Y_diag = np.einsum("bchls,bcshp->bclhp", CB * Lmask, xdt_c)
    # k3: chunk states from a zero start
    decay_to_end = np.exp(cs[..., -1:] - cs).transpose(0, 2, 3, 1)          # [b,c,Q,h]
    S = np.einsum("bclhn,bclh,bclhp->bchpn", B_c, decay_to_end, xdt_c)     # [b,c,h,p,n]
    # k4: serial state passing across chunks
    s_in = np.zeros((b, c + 1, h, p, n))
    s_in[:, 0] = 0.0 if init_state is None else np.asarray(init_state, np.float64)
    chunk_decay = np.exp(cs[..., -1])                                       # [b,h,c]
    for ci in range(c):
        s_in[:, ci + 1] = chunk_decay[:, :, ci][..., None, None] * s_in[:, ci] + S[:, ci]
    # k5 (state part): exp(cs) * C . s_in
    Y_off = np.einsum("bclhn,bchpn->bclhp", C_c, s_in[:, :c]) * np.exp(cs).transpose(0, 2, 3, 1)[..., None]
    y = Y_diag + Y_off
    if D is not None:
        y = y + np.asarray(D, np.float64)[None, None, None, :, None] * x_c
    y = y.reshape(b, Lp, h, p)[:, :L]
    return y, s_in[:, c]


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max|got - ref| / max|ref| over the whole tensor (0 when both vanish)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    if den == 0.0:
        return num
    return num / den
