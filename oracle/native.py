"""ctypes front end of the C oracle -- TEST INFRASTRUCTURE ONLY.

``gdn_forward_c`` runs the per-token fp64 recurrence of ``gdn_oracle.c`` over
every (sequence, head) pair, or over a chosen sample of pairs, with OpenMP.
Inputs may be numpy arrays or CPU torch tensors of any float dtype; they are
converted to fp32 (exact for bf16 and fp32 values).
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        lib.oracle_gdn_units.argtypes = [P, P, P, P, P, P, P, P,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         P, P, P, P, ctypes.c_int, P, P, ctypes.c_int]
        lib.oracle_gdn_units.restype = ctypes.c_int
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f32(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").float().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def spans(B: int, T: int, cu_seqlens=None) -> list:
    """(first row, length) of every sequence in the flattened [B*T] token rows."""
    if cu_seqlens is None:
        return [(b * T, T) for b in range(B)]
    if hasattr(cu_seqlens, "cpu"):  # torch tensor
        cu_seqlens = cu_seqlens.cpu().numpy()
    cu = [int(x) for x in np.asarray(cu_seqlens)]
    return [(cu[n], cu[n + 1] - cu[n]) for n in range(len(cu) - 1)]


def gdn_units_c(q, k, v, log_alpha, beta, S0, cu_seqlens, units: Sequence[Tuple[int, int]],
                erase=None, write=None, n_threads: int = 0):
    """Run the recurrence for the listed (sequence, head) units only.

    q, k: [B, T, H, dk]; v: [B, T, H, dv]; log_alpha, beta: [B, T, H];
    S0: [N, H, dv, dk] or None.  Returns a list of (out [len, dv], S_final
    [dv, dk]) fp64 arrays, one per unit.
    """
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    la, be = _f32(log_alpha), _f32(beta)
    er, wr = _f32(erase), _f32(write)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    sp = spans(B, T, cu_seqlens)
    units = list(units)
    n = len(units)
    ustart = np.array([sp[s][0] for s, _ in units], np.int64)
    ulen = np.array([sp[s][1] for s, _ in units], np.int64)
    uhead = np.array([h for _, h in units], np.int32)
    uout = np.zeros(n, np.int64)
    if n > 1:
        uout[1:] = np.cumsum(ulen)[:-1]
    out = np.zeros((int(ulen.sum()), dv), np.float64)
    Sf = np.zeros((n, dv, dk), np.float64)
    s0 = None
    if S0 is not None:
        S0a = _f32(S0)
        s0 = np.ascontiguousarray(np.stack([S0a[s, h] for s, h in units]) if n else
                                  np.zeros((0, dv, dk), np.float32))
    rc = lib.oracle_gdn_units(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(be), _ptr(er), _ptr(wr),
                              _ptr(s0), H, dk, dv, _ptr(ustart), _ptr(ulen), _ptr(uhead), _ptr(uout),
                              n, _ptr(out), _ptr(Sf), int(n_threads))
    if rc != 0:
        raise RuntimeError(f"oracle_gdn_units failed with code {rc}")
    res = []
    for u in range(n):
        res.append((out[uout[u]:uout[u] + ulen[u]], Sf[u]))
    return res


def gdn_forward_c(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None,
                  erase=None, write=None, n_threads: int = 0):
    """Full forward over every (sequence, head): returns (out [B, T, H, dv],
    S_final [N, H, dv, dk]) in fp64."""
    k_ = _f32(k)
    B, T, H, dk = k_.shape
    dv = (v.shape[-1])
    sp = spans(B, T, cu_seqlens)
    units = [(s, h) for s in range(len(sp)) for h in range(H)]
    res = gdn_units_c(q, k_, v, log_alpha, beta, S0, cu_seqlens, units, erase, write, n_threads)
    out = np.zeros((B * T, H, dv))
    Sf = np.zeros((len(sp), H, dv, dk))
    for (s, h), (o, S) in zip(units, res):
        r0, ln = sp[s]
        out[r0:r0 + ln, h] = o
        Sf[s, h] = S
    return out.reshape(B, T, H, dv), Sf
