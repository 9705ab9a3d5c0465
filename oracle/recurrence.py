"""The Gated DeltaNet recurrence, written out per token in fp64 (numpy).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Definition followed (qiita Nyysyyan, "Gated-DeltaNet" section, first equation
block):

    S_i = alpha_i S_{i-1} (I - beta_i k_i k_i^T) + beta_i v_i k_i^T
    h_i = S_i q_i

with S a dv x dk matrix, so the read happens after token i is written.  Plain
DeltaNet is alpha_i = 1 (same section).  alpha enters as log alpha.

For the special-case pins the erase strength and the write strength may be
given separately:

    S_i = alpha_i S_{i-1} (I - e_i k_i k_i^T) + w_i v_i k_i^T

which is the definition when e = w = beta, Mamba2 when e = 0 and w = 1, and
linear attention when also alpha = 1 (qiita Nyysyyan, "Mamba2" and "Linear
attention" sections).
"""
from __future__ import annotations

import numpy as np


def gdn_sequence(q, k, v, log_alpha, beta, S0=None, erase=None, write=None):
    """One sequence of one head.

    q, k: [L, dk]; v: [L, dv]; log_alpha, beta: [L]; S0: [dv, dk] or None.
    erase/write: [L] or None (None means beta).
    Returns (h [L, dv], S_L [dv, dk]) in fp64.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    a = np.exp(np.asarray(log_alpha, np.float64))
    b = np.asarray(beta, np.float64)
    e = b if erase is None else np.asarray(erase, np.float64)
    wr = b if write is None else np.asarray(write, np.float64)
    L, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, np.float64, copy=True)
    h = np.empty((L, dv))
    I = np.eye(dk)
    for i in range(L):
        kk = k[i]
        # alpha_i S_{i-1} (I - e_i k_i k_i^T) + w_i v_i k_i^T, as written.
        S = a[i] * S @ (I - e[i] * np.outer(kk, kk)) + wr[i] * np.outer(v[i], kk)
        h[i] = S @ q[i]
    return h, S


def gdn_sequence_gate_predict_write(q, k, v, log_alpha, beta, S0=None):
    """The same layer stated as gate -> predict -> correct -> write -> read.

    kkkzoz "linear-attention", "Gated DeltaNet" section: the old state is first
    scaled by the gate, the gated state predicts a value for k_t, the error
    against v_t is written back along k_t with strength eta_t (= beta), and the
    output is read from the new state with q_t.  Restated here from its meaning,
    independently of ``gdn_sequence``.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    L, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, np.float64, copy=True)
    out = np.empty((L, dv))
    for t in range(L):
        gated = np.exp(float(log_alpha[t])) * S
        pred = gated @ k[t]
        delta = v[t] - pred
        S = gated + float(beta[t]) * np.outer(delta, k[t])
        out[t] = S @ q[t]
    return out, S


def gdn_forward(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None):
    """Batched layout of the library: q, k [B, T, H, dk]; v [B, T, H, dv];
    log_alpha, beta [B, T, H]; S0 [N, H, dv, dk] or None; cu_seqlens [N+1] or
    None (then N = B and every sequence has T tokens).

    Every (sequence, head) pair is an independent recurrence.  A packed batch
    (B = 1) restarts the state at every cu_seqlens boundary.
    Returns (out [B, T, H, dv], S_final [N, H, dv, dk]) in fp64.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    la = np.asarray(log_alpha, np.float64)
    be = np.asarray(beta, np.float64)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        spans = [(b, 0, T) for b in range(B)]
    else:
        cu = [int(x) for x in np.asarray(cu_seqlens)]
        spans = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    out = np.zeros((B, T, H, dv))
    Sf = np.zeros((len(spans), H, dv, dk))
    for n, (b, t0, t1) in enumerate(spans):
        for h in range(H):
            s0 = None if S0 is None else np.asarray(S0, np.float64)[n, h]
            o, S = gdn_sequence(q[b, t0:t1, h], k[b, t0:t1, h], v[b, t0:t1, h],
                                la[b, t0:t1, h], be[b, t0:t1, h], s0)
            out[b, t0:t1, h] = o
            Sf[n, h] = S
    return out, Sf
