"""Gradients of the Gated DeltaNet recurrence, per token in fp64 (numpy).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The pages do not derive a backward pass (qiita Nyysyyan motivates the chunk form
by training but stops at the forward).  This is the plain reverse-mode derivative
of the recurrence of ``recurrence.gdn_sequence`` (Nyysyyan, "Gated-DeltaNet",
first equation block), written from the forward in its gate -> predict -> write
order:

    a_t = exp(log_alpha_t)
    p_t = S_{t-1} k_t                       (prediction of the old state)
    u_t = beta_t (v_t - a_t p_t)            (correction written along k_t)
    S_t = a_t S_{t-1} + u_t k_t^T           (= a_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T)
    o_t = S_t q_t

For a loss L with dL/do_t = dO_t and dL/dS_T = dS_T, walking t = T .. 1 with
G = dL/dS_t (G starts at dS_T):

    G      += dO_t q_t^T
    dq_t    = S_t^T dO_t
    du      = G k_t
    dv_t    = beta_t du
    dbeta_t = du . (v_t - a_t p_t)
    da      = <G, S_{t-1}> - beta_t du . p_t
    dp      = -beta_t a_t du
    dk_t    = G^T u_t + S_{t-1}^T dp
    G       = a_t G + dp k_t^T             (= a_t G (I - beta_t k_t k_t^T))
    dlog_alpha_t = a_t da

and dL/dS_0 = G at the end.  Pinned in tests/test_oracle_pins.py by central finite
differences of ``recurrence.gdn_sequence`` and by an autograd run of a separately
written torch forward.
"""
from __future__ import annotations

import numpy as np


def gdn_sequence_bwd(q, k, v, log_alpha, beta, S0, dO, dS_final=None):
    """One sequence of one head.  q, k: [L, dk]; v, dO: [L, dv]; log_alpha, beta:
    [L]; S0, dS_final: [dv, dk] or None.  Returns (dq, dk, dv, dlog_alpha, dbeta,
    dS0) in fp64."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dO = np.asarray(dO, np.float64)
    a = np.exp(np.asarray(log_alpha, np.float64))
    b = np.asarray(beta, np.float64)
    L, dk = k.shape
    dv = v.shape[1]
    # forward, keeping every state (small cases only)
    S = np.zeros((L + 1, dv, dk))
    if S0 is not None:
        S[0] = np.asarray(S0, np.float64)
    P = np.zeros((L, dv))
    U = np.zeros((L, dv))
    for t in range(L):
        P[t] = S[t] @ k[t]
        U[t] = b[t] * (v[t] - a[t] * P[t])
        S[t + 1] = a[t] * S[t] + np.outer(U[t], k[t])
    G = np.zeros((dv, dk)) if dS_final is None else np.array(dS_final, np.float64, copy=True)
    gq = np.zeros_like(q)
    gk = np.zeros_like(k)
    gv = np.zeros_like(v)
    gla = np.zeros(L)
    gb = np.zeros(L)
    for t in range(L - 1, -1, -1):
        S_prev, S_t = S[t], S[t + 1]
        G += np.outer(dO[t], q[t])
        gq[t] = S_t.T @ dO[t]
        du = G @ k[t]
        gv[t] = b[t] * du
        gb[t] = du @ (v[t] - a[t] * P[t])
        da = np.sum(G * S_prev) - b[t] * (du @ P[t])
        dp = -b[t] * a[t] * du
        gk[t] = G.T @ U[t] + S_prev.T @ dp
        G = a[t] * G + np.outer(dp, k[t])
        gla[t] = a[t] * da
    return gq, gk, gv, gla, gb, G


def gdn_backward(q, k, v, log_alpha, beta, S0, dO, dS_final=None, cu_seqlens=None):
    """Batched layout of the library: q, k [B, T, H, dk]; v, dO [B, T, H, dv];
    log_alpha, beta [B, T, H]; S0, dS_final [N, H, dv, dk] or None; cu_seqlens
    [N+1] or None.  Returns (dq, dk, dv, dlog_alpha, dbeta, dS0) in fp64 with the
    shapes of the inputs (dS0 [N, H, dv, dk])."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dO = np.asarray(dO, np.float64)
    la = np.asarray(log_alpha, np.float64)
    be = np.asarray(beta, np.float64)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        spans = [(b_, 0, T) for b_ in range(B)]
    else:
        cu = [int(x) for x in np.asarray(cu_seqlens)]
        spans = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    out = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(la),
           np.zeros_like(be)]
    dS0 = np.zeros((len(spans), H, dv, dk))
    for n, (b_, t0, t1) in enumerate(spans):
        for h in range(H):
            s0 = None if S0 is None else np.asarray(S0, np.float64)[n, h]
            dsf = None if dS_final is None else np.asarray(dS_final, np.float64)[n, h]
            r = gdn_sequence_bwd(q[b_, t0:t1, h], k[b_, t0:t1, h], v[b_, t0:t1, h],
                                 la[b_, t0:t1, h], be[b_, t0:t1, h], s0, dO[b_, t0:t1, h], dsf)
            for i in range(5):
                out[i][b_, t0:t1, h] = r[i]
            dS0[n, h] = r[5]
    return (*out, dS0)
