"""The pages' closed forms and identities, in fp64 numpy -- TEST INFRASTRUCTURE ONLY.

Matrices follow the column convention of qiita Nyysyyan (tokens are columns:
Q, K in R^{dk x L}, V in R^{dv x L}, H in R^{dv x L}) so that each function can be
read against the page's equations; ``chunked_wy_delta`` alone uses token rows,
the layout of the library.  Library routines used as single steps: matrix
products and ``np.linalg.solve`` (a triangular system solved densely).

Readings taken where the page is garbled:
* the WY matrix form writes "U_i" where the strict upper mask M^u_i is meant and
  loses a parenthesis; read W = (K - W (M^u o K^T K)) D_beta;
* "Gamma o K^T K" in the U matrix form is strictly upper (the page says so in
  words); the diagonal of Gamma is not used there;
* in the U/G induction one line writes gamma_{i-1} where gamma_i is meant.
"""
from __future__ import annotations

import numpy as np


def _gammas(alpha):
    """gamma_i = prod_{t<=i} alpha_t  (Nyysyyan, "Mamba2": definition of gamma)."""
    return np.cumprod(np.asarray(alpha, np.float64))


def _Gamma(gamma):
    """Upper-triangular Gamma_{ij} = gamma_j / gamma_i for i <= j, else 0
    (Nyysyyan, "Mamba2": the matrix Gamma)."""
    g = np.asarray(gamma, np.float64)
    L = len(g)
    G = np.zeros((L, L))
    for i in range(L):
        for j in range(i, L):
            G[i, j] = g[j] / g[i]
    return G


def causal_mask(L):
    """M_{ij} = 1 for j <= i (Nyysyyan, "Causal attention")."""
    return np.tril(np.ones((L, L)))


def linear_attention_matrix(Q, K, V):
    """H = V (M^T o (K^T Q))  (Nyysyyan, "Linear attention", matrix form)."""
    L = Q.shape[1]
    return V @ (causal_mask(L).T * (K.T @ Q))


def mamba2_matrix(Q, K, V, alpha, S0=None):
    """H = S0 Q D_gamma + V (Gamma o (K^T Q))  (Nyysyyan, "Mamba2", the S0 != O
    closed form)."""
    gamma = _gammas(alpha)
    H = V @ (_Gamma(gamma) * (K.T @ Q))
    if S0 is not None:
        H = H + S0 @ Q @ np.diag(gamma)
    return H


def A_matrix(k, beta):
    """A_i = I_d - beta_i k_i k_i^T  (Nyysyyan, "Gated-DeltaNet")."""
    k = np.asarray(k, np.float64)
    return np.eye(len(k)) - beta * np.outer(k, k)


def product_of_A(K, beta, i, start=0):
    """A_{start+1} A_{start+2} ... A_i as an explicit product (1-based i; i <=
    start gives the identity)."""
    d = K.shape[0]
    P = np.eye(d)
    for t in range(start, i):
        P = P @ A_matrix(K[:, t], beta[t])
    return P


def wy_vectors(K, beta):
    """w_1 = beta_1 k_1, w_i = beta_i (k_i - sum_{t<i} (k_i^T k_t) w_t)
    (Nyysyyan, "Gated-DeltaNet", the WY sequence)."""
    d, L = K.shape
    W = np.zeros((d, L))
    for i in range(L):
        acc = K[:, i].copy()
        for t in range(i):
            acc -= (K[:, i] @ K[:, t]) * W[:, t]
        W[:, i] = beta[i] * acc
    return W


def wy_matrix(K, beta):
    """W = K D_beta (I + (M^u o K^T K) D_beta)^{-1}  (Nyysyyan, "Gated-DeltaNet",
    WY in matrix form; M^u strictly upper)."""
    L = K.shape[1]
    Mu = np.triu(np.ones((L, L)), 1)
    Db = np.diag(beta)
    R = np.eye(L) + (Mu * (K.T @ K)) @ Db
    # X R = K D_beta  <=>  R^T X^T = (K D_beta)^T
    return np.linalg.solve(R.T, (K @ Db).T).T


def u_vectors(K, V, beta, alpha):
    """u_1 = beta_1 v_1, u_i = beta_i (v_i - sum_{s<i} (gamma_i/gamma_s)(k_s^T k_i) u_s)
    (Nyysyyan, "Gated-DeltaNet", the U sequence)."""
    gamma = _gammas(alpha)
    dv, L = V.shape
    U = np.zeros((dv, L))
    for i in range(L):
        acc = V[:, i].copy()
        for s in range(i):
            acc -= (gamma[i] / gamma[s]) * (K[:, s] @ K[:, i]) * U[:, s]
        U[:, i] = beta[i] * acc
    return U


def u_matrix(K, V, beta, alpha):
    """U = V D_beta (I + (Gamma o K^T K) D_beta)^{-1}, Gamma o K^T K strictly
    upper  (Nyysyyan, "Gated-DeltaNet", U in matrix form)."""
    gamma = _gammas(alpha)
    L = K.shape[1]
    Gs = np.triu(_Gamma(gamma), 1)
    Db = np.diag(beta)
    R = np.eye(L) + (Gs * (K.T @ K)) @ Db
    return np.linalg.solve(R.T, (V @ Db).T).T


def G_explicit(K, V, beta, alpha, i):
    """G_i = sum_{s<=i} beta_s (gamma_i/gamma_s) v_s k_s^T A_{s+1}...A_i by explicit
    products (Nyysyyan, "Gated-DeltaNet", second term of the unrolled state)."""
    gamma = _gammas(alpha)
    G = np.zeros((V.shape[0], K.shape[0]))
    for s in range(i):
        G += beta[s] * (gamma[i - 1] / gamma[s]) * np.outer(V[:, s], K[:, s]) @ product_of_A(K, beta, i, start=s + 1)
    return G


def unrolled_state(K, V, beta, alpha, S0, i):
    """S_i = gamma_i S0 A_1...A_i + G_i  (Nyysyyan, "Gated-DeltaNet", unrolled
    recurrence)."""
    gamma = _gammas(alpha)
    return gamma[i - 1] * S0 @ product_of_A(K, beta, i) + G_explicit(K, V, beta, alpha, i)


def gdn_matrix_form(Q, K, V, alpha, beta, S0=None):
    """Whole-sequence Gated DeltaNet output (Nyysyyan, "Gated-DeltaNet", final
    matrix form):

        H = S0 (Q - W (M^T o (K^T Q))) D_gamma + U (Gamma o (K^T Q))
    """
    L = Q.shape[1]
    gamma = _gammas(alpha)
    KtQ = K.T @ Q
    H = u_matrix(K, V, beta, alpha) @ (_Gamma(gamma) * KtQ)
    if S0 is not None:
        W = wy_matrix(K, beta)
        H = H + S0 @ (Q - W @ (causal_mask(L).T * KtQ)) @ np.diag(gamma)
    return H


def gdn_chunked(Q, K, V, alpha, beta, S0, chunk_lengths):
    """Chunk computation (Nyysyyan, "Chunk Computation"): split the tokens into
    chunks of the given (possibly unequal) lengths; each chunk computes its
    outputs with the matrix form, taking the previous chunk's final state as its
    S0, and hands on its own final state

        S_{C_j} = gamma_L S0 A_1...A_L + G_L = gamma_L S0 (I - W K^T) + U D K^T,
        D = diag(gamma_L / gamma_s),

    where gamma restarts at each chunk (products of the chunk's own alphas).
    Returns (H [dv, L_total], S_final).
    """
    dk = K.shape[0]
    dv = V.shape[0]
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, np.float64)
    outs = []
    t0 = 0
    for Lc in chunk_lengths:
        sl = slice(t0, t0 + Lc)
        Qc, Kc, Vc, ac, bc = Q[:, sl], K[:, sl], V[:, sl], alpha[sl], beta[sl]
        outs.append(gdn_matrix_form(Qc, Kc, Vc, ac, bc, S))
        gamma = _gammas(ac)
        W = wy_matrix(Kc, bc)
        U = u_matrix(Kc, Vc, bc, ac)
        S = gamma[-1] * S @ (np.eye(dk) - W @ Kc.T) + U @ np.diag(gamma[-1] / gamma) @ Kc.T
        t0 += Lc
    return np.concatenate(outs, axis=1), S


def chunked_wy_delta(q, k, v, log_alpha, beta, S0, C):
    """Token-row chunk form with the decayed WY factor, the arrangement the
    library computes (rows are tokens; S is dv x dk):

        g = cumsum(log alpha) inside the chunk,
        A = strictly-lower(diag(beta) K K^T o exp(g_i - g_j)),  T = (I + A)^{-1},
        W~ = T diag(beta e^g) K,  U = T diag(beta) V,
        delta = U - W~ S^T,
        O = diag(e^g) Q S^T + lower-incl-diag(Q K^T o exp(g_i - g_j)) delta,
        S <- e^{g_last} S + delta^T diag(e^{g_last - g}) K.

    W~ is gamma_i w_i with gamma measured from the chunk start (multiply the WY
    recursion of Nyysyyan's "Gated-DeltaNet" by gamma_i); with it the unrolled
    state reads S_i = gamma_i S + sum_{s<=i} (gamma_i/gamma_s)(u_s - S w~_s) k_s^T,
    which gives the three lines above.  The last chunk may be shorter than C.
    q, k: [L, dk]; v: [L, dv]. Returns (O [L, dv], S_final).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    la = np.asarray(log_alpha, np.float64)
    b = np.asarray(beta, np.float64)
    L, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, np.float64)
    O = np.zeros((L, dv))
    for t0 in range(0, L, C):
        t1 = min(L, t0 + C)
        Kc, Qc, Vc, bc = k[t0:t1], q[t0:t1], v[t0:t1], b[t0:t1]
        g = np.cumsum(la[t0:t1])
        n = t1 - t0
        D = np.exp(g[:, None] - g[None, :]) * np.tril(np.ones((n, n)))
        A = np.tril(bc[:, None] * (Kc @ Kc.T) * D, -1)
        T = np.linalg.solve(np.eye(n) + A, np.eye(n))
        Wt = T @ (bc[:, None] * np.exp(g)[:, None] * Kc)
        U = T @ (bc[:, None] * Vc)
        delta = U - Wt @ S.T
        O[t0:t1] = np.exp(g)[:, None] * (Qc @ S.T) + ((Qc @ Kc.T) * D) @ delta
        S = np.exp(g[-1]) * S + delta.T @ (np.exp(g[-1] - g)[:, None] * Kc)
    return O, S


def chunked_wy_delta_bwd(q, k, v, log_alpha, beta, S0, dO, dS_final, C):
    """The backward of ``chunked_wy_delta``, chunk by chunk in reverse (the pages
    derive none; this is the reverse-mode derivative of the chunk form above,
    written with matrices so that each line is a dense product a tensor-core kernel
    can take).  Per chunk, with S the chunk-start state, dS' the gradient of the
    chunk-end state, E = diag(e^{g_last - g}), P = lower-incl(Q K^T o D):

        d delta = P^T dO + E K dS'^T
        dS      = dO^T diag(e^g) Q + e^{g_last} dS' - d delta^T W~      (to the previous chunk)
        dP      = lower-incl(dO delta^T)
        dQ      = diag(e^g) dO S + (dP o D) K
        dK      = (dP o D)^T Q + E delta dS'  + diag(beta e^g) T^T dW + X K + X^T K
        dU      = d delta,  dW = -d delta S,  dV = diag(beta) T^T dU
        dT      = dU (diag(beta) V)^T + dW (diag(beta e^g) K)^T,  dA = -T^T dT T^T
        X       = strictly-lower(dA) o D o beta_i
        dbeta_i = (T^T dU)_i . v_i + e^{g_i} (T^T dW)_i . k_i + sum_j dA_ij (k_i . k_j) D_ij

    and the gate: every use of g (D, e^g, e^{g_last}) gives dg, and d log alpha is
    the reverse cumulative sum of dg inside the chunk.  Returns (dq, dk, dv,
    dlog_alpha, dbeta, dS0) like ``backward.gdn_sequence_bwd``.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    la = np.asarray(log_alpha, np.float64)
    b = np.asarray(beta, np.float64)
    dO = np.asarray(dO, np.float64)
    L, dk = k.shape
    dv = v.shape[1]
    # forward: chunk-start states
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, np.float64)
    starts = []
    bounds = [(t0, min(L, t0 + C)) for t0 in range(0, L, C)]
    for t0, t1 in bounds:
        starts.append(S.copy())
        _, S = chunked_wy_delta(q[t0:t1], k[t0:t1], v[t0:t1], la[t0:t1], b[t0:t1], S, C)
    dS = np.zeros((dv, dk)) if dS_final is None else np.array(dS_final, np.float64)
    gq, gk, gv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    gla, gb = np.zeros(L), np.zeros(L)
    for (t0, t1), S in zip(reversed(bounds), reversed(starts)):
        n = t1 - t0
        Kc, Qc, Vc, bc, dOc = k[t0:t1], q[t0:t1], v[t0:t1], b[t0:t1], dO[t0:t1]
        g = np.cumsum(la[t0:t1])
        eg, Gm = np.exp(g), np.exp(g[-1])
        E = np.exp(g[-1] - g)
        Mi = np.tril(np.ones((n, n)))
        D = np.exp(g[:, None] - g[None, :]) * Mi
        KK = Kc @ Kc.T
        A = np.tril(bc[:, None] * KK * D, -1)
        T = np.linalg.solve(np.eye(n) + A, np.eye(n))
        Wt = T @ ((bc * eg)[:, None] * Kc)
        U = T @ (bc[:, None] * Vc)
        delta = U - Wt @ S.T
        QK = Qc @ Kc.T
        P = QK * D
        dSn = dS  # gradient of this chunk's end state
        # output and state-update terms
        ddelta = P.T @ dOc + (E[:, None] * Kc) @ dSn.T
        dS_prev = dOc.T @ (eg[:, None] * Qc) + Gm * dSn - ddelta.T @ Wt
        dP = (dOc @ delta.T) * Mi
        dQ = eg[:, None] * (dOc @ S) + (dP * D) @ Kc
        dK = (dP * D).T @ Qc + E[:, None] * (delta @ dSn)
        # delta = U - W~ S^T
        dU = ddelta
        dW = -ddelta @ S
        TdU, TdW = T.T @ dU, T.T @ dW
        dV = bc[:, None] * TdU
        dK += (bc * eg)[:, None] * TdW
        db = np.sum(TdU * Vc, axis=1) + eg * np.sum(TdW * Kc, axis=1)
        # T = (I + A)^{-1}
        dT = dU @ (bc[:, None] * Vc).T + dW @ ((bc * eg)[:, None] * Kc).T
        dA = np.tril(-T.T @ dT @ T.T, -1)
        X = dA * D * bc[:, None]
        dK += X @ Kc + X.T @ Kc
        db += np.sum(dA * KK * D, axis=1)
        # gates: dD from A and P, d e^g from W~ and O, d e^{g_last} and E from S'
        dD = dA * bc[:, None] * KK + dP * QK
        dg = np.sum(dD * D, axis=1) - np.sum(dD * D, axis=0)
        deg = bc * np.sum(TdW * Kc, axis=1) + np.sum(dOc * (Qc @ S.T), axis=1)
        dg += deg * eg
        dE = np.sum((delta @ dSn) * Kc, axis=1)  # d(e^{g_last - g_s})
        dg -= dE * E
        dg[-1] += np.sum(dE * E) + np.sum(dSn * S) * Gm
        gq[t0:t1], gk[t0:t1], gv[t0:t1], gb[t0:t1] = dQ, dK, dV, db
        gla[t0:t1] = np.cumsum(dg[::-1])[::-1]
        dS = dS_prev
    return gq, gk, gv, gla, gb, dS
