"""Pins of the CPU oracle to facts the pages and the mathematics fix (CPU only).

Each check compares the oracle's per-token recurrence against something other
than itself: an identity proved on the pages, a closed form, an invariant, a
hand-derived example, or a second statement of the layer.  The last group plants
plausible mistakes in copies of the recurrence and shows that some pin fails for
each, so the pins have the power to catch them.
"""
import os

import numpy as np
import pytest

from oracle import derivations as D
from oracle import native
from oracle import recurrence as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(L, dk, dv, seed, alpha_mu=2.0, unit_keys=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((L, dk))
    k = rng.standard_normal((L, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=1, keepdims=True)
        q /= np.linalg.norm(q, axis=1, keepdims=True)
    v = rng.standard_normal((L, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    la = -np.log1p(np.exp(-(rng.standard_normal(L) + alpha_mu)))
    S0 = 0.1 * rng.standard_normal((dv, dk))
    return q, k, v, la, beta, S0


# ---------------------------------------------------------------- identities --

@pytest.mark.parametrize("dk,L", [(3, 12), (8, 12), (8, 5)])
def test_wy_identity(dk, L):
    """Nyysyyan "Gated-DeltaNet": A_1...A_i = I - sum_{t<=i} w_t k_t^T, by
    explicit products of the Householder-like factors, for every prefix i."""
    _, k, _, _, beta, _ = _rand(L, dk, 2, seed=dk * 100 + L, unit_keys=False)
    K = k.T * 0.7
    W = D.wy_vectors(K, beta)
    for i in range(1, L + 1):
        lhs = D.product_of_A(K, beta, i)
        rhs = np.eye(dk) - W[:, :i] @ K[:, :i].T
        assert np.abs(lhs - rhs).max() < 1e-12
    # the matrix form of the same W (triangular solve) gives the same vectors
    assert np.abs(D.wy_matrix(K, beta) - W).max() < 1e-12


@pytest.mark.parametrize("dk,dv,L", [(4, 3, 9), (8, 6, 11)])
def test_u_g_identity(dk, dv, L):
    """Nyysyyan "Gated-DeltaNet": G_i = sum_{s<=i} (gamma_i/gamma_s) u_s k_s^T."""
    _, k, v, la, beta, _ = _rand(L, dk, dv, seed=7 + L)
    K, V, alpha = k.T, v.T, np.exp(la)
    U = D.u_vectors(K, V, beta, alpha)
    gamma = np.cumprod(alpha)
    for i in range(1, L + 1):
        lhs = D.G_explicit(K, V, beta, alpha, i)
        rhs = sum((gamma[i - 1] / gamma[s]) * np.outer(U[:, s], K[:, s]) for s in range(i))
        assert np.abs(lhs - rhs).max() < 1e-12
    assert np.abs(D.u_matrix(K, V, beta, alpha) - U).max() < 1e-12


def test_unrolled_state_brute_force():
    """Nyysyyan "Gated-DeltaNet": the recurrence equals gamma_i S0 A_1..A_i + G_i."""
    dk, dv, L = 5, 4, 10
    q, k, v, la, beta, S0 = _rand(L, dk, dv, seed=3)
    for i in range(1, L + 1):
        _, S_rec = R.gdn_sequence(q[:i], k[:i], v[:i], la[:i], beta[:i], S0)
        S_unr = D.unrolled_state(k.T, v.T, beta, np.exp(la), S0, i)
        assert np.abs(S_rec - S_unr).max() < 1e-12


# -------------------------------------------------------------- closed forms --

@pytest.mark.parametrize("impl", ["numpy", "c"])
def test_mamba2_and_linear_attention_closed_forms(impl):
    """With the erase switched off and unit write strength the recurrence is
    Mamba2: H = S0 Q D_gamma + V (Gamma o K^T Q); with alpha = 1 too it is linear
    attention H = V (M^T o K^T Q)  (Nyysyyan, "Mamba2" and "Linear attention")."""
    dk, dv, L = 6, 5, 24
    q, k, v, la, beta, S0 = _rand(L, dk, dv, seed=11, unit_keys=False)
    zeros, ones = np.zeros(L), np.ones(L)
    if impl == "numpy":
        run = lambda la_, s0: R.gdn_sequence(q, k, v, la_, beta, s0, erase=zeros, write=ones)
    else:
        def run(la_, s0):
            out, Sf = native.gdn_forward_c(q[None, :, None], k[None, :, None], v[None, :, None],
                                           la_[None, :, None], beta[None, :, None],
                                           None if s0 is None else s0[None, None],
                                           erase=zeros[None, :, None], write=ones[None, :, None])
            return out[0, :, 0], Sf[0, 0]
        f32 = lambda x: x.astype(np.float32).astype(np.float64)
        q, k, v, la, S0 = f32(q), f32(k), f32(v), f32(la), f32(S0)
    h, _ = run(la, S0)
    H = D.mamba2_matrix(q.T, k.T, v.T, np.exp(la), S0)
    assert np.abs(h.T - H).max() < 1e-10
    h, _ = run(np.zeros(L), None)
    H = D.linear_attention_matrix(q.T, k.T, v.T)
    assert np.abs(h.T - H).max() < 1e-10


def test_full_sequence_matrix_form():
    """Nyysyyan "Gated-DeltaNet": H = S0 (Q - W (M^T o K^T Q)) D_gamma +
    U (Gamma o K^T Q), with W and U from triangular solves, equals the recurrence."""
    for (dk, dv, L, seed) in [(8, 6, 40, 1), (16, 16, 64, 2), (4, 8, 17, 3)]:
        q, k, v, la, beta, S0 = _rand(L, dk, dv, seed=seed)
        h, _ = R.gdn_sequence(q, k, v, la, beta, S0)
        H = D.gdn_matrix_form(q.T, k.T, v.T, np.exp(la), beta, S0)
        assert np.abs(h.T - H).max() < 1e-10


@pytest.mark.parametrize("lengths", [[16, 16, 16, 16], [5, 20, 1, 30, 8], [64]])
def test_chunk_computation_matches_recurrence(lengths):
    """Nyysyyan "Chunk Computation": chunks of unequal length, each with the
    previous chunk's final state as its S0, give the recurrence's outputs."""
    L = sum(lengths)
    q, k, v, la, beta, S0 = _rand(L, 8, 6, seed=L)
    h, S = R.gdn_sequence(q, k, v, la, beta, S0)
    H, S2 = D.gdn_chunked(q.T, k.T, v.T, np.exp(la), beta, S0, lengths)
    assert np.abs(h.T - H).max() < 1e-10
    assert np.abs(S - S2).max() < 1e-10


@pytest.mark.parametrize("C", [1, 2, 4, 16, 64])
def test_decayed_wy_chunk_form_matches_recurrence(C):
    """The token-row chunk form with the decayed W~ = T diag(beta e^g) K (the
    arrangement the library computes) equals the recurrence; T = 150 is not a
    multiple of any C > 2, so the last chunk is partial.  C = 1 is the
    recurrence itself, one token per chunk."""
    q, k, v, la, beta, S0 = _rand(150, 16, 12, seed=C)
    h, S = R.gdn_sequence(q, k, v, la, beta, S0)
    O, S2 = D.chunked_wy_delta(q, k, v, la, beta, S0, C)
    assert np.abs(h - O).max() < 1e-10
    assert np.abs(S - S2).max() < 1e-10


# --------------------------------------------------------------- invariants --

@pytest.mark.parametrize("gated", [False, True])
def test_write_invariant(gated):
    """Nyysyyan "Gated-DeltaNet" (DeltaNet, alpha = 1):
    S_i k_i = (1 - beta_i |k_i|^2) S_{i-1} k_i + beta_i |k_i|^2 v_i
    (the page's "v_k" read as v_i); with a gate the first term gains alpha_i."""
    dk, dv, L = 7, 5, 20
    q, k, v, la, beta, S0 = _rand(L, dk, dv, seed=5, unit_keys=False)
    if not gated:
        la = np.zeros(L)
    S_prev = S0
    for i in range(L):
        _, S_i = R.gdn_sequence(q[:i + 1], k[:i + 1], v[:i + 1], la[:i + 1], beta[:i + 1], S0)
        n2 = k[i] @ k[i]
        rhs = np.exp(la[i]) * (1 - beta[i] * n2) * (S_prev @ k[i]) + beta[i] * n2 * v[i]
        assert np.abs(S_i @ k[i] - rhs).max() < 1e-11
        S_prev = S_i


def test_exact_overwrite_reads_back_value():
    """Unit key, beta = 1, alpha = 1: S_i k_i = v_i exactly, so reading with
    q_i = k_i returns v_i (the write invariant's overwrite case)."""
    q, k, v, la, beta, S0 = _rand(30, 8, 8, seed=9)
    h, _ = R.gdn_sequence(k, k, v, np.zeros(30), np.ones(30), S0)
    assert np.abs(h - v).max() < 1e-12


def test_orthonormal_keys_columnwise_closed_form():
    """Keys along coordinate axes: every key column of S evolves alone,
    S[:, c] <- alpha (1 - beta) S[:, c] + beta v on the column being written and
    S[:, c] <- alpha S[:, c] elsewhere (the definition with k = e_c)."""
    dk, dv, L = 6, 4, 40
    rng = np.random.default_rng(4)
    cols = rng.integers(0, dk, L)
    k = np.eye(dk)[cols]
    q, _, v, la, beta, S0 = _rand(L, dk, dv, seed=4)
    h, S = R.gdn_sequence(q, k, v, la, beta, S0)
    Sc = S0.copy()
    for i in range(L):
        a = np.exp(la[i])
        Sc *= a
        c = cols[i]
        Sc[:, c] = (1 - beta[i]) * Sc[:, c] + beta[i] * v[i]
        assert np.abs(h[i] - Sc @ q[i]).max() < 1e-12
    assert np.abs(S - Sc).max() < 1e-12


def test_beta_zero_is_pure_decay():
    """beta = 0: nothing is written, h_t = gamma_t S0 q_t and S_T = gamma_T S0."""
    q, k, v, la, _, S0 = _rand(25, 6, 5, seed=8)
    h, S = R.gdn_sequence(q, k, v, la, np.zeros(25), S0)
    gamma = np.exp(np.cumsum(la))
    assert np.abs(h - gamma[:, None] * (q @ S0.T)).max() < 1e-12
    assert np.abs(S - gamma[-1] * S0).max() < 1e-12


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split("=")
            vals[key.strip()] = np.array([float(x) for x in rest.split()])
    return vals


@pytest.mark.parametrize("impl", ["numpy", "c"])
def test_hand_derived_two_token_example(impl):
    g = _read_golden("gdn_two_tokens_hand.txt")
    S0 = g["S0"].reshape(2, 2)
    k, q, v = g["k"].reshape(2, 2), g["q"].reshape(2, 2), g["v"].reshape(2, 2)
    la, be = np.log(g["alpha"]), g["beta"]
    if impl == "numpy":
        h, S = R.gdn_sequence(q, k, v, la, be, S0)
    else:
        out, Sf = native.gdn_forward_c(q[None, :, None], k[None, :, None], v[None, :, None],
                                       la[None, :, None], be[None, :, None], S0[None, None])
        h, S = out[0, :, 0], Sf[0, 0]
    assert np.abs(h.reshape(-1) - g["h"]).max() < 1e-6
    assert np.abs(S.reshape(-1) - g["S_final"]).max() < 1e-6


def test_gate_predict_write_statement_agrees():
    """kkkzoz "linear-attention", "Gated DeltaNet": gate -> predict -> delta ->
    write -> read is the same layer as the Nyysyyan update."""
    q, k, v, la, beta, S0 = _rand(64, 16, 8, seed=12)
    h1, S1 = R.gdn_sequence(q, k, v, la, beta, S0)
    h2, S2 = R.gdn_sequence_gate_predict_write(q, k, v, la, beta, S0)
    assert np.abs(h1 - h2).max() < 1e-12 and np.abs(S1 - S2).max() < 1e-12


# ----------------------------------------------------------- batch / layout --

def _batch(B, T, H, dk, dv, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, dk)).astype(np.float32)
    k = rng.standard_normal((B, T, H, dk)).astype(np.float32)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    la = (-np.log1p(np.exp(-(rng.standard_normal((B, T, H)) + 2)))).astype(np.float32)
    be = (1 / (1 + np.exp(-rng.standard_normal((B, T, H))))).astype(np.float32)
    S0 = (0.1 * rng.standard_normal((B, H, dv, dk))).astype(np.float32)
    return q, k, v, la, be, S0


def test_c_oracle_equals_numpy_oracle():
    q, k, v, la, be, S0 = _batch(2, 45, 3, 8, 6, seed=1)
    o1, s1 = native.gdn_forward_c(q, k, v, la, be, S0)
    o2, s2 = R.gdn_forward(q, k, v, la, be, S0)
    assert np.abs(o1 - o2).max() < 1e-12 and np.abs(s1 - s2).max() < 1e-12


def test_segment_hand_off():
    """Running [0, t) then [t, T) with the first S_final as the second S0 equals
    one pass (Nyysyyan "Chunk Computation": the state is the only thing passed)."""
    q, k, v, la, be, S0 = _batch(1, 100, 2, 8, 8, seed=2)
    o, s = native.gdn_forward_c(q, k, v, la, be, S0)
    for t in (1, 37, 64, 99):
        oa, sa = native.gdn_forward_c(q[:, :t], k[:, :t], v[:, :t], la[:, :t], be[:, :t], S0)
        ob, sb = native.gdn_forward_c(q[:, t:], k[:, t:], v[:, t:], la[:, t:], be[:, t:],
                                      sa.astype(np.float32))
        # the hand-off state is rounded to fp32 in between
        assert np.abs(np.concatenate([oa, ob], 1) - o).max() < 1e-5
        assert np.abs(sb - s).max() < 1e-5


def test_varlen_packed_equals_each_sequence_alone():
    lens = [5, 64, 1, 33]
    T = sum(lens)
    q, k, v, la, be, _ = _batch(1, T, 3, 8, 4, seed=3)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    S0 = (0.1 * np.random.default_rng(0).standard_normal((len(lens), 3, 4, 8))).astype(np.float32)
    o, s = native.gdn_forward_c(q, k, v, la, be, S0, cu_seqlens=cu)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        on, sn = native.gdn_forward_c(q[:, a:b], k[:, a:b], v[:, a:b], la[:, a:b], be[:, a:b], S0[n:n + 1])
        assert np.abs(o[:, a:b] - on).max() < 1e-13
        assert np.abs(s[n] - sn[0]).max() < 1e-13


def test_sampled_units_equal_full_run():
    q, k, v, la, be, S0 = _batch(3, 20, 4, 8, 4, seed=4)
    o, s = native.gdn_forward_c(q, k, v, la, be, S0)
    units = [(2, 1), (0, 3), (1, 0)]
    res = native.gdn_units_c(q, k, v, la, be, S0, None, units)
    for (b, h), (ou, su) in zip(units, res):
        assert np.abs(ou - o[b, :, h]).max() == 0 and np.abs(su - s[b, h]).max() == 0


# ------------------------------------------------------------ planted errors --
# Plausible mistakes, planted in copies of the recurrence (CPU only).  Each must
# be caught by at least one of the pins above.

def _mutant(kind):
    def run(q, k, v, la, beta, S0=None, erase=None, write=None):
        e = beta if erase is None else erase
        w = beta if write is None else write
        dk, dv = k.shape[1], v.shape[1]
        S = np.zeros((dv, dk)) if S0 is None else S0.copy()
        h = np.zeros((len(k), dv))
        for i in range(len(k)):
            a = np.exp(la[i])
            if kind == "read_before_write":
                h[i] = a * S @ q[i]
            if kind == "gate_after_write":
                S = a * (S @ (np.eye(dk) - e[i] * np.outer(k[i], k[i])) + w[i] * np.outer(v[i], k[i]))
            elif kind == "erase_sign":
                S = a * S @ (np.eye(dk) + e[i] * np.outer(k[i], k[i])) + w[i] * np.outer(v[i], k[i])
            elif kind == "no_beta_on_write":
                S = a * S @ (np.eye(dk) - e[i] * np.outer(k[i], k[i])) + np.outer(v[i], k[i])
            elif kind == "erase_on_left":
                S = a * (np.eye(dv) - e[i] * np.outer(v[i] / max(np.linalg.norm(v[i]), 1e-9), v[i] / max(np.linalg.norm(v[i]), 1e-9))) @ S + w[i] * np.outer(v[i], k[i])
            elif kind == "transposed_write":
                S = a * S @ (np.eye(dk) - e[i] * np.outer(k[i], k[i])) + w[i] * np.outer(k[i], v[i])
            else:
                S = a * S @ (np.eye(dk) - e[i] * np.outer(k[i], k[i])) + w[i] * np.outer(v[i], k[i])
            if kind != "read_before_write":
                h[i] = S @ q[i]
        return h, S
    return run


def _pins_fail(fn):
    """True when at least one pin (applied to fn as the recurrence) fails."""
    dk = dv = 6
    L = 20
    q, k, v, la, beta, S0 = _rand(L, dk, dv, seed=21, unit_keys=False)
    # Mamba2 closed form
    h, _ = fn(q, k, v, la, beta, S0, erase=np.zeros(L), write=np.ones(L))
    if np.abs(h.T - D.mamba2_matrix(q.T, k.T, v.T, np.exp(la), S0)).max() > 1e-8:
        return True
    # write invariant with the gate
    S_prev = S0
    for i in range(L):
        _, S_i = fn(q[:i + 1], k[:i + 1], v[:i + 1], la[:i + 1], beta[:i + 1], S0)
        n2 = k[i] @ k[i]
        rhs = np.exp(la[i]) * (1 - beta[i] * n2) * (S_prev @ k[i]) + beta[i] * n2 * v[i]
        if np.abs(S_i @ k[i] - rhs).max() > 1e-8:
            return True
        S_prev = S_i
    # full-sequence matrix form
    h, _ = fn(q, k, v, la, beta, S0)
    if np.abs(h.T - D.gdn_matrix_form(q.T, k.T, v.T, np.exp(la), beta, S0)).max() > 1e-8:
        return True
    return False


def test_pins_pass_on_the_oracle():
    assert not _pins_fail(lambda *a, **kw: R.gdn_sequence(*a, **kw))


@pytest.mark.parametrize("kind", ["read_before_write", "gate_after_write", "erase_sign",
                                  "no_beta_on_write", "erase_on_left", "transposed_write"])
def test_pins_catch_planted_mistake(kind):
    assert _pins_fail(_mutant(kind))
