"""Pins of the backward oracle (oracle/backward.py), CPU only.

The pages derive no backward pass, so the oracle's gradients are pinned to the
mathematics: central finite differences of the forward definition
(recurrence.gdn_sequence), and reverse-mode autograd through a torch forward written
separately in the update-as-written form S_t = a_t S_{t-1} (I - b_t k_t k_t^T) +
b_t v_t k_t^T.  Planted mistakes, applied to a copy of the oracle's own source,
each fail the finite-difference pin.
"""
import inspect

import numpy as np
import pytest
import torch

from oracle import backward as BW
from oracle import recurrence as R


def _rand(L, dk, dv, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((L, dk))
    k = rng.standard_normal((L, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    v = rng.standard_normal((L, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    la = -np.log1p(np.exp(-(rng.standard_normal(L) + 1.0)))
    S0 = 0.3 * rng.standard_normal((dv, dk))
    dO = rng.standard_normal((L, dv))
    dSf = rng.standard_normal((dv, dk))
    return [q, k, v, la, beta, S0], dO, dSf


def _loss(args, dO, dSf):
    q, k, v, la, beta, S0 = args
    o, S = R.gdn_sequence(q, k, v, la, beta, S0)
    return float(np.sum(o * dO) + np.sum(S * dSf))


def _finite_differences(args, dO, dSf, h=1e-6):
    grads = []
    for i, x in enumerate(args):
        g = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[i][idx] += h
            minus[i][idx] -= h
            g[idx] = (_loss(plus, dO, dSf) - _loss(minus, dO, dSf)) / (2 * h)
        grads.append(g)
    return grads  # q, k, v, log_alpha, beta, S0


def _fd_agrees(bwd, L=6, dk=3, dv=2, seed=0):
    args, dO, dSf = _rand(L, dk, dv, seed)
    fd = _finite_differences(args, dO, dSf)
    got = bwd(*args, dO, dSf)  # dq, dk, dv, dla, dbeta, dS0
    order = [0, 1, 2, 3, 4, 5]  # both in (q, k, v, log_alpha, beta, S0) order
    for j in order:
        scale = max(np.abs(fd[j]).max(), 1e-3)
        if np.abs(got[j] - fd[j]).max() > 1e-6 * scale:
            return False
    return True


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_backward_matches_finite_differences(seed):
    assert _fd_agrees(BW.gdn_sequence_bwd, seed=seed)


def test_backward_without_final_state_gradient():
    """dS_final = None means the loss does not see the final state."""
    args, dO, _ = _rand(7, 4, 3, 5)
    zero = np.zeros((3, 4))
    a = BW.gdn_sequence_bwd(*args, dO, None)
    b = BW.gdn_sequence_bwd(*args, dO, zero)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def _torch_forward(q, k, v, la, beta, S0):
    """The update as written on the page, S_t = a S (I - b k k^T) + b v k^T, o_t = S_t q_t."""
    S = S0
    outs = []
    eye = torch.eye(k.shape[1], dtype=torch.float64)
    for t in range(k.shape[0]):
        kt = k[t][:, None]
        S = torch.exp(la[t]) * S @ (eye - beta[t] * kt @ kt.T) + beta[t] * v[t][:, None] @ kt.T
        outs.append(S @ q[t])
    return torch.stack(outs), S


@pytest.mark.parametrize("L,dk,dv", [(9, 5, 4), (20, 8, 3)])
def test_backward_matches_autograd_of_the_update_as_written(L, dk, dv):
    args, dO, dSf = _rand(L, dk, dv, L + dk)
    ts = [torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in args]
    o, S = _torch_forward(*ts)
    loss = (o * torch.tensor(dO)).sum() + (S * torch.tensor(dSf)).sum()
    ref = torch.autograd.grad(loss, ts)
    got = BW.gdn_sequence_bwd(*args, dO, dSf)
    for g, r in zip(got, ref):
        assert np.allclose(g, r.numpy(), rtol=1e-11, atol=1e-12)


def test_batched_backward_equals_per_sequence():
    """The batched entry with a packed batch equals each sequence alone."""
    rng = np.random.default_rng(3)
    lens = [5, 1, 9]
    T, H, dk, dv = sum(lens), 2, 4, 3
    q = rng.standard_normal((1, T, H, dk))
    k = rng.standard_normal((1, T, H, dk))
    v = rng.standard_normal((1, T, H, dv))
    la = -np.abs(rng.standard_normal((1, T, H)))
    be = rng.uniform(0, 1, (1, T, H))
    dO = rng.standard_normal((1, T, H, dv))
    S0 = rng.standard_normal((3, H, dv, dk))
    dSf = rng.standard_normal((3, H, dv, dk))
    cu = np.array([0, 5, 6, 15])
    got = BW.gdn_backward(q, k, v, la, be, S0, dO, dSf, cu)
    for n in range(3):
        t0, t1 = cu[n], cu[n + 1]
        for h in range(H):
            ref = BW.gdn_sequence_bwd(q[0, t0:t1, h], k[0, t0:t1, h], v[0, t0:t1, h],
                                      la[0, t0:t1, h], be[0, t0:t1, h], S0[n, h],
                                      dO[0, t0:t1, h], dSf[n, h])
            for i in range(5):
                assert np.array_equal(got[i][0, t0:t1, h], ref[i])
            assert np.array_equal(got[5][n, h], ref[5])


PLANTS = {
    "dk_drops_prediction_term": ("gk[t] = G.T @ U[t] + S_prev.T @ dp", "gk[t] = G.T @ U[t]"),
    "dp_sign": ("dp = -b[t] * a[t] * du", "dp = b[t] * a[t] * du"),
    "state_gradient_not_decayed": ("G = a[t] * G + np.outer(dp, k[t])",
                                   "G = G + np.outer(dp, k[t])"),
    "dq_reads_old_state": ("gq[t] = S_t.T @ dO[t]", "gq[t] = S_prev.T @ dO[t]"),
    "dlog_alpha_misses_exp": ("gla[t] = a[t] * da", "gla[t] = da"),
    "output_gradient_on_key": ("G += np.outer(dO[t], q[t])", "G += np.outer(dO[t], k[t])"),
    "dbeta_ignores_prediction": ("gb[t] = du @ (v[t] - a[t] * P[t])", "gb[t] = du @ v[t]"),
}


@pytest.mark.parametrize("kind", sorted(PLANTS))
def test_finite_difference_pin_catches_planted_mistake(kind):
    old, new = PLANTS[kind]
    src = inspect.getsource(BW.gdn_sequence_bwd)
    assert old in src
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    assert not _fd_agrees(ns["gdn_sequence_bwd"])


@pytest.mark.parametrize("C,L", [(1, 7), (2, 9), (4, 13), (16, 40), (64, 64), (16, 37)])
def test_chunk_form_backward_equals_per_token_backward(C, L):
    """The chunk-form backward (matrix products per chunk, chunks in reverse) gives the
    per-token backward's gradients, for chunk lengths from 1 to 64 and ragged tails."""
    from oracle import derivations as D
    args, dO, dSf = _rand(L, 6, 5, C + L)
    ref = BW.gdn_sequence_bwd(*args, dO, dSf)
    got = D.chunked_wy_delta_bwd(*args, dO, dSf, C)
    for name, g, r in zip(("dq", "dk", "dv", "dla", "dbeta", "dS0"), got, ref):
        assert np.allclose(g, r, rtol=1e-9, atol=1e-11), (name, np.abs(g - r).max())


CHUNK_PLANTS = {
    "dK_misses_symmetric_gram_term": ("dK += X @ Kc + X.T @ Kc", "dK += X @ Kc"),
    "dA_sign": ("dA = np.tril(-T.T @ dT @ T.T, -1)", "dA = np.tril(T.T @ dT @ T.T, -1)"),
    "state_gradient_not_decayed": ("+ Gm * dSn -", "+ dSn -"),
    "gate_gradient_not_reverse_summed": ("gla[t0:t1] = np.cumsum(dg[::-1])[::-1]",
                                         "gla[t0:t1] = dg"),
    "delta_gradient_misses_state_write": ("ddelta = P.T @ dOc + (E[:, None] * Kc) @ dSn.T",
                                          "ddelta = P.T @ dOc"),
}


@pytest.mark.parametrize("kind", sorted(CHUNK_PLANTS))
def test_chunk_form_pin_catches_planted_mistake(kind):
    from oracle import derivations as D
    old, new = CHUNK_PLANTS[kind]
    src = inspect.getsource(D.chunked_wy_delta_bwd)
    assert old in src
    ns = {"np": np, "chunked_wy_delta": D.chunked_wy_delta}
    exec(src.replace(old, new), ns)
    args, dO, dSf = _rand(37, 6, 5, 3)
    ref = BW.gdn_sequence_bwd(*args, dO, dSf)
    got = ns["chunked_wy_delta_bwd"](*args, dO, dSf, 16)
    assert not all(np.allclose(g, r, rtol=1e-9, atol=1e-11) for g, r in zip(got, ref))


@pytest.mark.parametrize("L,C", [(37, 16), (65, 64), (1, 64)])
def test_zero_padded_tail_changes_no_gradient(L, C):
    """A ragged last chunk can be filled out to C tokens with q = k = v = dO = 0, beta = 0
    and log alpha = 0 (alpha = 1): such tokens leave the state unchanged (the erase and
    the write vanish with beta = 0, the gate with alpha = 1) and add nothing to any output,
    so the real tokens' gradients and dS0 are those of the unpadded sequence; the chunk
    form then works on whole chunks only (the chunked backward kernels rely on this).
    Checked on the chunk-form derivative itself."""
    from oracle import derivations as D
    args, dO, dSf = _rand(L, 6, 5, 300 + L)
    pad = (-L) % C
    padded = [np.concatenate([x, np.zeros((pad,) + x.shape[1:])]) for x in args[:5]] + [args[5]]
    dOp = np.concatenate([dO, np.zeros((pad, dO.shape[1]))])
    ref = D.chunked_wy_delta_bwd(*args, dO, dSf, C)
    got = D.chunked_wy_delta_bwd(*padded, dOp, dSf, C)
    for name, g, r in zip(("dq", "dk", "dv", "dla", "dbeta"), got[:5], ref[:5]):
        assert np.allclose(g[:L], r, rtol=1e-10, atol=1e-12), (name, np.abs(g[:L] - r).max())
    assert np.allclose(got[5], ref[5], rtol=1e-10, atol=1e-12)
    # the padding tokens' own dq, dk, dv, dbeta are 0 (their d log alpha is <G, S>, which
    # the padding does not use: those rows are never returned)
    per_token = BW.gdn_sequence_bwd(*padded, dOp, dSf)
    for j in (0, 1, 2, 4):
        assert np.abs(per_token[j][L:]).max() <= 1e-12, j
