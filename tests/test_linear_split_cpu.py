"""CPU pin of the algebra the linear mode's in-GPU split relies on, with the fp64 oracle only.

In the linear mode (erase 0, write 1: Nyysyyan, "Mamba2" section) the state over a segment
of tokens is the decayed sum of the writes, so it maps affinely with a scalar gain:
S_end = Gamma S_start + L, Gamma = e^{sum of log alpha over the segment}, L the segment's
end state from zero.  Each output is linear in the start state as well:
o_t = o_t(0) + e^{G_t} S_start q_t, G_t the sum of log alpha from the segment's first token
through t.  The GPU path runs the segments from zero (the first from S0), folds the start
states in order and adds that correction; here the same three steps on oracle segments must
give the unsplit oracle to fp64 rounding, and a plausible slip in any of them must not.
"""
import numpy as np
import pytest

from oracle.recurrence import gdn_sequence


def _inputs(L, dk, dv, seed, alpha_mu=2.0, resets=()):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((L, dk))
    k = rng.standard_normal((L, dk))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((L, dv))
    x = rng.normal(alpha_mu, 1.0, L)
    la = -np.logaddexp(0.0, -x)  # log sigmoid(x)
    for t in resets:
        la[t] = -np.inf
    S0 = 0.1 * rng.standard_normal((dv, dk))
    return q, k, v, la, S0


def _linear(q, k, v, la, S0):
    L = len(la)
    return gdn_sequence(q, k, v, la, np.zeros(L), S0, erase=np.zeros(L), write=np.ones(L))


def _split(q, k, v, la, S0, bounds, inclusive=True, fold_gain_of=None):
    """The split's three steps on oracle segments.  `inclusive` and `fold_gain_of` plant
    the slips the pins must catch (G_t without token t; a fold with the wrong segment's
    gain)."""
    outs, ends = [], []
    for r, (a, b) in enumerate(bounds):  # 1. segments from zero, the first from S0
        o, Lr = _linear(q[a:b], k[a:b], v[a:b], la[a:b], S0 if r == 0 else None)
        outs.append(o)
        ends.append(Lr)
    gam = [np.exp(la[a:b].sum()) for a, b in bounds]
    starts = [None, ends[0]]  # 2. fold: S_start_r = Gamma_{r-1} S_start_{r-1} + L_{r-1}
    for r in range(2, len(bounds)):
        g = gam[r - 1] if fold_gain_of is None else gam[fold_gain_of(r)]
        starts.append(g * starts[r - 1] + ends[r - 1])
    R = len(bounds)
    S_final = gam[R - 1] * starts[R - 1] + ends[R - 1] if R > 1 else ends[0]
    for r in range(1, R):  # 3. o_t += e^{G_t} S_start q_t
        a, b = bounds[r]
        G = np.cumsum(la[a:b])
        if not inclusive:
            G = G - la[a:b]
        outs[r] = outs[r] + np.exp(G)[:, None] * (q[a:b] @ starts[r].T)
    return np.concatenate(outs), S_final


def _bounds(L, R, C=64):
    """Whole-chunk segments, as even as the chunk count allows (the kernel's rule)."""
    nch = -(-L // C)
    per = -(-nch // R)
    return [(min(r * per * C, L), min((r + 1) * per * C, L)) for r in range(R)]


@pytest.mark.parametrize("L,R", [(200, 2), (333, 3), (600, 4), (1000, 4)])
@pytest.mark.parametrize("alpha_mu", [6.0, 2.0, -2.0, None],
                         ids=["slow", "mild", "strong", "no_gate"])
def test_split_equals_the_recurrence(L, R, alpha_mu):
    q, k, v, la, S0 = _inputs(L, 8, 6, seed=L + R, alpha_mu=alpha_mu or 0.0)
    if alpha_mu is None:
        la = np.zeros(L)  # linear attention: alpha = 1, Gamma = 1
    o_ref, S_ref = _linear(q, k, v, la, S0)
    o, S = _split(q, k, v, la, S0, _bounds(L, R))
    scale = np.abs(o_ref).max()
    assert np.abs(o - o_ref).max() <= 1e-12 * scale
    assert np.abs(S - S_ref).max() <= 1e-12 * np.abs(S_ref).max()


def test_split_with_resets_at_segment_edges():
    """alpha = 0 (log alpha = -inf) on a segment's last token, the next one's first, inside
    a segment and on the last token: exp(-inf) = 0 zeroes the gains and the correction."""
    L = 1000
    q, k, v, la, S0 = _inputs(L, 8, 6, seed=5, resets=(255, 256, 511, 600, 999))
    o_ref, S_ref = _linear(q, k, v, la, S0)
    o, S = _split(q, k, v, la, S0, _bounds(L, 4))
    assert np.abs(o - o_ref).max() <= 1e-12 * np.abs(o_ref).max()
    assert np.abs(S - S_ref).max() <= 1e-12 * max(np.abs(S_ref).max(), 1e-300)


def test_planted_slips_are_caught():
    """G_t summed through t - 1 instead of t, or the fold taking the gain of the segment
    being started instead of the one just finished, must visibly break the identity."""
    L = 600
    q, k, v, la, S0 = _inputs(L, 8, 6, seed=9)
    # slow decay whose rate changes between segments, so that every segment's gain is far
    # from 0 and from the others'
    la = np.where(np.arange(L) < 300, -0.0005, -0.01)
    o_ref, S_ref = _linear(q, k, v, la, S0)
    b = _bounds(L, 4)
    o, _ = _split(q, k, v, la, S0, b, inclusive=False)
    assert np.abs(o - o_ref).max() > 1e-3 * np.abs(o_ref).max()
    o, S = _split(q, k, v, la, S0, b, fold_gain_of=lambda r: r)
    assert np.abs(S - S_ref).max() > 1e-3 * np.abs(S_ref).max()
    assert np.abs(o - o_ref).max() > 1e-3 * np.abs(o_ref).max()
