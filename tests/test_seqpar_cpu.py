"""Sequence-parallel forward on CPU ranks (gloo): the host logic of
chunkwise_gated_deltanet_gb300.seqpar with the fp64 oracle as each rank's compute.

The split rests on the state map of a segment being affine, S_end = S_start M + L
(Nyysyyan, "Gated-DeltaNet": unrolled state and WY identity); the first tests pin
that property on the oracle itself, the rest check that segment bounds, the
exchange and the fold reproduce the unsplit oracle run.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from chunkwise_gated_deltanet_gb300 import seqpar
from oracle import recurrence as R

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _inputs(B=2, T=150, H=2, dk=16, dv=16, seed=0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T, H, dk, generator=g)
    k = torch.randn(B, T, H, dk, generator=g)
    q, k = q / q.norm(dim=-1, keepdim=True), k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(B, T, H, dv, generator=g)
    beta = torch.sigmoid(torch.randn(B, T, H, generator=g))
    la = -torch.nn.functional.softplus(-(torch.randn(B, T, H, generator=g) + 2.0))
    S0 = 0.1 * torch.randn(B, H, dv, dk, generator=g)
    return q, k, v, la, beta, S0


def _oracle_forward(q, k, v, la, beta, S0, C, linear, cu_seqlens=None):
    """Each (sequence, head) through the fp64 per-token recurrence (C is irrelevant
    to the definition).  Linear mode: erase 0, write 1.  With cu_seqlens, the members
    of a packed [1, T, ...] batch."""
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        spans = [(b, 0, T) for b in range(B)]
    else:
        cu = [int(x) for x in cu_seqlens.tolist()]
        spans = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    out = np.zeros((B, T, H, dv))
    Sf = np.zeros((len(spans), H, dv, dk))
    for n, (b, t0, t1) in enumerate(spans):
        for h in range(H):
            s0 = None if S0 is None else S0[n, h].double().numpy()
            kw = {}
            if linear:
                kw = dict(erase=np.zeros(t1 - t0), write=np.ones(t1 - t0))
            o, S = R.gdn_sequence(q[b, t0:t1, h].double().numpy(), k[b, t0:t1, h].double().numpy(),
                                  v[b, t0:t1, h].double().numpy(), la[b, t0:t1, h].double().numpy(),
                                  beta[b, t0:t1, h].double().numpy(), s0, **kw)
            out[b, t0:t1, h], Sf[n, h] = o, S
    return torch.from_numpy(out), torch.from_numpy(Sf)


def _oracle_fold(Ms, Ls):
    S = Ls[0].clone()
    for M, L in zip(Ms[1:], Ls[1:]):
        S = S @ M + L
    return S


ORACLE_OPS = seqpar.SegmentOps(_oracle_forward, _oracle_fold, torch.float64)


def _oracle_correct(q, la, S_start, out, S_end):
    """The linear mode's start-state correction from its formula, fp64, in place:
    o_t += e^{G_t} S_start q_t (G_t = sum of log alpha through t), S_end += e^{G_last}
    S_start ([N] Mamba2: the state is the decayed sum of the writes)."""
    B, T, H, _ = q.shape
    for b in range(B):
        for h in range(H):
            G = np.cumsum(la[b, :, h].double().numpy()) if la is not None else np.zeros(T)
            Ss = S_start[b, h].double().numpy()
            out[b, :, h] += torch.from_numpy(np.exp(G)[:, None] * (q[b, :, h].double().numpy()
                                                                  @ Ss.T))
            if S_end is not None:
                S_end[b, h] += torch.from_numpy(np.exp(G[-1] if T else 0.0) * Ss)


# the same compute with the linear mode's correction (fixed-length batches)
CORRECTING_OPS = seqpar.SegmentOps(_oracle_forward, _oracle_fold, torch.float64,
                                   correctable=lambda q, v, cu=None: cu is None,
                                   correct=_oracle_correct)


# ------------------------------------------------------ the affine property --

@pytest.mark.parametrize("linear", [False, True])
def test_segment_state_map_is_affine(linear):
    """S_end(X) = X M + L for any start X, with M from v = 0 and S0 = I and L from
    S0 = 0: the property the split rests on."""
    q, k, v, la, beta, _ = _inputs(B=1, T=40, H=1, dk=8, dv=5, seed=1)
    M, L = seqpar.segment_summary(q, k, v, la, beta, 16, linear, ORACLE_OPS)
    X = torch.randn(1, 1, 5, 8, generator=torch.Generator().manual_seed(2), dtype=torch.float64)
    _, S_end = _oracle_forward(q, k, v, la, beta, X, 16, linear)
    assert torch.allclose(S_end, X @ M + L, rtol=1e-12, atol=1e-12)
    if linear:  # the Mamba2 map is a scalar decay
        gamma = torch.exp(la.double().sum(1))[0, 0]
        assert torch.allclose(M[0, 0], gamma * torch.eye(8, dtype=torch.float64), atol=1e-14)


def test_transition_product_by_brute_force():
    """M equals the explicit ordered product of alpha_t (I - beta_t k_t k_t^T)."""
    q, k, v, la, beta, _ = _inputs(B=1, T=9, H=1, dk=6, dv=3, seed=3)
    M, _ = seqpar.segment_summary(q, k, v, la, beta, 16, False, ORACLE_OPS)
    P = np.eye(6)
    for t in range(9):
        kt = k[0, t, 0].double().numpy()
        P = P @ (np.exp(float(la[0, t, 0])) * (np.eye(6) - float(beta[0, t, 0]) * np.outer(kt, kt)))
    assert np.abs(M[0, 0].numpy() - P).max() < 1e-13


# ------------------------------------------------------------- segmentation --

@pytest.mark.parametrize("T,world,C", [(0, 3, 16), (1, 4, 16), (150, 2, 16), (150, 3, 64),
                                       (4096, 8, 64), (65, 5, 32), (64, 1, 64)])
def test_segment_bounds(T, world, C):
    b = seqpar.segment_bounds(T, world, C)
    assert len(b) == world and b[0][0] == 0 and b[-1][1] == T
    for (a0, a1), (b0, _) in zip(b, b[1:]):
        assert a1 == b0
    for a, e in b:
        assert 0 <= a <= e <= T and (a % C == 0 or a == T)


# --------------------------------------------------- one process, all ranks --

@pytest.mark.parametrize("world", [1, 2, 3, 5])
@pytest.mark.parametrize("linear", [False, True])
@pytest.mark.parametrize("ops", ["plain", "correcting"])
def test_emulated_split_matches_unsplit(world, linear, ops):
    """Every rank in turn; in the linear mode with a correcting compute the ranks r > 0
    keep their runs from zero and correct them after the exchange."""
    q, k, v, la, beta, S0 = _inputs(seed=world)
    o = ORACLE_OPS if ops == "plain" else CORRECTING_OPS
    out, Sf = seqpar.emulate(q, k, v, la, beta, S0, 16, world, linear, o)
    ref_o, ref_S = _oracle_forward(q, k, v, la, beta, S0, 16, linear)
    assert torch.allclose(out, ref_o, rtol=1e-10, atol=1e-12)
    assert torch.allclose(Sf, ref_S, rtol=1e-10, atol=1e-12)


PACKED_LENS = [5, 0, 70, 130, 1, 33]


def _packed_inputs(seed=0):
    q, k, v, la, beta, _ = _inputs(B=1, T=sum(PACKED_LENS), seed=seed)
    g = torch.Generator().manual_seed(seed + 100)
    S0 = 0.1 * torch.randn(len(PACKED_LENS), 2, 16, 16, generator=g)
    cu = torch.tensor([0] + list(np.cumsum(PACKED_LENS)), dtype=torch.int32)
    return q, k, v, la, beta, S0, cu


def test_packed_segments_cover_each_member_in_order():
    cu = torch.tensor([0] + list(np.cumsum(PACKED_LENS)), dtype=torch.int32)
    for world in (1, 2, 3, 4):
        parts = seqpar.packed_segments(cu, world, 16)
        seen = torch.cat([idx for idx, _ in parts])
        assert sorted(seen.tolist()) == list(range(int(cu[-1])))
        for n, L in enumerate(PACKED_LENS):
            pieces = [(int(c[n + 1] - c[n])) for _, c in parts]
            assert sum(pieces) == L
            b = seqpar.segment_bounds(L, world, 16)
            assert pieces == [e - a for a, e in b]


@pytest.mark.parametrize("world", [1, 2, 3, 5])
@pytest.mark.parametrize("linear", [False, True])
def test_emulated_packed_split_matches_unsplit(world, linear):
    q, k, v, la, beta, S0, cu = _packed_inputs(seed=world)
    out, Sf = seqpar.emulate(q, k, v, la, beta, S0, 16, world, linear, ORACLE_OPS, cu)
    ref_o, ref_S = _oracle_forward(q, k, v, la, beta, S0, 16, linear, cu)
    assert torch.allclose(out, ref_o, rtol=1e-10, atol=1e-12)
    assert torch.allclose(Sf, ref_S, rtol=1e-10, atol=1e-12)


# -------------------------------------------------------- gloo, real ranks --

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, linear, queue, correcting=False):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from chunkwise_gated_deltanet_gb300 import seqpar as sp
    from tests import test_seqpar_cpu as me
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v, la, beta, S0 = me._inputs(seed=7)
    bnd = sp.segment_bounds(q.shape[1], world, 16)[rank]
    seg = [sp.segment(t, bnd) for t in (q, k, v, la, beta)]
    out, Sf = sp.seqpar_chunk_fwd(*seg, S0 if rank == 0 else None, 16, linear=linear,
                                  ops=me.CORRECTING_OPS if correcting else me.ORACLE_OPS)
    queue.put((rank, bnd, out.numpy(), Sf.numpy()))
    dist.barrier()
    dist.destroy_process_group()


def _packed_rank_main(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from chunkwise_gated_deltanet_gb300 import seqpar as sp
    from tests import test_seqpar_cpu as me
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v, la, beta, S0, cu = me._packed_inputs(seed=9)
    idx, cu_r = sp.packed_segments(cu, world, 16)[rank]
    seg = [sp.packed_segment(t, idx) for t in (q, k, v, la, beta)]
    out, Sf = sp.seqpar_chunk_fwd(*seg, S0 if rank == 0 else None, 16, ops=me.ORACLE_OPS,
                                  cu_seqlens=cu_r)
    queue.put((rank, idx.numpy(), out.numpy(), Sf.numpy()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_packed_match_unsplit(world):
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_packed_rank_main, args=(r, world, port, queue))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((queue.get(timeout=300) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    q, k, v, la, beta, S0, cu = _packed_inputs(seed=9)
    ref_o, ref_S = _oracle_forward(q, k, v, la, beta, S0, 16, False, cu)
    got = np.zeros(ref_o.shape)
    for _, idx, o, _ in res:
        got[:, idx] = o
    assert np.allclose(got, ref_o.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(res[-1][3], ref_S.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("world,linear,correcting", [(2, False, False), (3, False, False),
                                                    (3, True, False), (2, True, True),
                                                    (3, True, True)])
def test_gloo_ranks_match_unsplit(world, linear, correcting):
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, linear, queue, correcting))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((queue.get(timeout=300) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    q, k, v, la, beta, S0 = _inputs(seed=7)
    ref_o, ref_S = _oracle_forward(q, k, v, la, beta, S0, 16, linear)
    got_o = np.concatenate([r[2] for r in res], axis=1)
    assert np.allclose(got_o, ref_o.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(res[-1][3], ref_S.numpy(), rtol=1e-10, atol=1e-12)
    assert [r[1] for r in res] == seqpar.segment_bounds(q.shape[1], world, 16)


def test_correcting_ranks_run_their_segment_once():
    """With the linear mode's correction, a rank r > 0 runs its segment once from zero
    (a middle rank's M pass beside it) before the exchange and no pass after it."""
    q, k, v, la, beta, S0 = _inputs(seed=3)
    calls = []

    def counting_forward(*a, **kw):
        calls.append(a[5] is None)  # S0 argument: None = from zero
        return _oracle_forward(*a, **kw)

    ops = seqpar.SegmentOps(counting_forward, _oracle_fold, torch.float64,
                            correctable=lambda q, v, cu=None: cu is None,
                            correct=_oracle_correct)
    world = 4
    bounds = seqpar.segment_bounds(q.shape[1], world, 16)
    segs = [[seqpar.segment(t, b) for t in (q, k, v, la, beta)] for b in bounds]
    first = [seqpar.phase1(r, world, *segs[r], S0, 16, True, ops) for r in range(world)]
    n1 = len(calls)
    assert n1 == 1 + 2 * (world - 2) + 1  # rank 0; (L, M) per middle rank; the last rank
    Ms = torch.stack([m for m, _, _ in first])
    Ls = torch.stack([l for _, l, _ in first])
    outs = [seqpar.phase2(r, *segs[r], 16, True, ops, Ms, Ls, first[r][2])
            for r in range(world)]
    assert len(calls) == n1  # no pass after the exchange
    ref_o, ref_S = _oracle_forward(q, k, v, la, beta, S0, 16, True)
    assert torch.allclose(torch.cat([o for o, _ in outs], dim=1), ref_o, rtol=1e-10,
                          atol=1e-12)
    assert torch.allclose(outs[-1][1], ref_S, rtol=1e-10, atol=1e-12)
