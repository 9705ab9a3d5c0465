"""Sequence-parallel (context-parallel) forward: the ranks of a process group each
own one contiguous, chunk-aligned segment of every sequence.

Over a segment of tokens the recurrence is an affine map of the state (Nyysyyan,
"Gated-DeltaNet": the WY identity for the product of the per-token factors
A_t = I - beta_t k_t k_t^T and the unrolled state S_i = gamma_i S_0 A_1..A_i + G_i):

    S_end = S_start M + L,
    M = ordered product of alpha_t (I - beta_t k_t k_t^T)   (dk x dk)
    L = the segment's final state from a zero start          (dv x dk)

Both come out of the chunk forward itself: L with S0 = 0, M with v = 0 and S0 = I
(the rows of I are carried through the same recurrence).  The forward then runs in
two phases around one exchange:

1. rank 0 runs its segment from the true S0 and publishes (-, S_end); every middle
   rank computes (M, L) of its segment; the last rank has nothing to publish.
2. all_gather of the (M, L) pairs (the exchange step: two state-sized tensors per
   rank and (sequence, head)).
3. rank r > 0 folds S_start = (((L_0) M_1 + L_1) M_2 + ...) over the ranks before it
   in one gdn_state_fold call and runs its segment from S_start.

Rank 0 runs one segment pass, a middle rank three (two of them independent), the
last rank one after the exchange.  The linear mode works the same way (there
M = (product of alpha_t) I, which the CUDA compute writes with one small kernel in place
of the M pass), except where the compute can correct a run's results for
its start state (``SegmentOps.correct``; in the linear mode the outputs are affine in
the start state with a scalar gain, o_t = o_t(0) + e^{G_t} S_start q_t): there every rank
r > 0 keeps the outputs and end state of its pass from zero and, after the exchange,
corrects them in place instead of running its segment again, so that every rank runs
one segment pass before the exchange and a cheap correction after it.  Fixed-length batches split every sequence at the same
chunk-aligned bounds; packed batches (cu_seqlens) split each member at its own bounds,
so that rank r holds a packed batch of the members' r-th segments (some of them empty:
an empty segment's map is M = I, L = 0, which the same passes give).

The compute is the CUDA library (``SegmentOps`` defaults to it); the functions take
an ``ops`` object so that the host logic can be exercised on CPU ranks.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional, Tuple

import torch


def segment_bounds(T: int, world: int, C: int) -> List[Tuple[int, int]]:
    """Contiguous token ranges [a, b) of the `world` segments of a length-T sequence.
    Every boundary is a multiple of the chunk length C (so each segment's chunks are
    the sequence's own chunks); trailing segments may be empty."""
    if world <= 0 or C <= 0 or T < 0:
        raise ValueError("segment_bounds: need world > 0, C > 0, T >= 0")
    n_chunks = -(-T // C)
    per = -(-n_chunks // world) if n_chunks else 0
    return [(min(r * per * C, T), min((r + 1) * per * C, T)) for r in range(world)]


def segment(t: Optional[torch.Tensor], bounds: Tuple[int, int]) -> Optional[torch.Tensor]:
    """Tokens [a, b) of a [B, T, ...] tensor, contiguous."""
    return None if t is None else t[:, bounds[0]:bounds[1]].contiguous()


def packed_segments(cu_seqlens: torch.Tensor, world: int, C: int):
    """The split of a packed batch: for every rank, (the indices of its tokens in the
    packed token axis, its own cu_seqlens).  Member n's tokens [cu[n], cu[n+1]) are cut
    at ``segment_bounds(len_n, world, C)``; rank r's batch is the members' r-th segments
    in member order, so that its cu_seqlens has the same N + 1 entries."""
    cu = [int(x) for x in cu_seqlens.tolist()]
    out = []
    for r in range(world):
        idx, lens = [], []
        for n in range(len(cu) - 1):
            a, b = segment_bounds(cu[n + 1] - cu[n], world, C)[r]
            idx.extend(range(cu[n] + a, cu[n] + b))
            lens.append(b - a)
        cu_r = torch.zeros(len(lens) + 1, dtype=torch.int32)
        if lens:
            cu_r[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
        out.append((torch.tensor(idx, dtype=torch.long), cu_r))
    return out


def packed_segment(t: Optional[torch.Tensor], idx: torch.Tensor) -> Optional[torch.Tensor]:
    """The tokens `idx` of a packed [1, T, ...] tensor, contiguous."""
    return None if t is None else t[:, idx.to(t.device)].contiguous()


@dataclasses.dataclass
class SegmentOps:
    """The compute a rank runs.  forward(q, k, v, log_alpha, beta, S0, C, linear
    [, cu_seqlens]) -> (out, S_final); fold(Ms, Ls) -> S after S = L_0,
    S <- S M_i + L_i for i >= 1 (Ms [count, N, H, dk, dk] and Ls [count, N, H, dv, dk]
    stacked; M_0 not read); states are state_dtype tensors.  summary(q, k, v,
    log_alpha, beta, C, linear[, cu_seqlens]) -> (M, L, out of the L pass), if given,
    replaces the two forward calls of ``segment_summary``.  cu_seqlens is passed only
    for packed batches.  correctable(q, v, cu_seqlens) -> bool and correct(q, log_alpha,
    S_start, out, S_end), if given, are the linear mode's start-state correction: it
    turns out and S_end of a run from a zero start state into those of the run from
    S_start, in place, for the tensors correctable accepts."""
    forward: Callable
    fold: Callable
    state_dtype: torch.dtype = torch.float32
    summary: Optional[Callable] = None
    correctable: Optional[Callable] = None
    correct: Optional[Callable] = None


_side_streams = {}


def _summary_streams(device: torch.device):
    """Two side streams per device, made once (streams taken afresh per call would
    each start an empty allocator pool)."""
    key = device.index if device.index is not None else torch.cuda.current_device()
    if key not in _side_streams:
        _side_streams[key] = (torch.cuda.Stream(device=device), torch.cuda.Stream(device=device))
    return _side_streams[key]


def cuda_ops() -> SegmentOps:
    """The CUDA library's entry points (device tensors, current stream)."""
    from . import gdn

    def forward(q, k, v, log_alpha, beta, S0, C, linear, cu_seqlens=None):
        if linear:
            return gdn.linear_chunk_fwd(q, k, v, log_alpha, S0, cu_seqlens, C=C)
        return gdn.chunk_fwd(q, k, v, log_alpha, beta, S0, cu_seqlens, C=C)

    def fold(Ms, Ls):
        out = torch.empty_like(Ls[0])
        gdn.gdn_state_fold(None, Ms, Ls, out)
        return out

    def summary(q, k, v, log_alpha, beta, C, linear, cu_seqlens=None):
        # the M pass (v = 0, S0 = I) and the L pass (S0 = 0) are independent: each
        # runs on a side stream of its own and takes the SMs the other leaves free.
        # Every buffer is allocated on the caller's stream, which waits for both
        # side streams before it goes on, so no buffer is reused under them.
        B, T, H, dk = k.shape
        dv = v.shape[-1]
        N = B if cu_seqlens is None else cu_seqlens.numel() - 1
        dev = k.device
        main = torch.cuda.current_stream(dev)
        if linear:  # M = (product of alpha_t) I: one small kernel instead of the M pass
            out_l = torch.empty((B, T, H, dv), dtype=v.dtype, device=dev)
            L = torch.empty((N, H, dv, dk), dtype=torch.float32, device=dev)
            M = torch.empty((N, H, dk, dk), dtype=torch.float32, device=dev)
            gdn.gdn_linear_chunk_fwd(q, k, v, log_alpha, None, out_l, L, C, cu_seqlens,
                                     stream=main)
            gdn.gdn_linear_segment_map(log_alpha, M, B, T, cu_seqlens, stream=main)
            return M, L, out_l
        I = torch.eye(dk, dtype=torch.float32, device=dev).expand(N, H, dk, dk).contiguous()
        vz = torch.zeros((B, T, H, dk), dtype=v.dtype, device=dev)
        out_m = torch.empty((B, T, H, dk), dtype=v.dtype, device=dev)
        out_l = torch.empty((B, T, H, dv), dtype=v.dtype, device=dev)
        M = torch.empty((N, H, dk, dk), dtype=torch.float32, device=dev)
        L = torch.empty((N, H, dv, dk), dtype=torch.float32, device=dev)
        sm, sl = _summary_streams(dev)
        sm.wait_stream(main)
        sl.wait_stream(main)
        for st, vv, s0, o, sf in ((sm, vz, I, out_m, M), (sl, v, None, out_l, L)):
            if linear:
                gdn.gdn_linear_chunk_fwd(q, k, vv, log_alpha, s0, o, sf, C, cu_seqlens,
                                         stream=st)
            else:
                gdn.gdn_chunk_fwd(q, k, vv, log_alpha, beta, s0, o, sf, C, cu_seqlens,
                                  stream=st)
        main.wait_stream(sm)
        main.wait_stream(sl)
        return M, L, out_l

    def correctable(q, v, cu_seqlens=None):
        return cu_seqlens is None and gdn.gdn_linear_state_correct_supported(
            q.shape[-1], v.shape[-1], q.dtype)

    def correct(q, log_alpha, S_start, out, S_end):
        gdn.gdn_linear_state_correct(q, log_alpha, S_start, out, S_end)

    return SegmentOps(forward, fold, torch.float32, summary, correctable, correct)


def _corrects(ops: SegmentOps, linear: bool, q, v, cu_seqlens) -> bool:
    """Whether the ranks r > 0 correct their runs from zero instead of running again."""
    return bool(linear and ops.correct is not None and ops.correctable is not None
                and ops.correctable(q, v, cu_seqlens))


def _fwd(ops: SegmentOps, q, k, v, log_alpha, beta, S0, C, linear, cu_seqlens):
    if cu_seqlens is None:
        return ops.forward(q, k, v, log_alpha, beta, S0, C, linear)
    return ops.forward(q, k, v, log_alpha, beta, S0, C, linear, cu_seqlens)


def segment_summary(q, k, v, log_alpha, beta, C: int, linear: bool, ops: SegmentOps,
                    cu_seqlens: Optional[torch.Tensor] = None, with_out: bool = False):
    """(M, L) of one segment: L = final state from zero, M = final state of the same
    recurrence with v = 0 and S0 = I (dv taken as dk); one pair per sequence.  With
    with_out, (M, L, the segment's outputs from zero)."""
    if ops.summary is not None:
        if cu_seqlens is None:
            M, L, out = ops.summary(q, k, v, log_alpha, beta, C, linear)
        else:
            M, L, out = ops.summary(q, k, v, log_alpha, beta, C, linear, cu_seqlens)
        return (M, L, out) if with_out else (M, L)
    B, T, H, dk = k.shape
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    I = torch.eye(dk, dtype=ops.state_dtype, device=k.device).expand(N, H, dk, dk).contiguous()
    vz = torch.zeros((B, T, H, dk), dtype=v.dtype, device=v.device)
    out, L = _fwd(ops, q, k, v, log_alpha, beta, None, C, linear, cu_seqlens)
    _, M = _fwd(ops, q, k, vz, log_alpha, beta, I, C, linear, cu_seqlens)
    return (M, L, out) if with_out else (M, L)


def fold(Ms: torch.Tensor, Ls: torch.Tensor, r: int, ops: SegmentOps):
    """S = (((L_0) M_1 + L_1) M_2 + ...) over segments 0 .. r-1 of the stacked
    summaries: the state at the start of segment r, from rank 0's published final
    state L_0 (its M_0 is not read)."""
    return ops.fold(Ms[:r], Ls[:r])


def phase1(rank: int, world: int, q, k, v, log_alpha, beta, S0, C: int, linear: bool,
           ops: SegmentOps, cu_seqlens: Optional[torch.Tensor] = None):
    """What a rank computes before the exchange.  Returns (M, L, result) where
    (M, L) is its contribution and result = (out, S_final) for rank 0; for a rank r > 0
    that corrects its run afterwards (see ``SegmentOps.correct``), its outputs and end
    state from a zero start; else None."""
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    dev = k.device
    if rank == 0:
        out, Sf = _fwd(ops, q, k, v, log_alpha, beta, S0, C, linear, cu_seqlens)
        M = torch.zeros((N, H, dk, dk), dtype=ops.state_dtype, device=dev)  # not read
        return M, Sf, (out, Sf)
    corrects = _corrects(ops, linear, q, v, cu_seqlens)
    if rank == world - 1:  # nobody needs the last segment's map
        zM = torch.zeros((N, H, dk, dk), dtype=ops.state_dtype, device=dev)
        zL = torch.zeros((N, H, dv, dk), dtype=ops.state_dtype, device=dev)
        if corrects:  # its run from zero, corrected after the exchange
            return zM, zL, _fwd(ops, q, k, v, log_alpha, beta, None, C, linear, cu_seqlens)
        return zM, zL, None
    if corrects:
        M, L, out = segment_summary(q, k, v, log_alpha, beta, C, linear, ops, cu_seqlens,
                                    with_out=True)
        return M, L, (out, L.clone())  # L goes out in the exchange; the copy is corrected
    M, L = segment_summary(q, k, v, log_alpha, beta, C, linear, ops, cu_seqlens)
    return M, L, None


def phase2(rank: int, q, k, v, log_alpha, beta, C: int, linear: bool, ops: SegmentOps,
           Ms: torch.Tensor, Ls: torch.Tensor, result,
           cu_seqlens: Optional[torch.Tensor] = None):
    """What a rank computes after the exchange: its segment from the folded start
    state (rank 0 already has its result), or, where phase 1 kept the run from zero,
    that run corrected for the start state.  Ms, Ls stack every rank's summary."""
    if rank == 0:
        return result
    S_start = fold(Ms, Ls, rank, ops)
    if result is not None and _corrects(ops, linear, q, v, cu_seqlens):
        out, S_end = result
        ops.correct(q, log_alpha, S_start, out, S_end)
        return out, S_end
    return _fwd(ops, q, k, v, log_alpha, beta, S_start, C, linear, cu_seqlens)


def seqpar_chunk_fwd(q, k, v, log_alpha, beta, S0, C: int, group=None, linear: bool = False,
                     ops: Optional[SegmentOps] = None,
                     cu_seqlens: Optional[torch.Tensor] = None):
    """This rank's part of a sequence-parallel forward.

    q, k, v, log_alpha, beta: this rank's segment of every sequence ([B, T_r, ...],
    the r-th range of ``segment_bounds``; for a packed batch, the rank's tokens from
    ``packed_segments`` with its cu_seqlens); S0: the sequences' initial state (read
    on rank 0 only) or None.  Returns (out of this segment, state at the end of this
    segment): on the last rank that is the sequences' final state.
    """
    import torch.distributed as dist
    ops = ops or cuda_ops()
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    M, L, res = phase1(rank, world, q, k, v, log_alpha, beta, S0, C, linear, ops, cu_seqlens)
    Ms = [torch.empty_like(M) for _ in range(world)]
    Ls = [torch.empty_like(L) for _ in range(world)]
    dist.all_gather(Ms, M.contiguous(), group=group)
    dist.all_gather(Ls, L.contiguous(), group=group)
    return phase2(rank, q, k, v, log_alpha, beta, C, linear, ops, torch.stack(Ms),
                  torch.stack(Ls), res, cu_seqlens)


def emulate(q, k, v, log_alpha, beta, S0, C: int, world: int, linear: bool = False,
            ops: Optional[SegmentOps] = None, cu_seqlens: Optional[torch.Tensor] = None):
    """Run every rank of a `world`-rank sequence-parallel forward in this process,
    one after another (the exchange is a list).  Returns (out of the whole
    sequences, final state); for checking the split on one device."""
    ops = ops or cuda_ops()
    if cu_seqlens is None:
        bounds = segment_bounds(k.shape[1], world, C)
        segs = [[segment(t, b) for t in (q, k, v, log_alpha, beta)] for b in bounds]
        cus = [None] * world
    else:
        parts = packed_segments(cu_seqlens, world, C)
        segs = [[packed_segment(t, idx) for t in (q, k, v, log_alpha, beta)]
                for idx, _ in parts]
        cus = [cu.to(cu_seqlens.device) for _, cu in parts]
    first = [phase1(r, world, *segs[r], S0, C, linear, ops, cus[r]) for r in range(world)]
    Ms = torch.stack([M for M, _, _ in first])
    Ls = torch.stack([L for _, L, _ in first])
    outs, Sf = [], None
    for r in range(world):
        out, Sf = phase2(r, *segs[r], C, linear, ops, Ms, Ls, first[r][2], cus[r])
        outs.append(out)
    if cu_seqlens is None:
        return torch.cat(outs, dim=1), Sf
    # the ranks' packed outputs back to the packed token order
    full = torch.empty((1, k.shape[1]) + tuple(outs[0].shape[2:]), dtype=outs[0].dtype,
                       device=outs[0].device)
    for (idx, _), o in zip(parts, outs):
        full[:, idx.to(full.device)] = o
    return full, Sf
