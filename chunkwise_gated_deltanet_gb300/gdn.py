"""Thin ctypes binding of ``libgdn.so`` (see include/gdn.h).

Argument marshalling only: every step of the forward runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current CUDA stream.  There is
no CPU fallback; if the library is missing or the tensors are not on a CUDA
device the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK, GDN_EINVAL, GDN_EDTYPE, GDN_ELAUNCH, GDN_ETIMEOUT, GDN_ECUDA = range(6)
GDN_F32, GDN_BF16 = 0, 1
GDN_PATH_NONE, GDN_PATH_SIMT, GDN_PATH_TCGEN05, GDN_PATH_TF32 = 0, 1, 2, 3
GDN_BWD_AUTO, GDN_BWD_TOKENS, GDN_BWD_CHUNKED = 0, 1, 2
EXPORTS = ("gdn_chunk_fwd", "gdn_chunk_fwd_host", "gdn_chunk_fwd_host_workspace_bytes",
           "gdn_decode_step_host", "gdn_decode_step_host_workspace_bytes",
           "gdn_chunk_bwd", "gdn_chunk_bwd_ex", "gdn_chunk_bwd_workspace_bytes", "gdn_bwd_select_path",
           "gdn_linear_chunk_fwd", "gdn_decode_step", "gdn_state_fold", "gdn_select_path", "gdn_launches_per_call",
           "gdn_check_status", "gdn_selftest_wait_timeout", "gdn_last_error", "gdn_version",
           "gdn_chunk_bwd_noalloc", "gdn_chunk_bwd_noalloc_max_scratch_bytes")


class GdnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"[gdn status {status}] {msg}")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libgdn.so (built by ``chunkwise_gated_deltanet_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libgdn.so is not built at {path}; run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.gdn_chunk_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, P, I, I, P]
    lib.gdn_chunk_fwd.restype = I
    lib.gdn_linear_chunk_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P, I, I, P]
    lib.gdn_linear_chunk_fwd.restype = I
    lib.gdn_decode_step.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P]
    lib.gdn_decode_step.restype = I
    Z = ctypes.c_size_t
    lib.gdn_chunk_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, Z,
                                  I, I, I, I, I, P, I, I, P]
    lib.gdn_chunk_bwd.restype = I
    lib.gdn_chunk_bwd_ex.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, Z,
                                     I, I, I, I, I, P, I, I, I, P]
    lib.gdn_chunk_bwd_ex.restype = I
    lib.gdn_chunk_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                          I, I, I, I, I, P, I, I, P]
    lib.gdn_chunk_bwd_noalloc.restype = I
    lib.gdn_chunk_bwd_noalloc_max_scratch_bytes.argtypes = []
    lib.gdn_chunk_bwd_noalloc_max_scratch_bytes.restype = ctypes.c_size_t
    lib.gdn_bwd_select_path.argtypes = [I, I, I]
    lib.gdn_bwd_select_path.restype = I
    lib.gdn_chunk_bwd_workspace_bytes.argtypes = [I, I, I, I, I, I]
    lib.gdn_chunk_bwd_workspace_bytes.restype = Z
    lib.gdn_chunk_fwd_host.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, Z, P]
    lib.gdn_chunk_fwd_host.restype = I
    lib.gdn_chunk_fwd_host_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I, I]
    lib.gdn_chunk_fwd_host_workspace_bytes.restype = Z
    lib.gdn_decode_step_host.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P, Z, P]
    lib.gdn_decode_step_host.restype = I
    lib.gdn_decode_step_host_workspace_bytes.argtypes = [I, I, I, I, I]
    lib.gdn_decode_step_host_workspace_bytes.restype = Z
    lib.gdn_state_fold.argtypes = [P, P, P, I, P, I, I, I, P]
    lib.gdn_state_fold.restype = I
    lib.gdn_linear_state_correct.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P]
    lib.gdn_linear_state_correct.restype = I
    lib.gdn_linear_state_correct_supported.argtypes = [I, I, I]
    lib.gdn_linear_state_correct_supported.restype = I
    lib.gdn_linear_segment_map.argtypes = [P, P, I, I, I, I, P, I, P]
    lib.gdn_linear_segment_map.restype = I
    for name in ("gdn_select_path", "gdn_launches_per_call"):
        getattr(lib, name).argtypes = [I, I, I, I]
        getattr(lib, name).restype = I
    lib.gdn_check_status.argtypes = [P]
    lib.gdn_check_status.restype = I
    lib.gdn_selftest_wait_timeout.argtypes = [P]
    lib.gdn_selftest_wait_timeout.restype = I
    lib.gdn_last_error.argtypes = []
    lib.gdn_last_error.restype = ctypes.c_char_p
    lib.gdn_version.restype = I
    _lib = lib
    return lib


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return GDN_F32
    if dt == torch.bfloat16:
        return GDN_BF16
    raise TypeError(f"q/k/v must be float32 or bfloat16, got {dt}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(status: int):
    if status != GDN_OK:
        raise GdnError(status, load_library().gdn_last_error().decode(errors="replace"))


def gdn_version() -> int:
    return load_library().gdn_version()


def gdn_select_path(dk: int, dv: int, C: int, dtype: torch.dtype) -> int:
    return load_library().gdn_select_path(dk, dv, C, _dtype_code(dtype))


def gdn_launches_per_call(dk: int, dv: int, C: int, dtype: torch.dtype) -> int:
    return load_library().gdn_launches_per_call(dk, dv, C, _dtype_code(dtype))


def gdn_linear_split_segments(N: int, H: int, T: int, dk: int, dv: int, C: int,
                              dtype: torch.dtype) -> int:
    """Segments per sequence of the linear mode's split on the current device (1: none)."""
    return load_library().gdn_linear_split_segments(N, H, T, dk, dv, C, _dtype_code(dtype))


def gdn_check_status(stream: Optional[torch.cuda.Stream] = None) -> None:
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(load_library().gdn_check_status(ctypes.c_void_p(s.cuda_stream)))


def _chunk_call(entry: str, q, k, v, log_alpha, beta, S0, out, S_final, C: int,
                cu_seqlens, stream) -> None:
    lib = load_library()
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    tensors = [q, k, v, log_alpha, beta, S0, out, S_final, cu_seqlens]
    for t in tensors:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{entry}: every tensor must be a contiguous CUDA tensor")
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    code = _dtype_code(v.dtype)
    if q.dtype != v.dtype or k.dtype != v.dtype or out.dtype != v.dtype:
        raise TypeError("q, k, v and out must share one dtype")
    for name, t in (("log_alpha", log_alpha), ("beta", beta), ("S0", S0), ("S_final", S_final)):
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    n_seqs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    s = ctypes.c_void_p((stream if stream is not None
                         else torch.cuda.current_stream(v.device)).cuda_stream)
    # the library resolves tensor maps, per-device state and streams on the current
    # device, which must be the tensors' device
    with torch.cuda.device(v.device):
        if entry == "gdn_chunk_fwd":
            st = lib.gdn_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                   _ptr(S0), _ptr(out), _ptr(S_final), B, H, T, dk, dv, C,
                                   _ptr(cu_seqlens), n_seqs, code, s)
        else:
            st = lib.gdn_linear_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(S0),
                                          _ptr(out), _ptr(S_final), B, H, T, dk, dv, C,
                                          _ptr(cu_seqlens), n_seqs, code, s)
    _check(st)


def gdn_selftest_wait_timeout(stream: Optional[torch.cuda.Stream] = None) -> None:
    """Launch the failure-detection self-test (a bounded wait that nothing satisfies);
    the next gdn_check_status on the stream raises GdnError(GDN_ETIMEOUT)."""
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(load_library().gdn_selftest_wait_timeout(ctypes.c_void_p(s.cuda_stream)))


def gdn_chunk_fwd(q, k, v, log_alpha, beta, S0, out, S_final, C: int,
                  cu_seqlens: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None) -> None:
    """Tensor-level call of the C entry point of the same name.

    Shapes: q, k [B, T, H, dk]; v, out [B, T, H, dv]; log_alpha, beta [B, T, H]
    fp32; S0, S_final [N, H, dv, dk] fp32 or None; cu_seqlens int32 [N+1] or None.
    All tensors contiguous on one CUDA device.  Launches on ``stream`` (default:
    the current torch stream) and returns without synchronising.
    """
    _chunk_call("gdn_chunk_fwd", q, k, v, log_alpha, beta, S0, out, S_final, C, cu_seqlens,
                stream)


def gdn_linear_chunk_fwd(q, k, v, log_alpha, S0, out, S_final, C: int,
                         cu_seqlens: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None) -> None:
    """Tensor-level call of the C entry point of the same name: the linear mode
    S_t = alpha_t S_{t-1} + v_t k_t^T (no beta; log_alpha None means alpha = 1).
    Shapes and stream behaviour as in ``gdn_chunk_fwd``."""
    _chunk_call("gdn_linear_chunk_fwd", q, k, v, log_alpha, None, S0, out, S_final, C,
                cu_seqlens, stream)


def chunk_fwd(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, C: int = 64,
              output_final_state: bool = True,
              pieces: Optional[int] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Allocate the outputs and run the forward.  Returns (out, S_final or None).

    Device tensors: runs on the current stream and returns device tensors.
    Host tensors (pinned, so that the copies are asynchronous): runs on the current
    CUDA device and returns pinned host tensors, synchronising before it returns.  A
    fixed-length batch goes through the native gdn_chunk_fwd_host: `pieces`
    consecutive token ranges (default: up to 4 of whole chunks), each starting from
    the previous one's final state, so that the copies of one range overlap the
    computation of the next.
    """
    if v.is_cuda:
        B, T, H, dk = k.shape
        dv = v.shape[-1]
        N = B if cu_seqlens is None else cu_seqlens.numel() - 1
        out = torch.empty((B, T, H, dv), dtype=v.dtype, device=v.device)
        Sf = (torch.empty((N, H, dv, dk), dtype=torch.float32, device=v.device)
              if output_final_state else None)
        gdn_chunk_fwd(q, k, v, log_alpha, beta, S0, out, Sf, C, cu_seqlens)
        return out, Sf
    return _chunk_fwd_host(q, k, v, log_alpha, beta, S0, cu_seqlens, C, output_final_state,
                           pieces, linear=False)


_host_ws = threading.local()


def _host_workspace(dev: torch.device, nbytes: int) -> torch.Tensor:
    """A device scratch buffer for the host path, kept per thread and device."""
    cache = getattr(_host_ws, "bufs", None)
    if cache is None:
        cache = _host_ws.bufs = {}
    t = cache.get(dev.index)
    if t is None or t.numel() < nbytes:
        t = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
        cache[dev.index] = t
    return t


def _chunk_fwd_host(q, k, v, log_alpha, beta, S0, cu_seqlens, C, output_final_state, pieces,
                    linear: bool):
    dev = torch.device("cuda", torch.cuda.current_device())
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    out_h = torch.empty((B, T, H, dv), dtype=v.dtype, pin_memory=True)
    Sf_h = (torch.empty((N, H, dv, dk), dtype=torch.float32, pin_memory=True)
            if output_final_state else None)
    stream = torch.cuda.current_stream(dev)
    if cu_seqlens is None:
        # the native pipelined path: copies overlap the computation, range by range
        lib = load_library()
        code = _dtype_code(v.dtype)
        for t in (q, k, v, log_alpha, beta, S0):
            if t is not None and (t.is_cuda or not t.is_contiguous()):
                raise ValueError("chunk_fwd: host inputs must be contiguous CPU tensors")
        npieces = pieces or 4
        nbytes = lib.gdn_chunk_fwd_host_workspace_bytes(B, H, T, dk, dv, C, code, npieces,
                                                        int(linear))
        ws = _host_workspace(dev, nbytes)
        _check(lib.gdn_chunk_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                      None if linear else _ptr(beta), _ptr(S0), _ptr(out_h),
                                      _ptr(Sf_h), B, H, T, dk, dv, C, code, npieces, _ptr(ws),
                                      ws.numel(), ctypes.c_void_p(stream.cuda_stream)))
        return out_h, Sf_h
    # packed batches: copy in, run, copy back
    mv = lambda t: None if t is None else t.to(dev, non_blocking=True)
    qd, kd, vd, lad, bed, S0d, cud = map(mv, (q, k, v, log_alpha, beta, S0, cu_seqlens))
    out = torch.empty((B, T, H, dv), dtype=v.dtype, device=dev)
    Sf = torch.empty((N, H, dv, dk), dtype=torch.float32, device=dev) if output_final_state else None
    if linear:
        gdn_linear_chunk_fwd(qd, kd, vd, lad, S0d, out, Sf, C, cud)
    else:
        gdn_chunk_fwd(qd, kd, vd, lad, bed, S0d, out, Sf, C, cud)
    out_h.copy_(out, non_blocking=True)
    if Sf_h is not None:
        Sf_h.copy_(Sf, non_blocking=True)
    stream.synchronize()
    return out_h, Sf_h


def linear_chunk_fwd(q, k, v, log_alpha=None, S0=None, cu_seqlens=None, C: int = 64,
                     output_final_state: bool = True, pieces: Optional[int] = None):
    """Allocate the outputs and run the linear-mode forward.  Returns (out, S_final or
    None).  Device tensors run on the current stream; pinned host tensors take the
    pipelined host path of ``chunk_fwd``."""
    if not v.is_cuda:
        return _chunk_fwd_host(q, k, v, log_alpha, None, S0, cu_seqlens, C, output_final_state,
                               pieces, linear=True)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    out = torch.empty((B, T, H, dv), dtype=v.dtype, device=v.device)
    Sf = torch.empty((N, H, dv, dk), dtype=torch.float32, device=v.device) if output_final_state else None
    gdn_linear_chunk_fwd(q, k, v, log_alpha, S0, out, Sf, C, cu_seqlens)
    return out, Sf


def gdn_decode_step(q, k, v, log_alpha, beta, S, out,
                    stream: Optional[torch.cuda.Stream] = None) -> None:
    """Tensor-level call of the C entry point of the same name (one token per
    (sequence, head), state updated in place).

    Shapes: q, k [N, H, dk]; v, out [N, H, dv]; log_alpha, beta [N, H] fp32;
    S [N, H, dv, dk] fp32.  All tensors contiguous on one CUDA device.  Launches on
    ``stream`` (default: the current torch stream) and returns without synchronising.
    """
    lib = load_library()
    N, H, dk = k.shape
    dv = v.shape[-1]
    for t in (q, k, v, log_alpha, beta, S, out):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("gdn_decode_step: every tensor must be a contiguous CUDA tensor")
    code = _dtype_code(v.dtype)
    if q.dtype != v.dtype or k.dtype != v.dtype or out.dtype != v.dtype:
        raise TypeError("q, k, v and out must share one dtype")
    for name, t in (("log_alpha", log_alpha), ("beta", beta), ("S", S)):
        if t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    s = stream if stream is not None else torch.cuda.current_stream(v.device)
    with torch.cuda.device(v.device):
        st = lib.gdn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S),
                                 _ptr(out), N, H, dk, dv, code, ctypes.c_void_p(s.cuda_stream))
    _check(st)


def decode_step(q, k, v, log_alpha, beta, S, pieces: int = 4) -> torch.Tensor:
    """One decode token for every (sequence, head): updates S in place and returns the
    output [N, H, dv] (same dtype as v).  Device tensors run on the current stream;
    pinned host tensors go through gdn_decode_step_host (copies pipelined over
    `pieces` slices of sequences) and the call returns with S and the output written."""
    if not v.is_cuda:
        lib = load_library()
        N, H, dk = k.shape
        dv = v.shape[-1]
        code = _dtype_code(v.dtype)
        for t in (q, k, v, log_alpha, beta, S):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("decode_step: host inputs must be contiguous CPU tensors")
        out = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
        dev = torch.device("cuda", torch.cuda.current_device())
        ws = _host_workspace(dev, lib.gdn_decode_step_host_workspace_bytes(N, H, dk, dv, code))
        s = torch.cuda.current_stream(dev)
        _check(lib.gdn_decode_step_host(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                        _ptr(S), _ptr(out), N, H, dk, dv, code, pieces, _ptr(ws),
                                        ws.numel(), ctypes.c_void_p(s.cuda_stream)))
        return out
    out = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    gdn_decode_step(q, k, v, log_alpha, beta, S, out)
    return out


def gdn_state_fold(S_in, M, L, S_out, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Tensor-level call of the C entry point of the same name: S <- S M_i + L_i for
    every step i, from S_in (None: zeros) into S_out.  M [count, ..., dk, dk] and
    L [count, ..., dv, dk] stack the steps; S_in, S_out [..., dv, dk].  fp32
    contiguous CUDA tensors; returns without synchronising."""
    lib = load_library()
    count = L.shape[0]
    dv, dk = L.shape[-2], L.shape[-1]
    units = L[0].numel() // (dv * dk)
    for name, t in (("S_in", S_in), ("M", M), ("L", L), ("S_out", S_out)):
        if t is None:
            continue
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.float32:
            raise ValueError(f"gdn_state_fold: {name} must be a contiguous fp32 CUDA tensor")
    if M is not None and (M.shape[0] != count or M.numel() != count * units * dk * dk):
        raise ValueError("gdn_state_fold: M and L do not describe the same steps and states")
    for name, t in (("S_in", S_in), ("S_out", S_out)):
        if t is not None and t.numel() != units * dv * dk:
            raise ValueError(f"gdn_state_fold: {name} does not hold one state per unit")
    s = stream if stream is not None else torch.cuda.current_stream(L.device)
    with torch.cuda.device(L.device):
        st = lib.gdn_state_fold(_ptr(S_in), _ptr(M), _ptr(L), count, _ptr(S_out), units, dv, dk,
                                ctypes.c_void_p(s.cuda_stream))
    _check(st)


def gdn_linear_state_correct_supported(dk: int, dv: int, dtype: torch.dtype) -> bool:
    return bool(load_library().gdn_linear_state_correct_supported(dk, dv, _dtype_code(dtype)))


def _correct_shapes(q, log_alpha, S_start, out, S_end) -> None:
    """gdn_linear_state_correct's shapes and dtypes (the C entry point sees only
    pointers): out like q's dtype [B, T, H, dv]; S_start, S_end fp32 [B, H, dv, dk];
    log_alpha fp32 [B, T, H]."""
    B, T, H, dk = q.shape
    dv = out.shape[-1]
    want = {"out": (out, (B, T, H, dv), q.dtype),
            "S_start": (S_start, (B, H, dv, dk), torch.float32),
            "log_alpha": (log_alpha, (B, T, H), torch.float32),
            "S_end": (S_end, (B, H, dv, dk), torch.float32)}
    for name, (t, shape, dt) in want.items():
        if t is not None and (tuple(t.shape) != shape or t.dtype != dt):
            raise ValueError(f"gdn_linear_state_correct: {name} must be {dt} of shape {shape}, "
                             f"got {t.dtype} {tuple(t.shape)}")


def _segment_map_shapes(log_alpha, M, B: int, T: int, cu_seqlens) -> None:
    """gdn_linear_segment_map's shapes and dtypes (the C entry point sees only pointers)."""
    if M.dim() != 4 or M.shape[2] != M.shape[3] or M.dtype != torch.float32:
        raise ValueError("gdn_linear_segment_map: M must be fp32 [N, H, dk, dk]")
    N, H = M.shape[0], M.shape[1]
    if log_alpha is not None and (tuple(log_alpha.shape) != (B, T, H) or
                                  log_alpha.dtype != torch.float32):
        raise ValueError(f"gdn_linear_segment_map: log_alpha must be fp32 of shape {(B, T, H)}")
    if cu_seqlens is None and N != B:
        raise ValueError("gdn_linear_segment_map: M must hold one map per sequence (N = B)")
    if cu_seqlens is not None and (cu_seqlens.dtype != torch.int32 or
                                   cu_seqlens.numel() != N + 1 or B != 1):
        raise ValueError("gdn_linear_segment_map: cu_seqlens must be int32 with N + 1 "
                         "entries (B = 1)")


def gdn_linear_state_correct(q, log_alpha, S_start, out, S_end,
                             stream: Optional[torch.cuda.Stream] = None) -> None:
    """Tensor-level call of the C entry point of the same name: out and S_end of a
    linear-mode run from a zero start state become the run's results from S_start
    (in place).  q [B, T, H, dk] bf16; log_alpha [B, T, H] fp32 or None; S_start,
    S_end (or None) [B, H, dv, dk] fp32; out [B, T, H, dv] bf16.  Contiguous CUDA
    tensors; returns without synchronising."""
    lib = load_library()
    B, T, H, dk = q.shape
    dv = out.shape[-1]
    for name, t in (("q", q), ("log_alpha", log_alpha), ("S_start", S_start), ("out", out),
                    ("S_end", S_end)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"gdn_linear_state_correct: {name} must be a contiguous CUDA tensor")
    _correct_shapes(q, log_alpha, S_start, out, S_end)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        st = lib.gdn_linear_state_correct(_ptr(q), _ptr(log_alpha), _ptr(S_start), _ptr(out),
                                          _ptr(S_end), B, H, T, dk, dv, _dtype_code(q.dtype),
                                          ctypes.c_void_p(s.cuda_stream))
    _check(st)


def gdn_linear_segment_map(log_alpha, M, B: int, T: int, cu_seqlens=None,
                           stream: Optional[torch.cuda.Stream] = None) -> None:
    """Tensor-level call of the C entry point of the same name: M [N, H, dk, dk] fp32
    gets (product of alpha_t over each sequence) I.  log_alpha [B, T, H] fp32 or None
    (alpha = 1); cu_seqlens int32 or None.  Returns without synchronising."""
    lib = load_library()
    N, H, dk = M.shape[0], M.shape[1], M.shape[-1]
    for name, t in (("log_alpha", log_alpha), ("M", M), ("cu_seqlens", cu_seqlens)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"gdn_linear_segment_map: {name} must be a contiguous CUDA tensor")
    _segment_map_shapes(log_alpha, M, B, T, cu_seqlens)
    s = stream if stream is not None else torch.cuda.current_stream(M.device)
    with torch.cuda.device(M.device):
        st = lib.gdn_linear_segment_map(_ptr(log_alpha), _ptr(M), B, H, T, dk, _ptr(cu_seqlens),
                                        N, ctypes.c_void_p(s.cuda_stream))
    _check(st)


def gdn_chunk_bwd_workspace_bytes(B: int, H: int, T: int, dk: int, dv: int, n_seqs: int) -> int:
    """Device workspace the backward needs (n_seqs: B, or the packed sequence count)."""
    return int(load_library().gdn_chunk_bwd_workspace_bytes(B, H, T, dk, dv, n_seqs))


def gdn_bwd_select_path(dk: int, dv: int, dtype: torch.dtype) -> int:
    """The backward path (GDN_BWD_TOKENS or GDN_BWD_CHUNKED) taken for these sizes."""
    return load_library().gdn_bwd_select_path(dk, dv, _dtype_code(dtype))


def gdn_chunk_bwd(q, k, v, log_alpha, beta, S0, d_out, dS_final, d_q, d_k, d_v, d_log_alpha,
                  d_beta, d_S0, workspace, cu_seqlens: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None, path: int = GDN_BWD_AUTO) -> None:
    """Tensor-level call of the C entry point gdn_chunk_bwd_ex (gdn_chunk_bwd for
    path = GDN_BWD_AUTO).  Inputs as for ``gdn_chunk_fwd``; d_out like out; dS_final like
    S_final (or None); the gradient outputs d_q, d_k, d_v (input dtype), d_log_alpha,
    d_beta (fp32) and d_S0 (fp32 or None); workspace a CUDA uint8 tensor of at least
    ``gdn_chunk_bwd_workspace_bytes`` bytes.  Launches on ``stream`` (default: current)
    without synchronising."""
    lib = load_library()
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    tensors = [q, k, v, log_alpha, beta, S0, d_out, dS_final, d_q, d_k, d_v, d_log_alpha,
               d_beta, d_S0, workspace, cu_seqlens]
    for t in tensors:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("gdn_chunk_bwd: every tensor must be a contiguous CUDA tensor")
    code = _dtype_code(v.dtype)
    for t in (q, k, d_out, d_q, d_k, d_v):
        if t.dtype != v.dtype:
            raise TypeError("q, k, v, d_out, d_q, d_k and d_v must share one dtype")
    for name, t in (("log_alpha", log_alpha), ("beta", beta), ("S0", S0), ("dS_final", dS_final),
                    ("d_log_alpha", d_log_alpha), ("d_beta", d_beta), ("d_S0", d_S0)):
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    n_seqs = B if cu_seqlens is None else cu_seqlens.numel() - 1
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = stream if stream is not None else torch.cuda.current_stream(v.device)
    with torch.cuda.device(v.device):
        st = lib.gdn_chunk_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                  _ptr(S0), _ptr(d_out), _ptr(dS_final), _ptr(d_q), _ptr(d_k),
                                  _ptr(d_v), _ptr(d_log_alpha), _ptr(d_beta), _ptr(d_S0),
                                  _ptr(workspace), ws_bytes, B, H, T, dk, dv, _ptr(cu_seqlens),
                                  0 if cu_seqlens is None else n_seqs, code, int(path),
                                  ctypes.c_void_p(s.cuda_stream))
    _check(st)


def gdn_chunk_bwd_noalloc(q, k, v, log_alpha, beta, S0, d_out, dS_final, d_q, d_k, d_v,
                          d_log_alpha, d_beta, d_S0, cu_seqlens: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None) -> None:
    """Tensor-level call of the C entry point of the same name: the per-token backward
    with the library's fixed scratch array instead of a workspace, for callers that
    cannot allocate device memory.  Arguments as for ``gdn_chunk_bwd`` without the
    workspace; sizes whose scratch exceeds the array raise GdnError(GDN_EINVAL)."""
    lib = load_library()
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    for t in (q, k, v, log_alpha, beta, S0, d_out, dS_final, d_q, d_k, d_v, d_log_alpha,
              d_beta, d_S0, cu_seqlens):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("gdn_chunk_bwd_noalloc: every tensor must be a contiguous CUDA tensor")
    code = _dtype_code(v.dtype)
    n_seqs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    s = stream if stream is not None else torch.cuda.current_stream(v.device)
    with torch.cuda.device(v.device):
        st = lib.gdn_chunk_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                       _ptr(S0), _ptr(d_out), _ptr(dS_final), _ptr(d_q),
                                       _ptr(d_k), _ptr(d_v), _ptr(d_log_alpha), _ptr(d_beta),
                                       _ptr(d_S0), B, H, T, dk, dv, _ptr(cu_seqlens), n_seqs,
                                       code, ctypes.c_void_p(s.cuda_stream))
    _check(st)


def chunk_bwd(q, k, v, log_alpha, beta, S0, d_out, dS_final=None, cu_seqlens=None,
              want_dS0: bool = True, path: int = GDN_BWD_AUTO):
    """Allocate the gradients and the workspace and run the backward on the current
    stream (device tensors), on ``path`` (GDN_BWD_AUTO, GDN_BWD_TOKENS or
    GDN_BWD_CHUNKED).  Returns (d_q, d_k, d_v, d_log_alpha, d_beta, d_S0 or None)."""
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    dev = v.device
    d_q, d_k, d_v = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    d_la = torch.empty_like(log_alpha)
    d_b = torch.empty_like(beta)
    d_S0 = torch.empty((N, H, dv, dk), dtype=torch.float32, device=dev) if want_dS0 else None
    nbytes = gdn_chunk_bwd_workspace_bytes(B, H, T, dk, dv, N)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    gdn_chunk_bwd(q, k, v, log_alpha, beta, S0, d_out, dS_final, d_q, d_k, d_v, d_la, d_b, d_S0,
                  ws, cu_seqlens, path=path)
    return d_q, d_k, d_v, d_la, d_b, d_S0


class GatedDeltaNetFunction(torch.autograd.Function):
    """(out, S_final) = the chunkwise forward of (q, k, v, log_alpha, beta, S0), with
    gradients from gdn_chunk_bwd.  Both directions run in the library's kernels on the
    current stream; device tensors only."""

    @staticmethod
    def forward(ctx, q, k, v, log_alpha, beta, S0, C, cu_seqlens):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        log_alpha, beta = log_alpha.contiguous(), beta.contiguous()
        S0 = None if S0 is None else S0.contiguous()
        out, Sf = chunk_fwd(q, k, v, log_alpha, beta, S0, cu_seqlens, C=C)
        ctx.save_for_backward(q, k, v, log_alpha, beta, S0, cu_seqlens)
        return out, Sf

    @staticmethod
    def backward(ctx, d_out, dS_final):
        q, k, v, log_alpha, beta, S0, cu_seqlens = ctx.saved_tensors
        if d_out is None:
            d_out = torch.zeros(v.shape, dtype=v.dtype, device=v.device)
        d_out = d_out.to(v.dtype).contiguous()
        dS_final = None if dS_final is None else dS_final.float().contiguous()
        want_dS0 = S0 is not None and ctx.needs_input_grad[5]
        d_q, d_k, d_v, d_la, d_b, d_S0 = chunk_bwd(q, k, v, log_alpha, beta, S0, d_out, dS_final,
                                                   cu_seqlens, want_dS0=want_dS0)
        return d_q, d_k, d_v, d_la, d_b, d_S0, None, None


def gated_delta_rule(q, k, v, log_alpha, beta, S0=None, C: int = 64, cu_seqlens=None):
    """Differentiable chunkwise Gated DeltaNet: returns (out, S_final); backward by
    gdn_chunk_bwd."""
    return GatedDeltaNetFunction.apply(q, k, v, log_alpha, beta, S0, C, cu_seqlens)
