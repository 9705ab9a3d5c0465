"""The allocation-free backward entry point, gdn_chunk_bwd_noalloc, on the GPU.

Some callers cannot allocate device memory: a plugin that is handed only its input and
output buffers, code running inside a caller's own memory pool, or a path that must not
risk the device-wide synchronisation an allocation can bring.  For them the library
offers the per-token backward with its scratch in a fixed array of its own device memory
instead of a caller-provided workspace.  These tests call that entry point through the
C ABI (ctypes, raw device pointers) and check its gradients against the existing entry
point, gdn_chunk_bwd_ex on the same per-token path with a workspace, twice in a row, so
that the array's contents left by one call cannot change the next call's results.  The
file is named to be collected last, after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import chunkwise_gated_deltanet_gb300 as gdn
import workloads
from tests.parity import TOL_F32_REL_MAX, to_device

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()
    return gdn.load_library()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _outputs(d, N):
    B, T, H, dk = d["k"].shape
    dv = d["v"].shape[-1]
    return [torch.full_like(d["q"], float("nan")), torch.full_like(d["k"], float("nan")),
            torch.full_like(d["v"], float("nan")), torch.full_like(d["log_alpha"], float("nan")),
            torch.full_like(d["beta"], float("nan")),
            torch.full((N, H, dv, dk), float("nan"), dtype=torch.float32, device=d["v"].device)]


def _noalloc(lib, d, g, N, stream):
    """One call of the new entry point through the C ABI; returns the six gradients."""
    B, T, H, dk = d["k"].shape
    dv = d["v"].shape[-1]
    o = _outputs(d, N)
    code = gdn.GDN_BF16 if d["v"].dtype == torch.bfloat16 else gdn.GDN_F32
    cu = d["cu_seqlens"]
    st = lib.gdn_chunk_bwd_noalloc(_p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["log_alpha"]),
                                   _p(d["beta"]), _p(d["S0"]), _p(g["d_out"]), _p(g["dS_final"]),
                                   *[_p(x) for x in o], B, H, T, dk, dv, _p(cu),
                                   0 if cu is None else N, code,
                                   ctypes.c_void_p(stream.cuda_stream))
    assert st == gdn.GDN_OK, lib.gdn_last_error().decode()
    return o


def _with_workspace(lib, d, g, N, stream):
    """The existing entry point on the same path, with a caller-supplied workspace."""
    B, T, H, dk = d["k"].shape
    dv = d["v"].shape[-1]
    o = _outputs(d, N)
    code = gdn.GDN_BF16 if d["v"].dtype == torch.bfloat16 else gdn.GDN_F32
    cu = d["cu_seqlens"]
    nbytes = lib.gdn_chunk_bwd_workspace_bytes(B, H, T, dk, dv, N)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=d["v"].device)
    st = lib.gdn_chunk_bwd_ex(_p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["log_alpha"]),
                              _p(d["beta"]), _p(d["S0"]), _p(g["d_out"]), _p(g["dS_final"]),
                              *[_p(x) for x in o], _p(ws), nbytes, B, H, T, dk, dv, _p(cu),
                              0 if cu is None else N, code, gdn.GDN_BWD_TOKENS,
                              ctypes.c_void_p(stream.cuda_stream))
    assert st == gdn.GDN_OK, lib.gdn_last_error().decode()
    return o


def _close(got, ref, bf16_store, what):
    """The backward tests' bound: max|delta| <= 1e-4 max|ref| (plus the bf16 storage
    rounding of each element for gradients stored in bf16)."""
    a = got.double().cpu().numpy()
    b = ref.double().cpu().numpy()
    assert np.isfinite(a).all(), f"{what}: non-finite values"
    d = np.abs(a - b)
    if bf16_store:
        d = d - 2.0 ** -8 * np.abs(b)
    assert d.max() <= TOL_F32_REL_MAX * max(np.abs(b).max(), 1e-30), what


CASES = [
    ("f32_d64", "gdn_f32_b2h4t1024d64c64", dict(B=2, H=2, T=300), False),
    ("bf16_d128", "gdn_bf16_b4h16t4096d128c64", dict(B=1, H=2, T=200), False),
    ("bf16_d128_packed", "gdn_bf16_b4h16t4096d128c64", dict(B=1, H=2, T=0), True),
]


@pytest.mark.parametrize("name,base,shape,packed", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_entry_point_twice(lib, name, base, shape, packed):
    w = W[base]
    if packed:
        lens = [0, 5, 64, 130, 1]
        inp = workloads.make_inputs(w, B=1, H=2, T=sum(lens), seed=3)
        inp["cu_seqlens"] = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
        inp["N"] = len(lens)
        inp["S0"] = torch.randn(len(lens), 2, w.dv, w.dk,
                                generator=torch.Generator().manual_seed(4)) * 0.1
    else:
        inp = workloads.make_inputs(w, seed=7, **shape)
    grads = workloads.make_grad_inputs(inp, seed=8)
    d, g = to_device(inp), to_device(grads)
    N = inp["N"]
    stream = torch.cuda.current_stream()
    ref = _with_workspace(lib, d, g, N, stream)
    bf16 = w.dtype == "bf16"
    for call in range(2):
        got = _noalloc(lib, d, g, N, stream)
        assert gdn.load_library().gdn_check_status(ctypes.c_void_p(stream.cuda_stream)) == 0
        torch.cuda.synchronize()
        for i, nm in enumerate(("d_q", "d_k", "d_v", "d_log_alpha", "d_beta", "d_S0")):
            _close(got[i], ref[i], bf16 and i < 3, f"{name} call {call}: {nm}")


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    """A problem whose scratch exceeds the fixed array is refused before any launch."""
    cap = lib.gdn_chunk_bwd_noalloc_max_scratch_bytes()
    assert cap == 64 << 20
    B, H, T, dk, dv = 1, 16, 4096, 128, 128
    assert lib.gdn_chunk_bwd_workspace_bytes(B, H, T, dk, dv, B) > cap
    dummy = torch.empty(16, dtype=torch.float32, device="cuda")
    p = _p(dummy)
    st = lib.gdn_chunk_bwd_noalloc(p, p, p, p, p, None, p, None, p, p, p, p, p, None,
                                   B, H, T, dk, dv, None, 0, gdn.GDN_BF16, None)
    assert st == gdn.GDN_EINVAL
    assert b"fixed" in lib.gdn_last_error()
