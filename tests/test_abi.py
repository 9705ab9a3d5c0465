"""Host-side checks of the C ABI (CPU only: no kernel is launched).

The library must load, export every function include/gdn.h declares, pick the
kernel path the header documents, and reject every invalid argument before any
launch.
"""
import ctypes
import os
import re

import pytest
import torch

import chunkwise_gated_deltanet_gb300 as gdn
from chunkwise_gated_deltanet_gb300 import build as gdn_build
from chunkwise_gated_deltanet_gb300 import gdn as binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def lib():
    gdn_build.build()
    return gdn.load_library()


def _declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(gdn_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    assert "gdn_chunk_fwd" in names and "gdn_last_error" in names
    assert set(binding.EXPORTS) <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libgdn.so does not export {name}"


def test_version(lib):
    assert gdn.gdn_version() >= 10000


@pytest.mark.parametrize("dk,dv,C,dt,path", [
    (128, 128, 64, torch.bfloat16, None),     # tensor-core path once available
    (128, 128, 64, torch.float32, gdn.GDN_PATH_TF32),
    (16, 16, 16, torch.float32, gdn.GDN_PATH_SIMT),
    (64, 64, 64, torch.float32, gdn.GDN_PATH_TF32),
    (64, 64, 64, torch.bfloat16, gdn.GDN_PATH_TF32),
    (64, 64, 32, torch.float32, gdn.GDN_PATH_TF32),
    (128, 128, 16, torch.bfloat16, gdn.GDN_PATH_TF32),
    (32, 32, 32, torch.float32, gdn.GDN_PATH_SIMT),
    (64, 128, 32, torch.bfloat16, gdn.GDN_PATH_SIMT),
    (48, 64, 64, torch.float32, gdn.GDN_PATH_NONE),
    (64, 64, 128, torch.float32, gdn.GDN_PATH_NONE),
    (64, 256, 64, torch.bfloat16, gdn.GDN_PATH_NONE),
])
def test_select_path(lib, dk, dv, C, dt, path):
    got = gdn.gdn_select_path(dk, dv, C, dt)
    if path is None:
        assert got in (gdn.GDN_PATH_SIMT, gdn.GDN_PATH_TCGEN05)
    else:
        assert got == path
    assert (gdn.gdn_launches_per_call(dk, dv, C, dt) > 0) == (got != gdn.GDN_PATH_NONE)


def _call(lib, **over):
    """Call gdn_chunk_fwd with fake (never dereferenced) aligned pointers."""
    a = dict(q=4096, k=8192, v=12288, la=16384, be=20480, S0=None, out=24576, Sf=None,
             B=2, H=4, T=128, dk=64, dv=64, C=64, cu=None, N=0, dt=gdn.GDN_F32, stream=None)
    a.update(over)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.gdn_chunk_fwd(P(a["q"]), P(a["k"]), P(a["v"]), P(a["la"]), P(a["be"]), P(a["S0"]),
                             P(a["out"]), P(a["Sf"]), a["B"], a["H"], a["T"], a["dk"], a["dv"],
                             a["C"], P(a["cu"]), a["N"], a["dt"], P(a["stream"]))


@pytest.mark.parametrize("over,code,word", [
    (dict(dt=7), binding.GDN_EDTYPE, "dtype"),
    (dict(q=None), binding.GDN_EINVAL, "non-NULL"),
    (dict(out=None), binding.GDN_EINVAL, "non-NULL"),
    (dict(la=None), binding.GDN_EINVAL, "non-NULL"),
    (dict(B=0), binding.GDN_EINVAL, "B > 0"),
    (dict(H=-1), binding.GDN_EINVAL, "H > 0"),
    (dict(T=-5), binding.GDN_EINVAL, "T >= 0"),
    (dict(dk=48), binding.GDN_EINVAL, "dk and dv"),
    (dict(dv=256), binding.GDN_EINVAL, "dk and dv"),
    (dict(C=8), binding.GDN_EINVAL, "C must be"),
    (dict(C=128), binding.GDN_EINVAL, "C must be"),
    (dict(cu=28672, N=3, B=2), binding.GDN_EINVAL, "B == 1"),
    (dict(cu=28672, N=0, B=1), binding.GDN_EINVAL, "N_seqs"),
    (dict(k=8200), binding.GDN_EINVAL, "k is not 16-byte aligned"),
    (dict(S0=36), binding.GDN_EINVAL, "S0 is not 16-byte aligned"),
    (dict(cu=28676, N=2, B=1), binding.GDN_EINVAL, "cu_seqlens is not 16-byte aligned"),
])
def test_invalid_arguments_rejected_before_launch(lib, over, code, word):
    assert _call(lib, **over) == code
    msg = lib.gdn_last_error().decode()
    assert word in msg, msg


def test_binding_rejects_host_tensors(lib):
    x = torch.zeros(1, 4, 1, 16)
    g = torch.zeros(1, 4, 1)
    with pytest.raises(ValueError):
        gdn.gdn_chunk_fwd(x, x, x, g, g, None, x.clone(), None, C=16)


def test_binding_has_no_cpu_path():
    """The product code never imports the oracle and has no CPU compute."""
    pkg = os.path.join(ROOT, "chunkwise_gated_deltanet_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert "oracle" not in src, fn
            assert "einsum" not in src and "matmul" not in src, fn


def test_missing_library_fails_loudly(tmp_path):
    saved = binding._lib
    binding._lib = None
    try:
        with pytest.raises(ImportError):
            binding.load_library(str(tmp_path / "nope.so"))
    finally:
        binding._lib = saved


def _call_decode(lib, **over):
    """Call gdn_decode_step with fake (never dereferenced) aligned pointers."""
    a = dict(q=4096, k=8192, v=12288, la=16384, be=20480, S=24576, out=28672,
             N=8, H=4, dk=64, dv=64, dt=gdn.GDN_F32, stream=None)
    a.update(over)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.gdn_decode_step(P(a["q"]), P(a["k"]), P(a["v"]), P(a["la"]), P(a["be"]), P(a["S"]),
                               P(a["out"]), a["N"], a["H"], a["dk"], a["dv"], a["dt"],
                               P(a["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(dt=7), gdn.GDN_EDTYPE if hasattr(gdn, "GDN_EDTYPE") else 2),
    (dict(dk=48), 1), (dict(dv=256), 1), (dict(N=-1), 1), (dict(H=-2), 1),
    (dict(q=None), 1), (dict(S=None), 1), (dict(out=None), 1), (dict(la=None), 1),
    (dict(k=8200), 1), (dict(S=24580), 1),
])
def test_decode_rejects_invalid_arguments(lib, over, code):
    assert _call_decode(lib, **over) == code
    assert lib.gdn_last_error()


def test_decode_empty_batch_launches_nothing(lib):
    # N * H == 0 returns OK before looking at the pointers (nothing to launch)
    assert _call_decode(lib, N=0, q=None, S=None, out=None) == binding.GDN_OK
    assert _call_decode(lib, H=0) == binding.GDN_OK


def _call_linear(lib, **over):
    """Call gdn_linear_chunk_fwd with fake (never dereferenced) aligned pointers."""
    a = dict(q=4096, k=8192, v=12288, la=16384, S0=None, out=24576, Sf=None,
             B=2, H=4, T=128, dk=64, dv=64, C=64, cu=None, N=0, dt=gdn.GDN_F32, stream=None)
    a.update(over)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.gdn_linear_chunk_fwd(P(a["q"]), P(a["k"]), P(a["v"]), P(a["la"]), P(a["S0"]),
                                    P(a["out"]), P(a["Sf"]), a["B"], a["H"], a["T"], a["dk"],
                                    a["dv"], a["C"], P(a["cu"]), a["N"], a["dt"], P(a["stream"]))


@pytest.mark.parametrize("over,code,word", [
    (dict(dt=3), binding.GDN_EDTYPE, "dtype"),
    (dict(v=None), binding.GDN_EINVAL, "non-NULL"),
    (dict(B=0), binding.GDN_EINVAL, "B > 0"),
    (dict(dk=24), binding.GDN_EINVAL, "dk and dv"),
    (dict(C=48), binding.GDN_EINVAL, "C must be"),
    (dict(cu=28672, N=3, B=2), binding.GDN_EINVAL, "B == 1"),
    (dict(la=16388), binding.GDN_EINVAL, "log_alpha is not 16-byte aligned"),
])
def test_linear_invalid_arguments_rejected_before_launch(lib, over, code, word):
    assert _call_linear(lib, **over) == code
    msg = lib.gdn_last_error().decode()
    assert msg.startswith("gdn_linear_chunk_fwd") and word in msg, msg


def test_chunk_fwd_still_requires_beta(lib):
    """Only the linear entry point may omit beta."""
    assert _call(lib, be=None) == binding.GDN_EINVAL
    assert "beta" in lib.gdn_last_error().decode()


def _call_fold(lib, **over):
    """Call gdn_state_fold with fake (never dereferenced) aligned pointers."""
    a = dict(S=4096, M=1 << 20, L=2 << 20, count=2, out=3 << 20, units=4, dv=64, dk=64,
             stream=None)
    a.update(over)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.gdn_state_fold(P(a["S"]), P(a["M"]), P(a["L"]), a["count"], P(a["out"]),
                              a["units"], a["dv"], a["dk"], P(a["stream"]))


@pytest.mark.parametrize("over,word", [
    (dict(units=-1), "units >= 0"),
    (dict(count=0), "count >= 1"),
    (dict(S=None, M=None), "non-NULL"),
    (dict(out=(2 << 20) + 4096), "overlaps S_in or L"),
    (dict(dk=48), "dk and dv"),
    (dict(L=None), "non-NULL"),
    (dict(M=None), "non-NULL"),
    (dict(out=3 << 20 | 8), "S_out is not 16-byte aligned"),
    (dict(out=4096 + 1024), "overlaps"),
    (dict(out=(1 << 20) + 4096), "overlaps"),
])
def test_state_fold_invalid_arguments(lib, over, word):
    assert _call_fold(lib, **over) == binding.GDN_EINVAL
    assert word in lib.gdn_last_error().decode()


def test_state_fold_empty_and_no_input_ok(lib):
    assert _call_fold(lib, units=0) == binding.GDN_OK


def _call_host(lib, **over):
    """Call gdn_chunk_fwd_host with fake (never dereferenced) pointers."""
    a = dict(q=4096, k=8192, v=12288, la=16384, be=20480, S0=None, out=24576, Sf=None,
             B=2, H=4, T=128, dk=64, dv=64, C=64, dt=gdn.GDN_F32, pieces=4, ws=1 << 20,
             ws_bytes=1 << 40, stream=None)
    a.update(over)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.gdn_chunk_fwd_host(P(a["q"]), P(a["k"]), P(a["v"]), P(a["la"]), P(a["be"]),
                                  P(a["S0"]), P(a["out"]), P(a["Sf"]), a["B"], a["H"], a["T"],
                                  a["dk"], a["dv"], a["C"], a["dt"], a["pieces"], P(a["ws"]),
                                  a["ws_bytes"], P(a["stream"]))


@pytest.mark.parametrize("over,code,word", [
    (dict(dt=9), binding.GDN_EDTYPE, "dtype"),
    (dict(B=0), binding.GDN_EINVAL, "B > 0"),
    (dict(pieces=0), binding.GDN_EINVAL, "pieces"),
    (dict(pieces=65), binding.GDN_EINVAL, "pieces"),
    (dict(q=None), binding.GDN_EINVAL, "non-NULL"),
    (dict(la=None), binding.GDN_EINVAL, "non-NULL"),
    (dict(ws_bytes=1024), binding.GDN_EINVAL, "workspace"),
    (dict(ws=(1 << 20) + 16), binding.GDN_EINVAL, "workspace"),
    (dict(ws=None), binding.GDN_EINVAL, "workspace"),
    (dict(C=8), binding.GDN_EINVAL, "C must be"),
])
def test_host_forward_invalid_arguments(lib, over, code, word):
    assert _call_host(lib, **over) == code
    assert word in lib.gdn_last_error().decode()


def test_host_forward_workspace_query(lib):
    f = lib.gdn_chunk_fwd_host_workspace_bytes
    full = f(4, 16, 4096, 128, 128, 64, gdn.GDN_BF16, 4, 0)
    lin = f(4, 16, 4096, 128, 128, 64, gdn.GDN_BF16, 4, 1)
    inputs = 4 * 4096 * 16 * (3 * 128 * 2 + 128 * 2 + 8)
    assert full >= inputs and lin < full
    assert f(4, 16, 4096, 128, 128, 64, gdn.GDN_BF16, 0, 0) == 0


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++11")])
def test_header_compiles_standalone(lang, std, tmp_path):
    """include/gdn.h is a plain C ABI: it compiles on its own as C99 and as C++11, with
    warnings as errors, and a C program can take the address of every entry point."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("use.c" if lang == "c" else "use.cpp")
    names = _declared_functions()
    src.write_text('#include "gdn.h"\n' + "void* entry_points[] = {\n" +
                   ",\n".join("  (void*)&%s" % n for n in names) + "\n};\n")
    r = subprocess.run([cc, "-std=" + std, "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def _call_bwd(lib, path, **over):
    """Call gdn_chunk_bwd_ex with fake (never dereferenced) aligned pointers."""
    a = dict(B=2, H=4, T=128, dk=64, dv=64, dt=gdn.GDN_F32)
    a.update(over)
    P = ctypes.c_void_p
    ptrs = [P(4096 * (i + 1)) for i in range(14)]
    ptrs[5] = ptrs[7] = ptrs[13] = None  # S0, dS_final, d_S0
    return lib.gdn_chunk_bwd_ex(*ptrs, P(1 << 20), ctypes.c_size_t(1 << 40), a["B"], a["H"],
                                a["T"], a["dk"], a["dv"], None, 0, a["dt"], path, None)


def test_bwd_select_path(lib):
    assert gdn.gdn_bwd_select_path(128, 128, torch.bfloat16) == gdn.GDN_BWD_CHUNKED
    assert gdn.gdn_bwd_select_path(64, 64, torch.float32) == gdn.GDN_BWD_CHUNKED
    for dk, dv in ((16, 16), (32, 32), (64, 128), (128, 64)):
        assert gdn.gdn_bwd_select_path(dk, dv, torch.float32) == gdn.GDN_BWD_TOKENS
    assert gdn.gdn_bwd_select_path(48, 48, torch.float32) == 0


def test_bwd_workspace_covers_both_paths(lib):
    for dk in (64, 128):
        a = lib.gdn_chunk_bwd_workspace_bytes(4, 16, 4096, dk, dk, 4)
        assert a > 0
    # chunk buffers: at least 16 [64 x d] and 3 [d x d] fp32 tiles per (chunk, head)
    assert lib.gdn_chunk_bwd_workspace_bytes(4, 16, 4096, 128, 128, 4) >= 64 * 16 * (
        16 * 64 * 128 + 3 * 128 * 128) * 4


@pytest.mark.parametrize("path,over,word", [
    (7, {}, "unknown backward path"),
    (-1, {}, "unknown backward path"),
    (gdn.GDN_BWD_CHUNKED, dict(dk=32, dv=32), "chunked path needs"),
    (gdn.GDN_BWD_CHUNKED, dict(dk=64, dv=128), "chunked path needs"),
])
def test_bwd_path_rejected_before_launch(lib, path, over, word):
    assert _call_bwd(lib, path, **over) == binding.GDN_EINVAL
    msg = lib.gdn_last_error().decode()
    assert word in msg, msg


def _call_correct(lib, **over):
    """Call gdn_linear_state_correct with fake (never dereferenced) aligned pointers."""
    a = dict(q=4096, la=8192, Ss=12288, out=16384, Se=20480, B=2, H=4, T=128, dk=128, dv=128,
             dt=gdn.GDN_BF16, stream=None)
    a.update(over)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.gdn_linear_state_correct(P(a["q"]), P(a["la"]), P(a["Ss"]), P(a["out"]),
                                        P(a["Se"]), a["B"], a["H"], a["T"], a["dk"], a["dv"],
                                        a["dt"], P(a["stream"]))


@pytest.mark.parametrize("over,code,word", [
    (dict(dk=64, dv=64), binding.GDN_EINVAL, "dk = dv = 128"),
    (dict(dt=gdn.GDN_F32), binding.GDN_EINVAL, "bf16"),
    (dict(dt=7), binding.GDN_EDTYPE, "qkv_dtype"),
    (dict(B=0), binding.GDN_EINVAL, "B, H > 0"),
    (dict(T=-1), binding.GDN_EINVAL, "T >= 0"),
    (dict(Ss=None), binding.GDN_EINVAL, "non-NULL"),
    (dict(q=None), binding.GDN_EINVAL, "non-NULL"),
    (dict(out=16388), binding.GDN_EINVAL, "out is not 16-byte aligned"),
])
def test_linear_state_correct_rejects_before_launch(lib, over, code, word):
    assert _call_correct(lib, **over) == code
    assert word in lib.gdn_last_error().decode()


def test_linear_state_correct_support_query(lib):
    assert lib.gdn_linear_state_correct_supported(128, 128, gdn.GDN_BF16) == 1
    assert lib.gdn_linear_state_correct_supported(64, 64, gdn.GDN_BF16) == 0
    assert lib.gdn_linear_state_correct_supported(128, 128, gdn.GDN_F32) == 0


@pytest.mark.parametrize("over,word", [
    (dict(B=0), "B, H > 0"),
    (dict(dk=48), "dk in"),
    (dict(M=None), "M must be non-NULL"),
    (dict(M=4100), "16-byte aligned"),
    (dict(cu=28672, N=0, B=1), "N_seqs > 0"),
    (dict(cu=28672, N=3, B=2), "B = 1"),
])
def test_linear_segment_map_rejects_before_launch(lib, over, word):
    a = dict(la=8192, M=4096, B=2, H=4, T=128, dk=128, cu=None, N=2, stream=None)
    a.update(over)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    st = lib.gdn_linear_segment_map(P(a["la"]), P(a["M"]), a["B"], a["H"], a["T"], a["dk"],
                                    P(a["cu"]), a["N"], P(a["stream"]))
    assert st == binding.GDN_EINVAL
    assert word in lib.gdn_last_error().decode()


def test_linear_correct_binding_checks_shapes_and_dtypes():
    """The bindings of the two linear-mode entry points refuse tensors whose shape or dtype
    the pointers cannot carry (checked on CPU tensors, before any device is touched)."""
    bf, f = torch.bfloat16, torch.float32
    q = torch.zeros(2, 8, 3, 128, dtype=bf)
    ok = dict(q=q, log_alpha=torch.zeros(2, 8, 3), S_start=torch.zeros(2, 3, 128, 128),
              out=torch.zeros(2, 8, 3, 128, dtype=bf), S_end=torch.zeros(2, 3, 128, 128))
    binding._correct_shapes(**ok)
    binding._correct_shapes(**dict(ok, log_alpha=None, S_end=None))
    for bad in (dict(S_start=torch.zeros(2, 3, 128, 128, dtype=bf)),
                dict(S_start=torch.zeros(1, 3, 128, 128)),
                dict(S_end=torch.zeros(2, 3, 128, 64)),
                dict(out=torch.zeros(2, 8, 3, 128, dtype=f)),
                dict(log_alpha=torch.zeros(2, 8, 4))):
        with pytest.raises(ValueError):
            binding._correct_shapes(**dict(ok, **bad))
    M = torch.zeros(2, 3, 64, 64)
    binding._segment_map_shapes(torch.zeros(2, 8, 3), M, 2, 8, None)
    binding._segment_map_shapes(None, M, 2, 8, None)
    binding._segment_map_shapes(torch.zeros(1, 8, 3), M, 1, 8, torch.tensor([0, 3, 8],
                                                                              dtype=torch.int32))
    for args in ((torch.zeros(2, 8, 3), torch.zeros(2, 3, 64, 32), 2, 8, None),
                 (torch.zeros(2, 8, 3), M.double(), 2, 8, None),
                 (torch.zeros(2, 9, 3), M, 2, 8, None),
                 (torch.zeros(2, 8, 3), torch.zeros(2, 4, 64, 64), 2, 8, None),
                 (None, M, 3, 8, None),
                 (None, M, 1, 8, torch.tensor([0, 8], dtype=torch.int32)),
                 (None, M, 1, 8, torch.tensor([0, 3, 8], dtype=torch.int64))):
        with pytest.raises(ValueError):
            binding._segment_map_shapes(*args)
