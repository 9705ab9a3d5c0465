"""GPU parity of the chunked backward (gdn_chunk_bwd_ex, GDN_BWD_CHUNKED) against the fp64
backward oracle, with the same bound as the per-token path: fp32 arithmetic on inputs
that fp64 holds exactly, max|delta| / max|ref| <= 1e-4, plus bf16 storage rounding for
d_q, d_k, d_v when the inputs are bf16.

The chunk form's derivative (Nyysyyan, "Gated-DeltaNet", WY representation and chunkwise
algorithm, differentiated per chunk) is itself pinned against the per-token backward in
tests/test_backward_pins.py; here the kernels meet the per-token oracle directly, over
ragged chunk tails, packed sequences with empty and one-token members, absent optional
arguments, gate resets (alpha = 0), and sampled units of the full headline workload.
"""
import dataclasses

import numpy as np
import pytest
import torch

import chunkwise_gated_deltanet_gb300 as gdn
import workloads
from oracle import backward as BW
from tests.parity import TOL_F32_REL_MAX, sample_units, to_device
from tests.test_backward_gpu import NAMES, _check, _compare, _oracle

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS
F32 = "gdn_f32_b2h4t1024d64c64"
BF16 = "gdn_bf16_b4h16t4096d128c64"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _gpu(inp, grads, path=gdn.GDN_BWD_CHUNKED, with_S0_grad=True, with_dSf=True):
    d = to_device(inp)
    g = to_device(grads)
    res = gdn.chunk_bwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"], g["d_out"],
                        g["dS_final"] if with_dSf else None, d["cu_seqlens"],
                        want_dS0=with_S0_grad, path=path)
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    return [None if x is None else x.float().cpu().numpy().astype(np.float64) for x in res]


def _with_S0(inp, seed):
    g = torch.Generator().manual_seed(seed)
    inp["S0"] = torch.randn(inp["S0"].shape if inp["S0"] is not None else
                            (inp["N"], inp["H"], inp["v"].shape[-1], inp["k"].shape[-1]),
                            generator=g) * 0.1
    return inp


def test_auto_path_is_chunked_for_supported_heads():
    assert gdn.gdn_bwd_select_path(128, 128, torch.bfloat16) == gdn.GDN_BWD_CHUNKED
    assert gdn.gdn_bwd_select_path(64, 64, torch.float32) == gdn.GDN_BWD_CHUNKED
    assert gdn.gdn_bwd_select_path(64, 128, torch.float32) == gdn.GDN_BWD_TOKENS


@pytest.mark.parametrize("T", [1, 5, 63, 64, 65, 129, 200])
def test_chunked_f32_lengths(T):
    inp = _with_S0(workloads.make_inputs(W[F32], B=2, H=3, T=T, seed=20 + T), 21)
    grads = workloads.make_grad_inputs(inp, seed=22)
    _compare(_gpu(inp, grads), _oracle(inp, grads), False)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunked_head_sizes_and_dtypes(d, dtype):
    w = dataclasses.replace(W[F32], dk=d, dv=d, dtype=dtype)
    inp = _with_S0(workloads.make_inputs(w, B=2, H=2, T=150, seed=31 + d), 32)
    grads = workloads.make_grad_inputs(inp, seed=33)
    _compare(_gpu(inp, grads), _oracle(inp, grads), dtype == "bf16")


def test_chunked_packed_sequences_with_empty_and_single_token_members():
    lens = [70, 0, 1, 130, 64, 3]
    inp = workloads.make_inputs(W[BF16], B=1, H=2, T=sum(lens), seed=41)
    inp["cu_seqlens"] = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    inp["N"] = len(lens)
    inp = _with_S0(inp, 42)
    grads = workloads.make_grad_inputs(inp, seed=43)
    _compare(_gpu(inp, grads), _oracle(inp, grads), True)


def test_chunked_optional_state_arguments():
    inp = workloads.make_inputs(W[F32], B=2, H=2, T=90, seed=51)
    inp["S0"] = None
    grads = workloads.make_grad_inputs(inp, seed=52)
    got = _gpu(inp, grads, with_S0_grad=False, with_dSf=False)
    assert got[5] is None
    ref = _oracle(inp, grads, with_dSf=False)
    _compare(got, ref, False)


def test_chunked_gate_resets():
    """alpha = 0 tokens at chunk starts, chunk ends and mid-chunk: the gradient of
    log alpha there is 0 up to rounding, and nothing reaches the state before."""
    inp = _with_S0(workloads.make_inputs(W[F32], B=2, H=2, T=200, seed=61), 62)
    la = inp["log_alpha"].clone()
    for t in (0, 5, 63, 64, 65, 130, 131, 199):
        la[:, t, :] = -float("inf")
    inp["log_alpha"] = la
    grads = workloads.make_grad_inputs(inp, seed=63)
    _compare(_gpu(inp, grads), _oracle(inp, grads), False)


def test_chunked_deterministic_and_close_to_the_token_path():
    inp = _with_S0(workloads.make_inputs(W[BF16], B=1, H=4, T=300, seed=71), 72)
    grads = workloads.make_grad_inputs(inp, seed=73)
    a = _gpu(inp, grads)
    b = _gpu(inp, grads)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    t = _gpu(inp, grads, path=gdn.GDN_BWD_TOKENS)
    for i, name in enumerate(NAMES):
        # both sides round to bf16 on their own for d_q, d_k, d_v: up to one bf16 ulp
        # (2^-7 relative) apart, on top of the fp32 bound
        d = np.abs(a[i] - t[i]) - (2.0 ** -7 * np.abs(t[i]) if i < 3 else 0.0)
        assert d.max() / np.abs(t[i]).max() <= TOL_F32_REL_MAX, name


def test_chunked_headline_size_sampled():
    """The full headline workload (bf16, B=4 H=16 T=4096 dk=dv=128) on the chunked path,
    compared on sampled (sequence, head) pairs that the oracle computes one by one."""
    inp = workloads.make_inputs(W[BF16])
    grads = workloads.make_grad_inputs(inp)
    got = _gpu(inp, grads)
    for n, h in sample_units(inp["N"], inp["H"], 3):
        ref = BW.gdn_sequence_bwd(inp["q"][n, :, h].double().numpy(),
                                  inp["k"][n, :, h].double().numpy(),
                                  inp["v"][n, :, h].double().numpy(),
                                  inp["log_alpha"][n, :, h].double().numpy(),
                                  inp["beta"][n, :, h].double().numpy(), None,
                                  grads["d_out"][n, :, h].double().numpy(),
                                  grads["dS_final"][n, h].double().numpy())
        for i, name in enumerate(NAMES):
            g = got[i][n, :, h] if i < 5 else got[5][n, h]
            _check(g, ref[i], i < 3, f"{name} unit ({n}, {h})")
