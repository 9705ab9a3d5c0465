"""GPU parity of the backward (gdn_chunk_bwd) against the fp64 backward oracle.

The oracle (oracle/backward.py) is the reverse-mode derivative of the per-token
recurrence, pinned to finite differences and autograd (tests/test_backward_pins.py).
The kernel computes in fp32 from inputs that fp64 holds exactly, so every gradient
stored in fp32 must match to max|delta| / max|ref| <= 1e-4; gradients stored in
bf16 (d_q, d_k, d_v for bf16 inputs) also get their own storage rounding,
|delta_i| <= 2^-8 |ref_i| + 1e-4 max|ref|.
"""
import dataclasses

import numpy as np
import pytest
import torch

import chunkwise_gated_deltanet_gb300 as gdn
import workloads
from oracle import backward as BW
from tests.parity import TOL_F32_REL_MAX, sample_units, to_device

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS
NAMES = ("d_q", "d_k", "d_v", "d_log_alpha", "d_beta", "d_S0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _gpu(inp, grads, with_S0_grad=True, with_dSf=True, path=gdn.GDN_BWD_AUTO):
    d = to_device(inp)
    g = to_device(grads)
    res = gdn.chunk_bwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"], g["d_out"],
                        g["dS_final"] if with_dSf else None, d["cu_seqlens"],
                        want_dS0=with_S0_grad, path=path)
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    return [None if x is None else x.float().cpu().numpy().astype(np.float64) for x in res]


def _oracle(inp, grads, with_dSf=True):
    return BW.gdn_backward(inp["q"].double().numpy(), inp["k"].double().numpy(),
                           inp["v"].double().numpy(), inp["log_alpha"].double().numpy(),
                           inp["beta"].double().numpy(),
                           None if inp["S0"] is None else inp["S0"].double().numpy(),
                           grads["d_out"].double().numpy(),
                           grads["dS_final"].double().numpy() if with_dSf else None,
                           None if inp["cu_seqlens"] is None else inp["cu_seqlens"].numpy())


def _check(got, ref, bf16_store, what):
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), what
    ref_max = max(np.abs(ref).max(), 1e-30) if ref.size else 1.0
    d = np.abs(got - ref)
    if bf16_store:
        d = d - 2.0 ** -8 * np.abs(ref)
    err = d.max() / ref_max if ref.size else 0.0
    assert err <= TOL_F32_REL_MAX, f"{what}: {err}"


def _compare(got, ref, bf16):
    for i, name in enumerate(NAMES):
        if got[i] is None:
            continue
        _check(got[i], ref[i], bf16 and i < 3, name)


@pytest.mark.parametrize("T", [1, 7, 8, 9, 70])
def test_backward_f32_lengths(T):
    w = W["gdn_f32_b2h4t1024d64c64"]
    inp = workloads.make_inputs(w, B=2, H=2, T=T, seed=T)
    grads = workloads.make_grad_inputs(inp, seed=T + 1)
    _compare(_gpu(inp, grads), _oracle(inp, grads), False)


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 128), (128, 64), (16, 128), (128, 16),
                                   (64, 32)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_head_sizes(dk, dv, dtype):
    w = dataclasses.replace(W["gdn_f32_b2h4t1024d64c64"], dk=dk, dv=dv, dtype=dtype)
    inp = workloads.make_inputs(w, B=1, H=2, T=45, seed=dk + dv)
    grads = workloads.make_grad_inputs(inp, seed=3)
    _compare(_gpu(inp, grads), _oracle(inp, grads), dtype == "bf16")


def test_backward_bf16_headline_shape():
    """The headline shape family (bf16, d = 128, no S0), several checkpoint blocks and
    a ragged tail on every (sequence, head)."""
    inp = workloads.make_inputs(W["gdn_bf16_b4h16t4096d128c64"], B=2, H=2, T=133, seed=2)
    grads = workloads.make_grad_inputs(inp, seed=4)
    _compare(_gpu(inp, grads), _oracle(inp, grads), True)


def test_backward_packed_sequences():
    w = W["gdn_bf16_varlen256_h16d128c64"]
    inp = workloads.make_inputs(w, n_seqs=4, H=2, seed=6)
    # an empty sequence in the middle: repeat one offset
    cu = inp["cu_seqlens"].tolist()
    cu = cu[:2] + [cu[1]] + cu[2:]
    inp["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32)
    inp["N"] = len(cu) - 1
    grads = workloads.make_grad_inputs(inp, seed=8)
    _compare(_gpu(inp, grads), _oracle(inp, grads), True)


def test_backward_optional_state_arguments():
    """No S0, no dS_final, no d_S0 requested."""
    w = W["gdn_f32_b2h4t1024d64c64"]
    inp = workloads.make_inputs(w, B=1, H=3, T=30, seed=9)
    inp["S0"] = None
    grads = workloads.make_grad_inputs(inp, seed=10)
    got = _gpu(inp, grads, with_S0_grad=False, with_dSf=False)
    assert got[5] is None
    _compare(got, _oracle(inp, grads, with_dSf=False), False)


def test_backward_empty_sequence_passes_state_gradient():
    w = W["gdn_f32_b2h4t1024d64c64"]
    inp = workloads.make_inputs(w, B=2, H=2, T=0)
    grads = workloads.make_grad_inputs(inp)
    got = _gpu(inp, grads)
    assert got[0].size == 0
    assert np.array_equal(got[5], grads["dS_final"].numpy().astype(np.float64))


def test_backward_deterministic():
    inp = workloads.make_inputs(W["gdn_bf16_b4h16t4096d128c64"], B=1, H=4, T=100, seed=11)
    grads = workloads.make_grad_inputs(inp, seed=12)
    a = _gpu(inp, grads)
    b = _gpu(inp, grads)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_backward_headline_size_sampled():
    """The headline workload at full size, compared on sampled (sequence, head)
    pairs that the oracle computes one by one."""
    inp = workloads.make_inputs(W["gdn_bf16_b4h16t4096d128c64"])
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


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_autograd_function_matches_oracle(dtype):
    """loss.backward() through gated_delta_rule gives the oracle's gradients."""
    w = dataclasses.replace(W["gdn_f32_b2h4t1024d64c64"], dtype=dtype)
    inp = workloads.make_inputs(w, B=2, H=2, T=37, seed=21)
    grads = workloads.make_grad_inputs(inp, seed=22)
    d = to_device(inp)
    leaves = [d[n].clone().requires_grad_(True) for n in ("q", "k", "v", "log_alpha", "beta", "S0")]
    out, Sf = gdn.gated_delta_rule(*leaves, C=64)
    loss = (out.float() * grads["d_out"].cuda().float()).sum() + (Sf * grads["dS_final"].cuda()).sum()
    loss.backward()
    torch.cuda.synchronize()
    got = [x.grad.float().cpu().numpy().astype(np.float64) for x in leaves]
    ref = _oracle(inp, grads)
    # the autograd loss multiplies by the bf16 d_out widened to fp32: the same values
    _compare(got, ref, dtype == "bf16")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_tokens_path_at_chunked_head_sizes(d, dtype):
    """d = 64 and 128 take the chunked path by default; the per-token path stays
    selectable there (GDN_BWD_TOKENS) and must meet the same bound, packed batches
    included."""
    w = dataclasses.replace(W["gdn_f32_b2h4t1024d64c64"], dk=d, dv=d, dtype=dtype)
    inp = workloads.make_inputs(w, B=2, H=2, T=77, seed=d + 5)
    grads = workloads.make_grad_inputs(inp, seed=d + 6)
    _compare(_gpu(inp, grads, path=gdn.GDN_BWD_TOKENS), _oracle(inp, grads), dtype == "bf16")
    lens = [40, 0, 75]
    inp = workloads.make_inputs(w, B=1, H=2, T=sum(lens), seed=d + 7)
    inp["cu_seqlens"] = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    inp["N"] = len(lens)
    inp["S0"] = None
    grads = workloads.make_grad_inputs(inp, seed=d + 8)
    _compare(_gpu(inp, grads, path=gdn.GDN_BWD_TOKENS), _oracle(inp, grads), dtype == "bf16")
