"""A gate of alpha = 0 (log alpha = -inf) forgets the whole state at that token: the
recurrence S_t = alpha_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T restarts from
the token's own write (Nyysyyan, "Gated-DeltaNet", first equation block, with alpha_t = 0).
Every path must match the fp64 oracle, which takes exp(-inf) = 0 exactly, with such
tokens at chunk starts, chunk ends, mid-chunk and back to back."""
import numpy as np
import pytest
import torch

import chunkwise_gated_deltanet_gb300 as gdn
import workloads
from oracle import backward as BW
from oracle import native
from tests.parity import TOL_F32_REL_MAX, assert_close, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS
RESETS = (0, 5, 63, 64, 65, 130, 131, 199, 255, 256, 299)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _reset(inp, T):
    la = inp["log_alpha"].clone()
    for t in RESETS:
        if t < T:
            la[:, t, :] = -float("inf")
    inp["log_alpha"] = la
    return inp


def _with_S0(inp, w, seed):
    g = torch.Generator().manual_seed(seed)
    inp["S0"] = torch.randn(inp["N"], inp["H"], w.dv, w.dk, generator=g) * 0.1
    return inp


@pytest.mark.parametrize("name,T", [("gdn_bf16_b4h16t4096d128c64", 300),
                                    ("gdn_f32_b2h4t1024d64c64", 200)])
def test_forward_with_resets(name, T):
    w = W[name]
    inp = _reset(_with_S0(workloads.make_inputs(w, B=2, H=2, T=T, seed=9), w, 10), T)
    fp32 = inp["dtype"] == "f32"
    o, s = run_gpu(inp, w.C)
    ro, rs = run_oracle(inp)
    assert_close(o, ro, fp32, "out", stored_bf16=not fp32)
    assert_close(s, rs, fp32, "S_final")


def test_forward_packed_with_resets():
    """A packed batch: resets inside sequences and on their first tokens."""
    w = W["gdn_bf16_b4h16t4096d128c64"]
    lens = [70, 1, 130, 99]
    inp = workloads.make_inputs(w, B=1, H=2, T=sum(lens), seed=11)
    inp["cu_seqlens"] = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    inp["N"] = len(lens)
    inp = _reset(_with_S0(inp, w, 12), sum(lens))
    o, s = run_gpu(inp, w.C)
    ro, rs = run_oracle(inp)
    assert_close(o, ro, False, "out", stored_bf16=True)
    assert_close(s, rs, False, "S_final")


def test_linear_mode_with_resets():
    w = W["gdn_bf16_b4h16t4096d128c64"]
    T = 300
    inp = _reset(_with_S0(workloads.make_inputs(w, B=2, H=2, T=T, seed=13), w, 14), T)
    d = to_device(inp)
    out, Sf = gdn.linear_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["S0"], None, C=64)
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    zeros = torch.zeros_like(inp["log_alpha"])
    ro, rs = native.gdn_forward_c(inp["q"], inp["k"], inp["v"], inp["log_alpha"], zeros,
                                  inp["S0"], None, erase=zeros, write=torch.ones_like(zeros))
    assert_close(out.float().cpu().numpy().astype(np.float64), ro, False, "out", stored_bf16=True)
    assert_close(Sf.cpu().numpy().astype(np.float64), rs, False, "S_final")


def test_decode_with_reset():
    w = workloads.DECODE_WORKLOADS["decode_f32_n64h8d64"]
    inp = workloads.make_decode_inputs(w, N=4, H=3, seed=15)
    inp["log_alpha"][1] = -float("inf")
    inp["log_alpha"][3, 2] = -float("inf")
    d = to_device(inp)
    S = d["S"].clone()
    out = gdn.decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S)
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    ro, rS = native.gdn_forward_c(inp["q"].unsqueeze(1), inp["k"].unsqueeze(1),
                                  inp["v"].unsqueeze(1), inp["log_alpha"].unsqueeze(1),
                                  inp["beta"].unsqueeze(1), inp["S"], None)
    got_o, got_S = out.cpu().numpy().astype(np.float64), S.cpu().numpy().astype(np.float64)
    assert np.isfinite(got_o).all() and np.isfinite(got_S).all()
    assert np.abs(got_S - rS).max() / np.abs(rS).max() <= TOL_F32_REL_MAX
    assert np.abs(got_o - ro[:, 0]).max() / np.abs(ro).max() <= TOL_F32_REL_MAX


def test_backward_with_resets():
    """The gradient through a reset: d log alpha = alpha * dL/dalpha = 0 there, and no
    gradient reaches the state before it through the gate."""
    w = W["gdn_f32_b2h4t1024d64c64"]
    T = 140
    inp = _reset(_with_S0(workloads.make_inputs(w, B=2, H=2, T=T, seed=16), w, 17), T)
    grads = workloads.make_grad_inputs(inp, seed=18)
    d, g = to_device(inp), to_device(grads)
    res = gdn.chunk_bwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"], g["d_out"],
                        g["dS_final"], None)
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    ref = BW.gdn_backward(inp["q"].double().numpy(), inp["k"].double().numpy(),
                          inp["v"].double().numpy(), inp["log_alpha"].double().numpy(),
                          inp["beta"].double().numpy(), inp["S0"].double().numpy(),
                          grads["d_out"].double().numpy(), grads["dS_final"].double().numpy(),
                          None)
    for name, got, r in zip(("d_q", "d_k", "d_v", "d_log_alpha", "d_beta", "d_S0"), res, ref):
        got = got.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all(), name
        assert np.abs(got - r).max() / max(np.abs(r).max(), 1e-30) <= TOL_F32_REL_MAX, name
