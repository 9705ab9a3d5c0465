"""GPU parity of the linear mode (gdn_linear_chunk_fwd) against the oracle.

The linear mode is the Mamba2 recurrence S_t = alpha_t S_{t-1} + v_t k_t^T,
o_t = S_t q_t (Nyysyyan, "Mamba2"; with alpha = 1 the "Linear attention" section).
The oracle is the per-token fp64 recurrence run with erase strength 0 and write
strength 1; the oracle pins tie that setting to both pages' closed forms.
Tolerances are those of the chunk forward (tests/parity.py).
"""
import dataclasses

import numpy as np
import pytest
import torch

import chunkwise_gated_deltanet_gb300 as gdn
import workloads
from oracle import native
from tests.parity import assert_close, sample_units, to_device

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _gates(inp, alpha_one: bool):
    la = torch.zeros_like(inp["log_alpha"]) if alpha_one else inp["log_alpha"]
    zeros = torch.zeros_like(la)
    return la, zeros, torch.ones_like(la)


def _oracle(inp, alpha_one: bool, units=None):
    la, zeros, ones = _gates(inp, alpha_one)
    if units is None:
        return native.gdn_forward_c(inp["q"], inp["k"], inp["v"], la, zeros, inp["S0"],
                                    inp["cu_seqlens"], erase=zeros, write=ones)
    return native.gdn_units_c(inp["q"], inp["k"], inp["v"], la, zeros, inp["S0"],
                              inp["cu_seqlens"], units, erase=zeros, write=ones)


def _gpu(inp, C: int, alpha_one: bool):
    d = to_device(inp)
    la = None if alpha_one else d["log_alpha"]
    out, Sf = gdn.linear_chunk_fwd(d["q"], d["k"], d["v"], la, d["S0"], d["cu_seqlens"], C=C)
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), Sf.cpu().numpy().astype(np.float64)


def _full(inp, C, alpha_one=False):
    fp32 = inp["dtype"] == "f32"
    o, s = _gpu(inp, C, alpha_one)
    ro, rs = _oracle(inp, alpha_one)
    assert_close(o, ro, fp32, "out", stored_bf16=not fp32)
    assert_close(s, rs, fp32, "S_final")


@pytest.mark.parametrize("alpha_one", [False, True], ids=["mamba2", "linear_attention"])
@pytest.mark.parametrize("C", [16, 32, 64])
def test_linear_f32(C, alpha_one):
    inp = workloads.make_inputs(W["gdn_f32_b2h4t1024d64c64"], B=2, H=3, T=203, seed=C)
    _full(inp, C, alpha_one)


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 128), (128, 64)])
def test_linear_f32_head_sizes(dk, dv):
    w = dataclasses.replace(W["gdn_f32_b2h4t1024d64c64"], dk=dk, dv=dv)
    inp = workloads.make_inputs(w, B=1, H=2, T=77, seed=dk + dv)
    _full(inp, 32)


@pytest.mark.parametrize("alpha_one", [False, True], ids=["mamba2", "linear_attention"])
def test_linear_bf16_tcgen05(alpha_one):
    """bf16 at dk = dv = 128, C = 64 runs the tcgen05 kernel; several chunks and a
    ragged tail on every (sequence, head), S0 given."""
    w = W["gdn_bf16_b4h16t4096d128c64"]
    assert gdn.gdn_select_path(128, 128, 64, torch.bfloat16) == gdn.GDN_PATH_TCGEN05
    inp = workloads.make_inputs(w, B=2, H=3, T=333, seed=5)
    inp["S0"] = torch.randn((2, 3, 128, 128), generator=torch.Generator().manual_seed(9)) * 0.1
    _full(inp, 64, alpha_one)


def test_linear_bf16_strong_decay():
    """Every chunk in the tcgen05 kernel's strong-decay form, in the linear mode."""
    w = workloads.Workload("decay_bf16", "bf16", B=1, H=2, T=200, dk=128, dv=128, C=64,
                           alpha_mu=-2.0, s0_std=0.1)
    _full(workloads.make_inputs(w), 64)


def test_linear_bf16_varlen():
    w = W["gdn_bf16_varlen256_h16d128c64"]
    inp = workloads.make_inputs(w, n_seqs=6, H=2, seed=3)
    _full(inp, 64)


def test_linear_bf16_headline_size_sampled():
    """The headline shape in the linear mode, compared on sampled (sequence, head)
    pairs that the oracle computes one by one."""
    w = W["gdn_bf16_b4h16t4096d128c64"]
    inp = workloads.make_inputs(w)
    o, s = _gpu(inp, 64, False)
    units = sample_units(inp["N"], inp["H"], 6)
    res = _oracle(inp, False, units)
    got_o = np.concatenate([o[n, :, h] for n, h in units])
    ref_o = np.concatenate([r[0] for r in res])
    assert_close(got_o, ref_o, False, "out (sampled)", stored_bf16=True)
    assert_close(np.stack([s[n, h] for n, h in units]), np.stack([r[1] for r in res]), False,
                 "S_final (sampled)")


def test_zero_write_reduces_to_pure_decay():
    """With beta = 0 the delta rule writes nothing, so gdn_chunk_fwd is a pure
    decay of S0; the linear mode with v = 0 is the same pure decay."""
    w = W["gdn_f32_b2h4t1024d64c64"]
    inp = workloads.make_inputs(w, B=1, H=2, T=130, seed=4)
    d = to_device(inp)
    _, s_gdn = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"],
                             torch.zeros_like(d["beta"]), d["S0"], None, C=64)
    _, s_lin = gdn.linear_chunk_fwd(d["q"], d["k"], torch.zeros_like(d["v"]), d["log_alpha"],
                                    d["S0"], None, C=64)
    torch.cuda.synchronize()
    ref = inp["S0"].double() * torch.exp(inp["log_alpha"].double().sum(1))[0][:, None, None]
    assert torch.allclose(s_gdn.cpu().double(), ref, rtol=1e-5, atol=1e-7)
    assert torch.allclose(s_lin.cpu().double(), ref, rtol=1e-5, atol=1e-7)


def test_linear_empty_sequence_returns_S0():
    w = W["gdn_f32_b2h4t1024d64c64"]
    inp = workloads.make_inputs(w, B=2, H=2, T=0)
    o, s = _gpu(inp, 64, False)
    assert o.size == 0
    ref = np.zeros_like(s) if inp["S0"] is None else inp["S0"].numpy()
    assert np.array_equal(s, ref)


@pytest.mark.parametrize("alpha_one", [False, True], ids=["mamba2", "linear_attention"])
def test_linear_bf16_packed_empty_and_short_sequences(alpha_one):
    """The tensor-core linear kernel on a packed batch with empty, one-token, one-chunk,
    one-chunk-plus-one and ragged sequences, each from its own S0: the chunk loop's
    first chunk, partial last chunks and sequences with no chunk at all."""
    base = W["gdn_bf16_b4h16t4096d128c64"]
    lens = [0, 1, 64, 65, 3, 0, 130, 17, 200]
    inp = workloads.make_inputs(base, B=1, H=2, T=sum(lens), seed=6)
    inp["cu_seqlens"] = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    inp["N"] = len(lens)
    g = torch.Generator().manual_seed(7)
    inp["S0"] = torch.randn(len(lens), 2, base.dv, base.dk, generator=g) * 0.1
    _full(inp, 64, alpha_one)


@pytest.mark.parametrize("B,H,T,R", [(1, 1, 600, 4), (1, 1, 520, 3), (2, 3, 333, 3),
                                     (4, 16, 300, 2), (2, 16, 1000, 4)])
@pytest.mark.parametrize("alpha_one", [False, True], ids=["mamba2", "linear_attention"])
def test_linear_split_over_more_sms(B, H, T, R, alpha_one):
    """Few (sequence, head) units: the tcgen05 path cuts each sequence into whole-chunk
    segments on more SMs, folds their end states and corrects the later segments' outputs;
    every unit against the oracle, S0 given, ragged tails.  T = 520 (9 chunks) would leave
    a fourth segment of 3-chunk segments empty, so it takes three."""
    w = W["gdn_bf16_b4h16t4096d128c64"]
    assert gdn.gdn_linear_split_segments(B, H, T, 128, 128, 64, torch.bfloat16) == R
    inp = workloads.make_inputs(w, B=B, H=H, T=T, seed=B + H)
    inp["S0"] = torch.randn((B, H, 128, 128), generator=torch.Generator().manual_seed(T)) * 0.1
    _full(inp, 64, alpha_one)


@pytest.mark.parametrize("alpha_mu", [2.0, -2.0], ids=["mild", "strong_decay"])
def test_linear_split_with_resets_at_segment_edges(alpha_mu):
    """Four segments of 256 tokens (B=1, H=2, T=1000): alpha = 0 (a full reset) on the last
    token of a segment, on the first token of the next, inside a later segment and on the
    sequence's last token, so the folded start states and the correction's gate sums meet
    exp(-inf) = 0 at the edges; mild and strong decay."""
    w = workloads.Workload("split_resets", "bf16", B=1, H=2, T=1000, dk=128, dv=128, C=64,
                           alpha_mu=alpha_mu, s0_std=0.1)
    assert gdn.gdn_linear_split_segments(1, 2, 1000, 128, 128, 64, torch.bfloat16) == 4
    inp = workloads.make_inputs(w, seed=21)
    la = inp["log_alpha"].clone()
    for t in (255, 256, 511, 600, 999):
        la[:, t, :] = -float("inf")
    inp["log_alpha"] = la
    _full(inp, 64)


@pytest.mark.parametrize("d,dtype,C", [(64, "f32", 64), (128, "f32", 64), (64, "bf16", 32),
                                       (128, "bf16", 16)])
@pytest.mark.parametrize("alpha_one", [False, True], ids=["mamba2", "linear_attention"])
def test_linear_on_the_tf32_chunk_path(d, dtype, C, alpha_one):
    """The shapes off the bf16 kernel run the linear mode on the TF32 chunk path (the
    gather's erase gates 0, so T = I and W~ = 0, and U = V): every unit against the
    oracle, S0 given, a ragged last chunk, with and without gates."""
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    assert gdn.gdn_select_path(d, d, C, dt) == gdn.GDN_PATH_TF32
    w = workloads.Workload("lin_tf32", dtype, B=2, H=2, T=333, dk=d, dv=d, C=C, alpha_mu=2.0,
                           s0_std=0.1)
    _full(workloads.make_inputs(w, seed=31 + d + C), C, alpha_one)


def test_linear_tf32_chunk_path_packed_with_resets():
    """A packed fp32 batch on the TF32 chunk path: empty, one-token, one-chunk, ragged
    members, each from its own S0, with alpha = 0 resets inside and at the first token."""
    lens = [0, 1, 64, 65, 130, 17]
    w = workloads.Workload("lin_tf32_packed", "f32", B=1, H=2, T=sum(lens), dk=128, dv=128,
                           C=64, alpha_mu=2.0, s0_std=0.0)
    inp = workloads.make_inputs(w, seed=41)
    inp["cu_seqlens"] = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    inp["N"] = len(lens)
    inp["S0"] = torch.randn(len(lens), 2, 128, 128,
                            generator=torch.Generator().manual_seed(42)) * 0.1
    la = inp["log_alpha"].clone()
    for t in (1, 2, 100, 200):
        la[:, t, :] = -float("inf")
    inp["log_alpha"] = la
    _full(inp, 64)


def test_linear_split_without_S0_or_final_state():
    """The split path with S0 = NULL (every segment from zero) and S_final not requested
    (the correction then writes no end state); the outputs against the oracle."""
    w = workloads.Workload("split_plain", "bf16", B=1, H=3, T=700, dk=128, dv=128, C=64,
                           alpha_mu=4.0, s0_std=0.0)
    assert gdn.gdn_linear_split_segments(1, 3, 700, 128, 128, 64, torch.bfloat16) > 1
    inp = workloads.make_inputs(w, seed=51)
    assert inp["S0"] is None
    d = to_device(inp)
    out, Sf = gdn.linear_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], None, None, C=64,
                                   output_final_state=False)
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    assert Sf is None
    ro, _ = _oracle(inp, False)
    assert_close(out.float().cpu().numpy().astype(np.float64), ro, False, "out",
                 stored_bf16=True)
