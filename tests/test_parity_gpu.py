"""GPU parity: the CUDA library against the fp64 oracle, element by element.

Every case is compared in full, the full-size workloads included (they run in the
same call the benchmark times, and the oracle runs every (sequence, head) unit).
Tolerances are in tests/parity.py.
"""
import numpy as np
import pytest
import torch

import chunkwise_gated_deltanet_gb300 as gdn
import workloads
from tests.parity import (assert_close, compare_all_units, run_gpu, run_oracle, to_device)

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _full_check(inp, C):
    fp32 = inp["dtype"] == "f32"
    o, s = run_gpu(inp, C)
    ro, rs = run_oracle(inp)
    eo = assert_close(o, ro, fp32, "out", stored_bf16=not fp32)
    es = assert_close(s, rs, fp32, "S_final")
    return eo, es


# ----------------------------------------------------------- the workloads --

def test_deltanet_f32_b1h1t64d16c16_full():
    _full_check(workloads.make_inputs(W["deltanet_f32_b1h1t64d16c16"]), 16)


def test_gdn_f32_b2h4t1024d64c64_full():
    _full_check(workloads.make_inputs(W["gdn_f32_b2h4t1024d64c64"]), 64)


@pytest.mark.parametrize("name", [
    "gdn_bf16_b4h16t4096d128c64",
    "gdn_bf16_b1h32t32768d128c64",
    "gdn_bf16_varlen256_h16d128c64",
])
def test_full_size_workload_every_unit(name):
    """The three full-size bf16 workloads, in the launch configuration the benchmark
    times, compared on every (sequence, head) unit against the oracle."""
    w = W[name]
    inp = workloads.make_inputs(w)
    o, s = run_gpu(inp, w.C, f64=False)
    assert np.isfinite(o).all() and np.isfinite(s).all()
    compare_all_units(inp, o, s)


def test_bf16_headline_shape_small_full():
    """Same shape family as the headline workload, small enough for a full
    oracle run: several chunks and a ragged tail on every (sequence, head)."""
    inp = workloads.make_inputs(W["gdn_bf16_b4h16t4096d128c64"], B=2, H=3, T=333)
    _full_check(inp, 64)


# --------------------------------------------------------------- edge cases --

@pytest.mark.parametrize("T", [0, 1, 5, 63, 64, 65, 200])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sequence_lengths(T, dtype):
    base = W["gdn_f32_b2h4t1024d64c64"] if dtype == "f32" else W["gdn_bf16_b4h16t4096d128c64"]
    inp = workloads.make_inputs(base, B=2, H=2, T=T)
    if T == 0:
        o, s = run_gpu(inp, base.C)
        S0 = inp["S0"]
        ref = np.zeros_like(s) if S0 is None else S0.numpy()
        assert o.size == 0 and np.array_equal(s, ref)
        return
    _full_check(inp, base.C)


@pytest.mark.parametrize("C", [16, 32, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_sizes(C, dtype):
    base = W["gdn_f32_b2h4t1024d64c64"] if dtype == "f32" else W["gdn_bf16_b4h16t4096d128c64"]
    inp = workloads.make_inputs(base, B=1, H=2, T=150)
    _full_check(inp, C)


@pytest.mark.parametrize("dk,dv", [(16, 64), (64, 128), (128, 32), (32, 16), (128, 128), (16, 16)])
def test_head_size_mix(dk, dv):
    w = workloads.Workload("mix", "f32", B=1, H=2, T=100, dk=dk, dv=dv, C=32, alpha_mu=2.0,
                           s0_std=0.1)
    _full_check(workloads.make_inputs(w), 32)


def test_strong_decay_and_plain_deltanet():
    w = workloads.Workload("decay", "f32", B=1, H=2, T=130, dk=64, dv=64, C=64, alpha_mu=-2.0,
                           s0_std=0.1)
    _full_check(workloads.make_inputs(w), 64)
    w = workloads.Workload("delta", "bf16", B=1, H=2, T=130, dk=128, dv=128, C=64,
                           alpha_mu=None, s0_std=0.1)
    _full_check(workloads.make_inputs(w), 64)


@pytest.mark.parametrize("alpha_mu", [-2.0, -0.3], ids=["all_strong", "mixed_forms"])
def test_tcgen05_strong_decay_forms(alpha_mu):
    """The tcgen05 kernel keeps a chunk in the factored frame only while its total decay
    is above 2^-80; alpha ~ sigmoid(N(-2, 1)) puts every chunk in the strong-decay form,
    sigmoid(N(-0.3, 1)) puts chunks on both sides of the threshold."""
    w = workloads.Workload("decay_bf16", "bf16", B=1, H=3, T=333, dk=128, dv=128, C=64,
                           alpha_mu=alpha_mu, s0_std=0.1)
    assert gdn.gdn_select_path(128, 128, 64, torch.bfloat16) == gdn.GDN_PATH_TCGEN05
    inp = workloads.make_inputs(w)
    per_chunk_bits = -inp["log_alpha"][0, :320].reshape(5, 64, 3).sum(1) * 1.4426950408889634
    if alpha_mu < -1:
        assert (per_chunk_bits > 80).all()
    else:
        assert (per_chunk_bits > 80).any() and (per_chunk_bits < 80).any()
    _full_check(inp, 64)


@pytest.mark.parametrize("beta_mode", ["zero", "one", "alternating"])
def test_tcgen05_beta_extremes(beta_mode):
    """beta = 0 writes nothing (the state only decays from S0, so every output is the
    carried state read out), beta = 1 with unit keys overwrites the stored value along k
    exactly (the write invariant of Nyysyyan's "Gated-DeltaNet" section), and the two
    alternate token by token; all through the tcgen05 kernel, to the plain bounds."""
    w = W["gdn_bf16_b4h16t4096d128c64"]
    inp = workloads.make_inputs(w, B=2, H=2, T=200, seed=21)
    if beta_mode == "zero":
        inp["beta"] = torch.zeros_like(inp["beta"])
    elif beta_mode == "one":
        inp["beta"] = torch.ones_like(inp["beta"])
    else:
        inp["beta"] = (torch.arange(200)[None, :, None] % 2).float().expand_as(inp["beta"]).contiguous()
    g = torch.Generator().manual_seed(22)
    inp["S0"] = torch.randn(2, 2, 128, 128, generator=g) * 0.1
    _full_check(inp, 64)


@pytest.mark.parametrize("beta_const", [0.0, 0.02, 0.1, 0.2, 0.3, 0.5])
@pytest.mark.parametrize("s0_std", [0.1, 1.0])
def test_tcgen05_weak_and_moderate_writes(beta_const, s0_std):
    """Constant write strengths on both sides of the bound below which a chunk takes the
    state operand of S Q^T as two bf16 terms, with a decaying carried state of two
    scales: the outputs meet the plain bounds whichever form a chunk takes."""
    w = W["gdn_bf16_b4h16t4096d128c64"]
    inp = workloads.make_inputs(w, B=1, H=3, T=400, seed=31)
    inp["beta"] = torch.full_like(inp["beta"], beta_const)
    g = torch.Generator().manual_seed(32)
    inp["S0"] = torch.randn(1, 3, 128, 128, generator=g) * s0_std
    _full_check(inp, 64)


def test_without_S0_and_without_S_final():
    inp = workloads.make_inputs(W["gdn_f32_b2h4t1024d64c64"], B=1, H=2, T=100)
    inp["S0"] = None
    o, s = run_gpu(inp, 64, S_final=False)
    assert s is None
    ro, _ = run_oracle(inp)
    assert_close(o, ro, True, "out")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_varlen_with_empty_and_short_sequences(dtype):
    base = W["gdn_f32_b2h4t1024d64c64"] if dtype == "f32" else W["gdn_bf16_b4h16t4096d128c64"]
    lens = [0, 1, 64, 65, 3, 0, 130, 17]
    T = sum(lens)
    inp = workloads.make_inputs(base, B=1, H=2, T=T)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    inp["cu_seqlens"] = cu
    inp["N"] = len(lens)
    g = torch.Generator().manual_seed(5)
    inp["S0"] = torch.randn(len(lens), 2, base.dv, base.dk, generator=g) * 0.1
    _full_check(inp, base.C)


def test_varlen_headline_shapes_small():
    w = W["gdn_bf16_varlen256_h16d128c64"]
    inp = workloads.make_inputs(w, n_seqs=6, H=2)
    _full_check(inp, 64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_segment_hand_off(dtype):
    """S_final of [0, t) passed as S0 of [t, T) equals one pass."""
    base = W["gdn_f32_b2h4t1024d64c64"] if dtype == "f32" else W["gdn_bf16_b4h16t4096d128c64"]
    inp = workloads.make_inputs(base, B=1, H=2, T=300)
    o, s = run_gpu(inp, base.C)
    t = 130
    a = dict(inp)
    b = dict(inp)
    for key in ("q", "k", "v", "log_alpha", "beta"):
        a[key] = inp[key][:, :t].contiguous()
        b[key] = inp[key][:, t:].contiguous()
    a["T"], b["T"] = t, 300 - t
    oa, sa = run_gpu(a, base.C)
    b["S0"] = torch.from_numpy(sa).float()
    ob, sb = run_gpu(b, base.C)
    fp32 = dtype == "f32"
    assert_close(np.concatenate([oa, ob], 1), o, fp32, "out hand-off", stored_bf16=not fp32)
    assert_close(sb, s, fp32, "S_final hand-off")


def test_deterministic():
    inp = workloads.make_inputs(W["gdn_bf16_b4h16t4096d128c64"], B=1, H=4, T=500)
    o1, s1 = run_gpu(inp, 64)
    o2, s2 = run_gpu(inp, 64)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_host_tensors_round_trip():
    """The public call with pinned host tensors copies in, runs and copies out."""
    inp = workloads.make_inputs(W["gdn_f32_b2h4t1024d64c64"], B=1, H=2, T=100)
    pin = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in inp.items()}
    out, Sf = gdn.chunk_fwd(pin["q"], pin["k"], pin["v"], pin["log_alpha"], pin["beta"],
                            pin["S0"], None, C=64)
    assert not out.is_cuda
    ro, rs = run_oracle(inp)
    assert_close(out.double().numpy(), ro, True, "out")
    assert_close(Sf.double().numpy(), rs, True, "S_final")


def test_selected_path_reported():
    p = gdn.gdn_select_path(128, 128, 64, torch.bfloat16)
    assert p in (gdn.GDN_PATH_SIMT, gdn.GDN_PATH_TCGEN05)
    assert gdn.gdn_select_path(64, 64, 64, torch.float32) == gdn.GDN_PATH_TF32
    assert gdn.gdn_select_path(16, 16, 16, torch.float32) == gdn.GDN_PATH_SIMT
