"""GPU parity of the single-token decode step (gdn_decode_step) against the oracle.

The oracle is the per-token recurrence itself (oracle.native, fp64): one token per
(sequence, head) with S0 = the state before the step.  The step computes in fp32
from inputs that fp64 holds exactly, so the state (stored fp32) must match to the
fp32 bound, max|delta| / max|ref| <= 1e-4, for both input dtypes.  fp32 outputs
take the same bound; bf16 outputs additionally get their own storage rounding,
|delta_i| <= 2^-8 |ref_i| + 1e-4 max|ref|.
"""
import numpy as np
import pytest
import torch

import chunkwise_gated_deltanet_gb300 as gdn
import workloads
from oracle import native
from tests.parity import TOL_F32_REL_MAX, run_gpu, to_device

pytestmark = pytest.mark.gpu

W_BF16 = workloads.DECODE_WORKLOADS["decode_bf16_n256h16d128"]
W_F32 = workloads.DECODE_WORKLOADS["decode_f32_n64h8d64"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunkwise_gated_deltanet_gb300 import build
    build.build()
    gdn.load_library()


def _oracle_step(inp):
    """The oracle on a one-token sequence per (sequence, head), starting from S."""
    o, S = native.gdn_forward_c(inp["q"].unsqueeze(1), inp["k"].unsqueeze(1),
                                inp["v"].unsqueeze(1), inp["log_alpha"].unsqueeze(1),
                                inp["beta"].unsqueeze(1), inp["S"], None)
    return o[:, 0], S


def _gpu_step(inp):
    d = to_device(inp)
    S = d["S"].clone()
    out = gdn.decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S)
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), S.cpu().numpy().astype(np.float64)


def _check(got_o, got_S, ref_o, ref_S, bf16_out: bool, what: str):
    assert np.isfinite(got_o).all() and np.isfinite(got_S).all(), what
    ds = np.abs(got_S - ref_S).max() / max(np.abs(ref_S).max(), 1e-30)
    assert ds <= TOL_F32_REL_MAX, f"{what}: state rel max {ds}"
    ref_max = max(np.abs(ref_o).max(), 1e-30)
    d = np.abs(got_o - ref_o)
    if bf16_out:
        excess = (d - 2.0 ** -8 * np.abs(ref_o)).max() / ref_max
        assert excess <= TOL_F32_REL_MAX, f"{what}: out excess {excess}"
    else:
        assert d.max() / ref_max <= TOL_F32_REL_MAX, f"{what}: out rel max {d.max() / ref_max}"


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (16, 128), (128, 16), (32, 64), (16, 16)])
@pytest.mark.parametrize("w", [W_BF16, W_F32], ids=["bf16", "f32"])
def test_decode_matches_oracle(w, dk, dv):
    inp = workloads.make_decode_inputs(w, N=12, H=3, dk=dk, dv=dv, seed=dk + dv)
    o, S = _gpu_step(inp)
    ro, rS = _oracle_step(inp)
    _check(o, S, ro, rS, w.dtype == "bf16", f"{w.dtype} dk={dk} dv={dv}")


@pytest.mark.parametrize("w", [W_BF16, W_F32], ids=["bf16", "f32"])
def test_decode_full_workload(w):
    inp = workloads.make_decode_inputs(w)
    o, S = _gpu_step(inp)
    ro, rS = _oracle_step(inp)
    _check(o, S, ro, rS, w.dtype == "bf16", w.name)


def test_decode_gate_extremes():
    """alpha = 1 (plain DeltaNet), alpha ~ 0 (state forgotten), beta = 0 (no write)."""
    inp = workloads.make_decode_inputs(W_F32, N=6, H=4, seed=7)
    inp["log_alpha"][0] = 0.0
    inp["log_alpha"][1] = -60.0
    inp["beta"][2] = 0.0
    o, S = _gpu_step(inp)
    ro, rS = _oracle_step(inp)
    _check(o, S, ro, rS, False, "gate extremes")


def test_decode_continues_the_chunk_forward():
    """T tokens by gdn_chunk_fwd, then 3 decode steps == the oracle on T + 3 tokens."""
    w = workloads.WORKLOADS["gdn_f32_b2h4t1024d64c64"]
    full = workloads.make_inputs(w, T=203, seed=3)
    T0 = 200
    head = dict(full)
    for name in ("q", "k", "v", "log_alpha", "beta"):
        head[name] = full[name][:, :T0].contiguous()
    head["T"] = T0
    _, S = run_gpu(head, C=64)
    state = torch.from_numpy(S).float().contiguous()
    outs = []
    for t in range(T0, T0 + 3):
        step = dict(q=full["q"][:, t].contiguous(), k=full["k"][:, t].contiguous(),
                    v=full["v"][:, t].contiguous(), log_alpha=full["log_alpha"][:, t].contiguous(),
                    beta=full["beta"][:, t].contiguous(), S=state)
        o, Snew = _gpu_step(step)
        outs.append(o)
        state = torch.from_numpy(Snew).float().contiguous()
    ro, rS = native.gdn_forward_c(full["q"], full["k"], full["v"], full["log_alpha"],
                                  full["beta"], full["S0"], None)
    got_o = np.stack(outs, axis=1)
    _check(got_o, state.numpy().astype(np.float64), ro[:, T0:], rS, False, "chunk + decode")


def test_decode_updates_in_place_and_empty_batch():
    inp = workloads.make_decode_inputs(W_BF16, N=2, H=2, seed=11)
    d = to_device(inp)
    S = d["S"].clone()
    ptr = S.data_ptr()
    out = torch.empty_like(d["v"])
    gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S, out)
    torch.cuda.synchronize()
    assert S.data_ptr() == ptr and not torch.equal(S, d["S"])
    empty = workloads.make_decode_inputs(W_BF16, N=0, H=2)
    e = to_device(empty)
    gdn.gdn_decode_step(e["q"], e["k"], e["v"], e["log_alpha"], e["beta"], e["S"],
                        torch.empty_like(e["v"]))
    gdn.gdn_check_status()


def test_decode_deterministic():
    inp = workloads.make_decode_inputs(W_BF16, N=16, H=4, seed=5)
    a = _gpu_step(inp)
    b = _gpu_step(inp)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("pieces", [1, 3, 4, 64])
def test_decode_host_path_equals_device_path(pieces):
    """decode_step on pinned host tensors (gdn_decode_step_host, copies pipelined over
    slices of sequences) gives bit for bit the device path's output and new state."""
    inp = workloads.make_decode_inputs(W_BF16, N=37, H=3, seed=13)
    d = to_device(inp)
    S_dev = d["S"].clone()
    out_dev = gdn.decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S_dev)
    h = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in inp.items()}
    S_host = h["S"].clone().pin_memory()
    out_host = gdn.decode_step(h["q"], h["k"], h["v"], h["log_alpha"], h["beta"], S_host,
                               pieces=pieces)
    torch.cuda.synchronize()
    assert not out_host.is_cuda
    assert torch.equal(out_dev.cpu(), out_host)
    assert torch.equal(S_dev.cpu(), S_host)
