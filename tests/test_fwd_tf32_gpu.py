"""The chunk form on the tensor cores for the shapes the bf16 headline kernel does not take
(GDN_PATH_TF32: dk = dv = 64 or 128, C = 16, 32 or 64, fp32 q/k/v, or bf16 off the bf16
kernel's shape), against the fp64 oracle element by element.  Its products and state
chain run in three TF32 passes, so the
fp32 bound (relative max error 1e-4) applies to every fp32 result, S_final of bf16 inputs
included; a bf16 output is also held to one bf16 rounding unit per element."""
import numpy as np
import pytest
import torch

import chunkwise_gated_deltanet_gb300 as gdn
import workloads
from tests.parity import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _wl(dtype, d, T, B=2, H=2, alpha_mu=2.0, C=64):
    return workloads.Workload("tf32", dtype, B=B, H=H, T=T, dk=d, dv=d, C=C,
                              alpha_mu=alpha_mu, s0_std=0.1)


def _check(inp, C=64):
    o, s = run_gpu(inp, C)
    ro, rs = run_oracle(inp)
    if inp["dtype"] == "f32":
        assert_close(o, ro, True, "out")
    else:
        assert_close(o, ro, False, "out", stored_bf16=True)
        # the output before its bf16 rounding is fp32-accurate: within half a bf16 unit
        d = np.abs(o - ro) - 2.0 ** -8 * np.abs(ro)
        assert d.max() <= 1e-4 * np.abs(ro).max(), "bf16 out beyond its rounding"
    assert_close(s, rs, True, "S_final")


@pytest.mark.parametrize("d,dtype,C", [(64, "f32", 64), (128, "f32", 64), (64, "bf16", 64),
                                       (64, "f32", 16), (128, "bf16", 32)])
def test_path_is_the_chunk_form(d, dtype, C):
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    assert gdn.gdn_select_path(d, d, C, dt) == gdn.GDN_PATH_TF32
    assert gdn.gdn_launches_per_call(d, d, C, dt) == 10


@pytest.mark.parametrize("C", [16, 32])
@pytest.mark.parametrize("d,dtype", [(64, "f32"), (128, "f32"), (128, "bf16")])
def test_shorter_chunks(d, dtype, C):
    """Chunks of 16 or 32 tokens: each padded to a 64-row entry, which must add nothing;
    lengths that leave a ragged last chunk."""
    _check(workloads.make_inputs(_wl(dtype, d, 150, C=C), seed=16), C)


def test_shorter_chunks_packed_and_reset():
    lens = [0, 17, 33, 100, 1]
    inp = workloads.make_inputs(_wl("f32", 128, sum(lens), B=1, C=16), seed=17)
    inp["cu_seqlens"] = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    inp["N"] = len(lens)
    g = torch.Generator().manual_seed(18)
    inp["S0"] = torch.randn(len(lens), 2, 128, 128, generator=g) * 0.1
    la = inp["log_alpha"].clone()
    la[:, 40] = -float("inf")
    inp["log_alpha"] = la
    _check(inp, 16)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
@pytest.mark.parametrize("d,dtype", [(64, "f32"), (128, "f32"), (64, "bf16")])
def test_lengths_and_shapes(d, dtype, T):
    _check(workloads.make_inputs(_wl(dtype, d, T), seed=11))


@pytest.mark.parametrize("d", [64, 128])
def test_packed_with_empty_and_short_sequences(d):
    lens = [0, 1, 64, 65, 3, 0, 130, 17]
    inp = workloads.make_inputs(_wl("f32", d, sum(lens), B=1), seed=12)
    inp["cu_seqlens"] = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    inp["N"] = len(lens)
    inp["S0"] = torch.randn(len(lens), 2, d, d, generator=torch.Generator().manual_seed(13)) * 0.1
    _check(inp)


def test_strong_decay_and_resets():
    """alpha = sigmoid(N(-2, 1)) (strong decay), and alpha = 0 at some tokens (full reset)."""
    inp = workloads.make_inputs(_wl("f32", 128, 300, alpha_mu=-2.0), seed=14)
    la = inp["log_alpha"].clone()
    la[:, 64] = -float("inf")
    la[:, 150] = -float("inf")
    inp["log_alpha"] = la
    _check(inp)


def test_without_S0_and_deterministic():
    inp = workloads.make_inputs(_wl("f32", 128, 333), seed=15)
    inp["S0"] = None
    o1, s1 = run_gpu(inp, 64)
    o2, s2 = run_gpu(inp, 64)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)
    ro, rs = run_oracle(inp)
    assert_close(o1, ro, True, "out")
    assert_close(s1, rs, True, "S_final")
