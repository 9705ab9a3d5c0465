"""The host-tensor path of chunk_fwd / linear_chunk_fwd (copies pipelined over token
ranges on separate streams, each range starting from the previous one's fp32 final
state) gives bit-for-bit the results of the device path where both run the same kernel
over the same chunks: the ranges are whole chunks, so the kernels see the same chunks and
the same fp32 state.  The linear mode's device path may split sequences over more SMs,
so there both paths are held to the oracle."""
import numpy as np
import pytest
import torch

import chunkwise_gated_deltanet_gb300 as gdn
import workloads
from oracle import native
from tests.parity import assert_close, to_device

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _pin(inp):
    return {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in inp.items()}


def _same(dev_res, host_res):
    for a, b in zip(dev_res, host_res):
        assert not b.is_cuda
        assert torch.equal(a.cpu(), b)


def _both_match_oracle_linear(dev_res, host_res, inp, alpha_one):
    """The linear mode's device path may split each sequence over more SMs (its segments'
    start states folded in fp32, a different order of sums than one pass), so the host
    path, which runs whole-chunk ranges in order, is held with it to the oracle."""
    z = torch.zeros_like(inp["log_alpha"])
    la = z if alpha_one else inp["log_alpha"]
    ro, rs = native.gdn_forward_c(inp["q"], inp["k"], inp["v"], la, z, inp["S0"],
                                  inp["cu_seqlens"], erase=z, write=torch.ones_like(z))
    for res in (dev_res, host_res):
        assert_close(res[0].float().cpu().numpy().astype(np.float64), ro, False, "out",
                     stored_bf16=True)
        assert_close(res[1].cpu().numpy().astype(np.float64), rs, False, "S_final")


@pytest.mark.parametrize("pieces", [1, 3, 4, 64])
@pytest.mark.parametrize("name,shrink", [
    ("gdn_bf16_b4h16t4096d128c64", dict(B=2, H=3, T=333)),
    ("gdn_f32_b2h4t1024d64c64", dict(B=2, H=2, T=200)),
])
def test_host_path_equals_device_path(name, shrink, pieces):
    w = W[name]
    inp = workloads.make_inputs(w, **shrink)
    if inp["S0"] is None:
        inp["S0"] = 0.1 * torch.randn((inp["N"], inp["H"], w.dv, w.dk),
                                      generator=torch.Generator().manual_seed(1))
    d, h = to_device(inp), _pin(inp)
    dev = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"], C=w.C)
    host = gdn.chunk_fwd(h["q"], h["k"], h["v"], h["log_alpha"], h["beta"], h["S0"], C=w.C,
                         pieces=pieces)
    torch.cuda.synchronize()
    _same(dev, host)


def test_host_path_linear_mode_and_packed_batch():
    w = W["gdn_bf16_b4h16t4096d128c64"]
    inp = workloads.make_inputs(w, B=2, H=2, T=300, seed=3)
    d, h = to_device(inp), _pin(inp)
    dev = gdn.linear_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], None, C=64)
    host = gdn.linear_chunk_fwd(h["q"], h["k"], h["v"], h["log_alpha"], None, C=64)
    torch.cuda.synchronize()
    _both_match_oracle_linear(dev, host, inp, False)
    pk = workloads.make_inputs(W["gdn_bf16_varlen256_h16d128c64"], n_seqs=3, H=2, seed=4)
    d, h = to_device(pk), _pin(pk)
    dev = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], None, d["cu_seqlens"])
    host = gdn.chunk_fwd(h["q"], h["k"], h["v"], h["log_alpha"], h["beta"], None,
                         h["cu_seqlens"])
    torch.cuda.synchronize()
    _same(dev, host)


def test_host_path_empty_sequence():
    w = W["gdn_f32_b2h4t1024d64c64"]
    inp = workloads.make_inputs(w, B=2, H=2, T=0)
    h = _pin(inp)
    out, Sf = gdn.chunk_fwd(h["q"], h["k"], h["v"], h["log_alpha"], h["beta"], h["S0"], C=64)
    assert out.numel() == 0 and torch.equal(Sf, inp["S0"])


def test_host_path_linear_attention_without_gates():
    """The linear mode with log_alpha = None (alpha = 1) through the native host path."""
    w = W["gdn_bf16_b4h16t4096d128c64"]
    inp = workloads.make_inputs(w, B=2, H=2, T=257, seed=8)
    d, h = to_device(inp), _pin(inp)
    dev = gdn.linear_chunk_fwd(d["q"], d["k"], d["v"], None, None, C=64)
    host = gdn.linear_chunk_fwd(h["q"], h["k"], h["v"], None, None, C=64, pieces=3)
    torch.cuda.synchronize()
    _both_match_oracle_linear(dev, host, inp, True)
