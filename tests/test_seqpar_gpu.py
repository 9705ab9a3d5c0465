"""GPU checks of the sequence-parallel pieces: gdn_state_fold against fp64 matrix
products, and the whole split (every rank run in turn on one device through
the CUDA library) against the unsplit oracle.  Tolerances are those of the chunk
forward (tests/parity.py)."""
import numpy as np
import pytest
import torch

import chunkwise_gated_deltanet_gb300 as gdn
import workloads
from chunkwise_gated_deltanet_gb300 import seqpar
from oracle import native
from tests.parity import assert_close, to_device

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _fold_ref(S_in, Ms, Ls):
    S = None if S_in is None else S_in.double()
    for M, L in zip(Ms.double(), Ls.double()):
        S = L if S is None else S @ M + L
    return S


def _rand(shape, g, scale=1.0):
    return torch.randn(*shape, generator=g) * scale


@pytest.mark.parametrize("dv,dk", [(128, 128), (16, 128), (128, 16), (64, 32), (16, 16),
                                   (32, 64)])
@pytest.mark.parametrize("count", [1, 2, 5])
@pytest.mark.parametrize("with_input", [True, False])
def test_state_fold_matches_matmul(dv, dk, count, with_input):
    g = torch.Generator().manual_seed(dv * 7 + dk + count)
    units = (3, 5)
    S = _rand((*units, dv, dk), g)
    Ms = _rand((count, *units, dk, dk), g, dk ** -0.5)
    Ls = _rand((count, *units, dv, dk), g)
    out = torch.empty(*units, dv, dk, device="cuda")
    gdn.gdn_state_fold(S.cuda() if with_input else None, Ms.cuda(), Ls.cuda(), out)
    torch.cuda.synchronize()
    ref = _fold_ref(S if with_input else None, Ms, Ls)
    err = (out.cpu().double() - ref).abs().max() / ref.abs().max()
    assert err <= 1e-5, err


@pytest.mark.parametrize("alias", ["S_in", "L"])
def test_state_fold_in_place(alias):
    g = torch.Generator().manual_seed(1)
    S, Ms, Ls = _rand((4, 64, 64), g), _rand((3, 4, 64, 64), g, 0.125), _rand((3, 4, 64, 64), g)
    Sd, Md, Ld = S.cuda(), Ms.cuda(), Ls.cuda()
    out = Sd if alias == "S_in" else Ld[0]
    gdn.gdn_state_fold(Sd, Md, Ld, out)
    torch.cuda.synchronize()
    ref = _fold_ref(S, Ms, Ls)
    assert (out.cpu().double() - ref).abs().max() / ref.abs().max() <= 1e-5


def _oracle(inp, linear):
    if not linear:
        return native.gdn_forward_c(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"],
                                    inp["S0"])
    z = torch.zeros_like(inp["log_alpha"])
    return native.gdn_forward_c(inp["q"], inp["k"], inp["v"], inp["log_alpha"], z, inp["S0"],
                                erase=z, write=torch.ones_like(z))


def _split(inp, C, world, linear):
    d = to_device(inp)
    out, Sf = seqpar.emulate(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"], C,
                             world, linear)
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), Sf.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("world", [2, 3, 4])
@pytest.mark.parametrize("linear", [False, True], ids=["gdn", "linear"])
def test_split_f32_simt(world, linear):
    inp = workloads.make_inputs(W["gdn_f32_b2h4t1024d64c64"], B=2, H=2, T=300, seed=world)
    o, s = _split(inp, 64, world, linear)
    ro, rs = _oracle(inp, linear)
    assert_close(o, ro, True, "out")
    assert_close(s, rs, True, "S_final")


@pytest.mark.parametrize("world,linear", [(3, False), (4, True)])
def test_split_bf16_tcgen05(world, linear):
    """The long-sequence workload's shape family (S0 given, strong gate) split over
    several segments of the tcgen05 path."""
    inp = workloads.make_inputs(W["gdn_bf16_b1h32t32768d128c64"], B=1, H=3, T=1500, seed=world)
    o, s = _split(inp, 64, world, linear)
    ro, rs = _oracle(inp, linear)
    assert_close(o, ro, False, "out", stored_bf16=True)
    assert_close(s, rs, False, "S_final")


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("name", ["gdn_f32_b2h4t1024d64c64", "gdn_bf16_varlen256_h16d128c64"],
                         ids=["f32_d64", "bf16_d128"])
def test_split_packed(name, world):
    """A packed batch (members of uneven lengths, one shorter than a chunk, one empty):
    each member cut at its own chunk-aligned bounds, the ranks' packed segments run
    through the library and folded, against the unsplit oracle."""
    w = W[name]
    lens = [5, 0, 70, 130, 1, 200]
    # the fixed-length generator of the same dtype and head size, packed by hand
    base = w if not w.varlen else W["gdn_bf16_b4h16t4096d128c64"]
    inp = workloads.make_inputs(base, B=1, H=2, T=sum(lens), seed=world)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    inp["cu_seqlens"] = cu
    inp["N"] = len(lens)
    inp["S0"] = 0.1 * torch.randn(len(lens), 2, w.dv, w.dk,
                                  generator=torch.Generator().manual_seed(world))
    d = to_device(inp)
    out, Sf = seqpar.emulate(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"], 64,
                             world, False, cu_seqlens=d["cu_seqlens"])
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    o = out.float().cpu().numpy().astype(np.float64)
    s = Sf.cpu().numpy().astype(np.float64)
    ro, rs = native.gdn_forward_c(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"],
                                  inp["S0"], inp["cu_seqlens"])
    fp32 = inp["dtype"] == "f32"
    assert_close(o, ro, fp32, "out", stored_bf16=not fp32)
    assert_close(s, rs, fp32, "S_final")
