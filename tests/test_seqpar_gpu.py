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


@pytest.mark.parametrize("alpha_one", [False, True], ids=["mamba2", "linear_attention"])
@pytest.mark.parametrize("B,H,T", [(2, 3, 333), (1, 1, 64), (4, 16, 200)])
def test_linear_state_correct_equals_the_run_from_S_start(B, H, T, alpha_one):
    """A linear-mode run from zero, then gdn_linear_state_correct with S_start, against
    the oracle's run from S_start (outputs and end state)."""
    w = W["linear_bf16_b4h16t4096d128c64"]
    inp = workloads.make_inputs(w, B=B, H=H, T=T, seed=B * T + H)
    if alpha_one:
        inp["log_alpha"] = torch.zeros_like(inp["log_alpha"])
    S_start = torch.randn(B, H, 128, 128, generator=torch.Generator().manual_seed(T)) * 0.1
    d = to_device(inp)
    la = None if alpha_one else d["log_alpha"]
    out, S_end = gdn.linear_chunk_fwd(d["q"], d["k"], d["v"], la, None, None, C=64)
    gdn.gdn_linear_state_correct(d["q"], la, S_start.cuda(), out, S_end)
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    ref = dict(inp, S0=S_start)
    ro, rs = _oracle(ref, True)
    assert_close(out.float().cpu().numpy().astype(np.float64), ro, False, "out",
                 stored_bf16=True)
    assert_close(S_end.cpu().numpy().astype(np.float64), rs, False, "S_final")


def test_linear_state_correct_edge_cases():
    """T = 0 adds S_start to S_end (no outputs); S_end = None corrects the outputs only;
    unsupported sizes are refused before any launch."""
    S_start = torch.randn(2, 2, 128, 128, device="cuda")
    S_end = torch.randn(2, 2, 128, 128, device="cuda")
    q0 = torch.empty(2, 0, 2, 128, dtype=torch.bfloat16, device="cuda")
    o0 = torch.empty(2, 0, 2, 128, dtype=torch.bfloat16, device="cuda")
    expect = S_end + S_start
    gdn.gdn_linear_state_correct(q0, None, S_start, o0, S_end)
    torch.cuda.synchronize()
    assert torch.equal(S_end, expect)
    w = W["linear_bf16_b4h16t4096d128c64"]
    inp = workloads.make_inputs(w, B=1, H=2, T=130, seed=5)
    d = to_device(inp)
    out, _ = gdn.linear_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], None, None, C=64,
                                  output_final_state=False)
    gdn.gdn_linear_state_correct(d["q"], d["log_alpha"], S_start[:1].contiguous(), out, None)
    torch.cuda.synchronize()
    ro, _ = _oracle(dict(inp, S0=S_start[:1].cpu()), True)
    assert_close(out.float().cpu().numpy().astype(np.float64), ro, False, "out",
                 stored_bf16=True)
    assert not gdn.gdn_linear_state_correct_supported(64, 64, torch.bfloat16)
    assert not gdn.gdn_linear_state_correct_supported(128, 128, torch.float32)
    qf = torch.zeros(1, 4, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gdn.GdnError):
        gdn.gdn_linear_state_correct(qf, None, torch.zeros(1, 2, 64, 64, device="cuda"),
                                     torch.zeros_like(qf), None)


@pytest.mark.parametrize("world", [2, 4])
def test_linear_split_corrects_instead_of_rerunning(world):
    """The bf16 d = 128 linear mode: ranks r > 0 correct their runs from zero (checked
    against the oracle; the correcting path is the one the CUDA ops choose here)."""
    inp = workloads.make_inputs(W["linear_bf16_b4h16t4096d128c64"], B=2, H=2, T=900,
                                seed=world + 40)
    inp["S0"] = torch.randn(2, 2, 128, 128, generator=torch.Generator().manual_seed(world)) * 0.1
    d = to_device(inp)
    assert seqpar.cuda_ops().correctable(d["q"], d["v"], None)
    o, s = _split(inp, 64, world, True)
    ro, rs = _oracle(inp, True)
    assert_close(o, ro, False, "out", stored_bf16=True)
    assert_close(s, rs, False, "S_final")


@pytest.mark.parametrize("packed", [False, True])
def test_linear_segment_map_is_the_gain_times_identity(packed):
    """M[n][h] = e^{sum of log alpha over the sequence} I, fixed-length and packed (an
    empty member gives I, a reset anywhere gives 0), against fp64 sums."""
    g = torch.Generator().manual_seed(3)
    if packed:
        lens = [0, 5, 64, 130, 1]
        T, B, N = sum(lens), 1, len(lens)
        cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    else:
        T, B, N, cu = 300, 2, 2, None
    H, dk = 3, 64
    la = -torch.nn.functional.softplus(-(torch.randn(B, T, H, generator=g) + 4.0)) * 0.05
    la[0, 7, 1] = -float("inf")
    M = torch.empty(N, H, dk, dk, device="cuda")
    gdn.gdn_linear_segment_map(la.cuda(), M, B, T, None if cu is None else cu.cuda())
    torch.cuda.synchronize()
    spans = [(n, 0, n * T, (n + 1) * T) for n in range(B)] if cu is None else \
        [(n, 0, int(cu[n]), int(cu[n + 1])) for n in range(N)]
    for n, _, a, b in spans:
        for h in range(H):
            flat = la.reshape(-1, H)[a:b, h].double()
            gam = float(torch.exp(flat.sum())) if b > a else 1.0
            ref = gam * np.eye(dk)
            got = M[n, h].double().cpu().numpy()
            assert np.abs(got - ref).max() <= 1e-5 * max(gam, 1e-30) + 1e-30, (n, h, gam)
    M1 = torch.empty(N, H, dk, dk, device="cuda")
    gdn.gdn_linear_segment_map(None, M1, B, T, None if cu is None else cu.cuda())
    torch.cuda.synchronize()
    assert torch.equal(M1, torch.eye(dk, device="cuda").expand(N, H, dk, dk))


@pytest.mark.parametrize("name", ["gdn_f32_b2h4t1024d64c64", "linear_bf16_b4h16t4096d128c64"])
@pytest.mark.parametrize("world", [2, 3])
def test_split_packed_linear_mode(name, world):
    """The linear mode on a packed batch: each member cut at its own bounds; the middle
    ranks' maps M = (prod alpha) I come from gdn_linear_segment_map with the ranks'
    cu_seqlens, the ranks run their segments again from the folded start states."""
    w = W[name]
    lens = [5, 0, 70, 130, 1, 200]
    inp = workloads.make_inputs(w, B=1, H=2, T=sum(lens), seed=world + 7)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    inp["cu_seqlens"] = cu
    inp["N"] = len(lens)
    inp["S0"] = 0.1 * torch.randn(len(lens), 2, w.dv, w.dk,
                                  generator=torch.Generator().manual_seed(world + 7))
    d = to_device(inp)
    out, Sf = seqpar.emulate(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"], 64,
                             world, True, cu_seqlens=d["cu_seqlens"])
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    o = out.float().cpu().numpy().astype(np.float64)
    s = Sf.cpu().numpy().astype(np.float64)
    z = torch.zeros_like(inp["log_alpha"])
    ro, rs = native.gdn_forward_c(inp["q"], inp["k"], inp["v"], inp["log_alpha"], z, inp["S0"],
                                  inp["cu_seqlens"], erase=z, write=torch.ones_like(z))
    fp32 = inp["dtype"] == "f32"
    assert_close(o, ro, fp32, "out", stored_bf16=not fp32)
    assert_close(s, rs, fp32, "S_final")


def test_linear_state_correct_many_units():
    """More (sequence, head) units than two CTAs an SM hold (B = 20, H = 16: 320): each
    correction CTA takes a run of whole sequences, folds a start state per sequence and
    writes each one's S_final; ragged last tiles (T = 100)."""
    w = W["linear_bf16_b4h16t4096d128c64"]
    inp = workloads.make_inputs(w, B=20, H=16, T=100, seed=61)
    S_start = torch.randn(20, 16, 128, 128, generator=torch.Generator().manual_seed(62)) * 0.1
    d = to_device(inp)
    out, S_end = gdn.linear_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], None, None, C=64)
    gdn.gdn_linear_state_correct(d["q"], d["log_alpha"], S_start.cuda(), out, S_end)
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    ro, rs = _oracle(dict(inp, S0=S_start), True)
    assert_close(out.float().cpu().numpy().astype(np.float64), ro, False, "out",
                 stored_bf16=True)
    assert_close(S_end.cpu().numpy().astype(np.float64), rs, False, "S_final")
