"""Helpers for the GPU parity tests: run the CUDA library, run the oracle, compare.

Tolerances (written here once, used by every parity test):
* fp32 q/k/v: max|delta| / max|ref| <= 1e-4, for out and for S_final.
* bf16 q/k/v with fp32 state, S_final (stored fp32):
  max|delta| <= 2e-2 * RMS(ref).
* bf16 out (stored bf16): every element |delta_i| <= 2e-2 * RMS(ref) + 2^-8 |ref_i|.
  The first term is the 2%-of-output-RMS bound on the computation; the second is
  the bf16 storage of that element (round-to-nearest moves a value by up to 2^-9
  of itself, and the computation can push it across one rounding boundary).
  Without it an exact fp32 result, rounded to bf16, already misses the bound on
  outputs near 10x the RMS.  RMS(delta)/RMS(ref) <= 2e-2 is checked as well.
"""
from __future__ import annotations

import numpy as np
import torch

import chunkwise_gated_deltanet_gb300 as gdn
from oracle import native

TOL_F32_REL_MAX = 1e-4
TOL_BF16_MAX_OVER_RMS = 2e-2
BF16_STORAGE_REL = 2.0 ** -8


def to_device(inp: dict, dev="cuda") -> dict:
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}


def run_gpu(inp: dict, C: int, S_final: bool = True, f64: bool = True):
    d = to_device(inp)
    out, Sf = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                            d["cu_seqlens"], C=C, output_final_state=S_final)
    gdn.gdn_check_status()
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    s = None if Sf is None else Sf.cpu().numpy()
    if f64:
        o = o.astype(np.float64)
        s = None if s is None else s.astype(np.float64)
    return o, s


def run_oracle(inp: dict):
    return native.gdn_forward_c(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"],
                                inp["S0"], inp["cu_seqlens"])


def errors(got: np.ndarray, ref: np.ndarray) -> dict:
    d = np.abs(got - ref)
    mx = float(d.max()) if d.size else 0.0
    rmax = float(np.abs(ref).max()) if ref.size else 0.0
    rms = float(np.sqrt((ref ** 2).mean())) if ref.size else 0.0
    return dict(max_abs=mx, rel_max=mx / rmax if rmax > 0 else mx,
                max_over_rms=mx / rms if rms > 0 else mx,
                rms_ratio=float(np.sqrt((d ** 2).mean())) / rms if rms > 0 else 0.0)


def assert_close(got, ref, fp32: bool, what: str, stored_bf16: bool = False):
    """fp32: relative max error.  bf16 inputs: 2e-2 of RMS(ref), plus one bf16
    rounding unit of each element when the result is stored in bf16."""
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    e = errors(got, ref)
    if fp32:
        assert e["rel_max"] <= TOL_F32_REL_MAX, f"{what}: {e}"
        return e
    rms = np.sqrt((ref ** 2).mean()) if ref.size else 0.0
    bound = TOL_BF16_MAX_OVER_RMS * rms
    if stored_bf16:
        bound = bound + BF16_STORAGE_REL * np.abs(ref)
    excess = np.abs(got - ref) - bound
    e["worst_excess_over_rms"] = float(excess.max() / rms) if ref.size and rms > 0 else 0.0
    assert (excess <= 0).all(), f"{what}: {e}"
    assert e["rms_ratio"] <= TOL_BF16_MAX_OVER_RMS, f"{what}: {e}"
    return e


def sample_units(N: int, H: int, count: int, seed: int = 0):
    """A deterministic sample of (sequence, head) pairs including both corners."""
    rng = np.random.default_rng(seed)
    units = {(0, 0), (N - 1, H - 1)}
    while len(units) < min(count, N * H):
        units.add((int(rng.integers(N)), int(rng.integers(H))))
    return sorted(units)


def compare_sampled(inp: dict, out: np.ndarray, Sf: np.ndarray, units, fp32: bool):
    """Compare the listed units of a full GPU run against the oracle run on
    those units alone."""
    res = native.gdn_units_c(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"],
                             inp["S0"], inp["cu_seqlens"], units)
    spans = native.spans(inp["B"], inp["T"], inp["cu_seqlens"])
    o_flat = out.reshape(inp["B"] * inp["T"], inp["H"], -1)
    got_o, ref_o, got_s, ref_s = [], [], [], []
    for (n, h), (ro, rs) in zip(units, res):
        r0, ln = spans[n]
        got_o.append(o_flat[r0:r0 + ln, h])
        ref_o.append(ro)
        got_s.append(Sf[n, h])
        ref_s.append(rs)
    eo = assert_close(np.concatenate(got_o), np.concatenate(ref_o), fp32, "out (sampled)",
                      stored_bf16=not fp32)
    es = assert_close(np.stack(got_s), np.stack(ref_s), fp32, "S_final (sampled)")
    return eo, es


def compare_all_units(inp: dict, out: np.ndarray, Sf: np.ndarray, block_rows: int = 1 << 14):
    """Every (sequence, head) unit of a full-size bf16 run against the oracle run on
    every unit, with the bf16 bounds of ``assert_close``; the comparison walks the
    token rows in blocks so that a multi-GB output needs no multi-GB temporaries.
    ``out`` may be fp32 (the bf16 outputs are exact in it)."""
    ref_o, ref_s = run_oracle(inp)
    assert out.shape == ref_o.shape and Sf.shape == ref_s.shape
    ro = ref_o.reshape(-1, ref_o.shape[-1])
    go = out.reshape(-1, out.shape[-1])
    ss = 0.0
    for r in range(0, ro.shape[0], block_rows):
        ss += float((ro[r:r + block_rows] ** 2).sum())
    rms = np.sqrt(ss / ro.size)
    worst, dss = -np.inf, 0.0
    for r in range(0, ro.shape[0], block_rows):
        g = go[r:r + block_rows].astype(np.float64)
        x = ro[r:r + block_rows]
        assert np.isfinite(g).all(), "out: non-finite values"
        d = np.abs(g - x)
        dss += float((d ** 2).sum())
        worst = max(worst, float((d - TOL_BF16_MAX_OVER_RMS * rms - BF16_STORAGE_REL * np.abs(x)).max()))
    e = dict(worst_excess_over_rms=worst / rms, rms_ratio=np.sqrt(dss / ro.size) / rms,
             units=int(ref_s.shape[0] * ref_s.shape[1]))
    assert worst <= 0, f"out (every unit): {e}"
    assert e["rms_ratio"] <= TOL_BF16_MAX_OVER_RMS, f"out (every unit): {e}"
    es = assert_close(Sf.astype(np.float64), ref_s, False, "S_final (every unit)")
    return e, es
