"""Seeded synthetic inputs for the chunkwise Gated DeltaNet forward.

This module is shared by the tests, ``bench.py`` and ``__graft_entry__.smoke``.
It only draws random numbers and shapes them; it holds none of the method's
arithmetic (no recurrence, no decay products, no solves).  Both the CUDA path and
the CPU oracle consume exactly the tensors it returns.

Recipe (the pages fix only the recurrence; the distributions are the five
workloads of the Gated DeltaNet forward that this library is measured on):

* q, k ~ N(0, 1), then divided by their L2 norm over the head dimension (in
  fp32), then cast to the workload's dtype.  The cast values are what both sides
  see, so they are not exactly unit-norm in bf16.
* v ~ N(0, 1), cast to the workload's dtype.
* beta = sigmoid(x), x ~ N(0, 1), fp32.
* log_alpha = log sigmoid(x) = -softplus(-x), x ~ N(mu, 1), fp32 (mu = 2 or 3);
  plain DeltaNet uses log_alpha = 0 (alpha = 1).
* S0 ~ N(0, 0.1^2) per (sequence, head) where the workload says so, else None.
* Packed variable-length batches draw lengths uniform in [lo, hi] first (they
  size every other tensor), then the tensors above over the packed tokens.

Draw order after the lengths: q, k, v, beta-logits, alpha-logits, S0, all from one
``torch.Generator`` seeded with the workload's seed, drawn in fp32 on the CPU.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "f32" or "bf16": the dtype of q, k, v and out
    B: int
    H: int
    T: int                # tokens per sequence (fixed-length) or 0 for packed
    dk: int
    dv: int
    C: int
    alpha_mu: Optional[float]   # None => plain DeltaNet (log_alpha = 0)
    s0_std: float               # 0 => S0 is None
    seed: int = 0
    n_seqs: int = 0             # >0 => packed variable-length batch (B must be 1)
    len_lo: int = 0
    len_hi: int = 0
    linear: bool = False        # True => the linear (Mamba2) mode: no beta, erase 0, write 1

    @property
    def varlen(self) -> bool:
        return self.n_seqs > 0


# The five workloads, by what they are.
WORKLOADS = {
    "deltanet_f32_b1h1t64d16c16": Workload(
        "deltanet_f32_b1h1t64d16c16", "f32", B=1, H=1, T=64, dk=16, dv=16, C=16,
        alpha_mu=None, s0_std=0.0),
    "gdn_f32_b2h4t1024d64c64": Workload(
        "gdn_f32_b2h4t1024d64c64", "f32", B=2, H=4, T=1024, dk=64, dv=64, C=64,
        alpha_mu=2.0, s0_std=0.1),
    "gdn_bf16_b4h16t4096d128c64": Workload(
        "gdn_bf16_b4h16t4096d128c64", "bf16", B=4, H=16, T=4096, dk=128, dv=128, C=64,
        alpha_mu=2.0, s0_std=0.0),
    "gdn_bf16_b1h32t32768d128c64": Workload(
        "gdn_bf16_b1h32t32768d128c64", "bf16", B=1, H=32, T=32768, dk=128, dv=128, C=64,
        alpha_mu=3.0, s0_std=0.1),
    "gdn_bf16_varlen256_h16d128c64": Workload(
        "gdn_bf16_varlen256_h16d128c64", "bf16", B=1, H=16, T=0, dk=128, dv=128, C=64,
        alpha_mu=2.0, s0_std=0.0, n_seqs=256, len_lo=64, len_hi=2048),
    # the headline sizes in the linear (Mamba2) mode: same draws, beta unused
    "linear_bf16_b4h16t4096d128c64": Workload(
        "linear_bf16_b4h16t4096d128c64", "bf16", B=4, H=16, T=4096, dk=128, dv=128, C=64,
        alpha_mu=2.0, s0_std=0.0, linear=True),
    # the long-sequence sizes in the linear mode (32 units: each sequence split over SMs)
    "linear_bf16_b1h32t32768d128c64": Workload(
        "linear_bf16_b1h32t32768d128c64", "bf16", B=1, H=32, T=32768, dk=128, dv=128, C=64,
        alpha_mu=3.0, s0_std=0.1, linear=True),
}

# The headline workload that bench.py times by default.
HEADLINE = "gdn_bf16_b4h16t4096d128c64"


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    # Data shaping only: scale each (token, head) row to unit length in fp32.
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def make_inputs(w: Workload, *, B: Optional[int] = None, H: Optional[int] = None,
                T: Optional[int] = None, n_seqs: Optional[int] = None,
                seed: Optional[int] = None) -> dict:
    """Draw the seeded inputs of workload ``w`` on the CPU.

    Keyword overrides shrink a workload (same distributions, fewer units) for
    tests.  Returns a dict with CPU tensors:

    q, k: [B, T, H, dk]; v: [B, T, H, dv] in the workload dtype (packed batches
    have B = 1 and T = total tokens); log_alpha, beta: [B, T, H] fp32;
    S0: [N, H, dv, dk] fp32 or None; cu_seqlens: int32 [N+1] or None;
    plus the integer sizes.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    T = w.T if T is None else T
    seed = w.seed if seed is None else seed
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    cu = None
    if w.varlen:
        n = w.n_seqs if n_seqs is None else n_seqs
        lens = torch.randint(w.len_lo, w.len_hi + 1, (n,), generator=g, dtype=torch.int64)
        cu = torch.zeros(n + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(lens, 0)
        B, T, N = 1, int(cu[-1]), n
        cu = cu.to(torch.int32)
    else:
        N = B
    dt = torch_dtype(w.dtype)
    q = _unit_rows(torch.randn(B, T, H, w.dk, generator=g)).to(dt)
    k = _unit_rows(torch.randn(B, T, H, w.dk, generator=g)).to(dt)
    v = torch.randn(B, T, H, w.dv, generator=g).to(dt)
    beta = torch.sigmoid(torch.randn(B, T, H, generator=g))
    if w.alpha_mu is None:
        log_alpha = torch.zeros(B, T, H)
    else:
        x = torch.randn(B, T, H, generator=g) + w.alpha_mu
        log_alpha = -torch.nn.functional.softplus(-x)
    S0 = None
    if w.s0_std > 0:
        S0 = torch.randn(N, H, w.dv, w.dk, generator=g) * w.s0_std
    return dict(q=q.contiguous(), k=k.contiguous(), v=v.contiguous(),
                log_alpha=log_alpha.contiguous(), beta=beta.contiguous(),
                S0=S0, cu_seqlens=cu, B=B, H=H, T=T, N=N, dk=w.dk, dv=w.dv,
                C=w.C, dtype=w.dtype)


def n_tokens(inp: dict) -> int:
    return inp["B"] * inp["T"]


# ---- single-token decode step (one token for each (sequence, head)) ----
# Recipe: q, k, v, beta, log_alpha as above with T = 1, plus the state
# S ~ N(0, s_std^2) per (sequence, head); draw order q, k, v, beta-logits,
# alpha-logits, S.  The batch is sized so that the state (N * H * dv * dk * 4
# bytes = 256 MiB at N = 256, H = 16, d = 128) is larger than the L2 cache.
@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    dtype: str
    N: int                # sequences
    H: int
    dk: int
    dv: int
    alpha_mu: float
    s_std: float
    seed: int = 0


DECODE_WORKLOADS = {
    "decode_bf16_n256h16d128": DecodeWorkload(
        "decode_bf16_n256h16d128", "bf16", N=256, H=16, dk=128, dv=128, alpha_mu=2.0, s_std=0.5),
    "decode_f32_n64h8d64": DecodeWorkload(
        "decode_f32_n64h8d64", "f32", N=64, H=8, dk=64, dv=64, alpha_mu=2.0, s_std=0.5),
}


def make_decode_inputs(w: DecodeWorkload, *, N: Optional[int] = None, H: Optional[int] = None,
                       dk: Optional[int] = None, dv: Optional[int] = None,
                       seed: Optional[int] = None) -> dict:
    """Draw the seeded inputs of decode workload ``w`` on the CPU: q, k [N, H, dk];
    v [N, H, dv] in the workload dtype; log_alpha, beta [N, H] fp32; S [N, H, dv, dk]
    fp32; plus the integer sizes."""
    N = w.N if N is None else N
    H = w.H if H is None else H
    dk = w.dk if dk is None else dk
    dv = w.dv if dv is None else dv
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    dt = torch_dtype(w.dtype)
    q = _unit_rows(torch.randn(N, H, dk, generator=g)).to(dt)
    k = _unit_rows(torch.randn(N, H, dk, generator=g)).to(dt)
    v = torch.randn(N, H, dv, generator=g).to(dt)
    beta = torch.sigmoid(torch.randn(N, H, generator=g))
    x = torch.randn(N, H, generator=g) + w.alpha_mu
    log_alpha = -torch.nn.functional.softplus(-x)
    S = torch.randn(N, H, dv, dk, generator=g) * w.s_std
    return dict(q=q.contiguous(), k=k.contiguous(), v=v.contiguous(),
                log_alpha=log_alpha.contiguous(), beta=beta.contiguous(), S=S.contiguous(),
                N=N, H=H, dk=dk, dv=dv, dtype=w.dtype)


def make_grad_inputs(inp: dict, seed: int = 1, ds_std: float = 0.1) -> dict:
    """Seeded upstream gradients for a backward test or benchmark of the inputs
    ``inp`` (from ``make_inputs``): d_out ~ N(0, 1) in the qkv dtype, shaped like out,
    and dS_final ~ N(0, ds_std^2) fp32, shaped like S_final."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    B, T, H, dk = inp["k"].shape
    dv = inp["v"].shape[-1]
    d_out = torch.randn(B, T, H, dv, generator=g).to(inp["v"].dtype)
    dS_final = ds_std * torch.randn(inp["N"], H, dv, dk, generator=g)
    return {"d_out": d_out, "dS_final": dS_final}
