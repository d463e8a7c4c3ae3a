"""Seeded synthetic inputs for the SwiAttn hot path (shared by tests and bench).

This module only draws random numbers; it holds none of the method's
arithmetic.  Everything is drawn on the CPU with ``torch.Generator`` so the
oracle and the GPU see bit-identical values (bf16 values widen exactly to
float64).  The recipes follow the workloads the SwiAttn report describes:
W = 1024 (section 2, training setup), an average routed (full-attention)
fraction of about 0.13 and about 0.05 in the easy case (section 3), 32K
context (sections 3 and 6).  No dataset or trained weight is involved.
"""
from __future__ import annotations

import math

import torch

# Phi^-1(0.87): with logit = h.w + b, h ~ N(0, I), the logit is
# N(b, ||w||^2), so b = -1.1264 ||w|| routes about 13 % of tokens.
Z_087 = 1.1263911290388013


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn(shape, dtype, gen: torch.Generator, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def bernoulli_gates(shape, frac: float, gen: torch.Generator) -> torch.Tensor:
    """Independent per-token gates, P(gate = 1) = frac; uint8."""
    return (torch.rand(*shape, generator=gen) < frac).to(torch.uint8)


def run_gates(N: int, frac: float, gen: torch.Generator, mean_run: float = 64.0,
              tol: float = None) -> torch.Tensor:
    """Two-state run process: routed runs ~ Geometric(mean mean_run), window runs
    ~ Geometric(mean mean_run*(1-frac)/frac), first state ~ Bernoulli(frac).
    With tol, whole sequences are redrawn until the realised routed fraction is
    within tol of frac (the same generator continues, so it stays seeded).
    Returns uint8 [N]."""
    while True:
        out = _run_gates_once(N, frac, gen, mean_run)
        if tol is None or abs(float(out.float().mean()) - frac) <= tol:
            return out


def _run_gates_once(N: int, frac: float, gen: torch.Generator, mean_run: float) -> torch.Tensor:
    out = torch.zeros(N, dtype=torch.uint8)
    state = 1 if float(torch.rand(1, generator=gen)) < frac else 0
    means = {1: mean_run, 0: mean_run * (1.0 - frac) / frac}
    pos = 0
    while pos < N:
        p = 1.0 / means[state]
        u = float(torch.rand(1, generator=gen))
        # Geometric on {1, 2, ...} with success probability p, by inversion.
        length = 1 + int(math.floor(math.log1p(-u) / math.log1p(-p))) if p < 1 else 1
        if state:
            out[pos:pos + length] = 1
        pos += length
        state ^= 1
    return out


def redraw_rows(h: torch.Tensor, rows, gen: torch.Generator) -> None:
    """Redraw the listed rows of a hidden-state matrix in place (used to keep
    router logits away from the gate threshold)."""
    rows = torch.as_tensor(rows, dtype=torch.long)
    if rows.numel():
        h[rows] = randn((rows.numel(), h.shape[1]), h.dtype, gen)


def attention_qkv(B, N, Hq, Hkv, d, dtype, gen):
    q = randn((B, N, Hq, d), dtype, gen)
    k = randn((B, N, Hkv, d), dtype, gen)
    v = randn((B, N, Hkv, d), dtype, gen)
    return q, k, v


def tiny_fp32(seed: int = 0) -> dict:
    """B=1, H=2, d=64, N=256, W=32, fp32; gates Bernoulli(0.13) per token."""
    g = _gen(seed)
    B, N, H, d, W = 1, 256, 2, 64, 32
    q, k, v = attention_qkv(B, N, H, H, d, torch.float32, g)
    gate = bernoulli_gates((B, N), 0.13, g)
    return dict(q=q, k=k, v=v, gate=gate, W=W, B=B, N=N, Hq=H, Hkv=H, d=d)


def router_inputs(T: int, D: int, dtype, seed: int, frac: float = 0.13) -> dict:
    """Hidden states h ~ N(0,1) [T,D], w ~ N(0,1/D), bias so ~frac route full."""
    g = _gen(seed)
    h = randn((T, D), dtype, g)
    w = randn((D,), dtype, g, std=1.0 / math.sqrt(D))
    wn = float(torch.linalg.vector_norm(w.to(torch.float64)))
    z = Z_087 if abs(frac - 0.13) < 1e-12 else _probit(1.0 - frac)
    return dict(h=h, w=w, bias=-z * wn, gen=g)


def _probit(p: float) -> float:
    from statistics import NormalDist
    return NormalDist().inv_cdf(p)


def prefill_4k(seed: int = 0) -> dict:
    """Single-layer prefill: B=1, H=16, d=128 (d_model 2048), N=4096, W=1024, bf16.
    Gates come from the router (caller runs it)."""
    B, N, H, d, W = 1, 4096, 16, 128, 1024
    r = router_inputs(B * N, H * d, torch.bfloat16, seed)
    q, k, v = attention_qkv(B, N, H, H, d, torch.bfloat16, r["gen"])
    return dict(h=r["h"], w=r["w"], bias=r["bias"], gen=r["gen"], q=q, k=k, v=v, W=W, B=B,
                N=N, Hq=H, Hkv=H, d=d)


def prefill_32k(frac: float = 0.13, seed: int = 0, N: int = 32768) -> dict:
    """Long-context prefill: B=1, H=16, d=128, N=32768, W=1024, bf16; gates in
    runs (mean routed run 64) at routed fraction frac (0.13 'standard',
    0.05 'easy'), realised fraction within 0.005 of frac."""
    g = _gen(seed)
    B, H, d, W = 1, 16, 128, 1024
    q, k, v = attention_qkv(B, N, H, H, d, torch.bfloat16, g)
    gate = run_gates(N, frac, g, tol=0.005).reshape(1, N)
    return dict(q=q, k=k, v=v, gate=gate, W=W, B=B, N=N, Hq=H, Hkv=H, d=d, frac=frac)


def decode_16x32k(seed: int = 0, B: int = 16, L: int = 32768, H: int = 16, d: int = 128,
                  W: int = 1024, frac: float = 0.13) -> dict:
    """Decode: B sequences with L cached tokens each (the newest token included),
    H heads, one query per sequence, per-sequence gate Bernoulli(frac), bf16."""
    g = _gen(seed)
    k = randn((B, L, H, d), torch.bfloat16, g)
    v = randn((B, L, H, d), torch.bfloat16, g)
    q = randn((B, H, d), torch.bfloat16, g)
    gate = bernoulli_gates((B,), frac, g)
    seq_lens = torch.full((B,), L, dtype=torch.int32)
    return dict(q=q, k_cache=k, v_cache=v, gate=gate, seq_lens=seq_lens, W=W, B=B, Lmax=L,
                Hq=H, Hkv=H, d=d)


def logits_with_margin(shape, gen, margin: float = 1e-3) -> torch.Tensor:
    """Router logits N(0,1) redrawn until every |logit| >= margin; fp32."""
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    while True:
        bad = x.abs() < margin
        if not bool(bad.any()):
            return x
        x[bad] = torch.randn(int(bad.sum()), generator=gen, dtype=torch.float32)


def dual_8k(seed: int = 0, B: int = 2, N: int = 8192) -> dict:
    """Dual-branch training forward: B=2, Hq=16, Hkv=4, d=128, N=8192, W=1024, bf16;
    logits N(0,1) with |logit| >= 1e-3, NLL ~ Gamma(2,1)."""
    g = _gen(seed)
    Hq, Hkv, d, W = 16, 4, 128, 1024
    q, k, v = attention_qkv(B, N, Hq, Hkv, d, torch.bfloat16, g)
    logits = logits_with_margin((B, N), g)
    # Gamma(2,1) is the sum of two Exp(1) draws.
    u = torch.rand(2, B, N, generator=g, dtype=torch.float64)
    nll = (-torch.log1p(-u)).sum(0).to(torch.float32)
    return dict(q=q, k=k, v=v, logits=logits, nll=nll, W=W, B=B, N=N, Hq=Hq, Hkv=Hkv, d=d,
                gamma_base=1e-3, eps=0.1, alpha=100.0)


def output_grad(shape, dtype, seed: int) -> torch.Tensor:
    """Upstream gradient of an attention output (the training backward's input):
    iid N(0,1) of the given shape and dtype, from its own seed."""
    return randn(shape, dtype, _gen(seed))
