"""Seeded synthetic inputs for the KDA forward.

This module only draws random numbers; it holds none of the method's
arithmetic.  Both the CUDA path's tests/benchmark and the fp64 oracle consume
the tensors it returns, so the two sides see identical bits.

Distributions follow the workloads of the KDA forward kernels (kernel-fun
``kda/_kernels/fwd_state.py`` host wrapper: bf16 q/k/v, fp32 per-dimension
log-decay g, fp32 initial/final state) and the standard KDA setup:

* q, k: N(0,1) in fp32, L2-normalised over K per token, then rounded to bf16;
* v: N(0,1) rounded to bf16;
* beta: sigmoid(N(0,1)) rounded to bf16, shape [B,T,H] (already activated);
* g: logsigmoid(N(mu,1)) in fp32, shape [B,T,H,K] (natural-log decay, < 0);
* h0: 0.1 * N(0,1) fp32 [N,H,K,V], or None (zero initial state);
* scale = K ** -0.5.

Generation runs on the CPU with ``torch.Generator`` (seed per workload) so the
bits do not depend on the device.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch
import torch.nn.functional as F


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    mu: float = 3.0
    h0: bool = True
    varlen: int = 0          # number of packed sequences (0 = fixed length)
    max_len: int = 8192      # varlen lengths are uniform in [1, max_len]
    seed: int = 20261202
    note: str = field(default="", compare=False)


# The five workloads of the KDA forward: a tiny two-chunk case the oracle
# finishes instantly, a mid-size case, the headline shape, a packed varlen
# batch and a single long sequence (few scan CTAs, long serial chain).
WORKLOADS = {
    "tiny": Workload("tiny", B=1, T=128, H=1, K=64, V=64, h0=False, seed=20261202),
    "mid": Workload("mid", B=1, T=4096, H=16, K=128, V=128, seed=20261203),
    "headline": Workload("headline", B=4, T=8192, H=32, K=128, V=128, seed=20261204),
    "varlen": Workload("varlen", B=1, T=0, H=32, K=128, V=128, varlen=16, seed=20261205),
    "long": Workload("long", B=1, T=65536, H=32, K=128, V=128, mu=5.0, h0=False,
                     seed=20261206),
    # a quarter of the headline's token-heads in two sequences (so the forward
    # runs unstaged, as at the headline): the size profiler captures of the
    # intra kernel run on (its inputs, ~0.4 GB, still exceed L2)
    "quarter": Workload("quarter", B=2, T=4096, H=32, K=128, V=128, seed=20261207),
    # the same token-heads as "quarter" spread over 128 heads: the scan kernel
    # runs the headline's grid (128 CTAs, 128-wide V tiles) on 32 chunks each
    "wide": Workload("wide", B=1, T=2048, H=128, K=128, V=128, seed=20261208),
    # the long single sequence at head dim 64
    "long_k64": Workload("long_k64", B=1, T=65536, H=32, K=64, V=64, mu=5.0, h0=False,
                         seed=20261209),
}


def varlen_lengths(n: int, max_len: int, seed: int) -> list[int]:
    """n sequence lengths uniform in [1, max_len] (seeded)."""
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(1, max_len + 1, (n,), generator=gen).tolist()


def cu_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def make_inputs(w: Workload, lengths=None, h0=None, dtype_g=torch.float32):
    """Draw the inputs of workload ``w`` on the CPU.

    Returns a dict with q, k, v (bf16 [B,T,H,K|V]), g (fp32 [B,T,H,K]), beta
    (bf16 [B,T,H]), h0 (fp32 [N,H,K,V] or None), cu_seqlens (int32 [N+1] or
    None), scale (float), N, and the shape fields.
    """
    gen = torch.Generator().manual_seed(w.seed)
    if w.varlen:
        if lengths is None:
            lengths = varlen_lengths(w.varlen, w.max_len, w.seed + 7919)
        cu = cu_from_lengths(lengths)
        B, T, N = 1, int(cu[-1]), len(lengths)
    elif lengths is not None:
        cu = cu_from_lengths(lengths)
        B, T, N = 1, int(cu[-1]), len(lengths)
    else:
        cu = None
        B, T, N = w.B, w.T, w.B
    H, K, V = w.H, w.K, w.V

    def unit_rows(shape):
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)
        return x.to(torch.bfloat16)

    q = unit_rows((B, T, H, K))
    k = unit_rows((B, T, H, K))
    v = torch.randn((B, T, H, V), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn((B, T, H), generator=gen)).to(torch.bfloat16)
    g = F.logsigmoid(torch.randn((B, T, H, K), generator=gen) + w.mu).to(dtype_g)
    if h0 is None and w.h0:
        h0 = 0.1 * torch.randn((N, H, K, V), generator=gen, dtype=torch.float32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, cu_seqlens=cu, scale=K ** -0.5,
                B=B, T=T, H=H, K=K, V=V, N=N)


def make_bwd_inputs(x: dict, seed: int = 0, dht: bool = True):
    """Upstream gradients for the reverse state scan of the inputs ``x`` (from
    :func:`make_inputs`), drawn on the CPU: do and dv_in bf16 [B,T,H,V] with
    N(0, 1) entries (dv_in stands for the chunk-local Aqk^T do term, of the same
    magnitude), dht fp32 [N,H,K,V] N(0, 0.1^2) or None."""
    gen = torch.Generator().manual_seed(1_000_003 + 31 * seed + int(x["T"]))
    B, T, H, K, V, N = x["B"], x["T"], x["H"], x["K"], x["V"], x["N"]
    do = torch.randn((B, T, H, V), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    dv_in = torch.randn((B, T, H, V), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    dh_t = 0.1 * torch.randn((N, H, K, V), generator=gen, dtype=torch.float32) if dht else None
    return dict(do=do, dv_in=dv_in, dht=dh_t)


def make_variant_inputs(w: Workload, io_dtype=torch.bfloat16, qk_heads=None, beta_logits=False,
                        state_dtype=torch.float32, lengths=None):
    """Inputs of workload ``w`` for the forward's interface variants, drawn on
    the CPU: q, k with ``qk_heads`` heads (default: w.H) and v, g, beta, h0 with
    w.H heads; q, k, v, beta in ``io_dtype`` (bf16 or fp16); beta either in
    (0, 1) (sigmoid of N(0,1)) or, with ``beta_logits``, the N(0,1) logits
    themselves; h0 (when the workload has one) in ``state_dtype``.  Same
    distributions as :func:`make_inputs` otherwise."""
    gen = torch.Generator().manual_seed(w.seed + 104729)
    if w.varlen or lengths is not None:
        if lengths is None:
            lengths = varlen_lengths(w.varlen, w.max_len, w.seed + 7919)
        cu = cu_from_lengths(lengths)
        B, T, N = 1, int(cu[-1]), len(lengths)
    else:
        cu = None
        B, T, N = w.B, w.T, w.B
    H, K, V = w.H, w.K, w.V
    Hqk = H if qk_heads is None else qk_heads

    def unit_rows(shape):
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        return (x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)).to(io_dtype)

    q = unit_rows((B, T, Hqk, K))
    k = unit_rows((B, T, Hqk, K))
    v = torch.randn((B, T, H, V), generator=gen, dtype=torch.float32).to(io_dtype)
    logits = torch.randn((B, T, H), generator=gen)
    beta = (logits if beta_logits else torch.sigmoid(logits)).to(io_dtype)
    g = F.logsigmoid(torch.randn((B, T, H, K), generator=gen) + w.mu)
    h0 = (0.1 * torch.randn((N, H, K, V), generator=gen, dtype=torch.float32)).to(state_dtype) if w.h0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, cu_seqlens=cu, scale=K ** -0.5,
                B=B, T=T, H=H, K=K, V=V, N=N, qk_heads=Hqk, beta_logits=beta_logits)


def make_inputs_on(w: Workload, device, with_bwd: bool = False):
    """Inputs of the workload ``w`` drawn directly on ``device`` with a
    generator seeded there (the distributions of :func:`make_inputs`; a packed
    workload takes the seeded lengths of :func:`make_inputs`).

    For problems whose tensors are too large to draw on the CPU in a test's
    time: the bits differ from :func:`make_inputs` (another generator), so a
    caller hands the oracle the slices it checks, copied back from the
    device.  ``with_bwd`` adds do, dv_in (N(0,1) bf16) and dht (N(0, 0.1^2)
    fp32), as :func:`make_bwd_inputs` draws them.
    """
    gen = torch.Generator(device=device).manual_seed(w.seed)
    H, K, V = w.H, w.K, w.V
    cu = None
    if w.varlen:  # the seeded lengths of make_inputs, packed as one row of sequences
        cu = cu_from_lengths(varlen_lengths(w.varlen, w.max_len, w.seed + 7919))
        B, T, N = 1, int(cu[-1]), w.varlen
    else:
        B, T, N = w.B, w.T, w.B

    def randn(shape):
        return torch.randn(shape, generator=gen, dtype=torch.float32, device=device)

    def unit_rows(shape):
        x = randn(shape)
        x /= x.norm(dim=-1, keepdim=True).clamp_min(1e-12)
        return x.to(torch.bfloat16)

    q = unit_rows((B, T, H, K))
    k = unit_rows((B, T, H, K))
    v = randn((B, T, H, V)).to(torch.bfloat16)
    beta = torch.sigmoid(randn((B, T, H))).to(torch.bfloat16)
    g = randn((B, T, H, K))
    g += w.mu
    g = F.logsigmoid(g)
    h0 = 0.1 * randn((N, H, K, V)) if w.h0 else None
    out = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, cu_seqlens=None if cu is None else cu.to(device),
               scale=K ** -0.5, B=B, T=T, H=H, K=K, V=V, N=N)
    if with_bwd:
        out.update(do=randn((B, T, H, V)).to(torch.bfloat16), dv_in=randn((B, T, H, V)).to(torch.bfloat16),
                   dht=0.1 * randn((N, H, K, V)))
    return out
