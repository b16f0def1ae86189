"""Seeded synthetic inputs for the KDA state path (shared by tests, smoke and bench).

This module holds none of the method's arithmetic: it only draws the
per-token inputs and checkpoints with the distributions of the workloads and
casts them.  Both the CUDA library and the oracle consume the identical cast
tensors it returns.

Input recipe (all drawn in fp32 from one seeded ``torch.Generator``, then cast):

* q, k ~ N(0, 1), each (token, head) vector L2-normalised over K;
* v ~ N(0, 1);
* gk = -softplus(N(0, 1))  (natural-log per-key-channel decay, <= 0);
* beta = sigmoid(N(0, 1));
* checkpoints ~ 0.02 * N(0, 1), fp32;
* draw order: q, k, v, gk, beta (then checkpoints), so a seed fixes everything.

Inputs of the fused prologue / epilogue (raw projection outputs and random-init
weights; the pages give no trained values):

* one fused q/k/v projection output [T, 3, H, K] ~ N(0, 1), read through views;
* pre-sigmoid beta b ~ N(0, 1), output gate ~ N(0, 1), gk as above;
* conv taps [3, H, K, 4] ~ 0.5 N(0, 1), RMSNorm weight ~ 1 + 0.1 N(0, 1);
* conv states ~ N(0, 1) in the dtype.

Workload shapes (K = V = 128):

* tiny:    1 sequence, T = 64, H = 1, fp32, zero initial state, seed 0;
* varlen:  8 sequences, lengths uniform in [64, 2048], H = 64, bf16, seed 1;
* long:    4 sequences x 24576 tokens, H = 96, bf16, checkpointed, pieces of 4096, seed 2;
* decode:  384 requests x 1 token, H = 64, bf16, pool of 512 slots, 69 layers, 10% CoW, seed 3;
* verify:  64 requests x 8 draft tokens, 69 layers, H = 64, bf16, pools of 128 slots, seed 4.
"""
from __future__ import annotations

import torch

K_DIM = 128
V_DIM = 128


def make_gen(seed: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, gen, device):
    return torch.randn(*shape, generator=gen, dtype=torch.float32, device=device)


def token_inputs(T: int, H: int, dtype=torch.bfloat16, gen=None, device: str = "cpu",
                 K: int = K_DIM, V: int = V_DIM, lead=()):
    """q, k, gk of shape lead + [T, H, K]; v lead + [T, H, V]; beta lead + [T, H]."""
    gen = gen if gen is not None else make_gen(0, device)
    shp = tuple(lead) + (T, H)
    q = _normal(shp + (K,), gen, device)
    q = q / q.norm(dim=-1, keepdim=True)
    k = _normal(shp + (K,), gen, device)
    k = k / k.norm(dim=-1, keepdim=True)
    v = _normal(shp + (V,), gen, device)
    gk = -torch.nn.functional.softplus(_normal(shp + (K,), gen, device))
    beta = torch.sigmoid(_normal(shp, gen, device))
    return {n: t.to(dtype).contiguous() for n, t in
            (("q", q), ("k", k), ("v", v), ("gk", gk), ("beta", beta))}


def raw_projections(T: int, H: int, dtype=torch.bfloat16, gen=None, device: str = "cpu",
                    K: int = K_DIM, lead=()):
    """Inputs of the fused prologue / epilogue: one fused q/k/v projection
    output qkv lead + [T, 3, H, K] ~ N(0, 1) (its [..., 0|1|2, :, :] slices are
    the raw q, k, v), the pre-sigmoid beta b lead + [T, H] ~ N(0, 1), the output
    gate lead + [T, H, K] ~ N(0, 1), and gk = -softplus(N(0, 1)) lead + [T, H, K]."""
    gen = gen if gen is not None else make_gen(0, device)
    shp = tuple(lead) + (T,)
    qkv = _normal(shp + (3, H, K), gen, device)
    b = _normal(shp + (H,), gen, device)
    gate = _normal(shp + (H, K), gen, device)
    gk = -torch.nn.functional.softplus(_normal(shp + (H, K), gen, device))
    return {n: t.to(dtype).contiguous() for n, t in
            (("qkv", qkv), ("b", b), ("gate", gate), ("gk", gk))}


def fused_weights(H: int, dtype=torch.bfloat16, gen=None, device: str = "cpu", K: int = K_DIM,
                  width: int = 4):
    """Random-init weights of the prologue / epilogue: conv taps [3, H, K, width]
    ~ 0.5 N(0, 1) and the RMSNorm weight [K] ~ 1 + 0.1 N(0, 1)."""
    gen = gen if gen is not None else make_gen(0, device)
    conv_w = 0.5 * _normal((3, H, K, width), gen, device)
    w_norm = 1.0 + 0.1 * _normal((K,), gen, device)
    return {"conv_w": conv_w.to(dtype).contiguous(), "w_norm": w_norm.to(dtype).contiguous()}


def checkpoint(shape, gen, device: str = "cpu", std: float = 0.02) -> torch.Tensor:
    return (_normal(tuple(shape), gen, device) * std).contiguous()


def varlen_lengths(n: int, lo: int, hi: int, gen) -> list:
    """n lengths drawn uniformly from the integers lo..hi (inclusive)."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen, device=gen.device).cpu()]


def cu_seqlens(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def accept_lengths(B: int, G: int, p: float, gen) -> torch.Tensor:
    """1 + (run of i.i.d. accepts with probability p), capped at G: values in
    1..G with mean 1 + sum_{i=1}^{G-1} p^i (2.70 for G = 8, p = 0.64)."""
    u = torch.rand(B, G - 1, generator=gen, device=gen.device).cpu()
    acc = torch.ones(B, dtype=torch.int32)
    alive = torch.ones(B, dtype=torch.bool)
    for i in range(G - 1):
        alive &= u[:, i] < p
        acc += alive.to(torch.int32)
    return acc


def draft_lengths(B: int, G: int, gen) -> torch.Tensor:
    """Trimmed verify windows: a draft count per request, uniform on 1..G (the
    pages give no distribution of the planner's window lengths)."""
    return torch.randint(1, G + 1, (B,), generator=gen, device=gen.device).cpu().to(torch.int32)


def slot_permutation(num_slots: int, gen) -> torch.Tensor:
    return torch.randperm(num_slots, generator=gen, device=gen.device).cpu().to(torch.int32)


# Workload descriptions (sizes only; tensors are drawn by the callers above).
WORKLOADS = {
    "tiny": dict(N=1, T=64, H=1, dtype="fp32", seed=0),
    "varlen": dict(N=8, lo=64, hi=2048, H=64, dtype="bf16", seed=1),
    "long": dict(N=4, T=24576, H=96, piece=4096, dtype="bf16", seed=2),
    "decode": dict(B=384, H=64, slots=512, layers=69, cow_frac=0.10, dtype="bf16", seed=3),
    "verify": dict(B=64, G=8, H=64, slots=128, layers=69, ring=16, accept_p=0.64, dtype="bf16",
                   seed=4),
}


# ---------------------------------------------------------------------------
# Full workload batches (same recipe for the benchmark and the parity tests).
# Large tensors are drawn on `device` with a generator seeded seed + 1000.
# ---------------------------------------------------------------------------

def varlen_batch(device: str = "cpu", seed: int = 1, H: int = 64, N: int = 8, lo: int = 64,
                 hi: int = 2048, dtype=torch.bfloat16):
    g = make_gen(seed)
    lengths = varlen_lengths(N, lo, hi, g)
    cu = cu_seqlens(lengths)
    gd = make_gen(seed + 1000, device)
    x = token_inputs(int(cu[-1]), H, dtype, gd, device=device)
    ck = checkpoint((N, H, K_DIM, V_DIM), gd, device=device)
    return dict(lengths=lengths, cu=cu, T=int(cu[-1]), H=H, N=N, x=x, ck=ck)


def long_batch(device: str = "cpu", seed: int = 2, H: int = 96, N: int = 4, T: int = 24576,
               dtype=torch.bfloat16):
    gd = make_gen(seed + 1000, device)
    x = token_inputs(N * T, H, dtype, gd, device=device)
    ck = checkpoint((N, H, K_DIM, V_DIM), gd, device=device)
    return dict(N=N, T=T, H=H, x=x, ck=ck)
