"""The operand precisions chosen for the chunked prefill's tensor-core products,
checked as a model on the CPU.

The chunk algebra of the tensor-core prefill (Gram matrices, unit-lower
triangular inverse, the state chain) is evaluated in fp64 with each group of
MMA operands rounded the way the kernel stores them, and compared with the
oracle's sequential recurrence on the workload's input recipe:

* all operands in bf16 misses the 2e-2 x RMS bar on o;
* the kernel's mix (the Gram product on TF32; [K~; Q~] S0, V' = V - K~ S0,
  [T Diag(b); Aqk] V' and U, K_end^T U on fp16 operands) stays well inside it.

This is a model of the design choice, not a test of the kernel; the GPU parity
tests compare the kernel itself with the oracle.
"""
import numpy as np
import pytest
import torch

import kda_inputs as gen
import oracle
from kda_testutil import TOL, rel_err

C = 64        # chunk length of the tensor-core prefill
REF_ROW = 31  # the Gram factors are split around this row of the chunk


def bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).float().to(torch.bfloat16).double().numpy()


def fp16(x):
    return np.ascontiguousarray(x).astype(np.float16).astype(np.float64)


def tf32(x):
    """fp32 with the low 13 mantissa bits dropped (10 explicit bits kept): how the
    5th-generation MMA reads fp32 operand tiles under kind::tf32."""
    a = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFFE000)
    return a.view(np.float32).astype(np.float64)


def chunk_model(q, k, v, gk, beta, S0, gram, chain):
    """One unit through the chunked form as the kernel computes it; gram rounds
    the operands of the Gram products, chain those of every product with the
    state or with U (and the stored V' = V - K~ S0)."""
    T = q.shape[0]
    S = S0.copy()
    o = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        L = min(C, T - c0)
        qc, kc, vc, bc = q[c0:c0 + L], k[c0:c0 + L], v[c0:c0 + L], beta[c0:c0 + L]
        G = np.cumsum(gk[c0:c0 + L], 0)
        Gref, GL = G[min(REF_ROW, L - 1)], G[-1]
        ef, eb = np.exp(G - Gref), np.exp(Gref - G)          # exp(G_r - G_ref), exp(G_ref - G_r)
        A = np.tril(gram(kc * ef) @ gram(kc * eb).T, -1) * bc[:, None]
        Aqk = np.tril(gram(qc * ef) @ gram(kc * eb).T)
        TB = np.linalg.inv(np.eye(L) + A) * bc[None, :]        # T Diag(beta)
        Sc = chain(S)
        Pk = chain(kc * np.exp(G)) @ Sc                        # K~ S0
        Pq = chain(qc * np.exp(G)) @ Sc                        # Q~ S0
        Vp = chain(vc - Pk)                                    # V' (V enters as given)
        U = chain(TB) @ Vp                                     # T Diag(b) (V - K~ S0)
        Uc = chain(U)
        o[c0:c0 + L] = Pq + chain(Aqk) @ Uc
        S = np.exp(GL)[:, None] * S + chain((kc * np.exp(GL - G)).T) @ Uc
    return o, S


@pytest.fixture(scope="module")
def cases():
    out = []
    for seed, T, ckpt in ((11, 523, False), (12, 700, True), (13, 300, False)):
        g = gen.make_gen(seed)
        x = gen.token_inputs(T, 1, torch.bfloat16, g)
        f = lambda t: t[:, 0].double().numpy()
        q, k, v, gk, beta = (f(x[n]) for n in ("q", "k", "v", "gk", "beta"))
        S0 = gen.checkpoint((128, 128), g).double().numpy() if ckpt else np.zeros((128, 128))
        out.append((q, k, v, gk, beta, S0, oracle.unit(q, k, v, gk, beta, S0)))
    return out


def worst(cases, **rnd):
    eo = es = 0.0
    for q, k, v, gk, beta, S0, (o_ref, S_ref) in cases:
        o, S = chunk_model(q, k, v, gk, beta, S0, **rnd)
        o16 = torch.from_numpy(o).float().to(torch.bfloat16)   # o is stored in bf16
        eo = max(eo, rel_err(o16, o_ref, torch.bfloat16))
        es = max(es, rel_err(torch.from_numpy(S), S_ref))
    return eo, es


def test_exact_operands_reproduce_the_oracle(cases):
    ident = lambda x: x
    eo, es = worst(cases, gram=ident, chain=ident)
    assert eo == 0.0 and es < 1e-12        # o: within its own bf16 rounding


def test_all_bf16_operands_miss_the_bar(cases):
    eo, _ = worst(cases, gram=bf16, chain=bf16)
    assert eo > TOL[torch.bfloat16]


def test_kernel_operand_mix_is_well_inside_the_bar(cases):
    eo, es = worst(cases, gram=tf32, chain=fp16)
    assert eo < 0.5 * TOL[torch.bfloat16] and es < 0.5 * TOL[torch.bfloat16]
