"""The operand precisions chosen for the chunked prefill's tensor-core products,
checked as a model on the CPU.

The chunk algebra of the tensor-core prefill (32-token chunks; Gram matrices,
unit-lower-triangular inverse, the state chain, every product on TF32) is
evaluated in fp64 with each MMA operand presented the way the kernel presents
it to the tensor core, and compared with the oracle's sequential recurrence on
the workload's input recipe:

* all operands in bf16 misses the 2e-2 x RMS bar on o;
* the kernel's formats stay well inside it: Kb and Aqk rounded to TF32 to
  nearest by the CUDA cores that write them; K~, Q~, V' and T Diag(b) written
  unrounded and the state S and U read from TMEM, all truncated to TF32 by the
  tensor core;
* Kb is the one tile that needs the rounding: truncating it as well moves the
  state's error past half the bar.

This is a model of the design choice, not a test of the kernel; the GPU parity
tests compare the kernel itself with the oracle.
"""
import numpy as np
import pytest
import torch

import kda_inputs as gen
import oracle
from kda_testutil import TOL, rel_err

C = 32        # chunk length of the tensor-core prefill


def bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).float().to(torch.bfloat16).double().numpy()


def f32(x):
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def tf32_trunc(x):
    """fp32 with the low 13 mantissa bits dropped (10 explicit bits kept): how the
    5th-generation MMA reads an fp32 operand it is given unrounded (here the
    state and U, read from TMEM)."""
    a = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFFE000)
    return a.view(np.float32).astype(np.float64)


def tf32_rna(x):
    """fp32 rounded to TF32, to nearest with ties away from zero (cvt.rna.tf32.f32):
    how the kernel stores the operand tiles its CUDA cores write."""
    a = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    a = ((a + 0x1000) & 0xFFFFE000).astype(np.uint32)
    return a.view(np.float32).astype(np.float64)


def chunk_model(q, k, v, gk, beta, S0, kt, qt, kb, vp, tb, aqk, tmem, store=f32):
    """One unit through the chunked form as the kernel computes it.  kt, qt,
    kb, vp, tb, aqk give the format of each operand tile (K~, Q~, Kb, V',
    T Diag(b), Aqk), tmem that of the operands read from TMEM (the state and
    U), store that of the fp32 accumulators."""
    T = q.shape[0]
    S = S0.copy()
    o = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        L = min(C, T - c0)
        qc, kc, vc, bc = q[c0:c0 + L], k[c0:c0 + L], v[c0:c0 + L], beta[c0:c0 + L]
        G = np.cumsum(gk[c0:c0 + L], 0)                       # decay from the chunk start
        Kt, Qt, Kb = kt(kc * np.exp(G)), qt(qc * np.exp(G)), kb(kc * np.exp(-G))
        A = np.tril(store(Kt @ Kb.T), -1) * bc[:, None]
        Aqk = np.tril(store(Qt @ Kb.T))
        TB = np.linalg.inv(np.eye(L) + A) * bc[None, :]        # T Diag(beta)
        Sc = tmem(S)
        Vp = vp(store(vc - Kt @ Sc))                           # V' = V - K~ S
        U = store(tb(TB) @ Vp)
        o[c0:c0 + L] = Qt @ Sc + aqk(Aqk) @ tmem(U)
        S = store(np.exp(G[-1])[:, None] * store(S + Kb.T @ tmem(U)))
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
    eo, es = worst(cases, kt=ident, qt=ident, kb=ident, vp=ident, tb=ident, aqk=ident, tmem=ident,
                   store=ident)
    assert eo == 0.0 and es < 1e-12        # o: within its own bf16 rounding


def test_all_bf16_operands_miss_the_bar(cases):
    eo, _ = worst(cases, kt=bf16, qt=bf16, kb=bf16, vp=bf16, tb=bf16, aqk=bf16, tmem=bf16)
    assert eo > TOL[torch.bfloat16]


KERNEL = dict(kt=tf32_trunc, qt=tf32_trunc, kb=tf32_rna, vp=tf32_trunc, tb=tf32_trunc, aqk=tf32_rna,
              tmem=tf32_trunc)


def test_kernel_operand_formats_are_well_inside_the_bar(cases):
    eo, es = worst(cases, **KERNEL)
    assert eo < 0.5 * TOL[torch.bfloat16] and es < 0.5 * TOL[torch.bfloat16]


def test_kb_needs_rounding_to_nearest(cases):
    _, es = worst(cases, **{**KERNEL, "kb": tf32_trunc})
    assert es > 0.5 * TOL[torch.bfloat16]
