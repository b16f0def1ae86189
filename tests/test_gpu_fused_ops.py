"""GPU parity of the fused prologue / epilogue around the recurrence:
kda_conv_prologue, kda_gated_rmsnorm and kda_decode_fused against the oracle
(oracle/fused_ops.py), plus the bit-exact contracts: the conv state holds exact
copies of raw inputs, two prologue calls continue one another exactly, and the
fused decode equals prologue + decode step + norm bit for bit."""
import numpy as np
import pytest
import torch

import kda_inputs as gen
from kda_testutil import assert_close, canary_fill, f64
from oracle import fused_ops as fo

pytestmark = pytest.mark.gpu
DEV = "cuda"
KD = VD = 128
DTYPES = pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kda_state_gb300 import _build
    _build.build()


def kda():
    import kda_state_gb300
    return kda_state_gb300


def _split(qkv):
    """Raw q, k, v views of a fused projection buffer [T, 3, H, K]."""
    return qkv[:, 0], qkv[:, 1], qkv[:, 2]


def _store(dtype):
    """The oracle stores intermediates as the unfused path does: in the dtype."""
    return fo.round_bf16 if dtype == torch.bfloat16 else fo.identity


def _ids(x):
    return torch.tensor(x, dtype=torch.int32, device=DEV)


@DTYPES
def test_conv_prologue_varlen(dtype):
    lengths = [1, 2, 3, 5, 64, 65, 130, 0]
    H, N, S = 3, 8, 12
    g = gen.make_gen(81)
    cu = gen.cu_seqlens(lengths)
    T = int(cu[-1])
    x = gen.raw_projections(T, H, dtype, g)
    wts = gen.fused_weights(H, dtype, g)
    cs = gen.checkpoint((S, 3, 3, H, KD), g, std=1.0).to(dtype).to(DEV)
    before = cs.clone()
    init = [-1, 1, 2, -1, 4, 5, 6, 7]
    out = [8, 1, 9, 10, -1, 5, 11, 0]      # in place for 1 and 5; 0 takes sequence 7's (empty) state
    qkv = x["qkv"].to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, k, v, beta = kda().kda_conv_prologue(*_split(qkv), x["b"].to(DEV), wts["conv_w"].to(DEV), cs,
                                            _ids(init), _ids(out), cu.to(DEV), cu, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rq, rk, rv, rb, rcs = fo.conv_prologue(*(f64(t) for t in _split(x["qkv"])), f64(x["b"]),
                                           f64(wts["conv_w"]), f64(before), cu.numpy(), init, out,
                                           store=_store(dtype))
    assert_close(q, rq, dtype, "q")
    assert_close(k, rk, dtype, "k")
    assert_close(v, rv, dtype, "v")
    assert_close(beta, rb, dtype, "beta")
    # the new conv states are copies of raw inputs (or of old state entries): exact
    assert np.array_equal(f64(cs), rcs), "conv state differs from the raw inputs it should hold"


@DTYPES
def test_conv_prologue_split_calls(dtype):
    """A sequence run as two calls, the second resuming from the conv state the
    first wrote in place, gives the one-call outputs and state bit for bit."""
    H, S, T = 2, 2, 150
    g = gen.make_gen(82, DEV)
    x = gen.raw_projections(T, H, dtype, g, device=DEV)
    wts = gen.fused_weights(H, dtype, g, device=DEV)
    cs0 = gen.checkpoint((S, 3, 3, H, KD), g, device=DEV, std=1.0).to(dtype)
    slot = _ids([0])
    cs_a = cs0.clone()
    whole = kda().kda_conv_prologue(*_split(x["qkv"]), x["b"], wts["conv_w"], cs_a, slot, slot,
                                    gen.cu_seqlens([T]).to(DEV), gen.cu_seqlens([T]))
    for cut in (1, 2, 64, 97):
        cs_b = cs0.clone()
        parts = []
        for lo, hi in ((0, cut), (cut, T)):
            cu = gen.cu_seqlens([hi - lo])
            parts.append(kda().kda_conv_prologue(*_split(x["qkv"][lo:hi]), x["b"][lo:hi],
                                                 wts["conv_w"], cs_b, slot, slot, cu.to(DEV), cu))
        torch.cuda.synchronize()
        for i in range(4):
            assert torch.equal(torch.cat([parts[0][i], parts[1][i]]), whole[i]), (cut, i)
        assert torch.equal(cs_b, cs_a)


@DTYPES
def test_gated_rmsnorm_strided(dtype):
    """o read at its own strides (a [T, H, 128] view inside a wider buffer)."""
    T, H = 37, 5
    g = gen.make_gen(83)
    big = torch.randn(T, H + 2, 2 * VD, generator=g).to(dtype).to(DEV)
    o = big[:, 1:H + 1, 64:64 + VD]
    gate = torch.randn(T, H, VD, generator=g).to(dtype).to(DEV)
    w = (1 + 0.1 * torch.randn(VD, generator=g)).to(dtype).to(DEV)
    out = kda().kda_gated_rmsnorm(o, gate, w)
    torch.cuda.synchronize()
    assert_close(out, fo.gated_rmsnorm(f64(o), f64(gate), f64(w)), dtype, "gated rmsnorm")


@DTYPES
def test_decode_fused_bit_exact_unfused(dtype):
    B, H, S = 6, 3, 10
    g = gen.make_gen(84)
    x = gen.raw_projections(1, H, dtype, g, lead=(B,))
    x = {n: t[:, 0] for n, t in x.items()}          # one token per request
    wts = gen.fused_weights(H, dtype, g)
    cs0 = gen.checkpoint((S, 3, 3, H, KD), g, std=1.0).to(dtype).to(DEV)
    pool0 = gen.checkpoint((S, H, KD, VD), g).to(DEV)
    ids = gen.slot_permutation(S, g)[:B]
    idd = ids.to(DEV)
    xd = {n: t.to(DEV) for n, t in x.items()}
    cw, wn = wts["conv_w"].to(DEV), wts["w_norm"].to(DEV)
    scale = 128 ** -0.5
    # fused
    cs_f, pool_f = cs0.clone(), pool0.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out_f = kda().kda_decode_fused(*_split(xd["qkv"]), xd["gk"], xd["b"], cw, cs_f, xd["gate"], wn,
                                   idd, pool_f, scale=scale, dev_err=err)
    # unfused: prologue (one-token sequences, conv state in the requests' slots), decode, norm
    cs_u, pool_u = cs0.clone(), pool0.clone()
    cu = torch.arange(B + 1, dtype=torch.int32)
    q, k, v, beta = kda().kda_conv_prologue(*_split(xd["qkv"]), xd["b"], cw, cs_u, idd, idd,
                                            cu.to(DEV), cu)
    o = kda().kda_decode_step(q, k, v, xd["gk"], beta, idd, pool_u, scale=scale)
    out_u = kda().kda_gated_rmsnorm(o, xd["gate"], wn)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out_f, out_u), "fused output differs from the unfused path"
    assert torch.equal(pool_f, pool_u), "fused KDA state differs from the unfused path"
    assert torch.equal(cs_f, cs_u), "fused conv state differs from the unfused path"
    ref_out, ref_pool, ref_cs = fo.decode_fused(*(f64(t) for t in _split(x["qkv"])), f64(x["gk"]),
                                                f64(x["b"]), f64(wts["conv_w"]), f64(cs0), f64(x["gate"]),
                                                f64(wts["w_norm"]), ids.numpy(), f64(pool0), scale=scale,
                                                store=_store(dtype))
    assert_close(out_f, ref_out, dtype, "fused decode out")
    assert_close(pool_f[idd.long()], ref_pool[ids.long().numpy()], dtype, "fused decode state")
    assert np.array_equal(f64(cs_f), ref_cs)


def test_decode_fused_bad_slot():
    B, H, S = 2, 2, 4
    g = gen.make_gen(85)
    x = {n: t[:, 0].to(DEV) for n, t in gen.raw_projections(1, H, torch.bfloat16, g, lead=(B,)).items()}
    wts = {n: t.to(DEV) for n, t in gen.fused_weights(H, torch.bfloat16, g).items()}
    cs = canary_fill(torch.empty(S, 3, 3, H, KD, dtype=torch.float32, device=DEV)).to(torch.bfloat16)
    pool = gen.checkpoint((S, H, KD, VD), g).to(DEV)
    cs_before, pool_before = cs.clone(), pool.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda().kda_decode_fused(*_split(x["qkv"]), x["gk"], x["b"], wts["conv_w"], cs, x["gate"],
                           wts["w_norm"], _ids([1, S + 2]), pool, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kda().KDA_DEVERR_SLOT_RANGE
    keep = torch.tensor([0, 2, 3], device=DEV)
    assert torch.equal(cs[keep], cs_before[keep]) and torch.equal(pool[keep], pool_before[keep])
    assert not torch.equal(pool[1], pool_before[1])
