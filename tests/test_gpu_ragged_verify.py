"""GPU parity of kda_verify_store_inputs_ragged: each request verifies its own
G_b <= G_max drafts, packed by cu_drafts.

Checked against the oracle's ragged verify; against the uniform verify (a
request's outputs are bit-identical to the uniform call's first G_b rows on
the same drafts); records of the verified steps exact, every other ring entry
and every output row of no request untouched; the fold of accept_len <= G_b
bit-identical to that many decode steps."""
import numpy as np
import pytest
import torch

import kda_inputs as gen
import oracle
from kda_testutil import assert_close, canary_fill, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
KD = VD = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kda_state_gb300 import _build
    _build.build()


def kda():
    import kda_state_gb300
    return kda_state_gb300


def _dev(x):
    return {n: t.to(DEV) for n, t in x.items()}


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("G_max", [8, 16, 24])
def test_ragged_verify_then_fold(dtype, G_max):
    g = gen.make_gen(51 + G_max)
    H, S = 2, 12
    Gb = [0, 1, 3, G_max, 5, 2, G_max - 1]
    B = len(Gb)
    R = kda().ring_len_for(G_max - 1)
    lead, tail = 1, 3                               # tokens that belong to no request
    cu = torch.tensor(np.concatenate([[lead], lead + np.cumsum(Gb)]), dtype=torch.int32)
    T = int(cu[-1]) + tail
    x = gen.token_inputs(T, H, dtype, g)
    xd = _dev(x)
    pool = gen.checkpoint((S, H, KD, VD), g).to(DEV)
    committed = pool.clone()
    ids = gen.slot_permutation(S, g)[:B]
    base = torch.randint(0, R, (B,), generator=g, dtype=torch.int32)
    ring = kda().make_ring(S, R, H, dtype, DEV)
    o = canary_fill(torch.empty(T, H, VD, dtype=torch.float32, device=DEV)).to(dtype)
    o_before = o.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    idd, based = ids.to(DEV), base.to(DEV)
    kda().kda_verify_store_inputs_ragged(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"],
                                         cu.to(DEV), G_max, idd, pool, ring, ring_base=based, o=o,
                                         dev_err=err)
    # the uniform call on the same drafts padded to G_max rows
    pad = {n: torch.zeros((B, G_max) + tuple(t.shape[1:]), dtype=t.dtype) for n, t in x.items()}
    for b in range(B):
        for n in pad:
            pad[n][b, :Gb[b]] = x[n][cu[b]:cu[b + 1]]
            pad[n][b, Gb[b]:] = x[n][:G_max - Gb[b]]      # arbitrary padding drafts
    padd = _dev(pad)
    ring_u = kda().make_ring(S, R, H, dtype, DEV)
    o_u = kda().kda_verify_store_inputs(padd["q"], padd["k"], padd["v"], padd["gk"], padd["beta"],
                                        idd, pool, ring_u, ring_base=based)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(pool, committed), "verify wrote the committed state"
    rows = torch.zeros(T, dtype=torch.bool)
    for b in range(B):
        rows[cu[b]:cu[b + 1]] = True
        assert torch.equal(o[cu[b]:cu[b + 1]], o_u[b, :Gb[b]]), "request %d differs from uniform" % b
    assert torch.equal(o[~rows.to(DEV)], o_before[~rows.to(DEV)]), "a row of no request was written"
    o_ref = oracle.verify_ragged(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["gk"]),
                                 f64(x["beta"]), cu.numpy(), f64(committed[ids.long().to(DEV)]))
    assert_close(o[rows.to(DEV)], o_ref[rows.numpy()], dtype, "ragged verify o")
    # records: the verified steps exact, every other entry of every slot untouched (zero)
    written = torch.zeros(S, R, dtype=torch.bool)
    for b in range(B):
        s = int(ids[b])
        ent = [(int(base[b]) + i) % R for i in range(Gb[b])]
        written[s, ent] = True
        sl = slice(int(cu[b]), int(cu[b + 1]))
        assert torch.equal(ring.k[s, ent].cpu(), x["k"][sl])
        assert torch.equal(ring.v[s, ent].cpu(), x["v"][sl])
        assert torch.equal(ring.beta[s, ent].cpu(), x["beta"][sl].float())
        np.testing.assert_allclose(f64(ring.decay[s, ent]), np.exp(f64(x["gk"][sl])), rtol=5e-7,
                                   atol=0)
    wd = written.to(DEV)
    for buf in (ring.k, ring.v, ring.decay, ring.beta):
        assert not buf[~wd].any(), "a ring entry past G_b was written"
    # fold accept_len <= G_b: bit-identical to that many decode steps
    accept = torch.tensor([min(a, gb) for a, gb in zip([0, 1, 2, G_max, 5, 1, 3], Gb)],
                          dtype=torch.int32)
    kda().kda_replay_fold([pool], [ring], idd, accept.to(DEV), max_accept=G_max, ring_base=based)
    ref = committed.clone()
    for i in range(G_max):
        sel = [b for b in range(B) if accept[b] > i]
        if not sel:
            continue
        tok = torch.tensor([int(cu[b]) + i for b in sel], device=DEV)
        kda().kda_decode_step(*(xd[n].index_select(0, tok).contiguous()
                                for n in ("q", "k", "v", "gk", "beta")),
                              idd[torch.tensor(sel, device=DEV)].contiguous(), ref)
    torch.cuda.synchronize()
    assert torch.equal(pool, ref), "fold after ragged verify is not bit-identical to decode"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_ragged_verify_bad_offsets(dtype):
    """A request whose offsets go backwards, one with more than G_max drafts,
    and one past total_tokens are skipped with KDA_DEVERR_SEQLENS; the others
    complete."""
    g = gen.make_gen(61)
    H, S, G_max = 2, 8, 8
    cu = torch.tensor([0, 3, 2, 12, 14, 40], dtype=torch.int32)   # b1 backwards, b2 10 > 8, b4 past T
    T = 16
    x = gen.token_inputs(T, H, dtype, g)
    xd = _dev(x)
    pool = gen.checkpoint((S, H, KD, VD), g).to(DEV)
    ring = kda().make_ring(S, 16, H, dtype, DEV)
    ids = torch.arange(5, dtype=torch.int32, device=DEV)
    o = torch.zeros(T, H, VD, dtype=dtype, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda().kda_verify_store_inputs_ragged(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"],
                                         cu.to(DEV), G_max, ids, pool, ring, o=o, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kda().KDA_DEVERR_SEQLENS
    for b, (lo, hi) in enumerate([(0, 3), (12, 14)]):
        S0 = f64(pool[[0, 3][b]])[None]
        sl = slice(lo, hi)
        ref = oracle.verify_ragged(f64(x["q"][sl]), f64(x["k"][sl]), f64(x["v"][sl]),
                                   f64(x["gk"][sl]), f64(x["beta"][sl]), [0, hi - lo], S0)
        assert_close(o[sl], ref, dtype, "request %d" % [0, 3][b])
    assert not o[3:12].any() and not o[14:].any()
    assert not ring.k[[1, 2, 4]].any()


def test_ragged_verify_all_empty():
    """Every request trims its window to zero drafts: nothing is read or
    written, no error is raised."""
    H, S = 2, 4
    g = gen.make_gen(62)
    pool = gen.checkpoint((S, H, KD, VD), g).to(DEV)
    before = pool.clone()
    ring = kda().make_ring(S, 16, H, torch.bfloat16, DEV)
    cu = torch.zeros(4, dtype=torch.int32, device=DEV)
    empty = torch.empty(0, H, KD, dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda().kda_verify_store_inputs_ragged(empty, empty, empty, empty,
                                         torch.empty(0, H, dtype=torch.bfloat16, device=DEV), cu, 8,
                                         torch.tensor([0, 1, 2], dtype=torch.int32, device=DEV),
                                         pool, ring, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(pool, before)
    assert not ring.k.any() and not ring.decay.any()
