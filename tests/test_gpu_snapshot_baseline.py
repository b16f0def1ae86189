"""GPU parity of the snapshot-per-step verify baseline (kda_verify_snapshot +
kda_snapshot_commit), the design ReplaySSM replaces.

Snapshot i and output i are bit-identical to i + 1 decode steps; the
committed state is never written by verify; the commit of accept a is
bit-identical to the ReplaySSM fold of a on the same drafts; outputs and
snapshots match the oracle; slots and snapshot slots not named stay
untouched."""
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
@pytest.mark.parametrize("G", [1, 3, 8])
def test_snapshot_verify_commit(dtype, G):
    g = gen.make_gen(71 + G)
    B, H, L, S = 5, 2, 2, 12
    NS = B + 1                                   # snapshot slot NS-1 is never named
    pools = [gen.checkpoint((S, H, KD, VD), g).to(DEV) for _ in range(L)]
    committed = [p.clone() for p in pools]
    xs = [gen.token_inputs(G, H, dtype, g, lead=(B,)) for _ in range(L)]
    ids = gen.slot_permutation(S, g)[:B]
    snap_ids = gen.slot_permutation(NS - 1, g)
    snaps = [canary_fill(torch.empty(NS, G, H, KD, VD, device=DEV)) for _ in range(L)]
    snap_before = [s.clone() for s in snaps]
    idd, snd = ids.to(DEV), snap_ids.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = []
    for l in range(L):
        xd = _dev(xs[l])
        outs.append(kda().kda_verify_snapshot(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"],
                                              idd, pools[l], snaps[l], snd, dev_err=err))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for l in range(L):
        assert torch.equal(pools[l], committed[l]), "verify wrote the committed state"
        assert torch.equal(snaps[l][NS - 1], snap_before[l][NS - 1]), "an unnamed snapshot slot"
        # bit-exact against decode steps on a copy of the committed pool
        ref = committed[l].clone()
        xd = _dev(xs[l])
        for i in range(G):
            od = kda().kda_decode_step(*(xd[n][:, i].contiguous() for n in ("q", "k", "v", "gk", "beta")),
                                       idd, ref)
            torch.cuda.synchronize()
            assert torch.equal(outs[l][:, i], od), "output %d differs from decode" % i
            assert torch.equal(snaps[l][snap_ids.long().to(DEV), i], ref[idd.long()]), (
                "snapshot %d differs from the decode state" % i)
        # against the oracle: outputs, and the states after every step
        x = xs[l]
        S0 = f64(committed[l][idd.long()])
        o_ref = oracle.verify(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["gk"]), f64(x["beta"]), S0)
        assert_close(outs[l], o_ref, dtype, "snapshot verify o")
        flat = {n: f64(t).reshape((B * G,) + tuple(t.shape[2:])) for n, t in x.items()}
        _, _, ck, _ = oracle.prefill_checkpoints(flat["q"], flat["k"], flat["v"], flat["gk"],
                                                 flat["beta"], np.arange(B + 1) * G, S0, 1, G)
        got = snaps[l][snap_ids.long().to(DEV)]          # [B, G, H, K, V]
        assert_close(got, ck, dtype, "snapshots")

    # commit vs the ReplaySSM fold of the same accept lengths (bit-exact)
    accept = torch.tensor([0, 1, min(3, G), G, min(2, G)], dtype=torch.int32)
    acc_d = accept.to(DEV)
    R = kda().ring_len_for(G - 1)
    rings = [kda().make_ring(S, R, H, dtype, DEV) for _ in range(L)]
    folded = [c.clone() for c in committed]
    for l in range(L):
        xd = _dev(xs[l])
        kda().kda_verify_store_inputs(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"], idd,
                                      folded[l], rings[l])
    kda().kda_replay_fold(folded, rings, idd, acc_d, max_accept=G)
    kda().kda_snapshot_commit(pools, snaps, idd, snd, acc_d, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for l in range(L):
        assert torch.equal(pools[l], folded[l]), "commit differs from the fold, layer %d" % l
        other = torch.ones(S, dtype=torch.bool)
        other[ids.long()] = False
        assert torch.equal(pools[l][other.to(DEV)], committed[l][other.to(DEV)])


def test_snapshot_commit_bad_ids():
    """An accept length above G and a snapshot slot out of range skip their
    requests with the matching error bits; the rest commit."""
    g = gen.make_gen(79)
    B, G, H, S, NS = 3, 4, 2, 6, 3
    pool = gen.checkpoint((S, H, KD, VD), g).to(DEV)
    before = pool.clone()
    snaps = gen.checkpoint((NS, G, H, KD, VD), g).to(DEV)
    ids = torch.tensor([0, 1, 2], dtype=torch.int32, device=DEV)
    snap_ids = torch.tensor([0, 7, 2], dtype=torch.int32, device=DEV)    # request 1: out of range
    accept = torch.tensor([2, 1, G + 1], dtype=torch.int32, device=DEV)  # request 2: above G
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda().kda_snapshot_commit([pool], [snaps], ids, snap_ids, accept, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == (kda().KDA_DEVERR_SLOT_RANGE | kda().KDA_DEVERR_ACCEPT_RANGE)
    assert torch.equal(pool[0], snaps[0, 1])
    assert torch.equal(pool[1:], before[1:])
