"""Full-size parity: the five workloads at their own sizes, launched the way
the benchmark launches them, checked against the oracle on sampled units
(the oracle computes each unit independently) and on properties that hold at
any size (committed states untouched by verify, fold == repeated decode bit
for bit, snapshots and copies exact, untouched slots unchanged)."""
import numpy as np
import pytest
import torch

import kda_inputs as gen
import oracle
from kda_testutil import assert_close, f64

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


def _host(x, heads):
    """Selected heads of token-major inputs, as float64 numpy."""
    idx = torch.tensor(heads, device=x["q"].device)
    return {n: f64(t.index_select(1, idx)) for n, t in x.items()}


@pytest.mark.parametrize("init", ["zero", "ckpt"])
def test_varlen_prefill_full(init):
    """8 sequences, lengths U[64, 2048] (seed 1), H = 64, bf16, zero or
    checkpointed initial states: every sequence on three heads vs the oracle."""
    w = gen.varlen_batch(DEV)
    x, N, H, cu = w["x"], w["N"], w["H"], w["cu"]
    pool = torch.zeros(2 * N, H, KD, VD, device=DEV)
    pool[:N] = w["ck"]
    init_slot = (torch.arange(N, dtype=torch.int32) if init == "ckpt"
                 else torch.full((N,), -1, dtype=torch.int32)).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = kda().kda_chunk_prefill(x["q"], x["k"], x["v"], x["gk"], x["beta"], cu.to(DEV), cu, pool,
                                init_slot, torch.arange(N, 2 * N, dtype=torch.int32, device=DEV),
                                dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    heads = [0, 29, 63]
    xs = _host(x, heads)
    S0 = f64(w["ck"][:, heads]) if init == "ckpt" else np.zeros((N, len(heads), KD, VD))
    o_ref, S_ref = oracle.prefill_varlen(xs["q"], xs["k"], xs["v"], xs["gk"], xs["beta"],
                                         cu.numpy(), S0)
    assert_close(o[:, heads], o_ref, torch.bfloat16, "o")
    assert_close(pool[N:, heads], S_ref, torch.bfloat16, "final states")


def test_varlen_prefill_checkpoints_full():
    """The varlen workload with a checkpoint every 256 tokens (the prefix
    cache's block), launched as the benchmark launches it: outputs and final
    states bit-identical to the plain prefill; every checkpoint bit-identical
    to the final state of a plain prefill of that prefix; three heads of every
    sequence vs the oracle."""
    w = gen.varlen_batch(DEV)
    x, N, H, cu = w["x"], w["N"], w["H"], w["cu"]
    I = 256
    lengths = (cu[1:] - cu[:-1]).tolist()
    cap = max(lengths) // I
    made = [L // I for L in lengths]
    slots = torch.arange(2 * N, 2 * N + N * cap, dtype=torch.int32).view(N, cap)
    pool = torch.zeros(2 * N + N * cap, H, KD, VD, device=DEV)
    pool[:N] = w["ck"]
    init = torch.arange(N, dtype=torch.int32, device=DEV)
    out = torch.arange(N, 2 * N, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = kda().kda_chunk_prefill_checkpoints(x["q"], x["k"], x["v"], x["gk"], x["beta"],
                                            cu.to(DEV), cu, pool, init, out, I, slots.to(DEV),
                                            dev_err=err)
    pool_p = torch.zeros(2 * N, H, KD, VD, device=DEV)
    pool_p[:N] = w["ck"]
    o_p = kda().kda_chunk_prefill(x["q"], x["k"], x["v"], x["gk"], x["beta"], cu.to(DEV), cu,
                                  pool_p, init, out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(o, o_p) and torch.equal(pool[N:2 * N], pool_p[N:])
    offs = cu.tolist()
    for m in range(cap):
        keep = [min(L, (m + 1) * I) for L in lengths]
        idx = torch.cat([torch.arange(offs[n], offs[n] + keep[n]) for n in range(N)]).to(DEV)
        xp = {k_: t.index_select(0, idx).contiguous() for k_, t in x.items()}
        cup = gen.cu_seqlens(keep)
        pool_q = pool_p.clone()
        pool_q[:N] = w["ck"]
        kda().kda_chunk_prefill(xp["q"], xp["k"], xp["v"], xp["gk"], xp["beta"], cup.to(DEV), cup,
                                pool_q, init, out)
        torch.cuda.synchronize()
        for n in range(N):
            if m < made[n]:
                assert torch.equal(pool[int(slots[n, m])], pool_q[N + n]), (m, n)
    heads = [0, 29, 63]
    xs = _host(x, heads)
    _, _, ck_ref, made_ref = oracle.prefill_checkpoints(
        xs["q"], xs["k"], xs["v"], xs["gk"], xs["beta"], cu.numpy(), f64(w["ck"][:, heads]), I, cap)
    assert list(made_ref) == made
    for n in range(N):
        for m in range(made[n]):
            assert_close(pool[int(slots[n, m])][heads], ck_ref[n, m], torch.bfloat16,
                         "checkpoint %d of sequence %d" % (m, n))


def test_decode_fused_full_layer():
    """One layer of the decode workload (384 requests x 64 heads, 512-slot
    pools) through conv + KDA + onorm, launched as the benchmark launches it:
    bit-identical to prologue + decode step + norm; untouched slots unchanged;
    the outputs of 16 requests vs the oracle (bf16 intermediates stored as the
    unfused path stores them)."""
    from oracle import fused_ops as fo
    B, H, S = 384, 64, 512
    g = gen.make_gen(3)
    ids = gen.slot_permutation(S, g)[:B].to(DEV)
    gd = gen.make_gen(1007, DEV)
    pool0 = gen.checkpoint((S, H, KD, VD), gd, device=DEV)
    cs0 = gen.checkpoint((S, 3, 3, H, KD), gd, device=DEV, std=1.0).to(torch.bfloat16)
    x = {n: t[:, 0] for n, t in gen.raw_projections(1, H, torch.bfloat16, gd, device=DEV,
                                                      lead=(B,)).items()}
    w = gen.fused_weights(H, torch.bfloat16, gd, device=DEV)
    raw = (x["qkv"][:, 0], x["qkv"][:, 1], x["qkv"][:, 2])
    scale = KD ** -0.5
    pool_f, cs_f = pool0.clone(), cs0.clone()
    out_f = kda().kda_decode_fused(*raw, x["gk"], x["b"], w["conv_w"], cs_f, x["gate"], w["w_norm"],
                                   ids, pool_f, scale=scale)
    pool_u, cs_u = pool0.clone(), cs0.clone()
    cu = torch.arange(B + 1, dtype=torch.int32)
    q, k, v, beta = kda().kda_conv_prologue(*raw, x["b"], w["conv_w"], cs_u, ids, ids, cu.to(DEV), cu)
    o = kda().kda_decode_step(q, k, v, x["gk"], beta, ids, pool_u, scale=scale)
    out_u = kda().kda_gated_rmsnorm(o, x["gate"], w["w_norm"])
    torch.cuda.synchronize()
    assert torch.equal(out_f, out_u) and torch.equal(pool_f, pool_u) and torch.equal(cs_f, cs_u)
    other = torch.ones(S, dtype=torch.bool, device=DEV)
    other[ids.long()] = False
    assert torch.equal(pool_f[other], pool0[other]) and torch.equal(cs_f[other], cs0[other])
    sel = torch.arange(0, B, B // 16, device=DEV)[:16]
    sid = ids[sel].long()
    ref_out, _, _ = fo.decode_fused(*(f64(t[sel]) for t in raw), f64(x["gk"][sel]), f64(x["b"][sel]),
                                    f64(w["conv_w"]), f64(cs0), f64(x["gate"][sel]), f64(w["w_norm"]),
                                    sid.cpu().numpy(), f64(pool0), scale=scale, store=fo.round_bf16)
    assert_close(out_f[sel], ref_out, torch.bfloat16, "fused decode out")


def test_long_prefill_pieces_full():
    """4 sequences x 24576 tokens, H = 96, bf16, from checkpoints, as six
    pieces of 4096 tokens that resume in place; after each piece the state is
    also written to a snapshot slot that alternates between two (ping-pong).
    Final states and outputs of sampled units vs the oracle over the whole
    sequence; the last snapshot equals the working slot; the other one equals
    the oracle's state after five pieces."""
    w = gen.long_batch(DEV)
    x, N, T, H = w["x"], w["N"], w["T"], w["H"]
    P = 4096
    pool = torch.zeros(3 * N, H, KD, VD, device=DEV)
    pool[:N] = w["ck"]
    work = torch.arange(N, dtype=torch.int32, device=DEV)
    snaps = [torch.arange(N, 2 * N, dtype=torch.int32, device=DEV),
             torch.arange(2 * N, 3 * N, dtype=torch.int32, device=DEV)]
    cu = gen.cu_seqlens([P] * N)
    cu_d = cu.to(DEV)
    o = torch.empty(N * T, H, VD, dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for piece in range(T // P):
        rows = torch.cat([torch.arange(n * T + piece * P, n * T + (piece + 1) * P) for n in range(N)]).to(DEV)
        sub = {k: t.index_select(0, rows) for k, t in x.items()}
        op = kda().kda_chunk_prefill(sub["q"], sub["k"], sub["v"], sub["gk"], sub["beta"], cu_d, cu,
                                     pool, work, work, snaps[piece % 2], dev_err=err)
        o.index_copy_(0, rows, op)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    last = (T // P - 1) % 2
    assert torch.equal(pool[snaps[last].long()], pool[work.long()])
    units = [(0, 0), (1, 47), (2, 95), (3, 13)]
    for n, h in units:
        sl = slice(n * T, (n + 1) * T)
        xs = {k: f64(t[sl, h]) for k, t in x.items()}
        S0 = f64(w["ck"][n, h])
        o_ref, S_ref = oracle.unit(xs["q"], xs["k"], xs["v"], xs["gk"], xs["beta"], S0)
        assert_close(o[sl, h], o_ref, torch.bfloat16, "o, unit %s" % ((n, h),))
        assert_close(pool[n, h], S_ref, torch.bfloat16, "final state, unit %s" % ((n, h),))
        cut = (T // P - 1) * P
        _, S5 = oracle.unit(xs["q"][:cut], xs["k"][:cut], xs["v"][:cut], xs["gk"][:cut],
                            xs["beta"][:cut], S0)
        assert_close(pool[snaps[1 - last][n].item(), h], S5, torch.bfloat16,
                     "snapshot after 5 pieces, unit %s" % ((n, h),))


def test_decode_full_layer():
    """384 requests x 1 token, H = 64, bf16, a 512-slot pool indexed by a
    seeded permutation, copy-on-write restores for 38 requests before the
    step (one layer of the 69-layer step, identical launches)."""
    B, H, S = 384, 64, 512
    g = gen.make_gen(3)
    perm = gen.slot_permutation(S, g)
    ids = perm[:B]
    n_cow = int(0.10 * B)
    cow_req = torch.randperm(B, generator=g)[:n_cow]
    cow_dst = ids[cow_req].to(torch.int32)
    cow_src = perm[B:][torch.randint(0, S - B, (n_cow,), generator=g)].to(torch.int32)
    gd = gen.make_gen(1003, DEV)
    pool = gen.checkpoint((S, H, KD, VD), gd, device=DEV)
    x = gen.token_inputs(B, H, torch.bfloat16, gd, device=DEV)
    before = pool.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda().kda_slot_copy([pool], cow_src.to(DEV), cow_dst.to(DEV), dev_err=err)
    o = kda().kda_decode_step(x["q"], x["k"], x["v"], x["gk"], x["beta"], ids.to(DEV), pool,
                              dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the state each request started from: its slot, or the copy-on-write source
    start = before[ids.long().to(DEV)].clone()
    start[cow_req.to(DEV)] = before[cow_src.long().to(DEV)]
    sample = torch.cat([cow_req[:4], torch.tensor([0, 1, 191, 383])]).unique()
    xs = {k: f64(t[sample.to(DEV)]) for k, t in x.items()}
    o_ref, S_ref = oracle.decode(xs["q"], xs["k"], xs["v"], xs["gk"], xs["beta"],
                                 f64(start[sample.to(DEV)]))
    assert_close(o[sample.to(DEV)], o_ref, torch.bfloat16, "o")
    assert_close(pool[ids[sample].long().to(DEV)], S_ref, torch.bfloat16, "S")
    untouched = torch.ones(S, dtype=torch.bool)
    untouched[ids.long()] = False
    assert torch.equal(pool[untouched.to(DEV)], before[untouched.to(DEV)])


def test_verify_fold_full():
    """64 requests x 8 draft tokens, 69 layers x H = 64, 128-slot pools, ring
    16, accept lengths 1..8 (mean about 2.7): 69 verify launches then one fold
    over all layers.  Committed states untouched by verify; every layer's
    fold bit-identical to repeated decode; sampled units vs the oracle."""
    B, G, H, S, R, Lyr = 64, 8, 64, 128, 16, 69
    g = gen.make_gen(4)
    ids = gen.slot_permutation(S, g)[:B]
    accept = gen.accept_lengths(B, G, 0.64, g)
    assert 1 <= int(accept.min()) and int(accept.max()) <= G
    gd = gen.make_gen(1004, DEV)
    pools = [gen.checkpoint((S, H, KD, VD), gd, device=DEV) for _ in range(Lyr)]
    rings = [kda().make_ring(S, R, H, torch.bfloat16, DEV) for _ in range(Lyr)]
    xs = [gen.token_inputs(G, H, torch.bfloat16, gd, device=DEV, lead=(B,)) for _ in range(Lyr)]
    committed = [p.clone() for p in pools]
    idd = ids.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = []
    for l in range(Lyr):
        x = xs[l]
        outs.append(kda().kda_verify_store_inputs(x["q"], x["k"], x["v"], x["gk"], x["beta"], idd,
                                                  pools[l], rings[l], dev_err=err))
    torch.cuda.synchronize()
    for l in range(Lyr):
        assert torch.equal(pools[l], committed[l]), "verify wrote layer %d" % l
    kda().kda_replay_fold(pools, rings, idd, accept.to(DEV), max_accept=G, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    reqs = [0, 17, 63]
    ref = torch.empty_like(pools[0])
    for l in range(Lyr):
        x = xs[l]
        ref.copy_(committed[l])
        for i in range(G):
            sel = (accept > i).nonzero().flatten().to(DEV)
            kda().kda_decode_step(*(x[n][sel, i].contiguous() for n in ("q", "k", "v", "gk", "beta")),
                                  idd[sel].contiguous(), ref)
        torch.cuda.synchronize()
        assert torch.equal(pools[l], ref), "fold differs from repeated decode, layer %d" % l
        if l not in (0, 34, 68):
            continue
        rs = torch.tensor(reqs, device=DEV)
        xh = {n: f64(t[rs]) for n, t in x.items()}
        S0 = f64(committed[l][idd[rs].long()])
        o_ref = oracle.verify(xh["q"], xh["k"], xh["v"], xh["gk"], xh["beta"], S0)
        assert_close(outs[l][rs], o_ref, torch.bfloat16, "verify o, layer %d" % l)
        S_ref = oracle.fold(xh["k"], xh["v"], xh["gk"], xh["beta"], accept[reqs].numpy(), S0)
        assert_close(pools[l][idd[rs].long()], S_ref, torch.bfloat16, "fold S, layer %d" % l)
    del pools, rings, xs, committed
    torch.cuda.empty_cache()
