"""GPU parity: every entry point of the C ABI against the oracle on seeded
inputs, at sizes the oracle finishes in seconds (several chunks, ragged tails,
empty sequences), plus the bit-exact contracts: fold == repeated decode,
verify never writes the committed state, copies and snapshots are exact, and
untouched slots keep their canary."""
import numpy as np
import pytest
import torch

import kda_inputs as gen
import oracle
from kda_testutil import TOL, assert_close, canary_fill, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
KD = VD = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kda_state_gb300 import _build
    _build.build()
    import kda_state_gb300 as kda
    kda.lib()


def kda():
    import kda_state_gb300
    return kda_state_gb300


def _dev(x):
    return {n: t.to(DEV) for n, t in x.items()}


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------

def run_prefill_case(lengths, H, dtype, init_kind, seed, scale=1.0):
    g = gen.make_gen(seed)
    N = len(lengths)
    cu = gen.cu_seqlens(lengths)
    T = int(cu[-1])
    x = gen.token_inputs(T, H, dtype, g)
    ck = gen.checkpoint((N, H, KD, VD), g)
    # slots: [0, N) checkpoints, [N, 2N) outputs, [2N, 3N) snapshots, 3N untouched canary
    pool = canary_fill(torch.empty(3 * N + 1, H, KD, VD, device=DEV))
    pool[:N] = ck.to(DEV)
    before = pool.clone()
    init = [(-1 if (init_kind == "zero" or (init_kind == "mixed" and n % 2 == 0)) else n)
            for n in range(N)]
    S0 = np.stack([np.zeros((H, KD, VD)) if init[n] < 0 else f64(ck[n]) for n in range(N)])
    dev_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    xd = _dev(x)
    o = kda().kda_chunk_prefill(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"], cu.to(DEV), cu,
                                pool, torch.tensor(init, dtype=torch.int32, device=DEV),
                                torch.arange(N, 2 * N, dtype=torch.int32, device=DEV),
                                torch.arange(2 * N, 3 * N, dtype=torch.int32, device=DEV),
                                scale=scale, dev_err=dev_err)
    torch.cuda.synchronize()
    assert int(dev_err.item()) == 0
    o_ref, S_ref = oracle.prefill_varlen(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["gk"]),
                                         f64(x["beta"]), cu.numpy(), S0, scale=scale)
    return dict(o=o, o_ref=o_ref, pool=pool, before=before, S_ref=S_ref, N=N, x=x, cu=cu, ck=ck)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("init_kind", ["zero", "ckpt", "mixed"])
def test_prefill_varlen_small(dtype, init_kind):
    r = run_prefill_case([1, 63, 64, 65, 200, 0, 130], 3, dtype, init_kind, seed=11)
    N, pool = r["N"], r["pool"]
    if r["cu"][-1] > 0:
        assert_close(r["o"], r["o_ref"], dtype, "o")
    assert_close(pool[N:2 * N], r["S_ref"], dtype, "final states")
    assert torch.equal(pool[2 * N:3 * N], pool[N:2 * N]), "snapshot differs from the final state"
    assert torch.equal(pool[:N], r["before"][:N]), "checkpoint slots were written"
    assert torch.equal(pool[3 * N], r["before"][3 * N]), "untouched slot was written"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_prefill_all_sequences_empty(dtype):
    """A batch without tokens: each output and snapshot slot receives its
    initial state bit for bit (zeros where init_slot is -1); nothing else is
    written and o is empty."""
    r = run_prefill_case([0, 0, 0], 2, dtype, "mixed", seed=13)
    N, pool = r["N"], r["pool"]
    assert r["o"].numel() == 0
    want = torch.from_numpy(r["S_ref"]).float()
    assert torch.equal(pool[N:2 * N].cpu(), want), "final states differ from the initial states"
    assert torch.equal(pool[2 * N:3 * N].cpu(), want), "snapshots differ from the initial states"
    assert torch.equal(pool[:N], r["before"][:N]), "checkpoint slots were written"
    assert torch.equal(pool[3 * N], r["before"][3 * N]), "untouched slot was written"


def test_decode_empty_batch_is_a_no_op():
    """B = 0: the call succeeds, launches nothing and leaves the pool as it was."""
    pool = canary_fill(torch.empty(2, 3, KD, VD, device=DEV))
    before = pool.clone()
    e = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device=DEV)
    o = kda().kda_decode_step(e(0, 3, KD), e(0, 3, KD), e(0, 3, VD), e(0, 3, KD), e(0, 3),
                              torch.empty(0, dtype=torch.int32, device=DEV), pool)
    torch.cuda.synchronize()
    assert o.shape == (0, 3, VD)
    assert torch.equal(pool, before)


def test_tiny_config():
    """1 sequence, T = 64, H = 1, fp32, zero state, seed 0; the oracle's
    chunked form with chunk 64 gives the same reference."""
    r = run_prefill_case([64], 1, torch.float32, "zero", seed=0)
    assert_close(r["o"], r["o_ref"], torch.float32, "o")
    assert_close(r["pool"][1:2], r["S_ref"], torch.float32, "S")
    x = r["x"]
    oc, Sc = oracle.unit(f64(x["q"][:, 0]), f64(x["k"][:, 0]), f64(x["v"][:, 0]),
                         f64(x["gk"][:, 0]), f64(x["beta"][:, 0]), np.zeros((KD, VD)), chunk=64)
    assert_close(r["o"][:, 0], oc, torch.float32, "o vs chunked")
    assert_close(r["pool"][1, 0], Sc, torch.float32, "S vs chunked")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_prefill_split_resume_in_place(dtype):
    """Prefill in two pieces, the second resuming in place from the first's
    output slot, matches the oracle's unsplit run."""
    g = gen.make_gen(12)
    H, lengths, cut = 2, [300, 129], [128, 64]
    x = gen.token_inputs(sum(lengths), H, dtype, g)
    xd = _dev(x)
    ck = gen.checkpoint((2, H, KD, VD), g)
    pool = ck.to(DEV).clone()
    slots = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
    offs = [0, lengths[0]]
    o = torch.empty(sum(lengths), H, VD, dtype=dtype, device=DEV)
    for piece in range(2):
        segs = [(offs[n] + (0 if piece == 0 else cut[n]),
                 offs[n] + (cut[n] if piece == 0 else lengths[n])) for n in range(2)]
        idx = torch.cat([torch.arange(a, b) for a, b in segs])
        cu = gen.cu_seqlens([b - a for a, b in segs])
        sub = {n: t[idx.to(DEV)].contiguous() for n, t in xd.items()}
        op = kda().kda_chunk_prefill(sub["q"], sub["k"], sub["v"], sub["gk"], sub["beta"],
                                     cu.to(DEV), cu, pool, slots, slots)
        o[idx.to(DEV)] = op
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.prefill_varlen(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["gk"]),
                                         f64(x["beta"]), gen.cu_seqlens(lengths).numpy(), f64(ck))
    assert_close(o, o_ref, dtype, "o")
    assert_close(pool, S_ref, dtype, "S")


def test_prefill_fp32_matches_decode_steps_bitwise():
    """The exact fp32 prefill and T decode steps run the same per-token
    arithmetic: identical states and outputs, bit for bit."""
    g = gen.make_gen(13)
    H, T = 2, 9
    x = gen.token_inputs(T, H, torch.float32, g)
    xd = _dev(x)
    ck = gen.checkpoint((1, H, KD, VD), g).to(DEV)
    pool_a = ck.clone()
    cu = gen.cu_seqlens([T])
    s = torch.zeros(1, dtype=torch.int32, device=DEV)
    o_a = kda().kda_chunk_prefill(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"], cu.to(DEV), cu,
                                  pool_a, s, s)
    pool_b = ck.clone()
    o_b = torch.empty_like(o_a)
    for t in range(T):
        o_b[t:t + 1] = kda().kda_decode_step(*(xd[n][t:t + 1] for n in ("q", "k", "v", "gk", "beta")),
                                             s, pool_b)
    torch.cuda.synchronize()
    assert torch.equal(pool_a, pool_b)
    assert torch.equal(o_a, o_b)


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_decode(dtype):
    g = gen.make_gen(21)
    B, H, S = 7, 3, 16
    x = gen.token_inputs(B, H, dtype, g)
    pool = gen.checkpoint((S, H, KD, VD), g).to(DEV)
    ids = gen.slot_permutation(S, g)[:B]
    before = pool.clone()
    xd = _dev(x)
    o = kda().kda_decode_step(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"], ids.to(DEV), pool,
                              scale=0.75)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.decode(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["gk"]),
                                 f64(x["beta"]), f64(before[ids.long().to(DEV)]), scale=0.75)
    assert_close(o, o_ref, dtype, "o")
    assert_close(pool[ids.long().to(DEV)], S_ref, dtype, "S")
    other = torch.ones(S, dtype=torch.bool)
    other[ids.long()] = False
    assert torch.equal(pool[other.to(DEV)], before[other.to(DEV)])


# ---------------------------------------------------------------------------
# verify + fold
# ---------------------------------------------------------------------------

def _verify_fold_setup(dtype, seed, B=5, G=8, H=2, L=3, S=12, R=16):
    g = gen.make_gen(seed)
    pools = [gen.checkpoint((S, H, KD, VD), g).to(DEV) for _ in range(L)]
    xs = [gen.token_inputs(G, H, dtype, g, lead=(B,)) for _ in range(L)]
    ids = gen.slot_permutation(S, g)[:B]
    base = torch.randint(0, R, (B,), generator=g, dtype=torch.int32)
    rings = [kda().make_ring(S, R, H, dtype, DEV) for _ in range(L)]
    return g, pools, xs, ids, base, rings


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_verify_then_fold(dtype):
    B, G, H, L, S, R = 5, 8, 2, 3, 12, 16
    g, pools, xs, ids, base, rings = _verify_fold_setup(dtype, 31, B, G, H, L, S, R)
    committed = [p.clone() for p in pools]
    idd, based = ids.to(DEV), base.to(DEV)
    outs = []
    for l in range(L):
        xd = _dev(xs[l])
        outs.append(kda().kda_verify_store_inputs(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"],
                                                  idd, pools[l], rings[l], ring_base=based,
                                                  scale=1.0))
    torch.cuda.synchronize()
    for l in range(L):
        assert torch.equal(pools[l], committed[l]), "verify wrote the committed state"
        x = xs[l]
        o_ref = oracle.verify(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["gk"]), f64(x["beta"]),
                              f64(committed[l][ids.long().to(DEV)]))
        assert_close(outs[l], o_ref, dtype, "verify o, layer %d" % l)
        # stored records: k, v as given, exp(gk) and beta as fp32
        for b in range(B):
            ent = [(int(base[b]) + i) % R for i in range(G)]
            s = int(ids[b])
            assert torch.equal(rings[l].k[s, ent].cpu(), x["k"][b])
            assert torch.equal(rings[l].v[s, ent].cpu(), x["v"][b])
            assert torch.equal(rings[l].beta[s, ent].cpu(), x["beta"][b].float())
            np.testing.assert_allclose(f64(rings[l].decay[s, ent]), np.exp(f64(x["gk"][b])),
                                       rtol=5e-7, atol=0)
    accept = torch.tensor([0, 1, 3, G, 5], dtype=torch.int32)
    kda().kda_replay_fold(pools, rings, idd, accept.to(DEV), max_accept=G, ring_base=based)
    torch.cuda.synchronize()
    for l in range(L):
        # bit-exact against the GPU's own sequential commit (decode steps)
        ref = committed[l].clone()
        xd = _dev(xs[l])
        for i in range(G):
            sel = (accept > i).nonzero().flatten()
            if sel.numel() == 0:
                continue
            seld = sel.to(DEV)
            kda().kda_decode_step(*(xd[n][seld, i].contiguous() for n in ("q", "k", "v", "gk", "beta")),
                                  idd[seld].contiguous(), ref)
        torch.cuda.synchronize()
        assert torch.equal(pools[l], ref), "fold is not bit-identical to decode, layer %d" % l
        x = xs[l]
        S_ref = oracle.fold(f64(x["k"]), f64(x["v"]), f64(x["gk"]), f64(x["beta"]), accept.numpy(),
                            f64(committed[l][ids.long().to(DEV)]))
        assert_close(pools[l][ids.long().to(DEV)], S_ref, dtype, "fold S, layer %d" % l)
        other = torch.ones(S, dtype=torch.bool)
        other[ids.long()] = False
        assert torch.equal(pools[l][other.to(DEV)], committed[l][other.to(DEV)])


# ---------------------------------------------------------------------------
# slot copy
# ---------------------------------------------------------------------------

def test_slot_copy_exact():
    g = gen.make_gen(41)
    P, S, H = 3, 10, 2
    pools = [gen.checkpoint((S, H, KD, VD), g).to(DEV) for _ in range(P)]
    before = [p.clone() for p in pools]
    src = torch.tensor([0, 3, 7], dtype=torch.int32)
    dst = torch.tensor([5, 1, 9], dtype=torch.int32)
    kda().kda_slot_copy(pools, src.to(DEV), dst.to(DEV))
    torch.cuda.synchronize()
    for p, b in zip(pools, before):
        exp = b.clone()
        exp[dst.long().to(DEV)] = b[src.long().to(DEV)]
        assert torch.equal(p, exp)


def test_slot_copy_odd_size():
    """A slot size that is not a multiple of the copy kernel's chunk."""
    g = gen.make_gen(42)
    pool = torch.randn(6, 12340, generator=torch.Generator().manual_seed(1)).to(DEV)
    before = pool.clone()
    kda().kda_slot_copy([pool], torch.tensor([4], dtype=torch.int32, device=DEV),
                        torch.tensor([2], dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    exp = before.clone()
    exp[2] = before[4]
    assert torch.equal(pool, exp)


# ---------------------------------------------------------------------------
# device-side error reporting (no trap; the bad unit is skipped)
# ---------------------------------------------------------------------------

def test_device_errors_are_reported_and_skipped():
    g = gen.make_gen(51)
    B, H, S = 3, 2, 6
    x = _dev(gen.token_inputs(B, H, torch.bfloat16, g))
    pool = gen.checkpoint((S, H, KD, VD), g).to(DEV)
    before = pool.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids = torch.tensor([1, 99, 4], dtype=torch.int32, device=DEV)
    kda().kda_decode_step(x["q"], x["k"], x["v"], x["gk"], x["beta"], ids, pool, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kda().KDA_DEVERR_SLOT_RANGE
    assert not torch.equal(pool[1], before[1]) and not torch.equal(pool[4], before[4])
    assert torch.equal(pool[[0, 2, 3, 5]], before[[0, 2, 3, 5]])

    # accept length beyond max_accept
    rings = [kda().make_ring(S, 16, H, torch.bfloat16, DEV)]
    err.zero_()
    kda().kda_replay_fold([pool], rings, torch.tensor([0, 2], dtype=torch.int32, device=DEV),
                          torch.tensor([9, 0], dtype=torch.int32, device=DEV), max_accept=8,
                          dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kda().KDA_DEVERR_ACCEPT_RANGE

    # device cu_seqlens disagreeing with the (valid) host copy
    err.zero_()
    xs = _dev(gen.token_inputs(8, H, torch.bfloat16, g))
    cu_host = torch.tensor([0, 3, 8], dtype=torch.int32)
    cu_bad = torch.tensor([0, 9, 8], dtype=torch.int32, device=DEV)
    sl = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
    kda().kda_chunk_prefill(xs["q"], xs["k"], xs["v"], xs["gk"], xs["beta"], cu_bad, cu_host,
                            pool, sl, sl, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kda().KDA_DEVERR_SEQLENS


@pytest.mark.parametrize("case", ["strong_decay_fallback", "growth_fallback", "long_draft_recurrent"])
def test_verify_other_paths(case):
    """Verify's other code paths: a draft whose cumulative decay leaves the
    range of the block form below (gk = -12 per step) or above (gk = +9 per
    step: the product passes 1e30 at the eighth draft, the state stays far
    inside fp32), and G = 20 > 16 drafts."""
    g = gen.make_gen(61)
    B, H, S = 3, 2, 6
    G, R = (20, 64) if case == "long_draft_recurrent" else (8, 16)
    x = gen.token_inputs(G, H, torch.bfloat16, g, lead=(B,))
    if case == "strong_decay_fallback":
        x["gk"] = torch.full_like(x["gk"], -12.0)
    if case == "growth_fallback":
        x["gk"] = torch.full_like(x["gk"], 9.0)
    pool = gen.checkpoint((S, H, KD, VD), g).to(DEV)
    committed = pool.clone()
    ids = torch.tensor([4, 0, 2], dtype=torch.int32, device=DEV)
    ring = kda().make_ring(S, R, H, torch.bfloat16, DEV)
    xd = _dev(x)
    o = kda().kda_verify_store_inputs(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"], ids, pool, ring)
    torch.cuda.synchronize()
    assert torch.equal(pool, committed)
    o_ref = oracle.verify(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["gk"]), f64(x["beta"]),
                          f64(committed[ids.long()]))
    assert_close(o, o_ref, torch.bfloat16, "verify o")
    for b in range(B):
        s = int(ids[b])
        assert torch.equal(ring.k[s, :G].cpu(), x["k"][b])
        assert torch.equal(ring.beta[s, :G].cpu(), x["beta"][b].float())


def test_verify_many_units_mixed():
    """Many units (more than can be resident at once): normal drafts, drafts on
    the strong-decay fallback and one out-of-range slot interleaved; every
    valid unit vs the oracle, the skipped request's outputs untouched."""
    g = gen.make_gen(62)
    B, G, H, S, R = 170, 8, 4, 180, 16
    x = gen.token_inputs(G, H, torch.bfloat16, g, lead=(B,))
    strong = torch.zeros(B, dtype=torch.bool)
    strong[::7] = True
    x["gk"][strong] = -12.0
    pool = gen.checkpoint((S, H, KD, VD), g).to(DEV)
    committed = pool.clone()
    ids = gen.slot_permutation(S, g)[:B].clone()
    ids[100] = S + 5                                   # out of range: reported and skipped
    ring = kda().make_ring(S, R, H, torch.bfloat16, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    xd = _dev(x)
    o = torch.full((B, G, H, VD), 7.0, dtype=torch.bfloat16, device=DEV)
    kda().kda_verify_store_inputs(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"], ids.to(DEV), pool,
                                  ring, o=o, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kda().KDA_DEVERR_SLOT_RANGE
    assert torch.equal(pool, committed)
    assert torch.all(o[100] == 7.0), "the skipped request's outputs were written"
    valid = [b for b in range(B) if b != 100]
    vb = torch.tensor(valid)
    o_ref = oracle.verify(f64(x["q"][vb]), f64(x["k"][vb]), f64(x["v"][vb]), f64(x["gk"][vb]),
                          f64(x["beta"][vb]), f64(committed[ids[vb].long()]))
    assert_close(o[vb.to(DEV)], o_ref, torch.bfloat16, "verify o")
    for b in (0, 1, 7, 169):
        s = int(ids[b])
        assert torch.equal(ring.k[s, :G].cpu(), x["k"][b])
        assert torch.equal(ring.v[s, :G].cpu(), x["v"][b])
        np.testing.assert_allclose(f64(ring.decay[s, :G]), np.exp(f64(x["gk"][b])), rtol=5e-7, atol=0)
