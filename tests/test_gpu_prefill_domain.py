"""The bf16 chunked prefill over the whole input domain of the recurrence.

The tensor-core path scales q and k by the chunk's cumulative decay exp(G) and
k by exp(-G) (TF32 operands); chunks whose products could leave fp32 range
(fast-forgetting key channels, a positive gk, large k, v or state) must still
give the oracle's result.  Every case here is compared with
the oracle at the bf16 tolerance; none may report an error, and the snapshot,
checkpoint and canary slots obey the same contracts as on ordinary inputs.
The prefill's own bounded wait is exercised through kda_selftest_prefill_wait.
"""
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


def strong_decay(gk, g, channels, lo, hi, tokens=None):
    """gk with the given key channels of every head set to -U[lo, hi] per token
    (seeded), on the given token rows (all by default)."""
    gk = gk.clone().float()
    rows = slice(None) if tokens is None else tokens
    sel = gk[rows][:, :, channels]
    u = torch.rand(sel.shape, generator=g) * (hi - lo) + lo
    gk[rows, :, channels] = -u
    return gk


def run(x, lengths, H, init_kind="ckpt", seed=0, ck_scale=1.0, inplace=False):
    """One kda_chunk_prefill call on bf16 inputs x against the oracle; returns
    the pool and the reference."""
    g = gen.make_gen(seed + 500)
    N = len(lengths)
    cu = gen.cu_seqlens(lengths)
    xb = {n: t.to(torch.bfloat16) for n, t in x.items()}
    ck = gen.checkpoint((N, H, KD, VD), g) * ck_scale
    pool = canary_fill(torch.empty(3 * N + 1, H, KD, VD, device=DEV))
    pool[:N] = ck.to(DEV)
    before = pool.clone()
    init = [(-1 if (init_kind == "zero" or (init_kind == "mixed" and n % 2 == 0)) else n)
            for n in range(N)]
    out = list(range(N)) if inplace else list(range(N, 2 * N))
    if inplace:
        init = list(range(N))
    S0 = np.stack([np.zeros((H, KD, VD)) if init[n] < 0 else f64(ck[n]) for n in range(N)])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    xd = {n: t.to(DEV) for n, t in xb.items()}
    o = kda().kda_chunk_prefill(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"], cu.to(DEV), cu,
                                pool, torch.tensor(init, dtype=torch.int32, device=DEV),
                                torch.tensor(out, dtype=torch.int32, device=DEV),
                                torch.arange(2 * N, 3 * N, dtype=torch.int32, device=DEV), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "the prefill reported device error bits %d" % int(err.item())
    o_ref, S_ref = oracle.prefill_varlen(f64(xb["q"]), f64(xb["k"]), f64(xb["v"]), f64(xb["gk"]),
                                         f64(xb["beta"]), cu.numpy(), S0)
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(pool[out], S_ref, torch.bfloat16, "final states")
    assert torch.equal(pool[2 * N:3 * N], pool[out]), "snapshot differs from the final state"
    assert torch.equal(pool[3 * N], before[3 * N]), "untouched slot was written"
    if not inplace:
        assert torch.equal(pool[:N], before[:N]), "checkpoint slots were written"
    return pool, o


LENGTHS = [200, 65, 130, 1]


def base_inputs(seed, lengths=LENGTHS, H=2):
    g = gen.make_gen(seed)
    T = int(sum(lengths))
    return gen.token_inputs(T, H, torch.float32, g), g


@pytest.mark.parametrize("lo,hi", [(3.0, 8.0), (8.0, 40.0)])
def test_fast_forgetting_channels(lo, hi):
    """A few key channels decay by 3 to 40 nats per token: their log-decay over
    a chunk leaves the range of exp(-G)."""
    x, g = base_inputs(21)
    x["gk"] = strong_decay(x["gk"], g, [0, 5, 77, 127], lo, hi)
    run(x, LENGTHS, 2, seed=21)


def test_every_channel_decays_by_six():
    x, g = base_inputs(22)
    x["gk"] = torch.full_like(x["gk"], -6.0)
    run(x, LENGTHS, 2, init_kind="mixed", seed=22)


def test_mixed_batch_of_normal_and_strong_decay_sequences():
    """Strong decays on the second and fourth sequences only, and on one chunk
    in the middle of the first: ordinary and exact chunks in one launch."""
    lengths = [300, 260, 64, 129]
    x, g = base_inputs(23, lengths)
    cu = gen.cu_seqlens(lengths).tolist()
    rows = torch.cat([torch.arange(cu[1], cu[2]), torch.arange(cu[3], cu[4]),
                      torch.arange(cu[0] + 128, cu[0] + 192)])
    gk = x["gk"].clone()
    gk[rows] = strong_decay(x["gk"], g, list(range(0, 128, 3)), 4.0, 9.0)[rows]
    x["gk"] = gk
    run(x, lengths, 2, seed=23)


def test_in_place_resume_across_a_strong_decay_chunk():
    """init_slot == out_slot (the long workload's pattern): a chunk that takes
    the exact path in the middle of the sequence, resumed in place."""
    lengths = [256, 190]
    x, g = base_inputs(24, lengths)
    gk = x["gk"].clone()
    gk[64:128] = strong_decay(x["gk"], g, [3, 9, 100], 5.0, 7.0)[64:128]
    x["gk"] = gk
    run(x, lengths, 2, seed=24, inplace=True)


def test_positive_log_decay():
    """gk > 0 on a few channels (growth): outside the pages' log-decay <= 0 but
    inside the recurrence's domain."""
    x, g = base_inputs(25)
    gk = x["gk"].clone()
    gk[:, :, [1, 2]] = 0.02
    x["gk"] = gk
    run(x, LENGTHS, 2, seed=25)


def test_large_q_v_k_and_state():
    """Magnitudes far beyond the input recipe's: |q| x 400 and |v| x 70000; |k|
    above 256 with beta scaled down so that beta |k|^2 stays below 2 (the
    delta rule is stable only there); a checkpoint of 5e6."""
    x, _ = base_inputs(26)
    x["q"] = x["q"] * 400.0
    x["v"] = x["v"] * 7.0e4
    run(x, LENGTHS, 2, seed=26)
    x, _ = base_inputs(31)
    x["k"] = x["k"] * 300.0
    x["beta"] = x["beta"] * 1.0e-5
    run(x, LENGTHS, 2, seed=31)
    x, _ = base_inputs(27)
    run(x, LENGTHS, 2, seed=27, ck_scale=5.0e6)


def test_checkpoints_across_strong_decay_chunks():
    """Multi-checkpoint prefill through chunks that take the exact path: each
    checkpoint equals the final state of a prefill of that prefix, bit for bit."""
    lengths = [384, 300]
    H, interval = 2, 128
    x, g = base_inputs(28, lengths, H)
    gk = x["gk"].clone()
    gk[100:230] = strong_decay(x["gk"], g, [0, 64, 65], 6.0, 12.0)[100:230]
    x["gk"] = gk
    xd = {n: t.to(torch.bfloat16).to(DEV) for n, t in x.items()}
    N = len(lengths)
    cu = gen.cu_seqlens(lengths)
    cap = max(lengths) // interval
    pool = canary_fill(torch.empty(2 * N + N * cap, H, KD, VD, device=DEV))
    slots = torch.arange(2 * N, 2 * N + N * cap, dtype=torch.int32).view(N, cap).to(DEV)
    init = torch.full((N,), -1, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda().kda_chunk_prefill_checkpoints(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"], cu.to(DEV),
                                        cu, pool, init, torch.arange(N, 2 * N, dtype=torch.int32,
                                                                     device=DEV),
                                        interval, slots, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    offs = cu.tolist()
    for m in range(cap):
        keep = [min((m + 1) * interval, L) for L in lengths]
        idx = torch.cat([torch.arange(offs[n], offs[n] + keep[n]) for n in range(N)]).to(DEV)
        cu_m = gen.cu_seqlens(keep)
        ref = torch.zeros(2 * N, H, KD, VD, device=DEV)
        kda().kda_chunk_prefill(*(xd[k][idx].contiguous() for k in ("q", "k", "v", "gk", "beta")),
                                cu_m.to(DEV), cu_m, ref, init,
                                torch.arange(N, 2 * N, dtype=torch.int32, device=DEV))
        torch.cuda.synchronize()
        for n in range(N):
            if (m + 1) * interval <= lengths[n]:
                assert torch.equal(pool[slots[n, m].item()], ref[N + n]), "checkpoint %d of %d" % (m, n)


def test_prefill_bounded_wait_gives_up_cleanly():
    """The prefill's own wait loop, on a barrier nothing arrives at (the first
    chunk's q, k, gk are never requested): KDA_DEVERR_TIMEOUT is reported, no
    slot is written, the tensor memory is released, and the next launch is
    bit-identical to the same launch made before."""
    lengths = [130, 64, 5]
    H = 2
    x, _ = base_inputs(29, lengths, H)
    xd = {n: t.to(torch.bfloat16).to(DEV) for n, t in x.items()}
    N = len(lengths)
    cu = gen.cu_seqlens(lengths)
    cud = cu.to(DEV)
    init = torch.arange(N, dtype=torch.int32, device=DEV)
    out = torch.arange(N, 2 * N, dtype=torch.int32, device=DEV)
    pool = canary_fill(torch.empty(2 * N, H, KD, VD, device=DEV))
    pool[:N] = gen.checkpoint((N, H, KD, VD), gen.make_gen(30)).to(DEV)
    args = (xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"], cud, cu, pool, init, out)
    o1 = kda().kda_chunk_prefill(*args)
    torch.cuda.synchronize()
    first = pool[N:].clone()
    pool[N:] = canary_fill(torch.empty_like(pool[N:]))
    before = pool.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda().kda_selftest_prefill_wait(*args, dev_err=err, wait_us=2000)
    torch.cuda.synchronize()
    assert int(err.item()) & kda().KDA_DEVERR_TIMEOUT
    assert torch.equal(pool, before), "a unit that gave up wrote a slot"
    err.zero_()
    o2 = kda().kda_chunk_prefill(*args, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(pool[N:], first) and torch.equal(o1, o2), "the next launch differs"
