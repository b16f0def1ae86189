"""GPU parity of kda_chunk_prefill_checkpoints: the state after every
``interval`` tokens of each sequence, written from the prefill's own launch.

Checked against the oracle (within the dtype's tolerance) and against two
bit-exact contracts: checkpointing changes no output and no final state, and
checkpoint m is bit for bit the final state of a plain prefill of the
sequence's first (m + 1) * interval tokens.  Slots the call must not touch
keep a canary pattern."""
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


def _prefix(xd, lengths, keep):
    """Inputs of every sequence cut to its first keep[n] tokens, repacked."""
    offs = np.concatenate([[0], np.cumsum(lengths)])
    idx = torch.cat([torch.arange(offs[n], offs[n] + keep[n]) for n in range(len(lengths))]
                    + [torch.zeros(0, dtype=torch.long)]).to(DEV)
    return {n: t.index_select(0, idx).contiguous() for n, t in xd.items()}, gen.cu_seqlens(keep)


def _plain(xd, cu, pool, init, out):
    o = kda().kda_chunk_prefill(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"], cu.to(DEV), cu,
                                pool, init, out)
    return o


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("interval,cap", [(64, 4), (256, 3)], ids=["i64", "i256"])
def test_prefill_checkpoints_small(dtype, interval, cap):
    lengths = [1, 63, 64, 65, 256, 300, 0, 700, 512]
    H, N = 3, 9
    g = gen.make_gen(21)
    cu = gen.cu_seqlens(lengths)
    x = gen.token_inputs(int(cu[-1]), H, dtype, g)
    xd = _dev(x)
    ck0 = gen.checkpoint((N, H, KD, VD), g)
    init = [-1 if n % 2 == 0 else n for n in range(N)]
    init_d = torch.tensor(init, dtype=torch.int32, device=DEV)
    # slots: [0, N) initial checkpoints, [N, 2N) outputs, then N * cap checkpoint
    # slots (row-major by sequence), then one slot that nothing may write
    base = 2 * N
    slots = torch.arange(base, base + N * cap, dtype=torch.int32).view(N, cap)
    slots[5, 0] = -1                        # sequence 5 skips its first checkpoint
    pool = canary_fill(torch.empty(base + N * cap + 1, H, KD, VD, device=DEV))
    pool[:N] = ck0.to(DEV)
    before = pool.clone()
    out = torch.arange(N, 2 * N, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = kda().kda_chunk_prefill_checkpoints(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"],
                                            cu.to(DEV), cu, pool, init_d, out, interval,
                                            slots.to(DEV), dev_err=err)
    # the same call without checkpoints, on its own pool
    pool_p = before.clone()
    o_p = _plain(xd, cu, pool_p, init_d, out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(o, o_p), "checkpointing changed the outputs"
    assert torch.equal(pool[N:2 * N], pool_p[N:2 * N]), "checkpointing changed the final states"
    assert torch.equal(pool[:N], before[:N]), "initial checkpoints were written"
    assert torch.equal(pool[-1], before[-1]), "an unnamed slot was written"

    made = [min(L // interval, cap) for L in lengths]
    for n in range(N):
        for m in range(cap):
            s = int(slots[n, m])
            if s >= 0 and m >= made[n]:
                assert torch.equal(pool[s], before[s]), "checkpoint %d of seq %d not due" % (m, n)
    assert torch.equal(pool[int(base + 5 * cap)], before[int(base + 5 * cap)]), "-1 slot written"

    # bit-exact: checkpoint m == final state of a plain prefill of the prefix
    for m in range(cap):
        due = [n for n in range(N) if m < made[n] and int(slots[n, m]) >= 0]
        if not due:
            continue
        keep = [min(L, (m + 1) * interval) for L in lengths]
        xp, cup = _prefix(xd, lengths, keep)
        pool_q = before.clone()
        _plain(xp, cup, pool_q, init_d, out)
        torch.cuda.synchronize()
        for n in due:
            assert torch.equal(pool[int(slots[n, m])], pool_q[N + n]), (
                "checkpoint %d of sequence %d differs from the prefix's final state" % (m, n))

    # against the oracle
    S0 = np.stack([np.zeros((H, KD, VD)) if init[n] < 0 else f64(ck0[n]) for n in range(N)])
    o_ref, S_ref, ck_ref, made_ref = oracle.prefill_checkpoints(
        f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["gk"]), f64(x["beta"]), cu.numpy(), S0,
        interval, cap)
    assert list(made_ref) == made
    assert_close(o, o_ref, dtype, "o")
    assert_close(pool[N:2 * N], S_ref, dtype, "final states")
    for n in range(N):
        for m in range(made[n]):
            s = int(slots[n, m])
            if s >= 0:
                assert_close(pool[s], ck_ref[n, m], dtype, "checkpoint %d of sequence %d" % (m, n))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_prefill_checkpoints_bad_slot(dtype):
    """A checkpoint slot out of range that the sequence would use: the unit is
    skipped (its output slot keeps its canary) and KDA_DEVERR_SLOT_RANGE is
    set; an out-of-range entry past the checkpoints a sequence makes is never
    read, and the other sequences complete normally."""
    lengths = [300, 100, 130]
    H, N, I = 2, 3, 128
    g = gen.make_gen(22)
    cu = gen.cu_seqlens(lengths)
    x = gen.token_inputs(int(cu[-1]), H, dtype, g)
    xd = _dev(x)
    num_slots = 8
    pool = canary_fill(torch.empty(num_slots, H, KD, VD, device=DEV))
    before = pool.clone()
    slots = torch.tensor([[5, num_slots + 3],      # sequence 0 makes 2: the second is bad
                          [-1, 1 << 20],           # sequence 1 makes none: never read
                          [6, 7 << 20]], dtype=torch.int32)   # sequence 2 makes 1
    init = torch.full((N,), -1, dtype=torch.int32, device=DEV)
    out = torch.tensor([0, 1, 2], dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda().kda_chunk_prefill_checkpoints(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"],
                                        cu.to(DEV), cu, pool, init, out, I, slots.to(DEV),
                                        dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kda().KDA_DEVERR_SLOT_RANGE
    assert torch.equal(pool[0], before[0]) and torch.equal(pool[5], before[5])
    _, S_ref, ck_ref, _ = oracle.prefill_checkpoints(
        f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["gk"]), f64(x["beta"]), cu.numpy(),
        np.zeros((N, H, KD, VD)), I, 2)
    assert_close(pool[1:3], S_ref[1:3], dtype, "final states")
    assert_close(pool[6], ck_ref[2, 0], dtype, "checkpoint")
    assert torch.equal(pool[7], before[7]) and torch.equal(pool[3:5], before[3:5])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_prefill_checkpoints_none_due(dtype):
    """An interval longer than every sequence makes no checkpoint: the call
    equals the plain prefill and leaves every checkpoint slot untouched."""
    lengths = [100, 0, 255]
    H, N = 2, 3
    g = gen.make_gen(23)
    cu = gen.cu_seqlens(lengths)
    x = gen.token_inputs(int(cu[-1]), H, dtype, g)
    xd = _dev(x)
    pool = canary_fill(torch.empty(2 * N + 2, H, KD, VD, device=DEV))
    before = pool.clone()
    init = torch.full((N,), -1, dtype=torch.int32, device=DEV)
    out = torch.arange(N, 2 * N, dtype=torch.int32, device=DEV)
    slots = torch.tensor([[6, 7]] * N, dtype=torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = kda().kda_chunk_prefill_checkpoints(xd["q"], xd["k"], xd["v"], xd["gk"], xd["beta"],
                                            cu.to(DEV), cu, pool, init, out, 256, slots.to(DEV),
                                            dev_err=err)
    pool_p = before.clone()
    o_p = _plain(xd, cu, pool_p, init, out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(o, o_p) and torch.equal(pool, pool_p)
    assert torch.equal(pool[6:], before[6:])
