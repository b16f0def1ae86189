"""Pins for the oracle of the prologue / epilogue around the recurrence
(oracle/fused_ops.py): each checks the oracle against something other than
itself -- numpy's convolution, closed forms, invariants, split-call
continuity, and a brute-force composition for the fused decode."""
import importlib.util

import numpy as np
import pytest

import oracle
from oracle import fused_ops

W = fused_ops.CONV_W


def _rng(seed):
    return np.random.default_rng(seed)


def _raw(rng, T, H, K):
    return [rng.standard_normal((T, H, K)) for _ in range(3)], rng.standard_normal((T, H))


def pin_conv_matches_numpy_convolve(fo):
    """The v stream (no norm) is silu(np.convolve(state ++ x, reversed taps))
    per channel; q and k are the same, L2-normalised per (token, head)."""
    rng = _rng(1)
    T, H, K, S = 9, 2, 5, 3
    (q, k, v), b = _raw(rng, T, H, K)
    w = rng.standard_normal((3, H, K, W))
    cs = rng.standard_normal((S, W - 1, 3, H, K))
    cu = [0, T]
    qo, ko, vo, beta, _ = fo.conv_prologue(q, k, v, b, w, cs, cu, [2], [-1])
    for s, (x, out) in enumerate([(q, qo), (k, ko), (v, vo)]):
        ref = np.zeros((T, H, K))
        for h in range(H):
            for c in range(K):
                full = np.concatenate([cs[2, :, s, h, c], x[:, h, c]])
                y = np.convolve(full, w[s, h, c, ::-1], mode="valid")
                ref[:, h, c] = y / (1 + np.exp(-y))
        if s < 2:
            ref = ref / np.sqrt(np.sum(ref * ref, axis=-1, keepdims=True) + 1e-6)
        np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(beta, 1 / (1 + np.exp(-b)), rtol=1e-15)


def pin_conv_state_update_and_zero_start(fo):
    """After a sequence the slot holds its last W-1 raw inputs (older ones from
    the previous state when it is shorter); init -1 starts from zeros, out -1
    writes nothing, and an empty sequence copies the state across."""
    rng = _rng(2)
    H, K, S = 1, 3, 6
    lens = [5, 1, 0, 2]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    (q, k, v), b = _raw(rng, T, H, K)
    w = rng.standard_normal((3, H, K, W))
    cs = rng.standard_normal((S, W - 1, 3, H, K))
    init, out = [-1, 1, 2, 3], [4, 1, 5, -1]
    *_, cs2 = fo.conv_prologue(q, k, v, b, w, cs, cu, init, out)
    raws = [q, k, v]
    for s in range(3):
        np.testing.assert_array_equal(cs2[4, :, s], raws[s][cu[0] + 2:cu[1]])       # 5 >= W-1
        np.testing.assert_array_equal(cs2[1, :, s], np.concatenate([cs[1, 1:, s], raws[s][cu[1]:cu[2]]]))
        np.testing.assert_array_equal(cs2[5, :, s], cs[2, :, s])                   # empty sequence
    np.testing.assert_array_equal(cs2[[0, 2, 3]], cs[[0, 2, 3]])                   # untouched
    # a zero start equals a state of zeros
    cz = np.zeros_like(cs)
    a = fo.conv_prologue(q, k, v, b, w, cs, cu, [-1, -1, -1, -1], [-1] * 4)
    z = fo.conv_prologue(q, k, v, b, w, cz, cu, [0, 0, 0, 0], [-1] * 4)
    for x, y in zip(a[:3], z[:3]):
        np.testing.assert_array_equal(x, y)


def pin_conv_split_calls_continue(fo):
    """Running a sequence in two calls, the second starting from the conv state
    the first left, gives the outputs of one call."""
    rng = _rng(3)
    T, H, K = 11, 2, 4
    (q, k, v), b = _raw(rng, T, H, K)
    w = rng.standard_normal((3, H, K, W))
    cs = rng.standard_normal((2, W - 1, 3, H, K))
    whole = fo.conv_prologue(q, k, v, b, w, cs, [0, T], [0], [1])
    for cut in (1, 2, 5):
        a = fo.conv_prologue(q[:cut], k[:cut], v[:cut], b[:cut], w, cs, [0, cut], [0], [1])
        bb = fo.conv_prologue(q[cut:], k[cut:], v[cut:], b[cut:], w, a[4], [0, T - cut], [1], [1])
        for i in range(4):
            np.testing.assert_allclose(np.concatenate([a[i], bb[i]]), whole[i], rtol=1e-14,
                                       atol=1e-15)
        np.testing.assert_array_equal(bb[4][1], whole[4][1])


def pin_norm_closed_forms(fo):
    """L2 norm: |x| = sqrt(ss / (ss + eps)).  Gated RMSNorm: with w = 1 and a
    saturated gate the output's mean square is ms / (ms + eps); it is
    scale-invariant at eps = 0; a zero gate halves it; w scales it per channel."""
    rng = _rng(4)
    x = rng.standard_normal((6, 3, 128))
    ss = np.sum(x * x, axis=-1)
    np.testing.assert_allclose(np.linalg.norm(fo.l2norm(x, 1e-6), axis=-1), np.sqrt(ss / (ss + 1e-6)),
                               rtol=1e-14)
    one = np.ones(128)
    big = np.full(x.shape, 60.0)
    out = fo.gated_rmsnorm(x, big, one, 1e-5)
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.mean(out * out, axis=-1), ms / (ms + 1e-5), rtol=1e-12)
    np.testing.assert_allclose(fo.gated_rmsnorm(7.5 * x, big, one, 0.0), fo.gated_rmsnorm(x, big, one, 0.0),
                               rtol=1e-13)
    np.testing.assert_allclose(fo.gated_rmsnorm(x, np.zeros(x.shape), one, 0.0),
                               0.5 * fo.gated_rmsnorm(x, big, one, 0.0), rtol=1e-13)
    wv = rng.uniform(0.5, 2.0, 128)
    np.testing.assert_allclose(fo.gated_rmsnorm(x, big, wv, 1e-5), wv * out, rtol=1e-13)
    assert fo.sigmoid(0.0) == 0.5 and abs(fo.silu(0.0)) == 0.0


def pin_decode_fused_brute_force(fo):
    """conv + KDA + onorm for one token per request, written out with explicit
    matrices: conv + SiLU, L2 norm, beta sigmoid, S = (I - b k k^T) Diag(e^g) S
    + b k v^T, o = S^T (scale q), then the gated RMSNorm; the pool changes only
    at the requests' slots and the conv state shifts in the new input."""
    rng = _rng(5)
    B, H, K, S = 3, 2, 128, 5
    q, k, v = (rng.standard_normal((B, H, K)) for _ in range(3))
    b = rng.standard_normal((B, H))
    gk = -np.log1p(np.exp(rng.standard_normal((B, H, K))))
    g = rng.standard_normal((B, H, K))
    w = rng.standard_normal((3, H, K, W)) * 0.5
    wn = rng.uniform(0.5, 1.5, K)
    cs = rng.standard_normal((S, W - 1, 3, H, K))
    pool = 0.02 * rng.standard_normal((S, H, K, K))
    ids = [3, 0, 4]
    out, pool2, cs2 = fo.decode_fused(q, k, v, gk, b, w, cs, g, wn, ids, pool, scale=0.3)
    for i, s in enumerate(ids):
        for h in range(H):
            ys = []
            for st, x in enumerate((q, k, v)):
                window = np.concatenate([cs[s, :, st, h], x[i, h][None]], axis=0)   # [W, K]
                y = np.sum(w[st, h] * window.T, axis=1)
                ys.append(y * (1 / (1 + np.exp(-y))))
            qq = ys[0] / np.sqrt(ys[0] @ ys[0] + 1e-6)
            kk = ys[1] / np.sqrt(ys[1] @ ys[1] + 1e-6)
            bb = 1 / (1 + np.exp(-b[i, h]))
            M = (np.eye(K) - bb * np.outer(kk, kk)) @ np.diag(np.exp(gk[i, h])) @ pool[s, h]
            Sn = M + bb * np.outer(kk, ys[2])
            o = Sn.T @ (0.3 * qq)
            ref = wn * o / np.sqrt(np.mean(o * o) + 1e-5) / (1 + np.exp(-g[i, h]))
            np.testing.assert_allclose(out[i, h], ref, rtol=1e-9, atol=1e-12)
            np.testing.assert_allclose(pool2[s, h], Sn, rtol=1e-10, atol=1e-14)
        for st, x in enumerate((q, k, v)):
            np.testing.assert_array_equal(cs2[s, :, st], np.concatenate([cs[s, 1:, st], x[i][None]]))
    other = [s for s in range(S) if s not in ids]
    np.testing.assert_array_equal(pool2[other], pool[other])
    np.testing.assert_array_equal(cs2[other], cs[other])


def pin_round_bf16_matches_library_cast(fo):
    """round_bf16 equals torch's float64 -> float32 -> bfloat16 cast, on random
    values, exact bf16 values, and the float32 midpoints between neighbours
    (ties go to the even neighbour)."""
    import torch
    rng = _rng(6)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-6, 6, 4000),
                        [0.0, -0.0, 1.0, -2.5, 3.0e38, 1.0e-40]])
    bf = torch.tensor(x).to(torch.float32).to(torch.bfloat16)
    lo = bf.to(torch.float32).numpy().view(np.uint32)
    mids = ((lo.astype(np.uint64) << 16 >> 16) | 0x8000).astype(np.uint32).view(np.float32)
    for v in (x, mids.astype(np.float64)):
        ref = torch.tensor(v).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
        np.testing.assert_array_equal(fo.round_bf16(v), ref)


def pin_store_rounds_every_intermediate(fo):
    """With store = round_bf16 the prologue's outputs are bf16 values, q and k
    are the rounded L2 norm of the rounded conv outputs, and the fused decode
    normalises the rounded o."""
    rng = _rng(7)
    T, H, K = 6, 2, 128
    (q, k, v), b = _raw(rng, T, H, K)
    w = 0.5 * rng.standard_normal((3, H, K, W))
    cs = rng.standard_normal((1, W - 1, 3, H, K))
    r = fo.round_bf16
    out = fo.conv_prologue(q, k, v, b, w, cs, [0, T], [0], [-1], store=r)
    plain = fo.conv_prologue(q, k, v, b, w, cs, [0, T], [0], [-1])
    for a in out[:4]:
        np.testing.assert_array_equal(r(a), a)
    np.testing.assert_array_equal(out[2], r(plain[2]))
    np.testing.assert_array_equal(out[3], r(plain[3]))
    y = plain[2] * 0   # recompute the conv outputs of q from the definition, rounded
    for t in range(T):
        win = np.concatenate([cs[0, :, 0], q[:t + 1]], axis=0)[t:t + W]
        y[t] = r(fo.silu(np.einsum("hki,ihk->hk", w[0], win)))
    np.testing.assert_array_equal(out[0], r(fo.l2norm(y)))
    # the fused decode norms the stored (rounded) o of the recurrence
    B = 3
    gk = -np.log1p(np.exp(rng.standard_normal((B, H, K))))
    gate = rng.standard_normal((B, H, K))
    wn = np.ones(K)
    pool = 0.02 * rng.standard_normal((4, H, K, K))
    cs4 = rng.standard_normal((4, W - 1, 3, H, K))
    ids = [2, 0, 3]
    got, _, _ = fo.decode_fused(q[:B], k[:B], v[:B], gk, b[:B], w, cs4, gate, wn, ids, pool,
                                store=r)
    pq, pk, pv, pb, _ = fo.conv_prologue(q[:B], k[:B], v[:B], b[:B], w, cs4, np.arange(B + 1), ids,
                                         ids, store=r)
    o, _ = oracle.decode(pq, pk, pv, gk, pb, pool[ids])
    np.testing.assert_array_equal(got, fo.gated_rmsnorm(r(o), gate, wn))
    assert not np.array_equal(got, fo.gated_rmsnorm(o, gate, wn))


PINS = [pin_conv_matches_numpy_convolve, pin_conv_state_update_and_zero_start,
        pin_conv_split_calls_continue, pin_norm_closed_forms, pin_decode_fused_brute_force,
        pin_round_bf16_matches_library_cast, pin_store_rounds_every_intermediate]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(fused_ops)


# planted mistakes: each mutant copy of oracle/fused_ops.py must fail a pin
MUTANTS = {
    "taps_reversed": ('np.einsum("hki,ihk->hk", w[s], x[t:t + CONV_W])',
                      'np.einsum("hki,ihk->hk", w[s][..., ::-1], x[t:t + CONV_W])'),
    "window_off_by_one": ("x[t:t + CONV_W]", "x[t + 1:t + 1 + CONV_W] if t + 1 + CONV_W <= x.shape[0] else x[t:t + CONV_W]"),
    "silu_dropped": ("outs[s][lo + t] = store(silu(y))", "outs[s][lo + t] = store(y)"),
    "round_truncates": ("r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16", "r = (u >> 16) << 16"),
    "round_ties_up": ("r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16", "r = ((u + 0x8000) >> 16) << 16"),
    "o_not_stored": ("return gated_rmsnorm(store(o), gate", "return gated_rmsnorm(o, gate"),
    "state_not_shifted": ("cs[so, :, s] = x[x.shape[0] - (CONV_W - 1):]", "cs[so, :, s] = x[:CONV_W - 1]"),
    "l2_eps_outside": ("return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)",
                       "return x / (np.sqrt(np.sum(x * x, axis=-1, keepdims=True)) + eps)"),
    "rms_sum_not_mean": ("np.mean(o * o, axis=-1, keepdims=True)", "np.sum(o * o, axis=-1, keepdims=True)"),
    "gate_silu": ("return _f64(w_norm) * o * r * sigmoid(_f64(g))",
                  "return _f64(w_norm) * o * r * silu(_f64(g))"),
    "beta_raw": ("return q, k, outs[2], store(sigmoid(_f64(b_raw))), cs",
                 "return q, k, outs[2], store(_f64(b_raw)), cs"),
    "v_normalised": ("return q, k, outs[2], store(sigmoid", "return q, k, l2norm(outs[2], eps_l2), store(sigmoid"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_fused_pins_catch_planted_mistakes(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(fused_ops.__file__).read()
    assert old in src, "mutation anchor not found: %s" % name
    path = tmp_path / ("mut_%s.py" % name)
    path.write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location("mut_%s" % name, str(path))
    mut = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mut)
    failed = []
    for pin in PINS:
        try:
            pin(mut)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "planted mistake %s passed every pin" % name
