"""Pins for the oracle: checks against facts other than the oracle itself.

Each pin is a closed form, an invariant the recurrence must satisfy, a brute
force on tiny inputs, or an agreement between two independently written forms
(sequential vs chunked).  Small odd dimensions (K != V) are used wherever a
transposed operand or a row/column mix-up could otherwise hide.

The pins are written as ``pin_*(orc)`` functions of an oracle namespace so that
``test_pins_catch_planted_mistakes`` can run them against copies of the oracle
source with a mistake planted in them.
"""
import os
import shutil

import numpy as np
import pytest

import oracle

pytestmark = []


def _rng(seed):
    return np.random.default_rng(seed)


def _unit_vecs(rng, n, d):
    x = rng.standard_normal((n, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def _inputs(rng, T, K, V, gk_scale=1.0):
    q = _unit_vecs(rng, T, K)
    k = _unit_vecs(rng, T, K)
    v = rng.standard_normal((T, V))
    gk = -np.log1p(np.exp(gk_scale * rng.standard_normal((T, K))))   # -softplus
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))               # sigmoid
    return q, k, v, gk, beta


# --------------------------------------------------------------------------
# pins (each raises AssertionError when violated)
# --------------------------------------------------------------------------

def pin_single_token_closed_form(orc):
    """S0 = 0, one token: S1 = beta k v^T and o1 = scale beta (k.q) v."""
    rng = _rng(1)
    K, V, scale = 5, 3, 0.7
    q, k, v, gk, beta = _inputs(rng, 1, K, V)
    o, S = orc.unit(q, k, v, gk, beta, np.zeros((K, V)), scale=scale)
    np.testing.assert_allclose(S, beta[0] * np.outer(k[0], v[0]), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(o[0], scale * beta[0] * np.dot(k[0], q[0]) * v[0], rtol=1e-13,
                               atol=1e-15)


def pin_identity_when_no_write_no_decay(orc):
    """beta = 0, gk = 0: the state is unchanged exactly and o_t = scale S0^T q_t."""
    rng = _rng(2)
    T, K, V, scale = 6, 5, 3, 1.3
    q, k, v, _, _ = _inputs(rng, T, K, V)
    S0 = rng.standard_normal((K, V))
    o, S = orc.unit(q, k, v, np.zeros((T, K)), np.zeros(T), S0, scale=scale)
    assert np.array_equal(S, S0)
    np.testing.assert_allclose(o, scale * q @ S0, rtol=1e-13, atol=1e-14)


def pin_pure_decay_closed_form(orc):
    """beta = 0, gk_t = g for every t: S_T = Diag(exp(T g)) S0 (rows = key channels,
    natural exponential)."""
    rng = _rng(3)
    T, K, V = 7, 5, 3
    q, k, v, _, _ = _inputs(rng, T, K, V)
    g = -rng.uniform(0.05, 0.9, K)
    S0 = rng.standard_normal((K, V))
    _, S = orc.unit(q, k, v, np.tile(g, (T, 1)), np.zeros(T), S0)
    np.testing.assert_allclose(S, np.exp(T * g)[:, None] * S0, rtol=1e-12, atol=1e-15)


def pin_write_exactness(orc):
    """beta = 1, |k| = 1: the updated state reads back v at key k (S_t^T k_t = v_t)
    for any decay and any previous state, so q_t = k_t gives o_t = scale v_t."""
    rng = _rng(4)
    T, K, V, scale = 5, 6, 4, 0.5
    _, k, v, gk, _ = _inputs(rng, T, K, V)
    S0 = rng.standard_normal((K, V))
    o, _ = orc.unit(k, k, v, gk, np.ones(T), S0, scale=scale)
    np.testing.assert_allclose(o, scale * v, rtol=1e-12, atol=1e-12)


def pin_delta_rule_geometry(orc):
    """One token, |k| = 1: for x orthogonal to k the read-out is the decayed old
    one, x^T S_1 = x^T Diag(alpha) S0, and at k it moves a fraction beta toward v,
    k^T S_1 = (1 - beta) k^T Diag(alpha) S0 + beta v^T.  These two facts fix S_1."""
    rng = _rng(5)
    K, V = 6, 4
    q, k, v, gk, beta = _inputs(rng, 1, K, V)
    S0 = rng.standard_normal((K, V))
    _, S1 = orc.unit(q, k, v, gk, beta, S0)
    M = np.exp(gk[0])[:, None] * S0
    basis = np.linalg.qr(np.column_stack([k[0], rng.standard_normal((K, K - 1))]))[0]
    for c in range(1, K):
        x = basis[:, c]
        np.testing.assert_allclose(x @ S1, x @ M, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(k[0] @ S1, (1 - beta[0]) * (k[0] @ M) + beta[0] * v[0], rtol=1e-11,
                               atol=1e-12)


def pin_affine_in_initial_state(orc):
    """S_T and o are affine in S0: f(aX + bY) = a f(X) + b f(Y) when a + b = 1."""
    rng = _rng(6)
    T, K, V = 9, 5, 4
    q, k, v, gk, beta = _inputs(rng, T, K, V)
    X, Y = rng.standard_normal((K, V)), rng.standard_normal((K, V))
    a, b = 1.7, -0.7
    oX, SX = orc.unit(q, k, v, gk, beta, X)
    oY, SY = orc.unit(q, k, v, gk, beta, Y)
    oZ, SZ = orc.unit(q, k, v, gk, beta, a * X + b * Y)
    np.testing.assert_allclose(SZ, a * SX + b * SY, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(oZ, a * oX + b * oY, rtol=1e-11, atol=1e-12)


def pin_brute_force_tiny(orc):
    """T <= 8, K = 4, V = 3: explicit matrix products of the definition
    S_t = (I - beta k k^T) Diag(exp(gk)) S_{t-1} + beta k v^T, o_t = S_t^T (scale q)."""
    rng = _rng(7)
    T, K, V, scale = 8, 4, 3, 0.9
    q, k, v, gk, beta = _inputs(rng, T, K, V)
    k = k * rng.uniform(0.5, 1.5, (T, 1))    # non-unit keys as well
    S0 = rng.standard_normal((K, V))
    o, S = orc.unit(q, k, v, gk, beta, S0, scale=scale)
    Sref = S0.copy()
    for t in range(T):
        P = np.eye(K) - beta[t] * np.outer(k[t], k[t])
        Sref = P @ np.diag(np.exp(gk[t])) @ Sref + beta[t] * np.outer(k[t], v[t])
        np.testing.assert_allclose(o[t], Sref.T @ (scale * q[t]), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S, Sref, rtol=1e-12, atol=1e-13)


def pin_split_resume(orc):
    """Running T1 tokens, then T2 tokens from the saved state, equals running
    T1 + T2 tokens at once (bit-exact in the sequential form)."""
    rng = _rng(8)
    T, K, V = 23, 8, 6
    q, k, v, gk, beta = _inputs(rng, T, K, V)
    S0 = 0.02 * rng.standard_normal((K, V))
    o, S = orc.unit(q, k, v, gk, beta, S0)
    for cut in (1, 8, 16, 22):
        o1, S1 = orc.unit(q[:cut], k[:cut], v[:cut], gk[:cut], beta[:cut], S0)
        o2, S2 = orc.unit(q[cut:], k[cut:], v[cut:], gk[cut:], beta[cut:], S1)
        assert np.array_equal(S2, S)
        assert np.array_equal(np.concatenate([o1, o2]), o)


def pin_chunked_equals_sequential(orc):
    """The chunked (UT) form equals the sequential form for several chunk sizes,
    T not a multiple of the chunk, at K = V = 128 and at small odd sizes."""
    for seed, (T, K, V) in enumerate([(70, 128, 128), (45, 7, 5)]):
        rng = _rng(20 + seed)
        q, k, v, gk, beta = _inputs(rng, T, K, V)
        S0 = 0.02 * rng.standard_normal((K, V))
        o, S = orc.unit(q, k, v, gk, beta, S0, scale=0.8)
        for C in (16, 32, 64):
            oc, Sc = orc.unit(q, k, v, gk, beta, S0, scale=0.8, chunk=C)
            assert np.abs(oc - o).max() <= 1e-12 * max(1.0, np.abs(o).max())
            assert np.abs(Sc - S).max() <= 1e-12 * max(1.0, np.abs(S).max())


def pin_fold_is_prefix_commit(orc):
    """Verify leaves the committed state untouched and its outputs are those of
    the recurrence over the draft; the fold of an accepted prefix a equals
    committing the first a tokens (bit-exact); a = 0 is a no-op."""
    rng = _rng(9)
    B, G, H, K, V = 3, 5, 2, 6, 4
    q = rng.standard_normal((B, G, H, K))
    k = rng.standard_normal((B, G, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, G, H, V))
    gk = -np.log1p(np.exp(rng.standard_normal((B, G, H, K))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, G, H))))
    S0 = rng.standard_normal((B, H, K, V))
    S0_copy = S0.copy()
    o = orc.verify(q, k, v, gk, beta, S0, scale=1.0)
    assert np.array_equal(S0, S0_copy)
    accept = np.array([0, 2, G])
    Sf = orc.fold(k, v, gk, beta, accept, S0)
    for b in range(B):
        for h in range(H):
            ou, _ = orc.unit(q[b, :, h], k[b, :, h], v[b, :, h], gk[b, :, h], beta[b, :, h], S0[b, h])
            np.testing.assert_allclose(o[b, :, h], ou, rtol=1e-13, atol=1e-14)
            a = accept[b]
            _, Sa = orc.unit(q[b, :a, h], k[b, :a, h], v[b, :a, h], gk[b, :a, h], beta[b, :a, h],
                             S0[b, h])
            assert np.array_equal(Sf[b, h], Sa)


def pin_batches_equal_units(orc):
    """The packed varlen / decode drivers equal per-unit runs (bit-exact): pins
    the token offsets, head strides and per-unit state bookkeeping."""
    rng = _rng(10)
    H, K, V = 3, 6, 5
    lens = [3, 1, 7]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = cu[-1]
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    v = rng.standard_normal((T, H, V))
    gk = -rng.uniform(0, 1, (T, H, K))
    beta = rng.uniform(0, 1, (T, H))
    S0 = rng.standard_normal((len(lens), H, K, V))
    o, S = orc.prefill_varlen(q, k, v, gk, beta, cu, S0, scale=0.6)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        for h in range(H):
            ou, Su = orc.unit(q[sl, h], k[sl, h], v[sl, h], gk[sl, h], beta[sl, h], S0[n, h], scale=0.6)
            assert np.array_equal(o[sl, h], ou)
            assert np.array_equal(S[n, h], Su)
    od, Sd = orc.decode(q[:2], k[:2], v[:2], gk[:2], beta[:2], S0[:2], scale=0.6)
    for b in range(2):
        for h in range(H):
            ou, Su = orc.unit(q[b:b + 1, h], k[b:b + 1, h], v[b:b + 1, h], gk[b:b + 1, h],
                              beta[b:b + 1, h], S0[b, h], scale=0.6)
            assert np.array_equal(od[b, h], ou[0])
            assert np.array_equal(Sd[b, h], Su)


def pin_checkpoints_are_prefix_states(orc):
    """Checkpoint m of a sequence is the state after its first (m + 1) * I
    tokens: written out as a brute-force product of the definition's per-token
    matrices on tiny sizes, for sequences that end on, before and between
    boundaries, with a cap on the number kept; the outputs and final states
    are those of the plain varlen run."""
    rng = _rng(13)
    H, K, V, I, cap = 2, 4, 3, 4, 2
    lens = [9, 3, 8, 12, 0]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    v = rng.standard_normal((T, H, V))
    gk = -rng.uniform(0, 1, (T, H, K))
    beta = rng.uniform(0, 1, (T, H))
    S0 = rng.standard_normal((len(lens), H, K, V))
    o, S, ck, made = orc.prefill_checkpoints(q, k, v, gk, beta, cu, S0, I, cap, scale=0.6)
    assert list(made) == [2, 0, 2, 2, 0]
    for n, L in enumerate(lens):
        for h in range(H):
            St = S0[n, h].copy()
            kept = []
            for t in range(cu[n], cu[n + 1]):
                P = np.eye(K) - beta[t, h] * np.outer(k[t, h], k[t, h])
                St = P @ np.diag(np.exp(gk[t, h])) @ St + beta[t, h] * np.outer(k[t, h], v[t, h])
                if (t - cu[n] + 1) % I == 0:
                    kept.append(St.copy())
            for m in range(cap):
                want = kept[m] if m < len(kept) else np.zeros((K, V))
                np.testing.assert_allclose(ck[n, m, h], want, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(S[n, h], St, rtol=1e-12, atol=1e-13)
    o2, S2 = orc.prefill_varlen(q, k, v, gk, beta, cu, S0, scale=0.6)
    assert np.array_equal(o, o2) and np.array_equal(S, S2)


def pin_ragged_verify_is_per_request_verify(orc):
    """Ragged verify: request b's outputs are those of the recurrence over its
    own G_b tokens from its committed state (brute-force matrix products of the
    definition), rows of no request stay zero, the committed states are not
    modified, and equal counts reproduce the uniform verify exactly."""
    rng = _rng(14)
    H, K, V, Gb = 2, 5, 4, [3, 0, 1, 4]
    cu = np.concatenate([[1], 1 + np.cumsum(Gb)])      # token 0 belongs to no request
    T = int(cu[-1]) + 4                                 # nor do the last four
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    v = rng.standard_normal((T, H, V))
    gk = -rng.uniform(0, 1, (T, H, K))
    beta = rng.uniform(0, 1, (T, H))
    S0 = rng.standard_normal((len(Gb), H, K, V))
    S0_copy = S0.copy()
    o = orc.verify_ragged(q, k, v, gk, beta, cu, S0, scale=0.7)
    assert np.array_equal(S0, S0_copy)
    assert not o[0].any() and not o[-1].any()
    for b in range(len(Gb)):
        for h in range(H):
            St = S0[b, h].copy()
            for t in range(cu[b], cu[b + 1]):
                P = np.eye(K) - beta[t, h] * np.outer(k[t, h], k[t, h])
                St = P @ np.diag(np.exp(gk[t, h])) @ St + beta[t, h] * np.outer(k[t, h], v[t, h])
                np.testing.assert_allclose(o[t, h], St.T @ (0.7 * q[t, h]), rtol=1e-12, atol=1e-13)
    G = 3
    assert len(Gb) * G <= T
    cu_u = np.arange(len(Gb) + 1) * G
    sl = slice(0, len(Gb) * G)
    ou = orc.verify_ragged(q[sl], k[sl], v[sl], gk[sl], beta[sl], cu_u, S0, scale=0.7)
    shp = lambda x: x[sl].reshape((len(Gb), G) + x.shape[1:])
    ov = orc.verify(shp(q), shp(k), shp(v), shp(gk), shp(beta), S0, scale=0.7)
    assert np.array_equal(ou, ov.reshape(ou.shape))


PINS = [
    pin_single_token_closed_form,
    pin_identity_when_no_write_no_decay,
    pin_pure_decay_closed_form,
    pin_write_exactness,
    pin_delta_rule_geometry,
    pin_affine_in_initial_state,
    pin_brute_force_tiny,
    pin_split_resume,
    pin_chunked_equals_sequential,
    pin_fold_is_prefix_commit,
    pin_batches_equal_units,
    pin_checkpoints_are_prefix_states,
    pin_ragged_verify_is_per_request_verify,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oracle)


def test_chunked_extreme_decay():
    """Strong decays (cumulative log-decay far below fp32 range over one chunk):
    the chunked form still equals the sequential one."""
    rng = _rng(11)
    T, K, V = 40, 16, 8
    q, k, v, gk, beta = _inputs(rng, T, K, V, gk_scale=4.0)
    gk = gk * 6.0
    S0 = rng.standard_normal((K, V))
    o, S = oracle.unit(q, k, v, gk, beta, S0)
    oc, Sc = oracle.unit(q, k, v, gk, beta, S0, chunk=32)
    assert np.abs(oc - o).max() <= 1e-11 * max(1.0, np.abs(o).max())
    assert np.abs(Sc - S).max() <= 1e-11 * max(1.0, np.abs(S).max())


def test_empty_units():
    """A zero-length sequence leaves its state unchanged and writes nothing."""
    rng = _rng(12)
    H, K, V = 2, 4, 4
    cu = np.array([0, 0, 3, 3])
    q = rng.standard_normal((3, H, K))
    S0 = rng.standard_normal((3, H, K, V))
    o, S = oracle.prefill_varlen(q, q, rng.standard_normal((3, H, V)), -np.ones((3, H, K)),
                                 np.ones((3, H)), cu, S0)
    assert np.array_equal(S[0], S0[0]) and np.array_equal(S[2], S0[2])


# --------------------------------------------------------------------------
# planted mistakes: each mutant copy of the oracle source must fail a pin
# --------------------------------------------------------------------------

MUTANTS = {
    "decay_dropped": ("double a = exp(gk[i]);", "double a = 1.0;"),
    "decay_base2": ("double a = exp(gk[i]);", "double a = exp2(gk[i]);"),
    "decay_on_columns": ("M[(size_t)i * V + j] = a * S[(size_t)i * V + j];",
                         "M[(size_t)i * V + j] = exp(gk[j % K]) * S[(size_t)i * V + j];"),
    "delta_sign_flipped": ("- beta * k[i] * kM[j]", "+ beta * k[i] * kM[j]"),
    "correction_undecayed": ("kM[j] += k[i] * M[(size_t)i * V + j];",
                             "kM[j] += k[i] * S[(size_t)i * V + j];"),
    "beta_dropped_on_write": ("+ beta * k[i] * v[j];", "+ k[i] * v[j];"),
    "scale_dropped": ("double sq = scale * q[i];", "double sq = q[i];"),
    "readout_transposed": ("o[j] += S[(size_t)i * V + j] * sq;",
                           "o[j] += S[(size_t)(j % K) * V + (i % V)] * scale * q[j % K];"),
    "readout_pre_update": ("    if (o) {\n        /* o = S^T (scale q) */",
                           "    if (o) {\n        for (int i = 0; i < K; ++i) for (int j = 0; j < V; ++j)"
                           " S[(size_t)i * V + j] = M[(size_t)i * V + j];\n        /* o = S^T (scale q) */"),
}


# mistakes in the packed-batch bookkeeping of the C source (every access stays
# in bounds, so a mutant fails a pin instead of crashing the test process)
MUTANTS.update({
    "batch_beta_token_stride": ("long sk = (long)J->H * J->K, sv = (long)J->H * J->V, sb = J->H;",
                                "long sk = (long)J->H * J->K, sv = (long)J->H * J->V, sb = 1;"),
    "batch_output_head_offset_dropped": ("double *o = J->o ? J->o + t0 * sv + (long)h * J->V : NULL;",
                                         "double *o = J->o ? J->o + t0 * sv : NULL;"),
    "batch_states_reversed": ("double *S = J->S + (size_t)u * J->K * J->V;",
                              "double *S = J->S + (size_t)(J->n_units - 1 - u) * J->K * J->V;"),
    "batch_gate_from_key": ("const double *gk = J->gk + t0 * sk + (long)h * J->K;",
                            "const double *gk = J->k + t0 * sk + (long)h * J->K;"),
})

# mistakes in the Python drivers (oracle/__init__.py), run against the same
# C library
PY_MUTANTS = {
    "fold_one_record_too_many": ("    Tn = np.repeat(acc, H)\n",
                                 "    Tn = np.repeat(np.minimum(acc + 1, G), H)\n"),
    "verify_writes_committed_state": (
        "    S = _f64(S0).reshape(B * H, *S0.shape[2:]).copy()   # scratch copy: S0 untouched\n"
        "    tok0 = np.repeat(np.arange(B) * G, H)",
        "    S = _f64(S0).reshape(B * H, *S0.shape[2:])\n"
        "    tok0 = np.repeat(np.arange(B) * G, H)"),
    "checkpoint_index_off_by_one": ("            m = start // interval\n",
                                    "            m = start // interval + 1\n"),
    "ragged_last_draft_dropped": (
        "    o, _ = _batch(tok0, np.repeat(cu[1:] - cu[:-1], H), head,",
        "    o, _ = _batch(tok0, np.repeat(np.maximum(cu[1:] - cu[:-1] - 1, 0), H), head,"),
    "varlen_state_to_next_sequence": ("    Sout = S0.copy()\n    for i, (n, h) in enumerate(units):\n"
                                      "        Sout[n, h] = S[i]\n    return o, Sout\n",
                                      "    Sout = S0.copy()\n    for i, (n, h) in enumerate(units):\n"
                                      "        Sout[(n + 1) % N, h] = S[i]\n    return o, Sout\n"),
}


def _failed_pins(orc):
    failed = []
    for pin in PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


def _driver_copy(old=None, new=None, name="copy"):
    """A fresh copy of the oracle's Python drivers, with one text substitution."""
    import types
    path = os.path.join(os.path.dirname(oracle.__file__), "__init__.py")
    src = open(path).read()
    if old is not None:
        assert src.count(old) == 1, "mutation anchor not found: %s" % name
        src = src.replace(old, new, 1)
    ns = {"__file__": path, "__name__": "oracle_%s" % name}
    exec(compile(src, path, "exec"), ns)
    return types.SimpleNamespace(**{f: ns[f] for f in ("unit", "prefill_varlen", "prefill_checkpoints",
                                                       "decode", "verify", "verify_ragged", "fold")})


def test_unmutated_driver_copy_passes_every_pin():
    """Control for the driver mutants: the copy loaded the same way passes."""
    assert _failed_pins(_driver_copy()) == []


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_pins_catch_planted_driver_mistakes(name):
    old, new = PY_MUTANTS[name]
    assert _failed_pins(_driver_copy(old, new, name)), "planted mistake %s passed every pin" % name


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")).read()
    assert old in src, "mutation anchor not found: %s" % name
    mpath = tmp_path / ("mut_%s.c" % name)
    mpath.write_text(src.replace(old, new, 1))
    mut = oracle.load_variant(str(mpath), str(tmp_path / ("mut_%s.so" % name)))
    assert _failed_pins(mut), "planted mistake %s passed every pin" % name
