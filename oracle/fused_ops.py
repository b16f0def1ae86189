"""Oracle of the prologue and epilogue around the KDA recurrence -- TEST
INFRASTRUCTURE ONLY (imported by tests/, the smoke check and the benchmark's CPU
legs; never by the product path).

Plain float64 numpy, written from the definitions.  The pages name the steps
(Kimi K3 on B200 deployment notes, items "prefill / decode kernel fusion" and
"other prefill switches": the short conv1d of q, k and v with SiLU and the
conv-state update, the beta sigmoid, and the gated RMSNorm of the output;
"SGLang and Miles Add Day-0 Support for Kimi K3", ladder step P5 "Conv + KDA +
Onorm Fusion") but not their constants or exact formulas.  The readings taken
here:

    conv    y_t[c] = sum_{i<W} w[c][i] x_{t-W+1+i}[c], W = 4, no bias; the
            inputs before a sequence come from its conv state (zeros if none)
    SiLU    y * sigmoid(y)
    q, k    x / sqrt(sum_c x_c^2 + eps_l2) per (token, head), eps_l2 = 1e-6
    beta    sigmoid(b)
    o norm  w[v] * o[v] / sqrt(mean_v o_v^2 + eps) * sigmoid(g[v]), eps = 1e-5

The unfused path stores its intermediates (conv + SiLU output, normalised q
and k, v, beta, the recurrence's o) in the activation dtype, and the pages'
fused kernels are bit-exact with it.  ``store`` is that storage: identity for
fp32, ``round_bf16`` for bf16 activations; every function rounds through it at
those points and computes in float64 between them.

Parity is pinned to these definitions (tests/test_oracle_fused_pins.py: a
library convolution and a library bf16 cast, closed forms, invariants,
split-call continuity, a brute-force composition); that they are the
definitions the pages' kernels use is a reading, not pinned.
"""
import numpy as np

import oracle

CONV_W = 4


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def identity(x):
    return x


def round_bf16(x):
    """Round to bfloat16 (nearest, ties to even), returned as float64: the value
    a bf16 tensor stores.  float64 -> float32 first (the kernels hold float32),
    then the low 16 bits of the float32 pattern are rounded away."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def silu(y):
    return y * sigmoid(y)


def l2norm(x, eps=1e-6):
    """x / sqrt(sum of squares over the last axis + eps)."""
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def conv_prologue(q_raw, k_raw, v_raw, b_raw, conv_w, conv_state, cu_seqlens, init_slot,
                  out_slot, eps_l2=1e-6, store=identity):
    """Short causal conv + SiLU of q, k, v over a packed varlen batch, L2 norm of
    q and k, beta = sigmoid(b), and the conv-state update.

    q_raw, k_raw, v_raw [T, H, K]; b_raw [T, H]; conv_w [3, H, K, W];
    conv_state [slots, W-1, 3, H, K] (the last W-1 raw inputs of each stream,
    oldest first); init_slot / out_slot [N] (-1: zeros / not written).
    ``store`` rounds the conv + SiLU outputs and the returned q, k, v, beta.
    Returns (q, k, v, beta, new conv_state)."""
    raws = [_f64(q_raw), _f64(k_raw), _f64(v_raw)]
    w = _f64(conv_w)
    cs = _f64(conv_state).copy()
    cs_in = cs.copy()
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, H, K = raws[0].shape
    outs = [np.zeros((T, H, K)) for _ in range(3)]
    for n in range(len(cu) - 1):
        lo, hi = cu[n], cu[n + 1]
        si, so = int(init_slot[n]), int(out_slot[n])
        for s in range(3):
            prev = cs_in[si, :, s] if si >= 0 else np.zeros((CONV_W - 1, H, K))
            x = np.concatenate([prev, raws[s][lo:hi]], axis=0)   # [W-1 + L, H, K]
            for t in range(hi - lo):
                y = np.einsum("hki,ihk->hk", w[s], x[t:t + CONV_W])
                outs[s][lo + t] = store(silu(y))
            if so >= 0:
                cs[so, :, s] = x[x.shape[0] - (CONV_W - 1):]
    q = store(l2norm(outs[0], eps_l2))
    k = store(l2norm(outs[1], eps_l2))
    return q, k, outs[2], store(sigmoid(_f64(b_raw))), cs


def gated_rmsnorm(o, g, w_norm, eps=1e-5):
    """w[v] * o[v] / sqrt(mean_v o^2 + eps) * sigmoid(g[v]) over the last axis."""
    o = _f64(o)
    r = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return _f64(w_norm) * o * r * sigmoid(_f64(g))


def decode_fused(q_raw, k_raw, v_raw, gk, b_raw, conv_w, conv_state, gate, w_norm, slot_ids,
                 S_pool, scale=1.0, eps_l2=1e-6, eps_norm=1e-5, store=identity):
    """One token per request through conv + KDA + onorm: conv_prologue with
    one-token sequences whose conv state lives in each request's slot, the
    decode recurrence on the slot's state, then gated_rmsnorm.

    q_raw, k_raw, v_raw, gk, gate [B, H, 128]; b_raw [B, H]; S_pool [slots, H,
    K, V].  Returns (out [B, H, V], new S_pool, new conv_state)."""
    B = q_raw.shape[0]
    ids = np.asarray(slot_ids, dtype=np.int64)
    q, k, v, beta, cs = conv_prologue(q_raw, k_raw, v_raw, b_raw, conv_w, conv_state,
                                      np.arange(B + 1), ids, ids, eps_l2, store)
    S = _f64(S_pool).copy()
    o, Sn = oracle.decode(q, k, v, gk, beta, S[ids], scale=scale)
    S[ids] = Sn
    return gated_rmsnorm(store(o), gate, w_norm, eps_norm), S, cs
