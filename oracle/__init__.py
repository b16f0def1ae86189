"""KDA oracle -- TEST INFRASTRUCTURE ONLY.

Plain double-precision CPU statement of the KDA gated delta-rule state path,
used to check the CUDA library.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference leg may import this package.  It
shares no code with the CUDA path (``kda_state_gb300``) and imports nothing
from it.

Recurrence, per (sequence or request, head) unit, state ``S`` of shape [K, V]::

    S_t = (I - beta_t k_t k_t^T) Diag(exp(gk_t)) S_{t-1} + beta_t k_t v_t^T
    o_t = S_t^T (scale * q_t)

Per-step inputs (v, k, gk, beta), K = V = 128, "verify never writes the
checkpoint" and "the fold replays only the accepted prefix": "SGLang and Miles
Add Day-0 Support for Kimi K3", section "ReplaySSM: raw-input replay for the
KDA state".  The [128, 128] fp32 state: Kimi K3 on B200 deployment notes,
timeline entry "FlashKDA".

The arithmetic lives in ``kda_oracle.c`` (compiled with gcc by ``build()``);
this module only marshals numpy float64 arrays.  Every function is pinned in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_default = None
_lock = threading.Lock()


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle's C source into a shared library (portable flags, no -march)."""
    stale = (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src)
    if force or stale:
        tmp = out + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.kda_oracle_unit.argtypes = [ctypes.c_int] * 3 + [ctypes.c_long] * 4 + [dp] * 5 + [
        ctypes.c_double, dp, dp]
    lib.kda_oracle_unit.restype = None
    lib.kda_oracle_unit_chunked.argtypes = [ctypes.c_int] * 4 + [ctypes.c_long] * 4 + [dp] * 5 + [
        ctypes.c_double, dp, dp]
    lib.kda_oracle_unit_chunked.restype = None
    lib.kda_oracle_batch.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_long),
                                     ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)] + [
        ctypes.c_int] * 4 + [dp] * 5 + [ctypes.c_double, dp, dp, ctypes.c_int]
    lib.kda_oracle_batch.restype = ctypes.c_int
    return lib


def _load():
    global _default
    with _lock:
        if _default is None:
            _default = _bind(build())
    return _default


def load_variant(src_path: str, out_path: str):
    """Build and bind another copy of the oracle source (used by the tests that
    plant mistakes in a copy of the oracle to show that the pins catch them).
    Returns a namespace with the same functions as this module."""
    lib = _bind(build(force=True, src=src_path, out=out_path))
    import types
    ns = types.SimpleNamespace()
    for name in ("unit", "prefill_varlen", "prefill_checkpoints", "decode", "verify",
                 "verify_ragged", "fold"):
        fn = globals()[name]
        ns.__dict__[name] = (lambda f: (lambda *a, **kw: f(*a, _lib=lib, **kw)))(fn)
    return ns


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return os.cpu_count() or 1


# --------------------------------------------------------------------------
# single unit
# --------------------------------------------------------------------------

def unit(q, k, v, gk, beta, S0, scale: float = 1.0, chunk: int = 0, _lib=None):
    """One unit: q, k, gk [T, K]; v [T, V]; beta [T]; S0 [K, V].

    Returns (o [T, V], S_T [K, V]).  ``chunk`` > 0 uses the chunked (UT) form.
    """
    q, k, v, gk, beta = (_f64(x) for x in (q, k, v, gk, beta))
    S = _f64(S0).copy()
    T, K = k.shape
    V = v.shape[1]
    o = np.zeros((T, V), np.float64)
    lib = _lib or _load()
    if chunk > 0:
        lib.kda_oracle_unit_chunked(T, K, V, chunk, K, V, 1, V, _ptr(q), _ptr(k), _ptr(v), _ptr(gk),
                                    _ptr(beta), float(scale), _ptr(S), _ptr(o))
    else:
        lib.kda_oracle_unit(T, K, V, K, V, 1, V, _ptr(q), _ptr(k), _ptr(v), _ptr(gk), _ptr(beta),
                            float(scale), _ptr(S), _ptr(o))
    return o, S


# --------------------------------------------------------------------------
# batches over packed [tokens, H, *] inputs
# --------------------------------------------------------------------------

def _batch(tok0, T, head, q, k, v, gk, beta, S, scale, want_o, chunk, nthreads, _lib=None):
    lib = _lib or _load()
    n = len(tok0)
    tok0 = np.ascontiguousarray(tok0, dtype=np.int64).astype(np.dtype("l"))
    T = np.ascontiguousarray(T, dtype=np.int32)
    head = np.ascontiguousarray(head, dtype=np.int32)
    H, K = q.shape[1], q.shape[2]
    V = v.shape[2]
    o = np.zeros(v.shape, np.float64) if want_o else None
    used = lib.kda_oracle_batch(n, tok0.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
                                T.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                head.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                H, K, V, int(chunk), _ptr(q), _ptr(k), _ptr(v), _ptr(gk), _ptr(beta),
                                float(scale), _ptr(S), _ptr(o) if want_o else None,
                                int(nthreads or default_threads()))
    return o, used


def prefill_varlen(q, k, v, gk, beta, cu_seqlens, S0, scale: float = 1.0, chunk: int = 0,
                   nthreads: int = 0, heads=None, seqs=None, _lib=None):
    """Varlen prefill: q/k/gk [T, H, K], v [T, H, V], beta [T, H], cu_seqlens [N+1],
    S0 [N, H, K, V] (initial states).  Returns (o [T, H, V], S [N, H, K, V]).

    ``seqs`` / ``heads`` restrict the run to a subset of units (outputs of other
    units stay zero, their states stay S0)."""
    q, k, v, gk, beta = (_f64(x) for x in (q, k, v, gk, beta))
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    H = q.shape[1]
    S0 = _f64(S0)
    seqs = list(range(N)) if seqs is None else list(seqs)
    heads = list(range(H)) if heads is None else list(heads)
    units = [(n, h) for n in seqs for h in heads]
    S = np.stack([S0[n, h] for n, h in units]) if units else np.zeros((0,) + S0.shape[2:])
    S = np.ascontiguousarray(S)
    o, used = _batch([cu[n] for n, _ in units], [cu[n + 1] - cu[n] for n, _ in units],
                     [h for _, h in units], q, k, v, gk, beta, S, scale, True, chunk, nthreads, _lib)
    Sout = S0.copy()
    for i, (n, h) in enumerate(units):
        Sout[n, h] = S[i]
    return o, Sout


def prefill_checkpoints(q, k, v, gk, beta, cu_seqlens, S0, interval: int, max_ckpts: int,
                        scale: float = 1.0, nthreads: int = 0, heads=None, seqs=None, _lib=None):
    """Varlen prefill that also returns the state after every ``interval``
    tokens of each sequence: checkpoint m of sequence n is the state once the
    recurrence has taken the sequence's first (m + 1) * interval tokens.

    Prefix caching keeps states only at fixed token boundaries (Kimi K3 on B200
    deployment notes, item "CuTe FlashKDA prefill": non-last chunks cut to
    multiples of the 256-token cache block so that the end-of-chunk state is an
    exact checkpoint).  Each sequence is run as consecutive pieces of
    ``interval`` tokens, each piece starting from the state the previous one
    left, and the state is read after every full piece.

    Returns (o [T, H, V], S [N, H, K, V], ckpt [N, max_ckpts, H, K, V],
    made [N]); checkpoints a sequence does not reach stay zero and made[n]
    counts the ones it does (at most max_ckpts)."""
    q, k, v, gk, beta = (_f64(x) for x in (q, k, v, gk, beta))
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    H = q.shape[1]
    S0 = _f64(S0)
    seqs = list(range(N)) if seqs is None else list(seqs)
    heads = list(range(H)) if heads is None else list(heads)
    units = [(n, h) for n in seqs for h in heads]
    lens = np.array([cu[n + 1] - cu[n] for n, _ in units], dtype=np.int64)
    S = np.stack([S0[n, h] for n, h in units]) if units else np.zeros((0,) + S0.shape[2:])
    S = np.ascontiguousarray(S)
    o = np.zeros(v.shape, np.float64)
    ckpt = np.zeros((N, max_ckpts, H) + S0.shape[2:], np.float64)
    made = np.zeros(N, np.int64)
    for n in seqs:
        made[n] = min((cu[n + 1] - cu[n]) // interval, max_ckpts)
    start = 0
    while units and start < lens.max():
        piece = np.clip(lens - start, 0, interval)
        op, _ = _batch([cu[n] + start for n, _ in units], piece, [h for _, h in units],
                       q, k, v, gk, beta, S, scale, True, 0, nthreads, _lib)
        for i, (n, h) in enumerate(units):
            sl = slice(cu[n] + start, cu[n] + start + piece[i])
            o[sl, h] = op[sl, h]
            m = start // interval
            if piece[i] == interval and m < max_ckpts:
                ckpt[n, m, h] = S[i]
        start += interval
    Sout = S0.copy()
    for i, (n, h) in enumerate(units):
        Sout[n, h] = S[i]
    return o, Sout, ckpt, made


def decode(q, k, v, gk, beta, S0, scale: float = 1.0, nthreads: int = 0, _lib=None):
    """One token per request: q/k/gk [B, H, K], v [B, H, V], beta [B, H],
    S0 [B, H, K, V] (the requests' slot states).  Returns (o [B, H, V], S)."""
    q, k, v, gk, beta = (_f64(x) for x in (q, k, v, gk, beta))
    B, H = q.shape[0], q.shape[1]
    S = _f64(S0).reshape(B * H, *S0.shape[2:]).copy()
    tok0 = np.repeat(np.arange(B), H)
    head = np.tile(np.arange(H), B)
    o, _ = _batch(tok0, np.ones(B * H), head, q, k, v, gk, beta, S, scale, True, 0, nthreads, _lib)
    return o, S.reshape(S0.shape)


def _seq_major(x):
    """[B, G, H, ...] -> [B*G, H, ...] (token-major packing, request b owns rows b*G..b*G+G-1)."""
    return _f64(x).reshape((x.shape[0] * x.shape[1],) + tuple(x.shape[2:]))


def verify(q, k, v, gk, beta, S0, scale: float = 1.0, nthreads: int = 0, _lib=None):
    """Speculative verify of G draft tokens per request from the committed
    states S0 [B, H, K, V] (never modified): q/k/gk [B, G, H, K], v [B, G, H, V],
    beta [B, G, H].  Returns o [B, G, H, V].  The records the method stores are
    the raw per-step inputs (v, k, gk, beta) themselves."""
    B, G, H = q.shape[0], q.shape[1], q.shape[2]
    S = _f64(S0).reshape(B * H, *S0.shape[2:]).copy()   # scratch copy: S0 untouched
    tok0 = np.repeat(np.arange(B) * G, H)
    head = np.tile(np.arange(H), B)
    o, _ = _batch(tok0, np.full(B * H, G), head, _seq_major(q), _seq_major(k), _seq_major(v),
                  _seq_major(gk), _seq_major(beta), S, scale, True, 0, nthreads, _lib)
    return o.reshape(v.shape)


def verify_ragged(q, k, v, gk, beta, cu_drafts, S0, scale: float = 1.0, nthreads: int = 0,
                  _lib=None):
    """Verify with a draft count per request ("SGLang and Miles Add Day-0
    Support for Kimi K3", section "Verify only what is worth verifying": the
    planner trims each request's window, and what remains is verified exactly as
    before).  q/k/gk [T, H, K], v [T, H, V], beta [T, H] packed by cu_drafts
    [B+1]; S0 [B, H, K, V] (never modified).  Request b runs the recurrence over
    its tokens cu_drafts[b] .. cu_drafts[b+1]-1 from S0[b].  Returns o [T, H, V]
    (rows of no request stay zero)."""
    q, k, v, gk, beta = (_f64(x) for x in (q, k, v, gk, beta))
    cu = np.asarray(cu_drafts, dtype=np.int64)
    B, H = len(cu) - 1, q.shape[1]
    S = _f64(S0).reshape(B * H, *S0.shape[2:]).copy()   # scratch copy: S0 untouched
    tok0 = np.repeat(cu[:-1], H)
    head = np.tile(np.arange(H), B)
    o, _ = _batch(tok0, np.repeat(cu[1:] - cu[:-1], H), head, q, k, v, gk, beta, S, scale, True,
                  0, nthreads, _lib)
    return o


def fold(rec_k, rec_v, rec_gk, rec_beta, accept, S0, nthreads: int = 0, _lib=None):
    """Replay the accepted prefix: records [B, G, H, *] in draft order, accept
    [B] in 0..G, S0 [B, H, K, V].  Request b applies its first accept[b] records
    to its state; accept 0 leaves it unchanged.  Returns the new states."""
    B, G, H = rec_k.shape[0], rec_k.shape[1], rec_k.shape[2]
    S = _f64(S0).reshape(B * H, *S0.shape[2:]).copy()
    acc = np.asarray(accept, dtype=np.int64)
    tok0 = np.repeat(np.arange(B) * G, H)
    head = np.tile(np.arange(H), B)
    Tn = np.repeat(acc, H)
    kk = _seq_major(rec_k)
    _batch(tok0, Tn, head, kk, kk, _seq_major(rec_v), _seq_major(rec_gk), _seq_major(rec_beta),
           S, 1.0, False, 0, nthreads, _lib)
    return S.reshape(S0.shape)
