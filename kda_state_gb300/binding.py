"""ctypes binding of libkda.so: the C entry points under the same names.

Argument marshalling only -- every step of the KDA path runs in the library's
CUDA kernels.  Tensors are torch tensors on the current CUDA device (PyTorch
supplies device memory and streams); shapes follow include/kda.h.  If the
library is missing the calls raise: there is no other implementation.

Errors that depend on device data (a slot id out of range, inconsistent
cu_seqlens, an accept length above the window, a wait that gave up) are found
by the kernels, which skip the affected unit and set KDA_DEVERR_* bits in
``dev_err``.  The calls never synchronise, so those bits cannot be raised here:
pass a zeroed int32 device tensor as ``dev_err`` and read it after the stream
has synchronised.  With ``dev_err=None`` (the default) such units are skipped
without a report.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARG = -1
KDA_ERR_UNSUPPORTED = -2
KDA_ERR_CUDA = -3
KDA_DTYPE_BF16 = 0
KDA_DTYPE_FP32 = 1
KDA_DEVERR_SLOT_RANGE = 1
KDA_DEVERR_ACCEPT_RANGE = 2
KDA_DEVERR_SEQLENS = 4
KDA_DEVERR_RANGE = 8
KDA_DEVERR_TIMEOUT = 16
KDA_MAX_LAYERS = 256
K_DIM = 128
V_DIM = 128

_DT = {torch.bfloat16: KDA_DTYPE_BF16, torch.float32: KDA_DTYPE_FP32}

_lib = None


class KdaError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__("%s failed: %s (%d)" % (fn, kda_status_string(status), status))
        self.status = status


class kda_ring(ctypes.Structure):
    """Mirror of the C struct ``kda_ring`` (one layer's ReplaySSM input ring)."""
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("decay", ctypes.c_void_p),
                ("beta", ctypes.c_void_p), ("ring_len", ctypes.c_int), ("reserved", ctypes.c_int)]


def lib() -> ctypes.CDLL:
    """Load libkda.so (built by ``kda_state_gb300._build.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libkda.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, ip = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
        L.kda_chunk_prefill.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, ip, ip, vp, i, ip, ip,
                                        ip, vp, f, ip, vp]
        L.kda_chunk_prefill_checkpoints.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, ip, ip,
                                                    vp, i, ip, ip, ip, i, ip, i, vp, f, ip, vp]
        L.kda_decode_step.argtypes = [i, i, i, i, i, vp, vp, vp, vp, vp, ip, vp, i, vp, f, ip, vp]
        L.kda_verify_store_inputs.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, ip, vp, i,
                                              ctypes.POINTER(kda_ring), ip, vp, f, ip, vp]
        L.kda_verify_store_inputs_ragged.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, ip, i,
                                                     ip, vp, i, ctypes.POINTER(kda_ring), ip, vp,
                                                     f, ip, vp]
        L.kda_replay_fold.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_void_p),
                                      ctypes.POINTER(kda_ring), i, i, ip, ip, ip, ip, vp]
        L.kda_verify_snapshot.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, ip, vp, i, vp, ip,
                                          i, vp, f, ip, vp]
        L.kda_snapshot_commit.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_void_p),
                                          ctypes.POINTER(ctypes.c_void_p), i, i, ip, ip, ip, ip,
                                          vp]
        ll = ctypes.c_longlong
        L.kda_conv_prologue.argtypes = [i, i, i, i, i, vp, vp, vp, ll, vp, vp, vp, i, ip, ip, ip, ip,
                                        vp, vp, vp, vp, f, ip, vp]
        L.kda_gated_rmsnorm.argtypes = [i, i, i, i, vp, ll, ll, vp, vp, f, vp, vp]
        L.kda_decode_fused.argtypes = [i, i, i, i, i, vp, vp, vp, ll, vp, vp, vp, vp, vp, vp, ip, vp,
                                       i, vp, f, f, f, ip, vp]
        L.kda_slot_copy.argtypes = [i, ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t, i, ip, ip,
                                    i, ip, vp]
        L.kda_selftest_bounded_wait.argtypes = [ip, i, vp]
        L.kda_selftest_prefill_wait.argtypes = [i, i, i, vp, vp, vp, vp, vp, ip, ip, vp, i, ip, ip,
                                                vp, ip, i, vp]
        for fn in ("kda_chunk_prefill", "kda_chunk_prefill_checkpoints", "kda_decode_step", "kda_verify_store_inputs",
                   "kda_verify_store_inputs_ragged", "kda_verify_snapshot",
                   "kda_snapshot_commit", "kda_conv_prologue", "kda_gated_rmsnorm",
                   "kda_decode_fused",
                   "kda_replay_fold", "kda_slot_copy", "kda_selftest_bounded_wait",
                   "kda_selftest_prefill_wait"):
            getattr(L, fn).restype = ctypes.c_int
        L.kda_status_string.argtypes = [ctypes.c_int]
        L.kda_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def kda_status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(fn, status):
    if status != KDA_OK:
        raise KdaError(fn, status)


def _dt(t):
    if t.dtype not in _DT:
        raise TypeError("unsupported dtype %s (bf16 or fp32)" % t.dtype)
    return _DT[t.dtype]


I32 = torch.int32
F32 = torch.float32


def _need(t, name, shape=None, dtype=None, device=None, dense=True, optional=False):
    """Check one tensor argument against the layout include/kda.h states (the C
    side receives a bare pointer and cannot): a CUDA tensor, on ``device`` when
    given, of ``dtype``, of ``shape`` (None matches any size) and, when
    ``dense``, contiguous.  Raises ValueError / TypeError before anything is
    launched."""
    if t is None:
        if optional:
            return
        raise ValueError("%s is required" % name)
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError("%s must be a CUDA tensor" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, the other operands on %s" % (name, t.device, device))
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s has dtype %s, expected %s" % (name, t.dtype, dtype))
    if shape is not None and (t.dim() != len(shape) or
                              any(e is not None and e != n for e, n in zip(shape, t.shape))):
        raise ValueError("%s has shape %s, expected [%s]" % (
            name, list(t.shape), ", ".join("*" if e is None else str(e) for e in shape)))
    if dense and not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _need_err(dev_err, device):
    """dev_err: None or a device int32 tensor of at least one element."""
    _need(dev_err, "dev_err", dtype=I32, device=device, optional=True)
    if dev_err is not None and dev_err.numel() < 1:
        raise ValueError("dev_err needs at least one element")


def _need_ring(ring, H, K, V, dtype, device, name="ring"):
    """A ring's four buffers: k, v [S, R, H, K|V] in the input dtype, decay
    [S, R, H, K] and beta [S, R, H] in fp32, one slot count and ring length."""
    _need(ring.k, name + ".k", (None, None, H, K), dtype, device)
    S, R = ring.k.shape[0], ring.k.shape[1]
    _need(ring.v, name + ".v", (S, R, H, V), dtype, device)
    _need(ring.decay, name + ".decay", (S, R, H, K), F32, device)
    _need(ring.beta, name + ".beta", (S, R, H), F32, device)


def _need_inputs(q, k, v, gk, beta, lead):
    """q, k, gk [*lead, H, K] and v [*lead, H, V], beta [*lead, H], one dtype
    (bf16 or fp32), dense, on q's device.  Returns (dtype, device, H, K, V)."""
    _need(q, "q", tuple(lead) + (None, None))
    dt, dev = q.dtype, q.device
    _dt(q)
    H, K = q.shape[-2], q.shape[-1]
    _need(k, "k", tuple(lead) + (H, K), dt, dev)
    _need(gk, "gk", tuple(lead) + (H, K), dt, dev)
    _need(v, "v", tuple(lead) + (H, None), dt, dev)
    _need(beta, "beta", tuple(lead) + (H,), dt, dev)
    return dt, dev, H, K, v.shape[-1]


# ---------------------------------------------------------------------------
# ReplaySSM ring helpers
# ---------------------------------------------------------------------------

def ring_len_for(gamma: int) -> int:
    """Ring length for gamma draft tokens: the smallest power of two that is at
    least 2 (gamma + 1) (gamma = 5 -> 12 -> 16)."""
    need = 2 * (int(gamma) + 1)
    r = 1
    while r < need:
        r <<= 1
    return r


def state_bytes(K: int = K_DIM, V: int = V_DIM) -> int:
    """Bytes of one (request, layer, head) fp32 state: 64 KB at K = V = 128."""
    return K * V * 4


def record_bytes(dtype=torch.bfloat16, K: int = K_DIM, V: int = V_DIM) -> int:
    """Bytes of one stored ring record: k and v in the input dtype, exp(gk) and
    beta in fp32 (1028 B for bf16 at K = V = 128)."""
    es = torch.tensor([], dtype=dtype).element_size()
    return K * es + V * es + K * 4 + 4


@dataclass
class RingBuffers:
    """One layer's ring: k, v [num_slots, R, H, K|V] (input dtype), decay
    [num_slots, R, H, K] and beta [num_slots, R, H] (fp32)."""
    k: torch.Tensor
    v: torch.Tensor
    decay: torch.Tensor
    beta: torch.Tensor

    @property
    def ring_len(self) -> int:
        return self.k.shape[1]

    def descriptor(self) -> kda_ring:
        return kda_ring(self.k.data_ptr(), self.v.data_ptr(), self.decay.data_ptr(),
                        self.beta.data_ptr(), self.ring_len, 0)


def make_ring(num_slots: int, ring_len: int, H: int, dtype=torch.bfloat16, device="cuda",
              K: int = K_DIM, V: int = V_DIM) -> RingBuffers:
    return RingBuffers(torch.zeros(num_slots, ring_len, H, K, dtype=dtype, device=device),
                       torch.zeros(num_slots, ring_len, H, V, dtype=dtype, device=device),
                       torch.zeros(num_slots, ring_len, H, K, dtype=torch.float32, device=device),
                       torch.zeros(num_slots, ring_len, H, dtype=torch.float32, device=device))


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def _need_prefill_common(cu_seqlens, N, state_pool, H, K, V, init_slot, out_slot, snap_slot,
                         dev_err, dev):
    if N < 0:
        raise ValueError("cu_seqlens_host needs N + 1 >= 1 entries")
    _need(cu_seqlens, "cu_seqlens", (N + 1,), I32, dev)
    _need(state_pool, "state_pool", (None, H, K, V), F32, dev)
    _need(init_slot, "init_slot", (N,), I32, dev)
    _need(out_slot, "out_slot", (N,), I32, dev)
    _need(snap_slot, "snap_slot", (N,), I32, dev, optional=True)
    _need_err(dev_err, dev)


def kda_chunk_prefill(q, k, v, gk, beta, cu_seqlens, cu_seqlens_host, state_pool, init_slot,
                      out_slot, snap_slot=None, o=None, scale: float = 1.0, dev_err=None,
                      stream=None):
    """q/k/gk [T, H, K], v [T, H, V], beta [T, H] on the device; cu_seqlens int32
    [N+1] on the device and its host copy; state_pool fp32 [slots, H, K, V];
    init_slot / out_slot / snap_slot int32 [N] on the device.  Returns o."""
    _need(q, "q", (None, None, None))
    T = q.shape[0]
    dt, dev, H, K, V = _need_inputs(q, k, v, gk, beta, (T,))
    host = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
    N = host.numel() - 1
    _need_prefill_common(cu_seqlens, N, state_pool, H, K, V, init_slot, out_slot, snap_slot,
                         dev_err, dev)
    if o is None:
        o = torch.empty(T, H, V, dtype=q.dtype, device=q.device)
    _need(o, "o", (T, H, V), dt, dev)
    hp = host.numpy().ctypes.data_as(ctypes.c_void_p)
    _check("kda_chunk_prefill", lib().kda_chunk_prefill(
        _dt(q), N, T, H, K, V, _p(q), _p(k), _p(v), _p(gk), _p(beta), _p(cu_seqlens), hp,
        _p(state_pool), state_pool.shape[0], _p(init_slot), _p(out_slot), _p(snap_slot), _p(o),
        float(scale), _p(dev_err), _stream(stream)))
    return o


def kda_chunk_prefill_checkpoints(q, k, v, gk, beta, cu_seqlens, cu_seqlens_host, state_pool,
                                  init_slot, out_slot, ckpt_interval: int, ckpt_slots,
                                  snap_slot=None, o=None, scale: float = 1.0, dev_err=None,
                                  stream=None):
    """``kda_chunk_prefill`` that also writes the state after every
    ``ckpt_interval`` tokens of sequence n into slot ``ckpt_slots[n, m]``
    (int32 [N, max_ckpts] on the device, -1 skips).  Returns o."""
    _need(q, "q", (None, None, None))
    T = q.shape[0]
    dt, dev, H, K, V = _need_inputs(q, k, v, gk, beta, (T,))
    host = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
    N = host.numel() - 1
    _need_prefill_common(cu_seqlens, N, state_pool, H, K, V, init_slot, out_slot, snap_slot,
                         dev_err, dev)
    _need(ckpt_slots, "ckpt_slots", (N, None), I32, dev)
    if o is None:
        o = torch.empty(T, H, V, dtype=q.dtype, device=q.device)
    _need(o, "o", (T, H, V), dt, dev)
    hp = host.numpy().ctypes.data_as(ctypes.c_void_p)
    _check("kda_chunk_prefill_checkpoints", lib().kda_chunk_prefill_checkpoints(
        _dt(q), N, T, H, K, V, _p(q), _p(k), _p(v), _p(gk), _p(beta), _p(cu_seqlens), hp,
        _p(state_pool), state_pool.shape[0], _p(init_slot), _p(out_slot), _p(snap_slot),
        int(ckpt_interval), _p(ckpt_slots), ckpt_slots.shape[1], _p(o), float(scale),
        _p(dev_err), _stream(stream)))
    return o


def kda_decode_step(q, k, v, gk, beta, slot_ids, state_pool, o=None, scale: float = 1.0,
                    dev_err=None, stream=None):
    """q/k/gk [B, H, K], v [B, H, V], beta [B, H]; slot_ids int32 [B].  Updates the
    pool in place and returns o [B, H, V]."""
    _need(q, "q", (None, None, None))
    B = q.shape[0]
    dt, dev, H, K, V = _need_inputs(q, k, v, gk, beta, (B,))
    _need(slot_ids, "slot_ids", (B,), I32, dev)
    _need(state_pool, "state_pool", (None, H, K, V), F32, dev)
    _need_err(dev_err, dev)
    if o is None:
        o = torch.empty(B, H, V, dtype=q.dtype, device=q.device)
    _need(o, "o", (B, H, V), dt, dev)
    _check("kda_decode_step", lib().kda_decode_step(
        _dt(q), B, H, K, V, _p(q), _p(k), _p(v), _p(gk), _p(beta), _p(slot_ids), _p(state_pool),
        state_pool.shape[0], _p(o), float(scale), _p(dev_err), _stream(stream)))
    return o


def kda_verify_store_inputs(q, k, v, gk, beta, slot_ids, state_pool, ring: RingBuffers,
                            ring_base=None, o=None, scale: float = 1.0, dev_err=None, stream=None):
    """q/k/gk [B, G, H, K], v [B, G, H, V], beta [B, G, H]; reads the pool, never
    writes it; stores the G records into ``ring``.  Returns o [B, G, H, V]."""
    _need(q, "q", (None, None, None, None))
    B, G = q.shape[0], q.shape[1]
    dt, dev, H, K, V = _need_inputs(q, k, v, gk, beta, (B, G))
    _need(slot_ids, "slot_ids", (B,), I32, dev)
    _need(state_pool, "state_pool", (None, H, K, V), F32, dev)
    _need_ring(ring, H, K, V, dt, dev)
    _need(ring_base, "ring_base", (B,), I32, dev, optional=True)
    _need_err(dev_err, dev)
    if o is None:
        o = torch.empty(B, G, H, V, dtype=q.dtype, device=q.device)
    _need(o, "o", (B, G, H, V), dt, dev)
    desc = ring.descriptor()
    _check("kda_verify_store_inputs", lib().kda_verify_store_inputs(
        _dt(q), B, G, H, K, V, _p(q), _p(k), _p(v), _p(gk), _p(beta), _p(slot_ids),
        _p(state_pool), state_pool.shape[0], ctypes.byref(desc), _p(ring_base), _p(o),
        float(scale), _p(dev_err), _stream(stream)))
    return o


def kda_verify_store_inputs_ragged(q, k, v, gk, beta, cu_drafts, G_max: int, slot_ids,
                                   state_pool, ring: RingBuffers, ring_base=None, o=None,
                                   scale: float = 1.0, dev_err=None, stream=None):
    """Verify with G_b <= G_max drafts per request: q/k/gk [T, H, K], v [T, H, V],
    beta [T, H] packed by cu_drafts (device int32 [B+1]).  Reads the pool, never
    writes it; stores request b's G_b records into ``ring``.  Returns o [T, H, V]
    (rows of no request are left as they were)."""
    _need(q, "q", (None, None, None))
    T = q.shape[0]
    dt, dev, H, K, V = _need_inputs(q, k, v, gk, beta, (T,))
    _need(cu_drafts, "cu_drafts", (None,), I32, dev)
    B = cu_drafts.numel() - 1
    if B < 0:
        raise ValueError("cu_drafts needs B + 1 >= 1 entries")
    _need(slot_ids, "slot_ids", (B,), I32, dev)
    _need(state_pool, "state_pool", (None, H, K, V), F32, dev)
    _need_ring(ring, H, K, V, dt, dev)
    _need(ring_base, "ring_base", (B,), I32, dev, optional=True)
    _need_err(dev_err, dev)
    if o is None:
        o = torch.zeros(T, H, V, dtype=q.dtype, device=q.device)
    _need(o, "o", (T, H, V), dt, dev)
    desc = ring.descriptor()
    _check("kda_verify_store_inputs_ragged", lib().kda_verify_store_inputs_ragged(
        _dt(q), B, int(G_max), H, K, V, _p(q), _p(k), _p(v), _p(gk), _p(beta), _p(cu_drafts), T,
        _p(slot_ids), _p(state_pool), state_pool.shape[0], ctypes.byref(desc), _p(ring_base),
        _p(o), float(scale), _p(dev_err), _stream(stream)))
    return o


def kda_replay_fold(state_pools, rings, slot_ids, accept_len, max_accept: int, ring_base=None,
                    dev_err=None, stream=None):
    """Fold the accepted prefixes of every layer in one launch.  state_pools: list
    of L fp32 pools [slots, H, K, V]; rings: list of L RingBuffers."""
    L = len(state_pools)
    if L != len(rings) or L == 0:
        raise ValueError("state_pools and rings must be non-empty lists of equal length")
    _need(state_pools[0], "state_pools[0]", (None, None, None, None), F32)
    S, H, K, V = state_pools[0].shape
    dev = state_pools[0].device
    for i, p in enumerate(state_pools):
        _need(p, "state_pools[%d]" % i, (S, H, K, V), F32, dev)
    dt = rings[0].k.dtype
    if dt not in _DT:
        raise TypeError("unsupported ring dtype %s (bf16 or fp32)" % dt)
    for i, r in enumerate(rings):
        _need_ring(r, H, K, V, dt, dev, "rings[%d]" % i)
    _need(slot_ids, "slot_ids", (None,), I32, dev)
    B = slot_ids.numel()
    _need(accept_len, "accept_len", (B,), I32, dev)
    _need(ring_base, "ring_base", (B,), I32, dev, optional=True)
    _need_err(dev_err, dev)
    ptrs = (ctypes.c_void_p * L)(*[p.data_ptr() for p in state_pools])
    descs = (kda_ring * L)(*[r.descriptor() for r in rings])
    _check("kda_replay_fold", lib().kda_replay_fold(
        _DT[rings[0].k.dtype], L, B, H, K, V, ptrs, descs, S, int(max_accept), _p(slot_ids),
        _p(accept_len), _p(ring_base), _p(dev_err), _stream(stream)))


def kda_verify_snapshot(q, k, v, gk, beta, slot_ids, state_pool, snaps, snap_ids, o=None,
                        scale: float = 1.0, dev_err=None, stream=None):
    """Snapshot-per-step verify: q/k/gk [B, G, H, K], v [B, G, H, V], beta
    [B, G, H]; writes the state after draft step i of request b to
    snaps[snap_ids[b], i] (snaps fp32 [num_snap_slots, G, H, K, V]); never writes
    the pool.  Returns o [B, G, H, V]."""
    _need(q, "q", (None, None, None, None))
    B, G = q.shape[0], q.shape[1]
    dt, dev, H, K, V = _need_inputs(q, k, v, gk, beta, (B, G))
    _need(slot_ids, "slot_ids", (B,), I32, dev)
    _need(state_pool, "state_pool", (None, H, K, V), F32, dev)
    _need(snaps, "snaps", (None, G, H, K, V), F32, dev)
    _need(snap_ids, "snap_ids", (B,), I32, dev)
    _need_err(dev_err, dev)
    if o is None:
        o = torch.empty(B, G, H, V, dtype=q.dtype, device=q.device)
    _need(o, "o", (B, G, H, V), dt, dev)
    _check("kda_verify_snapshot", lib().kda_verify_snapshot(
        _dt(q), B, G, H, K, V, _p(q), _p(k), _p(v), _p(gk), _p(beta), _p(slot_ids),
        _p(state_pool), state_pool.shape[0], _p(snaps), _p(snap_ids), snaps.shape[0], _p(o),
        float(scale), _p(dev_err), _stream(stream)))
    return o


def kda_snapshot_commit(state_pools, snaps, slot_ids, snap_ids, accept_len, dev_err=None,
                        stream=None):
    """Copy snapshot accept_len[b]-1 over slot slot_ids[b] in every layer, one
    launch.  state_pools / snaps: lists of L pools [slots, H, K, V] and snapshot
    buffers [num_snap_slots, G, H, K, V]."""
    L = len(state_pools)
    if L != len(snaps) or L == 0:
        raise ValueError("state_pools and snaps must be non-empty lists of equal length")
    _need(state_pools[0], "state_pools[0]", (None, None, None, None), F32)
    S, H, K, V = state_pools[0].shape
    dev = state_pools[0].device
    _need(snaps[0], "snaps[0]", (None, None, H, K, V), F32, dev)
    NS, G = snaps[0].shape[0], snaps[0].shape[1]
    for i in range(L):
        _need(state_pools[i], "state_pools[%d]" % i, (S, H, K, V), F32, dev)
        _need(snaps[i], "snaps[%d]" % i, (NS, G, H, K, V), F32, dev)
    _need(slot_ids, "slot_ids", (None,), I32, dev)
    B = slot_ids.numel()
    _need(snap_ids, "snap_ids", (B,), I32, dev)
    _need(accept_len, "accept_len", (B,), I32, dev)
    _need_err(dev_err, dev)
    pp = (ctypes.c_void_p * L)(*[p.data_ptr() for p in state_pools])
    sp = (ctypes.c_void_p * L)(*[p.data_ptr() for p in snaps])
    _check("kda_snapshot_commit", lib().kda_snapshot_commit(
        L, B, H, K, V, G, pp, sp, S, NS, _p(slot_ids), _p(snap_ids),
        _p(accept_len), _p(dev_err), _stream(stream)))


# ---------------------------------------------------------------------------
# fused prologue / epilogue around the recurrence
# ---------------------------------------------------------------------------

CONV_WIDTH = 4          # KDA_CONV_WIDTH
EPS_L2 = 1e-6           # q, k L2 norm
EPS_NORM = 1e-5         # gated RMSNorm of o


def _raw_stride(q_raw, k_raw, v_raw, K):
    """Token stride (elements) shared by three [T, H, K] raw views whose head
    and channel axes are dense (e.g. slices of one fused projection output)."""
    st = q_raw.stride(0)
    for x in (q_raw, k_raw, v_raw):
        if x.stride(-1) != 1 or x.stride(-2) != K or x.stride(0) != st:
            raise ValueError("q_raw, k_raw, v_raw need dense [H, K] rows and one token stride")
    return st


def make_conv_state(num_slots: int, H: int, dtype=torch.bfloat16, device="cuda", K: int = K_DIM):
    """Conv state pool [num_slots, W-1, 3, H, K] (zeros)."""
    return torch.zeros(num_slots, CONV_WIDTH - 1, 3, H, K, dtype=dtype, device=device)


def kda_conv_prologue(q_raw, k_raw, v_raw, b_raw, conv_w, conv_state, init_slot, out_slot,
                      cu_seqlens, cu_seqlens_host, eps_l2: float = EPS_L2, out=None, dev_err=None,
                      stream=None):
    """Short conv + SiLU of q, k, v ([T, H, K] views sharing a token stride), L2
    norm of q and k, beta = sigmoid(b_raw [T, H]); conv_w [3, H, K, W];
    conv_state [slots, W-1, 3, H, K] read at init_slot and written at out_slot
    (int32 [N] on the device, -1: zeros / none).  Returns (q, k, v, beta)."""
    _need(q_raw, "q_raw", (None, None, None), dense=False)
    T, H, K = q_raw.shape
    dt, dev = q_raw.dtype, q_raw.device
    _dt(q_raw)
    _need(k_raw, "k_raw", (T, H, K), dt, dev, dense=False)
    _need(v_raw, "v_raw", (T, H, K), dt, dev, dense=False)
    st = _raw_stride(q_raw, k_raw, v_raw, K)
    host = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
    N = host.numel() - 1
    if N < 0:
        raise ValueError("cu_seqlens_host needs N + 1 >= 1 entries")
    _need(b_raw, "b_raw", (T, H), dt, dev)
    _need(conv_w, "conv_w", (3, H, K, CONV_WIDTH), dt, dev)
    _need(conv_state, "conv_state", (None, CONV_WIDTH - 1, 3, H, K), dt, dev)
    _need(init_slot, "init_slot", (N,), I32, dev)
    _need(out_slot, "out_slot", (N,), I32, dev)
    _need(cu_seqlens, "cu_seqlens", (N + 1,), I32, dev)
    _need_err(dev_err, dev)
    if out is None:
        out = (torch.empty(T, H, K, dtype=q_raw.dtype, device=q_raw.device),
               torch.empty(T, H, K, dtype=q_raw.dtype, device=q_raw.device),
               torch.empty(T, H, K, dtype=q_raw.dtype, device=q_raw.device),
               torch.empty(T, H, dtype=q_raw.dtype, device=q_raw.device))
    q, k, v, beta = out
    for name, t in (("out[0]", q), ("out[1]", k), ("out[2]", v)):
        _need(t, name, (T, H, K), dt, dev)
    _need(beta, "out[3]", (T, H), dt, dev)
    hp = host.numpy().ctypes.data_as(ctypes.c_void_p)
    _check("kda_conv_prologue", lib().kda_conv_prologue(
        _dt(q_raw), N, T, H, K, _p(q_raw), _p(k_raw), _p(v_raw), st, _p(b_raw), _p(conv_w),
        _p(conv_state), conv_state.shape[0], _p(init_slot), _p(out_slot), _p(cu_seqlens), hp,
        _p(q), _p(k), _p(v), _p(beta), float(eps_l2), _p(dev_err), _stream(stream)))
    return q, k, v, beta


def kda_gated_rmsnorm(o, gate, w_norm, eps: float = EPS_NORM, out=None, stream=None):
    """out = w_norm * o / sqrt(mean o^2 + eps) * sigmoid(gate) per [token, head]
    row; o [T, H, V] may be strided (channel axis dense)."""
    _need(o, "o", (None, None, None), dense=False)
    T, H, V = o.shape
    dt, dev = o.dtype, o.device
    _dt(o)
    if o.stride(-1) != 1:
        raise ValueError("o needs a dense channel axis")
    _need(gate, "gate", (T, H, V), dt, dev)
    _need(w_norm, "w_norm", (V,), dt, dev)
    if out is None:
        out = torch.empty(T, H, V, dtype=o.dtype, device=o.device)
    _need(out, "out", (T, H, V), dt, dev)
    _check("kda_gated_rmsnorm", lib().kda_gated_rmsnorm(
        _dt(o), T, H, V, _p(o), o.stride(0), o.stride(1), _p(gate), _p(w_norm), float(eps),
        _p(out), _stream(stream)))
    return out


def kda_decode_fused(q_raw, k_raw, v_raw, gk, b_raw, conv_w, conv_state, gate, w_norm, slot_ids,
                     state_pool, out=None, scale: float = 1.0, eps_l2: float = EPS_L2,
                     eps_norm: float = EPS_NORM, dev_err=None, stream=None):
    """Conv + KDA + onorm for one token per request: raw q, k, v [B, H, K]
    (views sharing a token stride), gk, gate [B, H, K], b_raw [B, H]; the
    slot's conv state and KDA state are updated in place.  Returns out [B, H, V]."""
    _need(q_raw, "q_raw", (None, None, None), dense=False)
    B, H, K = q_raw.shape
    dt, dev = q_raw.dtype, q_raw.device
    _dt(q_raw)
    _need(k_raw, "k_raw", (B, H, K), dt, dev, dense=False)
    _need(v_raw, "v_raw", (B, H, K), dt, dev, dense=False)
    _need(state_pool, "state_pool", (None, H, K, None), F32, dev)
    V = state_pool.shape[-1]
    st = _raw_stride(q_raw, k_raw, v_raw, K)
    _need(gk, "gk", (B, H, K), dt, dev)
    _need(b_raw, "b_raw", (B, H), dt, dev)
    _need(conv_w, "conv_w", (3, H, K, CONV_WIDTH), dt, dev)
    _need(conv_state, "conv_state", (None, CONV_WIDTH - 1, 3, H, K), dt, dev)
    _need(gate, "gate", (B, H, V), dt, dev)
    _need(w_norm, "w_norm", (V,), dt, dev)
    _need(slot_ids, "slot_ids", (B,), I32, dev)
    _need_err(dev_err, dev)
    if out is None:
        out = torch.empty(B, H, V, dtype=q_raw.dtype, device=q_raw.device)
    _need(out, "out", (B, H, V), dt, dev)
    _check("kda_decode_fused", lib().kda_decode_fused(
        _dt(q_raw), B, H, K, V, _p(q_raw), _p(k_raw), _p(v_raw), st, _p(gk), _p(b_raw),
        _p(conv_w), _p(conv_state), _p(gate), _p(w_norm), _p(slot_ids), _p(state_pool),
        state_pool.shape[0], _p(out), float(scale), float(eps_l2), float(eps_norm), _p(dev_err),
        _stream(stream)))
    return out


def kda_slot_copy(pools, src, dst, dev_err=None, stream=None):
    """dst[i] <- src[i] in every pool of the list (int32 device index tensors)."""
    P = len(pools)
    if P == 0:
        raise ValueError("pools must be a non-empty list")
    _need(pools[0], "pools[0]", None, F32)
    dev = pools[0].device
    if pools[0].dim() < 1:
        raise ValueError("pools[0] needs a slot axis")
    for i, p in enumerate(pools):
        _need(p, "pools[%d]" % i, tuple(pools[0].shape), F32, dev)
    _need(src, "src", (None,), I32, dev)
    _need(dst, "dst", (src.numel(),), I32, dev)
    _need_err(dev_err, dev)
    ptrs = (ctypes.c_void_p * P)(*[p.data_ptr() for p in pools])
    slot_elems = pools[0][0].numel()
    _check("kda_slot_copy", lib().kda_slot_copy(
        P, ptrs, slot_elems, pools[0].shape[0], _p(src), _p(dst), src.numel(), _p(dev_err),
        _stream(stream)))


def kda_selftest_bounded_wait(dev_err, wait_us: int = 2000, stream=None):
    """One CTA waits, with the kernels' bounded-wait loop, on a barrier nothing
    arrives at; after wait_us it sets KDA_DEVERR_TIMEOUT in dev_err (a device
    int32 tensor) and returns."""
    _need(dev_err, "dev_err", dtype=I32)
    if dev_err.numel() < 1:
        raise ValueError("dev_err needs at least one element")
    _check("kda_selftest_bounded_wait", lib().kda_selftest_bounded_wait(_p(dev_err), int(wait_us),
                                                                       _stream(stream)))


def kda_selftest_prefill_wait(q, k, v, gk, beta, cu_seqlens, cu_seqlens_host, state_pool,
                              init_slot, out_slot, dev_err, o=None, wait_us: int = 1000,
                              stream=None):
    """The bf16 chunked prefill with the first chunk's q, k, gk never requested:
    every unit's first wait gives up after wait_us, sets KDA_DEVERR_TIMEOUT in
    dev_err and the unit writes no slot.  Arguments as ``kda_chunk_prefill``
    (bf16 only).  Returns o (not written by the abandoned units)."""
    _need(q, "q", (None, None, None), dtype=torch.bfloat16)
    T = q.shape[0]
    dt, dev, H, K, V = _need_inputs(q, k, v, gk, beta, (T,))
    host = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
    N = host.numel() - 1
    _need_prefill_common(cu_seqlens, N, state_pool, H, K, V, init_slot, out_slot, None, dev_err,
                         dev)
    if dev_err is None:
        raise ValueError("dev_err is required")
    if o is None:
        o = torch.empty(T, H, V, dtype=q.dtype, device=q.device)
    _need(o, "o", (T, H, V), dt, dev)
    hp = host.numpy().ctypes.data_as(ctypes.c_void_p)
    _check("kda_selftest_prefill_wait", lib().kda_selftest_prefill_wait(
        N, T, H, _p(q), _p(k), _p(v), _p(gk), _p(beta), _p(cu_seqlens), hp, _p(state_pool),
        state_pool.shape[0], _p(init_slot), _p(out_slot), _p(o), _p(dev_err), int(wait_us),
        _stream(stream)))
    return o
