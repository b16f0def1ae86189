"""Host-side checks that need no GPU: the library loads, exports every entry
point include/kda.h declares, rejects bad arguments before launching anything,
and its layout helpers agree with the sizes the pages print."""
import ctypes
import json
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from kda_state_gb300 import _build
    _build.build()
    import kda_state_gb300 as kda
    return kda.lib()


def declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "kda.h")).read()
    return sorted(set(re.findall(r"KDA_API\s+[\w\s\*]*?\b(kda_\w+)\s*\(", hdr)))


def test_header_declares_entry_points():
    names = declared_symbols()
    for n in ("kda_chunk_prefill", "kda_chunk_prefill_checkpoints", "kda_decode_step",
              "kda_verify_store_inputs", "kda_verify_store_inputs_ragged", "kda_replay_fold",
              "kda_verify_snapshot", "kda_snapshot_commit", "kda_conv_prologue",
              "kda_gated_rmsnorm", "kda_decode_fused", "kda_slot_copy", "kda_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_symbols():
        assert hasattr(L, n), n


def test_status_strings(L):
    import kda_state_gb300 as kda
    assert kda.kda_status_string(0) == "KDA_OK"
    assert kda.kda_status_string(-1) == "KDA_ERR_INVALID_ARG"
    assert kda.kda_status_string(-2) == "KDA_ERR_UNSUPPORTED"
    assert kda.kda_status_string(-3) == "KDA_ERR_CUDA"


FAKE = ctypes.c_void_p(4096)   # never dereferenced: every call below fails validation first


def test_decode_rejects_before_launch(L):
    # K != 128
    assert L.kda_decode_step(0, 4, 2, 64, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, FAKE,
                             1.0, None, None) == -2
    # bad dtype
    assert L.kda_decode_step(7, 4, 2, 128, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, FAKE,
                             1.0, None, None) == -2
    # null pointer
    assert L.kda_decode_step(0, 4, 2, 128, 128, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, FAKE,
                             1.0, None, None) == -1
    # misaligned pool
    assert L.kda_decode_step(0, 4, 2, 128, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                             ctypes.c_void_p(4100), 8, FAKE, 1.0, None, None) == -1
    # non-finite scale
    assert L.kda_decode_step(0, 4, 2, 128, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, FAKE,
                             float("nan"), None, None) == -1
    # empty batch: nothing to do
    assert L.kda_decode_step(0, 0, 2, 128, 128, None, None, None, None, None, None, None, 8, None,
                             1.0, None, None) == 0


def _cu(vals):
    arr = (ctypes.c_int32 * len(vals))(*vals)
    return arr


def test_prefill_rejects_bad_cu_seqlens(L):
    args = lambda cu, N, T: (0, N, T, 2, 128, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, cu, FAKE, 4,
                             FAKE, FAKE, None, FAKE, 1.0, None, None)
    assert L.kda_chunk_prefill(*args(_cu([0, 5, 3]), 2, 3)) == -1     # decreasing
    assert L.kda_chunk_prefill(*args(_cu([1, 5, 9]), 2, 9)) == -1     # cu[0] != 0
    assert L.kda_chunk_prefill(*args(_cu([0, 5, 9]), 2, 10)) == -1    # cu[N] != total
    assert L.kda_chunk_prefill(*args(None, 2, 9)) == -1               # host copy required
    assert L.kda_chunk_prefill(*(0, 0, 0, 2, 128, 128) + (None,) * 5 + (FAKE, _cu([0]), FAKE, 4,
                               FAKE, FAKE, None, None, 1.0, None, None)) == 0
    assert L.kda_chunk_prefill(*(0, 1, 4, 2, 128, 96) + (FAKE,) * 6 + (_cu([0, 4]), FAKE, 4,
                               FAKE, FAKE, None, FAKE, 1.0, None, None)) == -2


def test_prefill_checkpoints_rejects(L):
    def args(interval, slots, max_ckpts, cu=None, N=2, T=9):
        return (0, N, T, 2, 128, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                cu if cu is not None else _cu([0, 5, 9]), FAKE, 4, FAKE, FAKE, None, interval,
                slots, max_ckpts, FAKE, 1.0, None, None)
    assert L.kda_chunk_prefill_checkpoints(*args(0, FAKE, 1)) == -1      # no interval
    assert L.kda_chunk_prefill_checkpoints(*args(100, FAKE, 1)) == -1    # not a multiple of 64
    assert L.kda_chunk_prefill_checkpoints(*args(-64, FAKE, 1)) == -1
    assert L.kda_chunk_prefill_checkpoints(*args(256, None, 1)) == -1    # no slot list
    assert L.kda_chunk_prefill_checkpoints(*args(256, FAKE, 0)) == -1    # max_ckpts < 1
    # the plain prefill's own checks still apply
    assert L.kda_chunk_prefill_checkpoints(*args(256, FAKE, 2, _cu([0, 5, 3]), 2, 3)) == -1
    assert L.kda_chunk_prefill_checkpoints(*args(256, FAKE, 2, _cu([0]), 0, 0)) == 0


def test_verify_and_fold_ring_rules(L):
    import kda_state_gb300 as kda
    ring = kda.kda_ring(4096, 4096, 4096, 4096, 12, 0)           # not a power of two
    assert L.kda_verify_store_inputs(0, 2, 5, 2, 128, 128, *(FAKE,) * 6, FAKE, 4, ctypes.byref(ring),
                                     None, FAKE, 1.0, None, None) == -1
    ring.ring_len = 8                                              # 2 * G > R for G = 5
    assert L.kda_verify_store_inputs(0, 2, 5, 2, 128, 128, *(FAKE,) * 6, FAKE, 4, ctypes.byref(ring),
                                     None, FAKE, 1.0, None, None) == -1
    ring.ring_len = 16
    rag = lambda B, Gm, cu, T: (0, B, Gm, 2, 128, 128, *(FAKE,) * 5, cu, T, FAKE, FAKE, 4,
                                ctypes.byref(ring), None, FAKE, 1.0, None, None)
    assert L.kda_verify_store_inputs_ragged(*rag(2, 5, None, 6)) == -1    # no cu_drafts
    assert L.kda_verify_store_inputs_ragged(*rag(2, 9, FAKE, 6)) == -1    # 2 * G_max > R
    assert L.kda_verify_store_inputs_ragged(*rag(2, 0, FAKE, 6)) == -1    # G_max < 1
    assert L.kda_verify_store_inputs_ragged(*rag(2, 5, FAKE, -1)) == -1   # negative tokens
    assert L.kda_verify_store_inputs_ragged(*rag(0, 5, None, 0)) == 0     # empty batch
    rings = (kda.kda_ring * 2)(kda.kda_ring(4096, 4096, 4096, 4096, 16, 0),
                               kda.kda_ring(4096, 4096, 4096, 4096, 8, 0))   # ring lengths differ
    pools = (ctypes.c_void_p * 2)(4096, 4096)
    assert L.kda_replay_fold(0, 2, 2, 2, 128, 128, pools, rings, 4, 8, FAKE, FAKE, None, None,
                             None) == -1
    rings[1].ring_len = 16
    assert L.kda_replay_fold(0, 2, 2, 2, 128, 128, pools, rings, 4, 17, FAKE, FAKE, None, None,
                             None) == -1                             # max_accept > ring_len
    assert L.kda_replay_fold(0, 0, 2, 2, 128, 128, pools, rings, 4, 8, FAKE, FAKE, None, None,
                             None) == -1                             # no layers
    assert L.kda_replay_fold(0, 2, 0, 2, 128, 128, pools, rings, 4, 8, None, None, None, None,
                             None) == 0                              # empty batch


def test_snapshot_baseline_rejects(L):
    vs = lambda B, G, snaps, nsnap: (0, B, G, 2, 128, 128, *(FAKE,) * 5, FAKE, FAKE, 4, snaps, FAKE,
                                     nsnap, FAKE, 1.0, None, None)
    assert L.kda_verify_snapshot(*vs(2, 0, FAKE, 4)) == -1                   # G < 1
    assert L.kda_verify_snapshot(*vs(2, 65, FAKE, 4)) == -1                  # G > 64
    assert L.kda_verify_snapshot(*vs(2, 4, None, 4)) == -1                   # no snapshot buffer
    assert L.kda_verify_snapshot(*vs(2, 4, ctypes.c_void_p(4100), 4)) == -1  # misaligned
    assert L.kda_verify_snapshot(*vs(2, 4, FAKE, 0)) == -1                   # no snapshot slots
    assert L.kda_verify_snapshot(*vs(0, 4, None, 4)) == 0                    # empty batch
    pools = (ctypes.c_void_p * 2)(4096, 4096)
    snaps = (ctypes.c_void_p * 2)(4096, None)
    cm = lambda nl, B, G, sn: (nl, B, 2, 128, 128, G, pools, sn, 4, 4, FAKE, FAKE, FAKE, None, None)
    assert L.kda_snapshot_commit(*cm(2, 2, 4, snaps)) == -1                  # a null snapshot buffer
    snaps[1] = 4096
    assert L.kda_snapshot_commit(*cm(0, 2, 4, snaps)) == -1                  # no layers
    assert L.kda_snapshot_commit(*cm(257, 2, 4, snaps)) == -1                # too many layers
    assert L.kda_snapshot_commit(*cm(2, 2, 0, snaps)) == -1                  # G < 1
    assert L.kda_snapshot_commit(*cm(2, 0, 4, snaps)) == 0                   # empty batch


def test_fused_prologue_epilogue_rejects(L):
    cu = _cu([0, 5, 9])
    pro = lambda dt, K, stride, cuh, eps: (dt, 2, 9, 2, K, FAKE, FAKE, FAKE, stride, FAKE, FAKE,
                                           FAKE, 4, FAKE, FAKE, FAKE, cuh, FAKE, FAKE, FAKE, FAKE,
                                           eps, None, None)
    assert L.kda_conv_prologue(*pro(3, 128, 256, cu, 1e-6)) == -2        # bad dtype
    assert L.kda_conv_prologue(*pro(0, 64, 256, cu, 1e-6)) == -2         # K != 128
    assert L.kda_conv_prologue(*pro(0, 128, 255, cu, 1e-6)) == -1        # stride < H * K
    assert L.kda_conv_prologue(*pro(0, 128, 256, _cu([0, 5, 3]), 1e-6)) == -1
    assert L.kda_conv_prologue(*pro(0, 128, 256, None, 1e-6)) == -1      # host copy required
    assert L.kda_conv_prologue(*pro(0, 128, 256, cu, -1.0)) == -1        # negative eps
    assert L.kda_conv_prologue(*pro(0, 128, 256, cu, float("nan"))) == -1
    nrm = lambda V, T, o, eps: (0, T, 2, V, o, 256, 128, FAKE, FAKE, eps, FAKE, None)
    assert L.kda_gated_rmsnorm(*nrm(64, 3, FAKE, 1e-5)) == -2            # V != 128
    assert L.kda_gated_rmsnorm(*nrm(128, 3, None, 1e-5)) == -1           # no o
    assert L.kda_gated_rmsnorm(*nrm(128, 3, FAKE, -1e-5)) == -1
    assert L.kda_gated_rmsnorm(*nrm(128, 0, None, 1e-5)) == 0            # nothing to do
    dec = lambda B, stride, pool: (0, B, 2, 128, 128, FAKE, FAKE, FAKE, stride, FAKE, FAKE, FAKE,
                                   FAKE, FAKE, FAKE, FAKE, pool, 4, FAKE, 1.0, 1e-6, 1e-5, None,
                                   None)
    assert L.kda_decode_fused(*dec(2, 255, FAKE)) == -1                  # stride < H * K
    assert L.kda_decode_fused(*dec(2, 256, ctypes.c_void_p(4100))) == -1 # misaligned pool
    assert L.kda_decode_fused(*dec(0, 256, None)) == 0                   # empty batch


def test_slot_copy_rejects(L):
    pools = (ctypes.c_void_p * 1)(4096)
    assert L.kda_slot_copy(1, pools, 6, 4, FAKE, FAKE, 1, None, None) == -1      # not multiple of 4
    assert L.kda_slot_copy(0, pools, 16, 4, FAKE, FAKE, 1, None, None) == -1     # no pools
    assert L.kda_slot_copy(257, pools, 16, 4, FAKE, FAKE, 1, None, None) == -1   # too many pools
    assert L.kda_slot_copy(1, pools, 16, 4, None, None, 0, None, None) == 0      # nothing to copy


def test_size_and_alignment_limits_reject(L):
    """The remaining host checks, each met with every earlier check passing, so
    each call is refused by the check named beside it (nothing is launched)."""
    MIS = ctypes.c_void_p(4100)                    # not 16-byte aligned
    cu = _cu([0, 5, 9])
    pre = lambda H, q: (0, 2, 9, H, 128, 128, q, FAKE, FAKE, FAKE, FAKE, FAKE, cu, FAKE, 4, FAKE,
                        FAKE, None, FAKE, 1.0, None, None)
    assert L.kda_chunk_prefill(*pre(2, MIS)) == -1                  # bf16 q not 16-byte aligned
    assert L.kda_chunk_prefill(*pre((1 << 30) + 1, FAKE)) == -1     # N * H beyond 32 bits
    assert L.kda_chunk_prefill(*pre(0, FAKE)) == -1                 # H < 1
    dec = lambda B, H: (0, B, H, 128, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, FAKE, 1.0,
                        None, None)
    assert L.kda_decode_step(*dec(1 << 16, 1 << 16)) == -1          # B * H beyond 32 bits
    assert L.kda_decode_step(*dec(4, 0)) == -1                      # H < 1
    import kda_state_gb300 as kda
    ring = kda.kda_ring(4096, 4096, 4096, 4096, 256, 0)
    assert L.kda_verify_store_inputs(0, 2, 65, 2, 128, 128, *(FAKE,) * 6, FAKE, 4,
                                     ctypes.byref(ring), None, FAKE, 1.0, None, None) == -1   # G > 64
    rings = (kda.kda_ring * 2)(kda.kda_ring(4096, 4096, 4096, 4096, 16, 0),
                               kda.kda_ring(4096, 4096, 4096, 4096, 16, 0))
    for bad in (None, 4100):                                        # a null / misaligned pool
        pools = (ctypes.c_void_p * 2)(4096, bad)
        assert L.kda_replay_fold(0, 2, 2, 2, 128, 128, pools, rings, 4, 8, FAKE, FAKE, None, None,
                                 None) == -1
    pro = lambda H, stride: (0, 2, 9, H, 128, FAKE, FAKE, FAKE, stride, FAKE, FAKE, FAKE, 4, FAKE,
                             FAKE, FAKE, cu, FAKE, FAKE, FAKE, FAKE, 1e-6, None, None)
    assert L.kda_conv_prologue(*pro(2, 260)) == -1                  # stride not a multiple of 8
    assert L.kda_conv_prologue(*pro(65536, 65536 * 128)) == -1      # H > 65535 (the entry point's limit)


def test_layout_helpers_match_page_sizes():
    import kda_state_gb300 as kda
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "page_sizes.json")))
    sb = kda.state_bytes()
    assert sb == g["state_bytes_per_request_layer_head"]["value"]
    rb = kda.record_bytes(torch.bfloat16)
    e = g["raw_input_record_bytes"]
    assert abs(rb - e["value"]) <= e["rel_tol"] * e["value"]
    e = g["draft_window_snapshot_bytes"]
    assert e["gamma_plus_1"] * sb == e["value"]
    e = g["draft_window_ring_bytes"]
    assert abs(e["ring_len"] * rb - e["value"]) <= e["rel_tol"] * e["value"]
    assert 30 <= g["draft_window_snapshot_bytes"]["value"] / (e["ring_len"] * rb) <= 34
    e = g["ring_len_rule"]
    assert kda.ring_len_for(e["gamma"]) == e["value"]
    assert [kda.ring_len_for(x) for x in (0, 1, 3, 7)] == [2, 4, 8, 16]
    for key in ("state_read_per_request_step_bytes", "state_per_request_tp8_bytes"):
        e = g[key]
        assert abs(e["layers"] * e["heads"] * sb - e["value"]) <= e["rel_tol"] * e["value"]


def test_selftest_bounded_wait_rejects(L):
    assert L.kda_selftest_bounded_wait(None, 1000, None) == -1              # no status word
    assert L.kda_selftest_bounded_wait(FAKE, 0, None) == -1                 # limit below 1 us
    assert L.kda_selftest_bounded_wait(FAKE, 2000001, None) == -1           # limit above 2 s


def test_selftest_prefill_wait_rejects(L):
    cu = (ctypes.c_int32 * 2)(0, 4)
    args = lambda err, us, T=4: (1, T, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, cu, FAKE, 2, FAKE, FAKE,
                                 FAKE, err, us, None)
    assert L.kda_selftest_prefill_wait(*args(None, 1000)) == -1       # no status word
    assert L.kda_selftest_prefill_wait(*args(FAKE, 0)) == -1          # limit below 1 us
    assert L.kda_selftest_prefill_wait(*args(FAKE, 2000001)) == -1    # limit above 2 s
    assert L.kda_selftest_prefill_wait(*args(FAKE, 1000, T=0)) == -1  # no token to wait for


def test_binding_rejects_host_tensors():
    """Every wrapper checks its tensors before it touches the library: host
    (CPU) tensors, which the C side would take as device pointers, raise."""
    import kda_state_gb300 as kda
    T, H, K = 4, 2, 128
    x = {n: torch.zeros(T, H, K, dtype=torch.bfloat16) for n in ("q", "k", "v", "gk")}
    beta = torch.zeros(T, H, dtype=torch.bfloat16)
    cu = torch.tensor([0, T], dtype=torch.int32)
    ids = torch.zeros(1, dtype=torch.int32)
    pool = torch.zeros(1, H, K, K)
    with pytest.raises(ValueError, match="q must be a CUDA tensor"):
        kda.kda_chunk_prefill(x["q"], x["k"], x["v"], x["gk"], beta, cu, cu, pool, ids, ids)
    with pytest.raises(ValueError, match="q must be a CUDA tensor"):
        kda.kda_decode_step(x["q"], x["k"], x["v"], x["gk"], beta, ids, pool)
    with pytest.raises(ValueError, match="pools\\[0\\] must be a CUDA tensor"):
        kda.kda_slot_copy([pool], ids, ids)
    with pytest.raises(ValueError, match="o must be a CUDA tensor"):
        kda.kda_gated_rmsnorm(x["v"], x["v"], torch.zeros(K, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="dev_err must be a CUDA tensor"):
        kda.kda_selftest_bounded_wait(torch.zeros(1, dtype=torch.int32))
