"""GB300-native KDA (Kimi Delta Attention) recurrent-state library.

The compute runs in hand-written sm_103a CUDA kernels behind the C ABI of
``libkda.so`` (include/kda.h); this package is the thin Python binding.
"""
from .binding import (  # noqa: F401
    KDA_DEVERR_ACCEPT_RANGE,
    KDA_DEVERR_RANGE,
    KDA_DEVERR_TIMEOUT,
    KDA_DEVERR_SEQLENS,
    KDA_DEVERR_SLOT_RANGE,
    KDA_DTYPE_BF16,
    KDA_DTYPE_FP32,
    KDA_ERR_CUDA,
    KDA_ERR_INVALID_ARG,
    KDA_ERR_UNSUPPORTED,
    KDA_MAX_LAYERS,
    KDA_OK,
    KdaError,
    RingBuffers,
    kda_chunk_prefill,
    kda_chunk_prefill_checkpoints,
    kda_conv_prologue,
    kda_decode_fused,
    kda_decode_step,
    kda_gated_rmsnorm,
    kda_replay_fold,
    kda_ring,
    kda_selftest_bounded_wait,
    kda_selftest_prefill_wait,
    kda_slot_copy,
    kda_snapshot_commit,
    kda_status_string,
    kda_verify_store_inputs,
    kda_verify_store_inputs_ragged,
    kda_verify_snapshot,
    lib,
    make_conv_state,
    make_ring,
    record_bytes,
    ring_len_for,
    state_bytes,
)


def build(force: bool = False, verbose: bool = False) -> str:
    from ._build import build as _b
    return _b(force=force, verbose=verbose)
