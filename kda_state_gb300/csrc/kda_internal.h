// Internal launch interface between the C entry points (kda_api.cu) and the
// kernel translation units.  Host-side only; no device code here.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

struct DecodeArgs {
    int dt, B, H, num_slots;
    const void *q, *k, *v, *gk, *beta;
    const int32_t *slot_ids;
    float *pool;
    void *o;
    float scale;
    int32_t *err;
};

struct VerifyArgs {
    int dt, B, G, H, num_slots, ring_len;
    const void *q, *k, *v, *gk, *beta;
    const int32_t *slot_ids, *ring_base;
    // ragged drafts: request b's tokens are cu_drafts[b] .. cu_drafts[b+1]-1 of
    // [total_tokens][H][..] and number at most G; NULL: uniform [B][G][H][..]
    const int32_t *cu_drafts;
    int total_tokens;
    const float *pool;
    void *rk, *rv;
    float *rdecay, *rbeta;
    void *o;
    float scale;
    int32_t *err;
};

// One layer of a fold: its state pool and ring buffers.
struct FoldLayer {
    float *pool;
    void *rk, *rv;
    float *rdecay, *rbeta;
};

struct FoldParams {
    int L, B, H, num_slots, max_accept, ring_len;
    const int32_t *slot_ids, *accept, *ring_base;
    int32_t *err;
    FoldLayer layer[KDA_MAX_LAYERS];
};

struct CopyParams {
    int P, n, num_slots, chunks_per_copy;
    size_t slot_elems;
    const int32_t *src, *dst;
    int32_t *err;
    float *pool[KDA_MAX_LAYERS];
};

struct PrefillArgs {
    int dt, N, T_total, H, num_slots;
    const void *q, *k, *v, *gk, *beta;
    const int32_t *cu;            // device
    const int32_t *cu_host;       // host (validated)
    float *pool;
    const int32_t *init_slot, *out_slot, *snap_slot;
    void *o;
    float scale;
    int32_t *err;
    int ckpt_interval;             // 0: no checkpoints
    int max_ckpts;
    const int32_t *ckpt_slots;     // device [N][max_ckpts]
    uint64_t wait_ns = 0;          // limit of the kernel's waits (0: its default)
    int skip_first_load = 0;       // self-test only: the first chunk's q, k, gk are never requested
};

// Snapshot-per-step verify: the state after every draft step into a
// snapshot buffer [num_snap_slots][G][H][K][V].
struct SnapVerifyArgs {
    int dt, B, G, H, num_slots, num_snap_slots;
    const void *q, *k, *v, *gk, *beta;
    const int32_t *slot_ids, *snap_ids;
    const float *pool;
    float *snaps;
    void *o;
    float scale;
    int32_t *err;
};

// Commit of the snapshot baseline: snapshot accept-1 -> the request's slot,
// every layer, one launch.
struct SnapCommitParams {
    int L, B, H, G, num_slots, num_snap_slots, chunks_per_copy;
    const int32_t *slot_ids, *snap_ids, *accept;
    int32_t *err;
    float *pool[KDA_MAX_LAYERS];
    const float *snaps[KDA_MAX_LAYERS];
};

// Conv prologue over a packed varlen batch: grid (N x max_tiles, H).
struct PrologueArgs {
    int dt, N, T_total, H, num_slots, max_tiles;
    const void *q_raw, *k_raw, *v_raw, *b_raw;
    long long raw_stride;
    const void *conv_w;
    void *conv_state;
    const int32_t *init_slot, *out_slot, *cu;
    void *q, *k, *v, *beta;
    float eps;
    int32_t *err;
};

struct NormArgs {
    int dt, tokens, H;
    const void *o;
    long long o_token_stride, o_head_stride;
    const void *gate, *w_norm;
    float eps;
    void *out;
};

struct FusedDecodeArgs {
    int dt, B, H, num_slots;
    const void *q_raw, *k_raw, *v_raw;
    long long raw_stride;
    const void *gk, *b_raw, *conv_w;
    void *conv_state;
    const void *gate, *w_norm;
    const int32_t *slot_ids;
    float *pool;
    void *out;
    float scale, eps_l2, eps_norm;
    int32_t *err;
};

cudaError_t launch_conv_prologue(const PrologueArgs &a, cudaStream_t s);
cudaError_t launch_gated_rmsnorm(const NormArgs &a, cudaStream_t s);
cudaError_t launch_decode_fused(const FusedDecodeArgs &a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_verify_snapshot(const SnapVerifyArgs &a, cudaStream_t s);
cudaError_t launch_snapshot_commit(const SnapCommitParams &p, cudaStream_t s);
cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s);
cudaError_t launch_fold(const FoldParams &p, int dt, cudaStream_t s);
cudaError_t launch_slot_copy(const CopyParams &p, cudaStream_t s);
// Exact fp32 CUDA-core prefill (token by token, state in registers).
cudaError_t launch_prefill_recurrent(const PrefillArgs &a, cudaStream_t s);
// Chunked tensor-core prefill (bf16 inputs).
cudaError_t launch_prefill_chunked(const PrefillArgs &a, cudaStream_t s);

// One CTA waiting on a barrier nothing arrives at, for wait_us microseconds.
cudaError_t launch_selftest_wait(int32_t *err, int wait_us, cudaStream_t s);

}  // namespace kda
