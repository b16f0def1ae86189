// C entry points of libkda.so: argument validation, launch parameters, and the
// launch on the caller's stream.  No allocation, no synchronisation, no state.
// The contract of every function is documented in include/kda.h.
#include <algorithm>
#include <math.h>
#include <string.h>

#include "kda_internal.h"

namespace {

bool dtype_ok(int dt) { return dt == KDA_DTYPE_BF16 || dt == KDA_DTYPE_FP32; }
bool dims_ok(int K, int V) { return K == 128 && V == 128; }
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
int from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

}  // namespace

extern "C" {

KDA_API const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        default: return "KDA_ERR_UNKNOWN";
    }
}

static int prefill_impl(kda_dtype dt, int num_seqs, int total_tokens, int H, int K, int V,
                        const void *q, const void *k, const void *v, const void *gk,
                        const void *beta, const int32_t *cu_seqlens_dev,
                        const int32_t *cu_seqlens_host, float *state_pool, int num_slots,
                        const int32_t *init_slot, const int32_t *out_slot,
                        const int32_t *snap_slot, int ckpt_interval, const int32_t *ckpt_slots,
                        int max_ckpts, void *o, float scale, int32_t *dev_err, void *stream,
                        uint64_t wait_ns = 0, int skip_first_load = 0) {
    if (!dtype_ok(dt)) return KDA_ERR_UNSUPPORTED;
    if (!dims_ok(K, V)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_tokens < 0 || H < 1 || num_slots < 1 || !isfinite(scale))
        return KDA_ERR_INVALID_ARG;
    if (num_seqs == 0) return total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    if (!cu_seqlens_dev || !cu_seqlens_host || !state_pool || !init_slot || !out_slot)
        return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !gk || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(state_pool)) return KDA_ERR_INVALID_ARG;
    if ((long long)num_seqs * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens_host[0] != 0 || cu_seqlens_host[num_seqs] != total_tokens)
        return KDA_ERR_INVALID_ARG;
    for (int n = 0; n < num_seqs; ++n)
        if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_INVALID_ARG;

    kda::PrefillArgs a;
    a.dt = dt; a.N = num_seqs; a.T_total = total_tokens; a.H = H; a.num_slots = num_slots;
    a.q = q; a.k = k; a.v = v; a.gk = gk; a.beta = beta;
    a.cu = cu_seqlens_dev; a.cu_host = cu_seqlens_host;
    a.pool = state_pool; a.init_slot = init_slot; a.out_slot = out_slot; a.snap_slot = snap_slot;
    a.o = o; a.scale = scale; a.err = dev_err;
    a.ckpt_interval = ckpt_interval; a.max_ckpts = max_ckpts; a.ckpt_slots = ckpt_slots;
    a.wait_ns = wait_ns; a.skip_first_load = skip_first_load;
    cudaStream_t s = (cudaStream_t)stream;
    if (dt == KDA_DTYPE_BF16) {
        // the tensor-core kernel stages q, k, v, gk with TMA and stores o in 16-byte vectors
        if (total_tokens > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v) ||
                                 !aligned16(gk) || !aligned16(o)))
            return KDA_ERR_INVALID_ARG;
        return from_cuda(kda::launch_prefill_chunked(a, s));
    }
    return from_cuda(kda::launch_prefill_recurrent(a, s));
}

KDA_API int kda_chunk_prefill(kda_dtype dt, int num_seqs, int total_tokens, int H, int K, int V,
                              const void *q, const void *k, const void *v, const void *gk,
                              const void *beta, const int32_t *cu_seqlens_dev,
                              const int32_t *cu_seqlens_host, float *state_pool, int num_slots,
                              const int32_t *init_slot, const int32_t *out_slot,
                              const int32_t *snap_slot, void *o, float scale, int32_t *dev_err,
                              void *stream) {
    return prefill_impl(dt, num_seqs, total_tokens, H, K, V, q, k, v, gk, beta, cu_seqlens_dev,
                        cu_seqlens_host, state_pool, num_slots, init_slot, out_slot, snap_slot,
                        0, nullptr, 0, o, scale, dev_err, stream);
}

KDA_API int kda_chunk_prefill_checkpoints(kda_dtype dt, int num_seqs, int total_tokens, int H,
                                          int K, int V, const void *q, const void *k,
                                          const void *v, const void *gk, const void *beta,
                                          const int32_t *cu_seqlens_dev,
                                          const int32_t *cu_seqlens_host, float *state_pool,
                                          int num_slots, const int32_t *init_slot,
                                          const int32_t *out_slot, const int32_t *snap_slot,
                                          int ckpt_interval, const int32_t *ckpt_slots,
                                          int max_ckpts, void *o, float scale, int32_t *dev_err,
                                          void *stream) {
    if (ckpt_interval < 64 || ckpt_interval % 64 != 0 || max_ckpts < 1 || !ckpt_slots)
        return KDA_ERR_INVALID_ARG;
    if ((long long)num_seqs * max_ckpts > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    return prefill_impl(dt, num_seqs, total_tokens, H, K, V, q, k, v, gk, beta, cu_seqlens_dev,
                        cu_seqlens_host, state_pool, num_slots, init_slot, out_slot, snap_slot,
                        ckpt_interval, ckpt_slots, max_ckpts, o, scale, dev_err, stream);
}

KDA_API int kda_decode_step(kda_dtype dt, int B, int H, int K, int V, const void *q,
                            const void *k, const void *v, const void *gk, const void *beta,
                            const int32_t *slot_ids, float *state_pool, int num_slots, void *o,
                            float scale, int32_t *dev_err, void *stream) {
    if (!dtype_ok(dt)) return KDA_ERR_UNSUPPORTED;
    if (!dims_ok(K, V)) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || H < 1 || num_slots < 1 || !isfinite(scale)) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;
    if (!q || !k || !v || !gk || !beta || !slot_ids || !state_pool || !o)
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(state_pool)) return KDA_ERR_INVALID_ARG;
    if ((long long)B * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    kda::DecodeArgs a;
    a.dt = dt; a.B = B; a.H = H; a.num_slots = num_slots;
    a.q = q; a.k = k; a.v = v; a.gk = gk; a.beta = beta;
    a.slot_ids = slot_ids; a.pool = state_pool; a.o = o; a.scale = scale; a.err = dev_err;
    return from_cuda(kda::launch_decode(a, (cudaStream_t)stream));
}

static bool ring_ok(const kda_ring *r, int G) {
    if (!r || !r->k || !r->v || !r->decay || !r->beta) return false;
    const int R = r->ring_len;
    if (R < 2 || (R & (R - 1)) != 0) return false;
    return G >= 1 && 2 * G <= R;
}

static int verify_impl(kda_dtype dt, int B, int G, int H, int K, int V, const void *q,
                       const void *k, const void *v, const void *gk, const void *beta,
                       const int32_t *cu_drafts, int total_tokens, const int32_t *slot_ids,
                       const float *state_pool, int num_slots, const kda_ring *ring,
                       const int32_t *ring_base, void *o, float scale, int32_t *dev_err,
                       void *stream) {
    if (!dtype_ok(dt)) return KDA_ERR_UNSUPPORTED;
    if (!dims_ok(K, V)) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || H < 1 || num_slots < 1 || G < 1 || G > 64 || total_tokens < 0 ||
        !isfinite(scale))
        return KDA_ERR_INVALID_ARG;
    if (!ring_ok(ring, G)) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;
    if (!slot_ids || !state_pool) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !gk || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(state_pool)) return KDA_ERR_INVALID_ARG;
    if ((long long)B * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    kda::VerifyArgs a;
    a.dt = dt; a.B = B; a.G = G; a.H = H; a.num_slots = num_slots; a.ring_len = ring->ring_len;
    a.q = q; a.k = k; a.v = v; a.gk = gk; a.beta = beta;
    a.slot_ids = slot_ids; a.ring_base = ring_base; a.pool = state_pool;
    a.cu_drafts = cu_drafts; a.total_tokens = total_tokens;
    a.rk = ring->k; a.rv = ring->v; a.rdecay = ring->decay; a.rbeta = ring->beta;
    a.o = o; a.scale = scale; a.err = dev_err;
    return from_cuda(kda::launch_verify(a, (cudaStream_t)stream));
}

KDA_API int kda_verify_store_inputs(kda_dtype dt, int B, int G, int H, int K, int V,
                                    const void *q, const void *k, const void *v, const void *gk,
                                    const void *beta, const int32_t *slot_ids,
                                    const float *state_pool, int num_slots, const kda_ring *ring,
                                    const int32_t *ring_base, void *o, float scale,
                                    int32_t *dev_err, void *stream) {
    if (B > 0 && (!q || !k || !v || !gk || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if ((long long)B * G > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    return verify_impl(dt, B, G, H, K, V, q, k, v, gk, beta, nullptr, B * G, slot_ids,
                       state_pool, num_slots, ring, ring_base, o, scale, dev_err, stream);
}

KDA_API int kda_verify_store_inputs_ragged(kda_dtype dt, int B, int G_max, int H, int K, int V,
                                           const void *q, const void *k, const void *v,
                                           const void *gk, const void *beta,
                                           const int32_t *cu_drafts, int total_tokens,
                                           const int32_t *slot_ids, const float *state_pool,
                                           int num_slots, const kda_ring *ring,
                                           const int32_t *ring_base, void *o, float scale,
                                           int32_t *dev_err, void *stream) {
    if (B > 0 && !cu_drafts) return KDA_ERR_INVALID_ARG;
    return verify_impl(dt, B, G_max, H, K, V, q, k, v, gk, beta, cu_drafts, total_tokens,
                       slot_ids, state_pool, num_slots, ring, ring_base, o, scale, dev_err,
                       stream);
}

KDA_API int kda_replay_fold(kda_dtype dt, int num_layers, int B, int H, int K, int V,
                            float *const *state_pools, const kda_ring *rings, int num_slots,
                            int max_accept, const int32_t *slot_ids, const int32_t *accept_len,
                            const int32_t *ring_base, int32_t *dev_err, void *stream) {
    if (!dtype_ok(dt)) return KDA_ERR_UNSUPPORTED;
    if (!dims_ok(K, V)) return KDA_ERR_UNSUPPORTED;
    if (num_layers < 1 || num_layers > KDA_MAX_LAYERS || B < 0 || H < 1 || num_slots < 1)
        return KDA_ERR_INVALID_ARG;
    if (!state_pools || !rings) return KDA_ERR_INVALID_ARG;
    const int R = rings[0].ring_len;
    if (max_accept < 1 || max_accept > R || max_accept > 64) return KDA_ERR_INVALID_ARG;
    for (int l = 0; l < num_layers; ++l) {
        const kda_ring &r = rings[l];
        if (!state_pools[l] || !aligned16(state_pools[l])) return KDA_ERR_INVALID_ARG;
        if (!r.k || !r.v || !r.decay || !r.beta || r.ring_len != R || R < 2 || (R & (R - 1)))
            return KDA_ERR_INVALID_ARG;
    }
    if (B == 0) return KDA_OK;
    if (!slot_ids || !accept_len) return KDA_ERR_INVALID_ARG;
    if ((long long)num_layers * B * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    kda::FoldParams p;   // ~10 KB, copied into the launch parameters
    kda::FoldParams *pp = &p;
    pp->L = num_layers; pp->B = B; pp->H = H; pp->num_slots = num_slots;
    pp->max_accept = max_accept; pp->ring_len = R;
    pp->slot_ids = slot_ids; pp->accept = accept_len; pp->ring_base = ring_base; pp->err = dev_err;
    for (int l = 0; l < num_layers; ++l) {
        pp->layer[l].pool = state_pools[l];
        pp->layer[l].rk = rings[l].k;
        pp->layer[l].rv = rings[l].v;
        pp->layer[l].rdecay = rings[l].decay;
        pp->layer[l].rbeta = rings[l].beta;
    }
    return from_cuda(kda::launch_fold(p, dt, (cudaStream_t)stream));
}

KDA_API int kda_verify_snapshot(kda_dtype dt, int B, int G, int H, int K, int V, const void *q,
                                const void *k, const void *v, const void *gk, const void *beta,
                                const int32_t *slot_ids, const float *state_pool, int num_slots,
                                float *snaps, const int32_t *snap_ids, int num_snap_slots,
                                void *o, float scale, int32_t *dev_err, void *stream) {
    if (!dtype_ok(dt)) return KDA_ERR_UNSUPPORTED;
    if (!dims_ok(K, V)) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || H < 1 || num_slots < 1 || num_snap_slots < 1 || G < 1 || G > 64 ||
        !isfinite(scale))
        return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;
    if (!q || !k || !v || !gk || !beta || !slot_ids || !state_pool || !snaps || !snap_ids || !o)
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(state_pool) || !aligned16(snaps)) return KDA_ERR_INVALID_ARG;
    if ((long long)B * H > 0x7fffffffLL || (long long)B * G > 0x7fffffffLL)
        return KDA_ERR_INVALID_ARG;
    kda::SnapVerifyArgs a;
    a.dt = dt; a.B = B; a.G = G; a.H = H; a.num_slots = num_slots;
    a.num_snap_slots = num_snap_slots;
    a.q = q; a.k = k; a.v = v; a.gk = gk; a.beta = beta;
    a.slot_ids = slot_ids; a.snap_ids = snap_ids; a.pool = state_pool; a.snaps = snaps;
    a.o = o; a.scale = scale; a.err = dev_err;
    return from_cuda(kda::launch_verify_snapshot(a, (cudaStream_t)stream));
}

KDA_API int kda_snapshot_commit(int num_layers, int B, int H, int K, int V, int G,
                                float *const *state_pools, const float *const *snaps,
                                int num_slots, int num_snap_slots, const int32_t *slot_ids,
                                const int32_t *snap_ids, const int32_t *accept_len,
                                int32_t *dev_err, void *stream) {
    if (!dims_ok(K, V)) return KDA_ERR_UNSUPPORTED;
    if (num_layers < 1 || num_layers > KDA_MAX_LAYERS || B < 0 || H < 1 || num_slots < 1 ||
        num_snap_slots < 1 || G < 1 || G > 64)
        return KDA_ERR_INVALID_ARG;
    if (!state_pools || !snaps) return KDA_ERR_INVALID_ARG;
    for (int l = 0; l < num_layers; ++l)
        if (!state_pools[l] || !snaps[l] || !aligned16(state_pools[l]) || !aligned16(snaps[l]))
            return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;
    if (!slot_ids || !snap_ids || !accept_len) return KDA_ERR_INVALID_ARG;
    kda::SnapCommitParams p;   // ~4 KB of pointers, copied into the launch parameters
    p.L = num_layers; p.B = B; p.H = H; p.G = G; p.num_slots = num_slots;
    p.num_snap_slots = num_snap_slots; p.chunks_per_copy = 0;
    p.slot_ids = slot_ids; p.snap_ids = snap_ids; p.accept = accept_len; p.err = dev_err;
    for (int l = 0; l < num_layers; ++l) {
        p.pool[l] = state_pools[l];
        p.snaps[l] = snaps[l];
    }
    return from_cuda(kda::launch_snapshot_commit(p, (cudaStream_t)stream));
}

static bool cu_host_ok(const int32_t *cu, int N, int T) {
    if (!cu || cu[0] != 0 || cu[N] != T) return false;
    for (int n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return false;
    return true;
}

KDA_API int kda_conv_prologue(kda_dtype dt, int num_seqs, int total_tokens, int H, int K,
                              const void *q_raw, const void *k_raw, const void *v_raw,
                              long long raw_stride, const void *b_raw, const void *conv_w,
                              void *conv_state, int num_slots, const int32_t *init_slot,
                              const int32_t *out_slot, const int32_t *cu_seqlens_dev,
                              const int32_t *cu_seqlens_host, void *q, void *k, void *v,
                              void *beta, float eps_l2, int32_t *dev_err, void *stream) {
    if (!dtype_ok(dt)) return KDA_ERR_UNSUPPORTED;
    if (K != 128) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_tokens < 0 || H < 1 || num_slots < 1 || !(eps_l2 >= 0.f) ||
        !isfinite(eps_l2))
        return KDA_ERR_INVALID_ARG;
    if (num_seqs == 0) return total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    if (raw_stride < (long long)H * K) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens_dev || !cu_host_ok(cu_seqlens_host, num_seqs, total_tokens) || !conv_w ||
        !conv_state || !init_slot || !out_slot)
        return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q_raw || !k_raw || !v_raw || !b_raw || !q || !k || !v || !beta))
        return KDA_ERR_INVALID_ARG;
    // 16-byte vectors of 8 channels: every row start must be 16-byte aligned
    const long long vec = 16 / (dt == KDA_DTYPE_BF16 ? 2 : 4);
    if (raw_stride % vec != 0 || !aligned16(conv_w) || !aligned16(conv_state)) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!aligned16(q_raw) || !aligned16(k_raw) || !aligned16(v_raw) ||
                             !aligned16(q) || !aligned16(k) || !aligned16(v)))
        return KDA_ERR_INVALID_ARG;
    int max_len = 0;
    for (int n = 0; n < num_seqs; ++n)
        max_len = std::max(max_len, cu_seqlens_host[n + 1] - cu_seqlens_host[n]);
    const int max_tiles = std::max(1, (max_len + 63) / 64);
    if ((long long)num_seqs * max_tiles > 0x7fffffffLL || H > 65535) return KDA_ERR_INVALID_ARG;
    kda::PrologueArgs a;
    a.dt = dt; a.N = num_seqs; a.T_total = total_tokens; a.H = H; a.num_slots = num_slots;
    a.max_tiles = max_tiles;
    a.q_raw = q_raw; a.k_raw = k_raw; a.v_raw = v_raw; a.b_raw = b_raw; a.raw_stride = raw_stride;
    a.conv_w = conv_w; a.conv_state = conv_state; a.init_slot = init_slot; a.out_slot = out_slot;
    a.cu = cu_seqlens_dev; a.q = q; a.k = k; a.v = v; a.beta = beta; a.eps = eps_l2;
    a.err = dev_err;
    return from_cuda(kda::launch_conv_prologue(a, (cudaStream_t)stream));
}

KDA_API int kda_gated_rmsnorm(kda_dtype dt, int tokens, int H, int V, const void *o,
                              long long o_token_stride, long long o_head_stride,
                              const void *gate, const void *w_norm, float eps, void *out,
                              void *stream) {
    if (!dtype_ok(dt)) return KDA_ERR_UNSUPPORTED;
    if (V != 128) return KDA_ERR_UNSUPPORTED;
    if (tokens < 0 || H < 1 || !(eps >= 0.f) || !isfinite(eps)) return KDA_ERR_INVALID_ARG;
    if (tokens == 0) return KDA_OK;
    if ((long long)tokens * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    if (!o || !gate || !w_norm || !out || o_token_stride < 0 || o_head_stride < 0)
        return KDA_ERR_INVALID_ARG;
    const long long vec = 16 / (dt == KDA_DTYPE_BF16 ? 2 : 4);
    if (o_token_stride % vec != 0 || o_head_stride % vec != 0 || !aligned16(o) || !aligned16(gate) ||
        !aligned16(w_norm) || !aligned16(out))
        return KDA_ERR_INVALID_ARG;
    kda::NormArgs a;
    a.dt = dt; a.tokens = tokens; a.H = H; a.o = o; a.o_token_stride = o_token_stride;
    a.o_head_stride = o_head_stride; a.gate = gate; a.w_norm = w_norm; a.eps = eps; a.out = out;
    return from_cuda(kda::launch_gated_rmsnorm(a, (cudaStream_t)stream));
}

KDA_API int kda_decode_fused(kda_dtype dt, int B, int H, int K, int V, const void *q_raw,
                             const void *k_raw, const void *v_raw, long long raw_stride,
                             const void *gk, const void *b_raw, const void *conv_w,
                             void *conv_state, const void *gate, const void *w_norm,
                             const int32_t *slot_ids, float *state_pool, int num_slots,
                             void *out, float scale, float eps_l2, float eps_norm,
                             int32_t *dev_err, void *stream) {
    if (!dtype_ok(dt)) return KDA_ERR_UNSUPPORTED;
    if (!dims_ok(K, V)) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || H < 1 || num_slots < 1 || !isfinite(scale) || !(eps_l2 >= 0.f) ||
        !isfinite(eps_l2) || !(eps_norm >= 0.f) || !isfinite(eps_norm))
        return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;
    if (raw_stride < (long long)H * K) return KDA_ERR_INVALID_ARG;
    if (!q_raw || !k_raw || !v_raw || !gk || !b_raw || !conv_w || !conv_state || !gate ||
        !w_norm || !slot_ids || !state_pool || !out)
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(state_pool)) return KDA_ERR_INVALID_ARG;
    const long long vec = 16 / (dt == KDA_DTYPE_BF16 ? 2 : 4);
    if (raw_stride % vec != 0 || !aligned16(q_raw) || !aligned16(k_raw) || !aligned16(v_raw) ||
        !aligned16(gk) || !aligned16(conv_w) || !aligned16(conv_state) || !aligned16(gate) ||
        !aligned16(w_norm) || !aligned16(out))
        return KDA_ERR_INVALID_ARG;
    if ((long long)B * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    kda::FusedDecodeArgs a;
    a.dt = dt; a.B = B; a.H = H; a.num_slots = num_slots;
    a.q_raw = q_raw; a.k_raw = k_raw; a.v_raw = v_raw; a.raw_stride = raw_stride;
    a.gk = gk; a.b_raw = b_raw; a.conv_w = conv_w; a.conv_state = conv_state;
    a.gate = gate; a.w_norm = w_norm; a.slot_ids = slot_ids; a.pool = state_pool; a.out = out;
    a.scale = scale; a.eps_l2 = eps_l2; a.eps_norm = eps_norm; a.err = dev_err;
    return from_cuda(kda::launch_decode_fused(a, (cudaStream_t)stream));
}

KDA_API int kda_slot_copy(int num_pools, float *const *pools, size_t slot_elems, int num_slots,
                          const int32_t *src, const int32_t *dst, int n, int32_t *dev_err,
                          void *stream) {
    if (num_pools < 1 || num_pools > KDA_MAX_LAYERS || num_slots < 1 || n < 0 || !pools)
        return KDA_ERR_INVALID_ARG;
    if (slot_elems == 0 || (slot_elems & 3u) != 0) return KDA_ERR_INVALID_ARG;
    for (int i = 0; i < num_pools; ++i)
        if (!pools[i] || !aligned16(pools[i])) return KDA_ERR_INVALID_ARG;
    if (n == 0) return KDA_OK;
    if (!src || !dst) return KDA_ERR_INVALID_ARG;
    kda::CopyParams p;
    memset(&p, 0, sizeof(p));
    p.P = num_pools; p.n = n; p.num_slots = num_slots; p.slot_elems = slot_elems;
    p.src = src; p.dst = dst; p.err = dev_err;
    for (int i = 0; i < num_pools; ++i) p.pool[i] = pools[i];
    return from_cuda(kda::launch_slot_copy(p, (cudaStream_t)stream));
}

KDA_API int kda_selftest_prefill_wait(int num_seqs, int total_tokens, int H, const void *q,
                                      const void *k, const void *v, const void *gk,
                                      const void *beta, const int32_t *cu_seqlens_dev,
                                      const int32_t *cu_seqlens_host, float *state_pool,
                                      int num_slots, const int32_t *init_slot,
                                      const int32_t *out_slot, void *o, int32_t *dev_err,
                                      int wait_us, void *stream) {
    if (!dev_err || wait_us < 1 || wait_us > 2000000 || total_tokens < 1) return KDA_ERR_INVALID_ARG;
    return prefill_impl(KDA_DTYPE_BF16, num_seqs, total_tokens, H, 128, 128, q, k, v, gk, beta,
                        cu_seqlens_dev, cu_seqlens_host, state_pool, num_slots, init_slot, out_slot,
                        nullptr, 0, nullptr, 0, o, 1.0f, dev_err, stream,
                        (uint64_t)wait_us * 1000ull, 1);
}

KDA_API int kda_selftest_bounded_wait(int32_t *dev_err, int wait_us, void *stream) {
    if (!dev_err || wait_us < 1 || wait_us > 2000000) return KDA_ERR_INVALID_ARG;
    return from_cuda(kda::launch_selftest_wait(dev_err, wait_us, (cudaStream_t)stream));
}

}  // extern "C"
