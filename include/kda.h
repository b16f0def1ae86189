/*
 * kda.h -- C ABI of the GB300 KDA state library (libkda.so).
 *
 * Kimi Delta Attention (KDA) keeps one fp32 K x V recurrent state per
 * (sequence or request, head) and updates it with the gated delta rule
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(gk_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T (scale * q_t)
 *
 * with K = V = 128.  Sources for the shape of the problem: "SGLang and Miles
 * Add Day-0 Support for Kimi K3" (lmsys.org), sections "Hybrid KDA Memory
 * Management" (state overwritten in place, slot pools, copy-on-write and
 * snapshot copies ordered on the forward stream) and "ReplaySSM: raw-input
 * replay for the KDA state" (verify that never writes the checkpoint, stored
 * per-step inputs, one fold launch over all layers and heads, bit-identical
 * state); the Kimi K3 on B200 deployment notes (zdszero.github.io), timeline
 * entry "FlashKDA" (chunked prefill with a [128, 128] fp32 state) and
 * "DSPARK and KDA state" (per-slot input ring, power-of-two length at least
 * 2 (gamma + 1)).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Ownership: the caller allocates and owns every buffer.  The library
 *    allocates no memory, keeps no state between calls and never
 *    synchronises the device or the stream.
 *  - Pointers: "device" pointers must be CUDA device (or managed) memory of
 *    the current device; "host" pointers are read during the call only.
 *  - Layouts are dense, row-major, in elements of the stated dtype:
 *      state pool   float  [num_slots][H][K][V]   (row k = key channel)
 *      q, k, gk     dtype  [tokens][H][K]
 *      v, o         dtype  [tokens][H][V]
 *      beta         dtype  [tokens][H]
 *  - dtype: KDA_DTYPE_BF16 or KDA_DTYPE_FP32 for q, k, v, gk, beta and o; the
 *    state is always fp32.  gk is the natural-log decay (<= 0 in practice).
 *  - stream: a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All work is enqueued on it, so stream order is the happens-before
 *    between calls (e.g. a copy-on-write restore before the decode that
 *    reads the slot).
 *  - Errors found on the host (null pointer, negative size, K or V other
 *    than 128, bad dtype, ring length) return a negative kda_status and
 *    launch nothing.  A failed launch returns KDA_ERR_CUDA.  Errors that
 *    depend on device data (a slot id, an accept length, cu_seqlens) OR a
 *    KDA_DEVERR_* bit into *dev_err (if dev_err is not NULL) and skip the
 *    affected unit; nothing traps.  The caller reads *dev_err after its own
 *    synchronisation and clears it.
 *  - Slot ids within one call must be distinct (two units writing one slot
 *    race); the library does not check this.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,
    KDA_ERR_UNSUPPORTED = -2,
    KDA_ERR_CUDA = -3
} kda_status;

typedef enum { KDA_DTYPE_BF16 = 0, KDA_DTYPE_FP32 = 1 } kda_dtype;

/* Bits OR-ed into *dev_err by kernels. */
enum {
    KDA_DEVERR_SLOT_RANGE = 1,   /* a slot id outside [0, num_slots) */
    KDA_DEVERR_ACCEPT_RANGE = 2, /* an accept length outside [0, max_accept] */
    KDA_DEVERR_SEQLENS = 4,      /* cu_seqlens or cu_drafts not monotone or past total_tokens,
                                    or a draft count above G_max */
    KDA_DEVERR_RANGE = 8,        /* reserved: no kernel sets it.  The chunked prefill runs any
                                    chunk whose products could leave fp32 range (strong decays,
                                    positive gk, large k, v or state) through an fp32 recurrence
                                    instead of reporting it */
    KDA_DEVERR_TIMEOUT = 16      /* a kernel's bounded wait on its own copies gave up (the unit
                                    is abandoned, its slot is not written) */
};

/* Largest number of layers (fold) or pools (slot copy) one call takes: the
 * per-layer pointers travel in the launch parameters. */
#define KDA_MAX_LAYERS 256

/* Largest number of sequences for which prefill orders its work longest
 * first; larger batches run in batch order. */
#define KDA_MAX_LPT_SEQS 2048

/*
 * ReplaySSM input ring of ONE layer.  Record i of a verify call for the
 * request in slot s is stored at entry e = (ring_base + i) mod ring_len:
 *     k     dtype [num_slots][ring_len][H][K]   key as given
 *     v     dtype [num_slots][ring_len][H][V]   value as given
 *     decay float [num_slots][ring_len][H][K]   exp(gk) as the kernel computed it
 *     beta  float [num_slots][ring_len][H]      beta as the kernel read it
 * One record is 2*128*sizeof(dtype) + 128*4 + 4 bytes (1028 B for bf16),
 * against 64 KB for a snapshot of the state.  All four pointers are device
 * memory.  ring_len must be a power of two and at least 2*G.
 */
typedef struct {
    void *k;
    void *v;
    float *decay;
    float *beta;
    int ring_len;
    int reserved;
} kda_ring;

/*
 * kda_chunk_prefill -- varlen chunked prefill resuming from checkpoints.
 *
 * The pages' FlashKDA kernel (Kimi K3 on B200 deployment notes, timeline entry
 * "FlashKDA"; CuTe rewrite: one CTA per (sequence, head), fp32 [128,128] state
 * on chip, longest-first ordering) fuses a chunk's work and the state update
 * into one kernel.  This call does the same for a packed varlen batch.
 *
 *   dt              dtype of q, k, v, gk, beta and o
 *   num_seqs        N >= 0 sequences; total_tokens = cu_seqlens[N]
 *   H, K, V         heads, key and value dims (K = V = 128)
 *   q, k, gk        device [total_tokens][H][K]
 *   v               device [total_tokens][H][V]
 *   beta            device [total_tokens][H]
 *   cu_seqlens_dev  device int32 [N+1], sequence n = tokens cu[n] .. cu[n+1]-1
 *   cu_seqlens_host host int32 [N+1], the same values (required): validated
 *                   (cu[0] = 0, non-decreasing, cu[N] = total_tokens) and used
 *                   to order the work longest first; the device copy is still
 *                   checked per unit (KDA_DEVERR_SEQLENS)
 *   state_pool      device float [num_slots][H][K][V]
 *   init_slot       device int32 [N]: initial state slot, or -1 for zeros
 *   out_slot        device int32 [N]: slot receiving the final state (may equal
 *                   init_slot: in-place resume)
 *   snap_slot       device int32 [N] or NULL: if given and >= 0, an extra copy
 *                   of the final state (the snapshot taken at a chunk boundary)
 *   o               device [total_tokens][H][V], dtype dt
 *   scale           multiplies q
 *   dev_err         device int32 or NULL
 *   stream          cudaStream_t
 * bf16 runs the chunked tensor-core kernel; fp32 runs an exact fp32 kernel on
 * the CUDA cores.  Zero-length sequences copy init to out (or write zeros).
 * The chunked kernel is defined on every input the recurrence is: a chunk
 * whose products could leave fp32 range (a key channel's log-decay over the
 * 32-token chunk beyond 60 in magnitude, a positive gk, |k| above 256, a NaN,
 * or max |T Diag(beta)| x max |V - K~ S| above 1e6) is computed by the
 * recurrence in fp32 instead, slower but within the same tolerance.  A unit
 * whose bounded wait gave up (KDA_DEVERR_TIMEOUT) writes none of its slots.
 */
KDA_API int kda_chunk_prefill(kda_dtype dt, int num_seqs, int total_tokens, int H, int K, int V,
                              const void *q, const void *k, const void *v, const void *gk,
                              const void *beta, const int32_t *cu_seqlens_dev,
                              const int32_t *cu_seqlens_host, float *state_pool, int num_slots,
                              const int32_t *init_slot, const int32_t *out_slot,
                              const int32_t *snap_slot, void *o, float scale, int32_t *dev_err,
                              void *stream);

/*
 * kda_chunk_prefill_checkpoints -- kda_chunk_prefill that also writes the
 * state at every ckpt_interval tokens of each sequence.
 *
 * Prefix caching keeps exact states only at fixed token boundaries: the Kimi
 * K3 on B200 deployment notes (item "CuTe FlashKDA prefill") cut every
 * non-last chunk to a multiple of the cache's 256-token block so that the
 * kernel's end-of-chunk state is an exact checkpoint, and "SGLang and Miles Add
 * Day-0 Support for Kimi K3", section "Prefix caching for a recurrent state",
 * keeps such checkpoints sparsely on the radix tree.  This call emits every
 * one of a sequence's boundary states from the same launch as its prefill.
 *
 *   (all arguments of kda_chunk_prefill, same meaning)
 *   ckpt_interval  tokens between checkpoints, a positive multiple of 64
 *   ckpt_slots     device int32 [N][max_ckpts]: checkpoint m of sequence n (the
 *                  state after (m + 1) * ckpt_interval of its tokens in this
 *                  call) goes to slot ckpt_slots[n * max_ckpts + m]; -1 skips it;
 *                  checkpoints past max_ckpts or past the sequence are not made
 *   max_ckpts      >= 1
 * A checkpoint equals, bit for bit, the final state of the same call made on
 * the sequence's first (m + 1) * ckpt_interval tokens.
 */
KDA_API int kda_chunk_prefill_checkpoints(kda_dtype dt, int num_seqs, int total_tokens, int H,
                                          int K, int V, const void *q, const void *k,
                                          const void *v, const void *gk, const void *beta,
                                          const int32_t *cu_seqlens_dev,
                                          const int32_t *cu_seqlens_host, float *state_pool,
                                          int num_slots, const int32_t *init_slot,
                                          const int32_t *out_slot, const int32_t *snap_slot,
                                          int ckpt_interval, const int32_t *ckpt_slots,
                                          int max_ckpts, void *o, float scale, int32_t *dev_err,
                                          void *stream);

/*
 * kda_decode_step -- one token per request, state updated in place.
 *
 * The working slot is read and overwritten by every forward ("SGLang and Miles
 * Add Day-0 Support for Kimi K3", "Hybrid KDA Memory Management"); the pages'
 * fused decode kernel is ladder step P5 ("Kernels").
 *
 *   q, k, gk  device [B][H][K];  v, o device [B][H][V];  beta device [B][H]
 *   slot_ids  device int32 [B], distinct, each in [0, num_slots)
 *   state_pool device float [num_slots][H][K][V], updated in place
 * A request whose slot id is out of range is skipped (its o is not written).
 */
KDA_API int kda_decode_step(kda_dtype dt, int B, int H, int K, int V, const void *q,
                            const void *k, const void *v, const void *gk, const void *beta,
                            const int32_t *slot_ids, float *state_pool, int num_slots, void *o,
                            float scale, int32_t *dev_err, void *stream);

/*
 * kda_verify_store_inputs -- speculative verify of G draft tokens.
 *
 * Reads each request's committed state and NEVER writes it; emits o for the G
 * draft positions and stores each step's inputs (k, v, exp(gk), beta) into the
 * layer's ring ("ReplaySSM: raw-input replay for the KDA state").
 *
 *   q, k, gk   device [B][G][H][K];  v, o device [B][G][H][V];  beta [B][G][H]
 *   slot_ids   device int32 [B]
 *   state_pool device float [num_slots][H][K][V], read only
 *   ring       host pointer to this layer's ring descriptor (device buffers)
 *   ring_base  device int32 [B] or NULL (= 0): ring entry of draft step 0
 * Requires 1 <= G <= ring->ring_len / 2.
 * Arithmetic: the records are the decode step's values bit for bit (k, v as
 * given, exp(gk) and beta in fp32).  o is formed from the committed state in
 * one product; for bf16 inputs that product takes TF32 operands (rounded to
 * nearest, inside the bf16 output's tolerance), for fp32 inputs it is fp32
 * throughout.
 */
KDA_API int kda_verify_store_inputs(kda_dtype dt, int B, int G, int H, int K, int V,
                                    const void *q, const void *k, const void *v, const void *gk,
                                    const void *beta, const int32_t *slot_ids,
                                    const float *state_pool, int num_slots, const kda_ring *ring,
                                    const int32_t *ring_base, void *o, float scale,
                                    int32_t *dev_err, void *stream);

/*
 * kda_verify_store_inputs_ragged -- verify with a draft count per request.
 *
 * Under load a per-step planner trims each request's verify window to the
 * positions whose expected value covers their marginal cost, and the rest is
 * cut before the target forward runs; what remains is verified exactly as
 * before ("SGLang and Miles Add Day-0 Support for Kimi K3", section "Verify
 * only what is worth verifying").  Request b verifies its own G_b tokens:
 *
 *   q, k, gk   device [total_tokens][H][K];  v, o device [total_tokens][H][V];
 *              beta device [total_tokens][H]: request b's drafts are tokens
 *              cu_drafts[b] .. cu_drafts[b+1]-1
 *   cu_drafts  device int32 [B+1], non-decreasing, every G_b <= G_max and
 *              cu_drafts[B] <= total_tokens; a request that breaks this is
 *              skipped with KDA_DEVERR_SEQLENS
 *   G_max      bound on every G_b (1 <= G_max <= ring->ring_len / 2); it picks
 *              the kernel, so G_b = G_max for all b reproduces
 *              kda_verify_store_inputs bit for bit
 *   (other arguments as kda_verify_store_inputs)
 * Record i < G_b goes to ring entry (ring_base[b] + i) mod ring_len; entries
 * past G_b, and the o rows of no request, are not written.  G_b = 0 does
 * nothing.  The committed state is never written.  kda_replay_fold is
 * unchanged: it must be given accept_len[b] <= G_b.
 */
KDA_API int kda_verify_store_inputs_ragged(kda_dtype dt, int B, int G_max, int H, int K, int V,
                                           const void *q, const void *k, const void *v,
                                           const void *gk, const void *beta,
                                           const int32_t *cu_drafts, int total_tokens,
                                           const int32_t *slot_ids, const float *state_pool,
                                           int num_slots, const kda_ring *ring,
                                           const int32_t *ring_base, void *o, float scale,
                                           int32_t *dev_err, void *stream);

/*
 * kda_replay_fold -- commit the accepted prefix, all layers and heads, one launch.
 *
 * For every layer l, request b and head h: load the committed state from
 * state_pools[l] at slot_ids[b], apply the stored records 0 .. accept_len[b]-1
 * with the same per-token arithmetic as kda_decode_step, and overwrite the
 * slot.  The result is bit-identical to accept_len[b] calls of
 * kda_decode_step on the same inputs.  accept_len 0 leaves the slot untouched.
 *
 *   dt          dtype of the rings' k and v
 *   num_layers  L in [1, KDA_MAX_LAYERS]
 *   state_pools host array [L] of device pools float [num_slots][H][K][V]
 *   rings       host array [L] of ring descriptors (same ring_len for all)
 *   max_accept  upper bound for accept_len (<= ring_len)
 *   slot_ids    device int32 [B];  accept_len device int32 [B]
 *   ring_base   device int32 [B] or NULL (= 0)
 */
KDA_API int kda_replay_fold(kda_dtype dt, int num_layers, int B, int H, int K, int V,
                            float *const *state_pools, const kda_ring *rings, int num_slots,
                            int max_accept, const int32_t *slot_ids, const int32_t *accept_len,
                            const int32_t *ring_base, int32_t *dev_err, void *stream);

/*
 * kda_verify_snapshot / kda_snapshot_commit -- the snapshot-per-step verify
 * that ReplaySSM replaces, for comparing the two on the same workload.
 *
 * The baseline makes speculation reversible by saving the whole K x V state
 * after every draft step, 64 KB per request, layer and head times the draft
 * length, and the accepted length picks the saved state that becomes the slot
 * ("SGLang and Miles Add Day-0 Support for Kimi K3", section "ReplaySSM:
 * raw-input replay for the KDA state").
 *
 * kda_verify_snapshot: as kda_verify_store_inputs (same q, k, v, gk, beta, o,
 * slot_ids, state_pool; the committed state is never written), but instead of
 * ring records it writes the state after draft step i of request b to
 *   snaps  device float [num_snap_slots][G][H][K][V] at [snap_ids[b]][i]
 *   snap_ids device int32 [B], each in [0, num_snap_slots)
 * with the per-token arithmetic of kda_decode_step: snapshot i is
 * bit-identical to i + 1 decode steps.  1 <= G <= 64.
 *
 * kda_snapshot_commit: for every layer l and request b with a = accept_len[b]
 * >= 1, copies snaps[l][snap_ids[b]][a - 1] (all H heads) over
 * state_pools[l][slot_ids[b]]; a = 0 leaves the slot as it is.  One launch for
 * all layers; state_pools and snaps are host arrays of num_layers device
 * pointers (num_layers <= KDA_MAX_LAYERS).  accept_len outside [0, G] sets
 * KDA_DEVERR_ACCEPT_RANGE and skips the request.
 */
KDA_API int kda_verify_snapshot(kda_dtype dt, int B, int G, int H, int K, int V, const void *q,
                                const void *k, const void *v, const void *gk, const void *beta,
                                const int32_t *slot_ids, const float *state_pool, int num_slots,
                                float *snaps, const int32_t *snap_ids, int num_snap_slots,
                                void *o, float scale, int32_t *dev_err, void *stream);

KDA_API int kda_snapshot_commit(int num_layers, int B, int H, int K, int V, int G,
                                float *const *state_pools, const float *const *snaps,
                                int num_slots, int num_snap_slots, const int32_t *slot_ids,
                                const int32_t *snap_ids, const int32_t *accept_len,
                                int32_t *dev_err, void *stream);

/*
 * Fused prologue and epilogue around the recurrence.
 *
 * Around each KDA layer the pages fuse small steps into single kernels, each
 * bit-exact with the unfused path: the three short causal conv1d of q, k, v
 * with SiLU and the conv-state update; the beta copy and sigmoid; the conv
 * state gather and write-back; and the gated RMSNorm of the output read at its
 * raw strides (Kimi K3 on B200 deployment notes, items "prefill / decode kernel
 * fusion" and "other prefill switches"; "SGLang and Miles Add Day-0 Support for Kimi K3",
 * ladder step P5 "Conv + KDA + Onorm Fusion" for decode).  The pages give
 * neither the conv width nor the gate or norm formulas; this library uses:
 *
 *   conv     y_t[c] = sum_{i<W} w[c][i] x_{t-W+1+i}[c], W = KDA_CONV_WIDTH,
 *            no bias; x before the sequence start comes from the conv state
 *   SiLU     silu(y) = y / (1 + exp(-y))
 *   q, k     L2-normalised per (token, head): x / sqrt(sum x^2 + eps_l2)
 *   beta     sigmoid(b) = 1 / (1 + exp(-b))
 *   o norm   out = w_norm[v] * o[v] / sqrt(mean_v o^2 + eps_norm) * sigmoid(g[v])
 *
 * Every intermediate that an unfused path would store (conv + SiLU output,
 * normalised q and k, v, beta, o) is rounded to the dtype at the same point in
 * the fused kernels, so kda_decode_fused equals kda_conv_prologue (one token
 * per request) + kda_decode_step + kda_gated_rmsnorm bit for bit.
 *
 * Conv state pool: dtype [num_slots][KDA_CONV_WIDTH-1][3][H][K] -- for each
 * slot, the last W-1 raw inputs of q, k and v (stream 0, 1, 2), oldest first.
 * Conv weights: dtype [3][H][K][KDA_CONV_WIDTH].  (K = V = 128.)
 *
 * These kernels move 8 channels per 16-byte access: every device pointer must
 * be 16-byte aligned and every stride a multiple of 16 bytes (else
 * KDA_ERR_INVALID_ARG).
 */
#define KDA_CONV_WIDTH 4

/*
 * kda_conv_prologue -- conv + SiLU (+ L2 norm for q, k) and beta sigmoid for a
 * packed varlen batch, with the conv state read from and written to slots.
 *
 *   q_raw, k_raw, v_raw device dtype: token t, head h, channel c at
 *                   [t * raw_stride + h * K + c] (raw_stride >= H * K: the three
 *                   may be views of one fused projection output)
 *   b_raw           device dtype [total_tokens][H]
 *   conv_w          device dtype [3][H][K][KDA_CONV_WIDTH]
 *   conv_state      device dtype [num_slots][KDA_CONV_WIDTH-1][3][H][K]
 *   init_slot       device int32 [N]: slot holding sequence n's conv state, or
 *                   -1 for zeros
 *   out_slot        device int32 [N]: slot receiving its state after the
 *                   sequence, or -1 for none (may equal init_slot)
 *   cu_seqlens_dev / _host  as kda_chunk_prefill
 *   q, k, v         device dtype [total_tokens][H][K]; beta [total_tokens][H]
 * Slots out of range skip the sequence with KDA_DEVERR_SLOT_RANGE.
 */
KDA_API int kda_conv_prologue(kda_dtype dt, int num_seqs, int total_tokens, int H, int K,
                              const void *q_raw, const void *k_raw, const void *v_raw,
                              long long raw_stride, const void *b_raw, const void *conv_w,
                              void *conv_state, int num_slots, const int32_t *init_slot,
                              const int32_t *out_slot, const int32_t *cu_seqlens_dev,
                              const int32_t *cu_seqlens_host, void *q, void *k, void *v,
                              void *beta, float eps_l2, int32_t *dev_err, void *stream);

/*
 * kda_gated_rmsnorm -- out = w_norm * o / sqrt(mean o^2 + eps) * sigmoid(g),
 * per (token, head) row of V values.
 *
 *   o       device dtype, row (t, h) at [t * o_token_stride + h * o_head_stride]
 *           (the attention output read at its own strides, no copy)
 *   gate    device dtype [tokens][H][V];  w_norm device dtype [V]
 *   out     device dtype [tokens][H][V]
 */
KDA_API int kda_gated_rmsnorm(kda_dtype dt, int tokens, int H, int V, const void *o,
                              long long o_token_stride, long long o_head_stride,
                              const void *gate, const void *w_norm, float eps, void *out,
                              void *stream);

/*
 * kda_decode_fused -- conv + KDA + onorm: one token per request in one kernel.
 *
 * For request b (slot s = slot_ids[b]) and head h: conv of the new raw q, k, v
 * with the slot's conv state (updated in place), SiLU, L2 norm of q and k, beta
 * = sigmoid(b_raw), the decode step of kda_decode_step on the slot's KDA state
 * (in place), and the gated RMSNorm of o into out.  raw inputs as
 * kda_conv_prologue with one token per request; gk device dtype [B][H][K];
 * gate [B][H][V]; out [B][H][V]; conv_state has num_slots slots like
 * state_pool.  Bit-identical to the three unfused calls (see above).
 */
KDA_API int kda_decode_fused(kda_dtype dt, int B, int H, int K, int V, const void *q_raw,
                             const void *k_raw, const void *v_raw, long long raw_stride,
                             const void *gk, const void *b_raw, const void *conv_w,
                             void *conv_state, const void *gate, const void *w_norm,
                             const int32_t *slot_ids, float *state_pool, int num_slots,
                             void *out, float scale, float eps_l2, float eps_norm,
                             int32_t *dev_err, void *stream);

/*
 * kda_slot_copy -- dst slot <- src slot in every pool, bit-exact.
 *
 * The copy-on-write restore and the snapshot of "Hybrid KDA Memory
 * Management": kernels on the caller's (forward) stream.
 *
 *   num_pools   P in [1, KDA_MAX_LAYERS]; pools host array [P] of device pools
 *   slot_elems  floats per slot (H*K*V), a multiple of 4
 *   src, dst    device int32 [n]; pairs must not overlap (no slot is both a
 *               source and a destination in one call)
 */
KDA_API int kda_slot_copy(int num_pools, float *const *pools, size_t slot_elems, int num_slots,
                          const int32_t *src, const int32_t *dst, int n, int32_t *dev_err,
                          void *stream);

/*
 * kda_selftest_bounded_wait -- exercises the bounded-wait path of the kernels.
 *
 * Launches one CTA that waits, with the wait loop the kernels use on their
 * asynchronous copies, on a shared-memory barrier that nothing arrives at.
 * The wait gives up after wait_us microseconds, sets KDA_DEVERR_TIMEOUT in
 * *dev_err and the kernel returns: no fault, trap or hang, and the context
 * stays usable.  Not part of the KDA path; it lets a test see the timeout
 * status that a copy which never completes would produce.
 *
 *   dev_err  device int32 (required)
 *   wait_us  1 .. 2,000,000
 */
KDA_API int kda_selftest_bounded_wait(int32_t *dev_err, int wait_us, void *stream);

/*
 * kda_selftest_prefill_wait -- exercises the chunked prefill's own bounded wait.
 *
 * Runs the bf16 chunked prefill kernel (the kernel kda_chunk_prefill launches)
 * on the given batch, except that the first chunk's q, k and gk tiles are never
 * requested, so the first wait of every unit is on a barrier nothing arrives
 * at.  Each unit's waits give up after wait_us microseconds: KDA_DEVERR_TIMEOUT
 * is set in *dev_err, the unit writes no slot (out_slot keeps its contents),
 * frees its tensor memory and returns.  No fault, trap or hang; the context
 * stays usable and the next launch runs normally.  Not part of the KDA path.
 *
 *   arguments as kda_chunk_prefill (dtype bf16, K = V = 128, no snapshot,
 *   scale 1); total_tokens >= 1; dev_err required; wait_us 1 .. 2,000,000
 */
KDA_API int kda_selftest_prefill_wait(int num_seqs, int total_tokens, int H, const void *q,
                                      const void *k, const void *v, const void *gk,
                                      const void *beta, const int32_t *cu_seqlens_dev,
                                      const int32_t *cu_seqlens_host, float *state_pool,
                                      int num_slots, const int32_t *init_slot,
                                      const int32_t *out_slot, void *o, int32_t *dev_err,
                                      int wait_us, void *stream);

/* Human-readable name of a kda_status value. */
KDA_API const char *kda_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
