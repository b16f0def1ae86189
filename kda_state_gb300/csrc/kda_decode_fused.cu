// Fused decode of the KDA state library: conv + KDA + onorm in one kernel, one
// token per (request, head).  The new raw q, k, v go through the short conv
// with the slot's conv state (updated in place) and SiLU, q and k are
// L2-normalised, beta = sigmoid(b), the decode step updates the slot's state in
// place, and o leaves through the gated RMSNorm.
//
// The arithmetic is the unfused path's, step for step: the helpers and lane
// layout of kda_fused_ops.cuh (8 channels per lane, one 128-channel row per
// half-warp), the same rounding to the dtype wherever the unfused path stores
// an intermediate, and the decode step's stage_token / token_update.  So the
// result is bit-identical to kda_conv_prologue + kda_decode_step +
// kda_gated_rmsnorm.
//
// Persistent: each CTA walks units u = blockIdx.x, + gridDim.x, ...  While it
// computes unit u, bulk copies land unit u + gridDim.x's 64 KB state and small
// inputs (raw q, k, v, conv state, conv taps, gk, gate) in shared memory, so
// the conv, the barriers and the norm no longer sit between HBM transfers.
//
// Roles in the prologue: warp 0 runs the conv of q (lanes 0-15) and k (lanes
// 16-31); warp 1 the conv of v (lanes 0-15) and stages gk (lanes 16-31); warp 2
// stages the gate (lanes 0-15) and computes beta (lane 16); warp 7 issues the
// next unit's copies, one per lane; the norm epilogue runs on the lower half of
// warp 2.
//
// Paper correspondence: "SGLang and Miles Add Day-0 Support for Kimi K3"
// (lmsys.org), ladder step P5 "Conv + KDA + Onorm Fusion" in "Kernels"; the
// working slot is read and overwritten by every forward ("Hybrid KDA Memory
// Management").
#include "kda_async.cuh"
#include "kda_fused_ops.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

// The next unit's inputs, landed by bulk copies (every member a multiple of
// 16 bytes, so every member stays 16-byte aligned).
template <typename T>
struct FusedStage {
    float state[STATE_ELEMS];          // the slot's state, row-major [k][v]
    T raw[3][KD];                      // new raw q, k, v
    T conv[CONV_TAPS][3][KD];          // conv state rows [tap][stream]
    T taps[3][KD * CONV_W];            // conv weights of the head [stream][c][tap]
    T gk[KD];
    T gate[VD];
};

template <typename T>
struct FusedSmem {
    FusedStage<T> st;
    TokenIn in;
    Reduce red;
    alignas(16) T qs[KD];
    alignas(16) T ks[KD];
    alignas(16) T vs[VD];
    alignas(16) T gs[KD];
    alignas(16) T gate_s[VD];
    alignas(16) T wn_s[VD];
    alignas(16) float os[VD];
    alignas(8) uint64_t bar_state;   // the 64 KB state of the staged unit
    alignas(8) uint64_t bar_small;   // its small inputs
    T bs[2];
    int skip;   // the staged unit's slot is out of range
    int slot;   // the staged unit's slot
    int ok;     // the last waits succeeded
};

template <typename T>
__device__ __forceinline__ uint32_t small_bytes() {
    return (uint32_t)(sizeof(T) * (3 * KD + CONV_TAPS * 3 * KD + 3 * KD * CONV_W + KD + VD));
}

// The producer is warp PRODUCER, idle during the prologue: lane 0 arms the
// barrier (or marks the unit skipped), then each lane issues one copy.
constexpr int PRODUCER = 7;
constexpr int STATE_PIECES = 4;                     // 16 KB copies of the state
constexpr int SMALL_PIECES = 3 + 3 * CONV_TAPS + 3 + 2;   // raw, conv rows, taps, gk, gate

// Unit u's state into the stage; slot is its slot id (read ahead by lane 0).
// Returns the slot, or -1 when the unit is skipped.
template <typename T>
__device__ int stage_state(const FusedDecodeArgs &a, FusedSmem<T> &sm, uint32_t bar, int u, int slot,
                           int lane) {
    const int h = u - (u / a.H) * a.H;
    const bool bad = slot < 0 || slot >= a.num_slots;
    if (lane == 0) {
        sm.skip = bad;
        sm.slot = slot;
        if (bad) {
            if (h == 0) report(a.err, DEVERR_SLOT_RANGE);
            barrier_arrive(bar);
        } else {
            barrier_expect(bar, (uint32_t)(sizeof(float) * STATE_ELEMS));
        }
    }
    __syncwarp();
    if (bad) return -1;
    constexpr int PIECE = STATE_ELEMS / STATE_PIECES;
    if (lane < STATE_PIECES)
        bulk_copy(sm.st.state + lane * PIECE, a.pool + ((size_t)slot * a.H + h) * STATE_ELEMS + lane * PIECE,
                  PIECE * 4, bar);
    return slot;
}

// Unit u's small inputs into the stage (slot -1: skipped unit).
template <typename T>
__device__ void stage_small(const FusedDecodeArgs &a, FusedSmem<T> &sm, uint32_t bar, int u, int slot,
                            int lane) {
    if (lane == 0) {
        if (slot < 0) barrier_arrive(bar);
        else barrier_expect(bar, small_bytes<T>());
    }
    __syncwarp();
    if (slot < 0 || lane >= SMALL_PIECES) return;
    const int b = u / a.H, h = u - (u / a.H) * a.H;
    const T *cs = (const T *)a.conv_state;
    if (lane < 3) {
        const int s = lane;
        const T *raw = (const T *)(s == 0 ? a.q_raw : s == 1 ? a.k_raw : a.v_raw);
        bulk_copy(sm.st.raw[s], raw + (size_t)b * a.raw_stride + (size_t)h * KD, KD * sizeof(T), bar);
    } else if (lane < 3 + 3 * CONV_TAPS) {
        const int i = (lane - 3) / 3, s = (lane - 3) % 3;
        bulk_copy(sm.st.conv[i][s], cs + conv_state_idx(slot, i, s, a.H, h, 0), KD * sizeof(T), bar);
    } else if (lane < 3 + 3 * CONV_TAPS + 3) {
        const int s = lane - 3 - 3 * CONV_TAPS;
        bulk_copy(sm.st.taps[s], (const T *)a.conv_w + ((size_t)s * a.H + h) * KD * CONV_W,
                  KD * CONV_W * sizeof(T), bar);
    } else if (lane == SMALL_PIECES - 2) {
        bulk_copy(sm.st.gk, (const T *)a.gk + (size_t)u * KD, KD * sizeof(T), bar);
    } else {
        bulk_copy(sm.st.gate, (const T *)a.gate + (size_t)u * VD, VD * sizeof(T), bar);
    }
}

template <typename T>
__global__ void __launch_bounds__(CTA_THREADS, 2)
    decode_fused_kernel(const __grid_constant__ FusedDecodeArgs a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    FusedSmem<T> &sm = *reinterpret_cast<FusedSmem<T> *>(smem_raw);
    const int U = a.B * a.H;
    int u = blockIdx.x;
    if (u >= U) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, half = lane >> 4;
    const int c0 = (lane & 15) * LANE_CH;
    const uint32_t bar_s = shared_addr(&sm.bar_state), bar_x = shared_addr(&sm.bar_small);
    const bool beta_thread = warp == 2 && lane == 16;
    if (tid == 0) {
        barrier_init(bar_s, 1);
        barrier_init(bar_x, 1);
    }
    if (warp == 2 && half == 0) {
        Pack8<T> n;
        ld8((const T *)a.w_norm + c0, n);
        st8(sm.wn_s + c0, n);
    }
    float b_next = beta_thread ? to_f(((const T *)a.b_raw)[u]) : 0.f;
    __syncthreads();
    if (warp == PRODUCER) {
        fence_async_shared();
        const int sl = stage_state(a, sm, bar_s, u, a.slot_ids[u / a.H], lane);
        stage_small(a, sm, bar_x, u, sl, lane);
    }

    uint32_t phase = 0;
    for (; u < U; u += gridDim.x) {
        const int un = u + (int)gridDim.x;   // the unit staged during this one
        if (tid == 0) sm.ok = barrier_wait(bar_s, phase) && barrier_wait(bar_x, phase);
        __syncthreads();
        phase ^= 1;
        if (!sm.ok) {
            if (tid == 0) report(a.err, DEVERR_TIMEOUT);
            return;   // a copy never landed: nothing below may read the stage
        }
        const int skip = sm.skip, slot = sm.slot;
        const int h = u - (u / a.H) * a.H;
        const float b_raw = b_next;
        if (beta_thread && un < U)
            b_next = to_f(((const T *)a.b_raw)[un]);   // lands while this unit computes
        // the next unit's slot id, read while the state moves to registers
        const int slot_next = (warp == PRODUCER && un < U) ? a.slot_ids[un / a.H] : -1;
        StateRegs r;
        if (!skip) {
            // the state: stage -> registers (the thread mapping of state_load)
            const float4 *src =
                reinterpret_cast<const float4 *>(sm.st.state + warp * ROWS_PER_WARP * VD) + lane;
#pragma unroll
            for (int i = 0; i < ROWS_PER_WARP; ++i) r.s[i] = src[i * (VD / 4)];
        }
        __syncthreads();   // the state stage is consumed (and skip / slot read)
        int next_slot = -1;
        if (warp == PRODUCER && un < U) {
            fence_async_shared();
            next_slot = stage_state(a, sm, bar_s, un, slot_next, lane);
        }
        if (!skip) {
            // prologue from the stage; the new conv state goes straight to global memory
            if (warp == 0 || (warp == 1 && half == 0)) {
                const int s = warp == 0 ? half : 2;
                Pack8<T> wp[CONV_W], win[CONV_TAPS], x;
                ld8(sm.st.raw[s] + c0, x);
#pragma unroll
                for (int i = 0; i < CONV_TAPS; ++i) ld8(sm.st.conv[i][s] + c0, win[i]);
#pragma unroll
                for (int i = 0; i < CONV_W; ++i) ld8(sm.st.taps[s] + c0 * CONV_W + i * LANE_CH, wp[i]);
                float y[LANE_CH];
                conv8<T>(wp, win, x, y);
                if (warp == 0) l2norm8<T>(y, a.eps_l2);   // both halves of warp 0
                store8(s == 0 ? sm.qs + c0 : s == 1 ? sm.ks + c0 : sm.vs + c0, y);
                T *cs = (T *)a.conv_state;
#pragma unroll
                for (int i = 0; i < CONV_TAPS; ++i) st8(cs + conv_state_idx(slot, i, s, a.H, h, c0), win[i]);
            } else if (warp == 1) {
                Pack8<T> g;
                ld8(sm.st.gk + c0, g);
                st8(sm.gs + c0, g);
            } else if (warp == 2 && half == 0) {
                Pack8<T> g;
                ld8(sm.st.gate + c0, g);
                st8(sm.gate_s + c0, g);
            } else if (beta_thread) {
                sm.bs[0] = from_f<T>(sigmoid_f(b_raw));
            }
        }
        __syncthreads();   // the small stage is consumed
        if (warp == PRODUCER && un < U) {
            fence_async_shared();
            stage_small(a, sm, bar_x, un, next_slot, lane);
        }
        if (skip) continue;

        // the decode step, exactly as kda_decode_step runs it
        stage_token<T, true>(sm.in, sm.qs, sm.ks, sm.vs, sm.gs, sm.bs);
        __syncthreads();
        const float o = token_update<true>(r, sm.in, sm.red, a.scale);
        if (tid < VD) sm.os[tid] = round_t<T>(o);   // o as the decode step stores it
        state_store(r, a.pool + ((size_t)slot * a.H + h) * STATE_ELEMS);
        __syncthreads();

        // epilogue: gated RMSNorm, one row on the lower half of warp 2
        if (warp == 2) {
            float ov[LANE_CH];
#pragma unroll
            for (int e = 0; e < LANE_CH; ++e) ov[e] = half == 0 ? sm.os[c0 + e] : 0.f;
            const float f = rms_factor(row_sumsq(ov), a.eps_norm);
            if (half == 0) {
                float y[LANE_CH];
#pragma unroll
                for (int e = 0; e < LANE_CH; e += 2) {
                    const float2 r = gated_norm2(make_float2(ov[e], ov[e + 1]), f,
                                                 make_float2(to_f(sm.wn_s[c0 + e]), to_f(sm.wn_s[c0 + e + 1])),
                                                 make_float2(to_f(sm.gate_s[c0 + e]), to_f(sm.gate_s[c0 + e + 1])));
                    y[e] = r.x;
                    y[e + 1] = r.y;
                }
                store8((T *)a.out + (size_t)u * VD + c0, y);
            }
        }
    }
}

template <typename T>
cudaError_t launch_fused(const FusedDecodeArgs &a, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const size_t smem = sizeof(FusedSmem<T>);
    if ((e = set_smem(decode_fused_kernel<T>, smem)) != cudaSuccess) return e;
    const long long units = (long long)a.B * a.H;
    const unsigned grid = (unsigned)(units < 2LL * sms ? units : 2LL * sms);
    decode_fused_kernel<T><<<grid, CTA_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_fused(const FusedDecodeArgs &a, cudaStream_t s) {
    return a.dt == KDA_DTYPE_BF16 ? launch_fused<__nv_bfloat16>(a, s) : launch_fused<float>(a, s);
}

}  // namespace kda
