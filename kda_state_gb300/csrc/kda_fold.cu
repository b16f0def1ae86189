// Fold of the KDA state library: one launch over every (layer, request,
// head) replays the accepted prefix of the stored ReplaySSM records onto the
// committed state, in place.
// The (request, head) state of 128 x 128 fp32 lives in the registers of a
// 256-thread CTA and streams from/to HBM with 16-byte coalesced accesses;
// every token goes through the shared kda::token_update() of kda_common.cuh.
//
// fold_stream_kernel (up to 8 accepted steps, the ReplaySSM window of
// gamma + 1 = 8 drafts) is persistent: each CTA walks units and, while it
// replays one, bulk copies land the next unit's 64 KB state and records in
// shared memory.  fold_kernel loads each unit itself and serves longer
// windows.
//
// Paper correspondence: "SGLang and Miles Add Day-0 Support for Kimi K3"
// (lmsys.org), "ReplaySSM: raw-input replay for the KDA state": one fold launch
// over all layers and heads, only the accepted prefix replayed, with the gate
// values verify stored, and a state bit-identical to the recurrent baseline.
#include "kda_async.cuh"
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

// ---------------------------------------------------------------------------
// fold: one launch over (layer, request, head); replays records 0..a-1
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(CTA_THREADS, 2) fold_kernel(const __grid_constant__ FoldParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    Reduce &red = *reinterpret_cast<Reduce *>(smem);
    TokenIn *in = reinterpret_cast<TokenIn *>(smem + sizeof(Reduce));
    const int per_layer = p.B * p.H;
    const int l = blockIdx.x / per_layer;
    const int rem = blockIdx.x - l * per_layer;
    const int b = rem / p.H, h = rem - b * p.H;
    const int acc = p.accept[b];
    if (acc == 0) return;
    if (acc < 0 || acc > p.max_accept) {
        if (threadIdx.x == 0 && h == 0 && l == 0) report(p.err, DEVERR_ACCEPT_RANGE);
        return;
    }
    const int slot = p.slot_ids[b];
    if (slot < 0 || slot >= p.num_slots) {
        if (threadIdx.x == 0 && h == 0 && l == 0) report(p.err, DEVERR_SLOT_RANGE);
        return;
    }
    const FoldLayer &L = p.layer[l];
    float *S = L.pool + ((size_t)slot * p.H + h) * STATE_ELEMS;
    StateRegs r;
    state_load(r, S);
    const int base = p.ring_base ? p.ring_base[b] : 0;
    const int mask = p.ring_len - 1;
    // stage the records in batches of 8, every load of a batch issued first
    const int t = threadIdx.x;
    if (t < KD) {
        for (int i0 = 0; i0 < acc; i0 += 8) {
            T kr[8], vr[8];
            float dr[8], br[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (i0 + j < acc) {
                    const size_t e = ((size_t)slot * p.ring_len + ((base + i0 + j) & mask)) * p.H + h;
                    kr[j] = ((const T *)L.rk)[e * KD + t];
                    vr[j] = ((const T *)L.rv)[e * VD + t];
                    dr[j] = L.rdecay[e * KD + t];
                    if (t == 0) br[j] = L.rbeta[e];
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (i0 + j < acc) {
                    TokenIn &x = in[i0 + j];
                    x.k[t] = to_f(kr[j]);
                    x.alpha[t] = dr[j];
                    x.v[t] = to_f(vr[j]);
                    if (t == 0) x.beta = br[j];
                }
            }
        }
    }
    __syncthreads();
    for (int i = 0; i < acc; ++i) token_update<false>(r, in[i], red, 1.f);
    state_store(r, S);
}

// ---------------------------------------------------------------------------
// fold, persistent: the next unit's state and records arrive by bulk copy
// ---------------------------------------------------------------------------
constexpr int FOLD_RECS = 8;       // records staged per unit
constexpr int FOLD_PRODUCER = 7;   // the warp that issues the copies

template <typename T>
struct FoldRecs {
    T k[FOLD_RECS][KD];
    T v[FOLD_RECS][VD];
    float decay[FOLD_RECS][KD];
    float beta[FOLD_RECS];
};

template <typename T>
struct FoldSmem {
    float state[STATE_ELEMS];   // the staged unit's state (single buffer)
    FoldRecs<T> rec[2];         // records, double-buffered by unit parity
    TokenIn in[2];
    Reduce red;
    alignas(8) uint64_t bar[2];
    int acc[2], slot[2];        // per buffer: accepted steps (0: nothing to do), slot
    int ok;
};

struct UnitMeta {
    int acc, slot, base;
};

__device__ __forceinline__ void unit_coords(const FoldParams &p, int u, int &l, int &b, int &h) {
    const int per_layer = p.B * p.H;
    l = u / per_layer;
    const int rem = u - l * per_layer;
    b = rem / p.H;
    h = rem - b * p.H;
}

// Lane 0 of the producer: the unit's accept length, slot and ring base.
__device__ __forceinline__ UnitMeta load_meta(const FoldParams &p, int u) {
    int l, b, h;
    unit_coords(p, u, l, b, h);
    UnitMeta m;
    m.acc = p.accept[b];
    m.slot = p.slot_ids[b];
    m.base = p.ring_base ? p.ring_base[b] : 0;
    return m;
}

// The producer warp stages unit u into buffer q: lane 0 arms the barrier (two
// arrivals: the copies' byte count and the betas, which are plain loads), the
// lanes issue one copy each.
template <typename T>
__device__ void fold_stage(const FoldParams &p, FoldSmem<T> &sm, int q, int u, UnitMeta m, int lane) {
    int l, b, h;
    unit_coords(p, u, l, b, h);
    const uint32_t bar = shared_addr(&sm.bar[q]);
    const bool bad_acc = m.acc < 0 || m.acc > p.max_accept;
    const bool bad_slot = m.slot < 0 || m.slot >= p.num_slots;
    const bool live = m.acc > 0 && !bad_acc && !bad_slot;
    if (lane == 0) {
        if (m.acc != 0 && h == 0 && l == 0) {
            if (bad_acc) report(p.err, DEVERR_ACCEPT_RANGE);
            else if (bad_slot) report(p.err, DEVERR_SLOT_RANGE);
        }
        sm.acc[q] = live ? m.acc : 0;
        sm.slot[q] = m.slot;
        if (live) {
            barrier_expect(bar, (uint32_t)(sizeof(float) * STATE_ELEMS +
                                           m.acc * (sizeof(T) * (KD + VD) + sizeof(float) * KD)));
        } else {
            barrier_arrive(bar);
            barrier_arrive(bar);
        }
    }
    __syncwarp();
    if (!live) return;
    const FoldLayer &L = p.layer[l];
    constexpr int PIECE = STATE_ELEMS / 4;
    if (lane < 4)
        bulk_copy(sm.state + lane * PIECE, L.pool + ((size_t)m.slot * p.H + h) * STATE_ELEMS + lane * PIECE,
                  PIECE * 4, bar);
    const int mask = p.ring_len - 1;
    for (int i = lane; i < 3 * m.acc; i += 32) {
        const int j = i / 3, kind = i - 3 * j;
        const size_t e = ((size_t)m.slot * p.ring_len + ((m.base + j) & mask)) * p.H + h;
        if (kind == 0) bulk_copy(sm.rec[q].k[j], (const T *)L.rk + e * KD, KD * sizeof(T), bar);
        else if (kind == 1) bulk_copy(sm.rec[q].v[j], (const T *)L.rv + e * VD, VD * sizeof(T), bar);
        else bulk_copy(sm.rec[q].decay[j], L.rdecay + e * KD, KD * sizeof(float), bar);
    }
    if (lane < m.acc) {
        const size_t e = ((size_t)m.slot * p.ring_len + ((m.base + lane) & mask)) * p.H + h;
        sm.rec[q].beta[lane] = L.rbeta[e];
    }
    __syncwarp();
    if (lane == 0) barrier_arrive(bar);   // the betas are in place
}

template <typename T>
__global__ void __launch_bounds__(CTA_THREADS, 2) fold_stream_kernel(const __grid_constant__ FoldParams p) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    FoldSmem<T> &sm = *reinterpret_cast<FoldSmem<T> *>(smem_raw);
    const int U = p.L * p.B * p.H;
    int u = blockIdx.x;
    if (u >= U) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool producer = warp == FOLD_PRODUCER;
    const int G = gridDim.x;
    if (tid == 0) {
        barrier_init(shared_addr(&sm.bar[0]), 2);
        barrier_init(shared_addr(&sm.bar[1]), 2);
    }
    __syncthreads();
    // metadata of the unit the producer stages next (read one unit ahead)
    UnitMeta next{0, 0, 0};
    if (producer) {
        fold_stage(p, sm, 0, u, load_meta(p, u), lane);
        if (u + G < U) next = load_meta(p, u + G);
    }
    for (int k = 0; u < U; u += G, ++k) {
        const int q = k & 1;
        if (tid == 0) sm.ok = barrier_wait(shared_addr(&sm.bar[q]), (uint32_t)((k >> 1) & 1));
        __syncthreads();
        if (!sm.ok) {
            if (tid == 0) report(p.err, DEVERR_TIMEOUT);
            return;   // a copy never landed: nothing below may read the stage
        }
        const int acc = sm.acc[q], slot = sm.slot[q];
        StateRegs r;
        if (acc > 0) {
            const float4 *src = reinterpret_cast<const float4 *>(sm.state + warp * ROWS_PER_WARP * VD) + lane;
#pragma unroll
            for (int i = 0; i < ROWS_PER_WARP; ++i) r.s[i] = src[i * (VD / 4)];
        }
        __syncthreads();   // the state buffer is consumed; the other record buffer was replayed
        if (producer && u + G < U) {
            fence_async_shared();
            fold_stage(p, sm, q ^ 1, u + G, next, lane);
            if (u + 2 * G < U) next = load_meta(p, u + 2 * G);
        }
        if (acc == 0) continue;
        const FoldRecs<T> &rc = sm.rec[q];
        for (int i = 0; i < acc; ++i) {
            TokenIn &x = sm.in[i & 1];
            if (tid < KD) {
                x.k[tid] = to_f(rc.k[i][tid]);
                x.alpha[tid] = rc.decay[i][tid];
                x.v[tid] = to_f(rc.v[i][tid]);
                if (tid == 0) x.beta = rc.beta[i];
            }
            __syncthreads();
            token_update<false>(r, x, sm.red, 1.f);
        }
        int l, b, h;
        unit_coords(p, u, l, b, h);
        state_store(r, p.layer[l].pool + ((size_t)slot * p.H + h) * STATE_ELEMS);
    }
}

}  // namespace

cudaError_t launch_fold(const FoldParams &p, int dt, cudaStream_t s) {
    bool stream_ok = p.max_accept <= FOLD_RECS;
    for (int l = 0; l < p.L && stream_ok; ++l) {
        const FoldLayer &L = p.layer[l];
        stream_ok = ((uintptr_t)L.rk | (uintptr_t)L.rv | (uintptr_t)L.rdecay | (uintptr_t)L.pool) % 16 == 0;
    }
    if (stream_ok) {
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        const long long units = (long long)p.L * p.B * p.H;
        const unsigned grid = (unsigned)(units < 2LL * sms ? units : 2LL * sms);
        if (dt == KDA_DTYPE_BF16) {
            const size_t smem = sizeof(FoldSmem<__nv_bfloat16>);
            if ((e = set_smem(fold_stream_kernel<__nv_bfloat16>, smem)) != cudaSuccess) return e;
            fold_stream_kernel<__nv_bfloat16><<<grid, CTA_THREADS, smem, s>>>(p);
        } else {
            const size_t smem = sizeof(FoldSmem<float>);
            if ((e = set_smem(fold_stream_kernel<float>, smem)) != cudaSuccess) return e;
            fold_stream_kernel<float><<<grid, CTA_THREADS, smem, s>>>(p);
        }
        return cudaGetLastError();
    }
    const unsigned grid = (unsigned)p.L * (unsigned)p.B * (unsigned)p.H;
    const size_t smem = sizeof(Reduce) + (size_t)p.max_accept * sizeof(TokenIn);
    cudaError_t e;
    if (dt == KDA_DTYPE_BF16) {
        if ((e = set_smem(fold_kernel<__nv_bfloat16>, smem)) != cudaSuccess) return e;
        fold_kernel<__nv_bfloat16><<<grid, CTA_THREADS, smem, s>>>(p);
    } else {
        if ((e = set_smem(fold_kernel<float>, smem)) != cudaSuccess) return e;
        fold_kernel<float><<<grid, CTA_THREADS, smem, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace kda
