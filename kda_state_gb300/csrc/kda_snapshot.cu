// Snapshot-per-step speculative verify: the baseline that ReplaySSM replaces,
// kept so that the two can be compared on the same workload.
//
// Paper correspondence: "SGLang and Miles Add Day-0 Support for Kimi K3"
// (lmsys.org), "ReplaySSM: raw-input replay for the KDA state": the baseline
// makes a speculative step reversible by saving the whole K x V state after
// every draft step (64 KB per request, layer and head, times the draft length),
// and the accepted length then selects which saved state becomes the slot.
//
// verify_snapshot_kernel runs the draft on a register copy of the committed
// state with the shared per-token update (the decode arithmetic), so snapshot
// i is bit-identical to i + 1 decode steps; it never writes the committed
// state.  snapshot_commit_kernel copies snapshot accept-1 of every layer into
// the request's slot in one launch (accept 0 leaves the slot as it is).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

template <typename T>
__global__ void __launch_bounds__(CTA_THREADS, 2) verify_snapshot_kernel(SnapVerifyArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    Reduce &red = *reinterpret_cast<Reduce *>(smem);
    TokenIn *in = reinterpret_cast<TokenIn *>(smem + sizeof(Reduce));
    const int b = blockIdx.x / a.H, h = blockIdx.x - (blockIdx.x / a.H) * a.H;
    const int slot = a.slot_ids[b], sn = a.snap_ids[b];
    if (slot < 0 || slot >= a.num_slots || sn < 0 || sn >= a.num_snap_slots) {
        if (threadIdx.x == 0 && h == 0) report(a.err, DEVERR_SLOT_RANGE);
        return;
    }
    StateRegs r;
    state_load(r, a.pool + ((size_t)slot * a.H + h) * STATE_ELEMS);
    for (int i = 0; i < a.G; ++i) {
        const size_t tok = ((size_t)b * a.G + i) * a.H + h;     // [B][G][H]
        stage_token<T, true>(in[i], (const T *)a.q + tok * KD, (const T *)a.k + tok * KD,
                             (const T *)a.v + tok * VD, (const T *)a.gk + tok * KD,
                             (const T *)a.beta + tok);
    }
    __syncthreads();
    for (int i = 0; i < a.G; ++i) {
        const float o = token_update<true>(r, in[i], red, a.scale);
        if (threadIdx.x < VD)
            ((T *)a.o)[(((size_t)b * a.G + i) * a.H + h) * VD + threadIdx.x] = from_f<T>(o);
        state_store(r, a.snaps + (((size_t)sn * a.G + i) * a.H + h) * STATE_ELEMS);
    }
}

constexpr int COMMIT_THREADS = 256;
constexpr int COMMIT_VEC = 16;                                           // float4 per thread
constexpr size_t COMMIT_CHUNK = (size_t)COMMIT_THREADS * COMMIT_VEC * 4;  // floats per CTA

// grid: (layer, request, chunk of the request's H states)
__global__ void __launch_bounds__(COMMIT_THREADS)
    snapshot_commit_kernel(const __grid_constant__ SnapCommitParams p) {
    const int chunk = blockIdx.x % p.chunks_per_copy;
    const int lb = blockIdx.x / p.chunks_per_copy;
    const int l = lb / p.B, b = lb - l * p.B;
    const int acc = p.accept[b];
    const int slot = p.slot_ids[b], sn = p.snap_ids[b];
    if (acc < 0 || acc > p.G) {
        if (threadIdx.x == 0 && chunk == 0 && l == 0) report(p.err, DEVERR_ACCEPT_RANGE);
        return;
    }
    if (slot < 0 || slot >= p.num_slots || sn < 0 || sn >= p.num_snap_slots) {
        if (threadIdx.x == 0 && chunk == 0 && l == 0) report(p.err, DEVERR_SLOT_RANGE);
        return;
    }
    if (acc == 0) return;
    const size_t elems = (size_t)p.H * STATE_ELEMS;   // one step's H states are contiguous
    const float4 *src = reinterpret_cast<const float4 *>(
        p.snaps[l] + ((size_t)sn * p.G + (acc - 1)) * elems);
    float4 *dst = reinterpret_cast<float4 *>(p.pool[l] + (size_t)slot * elems);
    const size_t nvec = elems / 4;
    const size_t v0 = (size_t)chunk * (COMMIT_CHUNK / 4) + threadIdx.x;
    float4 buf[COMMIT_VEC];
#pragma unroll
    for (int j = 0; j < COMMIT_VEC; ++j) {
        const size_t v = v0 + (size_t)j * COMMIT_THREADS;
        if (v < nvec) buf[j] = __ldcs(src + v);
    }
#pragma unroll
    for (int j = 0; j < COMMIT_VEC; ++j) {
        const size_t v = v0 + (size_t)j * COMMIT_THREADS;
        if (v < nvec) __stcs(dst + v, buf[j]);
    }
}

}  // namespace

cudaError_t launch_verify_snapshot(const SnapVerifyArgs &a, cudaStream_t s) {
    const unsigned grid = (unsigned)a.B * (unsigned)a.H;
    const size_t smem = sizeof(Reduce) + (size_t)a.G * sizeof(TokenIn);
    cudaError_t e;
    if (a.dt == KDA_DTYPE_BF16) {
        if ((e = set_smem(verify_snapshot_kernel<__nv_bfloat16>, smem)) != cudaSuccess) return e;
        verify_snapshot_kernel<__nv_bfloat16><<<grid, CTA_THREADS, smem, s>>>(a);
    } else {
        if ((e = set_smem(verify_snapshot_kernel<float>, smem)) != cudaSuccess) return e;
        verify_snapshot_kernel<float><<<grid, CTA_THREADS, smem, s>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_snapshot_commit(const SnapCommitParams &p_in, cudaStream_t s) {
    SnapCommitParams p = p_in;
    p.chunks_per_copy = (int)(((size_t)p.H * STATE_ELEMS + COMMIT_CHUNK - 1) / COMMIT_CHUNK);
    const size_t grid = (size_t)p.L * p.B * p.chunks_per_copy;
    if (grid == 0) return cudaSuccess;
    if (grid > 0x7fffffffu) return cudaErrorInvalidConfiguration;
    snapshot_commit_kernel<<<(unsigned)grid, COMMIT_THREADS, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
