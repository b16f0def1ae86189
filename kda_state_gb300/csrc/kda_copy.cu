// Slot copy: dst slot <- src slot in every pool, bit-exact.
//
// The copy-on-write restore of a cached checkpoint into a working slot and the
// snapshot of a working slot at a track boundary are both plain copies enqueued
// on the forward stream, so stream order gives the happens-before ("SGLang and
// Miles Add Day-0 Support for Kimi K3", "Hybrid KDA Memory Management", "Three
// state moves on the forward stream").  HBM-bound: 16-byte loads, all issued
// before the stores, evict-first caching (each byte is touched once).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int COPY_THREADS = 256;
constexpr int COPY_VEC_PER_THREAD = 16;
constexpr size_t COPY_CHUNK = (size_t)COPY_THREADS * COPY_VEC_PER_THREAD * 4;  // floats per CTA

__global__ void __launch_bounds__(COPY_THREADS) slot_copy_kernel(const __grid_constant__ CopyParams p) {
    const int chunk = blockIdx.x % p.chunks_per_copy;
    const int pair = blockIdx.x / p.chunks_per_copy;
    const int pool = pair / p.n, i = pair - pool * p.n;
    const int s = p.src[i], d = p.dst[i];
    if (s < 0 || s >= p.num_slots || d < 0 || d >= p.num_slots) {
        if (threadIdx.x == 0 && chunk == 0 && pool == 0) report(p.err, DEVERR_SLOT_RANGE);
        return;
    }
    const float4 *src = reinterpret_cast<const float4 *>(p.pool[pool] + (size_t)s * p.slot_elems);
    float4 *dst = reinterpret_cast<float4 *>(p.pool[pool] + (size_t)d * p.slot_elems);
    const size_t nvec = p.slot_elems / 4;
    const size_t v0 = (size_t)chunk * (COPY_CHUNK / 4) + threadIdx.x;
    float4 buf[COPY_VEC_PER_THREAD];
#pragma unroll
    for (int j = 0; j < COPY_VEC_PER_THREAD; ++j) {
        const size_t v = v0 + (size_t)j * COPY_THREADS;
        if (v < nvec) buf[j] = __ldcs(src + v);
    }
#pragma unroll
    for (int j = 0; j < COPY_VEC_PER_THREAD; ++j) {
        const size_t v = v0 + (size_t)j * COPY_THREADS;
        if (v < nvec) __stcs(dst + v, buf[j]);
    }
}

}  // namespace

cudaError_t launch_slot_copy(const CopyParams &p_in, cudaStream_t s) {
    CopyParams p = p_in;
    p.chunks_per_copy = (int)((p.slot_elems + COPY_CHUNK - 1) / COPY_CHUNK);
    const size_t grid = (size_t)p.P * p.n * p.chunks_per_copy;
    if (grid == 0) return cudaSuccess;
    if (grid > 0x7fffffffu) return cudaErrorInvalidConfiguration;
    slot_copy_kernel<<<(unsigned)grid, COPY_THREADS, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
