// Decode step of the KDA state library: one token per (request, head),
// the state updated in place in its slot.
// The (request, head) state of 128 x 128 fp32 lives in the registers of a
// 256-thread CTA and streams from/to HBM with 16-byte coalesced accesses;
// every token goes through the shared kda::token_update() of kda_common.cuh.
//
// Paper correspondence: "SGLang and Miles Add Day-0 Support for Kimi K3"
// (lmsys.org), "Hybrid KDA Memory Management": the working slot is read and
// overwritten by every forward.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

// ---------------------------------------------------------------------------
// decode: one token per (request, head), in place
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(CTA_THREADS, 2) decode_kernel(DecodeArgs a) {
    __shared__ TokenIn in;
    __shared__ Reduce red;
    const int unit = blockIdx.x;
    const int b = unit / a.H, h = unit - b * a.H;
    const int slot = a.slot_ids[b];
    if (slot < 0 || slot >= a.num_slots) {
        if (threadIdx.x == 0 && h == 0) report(a.err, DEVERR_SLOT_RANGE);
        return;
    }
    float *S = a.pool + ((size_t)slot * a.H + h) * STATE_ELEMS;
    StateRegs r;
    state_load(r, S);
    const size_t tk = (size_t)unit * KD, tv = (size_t)unit * VD;
    stage_token<T, true>(in, (const T *)a.q + tk, (const T *)a.k + tk, (const T *)a.v + tv,
                         (const T *)a.gk + tk, (const T *)a.beta + unit);
    __syncthreads();
    const float o = token_update<true>(r, in, red, a.scale);
    if (threadIdx.x < VD) ((T *)a.o)[tv + threadIdx.x] = from_f<T>(o);
    state_store(r, S);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
    const unsigned grid = (unsigned)a.B * (unsigned)a.H;
    if (a.dt == KDA_DTYPE_BF16)
        decode_kernel<__nv_bfloat16><<<grid, CTA_THREADS, 0, s>>>(a);
    else
        decode_kernel<float><<<grid, CTA_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
