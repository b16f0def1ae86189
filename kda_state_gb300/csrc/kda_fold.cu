// Fold of the KDA state library: one launch over every (layer, request,
// head) replays the accepted prefix of the stored ReplaySSM records onto the
// committed state, in place.
// The (request, head) state of 128 x 128 fp32 lives in the registers of a
// 256-thread CTA and streams from/to HBM with 16-byte coalesced accesses;
// every token goes through the shared kda::token_update() of kda_common.cuh.
//
// Paper correspondence: "SGLang and Miles Add Day-0 Support for Kimi K3"
// (lmsys.org), "ReplaySSM: raw-input replay for the KDA state": one fold launch
// over all layers and heads, only the accepted prefix replayed, with the gate
// values verify stored, and a state bit-identical to the recurrent baseline.
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

}  // namespace

cudaError_t launch_fold(const FoldParams &p, int dt, cudaStream_t s) {
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
