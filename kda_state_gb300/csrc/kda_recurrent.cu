// CUDA-core kernels of the KDA state library: decode step, speculative verify
// with ReplaySSM input records, the fold over all layers and heads, and the
// exact fp32 prefill.  All of them hold one (request, head) state of
// 128 x 128 fp32 in the registers of a 256-thread CTA and stream it from/to
// HBM with 16-byte coalesced accesses; every token goes through the same
// kda::token_update() (see kda_common.cuh).
//
// Paper correspondence: "SGLang and Miles Add Day-0 Support for Kimi K3"
// (lmsys.org) -- "Hybrid KDA Memory Management" for the in-place slot update,
// "ReplaySSM: raw-input replay for the KDA state" for verify (reads the
// checkpoint, never writes it, stores (k, v, gate, beta) per step) and the
// fold (one launch over all layers and heads, replays only the accepted prefix
// with the stored gate values, overwrites the slot in place).
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

// ---------------------------------------------------------------------------
// verify: G draft tokens from the committed state, which is never written;
// record i goes to ring entry (base + i) mod R of the request's slot.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(CTA_THREADS, 2) verify_kernel(VerifyArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    Reduce &red = *reinterpret_cast<Reduce *>(smem);
    TokenIn *in = reinterpret_cast<TokenIn *>(smem + sizeof(Reduce));
    const int unit = blockIdx.x;
    const int b = unit / a.H, h = unit - b * a.H;
    const int slot = a.slot_ids[b];
    if (slot < 0 || slot >= a.num_slots) {
        if (threadIdx.x == 0 && h == 0) report(a.err, DEVERR_SLOT_RANGE);
        return;
    }
    StateRegs r;
    state_load(r, a.pool + ((size_t)slot * a.H + h) * STATE_ELEMS);
    const int base = a.ring_base ? a.ring_base[b] : 0;
    const int mask = a.ring_len - 1;
    for (int i = 0; i < a.G; ++i) {
        const size_t tok = ((size_t)b * a.G + i) * a.H + h;     // [B][G][H]
        const size_t e = ((size_t)slot * a.ring_len + ((base + i) & mask)) * a.H + h;
        stage_token<T, true>(in[i], (const T *)a.q + tok * KD, (const T *)a.k + tok * KD,
                             (const T *)a.v + tok * VD, (const T *)a.gk + tok * KD,
                             (const T *)a.beta + tok, (T *)a.rk + e * KD, (T *)a.rv + e * VD,
                             a.rdecay + e * KD, a.rbeta + e);
    }
    __syncthreads();
    for (int i = 0; i < a.G; ++i) {
        const float o = token_update<true>(r, in[i], red, a.scale);
        if (threadIdx.x < VD)
            ((T *)a.o)[(((size_t)b * a.G + i) * a.H + h) * VD + threadIdx.x] = from_f<T>(o);
    }
}

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
    for (int i = 0; i < acc; ++i) {
        const size_t e = ((size_t)slot * p.ring_len + ((base + i) & mask)) * p.H + h;
        stage_record<T>(in[i], (const T *)L.rk + e * KD, (const T *)L.rv + e * VD,
                        L.rdecay + e * KD, L.rbeta + e);
    }
    __syncthreads();
    for (int i = 0; i < acc; ++i) token_update<false>(r, in[i], red, 1.f);
    state_store(r, S);
}

// ---------------------------------------------------------------------------
// exact prefill: one CTA per (sequence, head), tokens in order
// ---------------------------------------------------------------------------
constexpr int PREFILL_STAGE = 8;   // tokens staged per round

template <typename T>
__global__ void __launch_bounds__(CTA_THREADS, 2) prefill_rec_kernel(PrefillArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    Reduce &red = *reinterpret_cast<Reduce *>(smem);
    TokenIn *in = reinterpret_cast<TokenIn *>(smem + sizeof(Reduce));
    const int n = blockIdx.x / a.H, h = blockIdx.x - (blockIdx.x / a.H) * a.H;
    const int bos = a.cu[n], eos = a.cu[n + 1];
    if (bos < 0 || eos < bos || eos > a.T_total) {
        if (threadIdx.x == 0 && h == 0) report(a.err, DEVERR_SEQLENS);
        return;
    }
    const int si = a.init_slot[n], so = a.out_slot[n];
    const int ss = a.snap_slot ? a.snap_slot[n] : -1;
    if (si < -1 || si >= a.num_slots || so < 0 || so >= a.num_slots || ss >= a.num_slots) {
        if (threadIdx.x == 0 && h == 0) report(a.err, DEVERR_SLOT_RANGE);
        return;
    }
    StateRegs r;
    if (si >= 0)
        state_load(r, a.pool + ((size_t)si * a.H + h) * STATE_ELEMS);
    else
        state_zero(r);
    for (int t0 = bos; t0 < eos; t0 += PREFILL_STAGE) {
        const int cnt = min(PREFILL_STAGE, eos - t0);
        __syncthreads();   // previous round's inputs are no longer read
        for (int i = 0; i < cnt; ++i) {
            const size_t tok = (size_t)(t0 + i) * a.H + h;
            stage_token<T, true>(in[i], (const T *)a.q + tok * KD, (const T *)a.k + tok * KD,
                                 (const T *)a.v + tok * VD, (const T *)a.gk + tok * KD,
                                 (const T *)a.beta + tok);
        }
        __syncthreads();
        for (int i = 0; i < cnt; ++i) {
            const float o = token_update<true>(r, in[i], red, a.scale);
            if (threadIdx.x < VD)
                ((T *)a.o)[((size_t)(t0 + i) * a.H + h) * VD + threadIdx.x] = from_f<T>(o);
        }
    }
    state_store(r, a.pool + ((size_t)so * a.H + h) * STATE_ELEMS);
    if (ss >= 0) state_store(r, a.pool + ((size_t)ss * a.H + h) * STATE_ELEMS);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
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

cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s) {
    const unsigned grid = (unsigned)a.B * (unsigned)a.H;
    const size_t smem = sizeof(Reduce) + (size_t)a.G * sizeof(TokenIn);
    cudaError_t e;
    if (a.dt == KDA_DTYPE_BF16) {
        if ((e = set_smem(verify_kernel<__nv_bfloat16>, smem)) != cudaSuccess) return e;
        verify_kernel<__nv_bfloat16><<<grid, CTA_THREADS, smem, s>>>(a);
    } else {
        if ((e = set_smem(verify_kernel<float>, smem)) != cudaSuccess) return e;
        verify_kernel<float><<<grid, CTA_THREADS, smem, s>>>(a);
    }
    return cudaGetLastError();
}

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

cudaError_t launch_prefill_recurrent(const PrefillArgs &a, cudaStream_t s) {
    const unsigned grid = (unsigned)a.N * (unsigned)a.H;
    const size_t smem = sizeof(Reduce) + PREFILL_STAGE * sizeof(TokenIn);
    cudaError_t e;
    if (a.dt == KDA_DTYPE_BF16) {
        if ((e = set_smem(prefill_rec_kernel<__nv_bfloat16>, smem)) != cudaSuccess) return e;
        prefill_rec_kernel<__nv_bfloat16><<<grid, CTA_THREADS, smem, s>>>(a);
    } else {
        if ((e = set_smem(prefill_rec_kernel<float>, smem)) != cudaSuccess) return e;
        prefill_rec_kernel<float><<<grid, CTA_THREADS, smem, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kda
