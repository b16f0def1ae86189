// Exact fp32 prefill of the KDA state library: one CTA per (sequence, head),
// tokens in order, with the optional checkpoints every ckpt_interval tokens.
// The (request, head) state of 128 x 128 fp32 lives in the registers of a
// 256-thread CTA and streams from/to HBM with 16-byte coalesced accesses;
// every token goes through the shared kda::token_update() of kda_common.cuh.
//
// Paper correspondence: the Kimi K3 on B200 deployment notes, timeline entry
// "FlashKDA" (varlen prefill over a [128, 128] fp32 state per sequence and
// head) and item "CuTe FlashKDA prefill" (exact states at fixed boundaries).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

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
    const int nck = ckpt_count(eos - bos, a.ckpt_interval, a.max_ckpts);
    if (si < -1 || si >= a.num_slots || so < 0 || so >= a.num_slots || ss >= a.num_slots ||
        !ckpt_slots_ok(a.ckpt_slots, n, nck, a.max_ckpts, a.num_slots)) {
        if (threadIdx.x == 0 && h == 0) report(a.err, DEVERR_SLOT_RANGE);
        return;
    }
    StateRegs r;
    if (si >= 0)
        state_load(r, a.pool + ((size_t)si * a.H + h) * STATE_ELEMS);
    else
        state_zero(r);
    // a checkpoint interval is a multiple of 64, so checkpoints fall on stage ends
    static_assert(64 % PREFILL_STAGE == 0, "stages must tile a checkpoint interval");
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
        const int done = t0 + cnt - bos;
        if (nck > 0 && done % a.ckpt_interval == 0 && done / a.ckpt_interval <= nck) {
            const int cs = a.ckpt_slots[(size_t)n * a.max_ckpts + done / a.ckpt_interval - 1];
            if (cs >= 0) state_store(r, a.pool + ((size_t)cs * a.H + h) * STATE_ELEMS);
        }
    }
    state_store(r, a.pool + ((size_t)so * a.H + h) * STATE_ELEMS);
    if (ss >= 0) state_store(r, a.pool + ((size_t)ss * a.H + h) * STATE_ELEMS);
}

}  // namespace

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
