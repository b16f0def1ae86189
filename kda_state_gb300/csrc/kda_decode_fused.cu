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
// The shape of kda_decode_step: one 256-thread CTA per (request, head), two per
// SM, the 64 KB state streamed straight into registers with 16-byte coalesced
// loads.  Those loads are issued first, so the conv, the L2 norms and beta run
// while the state is in flight; the CTAs resident beside it overlap their
// transfers with this one's barriers and norm.  Roles: warp 0 runs the conv
// of q (lanes 0-15) and k (lanes 16-31), warp 1 the conv of v (lanes 0-15),
// lane 16 of warp 2 computes beta; the norm epilogue runs on the lower half of
// warp 2.
//
// Paper correspondence: "SGLang and Miles Add Day-0 Support for Kimi K3"
// (lmsys.org), ladder step P5 "Conv + KDA + Onorm Fusion" in "Kernels"; the
// working slot is read and overwritten by every forward ("Hybrid KDA Memory
// Management").
#include "kda_fused_ops.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

template <typename T>
__global__ void __launch_bounds__(CTA_THREADS, 2)
    decode_fused_kernel(const __grid_constant__ FusedDecodeArgs a) {
    __shared__ TokenIn in;
    __shared__ Reduce red;
    __shared__ __align__(16) T qs[KD];
    __shared__ __align__(16) T ks[KD];
    __shared__ __align__(16) T vs[VD];
    __shared__ __align__(16) float os[VD];
    __shared__ T bs[2];
    const int u = blockIdx.x;
    const int b = u / a.H, h = u - b * a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, half = lane >> 4;
    const int c0 = (lane & 15) * LANE_CH;
    const int slot = a.slot_ids[b];
    if (slot < 0 || slot >= a.num_slots) {
        if (tid == 0 && h == 0) report(a.err, DEVERR_SLOT_RANGE);
        return;
    }
    float *S = a.pool + ((size_t)slot * a.H + h) * STATE_ELEMS;
    // The small inputs are requested first and the 64 KB state right after
    // them, so that the conv, the L2 norms and beta run while the state is in
    // flight, and no later step waits for a second round trip: the conv rows
    // (warps 0, 1), gk (threads 0..127), b, gate and the norm weights (warp 2).
    const bool conv_lanes = warp == 0 || (warp == 1 && half == 0);
    const int s = warp == 0 ? half : 2;   // conv stream of the conv lanes: q, k, v
    T *cs = (T *)a.conv_state;
    Pack8<T> wp[CONV_W], win[CONV_TAPS], x;
    if (conv_lanes) {
        const T *raw = (const T *)(s == 0 ? a.q_raw : s == 1 ? a.k_raw : a.v_raw);
        const T *taps = (const T *)a.conv_w + ((size_t)s * a.H + h) * KD * CONV_W + c0 * CONV_W;
        ld8(raw + (size_t)b * a.raw_stride + (size_t)h * KD + c0, x);
#pragma unroll
        for (int i = 0; i < CONV_TAPS; ++i) ld8(cs + conv_state_idx(slot, i, s, a.H, h, c0), win[i]);
#pragma unroll
        for (int i = 0; i < CONV_W; ++i) ld8(taps + i * LANE_CH, wp[i]);
    }
    const T gk_t = tid < KD ? ((const T *)a.gk)[(size_t)u * KD + tid] : from_f<T>(0.f);
    const bool norm_lanes = warp == 2 && half == 0;
    const bool beta_lane = warp == 2 && lane == 16;
    const T b_t = beta_lane ? ((const T *)a.b_raw)[u] : from_f<T>(0.f);
    Pack8<T> gt, wn;
    if (norm_lanes) {
        ld8((const T *)a.gate + (size_t)u * VD + c0, gt);
        ld8((const T *)a.w_norm + c0, wn);
    }
    StateRegs r;
    state_load(r, S);

    // prologue; the new conv state goes straight back to global memory
    if (conv_lanes) {
        float y[LANE_CH];
        conv8<T>(wp, win, x, y);
        if (warp == 0) l2norm8<T>(y, a.eps_l2);   // both halves of warp 0
        store8(s == 0 ? qs + c0 : s == 1 ? ks + c0 : vs + c0, y);
#pragma unroll
        for (int i = 0; i < CONV_TAPS; ++i) st8(cs + conv_state_idx(slot, i, s, a.H, h, c0), win[i]);
    } else if (beta_lane) {
        bs[0] = from_f<T>(sigmoid_f(to_f(b_t)));
    }
    if (tid < KD) in.alpha[tid] = expf(to_f(gk_t));   // exp(gk), as stage_token forms it
    __syncthreads();

    // the decode step, exactly as kda_decode_step runs it (alpha staged above)
    stage_token<T, true, false>(in, qs, ks, vs, nullptr, bs);
    __syncthreads();
    const float o = token_update<true>(r, in, red, a.scale);
    if (tid < VD) os[tid] = round_t<T>(o);   // o as the decode step stores it
    state_store(r, S);
    __syncthreads();

    // epilogue: gated RMSNorm, one row on the lower half of warp 2
    if (warp == 2) {
        float ov[LANE_CH];
#pragma unroll
        for (int e = 0; e < LANE_CH; ++e) ov[e] = half == 0 ? os[c0 + e] : 0.f;
        const float f = rms_factor(row_sumsq(ov), a.eps_norm);
        if (half == 0) {
            float y[LANE_CH];
#pragma unroll
            for (int e = 0; e < LANE_CH; e += 2) {
                const float2 rr = gated_norm2(make_float2(ov[e], ov[e + 1]), f, el2(wn, e / 2), el2(gt, e / 2));
                y[e] = rr.x;
                y[e + 1] = rr.y;
            }
            store8((T *)a.out + (size_t)u * VD + c0, y);
        }
    }
}

template <typename T>
cudaError_t launch_fused(const FusedDecodeArgs &a, cudaStream_t s) {
    const unsigned grid = (unsigned)a.B * (unsigned)a.H;
    decode_fused_kernel<T><<<grid, CTA_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_fused(const FusedDecodeArgs &a, cudaStream_t s) {
    return a.dt == KDA_DTYPE_BF16 ? launch_fused<__nv_bfloat16>(a, s) : launch_fused<float>(a, s);
}

}  // namespace kda
