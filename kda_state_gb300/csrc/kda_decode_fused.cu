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
// kda_gated_rmsnorm.  Every global load of the prologue and epilogue is issued
// at the start, ahead of the 64 KB state load, so the conv runs while the state
// streams in.
//
// Roles: warp 0 runs the conv of q (lanes 0-15) and k (lanes 16-31); warp 1 the
// conv of v (lanes 0-15) and stages gk (lanes 16-31); warp 2 holds the gate and
// norm weight (lanes 0-15) for the epilogue and computes beta (lane 16).
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
__global__ void __launch_bounds__(CTA_THREADS, 2) decode_fused_kernel(FusedDecodeArgs a) {
    __shared__ TokenIn in;
    __shared__ Reduce red;
    __shared__ __align__(16) T qs[KD], ks[KD], vs[VD], gs[KD], gate_s[VD], wn_s[VD];
    __shared__ T bs[1];
    __shared__ __align__(16) float os[VD];
    const int unit = blockIdx.x;
    const int b = unit / a.H, h = unit - b * a.H;
    const int slot = a.slot_ids[b];
    if (slot < 0 || slot >= a.num_slots) {
        if (threadIdx.x == 0 && h == 0) report(a.err, DEVERR_SLOT_RANGE);
        return;
    }
    float *S = a.pool + ((size_t)slot * a.H + h) * STATE_ELEMS;
    StateRegs r;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, half = lane >> 4;
    const int c0 = (lane & 15) * LANE_CH;
    const size_t col = (size_t)h * KD + c0;
    T *cs = (T *)a.conv_state;
    const bool conv = warp == 0 || (warp == 1 && half == 0);
    const int s = warp == 0 ? half : 2;
    Pack8<T> w[CONV_W], win[CONV_TAPS], x;
    if (conv) {
        const T *raw = (const T *)(s == 0 ? a.q_raw : s == 1 ? a.k_raw : a.v_raw);
        ld8(raw + (size_t)b * a.raw_stride + col, x);
#pragma unroll
        for (int i = 0; i < CONV_TAPS; ++i) ld8(cs + conv_state_idx(slot, i, s, a.H, h, c0), win[i]);
        load_taps((const T *)a.conv_w, s, a.H, h, c0, w);
    } else if (warp == 1) {
        Pack8<T> g;
        ld8((const T *)a.gk + (size_t)unit * KD + c0, g);
        st8(gs + c0, g);
    } else if (warp == 2) {
        if (half == 0) {
            Pack8<T> g, n;
            ld8((const T *)a.gate + (size_t)unit * VD + c0, g);
            ld8((const T *)a.w_norm + c0, n);
            st8(gate_s + c0, g);
            st8(wn_s + c0, n);
        } else if (lane == 16) {
            bs[0] = from_f<T>(sigmoid_f(to_f(((const T *)a.b_raw)[unit])));
        }
    }
    // the 64 KB state streams in while the small loads above are consumed
    state_load(r, S);
    if (conv) {
        float y[LANE_CH];
        conv8<T>(w, win, x, y);
        if (warp == 0) l2norm8<T>(y, a.eps_l2);   // both halves of warp 0
        store8(s == 0 ? qs + c0 : s == 1 ? ks + c0 : vs + c0, y);
#pragma unroll
        for (int i = 0; i < CONV_TAPS; ++i) st8(cs + conv_state_idx(slot, i, s, a.H, h, c0), win[i]);
    }
    __syncthreads();

    // the decode step, exactly as kda_decode_step runs it
    stage_token<T, true>(in, qs, ks, vs, gs, bs);
    __syncthreads();
    const float o = token_update<true>(r, in, red, a.scale);
    if (threadIdx.x < VD) os[threadIdx.x] = round_t<T>(o);   // o as the decode step stores it
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
            for (int e = 0; e < LANE_CH; ++e)
                y[e] = gated_norm(ov[e], f, to_f(wn_s[c0 + e]), to_f(gate_s[c0 + e]));
            store8((T *)a.out + (size_t)unit * VD + c0, y);
        }
    }
}

}  // namespace

cudaError_t launch_decode_fused(const FusedDecodeArgs &a, cudaStream_t s) {
    const unsigned grid = (unsigned)a.B * (unsigned)a.H;
    if (a.dt == KDA_DTYPE_BF16)
        decode_fused_kernel<__nv_bfloat16><<<grid, CTA_THREADS, 0, s>>>(a);
    else
        decode_fused_kernel<float><<<grid, CTA_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
