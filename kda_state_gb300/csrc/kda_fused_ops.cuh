// Device helpers of the fused prologue / epilogue around the recurrence: the
// short causal conv with SiLU, L2 norm, beta sigmoid and gated RMSNorm.
//
// Layout shared by every kernel that computes these steps: a 128-channel row
// (one token and head) is held by 16 consecutive lanes of a warp, lane j of the
// half-warp owning channels 8j .. 8j+7, moved as 16-byte vectors (bf16) or
// pairs of them (fp32).  A row's sum of squares is a sequential FMA chain over
// the lane's 8 values followed by a butterfly over the 16 lanes, with explicit
// round-to-nearest intrinsics so nothing can be contracted differently in two
// kernels.  The fused decode kernel and the unfused prologue / norm kernels go
// through these same helpers, which is what makes them bit-identical.
#pragma once

#include "kda_common.cuh"
#include "../../include/kda.h"

namespace kda {

constexpr int CONV_W = KDA_CONV_WIDTH;
constexpr int CONV_TAPS = CONV_W - 1;   // raw inputs kept in the conv state
constexpr int ROW_LANES = 16;           // lanes per 128-channel row
constexpr int LANE_CH = 8;              // channels per lane

// exp(-x) as 2^(-x log2 e) (a change of base) on the PTX ex2.approx
// instruction, and 1 / d on rcp.approx: a few instructions, relative error
// near 2^-22.  Every kernel calls these same helpers, so the fused and
// unfused paths stay bit-identical.  For a large negative argument exp(-x)
// overflows to +inf and the reciprocal gives 0, the limit of both functions.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float sigmoid_f(float x) {
    return rcp_approx(__fadd_rn(1.f, ex2_approx(__fmul_rn(x, -1.4426950408889634f))));
}
__device__ __forceinline__ float silu_f(float y) { return __fmul_rn(y, sigmoid_f(y)); }

// The value an unfused path would store and read back.
template <typename T>
__device__ __forceinline__ float round_t(float x) {
    return to_f(from_f<T>(x));
}

// 8 consecutive elements (16-byte aligned) as float.
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&x)[LANE_CH]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void load8(const float *p, float (&x)[LANE_CH]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
// Store 8 values rounded to the element type (16-byte aligned).
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float (&x)[LANE_CH]) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    *reinterpret_cast<uint4 *>(p) = u;
}
__device__ __forceinline__ void store8(float *p, const float (&x)[LANE_CH]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

// 8 consecutive elements kept packed in registers (16 bytes for bf16, 32 for
// fp32) until used; el() unpacks element e (a compile-time index once
// unrolled).
template <typename T> struct Pack8;
template <> struct Pack8<__nv_bfloat16> { uint4 u; };
template <> struct Pack8<float> { float4 a, b; };

__device__ __forceinline__ void ld8(const __nv_bfloat16 *p, Pack8<__nv_bfloat16> &v) {
    v.u = *reinterpret_cast<const uint4 *>(p);
}
__device__ __forceinline__ void ld8(const float *p, Pack8<float> &v) {
    v.a = reinterpret_cast<const float4 *>(p)[0];
    v.b = reinterpret_cast<const float4 *>(p)[1];
}
__device__ __forceinline__ void st8(__nv_bfloat16 *p, const Pack8<__nv_bfloat16> &v) {
    *reinterpret_cast<uint4 *>(p) = v.u;
}
__device__ __forceinline__ void st8(float *p, const Pack8<float> &v) {
    reinterpret_cast<float4 *>(p)[0] = v.a;
    reinterpret_cast<float4 *>(p)[1] = v.b;
}
__device__ __forceinline__ void zero8(Pack8<__nv_bfloat16> &v) { v.u = make_uint4(0, 0, 0, 0); }
__device__ __forceinline__ void zero8(Pack8<float> &v) {
    v.a = make_float4(0.f, 0.f, 0.f, 0.f);
    v.b = v.a;
}
__device__ __forceinline__ float el(const Pack8<__nv_bfloat16> &v, int e) {
    const uint32_t w = e < 2 ? v.u.x : e < 4 ? v.u.y : e < 6 ? v.u.z : v.u.w;
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
}
__device__ __forceinline__ float el(const Pack8<float> &v, int e) {
    return e == 0 ? v.a.x : e == 1 ? v.a.y : e == 2 ? v.a.z : e == 3 ? v.a.w
         : e == 4 ? v.b.x : e == 5 ? v.b.y : e == 6 ? v.b.z : v.b.w;
}

// Causal conv of one channel and SiLU: win[0..W-2] are the previous raw
// inputs, oldest first; x is the current one; w the channel's W taps.
__device__ __forceinline__ float conv_silu(const float *w, const float *win, float x) {
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < CONV_TAPS; ++i) acc = __fmaf_rn(w[i], win[i], acc);
    acc = __fmaf_rn(w[CONV_TAPS], x, acc);
    return silu_f(acc);
}

// Sum of squares of the row held by this lane's half-warp (every lane of the
// warp must call it; each half-warp reduces its own row).  All 16 lanes of a
// half-warp get the same bits: IEEE addition is commutative, so the two lanes
// of each butterfly pair add the same operands.
__device__ __forceinline__ float row_sumsq(const float (&x)[LANE_CH]) {
    float p = __fmul_rn(x[0], x[0]);
#pragma unroll
    for (int i = 1; i < LANE_CH; ++i) p = __fmaf_rn(x[i], x[i], p);
#pragma unroll
    for (int off = ROW_LANES / 2; off > 0; off >>= 1)
        p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, off));
    return p;
}

// 1 / sqrt(sum of squares + eps): the L2-norm factor of q and k.
__device__ __forceinline__ float l2_factor(float ss, float eps) { return rsqrtf(__fadd_rn(ss, eps)); }

// 1 / sqrt(mean of squares + eps) over V channels: the RMSNorm factor (the
// mean is an exact scaling by 2^-7).
__device__ __forceinline__ float rms_factor(float ss, float eps) {
    static_assert(VD == 128, "the mean scales by 2^-7");
    return rsqrtf(__fadd_rn(__fmul_rn(ss, 0.0078125f), eps));
}

// One channel of the gated RMSNorm output.
__device__ __forceinline__ float gated_norm(float o, float r, float w, float g) {
    return __fmul_rn(__fmul_rn(__fmul_rn(o, r), w), sigmoid_f(g));
}

// Conv state element: [slot][tap][stream][H][K].
__device__ __forceinline__ size_t conv_state_idx(int slot, int tap, int stream, int H, int h, int c) {
    return (((size_t)slot * CONV_TAPS + tap) * 3 + stream) * ((size_t)H * KD) + (size_t)h * KD + c;
}

// The W taps of 8 channels c0 .. c0+7 of one stream and head: 8 x W elements,
// contiguous in conv_w [3][H][K][W] (16-byte aligned); tap i of channel e is
// element (e W + i) of the run.  Kept packed (load_taps) or unpacked once into
// floats (unpack_taps) -- the values are the same.
template <typename T>
__device__ __forceinline__ void load_taps(const T *conv_w, int stream, int H, int h, int c0,
                                          Pack8<T> (&w)[CONV_W]) {
    const T *p = conv_w + (((size_t)stream * H + h) * KD + c0) * CONV_W;
#pragma unroll
    for (int i = 0; i < CONV_W; ++i) ld8(p + i * LANE_CH, w[i]);
}
template <typename T>
__device__ __forceinline__ void unpack_taps(const Pack8<T> (&p)[CONV_W], float (&w)[LANE_CH][CONV_W]) {
#pragma unroll
    for (int e = 0; e < LANE_CH; ++e)
#pragma unroll
        for (int i = 0; i < CONV_W; ++i) w[e][i] = el(p[(e * CONV_W + i) / LANE_CH], (e * CONV_W + i) % LANE_CH);
}
template <typename T>
__device__ __forceinline__ float tap(const Pack8<T> (&w)[CONV_W], int e, int i) {
    return el(w[(e * CONV_W + i) / LANE_CH], (e * CONV_W + i) % LANE_CH);
}
__device__ __forceinline__ float tap(const float (&w)[LANE_CH][CONV_W], int e, int i) { return w[e][i]; }

// Conv windows (the W-1 previous raw inputs of 8 channels): packed rows or
// floats, with the same values.
template <typename T>
__device__ __forceinline__ float wget(const Pack8<T> (&win)[CONV_TAPS], int i, int e) { return el(win[i], e); }
__device__ __forceinline__ float wget(const float (&win)[CONV_TAPS][LANE_CH], int i, int e) { return win[i][e]; }
template <typename T>
__device__ __forceinline__ void wshift(Pack8<T> (&win)[CONV_TAPS], const Pack8<T> &x) {
#pragma unroll
    for (int i = 0; i + 1 < CONV_TAPS; ++i) win[i] = win[i + 1];
    win[CONV_TAPS - 1] = x;
}
template <typename T>
__device__ __forceinline__ void wshift(float (&win)[CONV_TAPS][LANE_CH], const Pack8<T> &x) {
#pragma unroll
    for (int e = 0; e < LANE_CH; ++e) {
#pragma unroll
        for (int i = 0; i + 1 < CONV_TAPS; ++i) win[i][e] = win[i + 1][e];
        win[CONV_TAPS - 1][e] = el(x, e);
    }
}

// Conv + SiLU of one token on 8 channels; shifts x into the window.  y gets
// the outputs rounded to T (the stored conv output).
template <typename T, typename Taps, typename Win>
__device__ __forceinline__ void conv8(const Taps &w, Win &win, const Pack8<T> &x, float (&y)[LANE_CH]) {
#pragma unroll
    for (int e = 0; e < LANE_CH; ++e) {
        float wt[CONV_W], wv[CONV_TAPS];
#pragma unroll
        for (int i = 0; i < CONV_W; ++i) wt[i] = tap(w, e, i);
#pragma unroll
        for (int i = 0; i < CONV_TAPS; ++i) wv[i] = wget(win, i, e);
        y[e] = round_t<T>(conv_silu(wt, wv, el(x, e)));
    }
    wshift(win, x);
}

// L2-normalise a rounded q or k row (every lane of the warp must call it).
template <typename T>
__device__ __forceinline__ void l2norm8(float (&y)[LANE_CH], float eps) {
    const float f = l2_factor(row_sumsq(y), eps);
#pragma unroll
    for (int e = 0; e < LANE_CH; ++e) y[e] = __fmul_rn(y[e], f);
}

}  // namespace kda
