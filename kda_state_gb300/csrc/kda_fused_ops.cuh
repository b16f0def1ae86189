// Device helpers of the fused prologue / epilogue around the recurrence: the
// short causal conv with SiLU, L2 norm, beta sigmoid and gated RMSNorm.
//
// Layout shared by every kernel that computes these steps: a 128-channel row
// (one token and head) is held by 16 consecutive lanes of a warp, lane j of the
// half-warp owning channels 8j .. 8j+7, moved as 16-byte vectors (bf16) or
// pairs of them (fp32).  The arithmetic runs on channel pairs (2p, 2p + 1)
// through the two-wide fp32 instructions (__ffma2_rn, __fmul2_rn, __fadd2_rn):
// each half rounds exactly as the scalar round-to-nearest instruction would, in
// half the issue slots.  A row's sum of squares is two FMA chains over the
// lane's even and odd channels, their sum, and a butterfly over the 16 lanes.
// Explicit round-to-nearest intrinsics leave nothing to be contracted
// differently in two kernels: the fused decode kernel and the unfused prologue
// / norm kernels go through these same helpers, which is what makes them
// bit-identical.
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
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
// sigmoid_f and SiLU on a channel pair (the same operations per half).
__device__ __forceinline__ float2 sigmoid2(float2 x) {
    const float2 e = __fmul2_rn(x, f2(-1.4426950408889634f));
    const float2 d = __fadd2_rn(f2(1.f), make_float2(ex2_approx(e.x), ex2_approx(e.y)));
    return make_float2(rcp_approx(d.x), rcp_approx(d.y));
}
__device__ __forceinline__ float2 silu2(float2 y) { return __fmul2_rn(y, sigmoid2(y)); }

// The value an unfused path would store and read back.
template <typename T>
__device__ __forceinline__ float round_t(float x) {
    return to_f(from_f<T>(x));
}
template <typename T> __device__ __forceinline__ float2 round2(float2 x);
template <> __device__ __forceinline__ float2 round2<float>(float2 x) { return x; }
template <> __device__ __forceinline__ float2 round2<__nv_bfloat16>(float2 x) {
    return __bfloat1622float2(__floats2bfloat162_rn(x.x, x.y));
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
// Elements 2p and 2p + 1.
template <typename T>
__device__ __forceinline__ float2 el2(const Pack8<T> &v, int p) {
    return make_float2(el(v, 2 * p), el(v, 2 * p + 1));
}

// Sum of squares of the row held by this lane's half-warp (every lane of the
// warp must call it; each half-warp reduces its own row).  All 16 lanes of a
// half-warp get the same bits: IEEE addition is commutative, so the two lanes
// of each butterfly pair add the same operands.
__device__ __forceinline__ float row_sumsq(const float (&x)[LANE_CH]) {
    float2 q = __fmul2_rn(make_float2(x[0], x[1]), make_float2(x[0], x[1]));
#pragma unroll
    for (int i = 2; i < LANE_CH; i += 2) {
        const float2 v = make_float2(x[i], x[i + 1]);
        q = __ffma2_rn(v, v, q);
    }
    float p = __fadd_rn(q.x, q.y);
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

// Two channels of the gated RMSNorm output: o r w sigmoid(g), left to right.
__device__ __forceinline__ float2 gated_norm2(float2 o, float r, float2 w, float2 g) {
    return __fmul2_rn(__fmul2_rn(__fmul2_rn(o, f2(r)), w), sigmoid2(g));
}

// Conv state element: [slot][tap][stream][H][K].
__device__ __forceinline__ size_t conv_state_idx(int slot, int tap, int stream, int H, int h, int c) {
    return (((size_t)slot * CONV_TAPS + tap) * 3 + stream) * ((size_t)H * KD) + (size_t)h * KD + c;
}

// The W taps of 8 channels c0 .. c0+7 of one stream and head: 8 x W elements,
// contiguous in conv_w [3][H][K][W] (16-byte aligned); tap i of channel e is
// element (e W + i) of the run.  Kept packed (load_taps) or unpacked once into
// float pairs, w[p][i] = taps i of channels 2p and 2p + 1 (unpack_taps) -- the
// values are the same.
template <typename T>
__device__ __forceinline__ void load_taps(const T *conv_w, int stream, int H, int h, int c0,
                                          Pack8<T> (&w)[CONV_W]) {
    const T *p = conv_w + (((size_t)stream * H + h) * KD + c0) * CONV_W;
#pragma unroll
    for (int i = 0; i < CONV_W; ++i) ld8(p + i * LANE_CH, w[i]);
}
template <typename T>
__device__ __forceinline__ float tap(const Pack8<T> (&w)[CONV_W], int e, int i) {
    return el(w[(e * CONV_W + i) / LANE_CH], (e * CONV_W + i) % LANE_CH);
}
template <typename T>
__device__ __forceinline__ void unpack_taps(const Pack8<T> (&p)[CONV_W], float2 (&w)[LANE_CH / 2][CONV_W]) {
#pragma unroll
    for (int q = 0; q < LANE_CH / 2; ++q)
#pragma unroll
        for (int i = 0; i < CONV_W; ++i) w[q][i] = make_float2(tap(p, 2 * q, i), tap(p, 2 * q + 1, i));
}
template <typename T>
__device__ __forceinline__ float2 tap2(const Pack8<T> (&w)[CONV_W], int p, int i) {
    return make_float2(tap(w, 2 * p, i), tap(w, 2 * p + 1, i));
}
__device__ __forceinline__ float2 tap2(const float2 (&w)[LANE_CH / 2][CONV_W], int p, int i) { return w[p][i]; }

// Conv windows (the W-1 previous raw inputs of 8 channels, oldest first): packed
// rows or float pairs, with the same values.
template <typename T>
__device__ __forceinline__ float2 wget2(const Pack8<T> (&win)[CONV_TAPS], int i, int p) { return el2(win[i], p); }
__device__ __forceinline__ float2 wget2(const float2 (&win)[CONV_TAPS][LANE_CH / 2], int i, int p) {
    return win[i][p];
}
template <typename T>
__device__ __forceinline__ void wshift(Pack8<T> (&win)[CONV_TAPS], const Pack8<T> &x) {
#pragma unroll
    for (int i = 0; i + 1 < CONV_TAPS; ++i) win[i] = win[i + 1];
    win[CONV_TAPS - 1] = x;
}
template <typename T>
__device__ __forceinline__ void wshift(float2 (&win)[CONV_TAPS][LANE_CH / 2], const Pack8<T> &x) {
#pragma unroll
    for (int p = 0; p < LANE_CH / 2; ++p) {
#pragma unroll
        for (int i = 0; i + 1 < CONV_TAPS; ++i) win[i][p] = win[i + 1][p];
        win[CONV_TAPS - 1][p] = el2(x, p);
    }
}

// Causal conv + SiLU of one token on 8 channels: per channel the taps times
// the window (oldest first) then the current input, accumulated by FMA from 0;
// shifts x into the window.  y gets the outputs rounded to T (the stored conv
// output).
template <typename T, typename Taps, typename Win>
__device__ __forceinline__ void conv8(const Taps &w, Win &win, const Pack8<T> &x, float (&y)[LANE_CH]) {
#pragma unroll
    for (int p = 0; p < LANE_CH / 2; ++p) {
        float2 acc = f2(0.f);
#pragma unroll
        for (int i = 0; i < CONV_TAPS; ++i) acc = __ffma2_rn(tap2(w, p, i), wget2(win, i, p), acc);
        acc = __ffma2_rn(tap2(w, p, CONV_TAPS), el2(x, p), acc);
        const float2 r = round2<T>(silu2(acc));
        y[2 * p] = r.x;
        y[2 * p + 1] = r.y;
    }
    wshift(win, x);
}

// L2-normalise a rounded q or k row (every lane of the warp must call it).
template <typename T>
__device__ __forceinline__ void l2norm8(float (&y)[LANE_CH], float eps) {
    const float f = l2_factor(row_sumsq(y), eps);
#pragma unroll
    for (int p = 0; p < LANE_CH / 2; ++p) {
        const float2 v = __fmul2_rn(make_float2(y[2 * p], y[2 * p + 1]), f2(f));
        y[2 * p] = v.x;
        y[2 * p + 1] = v.y;
    }
}

}  // namespace kda
