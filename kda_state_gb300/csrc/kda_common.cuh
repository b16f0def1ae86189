// Shared device code of the KDA state library: dtype helpers and the
// per-token CTA update of one 128 x 128 fp32 state held in registers.
//
// The gated delta rule for one token on one (request, head) state S[k][v]:
//     alpha = exp(gk)                    (per key channel k)
//     S'    = Diag(alpha) S              (row k scaled by alpha_k)
//     w     = S'^T k                     (length V)
//     u     = beta (v - w)
//     S     = S' + k u^T
//     o     = scale S^T q = scale (S'^T q + u (k . q))
// ("SGLang and Miles Add Day-0 Support for Kimi K3", "ReplaySSM: raw-input
// replay for the KDA state": per-step inputs (v, k, gk, beta), K = V = 128.)
//
// Decode, verify, fold and the exact fp32 prefill all run token_update() with
// the same CTA shape, so the state arithmetic (explicit round-to-nearest
// intrinsics, fixed reduction order) is identical in all of them; this is what
// makes the fold's committed state bit-identical to repeated decode steps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int KD = 128;
constexpr int VD = 128;
constexpr int STATE_ELEMS = KD * VD;
constexpr int CTA_THREADS = 256;
constexpr int CTA_WARPS = CTA_THREADS / 32;
constexpr int ROWS_PER_WARP = KD / CTA_WARPS;  // 16 rows of the state per warp

enum {
    DEVERR_SLOT_RANGE = 1,
    DEVERR_ACCEPT_RANGE = 2,
    DEVERR_SEQLENS = 4,
    DEVERR_RANGE = 8,
    DEVERR_TIMEOUT = 16
};

__device__ __forceinline__ void report(int32_t *err, int bits) {
    if (err) atomicOr(err, bits);
}

// Checkpoints a prefill unit of len tokens makes: one after every interval
// tokens, at most max_ckpts (interval 0: none).
__device__ __forceinline__ int ckpt_count(int len, int interval, int max_ckpts) {
    return interval > 0 ? min(len / interval, max_ckpts) : 0;
}

// Block-wide check that every checkpoint slot sequence n will use lies in
// [-1, num_slots).  Every thread of the block must call it.
__device__ __forceinline__ bool ckpt_slots_ok(const int32_t *slots, int n, int count,
                                              int max_ckpts, int num_slots) {
    int bad = 0;
    for (int m = threadIdx.x; m < count; m += blockDim.x) {
        const int s = slots[(size_t)n * max_ckpts + m];
        bad |= s < -1 || s >= num_slots;
    }
    return !__syncthreads_or(bad);
}

// fp32 -> tf32 bit pattern, round to nearest.
__device__ __forceinline__ uint32_t tf32_bits(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
// d (16x8, fp32) += a (16x8, tf32, row) * b (8x8, tf32, col): one warp-level MMA.
__device__ __forceinline__ void mma16n8k8_tf32(float (&d)[4], const uint32_t (&a)[4],
                                               const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9},"
        " {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// One token's inputs, staged in shared memory as fp32.
struct TokenIn {
    float alpha[KD];   // exp(gk), exactly as every kernel computes (or stores) it
    float k[KD];
    float q[KD];
    float v[VD];
    float beta;
    float kq_part[4];  // partial dot products k . q of warps 0..3
    float pad[3];
};

// Cross-warp reduction buffers.
struct Reduce {
    float w[CTA_WARPS][VD];
    float p[CTA_WARPS][VD];
    float u[VD];
};

// This thread's slice of the state: rows ROWS_PER_WARP*warp + i, columns
// 4*lane .. 4*lane+3.  A warp reads or writes one full 512-byte row per i.
struct StateRegs {
    float4 s[ROWS_PER_WARP];
};

__device__ __forceinline__ void state_load(StateRegs &r, const float *__restrict__ S) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float4 *p = reinterpret_cast<const float4 *>(S + warp * ROWS_PER_WARP * VD) + lane;
#pragma unroll
    for (int i = 0; i < ROWS_PER_WARP; ++i) r.s[i] = __ldcs(p + i * (VD / 4));
}

__device__ __forceinline__ void state_zero(StateRegs &r) {
#pragma unroll
    for (int i = 0; i < ROWS_PER_WARP; ++i) r.s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ void state_store(const StateRegs &r, float *__restrict__ S) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float4 *p = reinterpret_cast<float4 *>(S + warp * ROWS_PER_WARP * VD) + lane;
#pragma unroll
    for (int i = 0; i < ROWS_PER_WARP; ++i) __stcs(p + i * (VD / 4), r.s[i]);
}

// Stage one token's inputs (threads 0..127 each take one channel).  If rec_*
// pointers are given, the step's record for the ReplaySSM ring is written too:
// k and v as given, exp(gk) and beta as fp32.  Without ALPHA the caller has
// staged in.alpha itself (gk is not read).
template <typename T, bool NEED_Q, bool ALPHA = true>
__device__ __forceinline__ void stage_token(TokenIn &in, const T *__restrict__ q,
                                            const T *__restrict__ k, const T *__restrict__ v,
                                            const T *__restrict__ gk, const T *__restrict__ beta,
                                            T *rec_k = nullptr, T *rec_v = nullptr,
                                            float *rec_decay = nullptr,
                                            float *rec_beta = nullptr) {
    const int t = threadIdx.x;
    if (t < KD) {
        const T kr = k[t], vr = v[t];
        const float kk = to_f(kr);
        in.k[t] = kk;
        in.v[t] = to_f(vr);
        if (ALPHA) {
            const float a = expf(to_f(gk[t]));
            in.alpha[t] = a;
            if (rec_k) rec_decay[t] = a;
        }
        if (rec_k) {
            rec_k[t] = kr;
            rec_v[t] = vr;
        }
        if (NEED_Q) {
            const float qq = to_f(q[t]);
            in.q[t] = qq;
            float d = kk * qq;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            if ((t & 31) == 0) in.kq_part[t >> 5] = d;
        }
        if (t == 0) {
            const float b = to_f(beta[0]);
            in.beta = b;
            if (rec_beta) rec_beta[0] = b;
        }
    }
}

// One token of the recurrence on the CTA's register-resident state.
// Requires every thread of the CTA; `in` must be visible (synchronised).  With
// OUT, threads 0..127 return o[threadIdx.x] (already multiplied by scale).
// The state arithmetic does not depend on OUT.
template <bool OUT>
__device__ __forceinline__ float token_update(StateRegs &r, const TokenIn &in, Reduce &red,
                                              float scale) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float4 wa = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 pa = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < ROWS_PER_WARP; ++i) {
        const int row = warp * ROWS_PER_WARP + i;
        const float a = in.alpha[row];
        const float kk = in.k[row];
        float4 s = r.s[i];
        s.x = __fmul_rn(a, s.x);
        s.y = __fmul_rn(a, s.y);
        s.z = __fmul_rn(a, s.z);
        s.w = __fmul_rn(a, s.w);
        r.s[i] = s;
        wa.x = __fmaf_rn(s.x, kk, wa.x);
        wa.y = __fmaf_rn(s.y, kk, wa.y);
        wa.z = __fmaf_rn(s.z, kk, wa.z);
        wa.w = __fmaf_rn(s.w, kk, wa.w);
        if (OUT) {
            const float qq = in.q[row];
            pa.x = __fmaf_rn(s.x, qq, pa.x);
            pa.y = __fmaf_rn(s.y, qq, pa.y);
            pa.z = __fmaf_rn(s.z, qq, pa.z);
            pa.w = __fmaf_rn(s.w, qq, pa.w);
        }
    }
    reinterpret_cast<float4 *>(red.w[warp])[lane] = wa;
    if (OUT) reinterpret_cast<float4 *>(red.p[warp])[lane] = pa;
    __syncthreads();
    float o = 0.f;
    if (threadIdx.x < VD) {
        const int c = threadIdx.x;
        float ws = red.w[0][c];
#pragma unroll
        for (int j = 1; j < CTA_WARPS; ++j) ws = __fadd_rn(ws, red.w[j][c]);
        const float u = __fmul_rn(in.beta, __fsub_rn(in.v[c], ws));
        red.u[c] = u;
        if (OUT) {
            float ps = red.p[0][c];
#pragma unroll
            for (int j = 1; j < CTA_WARPS; ++j) ps += red.p[j][c];
            const float kq = (in.kq_part[0] + in.kq_part[1]) + (in.kq_part[2] + in.kq_part[3]);
            o = scale * (ps + u * kq);
        }
    }
    __syncthreads();
    const float4 u4 = reinterpret_cast<const float4 *>(red.u)[lane];
#pragma unroll
    for (int i = 0; i < ROWS_PER_WARP; ++i) {
        const float kk = in.k[warp * ROWS_PER_WARP + i];
        float4 s = r.s[i];
        s.x = __fmaf_rn(kk, u4.x, s.x);
        s.y = __fmaf_rn(kk, u4.y, s.y);
        s.z = __fmaf_rn(kk, u4.z, s.z);
        s.w = __fmaf_rn(kk, u4.w, s.w);
        r.s[i] = s;
    }
    return o;
}

// Opt a kernel into more than 48 KB of dynamic shared memory when it needs it.
template <typename Kernel>
cudaError_t set_smem(Kernel kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace kda
