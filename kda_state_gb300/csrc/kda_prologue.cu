// Prologue and epilogue around the KDA recurrence for a packed batch: the short
// causal conv of q, k, v with SiLU and the conv-state update, the L2 norm of q
// and k, beta = sigmoid(b) (one kernel), and the gated RMSNorm of the output
// read at its own strides (another).  Both move 16-byte vectors, 8 channels
// per lane, and reduce each 128-channel row over a half-warp with the helpers
// of kda_fused_ops.cuh.  The prologue streams its raw inputs through a
// per-warp ring of asynchronous copies (cp.async) so that each warp keeps
// PRO_DEPTH - 1 tokens in flight while it computes.
//
// Paper correspondence: Kimi K3 on B200 deployment notes, items "prefill /
// decode kernel fusion" and "other prefill switches": the three conv1d, the
// beta copy + sigmoid and the conv-state gather / write-back fused into one
// kernel, and the output layout copy folded into the gated RMSNorm, each
// bit-exact with the unfused path.
#include "kda_fused_ops.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int PRO_TILE = 64;                  // tokens per CTA
constexpr int PRO_HEADS = 2;                  // heads per CTA
constexpr int PRO_THREADS = 3 * 32;           // warp w: stream w, heads lane / 16
constexpr int PRO_DEPTH = 16;                 // ring slots per warp
constexpr int PRO_TOK = 4;                    // tokens per iteration (independent chains)

// 16-byte asynchronous copy global -> shared (zero-filled when !ok: no global
// read), one commit group per call site, and the wait for all but the newest
// N groups of this thread.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool ok) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(ok ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
template <typename T>
__device__ __forceinline__ void cp_async_pack(Pack8<T> *dst, const T *src, bool ok) {
    static_assert(sizeof(Pack8<T>) % 16 == 0, "16-byte pieces");
#pragma unroll
    for (int i = 0; i < (int)sizeof(Pack8<T>) / 16; ++i)
        cp_async16(reinterpret_cast<uint8_t *>(dst) + 16 * i, reinterpret_cast<const uint8_t *>(src) + 16 * i, ok);
}

// grid: (N x max_tiles, ceil(H / 2)).  The CTA of tile 0 also reads the
// sequence's conv state and writes the new one, so an in-place slot has one
// reader and one writer, both in the same CTA.
template <typename T>
__global__ void __launch_bounds__(PRO_THREADS) conv_prologue_kernel(const PrologueArgs a) {
    const int tile = blockIdx.x % a.max_tiles, n = blockIdx.x / a.max_tiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = warp;
    const int h = blockIdx.y * PRO_HEADS + (lane >> 4);
    const int c0 = (lane & 15) * LANE_CH;
    const bool live = h < a.H;   // a partial last head group leaves some half-warps idle
    const int bos = a.cu[n], eos = a.cu[n + 1];
    if (bos < 0 || eos < bos || eos > a.T_total) {
        if (threadIdx.x == 0 && tile == 0 && blockIdx.y == 0) report(a.err, DEVERR_SEQLENS);
        return;
    }
    const int t0 = bos + tile * PRO_TILE;
    if (tile > 0 && t0 >= eos) return;
    const int si = a.init_slot[n], so = a.out_slot[n];
    if (si < -1 || si >= a.num_slots || so < -1 || so >= a.num_slots) {
        if (threadIdx.x == 0 && tile == 0 && blockIdx.y == 0) report(a.err, DEVERR_SLOT_RANGE);
        return;
    }
    const int cnt = min(PRO_TILE, eos - t0);
    const T *__restrict__ raw = (const T *)(s == 0 ? a.q_raw : s == 1 ? a.k_raw : a.v_raw);
    T *__restrict__ dst = (T *)(s == 0 ? a.q : s == 1 ? a.k : a.v);
    T *cs = (T *)a.conv_state;
    const size_t col = (size_t)(live ? h : 0) * KD + c0;
    const size_t hk = (size_t)a.H * KD;

    // taps and windows unpacked once into channel pairs: every token reuses them
    float2 w[LANE_CH / 2][CONV_W], win[CONV_TAPS][LANE_CH / 2];
    {
        Pack8<T> wp[CONV_W], wn[CONV_TAPS];
#pragma unroll
        for (int i = 0; i < CONV_W; ++i) zero8(wp[i]);
#pragma unroll
        for (int i = 0; i < CONV_TAPS; ++i) zero8(wn[i]);
        if (live) {
            load_taps((const T *)a.conv_w, s, a.H, h, c0, wp);
            if (tile == 0) {
                if (si >= 0)
#pragma unroll
                    for (int i = 0; i < CONV_TAPS; ++i) ld8(cs + conv_state_idx(si, i, s, a.H, h, c0), wn[i]);
            } else {
#pragma unroll
                for (int i = 0; i < CONV_TAPS; ++i)
                    ld8(raw + (size_t)(t0 - CONV_TAPS + i) * a.raw_stride + col, wn[i]);
            }
        }
        unpack_taps(wp, w);
#pragma unroll
        for (int i = 0; i < CONV_TAPS; ++i)
#pragma unroll
            for (int q = 0; q < LANE_CH / 2; ++q) win[i][q] = el2(wn[i], q);
    }
    // Ring of PRO_DEPTH token slots per warp; lane l owns bytes [l, l + 1) x
    // sizeof(Pack8<T>) of every slot and reads back only what it copied, so no
    // lane waits for another.  Tokens go PRO_TOK per iteration (independent
    // chains after the conv); the iteration at token j copies tokens
    // j + PRO_DEPTH - PRO_TOK .. j + PRO_DEPTH - 1 into the slots of tokens
    // j - PRO_TOK .. j - 1, read and consumed by the previous iteration.  A
    // token past the tile is zero-filled, computed and not stored.
    static_assert((PRO_DEPTH & (PRO_DEPTH - 1)) == 0 && PRO_DEPTH > PRO_TOK, "ring");
    __shared__ __align__(16) Pack8<T> ring[PRO_THREADS / 32][PRO_DEPTH][32];
    Pack8<T> (&my)[PRO_DEPTH][32] = ring[warp];
    const T *gsrc = raw + (size_t)t0 * a.raw_stride + col;   // row t0: valid whenever cnt > 0
    const T *gnext = gsrc;
    int jn = 0;   // next token to copy
    auto issue = [&]() {
        const bool ok = live && jn < cnt;
        cp_async_pack<T>(&my[jn & (PRO_DEPTH - 1)][lane], ok ? gnext : gsrc, ok);
        cp_async_commit();
        gnext += a.raw_stride;
        ++jn;
    };
#pragma unroll 1
    for (int j = 0; j < PRO_DEPTH - PRO_TOK && cnt > 0; ++j) issue();   // none for an empty sequence
    T *dptr = dst + (size_t)t0 * hk + col;
#pragma unroll 1
    for (int j = 0; j < cnt; j += PRO_TOK) {   // cnt is uniform across the CTA
#pragma unroll
        for (int u = 0; u < PRO_TOK; ++u) issue();
        cp_async_wait<PRO_DEPTH - PRO_TOK>();   // tokens j .. j + PRO_TOK - 1 have landed
        Pack8<T> x[PRO_TOK];
#pragma unroll
        for (int u = 0; u < PRO_TOK; ++u) x[u] = my[(j + u) & (PRO_DEPTH - 1)][lane];
        float y[PRO_TOK][LANE_CH];
#pragma unroll
        for (int u = 0; u < PRO_TOK; ++u) conv8<T>(w, win, x[u], y[u]);
        if (s < 2) {
#pragma unroll
            for (int u = 0; u < PRO_TOK; ++u) l2norm8<T>(y[u], a.eps);
        }
        if (live) {
#pragma unroll
            for (int u = 0; u < PRO_TOK; ++u)
                if (j + u < cnt) store8(dptr + u * hk, y[u]);
        }
        dptr += PRO_TOK * hk;
    }
    cp_async_wait<0>();
    if (s == 2 && live) {
        for (int i = lane & 15; i < cnt; i += ROW_LANES) {
            const size_t bi = (size_t)(t0 + i) * a.H + h;
            ((T *)a.beta)[bi] = from_f<T>(sigmoid_f(to_f(((const T *)a.b_raw)[bi])));
        }
    }
    if (tile == 0 && so >= 0 && live) {
        // the last W-1 raw inputs of the sequence, from the old state where it
        // is shorter (this CTA is the slot's only reader and writer, and it has
        // not written it yet)
        const int len = eos - bos;
#pragma unroll
        for (int i = 0; i < CONV_TAPS; ++i) {
            const int p = len - CONV_TAPS + i;   // position relative to the sequence start
            Pack8<T> v;
            if (p >= 0)
                ld8(raw + (size_t)(bos + p) * a.raw_stride + col, v);
            else if (si >= 0)
                ld8(cs + conv_state_idx(si, p + CONV_TAPS, s, a.H, h, c0), v);
            else
                zero8(v);
            st8(cs + conv_state_idx(so, i, s, a.H, h, c0), v);
        }
    }
}

// Grid-stride over groups of NORM_PAIRS pairs of (token, head) rows, one row
// per half-warp: all loads of a group are issued before any row is computed,
// so each warp keeps NORM_PAIRS x 1 KB in flight.
constexpr int NORM_PAIRS = 4;

template <typename T>
__global__ void __launch_bounds__(CTA_THREADS) gated_rmsnorm_kernel(const NormArgs a) {
    const int lane = threadIdx.x & 31, c0 = (lane & 15) * LANE_CH;
    const unsigned rows = (unsigned)a.tokens * (unsigned)a.H;   // < 2^31 (checked on the host)
    float wn[LANE_CH];
    load8((const T *)a.w_norm + c0, wn);
    const unsigned nwarps = gridDim.x * (CTA_THREADS / 32);
    for (unsigned grp = blockIdx.x * (CTA_THREADS / 32) + (threadIdx.x >> 5); grp * 2 * NORM_PAIRS < rows;
         grp += nwarps) {
        Pack8<T> ov[NORM_PAIRS], gv[NORM_PAIRS];
        bool live[NORM_PAIRS];
#pragma unroll
        for (int j = 0; j < NORM_PAIRS; ++j) {
            const unsigned row = (grp * NORM_PAIRS + j) * 2 + (lane >> 4);
            live[j] = row < rows;
            if (live[j]) {
                const unsigned t = row / (unsigned)a.H, h = row - t * (unsigned)a.H;
                ld8((const T *)a.o + (size_t)t * a.o_token_stride + (size_t)h * a.o_head_stride + c0, ov[j]);
                ld8((const T *)a.gate + (size_t)row * VD + c0, gv[j]);
            } else {
                zero8(ov[j]);
                zero8(gv[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < NORM_PAIRS; ++j) {
            float o[LANE_CH];
#pragma unroll
            for (int e = 0; e < LANE_CH; ++e) o[e] = el(ov[j], e);
            const float f = rms_factor(row_sumsq(o), a.eps);
            float y[LANE_CH];
#pragma unroll
            for (int e = 0; e < LANE_CH; e += 2) {
                const float2 r = gated_norm2(make_float2(o[e], o[e + 1]), f, make_float2(wn[e], wn[e + 1]),
                                             el2(gv[j], e / 2));
                y[e] = r.x;
                y[e + 1] = r.y;
            }
            if (live[j]) store8((T *)a.out + (size_t)((grp * NORM_PAIRS + j) * 2 + (lane >> 4)) * VD + c0, y);
        }
    }
}

}  // namespace

cudaError_t launch_conv_prologue(const PrologueArgs &a, cudaStream_t s) {
    const dim3 grid((unsigned)(a.N * a.max_tiles), (unsigned)((a.H + PRO_HEADS - 1) / PRO_HEADS));
    if (a.dt == KDA_DTYPE_BF16)
        conv_prologue_kernel<__nv_bfloat16><<<grid, PRO_THREADS, 0, s>>>(a);
    else
        conv_prologue_kernel<float><<<grid, PRO_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gated_rmsnorm(const NormArgs &a, cudaStream_t s) {
    const size_t rows = (size_t)a.tokens * a.H;
    if (rows == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t want = (rows + 16 * NORM_PAIRS - 1) / (16 * NORM_PAIRS);   // 8 warps of 2 x NORM_PAIRS rows
    const size_t cap = (size_t)(sms > 0 ? sms : 152) * 16;
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    if (a.dt == KDA_DTYPE_BF16)
        gated_rmsnorm_kernel<__nv_bfloat16><<<grid, CTA_THREADS, 0, s>>>(a);
    else
        gated_rmsnorm_kernel<float><<<grid, CTA_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
