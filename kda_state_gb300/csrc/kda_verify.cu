// Speculative verify of the KDA state library with ReplaySSM input records.
//
// Paper correspondence: "SGLang and Miles Add Day-0 Support for Kimi K3"
// (lmsys.org), "ReplaySSM: raw-input replay for the KDA state": verify reads the
// committed checkpoint, never writes it, and stores each draft step's
// (k, v, gate, beta) into a per-slot ring.
#include "kda_async.cuh"
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

// ---------------------------------------------------------------------------
// verify: G draft tokens from the committed state, which is never written;
// record i goes to ring entry (base + i) mod R of the request's slot.  With
// ragged drafts request b verifies its own G_b <= G tokens, packed by
// cu_drafts; the uniform call is the case cu_drafts[b] = b G.
// ---------------------------------------------------------------------------

// Request b's first token and draft count; false (and an error bit) when the
// ragged offsets are inconsistent.
__device__ __forceinline__ bool draft_span(const VerifyArgs &a, int b, size_t &tok0, int &G) {
    if (!a.cu_drafts) {
        tok0 = (size_t)b * a.G;
        G = a.G;
        return true;
    }
    const int lo = a.cu_drafts[b], hi = a.cu_drafts[b + 1];
    if (lo < 0 || hi < lo || hi - lo > a.G || hi > a.total_tokens) return false;
    tok0 = (size_t)lo;
    G = hi - lo;
    return true;
}

// Recurrent form: the G tokens one after another on a register copy of the
// state (the decode arithmetic).  Used for G > 16 and as the fallback of the
// draft-block form below.
template <typename T>
__device__ __forceinline__ void verify_unit_recurrent(const VerifyArgs &a, int b, int h, int slot,
                                                      size_t tok0, int G, unsigned char *smem) {
    Reduce &red = *reinterpret_cast<Reduce *>(smem);
    TokenIn *in = reinterpret_cast<TokenIn *>(smem + sizeof(Reduce));
    StateRegs r;
    state_load(r, a.pool + ((size_t)slot * a.H + h) * STATE_ELEMS);
    const int base = a.ring_base ? a.ring_base[b] : 0;
    const int mask = a.ring_len - 1;
    for (int i = 0; i < G; ++i) {
        const size_t tok = (tok0 + i) * a.H + h;     // [tokens][H]
        const size_t e = ((size_t)slot * a.ring_len + ((base + i) & mask)) * a.H + h;
        stage_token<T, true>(in[i], (const T *)a.q + tok * KD, (const T *)a.k + tok * KD,
                             (const T *)a.v + tok * VD, (const T *)a.gk + tok * KD,
                             (const T *)a.beta + tok, (T *)a.rk + e * KD, (T *)a.rv + e * VD,
                             a.rdecay + e * KD, a.rbeta + e);
    }
    __syncthreads();
    for (int i = 0; i < G; ++i) {
        const float o = token_update<true>(r, in[i], red, a.scale);
        if (threadIdx.x < VD)
            ((T *)a.o)[((tok0 + i) * a.H + h) * VD + threadIdx.x] = from_f<T>(o);
    }
}

template <typename T>
__global__ void __launch_bounds__(CTA_THREADS, 2) verify_kernel(VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int unit = blockIdx.x;
    const int b = unit / a.H, h = unit - b * a.H;
    size_t tok0;
    int G;
    if (!draft_span(a, b, tok0, G)) {
        if (threadIdx.x == 0 && h == 0) report(a.err, DEVERR_SEQLENS);
        return;
    }
    const int slot = a.slot_ids[b];
    if (slot < 0 || slot >= a.num_slots) {
        if (threadIdx.x == 0 && h == 0) report(a.err, DEVERR_SLOT_RANGE);
        return;
    }
    if (G == 0) return;
    verify_unit_recurrent<T>(a, b, h, slot, tok0, G, smem);
}

// Draft-block form (G <= GM): all G outputs from h0 at once.  With
// E_r = exp(sum_{j<=r} gk_j) (the product of the step decays) per key channel,
//     A[r][j]   = b_r <k_r E_r, k_j / E_j>   (j < r),   T = (I + A)^-1
//     Aqk[r][j] = <q_r E_r, k_j / E_j>       (j <= r)
//     W = T Diag(b) (K . E),  U~ = T Diag(b) V,  U = U~ - W h0
//     O = (Q . E) h0 + Aqk U
// The state is read once; the G x 128 x 128 products with h0 run on the CUDA
// cores in fp32 (2G vectors against the register-resident h0).  A unit whose
// decay over the draft leaves fp32 range for 1/E falls back to the recurrent
// form.  Thread mapping for h0: warp w owns columns 16w .. 16w+15, lane l
// column 16w + (l & 15) and rows 64 (l >> 4) .. + 63.
constexpr int XS = KD + 4;   // padded row stride of W and q . E (conflict-free fragment loads)

constexpr int HS = KD + 8;   // row stride of the staged h0: conflict-free B-fragment loads

// H0S: h0 staged in shared memory by bulk copies (the tensor path), one row
// of 512 bytes per copy into rows HS floats apart.
template <int GM, bool H0S>
struct VerifyBlockSmem {
    float kg[GM][KD];   // k . E
    float kn[GM][KD];   // k / E
    float qg[GM][XS];   // q . E
    float v[GM][VD];
    float w[GM][XS];    // W
    float ut[GM][VD];   // U~
    float akk[GM][GM], aqk[GM][GM], tb[GM][GM];
    float beta[GM];
    int fallback;
    int h0_ok;
    alignas(8) uint64_t bar;
    alignas(16) float h0s[H0S ? KD : 1][HS];
};

// ---------------------------------------------------------------------------
// Block-form phases of one unit.  Each is followed by a block barrier in the
// caller.
// ---------------------------------------------------------------------------
template <int GM, bool H0S>
__device__ __forceinline__ void block_gram(VerifyBlockSmem<GM, H0S> &sm, int G, int warp, int lane) {
    // Gram rows: warp w takes draft rows r = w, w + 8, ...; each lane holds 4
    // channels of k_r E_r and q_r E_r and accumulates the row's products with
    // every k_j / E_j, then one butterfly per product (independent, so they
    // overlap).  A[r][j] = b_r <k_r E_r, k_j / E_j> (j < r), Aqk[r][j] =
    // <q_r E_r, k_j / E_j> (j <= r).
    for (int r = warp; r < G; r += CTA_WARPS) {
        const float4 kr4 = reinterpret_cast<const float4 *>(sm.kg[r])[lane];
        const float4 qr4 = reinterpret_cast<const float4 *>(sm.qg[r])[lane];
        float dk[GM], dq[GM];
#pragma unroll
        for (int j = 0; j < GM; ++j) {
            dk[j] = 0.f;
            dq[j] = 0.f;
            if (j <= r) {
                const float4 y = reinterpret_cast<const float4 *>(sm.kn[j])[lane];
                dk[j] = kr4.x * y.x + kr4.y * y.y + kr4.z * y.z + kr4.w * y.w;
                dq[j] = qr4.x * y.x + qr4.y * y.y + qr4.z * y.z + qr4.w * y.w;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
            for (int j = 0; j < GM; ++j) {
                dk[j] += __shfl_xor_sync(0xffffffffu, dk[j], off);
                dq[j] += __shfl_xor_sync(0xffffffffu, dq[j], off);
            }
        }
        if (lane == 0) {
            const float br = sm.beta[r];
#pragma unroll
            for (int j = 0; j < GM; ++j) {
                if (j < r) sm.akk[r][j] = dk[j] * br;
                if (j <= r) sm.aqk[r][j] = dq[j];
            }
        }
    }
}

template <int GM, bool H0S>
__device__ __forceinline__ void block_solve(VerifyBlockSmem<GM, H0S> &sm, int G, int warp, int lane) {
    // T = (I + A)^-1 by forward substitution (lane = column), then T Diag(b).
    // Each row's entries of A are loaded before its FMA chain (they do not
    // depend on x), so the loads overlap the previous rows' chains.
    if (warp == 0 && lane < G) {
        const int cc = lane;
        float x[GM];
#pragma unroll
        for (int r = 0; r < GM; ++r) x[r] = (r == cc) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < GM; ++r) {
            float ar[GM];
#pragma unroll
            for (int j = 0; j < GM; ++j) ar[j] = (j < r) ? sm.akk[r][j] : 0.f;
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < GM; ++j)
                if (j < r) acc = fmaf(ar[j], x[j], acc);
            if (r < G && r > cc) x[r] = -acc;
        }
        const float bc = sm.beta[cc];
#pragma unroll
        for (int r = 0; r < GM; ++r)
            if (r < G) sm.tb[r][cc] = (r >= cc) ? x[r] * bc : 0.f;
    }
}

template <int GM, bool H0S>
__device__ __forceinline__ void block_wu(VerifyBlockSmem<GM, H0S> &sm, int G, int tid) {
    // W = T Diag(b) (K . E) and U~ = T Diag(b) V, one column per thread
    const int c = tid & (KD - 1);
    const bool do_w = tid < KD;
    for (int r = 0; r < GM; ++r) {
        float acc = 0.f;
        if (r < G)
            for (int j = 0; j <= r; ++j) acc = fmaf(sm.tb[r][j], do_w ? sm.kg[j][c] : sm.v[j][c], acc);
        if (do_w) {
            sm.w[r][c] = acc;
            if (r >= G) sm.qg[r][c] = 0.f;
        } else {
            sm.ut[r][c] = acc;
        }
    }
}

// [W; Q . E] h0 on warp-level TF32 MMAs with h0 from shared memory, then
// U = U~ - W h0 and O = (Q . E) h0 + Aqk U; writes the G output rows.
template <typename T>
__device__ __forceinline__ void block_tensor_out(VerifyBlockSmem<8, true> &sm, const VerifyArgs &a,
                                                 size_t tok0, int G, int h, int warp, int lane) {
    constexpr int GM = 8;
    const int g = lane >> 2, t4 = lane & 3;
    // [W; Q . E] (16 x 128) h0 (128 x 16 columns of this warp): 16 k-steps x
    // 2 n-tiles of m16n8k8 TF32.  Row g of the result is W row g (c[.][0..1])
    // and (Q . E) row g (c[.][2..3]) at columns 16w + 8nt + 2t4 (+1).
    float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
        const int k = 8 * ks + t4;
        const uint32_t af[4] = {tf32_bits(sm.w[g][k]), tf32_bits(sm.qg[g][k]),
                                tf32_bits(sm.w[g][k + 4]), tf32_bits(sm.qg[g][k + 4])};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const float *hb = &sm.h0s[8 * ks + t4][16 * warp + 8 * nt + g];
            const uint32_t bf[2] = {tf32_bits(hb[0]), tf32_bits(hb[4 * HS])};
            mma16n8k8_tf32(c[nt], af, bf);
        }
    }
    // U = U~ - W h0 for row g; O = (Q . E) h0 + Aqk U, U rows from the lanes
    // holding them (lane 4j + t4)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int c0 = 16 * warp + 8 * nt + 2 * t4;
        const float u0 = sm.ut[g][c0] - c[nt][0], u1 = sm.ut[g][c0 + 1] - c[nt][1];
        float o0 = c[nt][2], o1 = c[nt][3];
#pragma unroll
        for (int j = 0; j < GM; ++j) {
            const float uj0 = __shfl_sync(0xffffffffu, u0, 4 * j + t4);
            const float uj1 = __shfl_sync(0xffffffffu, u1, 4 * j + t4);
            if (j <= g && j < G) {
                const float aq = sm.aqk[g][j];
                o0 = fmaf(aq, uj0, o0);
                o1 = fmaf(aq, uj1, o1);
            }
        }
        if (g < G) {
            T *dst = (T *)a.o + ((tok0 + g) * a.H + h) * VD + c0;
            dst[0] = from_f<T>(a.scale * o0);
            dst[1] = from_f<T>(a.scale * o1);
        }
    }
}

template <typename T, int GM>
__global__ void __launch_bounds__(CTA_THREADS, 2) verify_block_kernel(VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr bool TENSOR = (sizeof(T) == 2) && (GM == 8);
    VerifyBlockSmem<GM, TENSOR> &sm = *reinterpret_cast<VerifyBlockSmem<GM, TENSOR> *>(smem);
    const int unit = blockIdx.x;
    const int b = unit / a.H, h = unit - b * a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    size_t tok0;
    int G;
    if (!draft_span(a, b, tok0, G)) {
        if (tid == 0 && h == 0) report(a.err, DEVERR_SEQLENS);
        return;
    }
    const int slot = a.slot_ids[b];
    if (slot < 0 || slot >= a.num_slots) {
        if (tid == 0 && h == 0) report(a.err, DEVERR_SLOT_RANGE);
        return;
    }
    if (G == 0) return;
    // h0 (read-only).  Tensor path (bf16 inputs, G <= 8): 128 bulk copies, one
    // row each, land it in shared memory while the draft is staged and its
    // matrices formed; the m16n8k8 B fragments are read from there.  CUDA-core
    // path: registers, column 16w + (lane & 15), rows 64 (lane >> 4) .. + 63.
    const float *S0 = a.pool + ((size_t)slot * a.H + h) * STATE_ELEMS;
    const int col = 16 * warp + (lane & 15), hr = lane >> 4;
    float s[TENSOR ? 1 : 64];
    const uint32_t bar = shared_addr(&sm.bar);
    if (tid == 0) {
        sm.fallback = 0;   // set by the staging below, after the barrier
        if (TENSOR) {
            barrier_init(bar, 1);
            barrier_expect(bar, (uint32_t)(sizeof(float) * STATE_ELEMS));
        }
    }
    if (!TENSOR) {
#pragma unroll
        for (int i = 0; i < 64; ++i) s[i] = __ldg(S0 + (size_t)(64 * hr + i) * VD + col);
    }
    __syncthreads();   // the reset, and the barrier the h0 copies (issued after the draft's loads) complete on
    const int base = a.ring_base ? a.ring_base[b] : 0;
    const int mask = a.ring_len - 1;
    // stage the draft, store the records; running decay products per channel.
    // All loads of the draft are issued before the first store.
    if (tid < KD) {
        const int c = tid;
        T kr[GM], qr[GM], gr[GM];
#pragma unroll
        for (int i = 0; i < GM; ++i) {
            if (i < G) {
                const size_t tok = (tok0 + i) * a.H + h;
                kr[i] = ((const T *)a.k)[tok * KD + c];
                qr[i] = ((const T *)a.q)[tok * KD + c];
                gr[i] = ((const T *)a.gk)[tok * KD + c];
            }
        }
        // h0 streams in behind the draft (8 KB), which the Gram, the solve and
        // W / U~ need first; only the final product waits for h0
        if (TENSOR) bulk_copy(sm.h0s[c], S0 + (size_t)c * VD, VD * sizeof(float), bar);
        float E = 1.f;
        bool tiny = false;
#pragma unroll
        for (int i = 0; i < GM; ++i) {
            if (i < G) {
                const size_t e = ((size_t)slot * a.ring_len + ((base + i) & mask)) * a.H + h;
                const float alpha = expf(to_f(gr[i]));
                ((T *)a.rk)[e * KD + c] = kr[i];
                a.rdecay[e * KD + c] = alpha;
                E *= alpha;
                tiny |= !(E > 1e-30f && E < 1e30f);   // outside: the recurrent fallback
                const float kk = to_f(kr[i]), qq = to_f(qr[i]);
                sm.kg[i][c] = kk * E;
                sm.kn[i][c] = __fdividef(kk, E);   // used only for E in (1e-30, 1e30): within 2 ulp
                sm.qg[i][c] = qq * E;
            }
        }
        if (tiny) sm.fallback = 1;
    } else {
        const int c = tid - KD;
        T vr[GM], br[GM];
#pragma unroll
        for (int i = 0; i < GM; ++i) {
            if (i < G) {
                const size_t tok = (tok0 + i) * a.H + h;
                vr[i] = ((const T *)a.v)[tok * VD + c];
                if (c == 0) br[i] = ((const T *)a.beta)[tok];
            }
        }
#pragma unroll
        for (int i = 0; i < GM; ++i) {
            if (i < G) {
                const size_t e = ((size_t)slot * a.ring_len + ((base + i) & mask)) * a.H + h;
                ((T *)a.rv)[e * VD + c] = vr[i];
                sm.v[i][c] = to_f(vr[i]);
                if (c == 0) {
                    const float bb = to_f(br[i]);
                    a.rbeta[e] = bb;
                    sm.beta[i] = bb;
                }
            }
        }
    }
    __syncthreads();
    if (sm.fallback) {
        // The records above are the same ones the recurrent form stores; it
        // rewrites them identically.  Its scratch reuses this shared memory,
        // so the h0 copies must have landed first.
        if (TENSOR && tid == 0) sm.h0_ok = barrier_wait(bar, 0);
        __syncthreads();
        if (TENSOR && !sm.h0_ok) {
            if (tid == 0) report(a.err, DEVERR_TIMEOUT);
            return;
        }
        verify_unit_recurrent<T>(a, b, h, slot, tok0, G, smem);
        return;
    }
    block_gram(sm, G, warp, lane);
    __syncthreads();
    block_solve(sm, G, warp, lane);
    __syncthreads();
    block_wu(sm, G, tid);
    if (TENSOR && tid == 0) sm.h0_ok = barrier_wait(bar, 0);   // h0 has landed
    __syncthreads();
    if constexpr (TENSOR) {
        if (!sm.h0_ok) {
            if (tid == 0) report(a.err, DEVERR_TIMEOUT);
            return;
        }
        block_tensor_out<T>(sm, a, tok0, G, h, warp, lane);
    } else {
        // [W; Q . E] h0 for this thread's column: partial over its 64 rows, then
        // the other row half via one shuffle.  acc[i] (i < GM) is row i of W,
        // acc[GM + i] row i of Q . E.
        float acc[2 * GM];
#pragma unroll
        for (int i = 0; i < 2 * GM; ++i) acc[i] = 0.f;
#pragma unroll
        for (int k4 = 0; k4 < 16; ++k4) {
            const int k = 64 * hr + 4 * k4;
#pragma unroll
            for (int i = 0; i < 2 * GM; ++i) {
                if ((i < GM ? i : i - GM) < G) {
                    const float *row = (i < GM) ? sm.w[i] : sm.qg[i - GM];
                    const float4 x = *reinterpret_cast<const float4 *>(row + k);
                    acc[i] = fmaf(x.x, s[4 * k4], acc[i]);
                    acc[i] = fmaf(x.y, s[4 * k4 + 1], acc[i]);
                    acc[i] = fmaf(x.z, s[4 * k4 + 2], acc[i]);
                    acc[i] = fmaf(x.w, s[4 * k4 + 3], acc[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 2 * GM; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 16);
        // U = U~ - W h0;  O = (Q . E) h0 + Aqk U;  each row half writes half the rows
        float u[GM];
#pragma unroll
        for (int r = 0; r < GM; ++r) u[r] = (r < G) ? sm.ut[r][col] - acc[r] : 0.f;
        const int half = (G + 1) / 2;
#pragma unroll
        for (int r = 0; r < GM; ++r) {
            if (r < G && ((r < half) == (hr == 0))) {
                float o = acc[GM + r];
#pragma unroll
                for (int j = 0; j <= r; ++j) o = fmaf(sm.aqk[r][j], u[j], o);
                ((T *)a.o)[((tok0 + r) * a.H + h) * VD + col] = from_f<T>(a.scale * o);
            }
        }
    }
}

}  // namespace

template <typename T, int GM>
cudaError_t launch_verify_block(const VerifyArgs &a, cudaStream_t s) {
    const unsigned grid = (unsigned)a.B * (unsigned)a.H;
    const size_t rec = sizeof(Reduce) + (size_t)a.G * sizeof(TokenIn);   // fallback's needs
    constexpr bool TENSOR = (sizeof(T) == 2) && (GM == 8);
    const size_t blk = sizeof(VerifyBlockSmem<GM, TENSOR>);
    const size_t smem = blk > rec ? blk : rec;
    cudaError_t e = set_smem(verify_block_kernel<T, GM>, smem);
    if (e != cudaSuccess) return e;
    verify_block_kernel<T, GM><<<grid, CTA_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

// The recurrent fallback's scratch (Reduce + G TokenIn) must stay below h0s,
// where copies may be in flight.
cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s) {
    const bool bf = a.dt == KDA_DTYPE_BF16;
    if (a.G <= 8)
        return bf ? launch_verify_block<__nv_bfloat16, 8>(a, s) : launch_verify_block<float, 8>(a, s);
    if (a.G <= 16)
        return bf ? launch_verify_block<__nv_bfloat16, 16>(a, s) : launch_verify_block<float, 16>(a, s);
    const unsigned grid = (unsigned)a.B * (unsigned)a.H;
    const size_t smem = sizeof(Reduce) + (size_t)a.G * sizeof(TokenIn);
    cudaError_t e;
    if (bf) {
        if ((e = set_smem(verify_kernel<__nv_bfloat16>, smem)) != cudaSuccess) return e;
        verify_kernel<__nv_bfloat16><<<grid, CTA_THREADS, smem, s>>>(a);
    } else {
        if ((e = set_smem(verify_kernel<float>, smem)) != cudaSuccess) return e;
        verify_kernel<float><<<grid, CTA_THREADS, smem, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kda
