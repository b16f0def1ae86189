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

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

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
//     O = (Q . E) h0 + Aqk U = M h0 + N,  M = Q . E - Aqk W,  N = Aqk U~
// M and N depend on the draft alone, so h0 enters one G x 128 x 128 product
// that streams h0 once from L2: a bulk prefetch asks for it when the unit
// starts, and nothing of h0 is staged in shared memory.  For bf16 inputs the
// product runs as warp-level TF32 MMAs (operands rounded to nearest, within the
// bf16 output's bound), for fp32 inputs as fp32 FMAs (the fp32 bound is beyond
// TF32).  A unit whose decay products over the draft leave
// (1e-30, 1e30), where k / E stops being exact in fp32, takes the recurrence
// instead (verify_unit_sliced).
template <int GM>
struct VerifyBlockSmem {
    float kg[GM][KD];   // k . E; in the recurrent path alpha = exp(gk)
    float kn[GM][KD];   // k / E, then N (bf16 inputs); in the recurrent path k
    float qg[GM][KD + 4];   // q . E, then M = Q . E - Aqk W; in the recurrent path q
                            // (rows padded: the MMA product's fragment loads are conflict-free)
    float v[GM][VD];    // v, then the k-half 0 partial of M h0
    float akk[GM][GM], aqk[GM][GM], tb[GM][GM];
    float beta[GM];
    float kq[GM];       // recurrent path: k . q per token
    float red[2][8][32];   // recurrent path: partial sums of S'^T k and S'^T q
    float u[32];
};

// ---------------------------------------------------------------------------
// Block-form phases of one unit.  Each is followed by a block barrier in the
// caller.
// ---------------------------------------------------------------------------
template <int GM>
__device__ __forceinline__ void block_gram(VerifyBlockSmem<GM> &sm, int G, int warp, int lane) {
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
        // Reduce the 2 GM partial sums across the warp by halving: at each step a
        // lane keeps half of its values and adds its partner's copy of that half,
        // so the steps move GM, GM / 2, ... values instead of all 2 GM each time.
        // Afterwards lane l holds the total of value (l >> s) (s = 1 for GM = 8,
        // 0 for GM = 16): values 0 .. GM-1 are dk, GM .. 2GM-1 are dq.
        float v[2 * GM];
#pragma unroll
        for (int j = 0; j < GM; ++j) {
            v[j] = dk[j];
            v[GM + j] = dq[j];
        }
#pragma unroll
        for (int n = 2 * GM, off = 16; n > 1; n >>= 1, off >>= 1) {
            const bool hi = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < n / 2; ++i) {
                const float send = hi ? v[i] : v[i + n / 2];
                const float keep = hi ? v[i + n / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        }
        constexpr int SH = GM == 8 ? 1 : 0;
        if (SH) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
        const int idx = lane >> SH;
        if ((lane & ((1 << SH) - 1)) == 0) {
            if (idx < GM) {
                if (idx < r) sm.akk[r][idx] = v[0] * sm.beta[r];
            } else if (idx - GM <= r) {
                sm.aqk[r][idx - GM] = v[0];
            }
        }
    }
}

template <int GM>
__device__ __forceinline__ void block_solve(VerifyBlockSmem<GM> &sm, int G, int warp, int lane) {
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

// The recurrence over the draft, one 32-column slice of the state at a time
// (the update separates by value column): thread t holds rows 16 (t / 32) ..
// + 15 of column 32 slice + (t % 32).  Its token inputs (alpha, k, q, v, beta,
// k . q) are staged first; o of every token is stored.  Used when the block
// form's k / E would leave fp32's exact range.
template <typename T, int GM>
__device__ __noinline__ void verify_unit_sliced(const VerifyArgs &a, VerifyBlockSmem<GM> &sm, const float *S0,
                                                size_t tok0, int G, int h) {
    const int t = threadIdx.x, cl = t & 31, rg = t >> 5;
    if (t < KD) {
        for (int i = 0; i < G; ++i) {
            const size_t tok = (tok0 + i) * a.H + h;
            const float kk = to_f(((const T *)a.k)[tok * KD + t]);
            const float qq = to_f(((const T *)a.q)[tok * KD + t]);
            sm.kg[i][t] = expf(to_f(((const T *)a.gk)[tok * KD + t]));
            sm.kn[i][t] = kk;
            sm.qg[i][t] = qq;
            float d = kk * qq;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            if ((t & 31) == 0) sm.red[0][t >> 5][i] = d;   // k . q, 4 warps' parts
        }
    }
    __syncthreads();
    if (t < GM && t < G) sm.kq[t] = (sm.red[0][0][t] + sm.red[0][1][t]) + (sm.red[0][2][t] + sm.red[0][3][t]);
    __syncthreads();
    for (int sl = 0; sl < VD / 32; ++sl) {
        const int col = 32 * sl + cl;
        float s[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) s[j] = S0[(size_t)(16 * rg + j) * VD + col];
        for (int i = 0; i < G; ++i) {
            float pw = 0.f, pq = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int kr = 16 * rg + j;
                s[j] *= sm.kg[i][kr];
                pw = fmaf(s[j], sm.kn[i][kr], pw);
                pq = fmaf(s[j], sm.qg[i][kr], pq);
            }
            sm.red[0][rg][cl] = pw;
            sm.red[1][rg][cl] = pq;
            __syncthreads();
            if (rg == 0) {
                float w = 0.f, ps = 0.f;
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    w += sm.red[0][g][cl];
                    ps += sm.red[1][g][cl];
                }
                const float u = sm.beta[i] * (sm.v[i][col] - w);
                sm.u[cl] = u;
                ((T *)a.o)[((tok0 + i) * a.H + h) * VD + col] = from_f<T>(a.scale * (ps + u * sm.kq[i]));
            }
            __syncthreads();
            const float u = sm.u[cl];
#pragma unroll
            for (int j = 0; j < 16; ++j) s[j] = fmaf(sm.kn[i][16 * rg + j], u, s[j]);
        }
    }
}

// o = scale (M h0 + N) on fp32 FMAs (fp32 inputs): thread (column c, half hf)
// sums over rows 64 hf .. 64 hf + 63 of h0, 16 rows' loads in flight at a
// time; each warp load is one 128-byte piece of a row.  Rows of M past G are
// zero.  N is in registers of threads 128..255 (column c).
template <typename T, int GM>
__device__ __forceinline__ void verify_product_fma(const VerifyArgs &a, VerifyBlockSmem<GM> &sm, const float *S0,
                                                   size_t tok0, int G, int h, const float (&n)[GM]) {
    const int tid = threadIdx.x, c = tid & (KD - 1), hf = tid >> 7;
    float acc[GM];
#pragma unroll
    for (int r = 0; r < GM; ++r) acc[r] = 0.f;
    const float *hp = S0 + (size_t)(64 * hf) * VD + c;
#pragma unroll 1
    for (int k16 = 0; k16 < 4; ++k16) {
        float hv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) hv[e] = __ldcs(hp + (size_t)(16 * k16 + e) * VD);
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
            const int kk = 64 * hf + 16 * k16 + 4 * e4;
#pragma unroll
            for (int r = 0; r < GM; ++r) {
                if (r < G) {
                    const float4 m = *reinterpret_cast<const float4 *>(&sm.qg[r][kk]);
                    acc[r] = fmaf(m.x, hv[4 * e4], acc[r]);
                    acc[r] = fmaf(m.y, hv[4 * e4 + 1], acc[r]);
                    acc[r] = fmaf(m.z, hv[4 * e4 + 2], acc[r]);
                    acc[r] = fmaf(m.w, hv[4 * e4 + 3], acc[r]);
                }
            }
        }
    }
    if (hf == 0) {
#pragma unroll
        for (int r = 0; r < GM; ++r) sm.v[r][c] = acc[r];
    }
    __syncthreads();
    if (hf == 1) {
#pragma unroll
        for (int r = 0; r < GM; ++r)
            if (r < G)
                ((T *)a.o)[((tok0 + r) * a.H + h) * VD + c] = from_f<T>(a.scale * ((sm.v[r][c] + acc[r]) + n[r]));
    }
}

// o = scale (M h0 + N) as warp-level TF32 MMAs (bf16 inputs).  Warp w covers
// value columns 32 (w & 3) .. + 31 over key rows 64 (w >> 2) .. + 63, in eight
// k-steps of m16n8k8 (M's rows 0..15 as the A operand, rows past G zero).  The
// warp's 32 columns form four n-tiles whose column n of tile j is value column
// 4 n + j of the group, so lane (g, t4) takes its B operands of all four tiles
// for key row k from one 16-byte load of h0[k][4 g .. 4 g + 3] (each warp load
// reads four whole 128-byte row pieces), and its results for draft row g are
// the group's value columns 8 t4 .. 8 t4 + 7.  The k-half 0 warps leave their
// partial sums in sm.v; the k-half 1 warps add them and N (sm.kn) and store o.
template <typename T, int GM>
__device__ __forceinline__ void verify_product_mma(const VerifyArgs &a, VerifyBlockSmem<GM> &sm, const float *S0,
                                                   size_t tok0, int G, int h, int warp, int lane) {
    static_assert(GM == 8 || GM == 16, "draft rows fill one or two 8-row halves of the A operand");
    const int cg = warp & 3, kh = warp >> 2, g = lane >> 2, t4 = lane & 3;
    const int c0 = 32 * cg;
    float d[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
    const float *hp = S0 + (size_t)(64 * kh + t4) * VD + c0 + 4 * g;
#pragma unroll 1
    for (int s2 = 0; s2 < 4; ++s2) {   // two k-steps per batch: four 16-byte loads in flight
        float4 hb[2][2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            hb[s][0] = __ldcs(reinterpret_cast<const float4 *>(hp + (size_t)(16 * s2 + 8 * s) * VD));
            hb[s][1] = __ldcs(reinterpret_cast<const float4 *>(hp + (size_t)(16 * s2 + 8 * s + 4) * VD));
        }
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int k0 = 64 * kh + 16 * s2 + 8 * s;
            uint32_t af[4];
            af[0] = tf32_bits(sm.qg[g][k0 + t4]);
            af[2] = tf32_bits(sm.qg[g][k0 + t4 + 4]);
            af[1] = GM == 16 ? tf32_bits(sm.qg[(g + 8) % GM][k0 + t4]) : 0u;
            af[3] = GM == 16 ? tf32_bits(sm.qg[(g + 8) % GM][k0 + t4 + 4]) : 0u;
            const float lo[4] = {hb[s][0].x, hb[s][0].y, hb[s][0].z, hb[s][0].w};
            const float hi[4] = {hb[s][1].x, hb[s][1].y, hb[s][1].z, hb[s][1].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t bf[2] = {tf32_bits(lo[j]), tf32_bits(hi[j])};
                mma16n8k8_tf32(d[j], af, bf);
            }
        }
    }
    // this thread's results: rows g (and g + 8), value columns c0 + 8 t4 + e:
    // e < 4 from tile e's first column pair entry, e >= 4 from tile e - 4's second
    float* part0 = &sm.v[g][c0 + 8 * t4];
    if (kh == 0) {
        *reinterpret_cast<float4 *>(part0) = make_float4(d[0][0], d[1][0], d[2][0], d[3][0]);
        *reinterpret_cast<float4 *>(part0 + 4) = make_float4(d[0][1], d[1][1], d[2][1], d[3][1]);
        if (GM == 16) {
            float *p1 = &sm.v[(g + 8) % GM][c0 + 8 * t4];
            *reinterpret_cast<float4 *>(p1) = make_float4(d[0][2], d[1][2], d[2][2], d[3][2]);
            *reinterpret_cast<float4 *>(p1 + 4) = make_float4(d[0][3], d[1][3], d[2][3], d[3][3]);
        }
    }
    __syncthreads();
    if (kh == 1) {
#pragma unroll
        for (int hr = 0; hr < (GM == 16 ? 2 : 1); ++hr) {
            const int r = g + 8 * hr;
            if (r < G) {
                const float *p0 = &sm.v[r][c0 + 8 * t4];
                const float *nn = &sm.kn[r][c0 + 8 * t4];
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float mine = e < 4 ? d[e][2 * hr] : d[e - 4][2 * hr + 1];
                    y[e] = a.scale * ((p0[e] + mine) + nn[e]);
                }
                uint4 w;
                w.x = pack_bf2(y[0], y[1]);
                w.y = pack_bf2(y[2], y[3]);
                w.z = pack_bf2(y[4], y[5]);
                w.w = pack_bf2(y[6], y[7]);
                *reinterpret_cast<uint4 *>((T *)a.o + ((tok0 + r) * a.H + h) * VD + c0 + 8 * t4) = w;
            }
        }
    }
}

template <typename T, int GM>
__global__ void __launch_bounds__(CTA_THREADS, 4) verify_block_kernel(VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    VerifyBlockSmem<GM> &sm = *reinterpret_cast<VerifyBlockSmem<GM> *>(smem);
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
    // h0 (read-only): into L2 now, read once by the final product
    const float *S0 = a.pool + ((size_t)slot * a.H + h) * STATE_ELEMS;
    if (tid < 4) prefetch_l2(S0 + tid * (STATE_ELEMS / 4), STATE_ELEMS);   // four 16 KB requests
    const int base = a.ring_base ? a.ring_base[b] : 0;
    const int mask = a.ring_len - 1;
    // stage the draft, store the records; running decay products per channel.
    // All loads of the draft are issued before the first store.
    bool tiny = false;
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
        float E = 1.f;
#pragma unroll
        for (int i = 0; i < GM; ++i) {
            if (i < G) {
                const size_t e = ((size_t)slot * a.ring_len + ((base + i) & mask)) * a.H + h;
                const float alpha = expf(to_f(gr[i]));
                ((T *)a.rk)[e * KD + c] = kr[i];
                a.rdecay[e * KD + c] = alpha;
                E *= alpha;
                tiny |= !(E > 1e-30f && E < 1e30f);   // outside: the recurrent path
                const float kk = to_f(kr[i]), qq = to_f(qr[i]);
                sm.kg[i][c] = kk * E;
                sm.kn[i][c] = __fdividef(kk, E);   // used only for E in (1e-30, 1e30): within 2 ulp
                sm.qg[i][c] = qq * E;
            }
        }
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
    if (__syncthreads_or(tiny)) {   // uniform
        verify_unit_sliced<T, GM>(a, sm, S0, tok0, G, h);
        return;
    }
    block_gram(sm, G, warp, lane);
    __syncthreads();
    block_solve(sm, G, warp, lane);
    __syncthreads();
    // W and M = Q . E - Aqk W (threads 0..127, column c, M in place of Q . E);
    // U~ and N = Aqk U~ (threads 128..255, column c, N kept in registers)
    const int c = tid & (KD - 1);
    float n[GM];
    if (tid < KD) {
        float w[GM];
#pragma unroll
        for (int r = 0; r < GM; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j <= r; ++j) acc = fmaf(sm.tb[r][j], sm.kg[j][c], acc);
            w[r] = r < G ? acc : 0.f;
        }
#pragma unroll
        for (int r = 0; r < GM; ++r) {
            float m = r < G ? sm.qg[r][c] : 0.f;
#pragma unroll
            for (int j = 0; j <= r; ++j) m = fmaf(-sm.aqk[r][j], w[j], m);
            sm.qg[r][c] = r < G ? m : 0.f;
        }
    } else {
        float ut[GM];
#pragma unroll
        for (int r = 0; r < GM; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j <= r; ++j) acc = fmaf(sm.tb[r][j], sm.v[j][c], acc);
            ut[r] = r < G ? acc : 0.f;
        }
#pragma unroll
        for (int r = 0; r < GM; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j <= r; ++j) acc = fmaf(sm.aqk[r][j], ut[j], acc);
            n[r] = acc;
        }
    }
    if constexpr (sizeof(T) == 2) {
        if (tid >= KD) {
#pragma unroll
            for (int r = 0; r < GM; ++r) sm.kn[r][c] = n[r];   // N, for the threads that store o
        }
        __syncthreads();
        verify_product_mma<T, GM>(a, sm, S0, tok0, G, h, warp, lane);
    } else {
        __syncthreads();
        verify_product_fma<T, GM>(a, sm, S0, tok0, G, h, n);
    }
}

}  // namespace

template <typename T, int GM>
cudaError_t launch_verify_block(const VerifyArgs &a, cudaStream_t s) {
    const unsigned grid = (unsigned)a.B * (unsigned)a.H;
    const size_t smem = sizeof(VerifyBlockSmem<GM>);
    cudaError_t e = set_smem(verify_block_kernel<T, GM>, smem);
    if (e != cudaSuccess) return e;
    verify_block_kernel<T, GM><<<grid, CTA_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

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
