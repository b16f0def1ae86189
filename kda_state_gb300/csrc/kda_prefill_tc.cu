// Chunked KDA prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One CTA (512 threads) per (sequence, head) unit walks the sequence in chunks
// of C = 64 tokens.  The pages' FlashKDA fuses a chunk's work and the state
// update into one kernel with intermediates on chip (Kimi K3 on B200 deployment
// notes, timeline entry "FlashKDA"); its CuTe rewrite keeps the fp32 state in
// TMEM and issues the longest sequences first.  Both ideas are kept here; the
// chunk size, the transposed formulation and the two-group pipeline are this
// kernel's own.
//
// Chunk algebra (from the recurrence
//     S_t = (I - b_t k_t k_t^T) Diag(exp(gk_t)) S_{t-1} + b_t k_t v_t^T,  o_t = S_t^T q_t
// unrolled over a chunk).  With G_r = sum_{j<=r} gk_j per key channel, S0 the
// state entering the chunk and G_L the last row's G:
//     A[r][j]  = b_r <k_r, exp(G_r - G_j) . k_j>  (j < r),   T = (I + A)^-1
//     TB       = T Diag(b)
//     U        = TB (V - K~ S0),                 K~ = K . exp(G)
//     O        = Q~ S0 + Aqk U,                  Q~ = Q . exp(G),
//                Aqk[r][j] = <q_r, exp(G_r - G_j) . k_j>  (j <= r)
//     S_L      = Diag(exp(G_L)) S0 + K_end^T U,  K_end = K . exp(G_L - G)
// The pairwise factors exp(G_r - G_j) are split as exp(G_r - G_ref) x
// exp(G_ref - G_j) around the chunk's row 31.
//
// Everything that touches the state is computed transposed, so that every
// state-side product has the 128 value channels on the TMEM lanes:
//     P   = S0^T [K~^T | Q~^T]        (A = fp16 S0^T in TMEM)   -> (K~ S0)^T, and O^T's start
//     U^T = V^T TB^T - (K~ S0)^T TB^T  (A = V^T in shared memory, then -(K~ S0)^T in TMEM)
//     O^T += U^T Aqk^T,  S^T += U^T K_end  (A = fp16 U^T in TMEM)
// and the fp32 state S^T itself lives in TMEM.  The Gram product
// [K e^{G-Gref}; Q e^{G-Gref}] (K e^{Gref-G})^T runs on TF32 (its factors span
// up to exp(+-80)); the other operands are bounded and use fp16.
//
// Two warp groups run a two-stage pipeline over the chunks of the unit:
//   warps 0-7  (intra-chunk): chunk c's cumulative decays, exponentials and
//              operand tiles, the Gram product, and the 64 x 64 unit-lower
//              triangular inverse in 16 x 16 blocks: nothing that depends on
//              the state;
//   warps 8-15 (state): chunk c-1's three state products, their TMEM
//              read-outs, the state pass (checkpoints, the fp16 copy of S^T,
//              the decay of S^T by exp(G_L)) and o.
// Hand-offs are mbarriers, one per buffer parity where a producer can run a
// chunk ahead; every wait is bounded, and a wait that gives up reports
// KDA_DEVERR_TIMEOUT and abandons the unit without writing its slots.
//
// Exactness over the whole input domain: a chunk whose factors or operands
// would leave the formats above (a key channel's log-decay over half a chunk
// beyond 80 in magnitude, a positive gk, |q| or |k| above 256, |v|, T Diag(b),
// Aqk, K~ S0, U or S above 60000) does not use the tensor-core result: the
// state group applies the recurrence to it token by token in fp32 on the CUDA
// cores, from the state entering the chunk, which the tensor-core path has
// not modified when each of these checks is decided.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <numeric>
#include <vector>

#include "kda_async.cuh"
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace tc {

constexpr int C = 64;              // chunk length
constexpr int NT = 512;            // threads per CTA
constexpr int NG = 256;            // threads per warp group
constexpr int BAR_I = 1;           // named barrier of the intra-chunk group
constexpr int BAR_S = 2;           // named barrier of the state group
constexpr int AS = 68;             // row stride (floats) of the fp32 A scratch

// Shared-memory map (byte offsets from a 1024-aligned base).
// R1 [0, 96K): the Gram operands from the prep to the end of the Gram product;
// then the next chunk's raw q, k, gk (TMA) and the triangular-solve scratch.
constexpr uint32_t OP_A1 = 0;          // [Kf; Qr] fp32, 128 rows x 128 ch, K-major A (tf32)
constexpr uint32_t OP_B1 = 65536;      // Kb fp32, 64 rows x 128 ch, K-major B (tf32)
constexpr uint32_t RAW_Q = 0;          // 64 tokens x 128 ch bf16, 2 boxes of 64 ch (TMA)
constexpr uint32_t RAW_K = 16384;
constexpr uint32_t RAW_G = 32768;
constexpr uint32_t SCR_A = 49152;      // fp32 A [64][AS]
constexpr uint32_t SCR_T = 66560;      // fp32 T [64][64], columns swizzled by row
constexpr uint32_t SCR_RW = 82944;     // per-warp 16 x 8 scratch of the block-column solve (6 warps)
constexpr uint32_t R1_END = 98304;
constexpr uint32_t OP_KQ = 98304;      // [K~; Q~] fp16, 128 rows x 128 ch, K-major B of P
constexpr uint32_t OP_V = 131072;      // 2 x v: raw bf16 (TMA), then fp16 in place; MN-major A of U
constexpr uint32_t OP_KE = 163840;     // 2 x K_end fp16, 64 tokens x 128 ch, MN-major B of dS
constexpr uint32_t OP_TB = 196608;     // T Diag(b) fp16 [64 r][64 j], K-major B of U
constexpr uint32_t OP_AQK = 204800;    // Aqk fp16 [64 r][64 j], K-major B of O
constexpr uint32_t SM_BETA = 212992;   // fp32 [2][64], by chunk parity
constexpr uint32_t SM_GAM = 213504;    // fp32 [2][128]: exp(G_L), by chunk parity
constexpr uint32_t SM_FB = 214528;     // recurrent path: 2 x {alpha, k, q, v}[128] fp32
constexpr uint32_t FB_P = SM_FB + 4096;   // its partial sums [2 x pk | 2 x pq][128]
constexpr uint32_t FB_X = SM_FB + 6144;   // [2][4] k.q partials, [2] beta
constexpr uint32_t SM_BAR = SM_FB + 6272;
constexpr uint32_t SM_MISC = SM_BAR + 128;   // TMEM base, flags
constexpr uint32_t SMEM_USED = SM_MISC + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;   // + alignment slack
static_assert(SCR_A + 64 * AS * 4 <= SCR_T && SCR_T + 64 * 64 * 4 <= SCR_RW, "solve scratch overlaps");
static_assert(SCR_RW + 6 * 16 * 8 * 4 <= R1_END, "R scratch misplaced");
static_assert(RAW_G + 16384 <= SCR_A, "raw tiles overlap the solve scratch");
static_assert(OP_KQ % 1024 == 0 && OP_V % 1024 == 0 && OP_KE % 1024 == 0 && OP_TB % 1024 == 0 &&
              OP_AQK % 1024 == 0, "swizzled tiles must be 1024-aligned");
static_assert(OP_AQK + 8192 <= SM_BETA, "tiles overlap");
static_assert(SM_BAR % 8 == 0, "mbarrier alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");

// mbarriers (byte offsets from SM_BAR); MB_V, MB_PREP and MB_TB are pairs, by chunk parity
enum { MB_RAW = 0, MB_V = 8, MB_G1 = 24, MB_PREP = 32, MB_TB = 48, MB_P = 64, MB_U = 72, MB_G4 = 80,
       MB_COUNT = 11 };

// TMEM columns (512 allocated; one CTA per SM)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;       // S^T fp32: lane v, column k
constexpr uint32_t TM_S16 = 128;   // S^T fp16, two k per column: A of P
constexpr uint32_t TM_G1 = 192;    // Gram: lanes 0-63 A rows, 64-127 Aqk rows; 64 columns
constexpr uint32_t TM_KS = 256;    // (K~ S0)^T fp32 [v][token]; then -(K~ S0)^T fp16 (A of U)
constexpr uint32_t TM_U = 320;     // U^T fp32 [v][token]; then fp16 (A of O and dS)
constexpr uint32_t TM_O = 384;     // 2 x O^T fp32 [v][token], by chunk parity

constexpr uint64_t WAIT_NS = 2000000000ull;   // bounded waits: 2 s
constexpr float FP16_LIMIT = 60000.f;         // fp16 operands must stay below this
constexpr float QK_LIMIT = 256.f;             // |q|, |k| bound of the tensor-core path
constexpr float D_LIMIT = 80.f;               // |G_r - G_ref| bound (natural log)

enum { FLAG_TIMEOUT = 1 };

struct Params {
    CUtensorMap tq, tk, tg, tv;
    int N, T_total, H, num_slots, lpt;
    const __nv_bfloat16 *q, *k, *gk, *v, *beta;
    const int32_t *cu;
    float *pool;
    const int32_t *init_slot, *out_slot, *snap_slot;
    __nv_bfloat16 *o;
    float scale;
    int32_t *err;
    int ckpt_chunks, max_ckpts;     // checkpoint every ckpt_chunks chunks (0: none)
    const int32_t *ckpt_slots;
    uint64_t wait_ns;               // limit of every wait
    int skip_first_load;            // self-test: chunk 0's q, k, gk are never requested
    int32_t order[KDA_MAX_LPT_SEQS];
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Named barrier over one warp group.
__device__ __forceinline__ void group_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(NG) : "memory");
}
// Named barrier over one warp group that also ORs a predicate across it: every
// thread of the group gets the same result.
__device__ __forceinline__ bool group_sync_or(int id, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, %2, %3, q;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(NG)
        : "memory");
    return r != 0;
}
// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, fp32 accumulate; fmt 0 = fp16 (kind::f16), 2 = tf32
// (kind::tf32).  A and B always share one format.
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn, int fmt) {
    return (1u << 4) | ((uint32_t)fmt << 7) | ((uint32_t)fmt << 10) | ((uint32_t)a_mn << 15) |
           ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D (TMEM) (+)= A (shared memory) x B (shared memory)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc));
}
// D (TMEM) (+)= A (TMEM: lane = row, two 16-bit k per column, low half first) x B (shared memory)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
        "r"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void mma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// TMEM loads and stores complete inside their own asm statement (the wait is
// part of it): the compiler sees the registers written, or free again, only
// once the asynchronous transfer is done, so no spill or reuse of a register
// can race with it.
#define KDA_TMEM_LD32(taddr, r)                                                                   \
    asm volatile(                                                                                 \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"  \
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"     \
        "tcgen05.wait::ld.sync.aligned;"                                                          \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),            \
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),            \
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])             \
        : "r"(taddr)                                                                              \
        : "memory")
#define KDA_TMEM_ST32(taddr, r)                                                                    \
    asm volatile(                                                                                  \
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"         \
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),                                              \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),    \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),           \
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),         \
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),         \
        "r"(r[29]), "r"(r[30]), "r"(r[31])                                                          \
        : "memory")
#define KDA_TMEM_ST16(taddr, r)                                                                    \
    asm volatile(                                                                                  \
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
        "%14,%15,%16};\n"                                                                         \
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),                                              \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),    \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),           \
        "r"(r[15])                                                                                  \
        : "memory")

// Byte offset of the 16-byte chunk holding columns col..col+7 (col % 8 == 0) of
// row `row` in a tile of `rows` rows x 128 16-bit columns stored as two boxes of
// 64 columns, each box rows x 128 B with the 128-byte swizzle (chunk index
// XOR row % 8).  This is both the TMA SWIZZLE_128B layout of a 64-column box and
// the canonical SW128 operand layout (K-major when columns are K, MN-major when
// columns are M or N).
__device__ __forceinline__ uint32_t chunk_off(int row, int col, int rows) {
    return (uint32_t)((col >> 6) * rows * 128 + row * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4));
}
// Byte offset of the 16-byte chunk holding fp32 columns col..col+3 (col % 4 ==
// 0) of a tile of `rows` rows x 128 fp32 columns stored as four boxes of 32
// columns (rows x 128 B each, 128-byte swizzle).
__device__ __forceinline__ uint32_t chunk32_off(int row, int col, int rows) {
    return (uint32_t)((col >> 5) * rows * 128 + row * 128 + ((((col >> 2) & 7) ^ (row & 7)) << 4));
}
__device__ __forceinline__ void store_f32x8(uint8_t *base, uint32_t tile, int row, int col, int rows,
                                            const float *v8) {
    *reinterpret_cast<float4 *>(base + tile + chunk32_off(row, col, rows)) =
        make_float4(v8[0], v8[1], v8[2], v8[3]);
    *reinterpret_cast<float4 *>(base + tile + chunk32_off(row, col + 4, rows)) =
        make_float4(v8[4], v8[5], v8[6], v8[7]);
}
__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ void store_f16(uint8_t *base, uint32_t off, const float *v8) {
    *reinterpret_cast<uint4 *>(base + off) =
        make_uint4(pack_f16x2(v8[0], v8[1]), pack_f16x2(v8[2], v8[3]), pack_f16x2(v8[4], v8[5]),
                   pack_f16x2(v8[6], v8[7]));
}
__device__ __forceinline__ void unpack_bf16(const uint4 &w, float *v8) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v8[2 * i] = f.x;
        v8[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ float bf16_to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
// 2^x on the special-function unit (one MUFU op; relative error ~2^-22, far
// below the fp16 / tf32 rounding of the operands it feeds).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Bounded wait of one thread; a wait that gives up raises the CTA's timeout flag.
__device__ __forceinline__ void wait_or_flag(uint32_t bar, uint32_t parity, uint64_t limit, int *flags) {
    if (!barrier_wait_for(bar, parity, limit)) atomicOr(flags, FLAG_TIMEOUT);
}
__device__ __forceinline__ bool timed_out(const int *flags) {
    return (*reinterpret_cast<const volatile int *>(flags) & FLAG_TIMEOUT) != 0;
}

// ---------------------------------------------------------------------------
// 64 x 64 unit-lower-triangular inverse, off-diagonal blocks.
// A is fp32 [64][AS] (strictly lower, rows scaled by beta); T is fp32 [64][64]
// with its columns XOR-swizzled by row: T[r][c] lives at r*64 + tsw(r, c).
// Block column J belongs to two warps (8 columns each): for I = J+1 .. 3 they form
//     R = sum_{K=J}^{I-1} A_IK T_KJ,   T_IJ = -T_II R
// from blocks of lower levels only, so the warps need no group-wide barrier.
// The 16 x 16 x 16 products run as warp-level m16n8k8 TF32 MMAs (fp32
// accumulate): they are latency-bound and far below the 64-row minimum of the
// 5th-generation MMA.  T Diag(b) is stored in fp16 as the B operand of U.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int tsw(int r, int c) { return c ^ ((r & 3) << 3); }
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32_warp(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9},"
        " {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
constexpr int RW = 8;    // row stride (floats) of a warp's 16 x 8 R scratch

// Magnitude bound of a stored fp16 operand value: |x|, or a value above every
// limit when x is NaN.
__device__ __forceinline__ float mag(float x) { return x == x ? fabsf(x) : 3.0e38f; }

// T Diag(beta) element pair (r, c), (r, c + 1), c even, as fp16 into the
// K-major TB tile (64 token columns, one 128-byte row per r); returns the
// larger magnitude.
__device__ __forceinline__ float store_tb2(uint8_t *tb, int r, int c, float t0, float t1, const float *beta) {
    const float a = t0 * beta[c], b = t1 * beta[c + 1];
    *reinterpret_cast<uint32_t *>(tb + r * 128 + ((((c >> 3) ^ r) & 7) << 4) + (c & 7) * 2) =
        pack_f16x2(a, b);
    return fmaxf(mag(a), mag(b));
}

template <int J>
__device__ __forceinline__ float solve_block_column(const float *As, float *Ts, float *Rw, int lane,
                                                    uint8_t *tb, const float *beta, int nt) {
    // This warp owns the 8 columns 16J + 8nt .. +7 of block column J; the two
    // halves of a block column never read each other's results.
    const int g = lane >> 2, t4 = lane & 3;
    float bound = 0.f;
#pragma unroll
    for (int I = J + 1; I < 4; ++I) {
        float rc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int K = J; K < I; ++K) {
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const float *ar = As + (16 * I + g) * AS + 16 * K + 8 * ks + t4;
                const uint32_t a[4] = {to_tf32(ar[0]), to_tf32(ar[8 * AS]), to_tf32(ar[4]),
                                       to_tf32(ar[8 * AS + 4])};
                const int rr = 16 * K + 8 * ks + t4;   // rr % 4 == t4, also for rr + 4
                const int cc = (16 * J + 8 * nt + g) ^ (t4 << 3);
                const uint32_t b[2] = {to_tf32(Ts[rr * 64 + cc]), to_tf32(Ts[(rr + 4) * 64 + cc])};
                mma_tf32_warp(rc, a, b);
            }
        }
        Rw[g * RW + 2 * t4] = rc[0];
        Rw[g * RW + 2 * t4 + 1] = rc[1];
        Rw[(g + 8) * RW + 2 * t4] = rc[2];
        Rw[(g + 8) * RW + 2 * t4 + 1] = rc[3];
        __syncwarp();
        float tc[4] = {0.f, 0.f, 0.f, 0.f};
        const int sw = (g & 3) << 3;   // swizzle of rows 16I + g and 16I + g + 8
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const int c0 = (16 * I + 8 * ks + t4) ^ sw, c1 = (16 * I + 8 * ks + t4 + 4) ^ sw;
            const uint32_t a[4] = {to_tf32(Ts[(16 * I + g) * 64 + c0]), to_tf32(Ts[(16 * I + g + 8) * 64 + c0]),
                                   to_tf32(Ts[(16 * I + g) * 64 + c1]), to_tf32(Ts[(16 * I + g + 8) * 64 + c1])};
            const uint32_t b[2] = {to_tf32(Rw[(8 * ks + t4) * RW + g]), to_tf32(Rw[(8 * ks + t4 + 4) * RW + g])};
            mma_tf32_warp(tc, a, b);
        }
        const int cl = 16 * J + 8 * nt + 2 * t4;
        const int c = cl ^ sw;
        Ts[(16 * I + g) * 64 + c] = -tc[0];
        Ts[(16 * I + g) * 64 + c + 1] = -tc[1];
        Ts[(16 * I + g + 8) * 64 + c] = -tc[2];
        Ts[(16 * I + g + 8) * 64 + c + 1] = -tc[3];
        bound = fmaxf(bound, store_tb2(tb, 16 * I + g, cl, -tc[0], -tc[1], beta));
        bound = fmaxf(bound, store_tb2(tb, 16 * I + g + 8, cl, -tc[2], -tc[3], beta));
        __syncwarp();
    }
    return bound;
}

// 32 columns of an O^T buffer (lane v, tokens tok0 .. tok0 + 31 of the unit's
// head), scaled and stored as bf16 for the first nvalid tokens.
__device__ __forceinline__ void store_o_cols(const Params &p, uint32_t taddr, int tok0, int nvalid, int h,
                                             int v) {
    uint32_t r[32];
    KDA_TMEM_LD32(taddr, r);
    __nv_bfloat16 *dst = p.o + ((size_t)tok0 * p.H + h) * VD + v;
    const size_t stride = (size_t)p.H * VD;
    const float sc = p.scale;
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (j < nvalid) dst[j * stride] = __float2bfloat16_rn(sc * __uint_as_float(r[j]));
}

// The recurrence over one chunk on the CUDA cores, in fp32, run by the state
// group: this thread's S[64 hh + j][v] (j < 64) is read from TMEM S^T on entry
// and written back on exit; o of every token is stored.
__device__ __noinline__ void chunk_recurrent(const Params &p, uint8_t *sm, uint32_t lb, int t0, int L, int h,
                                             int st, int v, int hh) {
    const int lane = st & 31, sw = st >> 5;
    float *part = reinterpret_cast<float *>(sm + FB_P);        // [2 pk | 2 pq][128]
    float *xs = reinterpret_cast<float *>(sm + FB_X);          // [2][4] k.q partials, [2] beta
    float s[64];
    KDA_TMEM_LD32(lb + TM_S + 64 * hh, reinterpret_cast<uint32_t *>(s));
    KDA_TMEM_LD32(lb + TM_S + 64 * hh + 32, (reinterpret_cast<uint32_t *>(s) + 32));
    for (int t = 0; t < L; ++t) {
        const int tg = t0 + t, b = t & 1;
        float *fb = reinterpret_cast<float *>(sm + SM_FB + b * 2048);   // alpha, k, q, v
        const size_t row = ((size_t)tg * p.H + h) * KD;
        if (st < 128) {
            const float g = bf16_to_f(p.gk[row + st]);
            const float kk = bf16_to_f(p.k[row + st]), qq = bf16_to_f(p.q[row + st]);
            fb[st] = expf(g);
            fb[128 + st] = kk;
            fb[256 + st] = qq;
            float kq = kk * qq;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
            if (lane == 0) xs[b * 4 + sw] = kq;
        } else {
            fb[384 + st - 128] = bf16_to_f(p.v[((size_t)tg * p.H + h) * VD + st - 128]);
            if (st == 128) xs[8 + b] = bf16_to_f(p.beta[(size_t)tg * p.H + h]);
        }
        group_sync(BAR_S);
        float pk = 0.f, pq = 0.f;
        const float4 *al = reinterpret_cast<const float4 *>(fb + 64 * hh);
        const float4 *kv = reinterpret_cast<const float4 *>(fb + 128 + 64 * hh);
        const float4 *qv = reinterpret_cast<const float4 *>(fb + 256 + 64 * hh);
#pragma unroll
        for (int j4 = 0; j4 < 16; ++j4) {
            const float4 a = al[j4], kk = kv[j4], qq = qv[j4];
            s[4 * j4] *= a.x; s[4 * j4 + 1] *= a.y; s[4 * j4 + 2] *= a.z; s[4 * j4 + 3] *= a.w;
            pk = fmaf(s[4 * j4], kk.x, pk); pk = fmaf(s[4 * j4 + 1], kk.y, pk);
            pk = fmaf(s[4 * j4 + 2], kk.z, pk); pk = fmaf(s[4 * j4 + 3], kk.w, pk);
            pq = fmaf(s[4 * j4], qq.x, pq); pq = fmaf(s[4 * j4 + 1], qq.y, pq);
            pq = fmaf(s[4 * j4 + 2], qq.z, pq); pq = fmaf(s[4 * j4 + 3], qq.w, pq);
        }
        part[hh * 128 + v] = pk;
        part[256 + hh * 128 + v] = pq;
        group_sync(BAR_S);
        const float w = part[v] + part[128 + v];
        const float sq = part[256 + v] + part[384 + v];
        const float kq = (xs[b * 4] + xs[b * 4 + 1]) + (xs[b * 4 + 2] + xs[b * 4 + 3]);
        const float u = xs[8 + b] * (fb[384 + v] - w);
#pragma unroll
        for (int j4 = 0; j4 < 16; ++j4) {
            const float4 kk = kv[j4];
            s[4 * j4] = fmaf(kk.x, u, s[4 * j4]); s[4 * j4 + 1] = fmaf(kk.y, u, s[4 * j4 + 1]);
            s[4 * j4 + 2] = fmaf(kk.z, u, s[4 * j4 + 2]); s[4 * j4 + 3] = fmaf(kk.w, u, s[4 * j4 + 3]);
        }
        if (hh == 0) p.o[((size_t)tg * p.H + h) * VD + v] = __float2bfloat16_rn(p.scale * (sq + u * kq));
    }
    KDA_TMEM_ST32(lb + TM_S + 64 * hh, reinterpret_cast<const uint32_t *>(s));
    KDA_TMEM_ST32(lb + TM_S + 64 * hh + 32, (reinterpret_cast<const uint32_t *>(s) + 32));
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(NT, 1) prefill_tc_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *beta_s = reinterpret_cast<float *>(sm + SM_BETA);
    float *gam_s = reinterpret_cast<float *>(sm + SM_GAM);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + SM_MISC);
    int *flags = reinterpret_cast<int *>(sm + SM_MISC + 4);
    int *flag_prep = reinterpret_cast<int *>(sm + SM_MISC + 8);   // [2]
    int *flag_tb = reinterpret_cast<int *>(sm + SM_MISC + 16);    // [2]
    const uint32_t mb = sbase + SM_BAR;
    const uint64_t wait_ns = p.wait_ns ? p.wait_ns : WAIT_NS;

    // ---- the unit: longest sequences first ------------------------------
    const int ui = blockIdx.x / p.H, h = blockIdx.x - (blockIdx.x / p.H) * p.H;
    const int n = p.lpt ? p.order[ui] : ui;
    const int bos = p.cu[n], eos = p.cu[n + 1];
    if (bos < 0 || eos < bos || eos > p.T_total) {
        if (tid == 0 && h == 0) report(p.err, DEVERR_SEQLENS);
        return;
    }
    const int si = p.init_slot[n], so = p.out_slot[n];
    const int ss = p.snap_slot ? p.snap_slot[n] : -1;
    const int nck = ckpt_count(eos - bos, p.ckpt_chunks * C, p.max_ckpts);
    if (si < -1 || si >= p.num_slots || so < 0 || so >= p.num_slots || ss >= p.num_slots ||
        !ckpt_slots_ok(p.ckpt_slots, n, nck, p.max_ckpts, p.num_slots)) {
        if (tid == 0 && h == 0) report(p.err, DEVERR_SLOT_RANGE);
        return;
    }
    const int nchunks = (eos - bos + C - 1) / C;

    // ---- set-up -----------------------------------------------------------
    if (tid == 0) {
        for (int i = 0; i < MB_COUNT; ++i) barrier_init(mb + 8 * i, 1);
        *flags = 0;
        flag_prep[0] = flag_prep[1] = flag_tb[0] = flag_tb[1] = 0;
        if (nchunks > 0 && !p.skip_first_load) {
            barrier_expect(mb + MB_RAW, 3 * 16384);
            for (int b = 0; b < 2; ++b) {
                tma_load_3d(sbase + RAW_Q + b * 8192, &p.tq, mb + MB_RAW, 64 * b, h, bos);
                tma_load_3d(sbase + RAW_K + b * 8192, &p.tk, mb + MB_RAW, 64 * b, h, bos);
                tma_load_3d(sbase + RAW_G + b * 8192, &p.tg, mb + MB_RAW, 64 * b, h, bos);
            }
        }
        for (int i = 0; i < 2 && i < nchunks; ++i) {
            barrier_expect(mb + MB_V + 8 * i, 16384);
            for (int b = 0; b < 2; ++b)
                tma_load_3d(sbase + OP_V + i * 16384 + b * 8192, &p.tv, mb + MB_V + 8 * i, 64 * b, h,
                            bos + i * C);
        }
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const float LOG2E = 1.4426950408889634f;

    if (warp < 8) {
        // =================== intra-chunk group ===================
        const int it = tid;
        const int lq = warp & 3, hh = warp >> 2;   // TMEM lane quarter, column half of the Gram read-out
        float *As = reinterpret_cast<float *>(sm + SCR_A);
        float *Ts = reinterpret_cast<float *>(sm + SCR_T);
        float *Rws = reinterpret_cast<float *>(sm + SCR_RW);
        const unsigned short *beta_bits = reinterpret_cast<const unsigned short *>(p.beta);
        unsigned short beta_raw = 0;
        bool beta_ok = false;
        if (it < C && nchunks > 0) {
            beta_ok = it < eos - bos;
            beta_raw = __ldg(beta_bits + (size_t)(beta_ok ? bos + it : bos) * p.H + h);
        }
        constexpr uint32_t ID_G1 = idesc(128, 64, 0, 0, 2);
        // prep: warp w owns key channels 16w .. 16w+15 (two 8-channel halves);
        // lane l owns rows 2l and 2l + 1, taken in the order rA, rB so that the 8
        // lanes of each quarter-warp meet all 8 positions of the 128-byte swizzle.
        const int swr = (lane >> 2) & 1;
        const int rA = 2 * lane + swr, rB = 2 * lane + 1 - swr;
        for (int c = 0; c < nchunks; ++c) {
            const int t0 = bos + c * C;
            const int L = min(C, eos - t0);
            const int par = c & 1;

            // (1) beta of this chunk; the next chunk's is loaded
            if (it < C) {
                beta_s[par * 64 + it] = beta_ok ? __uint_as_float((uint32_t)beta_raw << 16) : 0.f;
                const int tn = t0 + C + it;
                beta_ok = c + 1 < nchunks && tn < eos;
                beta_raw = __ldg(beta_bits + (size_t)(beta_ok ? tn : bos) * p.H + h);
            }
            // (2) this chunk's raw q, k, gk into registers
            if (it == 0) wait_or_flag(mb + MB_RAW, (uint32_t)par, wait_ns, flags);
            if (group_sync_or(BAR_I, timed_out(flags))) break;
            uint4 wq[2][2], wk[2][2], wg[2][2];
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {
                const int ch = 16 * warp + 8 * hq;
                wq[hq][0] = *reinterpret_cast<const uint4 *>(sm + RAW_Q + chunk_off(rA, ch, 64));
                wq[hq][1] = *reinterpret_cast<const uint4 *>(sm + RAW_Q + chunk_off(rB, ch, 64));
                wk[hq][0] = *reinterpret_cast<const uint4 *>(sm + RAW_K + chunk_off(rA, ch, 64));
                wk[hq][1] = *reinterpret_cast<const uint4 *>(sm + RAW_K + chunk_off(rB, ch, 64));
                wg[hq][0] = *reinterpret_cast<const uint4 *>(sm + RAW_G + chunk_off(rA, ch, 64));
                wg[hq][1] = *reinterpret_cast<const uint4 *>(sm + RAW_G + chunk_off(rB, ch, 64));
            }
            // the state group has released [K~; Q~] (P of the previous chunk is
            // done, hence also the products that read this parity's K_end), and
            // this chunk's v has landed
            if (it == 0) {
                if (c >= 1) wait_or_flag(mb + MB_P, (uint32_t)((c - 1) & 1), wait_ns, flags);
                wait_or_flag(mb + MB_V + 8 * par, (uint32_t)((c >> 1) & 1), wait_ns, flags);
            }
            if (group_sync_or(BAR_I, timed_out(flags))) break;   // also: R1's raw tiles are read

            // (3) v -> fp16 in place (rows past the sequence become zero)
            float vmax = 0.f;
            {
                uint8_t *vt = sm + OP_V + par * 16384;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int q4 = it + NG * i;            // 16-byte chunk 0..1023
                    const int row = (q4 >> 3) & 63;        // token row (2 boxes of 64 rows x 128 B)
                    const uint4 w = *reinterpret_cast<const uint4 *>(vt + 16 * q4);
                    float f[8];
                    unpack_bf16(w, f);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        f[j] = row < L ? f[j] : 0.f;
                        vmax = fmaxf(vmax, mag(f[j]));
                    }
                    store_f16(vt, 16 * q4, f);
                }
            }
            // (4) cumulative decays, exponentials and the operand tiles
            float dmax = 0.f, qkmax = 0.f, gmax = 0.f;
            const bool vA = rA < L, vB = rB < L;
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {
                const int ch = 16 * warp + 8 * hq;
                float gA[8], gB[8];
                unpack_bf16(wg[hq][0], gA);
                unpack_bf16(wg[hq][1], gB);
                float gref[8], glast[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float a = vA ? gA[i] : 0.f, b = vB ? gB[i] : 0.f;
                    gmax = fmaxf(gmax, fmaxf(a == a ? a : 1.f, b == b ? b : 1.f));
                    float s2 = a + b;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float t = __shfl_up_sync(0xffffffffu, s2, off);
                        if (lane >= off) s2 += t;
                    }
                    const float odd = swr ? a : b;   // the term of row 2l + 1
                    gA[i] = swr ? s2 : s2 - odd;
                    gB[i] = swr ? s2 - odd : s2;
                    gref[i] = __shfl_sync(0xffffffffu, s2, 15);    // G at row 31
                    glast[i] = __shfl_sync(0xffffffffu, s2, 31);   // G at row 63 (= last valid row)
                }
                float egr[8], elr[8];   // per channel: exp(G_ref), exp(G_L - G_ref)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    egr[i] = ex2(gref[i] * LOG2E);
                    elr[i] = ex2((glast[i] - gref[i]) * LOG2E);
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int r = half ? rB : rA;
                    const bool valid = half ? vB : vA;
                    const float *g = half ? gB : gA;
                    float qq[8], kk[8];
                    unpack_bf16(wq[hq][half], qq);
                    unpack_bf16(wk[hq][half], kk);
                    float kf[8], kb[8], kt[8], ke[8], qr[8], qt[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float q_ = valid ? qq[i] : 0.f, k_ = valid ? kk[i] : 0.f;
                        qkmax = fmaxf(qkmax, fmaxf(mag(q_), mag(k_)));
                        const float d = (g[i] - gref[i]) * LOG2E;
                        dmax = fmaxf(dmax, mag(d));
                        const float ef = ex2(d);                 // exp(G_r - G_ref)
                        const float eb = ex2(-d);                // exp(G_ref - G_r)
                        kf[i] = k_ * ef;
                        kb[i] = k_ * eb;
                        kt[i] = k_ * (egr[i] * ef);              // k exp(G_r)
                        ke[i] = k_ * (elr[i] * eb);              // k exp(G_L - G_r)
                        qr[i] = q_ * ef;
                        qt[i] = q_ * (egr[i] * ef);              // q exp(G_r)
                    }
                    store_f32x8(sm, OP_A1, r, ch, 128, kf);
                    store_f32x8(sm, OP_A1, 64 + r, ch, 128, qr);
                    store_f32x8(sm, OP_B1, r, ch, 64, kb);
                    store_f16(sm, OP_KQ + chunk_off(r, ch, 128), kt);
                    store_f16(sm, OP_KQ + chunk_off(64 + r, ch, 128), qt);
                    store_f16(sm, OP_KE + par * 16384 + chunk_off(r, ch, 64), ke);
                }
                if (lane == 31) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) gam_s[par * 128 + ch + i] = expf(glast[i]);
                }
            }
            const bool bad = !(dmax <= D_LIMIT * LOG2E) || !(qkmax <= QK_LIMIT) || !(gmax <= 0.f) ||
                             !(vmax <= FP16_LIMIT);
            fence_proxy_async();
            const bool prep_bad = group_sync_or(BAR_I, bad);
            if (it == 0) {
                flag_prep[par] = prep_bad;
                barrier_arrive(mb + MB_PREP + 8 * par);   // release: the tiles, gamma and the flag
                // (5) the Gram product on TF32: [Kf; Qr] Kb^T, 16 steps of K = 8
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < 16; ++s)
                    mma_tf32(tmem + TM_G1, sdesc(sbase + OP_A1 + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024),
                             sdesc(sbase + OP_B1 + (s >> 2) * 8192 + (s & 3) * 32, 16, 1024), ID_G1, s > 0);
                mma_commit(mb + MB_G1);
                wait_or_flag(mb + MB_G1, (uint32_t)par, wait_ns, flags);
                // Aqk's tile is free once the previous chunk's O product is done
                if (c >= 1) wait_or_flag(mb + MB_G4, (uint32_t)((c - 1) & 1), wait_ns, flags);
            }
            if (group_sync_or(BAR_I, timed_out(flags))) break;
            tc_fence_after();
            // the Gram operands are consumed: the next chunk's raw q, k, gk into R1
            if (it == 0 && c + 1 < nchunks) {
                barrier_expect(mb + MB_RAW, 3 * 16384);
                for (int b = 0; b < 2; ++b) {
                    tma_load_3d(sbase + RAW_Q + b * 8192, &p.tq, mb + MB_RAW, 64 * b, h, t0 + C);
                    tma_load_3d(sbase + RAW_K + b * 8192, &p.tk, mb + MB_RAW, 64 * b, h, t0 + C);
                    tma_load_3d(sbase + RAW_G + b * 8192, &p.tg, mb + MB_RAW, 64 * b, h, t0 + C);
                }
            }
            __syncwarp();
            // (6) A -> fp32 scratch (strictly lower, x beta_r); Aqk -> fp16 tile (lower incl. diagonal)
            float tbmax = 0.f;
            {
                uint32_t r[32];
                KDA_TMEM_LD32(tmem + ((uint32_t)(32 * lq) << 16) + TM_G1 + 32 * hh, r);
                const int row = 32 * (lq & 1) + lane;
                if (lq < 2) {
                    const float b = beta_s[par * 64 + row];
                    float4 *dst = reinterpret_cast<float4 *>(As + row * AS + 32 * hh);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float v4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int col = 32 * hh + 4 * j + e;
                            v4[e] = col < row ? __uint_as_float(r[4 * j + e]) * b : 0.f;
                        }
                        dst[j] = make_float4(v4[0], v4[1], v4[2], v4[3]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float v8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int col = 32 * hh + 8 * j + e;
                            v8[e] = col <= row ? __uint_as_float(r[8 * j + e]) : 0.f;
                            tbmax = fmaxf(tbmax, mag(v8[e]));
                        }
                        store_f16(sm, OP_AQK + (uint32_t)row * 128 + ((((4 * hh + j) ^ row) & 7) << 4), v8);
                    }
                }
            }
            tc_fence_before();
            // T Diag(b)'s tile is free once the previous chunk's U product is done
            if (it == 0 && c >= 1) wait_or_flag(mb + MB_U, (uint32_t)((c - 1) & 1), wait_ns, flags);
            if (group_sync_or(BAR_I, timed_out(flags))) break;

            // (7) T = (I + A)^-1 in 16 x 16 blocks: diagonal blocks T_II by forward
            //     substitution (warps 0-1, one block per half-warp, lane = column);
            //     warps 2-7 zero the blocks of T Diag(b) above the diagonal.
            const float *bet = beta_s + par * 64;
            if (warp < 2) {
                const int I = 2 * warp + (lane >> 4), col = lane & 15;
                const float *Ab = As + 16 * I * AS + 16 * I;   // diagonal block I, row stride AS
                // Column-oriented substitution: once x[j] is final, every later row
                // takes its term.  The chain is one FMA per step; rows load their
                // four entries of a column group as one 16-byte vector.
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) x[r] = (r == col) ? 1.f : 0.f;
#pragma unroll
                for (int j0 = 0; j0 < 16; j0 += 4) {
                    float4 a[16];
#pragma unroll
                    for (int r = j0 + 1; r < 16; ++r) a[r] = *reinterpret_cast<const float4 *>(Ab + r * AS + j0);
#pragma unroll
                    for (int j = j0; j < j0 + 4 && j < 15; ++j) {
#pragma unroll
                        for (int r = j + 1; r < 16; ++r) {
                            const float e = (j & 3) == 0 ? a[r].x : (j & 3) == 1 ? a[r].y : (j & 3) == 2 ? a[r].z : a[r].w;
                            x[r] = fmaf(-e, x[j], x[r]);
                        }
                    }
                }
                const int cI = 16 * I + col;
                const float bc = bet[cI];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const int rr = 16 * I + r;
                    Ts[rr * 64 + tsw(r, cI)] = x[r];
                    const float tv = x[r] * bc;
                    tbmax = fmaxf(tbmax, mag(tv));
                    *reinterpret_cast<__half *>(sm + OP_TB + rr * 128 + ((((cI >> 3) ^ rr) & 7) << 4) +
                                                (cI & 7) * 2) = __float2half_rn(tv);
                }
            } else {
                // 6 upper blocks x 16 rows x two 16-byte chunks = 192 chunks, one per thread
                const int t = it - 64;                   // 0 .. 191
                const int blk = t >> 5, rem = t & 31, r = rem >> 1, h2 = rem & 1;
                const int I = (blk < 3) ? 0 : (blk < 5 ? 1 : 2);
                const int J = (blk < 3) ? blk + 1 : (blk < 5 ? blk - 1 : 3);
                const int rr = 16 * I + r, cchunk = 2 * J + h2;
                *reinterpret_cast<uint4 *>(sm + OP_TB + rr * 128 + (((cchunk ^ rr) & 7) << 4)) =
                    make_uint4(0, 0, 0, 0);
            }
            group_sync(BAR_I);
            if (warp < 2) tbmax = fmaxf(tbmax, solve_block_column<0>(As, Ts, Rws + warp * 16 * RW, lane, sm + OP_TB, bet, warp & 1));
            else if (warp < 4) tbmax = fmaxf(tbmax, solve_block_column<1>(As, Ts, Rws + warp * 16 * RW, lane, sm + OP_TB, bet, warp & 1));
            else if (warp < 6) tbmax = fmaxf(tbmax, solve_block_column<2>(As, Ts, Rws + warp * 16 * RW, lane, sm + OP_TB, bet, warp & 1));
            fence_proxy_async();
            const bool tb_bad = group_sync_or(BAR_I, !(tbmax <= FP16_LIMIT));
            if (it == 0) {
                flag_tb[par] = tb_bad;
                barrier_arrive(mb + MB_TB + 8 * par);
            }
        }
    } else {
        // =================== state group ===================
        const int st = tid - NG;                   // 0 .. 255
        const int sw = warp - 8;
        const int lq = sw & 3, hh = sw >> 2;       // TMEM lane quarter; key-column half / token half
        const int v = 32 * lq + lane;              // the value channel on this thread's TMEM lane
        const uint32_t lb = tmem + ((uint32_t)(32 * lq) << 16);
        constexpr uint32_t ID_P = idesc(128, 64, 0, 0, 0);
        constexpr uint32_t ID_UV = idesc(128, 64, 1, 0, 0);
        constexpr uint32_t ID_UT = idesc(128, 64, 0, 0, 0);
        constexpr uint32_t ID_DS = idesc(128, 128, 0, 1, 0);
        // initial state: S^T[v][k], k = 64 hh .. 64 hh + 63 (each warp load is one 128-byte row segment)
        {
            float s[64];
            if (si >= 0) {
                const float *src = p.pool + ((size_t)si * p.H + h) * STATE_ELEMS + (size_t)(64 * hh) * VD + v;
#pragma unroll
                for (int j = 0; j < 64; ++j) s[j] = __ldcs(src + (size_t)j * VD);
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) s[j] = 0.f;
            }
            KDA_TMEM_ST32(lb + TM_S + 64 * hh, reinterpret_cast<const uint32_t *>(s));
            KDA_TMEM_ST32(lb + TM_S + 64 * hh + 32, (reinterpret_cast<const uint32_t *>(s) + 32));
        }
        bool fb_prev = false, stopped = false;
        for (int c = 0; c < nchunks; ++c) {
            const int t0 = bos + c * C;
            const int L = min(C, eos - t0);
            const int par = c & 1;
            // (1) chunk c's operand tiles are ready; the previous chunk's products are done
            if (st == 0) {
                wait_or_flag(mb + MB_PREP + 8 * par, (uint32_t)((c >> 1) & 1), wait_ns, flags);
                if (c >= 1) wait_or_flag(mb + MB_G4, (uint32_t)((c - 1) & 1), wait_ns, flags);
            }
            if (group_sync_or(BAR_S, timed_out(flags))) { stopped = true; break; }
            tc_fence_after();
            bool fb = flag_prep[par] != 0;
            // (2) the state pass: S_{c-1} -> checkpoint, fp16 copy for P
            {
                const int m = c / max(p.ckpt_chunks, 1) - 1;
                float *ck = nullptr;
                if (nck > 0 && c > 0 && c % p.ckpt_chunks == 0 && m < nck) {
                    const int cs = p.ckpt_slots[(size_t)n * p.max_ckpts + m];
                    if (cs >= 0) ck = p.pool + ((size_t)cs * p.H + h) * STATE_ELEMS + (size_t)(64 * hh) * VD + v;
                }
                float smax = 0.f;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t r[32];
                    KDA_TMEM_LD32(lb + TM_S + 64 * hh + 32 * half, r);
                    if (ck) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) __stcs(ck + (size_t)(32 * half + j) * VD, __uint_as_float(r[j]));
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float a = __uint_as_float(r[2 * j]), b = __uint_as_float(r[2 * j + 1]);
                        smax = fmaxf(smax, fmaxf(mag(a), mag(b)));
                        pk[j] = pack_f16x2(a, b);
                    }
                    KDA_TMEM_ST16(lb + TM_S16 + 32 * hh + 16 * half, pk);
                }
                tc_fence_before();
                fb = group_sync_or(BAR_S, fb || !(smax <= FP16_LIMIT));
            }
            // (3) P = S0^T [K~^T | Q~^T]
            if (st == 0) {
                tc_fence_after();
                if (!fb) {
#pragma unroll
                    for (int s8 = 0; s8 < 8; ++s8)
                        mma_ts(tmem + TM_KS, tmem + TM_S16 + 8 * s8,
                               sdesc(sbase + OP_KQ + (s8 >> 2) * 16384 + (s8 & 3) * 32, 16, 1024), ID_P, s8 > 0);
#pragma unroll
                    for (int s8 = 0; s8 < 8; ++s8)
                        mma_ts(tmem + TM_O + 64 * par, tmem + TM_S16 + 8 * s8,
                               sdesc(sbase + OP_KQ + (s8 >> 2) * 16384 + 8192 + (s8 & 3) * 32, 16, 1024), ID_P,
                               s8 > 0);
                    mma_commit(mb + MB_P);
                } else {
                    barrier_arrive(mb + MB_P);
                }
            }
            __syncwarp();
            // (4) O of the previous chunk (a full chunk) while P runs
            if (c >= 1 && !fb_prev) {
                store_o_cols(p, lb + TM_O + 64 * (par ^ 1) + 32 * hh, t0 - C + 32 * hh, 32, h, v);
                tc_fence_before();
            }
            // (5) -(K~ S0)^T -> fp16 in TMEM (A of U)
            if (!fb) {
                if (st == 0) wait_or_flag(mb + MB_P, (uint32_t)par, wait_ns, flags);
                if (group_sync_or(BAR_S, timed_out(flags))) { stopped = true; break; }
                tc_fence_after();
                uint32_t r[32];
                KDA_TMEM_LD32(lb + TM_KS + 32 * hh, r);
                float kmax = 0.f;
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float a = __uint_as_float(r[2 * j]), b = __uint_as_float(r[2 * j + 1]);
                    kmax = fmaxf(kmax, fmaxf(mag(a), mag(b)));
                    pk[j] = pack_f16x2(-a, -b);
                }
                KDA_TMEM_ST16(lb + TM_KS + 32 * hh, pk);
                tc_fence_before();
                fb = group_sync_or(BAR_S, !(kmax <= FP16_LIMIT));
            }
            // (6) T Diag(b) and Aqk of chunk c are ready.  Waited on every path,
            //     also when the chunk takes the recurrence: the U and G4 barriers
            //     below then complete chunk c's phase only after the intra group
            //     has finished chunk c, so they are never two phases ahead of its
            //     waits on them (a parity wait cannot tell those phases apart).
            if (st == 0) wait_or_flag(mb + MB_TB + 8 * par, (uint32_t)((c >> 1) & 1), wait_ns, flags);
            if (group_sync_or(BAR_S, timed_out(flags))) { stopped = true; break; }
            if (!fb) fb = flag_tb[par] != 0;
            // (7) U^T = V^T TB^T - (K~ S0)^T TB^T
            if (st == 0) {
                tc_fence_after();
                if (!fb) {
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4)
                        mma_ss(tmem + TM_U, sdesc(sbase + OP_V + par * 16384 + s4 * 2048, 8192, 1024),
                               sdesc(sbase + OP_TB + s4 * 32, 16, 1024), ID_UV, s4 > 0);
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4)
                        mma_ts(tmem + TM_U, tmem + TM_KS + (s4 >> 1) * 32 + (s4 & 1) * 8,
                               sdesc(sbase + OP_TB + s4 * 32, 16, 1024), ID_UT, 1);
                    mma_commit(mb + MB_U);
                    wait_or_flag(mb + MB_U, (uint32_t)par, wait_ns, flags);
                } else {
                    barrier_arrive(mb + MB_U);
                }
                // v of chunk c + 2 into this parity's buffer, free now
                if (c + 2 < nchunks && !timed_out(flags)) {
                    barrier_expect(mb + MB_V + 8 * par, 16384);
                    for (int b = 0; b < 2; ++b)
                        tma_load_3d(sbase + OP_V + par * 16384 + b * 8192, &p.tv, mb + MB_V + 8 * par, 64 * b,
                                    h, t0 + 2 * C);
                }
            }
            __syncwarp();
            // (8) U^T -> fp16 in TMEM (A of O and dS)
            if (!fb) {
                if (group_sync_or(BAR_S, timed_out(flags))) { stopped = true; break; }
                tc_fence_after();
                uint32_t r[32];
                KDA_TMEM_LD32(lb + TM_U + 32 * hh, r);
                float umax = 0.f;
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float a = __uint_as_float(r[2 * j]), b = __uint_as_float(r[2 * j + 1]);
                    umax = fmaxf(umax, fmaxf(mag(a), mag(b)));
                    pk[j] = pack_f16x2(a, b);
                }
                KDA_TMEM_ST16(lb + TM_U + 32 * hh, pk);
                tc_fence_before();
                fb = group_sync_or(BAR_S, !(umax <= FP16_LIMIT));
            }
            if (!fb) {
                // (9) S^T <- S^T Diag(exp(G_L)), then O^T += U^T Aqk^T and S^T += U^T K_end
                const float4 *gm = reinterpret_cast<const float4 *>(gam_s + par * 128 + 64 * hh);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t r[32];
                    KDA_TMEM_LD32(lb + TM_S + 64 * hh + 32 * half, r);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 g4 = gm[8 * half + j4];
                        r[4 * j4] = __float_as_uint(__uint_as_float(r[4 * j4]) * g4.x);
                        r[4 * j4 + 1] = __float_as_uint(__uint_as_float(r[4 * j4 + 1]) * g4.y);
                        r[4 * j4 + 2] = __float_as_uint(__uint_as_float(r[4 * j4 + 2]) * g4.z);
                        r[4 * j4 + 3] = __float_as_uint(__uint_as_float(r[4 * j4 + 3]) * g4.w);
                    }
                    KDA_TMEM_ST32(lb + TM_S + 64 * hh + 32 * half, r);
                }
                tc_fence_before();
                group_sync(BAR_S);
                if (st == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4) {
                        const uint32_t a = tmem + TM_U + (s4 >> 1) * 32 + (s4 & 1) * 8;
                        mma_ts(tmem + TM_O + 64 * par, a, sdesc(sbase + OP_AQK + s4 * 32, 16, 1024), ID_UT, 1);
                        mma_ts(tmem + TM_S, a, sdesc(sbase + OP_KE + par * 16384 + s4 * 2048, 8192, 1024), ID_DS, 1);
                    }
                    mma_commit(mb + MB_G4);
                }
                __syncwarp();
            } else {
                // (9') the recurrence over this chunk, from S_{c-1} (untouched in TMEM)
                if (st == 0) barrier_arrive(mb + MB_G4);
                __syncwarp();
                chunk_recurrent(p, sm, lb, t0, L, h, st, v, hh);
                tc_fence_before();
            }
            fb_prev = fb;
        }
        // the last chunk's products, and its O
        if (nchunks > 0 && !stopped) {
            if (st == 0) wait_or_flag(mb + MB_G4, (uint32_t)((nchunks - 1) & 1), wait_ns, flags);
            const bool to = group_sync_or(BAR_S, timed_out(flags));
            tc_fence_after();
            if (!to && !fb_prev) {
                const int tl = bos + (nchunks - 1) * C;
                store_o_cols(p, lb + TM_O + 64 * ((nchunks - 1) & 1) + 32 * hh, tl + 32 * hh,
                             eos - tl - 32 * hh, h, v);
            }
        }
    }

    // ---- tail: the final state, unless a wait gave up ---------------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (timed_out(flags)) {
        if (tid == 0) {
            report(p.err, DEVERR_TIMEOUT);
            // copies issued at set-up that no consumer waited for: let them land
            // (bounded) before the CTA's shared memory is released
            if (p.skip_first_load)
                for (int i = 0; i < 2 && i < nchunks; ++i) barrier_wait_for(mb + MB_V + 8 * i, 0, wait_ns);
        }
    } else if (warp >= 8) {
        const int sw = warp - 8, lq = sw & 3, hh = sw >> 2, v = 32 * lq + lane;
        const uint32_t lb = tmem + ((uint32_t)(32 * lq) << 16);
        const size_t off = (size_t)(64 * hh) * VD + v;
        float *d0 = p.pool + ((size_t)so * p.H + h) * STATE_ELEMS + off;
        float *d1 = ss >= 0 ? p.pool + ((size_t)ss * p.H + h) * STATE_ELEMS + off : nullptr;
        // a checkpoint that falls on the sequence's end
        const int m = nchunks / max(p.ckpt_chunks, 1) - 1;
        float *d2 = nullptr;
        if (nck > 0 && nchunks > 0 && nchunks % p.ckpt_chunks == 0 && m < nck) {
            const int cs = p.ckpt_slots[(size_t)n * p.max_ckpts + m];
            if (cs >= 0) d2 = p.pool + ((size_t)cs * p.H + h) * STATE_ELEMS + off;
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t r[32];
            KDA_TMEM_LD32(lb + TM_S + 64 * hh + 32 * half, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float x = __uint_as_float(r[j]);
                const size_t e = (size_t)(32 * half + j) * VD;
                __stcs(d0 + e, x);
                if (d1) __stcs(d1 + e, x);
                if (d2) __stcs(d2 + e, x);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS));
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [T][H][128] bf16 viewed as a 3-D tensor {128, H, T}; boxes of 64 channels x 1 head x 64 tokens.
bool make_map(CUtensorMap *m, const void *base, int H, int T) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

cudaError_t launch_prefill_chunked(const PrefillArgs &a, cudaStream_t s) {
    using namespace tc;
    Params p;   // ~9 KB, copied into the launch parameters
    memset(&p, 0, sizeof(p));
    if (a.T_total > 0) {
        if (!make_map(&p.tq, a.q, a.H, a.T_total) || !make_map(&p.tk, a.k, a.H, a.T_total) ||
            !make_map(&p.tg, a.gk, a.H, a.T_total) || !make_map(&p.tv, a.v, a.H, a.T_total))
            return cudaErrorInvalidValue;
    }
    p.N = a.N; p.T_total = a.T_total; p.H = a.H; p.num_slots = a.num_slots;
    p.q = (const __nv_bfloat16 *)a.q; p.k = (const __nv_bfloat16 *)a.k;
    p.gk = (const __nv_bfloat16 *)a.gk; p.v = (const __nv_bfloat16 *)a.v;
    p.beta = (const __nv_bfloat16 *)a.beta; p.cu = a.cu; p.pool = a.pool;
    p.init_slot = a.init_slot; p.out_slot = a.out_slot; p.snap_slot = a.snap_slot;
    p.o = (__nv_bfloat16 *)a.o; p.scale = a.scale; p.err = a.err;
    p.ckpt_chunks = a.ckpt_interval / C; p.max_ckpts = a.max_ckpts; p.ckpt_slots = a.ckpt_slots;
    p.wait_ns = a.wait_ns;
    p.skip_first_load = a.skip_first_load;
    p.lpt = a.N <= KDA_MAX_LPT_SEQS;
    if (p.lpt) {
        std::vector<int> idx(a.N);
        std::iota(idx.begin(), idx.end(), 0);
        std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) {
            return a.cu_host[x + 1] - a.cu_host[x] > a.cu_host[y + 1] - a.cu_host[y];
        });
        for (int i = 0; i < a.N; ++i) p.order[i] = idx[i];
    }
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<<<(unsigned)(a.N * a.H), NT, SMEM_BYTES, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
