// Chunked KDA prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One CTA (512 threads) per (sequence, head) unit walks the sequence in chunks
// of C = 64 tokens with the fp32 128 x 128 state held in registers across
// chunks (32 values per thread); every chunk-sized contraction runs as a
// tcgen05.mma (operands in shared memory, fp32 accumulators in TMEM).  The
// pages' FlashKDA fuses a chunk's work and the state update into one kernel
// with intermediates on chip (Kimi K3 on B200 deployment notes, timeline entry
// "FlashKDA"); its CuTe rewrite keeps the state on chip and issues the longest
// sequences first.  Both ideas are kept here; the chunk size, the state
// placement (registers, not TMEM) and the work split are this kernel's own.
//
// Chunk algebra (derived from the recurrence
//     S_t = (I - b_t k_t k_t^T) Diag(exp(gk_t)) S_{t-1} + b_t k_t v_t^T,  o_t = S_t^T q_t
// by unrolling it over the chunk).  With G_r = sum_{j<=r} gk_j per key channel,
// S0 the state entering the chunk, G_L the last row's G, K~ = K . exp(G),
// Q~ = Q . exp(G) and K_end = K . exp(G_L - G):
//     A[r][j]   = b_r <k_r, exp(G_r - G_j) . k_j>  (j < r),  T = (I + A)^-1
//     Aqk[r][j] = <q_r, exp(G_r - G_j) . k_j>       (j <= r)
//     U         = T Diag(b) (V - K~ S0)
//     O         = Q~ S0 + Aqk U
//     S_L       = Diag(exp(G_L)) S0 + K_end^T U
// (U is the usual U~ - W S0 with U~ = T Diag(b) V and W = T Diag(b) K~, taken
// in one product.)  The pairwise factors exp(G_r - G_j) of the Gram matrices
// are split as exp(G_r - G_ref) * exp(G_ref - G_j) around the chunk's row 31,
// which keeps both factors in fp32 range while a key channel's decay over half
// a chunk stays within 79 (natural log).
//
// Per chunk (M = 128 throughout; shared-memory operands in the 128-byte-
// swizzled canonical layouts):
//   G1  [Kf; Qr] (128x128) x Kb^T   (tf32)  -> TMEM cols [0,64): A (rows 0-63), Aqk (64-127)
//   P   [K~; Q~] (128x128) x S0     (fp16)  -> cols 256.. (by chunk parity): K~ S0, Q~ S0
//   U   [T Diag(b); Aqk] (128x64) x V'      -> cols [0,128), rows 0-63 kept; V' = V - K~ S0
//   G4a [T Diag(b); Aqk] (128x64) x U (+=)  -> P's rows 64-127 become O
//   G4b K_end^T (128x64) x U                -> cols [0,128): the state increment
// P depends on the previous chunk's state only, so it is issued with G1 and
// read out (into V', in place of v) while the triangular solve runs; O stays in
// TMEM until the next chunk's solve phase, where the warps of lanes 64..127
// write it out.  CUDA cores do the cumulative decays and exponentials (prep),
// the 64x64 unit-lower-triangular inverse (16x16 blocks: substitution on the
// diagonal, warp-level TF32 MMAs off it), the TMEM read-outs and the fp32 state
// update.
//
// Operand precision: the Gram factors span exp(+-26) and need an 8-bit
// exponent, so G1 runs on TF32 (fp32 operand tiles); the operands of P, U and
// G4 are bounded or checked (|.| <= 1 for the decayed q, k and Aqk; |q|, |k| <=
// 256; T Diag(b), V', U and S below 60000) and use fp16's 11-bit significand.
// All operands in bf16 would give about 3e-2 x RMS on o; this mix about 8e-3
// (a CPU model of the chunk algebra with the kernel's roundings).
//
// Exactness over the whole input domain: a chunk whose factors or operands
// would leave those formats (the decay bound, a positive gk, |q| or |k| above
// 256, Aqk, T Diag(b), V', U or S above 60000, or a NaN) does not use the
// tensor-core result: all 512 threads apply the recurrence to it token by
// token in fp32 on the CUDA cores, from the state entering the chunk (still in
// registers: every check is decided before the chunk's state update).
//
// All waits are bounded (barrier_wait_for, the wait loop of the library's
// other kernels, with a per-launch limit); a wait that gives up reports
// KDA_DEVERR_TIMEOUT, frees TMEM and abandons the unit without writing its
// slots.  Data movement: raw q, k, gk, v tiles arrive by TMA one chunk ahead
// and are taken into registers while the previous chunk's G4 runs; the unit's
// initial state arrives by four tensor copies into a swizzled staging tile and
// the final state leaves as whole 512-byte rows through it.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <numeric>
#include <type_traits>
#include <vector>

#include "kda_async.cuh"
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace tc {

constexpr int C = 64;              // chunk length
constexpr int NT = 512;            // threads per CTA
constexpr int AS = 68;             // row stride (floats) of the fp32 A scratch

// Shared-memory map (byte offsets from a 1024-aligned base).  Region R1
// [0, 96K) holds the G1 operands from the end of the prep to the end of G1,
// then the next chunk's raw q, k, gk (TMA), the triangular-solve scratch and
// the [T Diag(b); 0; Aqk] tile.  The prep reads its raw tiles into registers
// before it overwrites R1.
constexpr uint32_t OP_A1 = 0;          // [Kf; Qr], fp32 (tf32 MMA), 128 rows x 128 ch, K-major A
constexpr uint32_t OP_B1 = 65536;      // Kb, fp32, 64 rows x 128 ch, K-major B
constexpr uint32_t RAW_Q = 0;          // 64 tokens x 128 ch bf16, 2 boxes of 64 ch (TMA)
constexpr uint32_t RAW_K = 16384;
constexpr uint32_t RAW_G = 32768;
constexpr uint32_t SCR_A = 49152;      // fp32 A [64][AS]
// [T Diag(b); Aqk] (fp16, K-major, 64 token columns): the A operand of both U
// and O.  U = [T Diag(b); Aqk] V' keeps rows 0-63 (its rows 64-127, Aqk V', are
// never read), and O = [T Diag(b); Aqk] U added onto P keeps rows 64-127 (its
// rows 0-63 land on K~ S0, which is no longer needed), so no zero rows are kept.
constexpr uint32_t OP_TBZ = 69632;
constexpr uint32_t SCR_RW = 94208;     // per-warp R scratch of the solve (6 x 16 x RW floats)
constexpr uint32_t R1_END = 98304;
// The recurrent path (a chunk outside the operand formats) reuses the solve
// scratch for its per-token inputs and partial sums, and the staging tile for
// the fp32 state as [128][129] (padded rows: conflict-free by row and column).
constexpr uint32_t FB_IN = SCR_A;            // 2 x {alpha, k, q, v}[128] fp32
constexpr uint32_t FB_P = SCR_A + 4096;      // [4 pk | 4 pq][128] fp32
constexpr uint32_t FB_X = SCR_A + 8192;      // [2][4] k.q partials, [2] beta
constexpr int FB_LD = 129;                   // row stride (floats) of the staged state
constexpr uint32_t RAW_V = 98304;      // v (bf16, TMA), then V' = V - K~ S0 in place (fp16): MN-major B of U
constexpr uint32_t OP_OST = 114688;    // staging of the previous chunk's O for its tensor store (8 x 2 KB)
constexpr uint32_t OP_A3 = 131072;     // [K~; Q~] = [K; Q] . exp(G), fp16, 128 rows x 128 ch, K-major A of P
constexpr uint32_t OP_S = 163840;      // S0, fp16, 128 rows (k) x 128 (v), MN-major B
constexpr uint32_t OP_KE = 196608;     // K . exp(G_L - G), fp16, 64 tokens x 128 ch, MN-major A
constexpr uint32_t OP_U = 212992;      // U, fp16, 64 tokens x 128 v, MN-major B
constexpr uint32_t SCR_T = OP_U;       // during the solve: fp32 T [64][64] (before U is read out)
// Before the first chunk and after the last, the fp32 state passes through a
// 64 KB staging tile here (KT, [-W; Q~] and the first half of S0).  In: four
// tensor copies, box j = columns 32j .. 32j+31 of the 128 rows, 128 bytes per
// row with its 16-byte chunks XOR-swizzled by (row & 7).  Out: rows of 512
// bytes, chunks XOR-swizzled by (row & 7), stored as whole rows.  Either way
// each thread's 128-byte row segment moves without bank conflicts.
constexpr uint32_t STG = OP_OST;
constexpr uint32_t SM_BETA = 229376;   // fp32 [64]
constexpr uint32_t SM_GAM = SM_BETA + 256;   // fp32 [2][128]: exp(G_L), by chunk parity
constexpr uint32_t SM_BAR = SM_GAM + 1024;   // 5 mbarriers
constexpr uint32_t SM_MISC = SM_BAR + 64;    // TMEM base, flags
constexpr uint32_t SMEM_USED = SM_MISC + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;   // + alignment slack
static_assert(SCR_A + 64 * AS * 4 <= OP_TBZ, "solve scratch overlaps the TBZ tile");
static_assert(OP_TBZ + 128 * 128 <= SCR_RW && SCR_RW + 6 * 16 * 8 * 4 <= R1_END, "R scratch misplaced");
static_assert(OP_TBZ % 1024 == 0 && OP_TBZ + 128 * 128 <= R1_END, "TBZ tile misplaced");
static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");
static_assert(FB_X + 64 <= SCR_A + 64 * AS * 4, "recurrent scratch overflows the solve scratch");
static_assert(STG + 128 * FB_LD * 4 <= OP_KE, "staged state overlaps K_end");

// TMEM columns (512 allocated; one CTA per SM): the Gram product, then U,
// then the state increment share columns 0..127; P = [K~; Q~] S0 of a chunk
// (rows 64..127 becoming its O) lives in columns 256..383 or 384..511 by
// chunk parity, so that the previous chunk's O survives the next P.
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_P = 256;
constexpr uint64_t WAIT_NS = 2000000000ull;   // bounded waits: 2 s
constexpr float FP16_LIMIT = 60000.f;         // fp16 operands must stay below this
constexpr float QK_LIMIT = 256.f;             // |q|, |k| bound of the tensor-core path
constexpr float D_LIMIT = 80.f;               // |G_r - G_ref| bound (natural log)

enum { FLAG_TIMEOUT = 1 };

struct Params {
    CUtensorMap tq, tk, tg, tv;
    CUtensorMap to;   // o: boxes of 32 channels x 1 head x 32 tokens, 64-byte swizzle
    CUtensorMap tpool;   // the state pool as [slots * H * 128][128] fp32: boxes of 32 columns x 128 rows
    int N, T_total, H, num_slots, lpt;
    const __nv_bfloat16 *beta;
    const int32_t *cu;
    float *pool;
    const int32_t *init_slot, *out_slot, *snap_slot;
    __nv_bfloat16 *o;
    float scale;
    int32_t *err;
    int ckpt_chunks, max_ckpts;     // checkpoint every ckpt_chunks chunks (0: none)
    const int32_t *ckpt_slots;
    const __nv_bfloat16 *q, *k, *gk, *v;   // the recurrent path reads its tokens directly
    uint64_t wait_ns;                       // limit of every wait
    int skip_first_load;                    // self-test: chunk 0's q, k, gk are never requested
    int32_t order[KDA_MAX_LPT_SEQS];
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// Completion of this CTA's MMAs: thread 0 waits (bounded) on the commit
// barrier, the block synchronises, every thread fences before reading TMEM.
__device__ __forceinline__ void mma_wait_all(uint32_t bar, uint32_t parity, int *flags, uint64_t lim) {
    if (threadIdx.x == 0 && !barrier_wait_for(bar, parity, lim)) atomicOr(flags, FLAG_TIMEOUT);
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}
// Bulk tensor store of a shared-memory box; completes in this thread's bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's bulk stores have read their shared-memory source.
__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's bulk stores are complete.
__device__ __forceinline__ void tma_store_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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
// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, fp32 accumulate; fmt 1 = bf16, 0 = fp16 (kind::f16),
// 2 = tf32 (kind::tf32).  A and B always share one format.
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn, int fmt) {
    return (1u << 4) | ((uint32_t)fmt << 7) | ((uint32_t)fmt << 10) | ((uint32_t)a_mn << 15) |
           ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc));
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
#define KDA_TMEM_LD16(taddr, r)                                                                   \
    asm volatile(                                                                                 \
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"  \
        "%14,%15}, [%16];\n"                                                                     \
        "tcgen05.wait::ld.sync.aligned;"                                                          \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
          "=r"(r[14]), "=r"(r[15])                                                                \
        : "r"(taddr)                                                                              \
        : "memory")
// The TMEM loads above complete inside their own asm statement (the wait is
// part of it): the compiler sees their registers written only once the
// asynchronous transfer is done, so no spill or reuse of a register races
// with it.

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
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
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
// 2^x on the special-function unit (one MUFU op; relative error ~2^-22, far
// below the bf16/fp16 rounding of the operands it feeds).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// max(a, b), NaN if either is NaN (one instruction; fmaxf would drop the NaN).
__device__ __forceinline__ float maxnan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}
// max(a, b, c), NaN if any is NaN (one three-input instruction on sm_100+).
__device__ __forceinline__ float maxnan3(float a, float b, float c) {
    float d;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// Largest magnitude of n (even) values; NaN when one is NaN, so a check
// written as !(absmax <= limit) also rejects NaN.
__device__ __forceinline__ float absmax(const float *v, int n) {
    float m = 0.f;
    for (int i = 0; i < n; i += 2) m = maxnan3(m, fabsf(v[i]), fabsf(v[i + 1]));
    return m;
}

// ---------------------------------------------------------------------------
// 64 x 64 unit-lower-triangular inverse, off-diagonal blocks.
// A is fp32 [64][AS] (strictly lower, rows scaled by beta); T is fp32 [64][64]
// with its columns XOR-swizzled by row: T[r][c] lives at r*64 + tsw(r, c).
// Block column J belongs to two warps (8 columns each): for I = J+1 .. 3 they form
//     R = sum_{K=J}^{I-1} A_IK T_KJ,   T_IJ = -T_II R
// from blocks of lower levels only, so the warps need no block-wide barrier.
// The 16 x 16 x 16 products run as warp-level m16n8k8 TF32 MMAs (fp32
// accumulate): they are latency-bound and far below the 64-row minimum of the
// 5th-generation MMA; T is rounded to bf16 right after.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int tsw(int r, int c) { return c ^ ((r & 3) << 3); }
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9},"
        " {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
constexpr int RW = 8;    // row stride (floats) of a warp's 16 x 8 R scratch

// T Diag(beta) element pair (r, c), (r, c + 1), c even, as fp16 into the
// K-major [T Diag(b); 0; Aqk] tile (64 token columns, one 128-byte row per r);
// returns the larger magnitude (NaN if either is NaN).
__device__ __forceinline__ float store_tb2(uint8_t *tbz, int r, int c, float t0, float t1,
                                           const float *beta) {
    const float a = t0 * beta[c], b = t1 * beta[c + 1];
    *reinterpret_cast<uint32_t *>(tbz + r * 128 + ((((c >> 3) ^ r) & 7) << 4) + (c & 7) * 2) =
        pack_f16x2(a, b);
    return maxnan3(0.f, fabsf(a), fabsf(b));
}

template <int J>
__device__ __forceinline__ float solve_block_column(const float *As, float *Ts, float *Rw, int lane,
                                                   uint8_t *tbz, const float *beta, int nt) {
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
                mma_tf32(rc, a, b);
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
            mma_tf32(tc, a, b);
        }
        const int cl = 16 * J + 8 * nt + 2 * t4;
        const int c = cl ^ sw;
        Ts[(16 * I + g) * 64 + c] = -tc[0];
        Ts[(16 * I + g) * 64 + c + 1] = -tc[1];
        Ts[(16 * I + g + 8) * 64 + c] = -tc[2];
        Ts[(16 * I + g + 8) * 64 + c + 1] = -tc[3];
        bound = maxnan3(bound, store_tb2(tbz, 16 * I + g, cl, -tc[0], -tc[1], beta),
                        store_tb2(tbz, 16 * I + g + 8, cl, -tc[2], -tc[3], beta));
        __syncwarp();
    }
    return bound;
}

// O of a chunk, from rows 64..127 of its P columns (TMEM column ocol on):
// this warp's lane quarter lq (2 or 3) and columns 32 cq .. 32 cq + 31, scaled,
// rounded to bf16 and stored for the chunk's first L tokens (the chunk starts
// at token t0).
__device__ __forceinline__ void store_o(const Params &p, uint32_t tmem, uint32_t ocol, int lq, int cq, int lane,
                                        int t0, int L, int h) {
    uint32_t r[32];
    KDA_TMEM_LD32(tmem + ((uint32_t)(32 * lq) << 16) + ocol + 32 * cq, r);
    const int row = 32 * (lq - 2) + lane;
    if (row < L) {
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + ((size_t)(t0 + row) * p.H + h) * VD + 32 * cq);
        const float sc = p.scale;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float *f = reinterpret_cast<const float *>(r + 8 * j);
            dst[j] = make_uint4(pack_bf16x2(sc * f[0], sc * f[1]), pack_bf16x2(sc * f[2], sc * f[3]),
                                pack_bf16x2(sc * f[4], sc * f[5]), pack_bf16x2(sc * f[6], sc * f[7]));
        }
    }
}

// O of a full chunk by tensor store: the warp stages its 32 tokens x 32
// channels as one 64-byte-swizzled box (2 KB) in the staging tile, and lane 0
// stores it; lane 0 waits for the box to be read (tma_store_wait_read) before
// the staging tile is written again.
__device__ __forceinline__ void store_o_tma(const Params &p, uint8_t *sm, uint32_t sbase, uint32_t tmem,
                                            uint32_t ocol, int lq, int cq, int lane, int t0, int h) {
    uint32_t r[32];
    KDA_TMEM_LD32(tmem + ((uint32_t)(32 * lq) << 16) + ocol + 32 * cq, r);
    const int box = 4 * (lq - 2) + cq;
    const uint32_t stage = OP_OST + box * 2048;
    const float sc = p.scale;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float *f = reinterpret_cast<const float *>(r + 8 * j);
        *reinterpret_cast<uint4 *>(sm + stage + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
            make_uint4(pack_bf16x2(sc * f[0], sc * f[1]), pack_bf16x2(sc * f[2], sc * f[3]),
                       pack_bf16x2(sc * f[4], sc * f[5]), pack_bf16x2(sc * f[6], sc * f[7]));
    }
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) tma_store_3d(&p.to, sbase + stage, 32 * cq, h, t0 + 32 * (lq - 2));
}

// The recurrence over one chunk on the CUDA cores, in fp32, by all 512
// threads: thread t keeps S[32 (t / 128) + j][t % 128] (j < 32), read from and
// written back to the staged state P ([128][FB_LD] fp32); o of every token is
// stored.  Per token: the inputs are staged (alpha = exp(gk), k, q, v, beta;
// double-buffered by token parity), each thread decays its 32 rows and forms
// its share of S'^T k and S'^T q, and after the shares are summed it applies
// u = beta (v - S'^T k) and o = scale (S'^T q + u (k . q)).
__device__ __noinline__ void chunk_recurrent(const Params &p, uint8_t *sm, float *P, int t0, int L, int h) {
    const int t = threadIdx.x, v = t & 127, kq = t >> 7, lane = t & 31, w = t >> 5;
    float *part = reinterpret_cast<float *>(sm + FB_P);   // [4 pk | 4 pq][128]
    float *xs = reinterpret_cast<float *>(sm + FB_X);     // [2][4] k.q partials, [2] beta
    float s[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) s[j] = P[(32 * kq + j) * FB_LD + v];
    for (int tk = 0; tk < L; ++tk) {
        const int tg = t0 + tk, b = tk & 1;
        float *in = reinterpret_cast<float *>(sm + FB_IN + b * 2048);   // alpha, k, q, v
        const size_t row = ((size_t)tg * p.H + h) * KD;
        if (t < 128) {
            const float kk = __bfloat162float(p.k[row + t]), qq = __bfloat162float(p.q[row + t]);
            in[t] = expf(__bfloat162float(p.gk[row + t]));
            in[128 + t] = kk;
            in[256 + t] = qq;
            float x = kk * qq;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
            if (lane == 0) xs[b * 4 + w] = x;
        } else if (t < 256) {
            in[384 + t - 128] = __bfloat162float(p.v[row + t - 128]);
            if (t == 128) xs[8 + b] = __bfloat162float(p.beta[(size_t)tg * p.H + h]);
        }
        __syncthreads();
        const float4 *al = reinterpret_cast<const float4 *>(in + 32 * kq);
        const float4 *kv = reinterpret_cast<const float4 *>(in + 128 + 32 * kq);
        const float4 *qv = reinterpret_cast<const float4 *>(in + 256 + 32 * kq);
        float pk = 0.f, pq = 0.f;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
            const float4 a = al[j4], kk = kv[j4], qq = qv[j4];
            s[4 * j4] *= a.x; s[4 * j4 + 1] *= a.y; s[4 * j4 + 2] *= a.z; s[4 * j4 + 3] *= a.w;
            pk = fmaf(s[4 * j4], kk.x, pk); pk = fmaf(s[4 * j4 + 1], kk.y, pk);
            pk = fmaf(s[4 * j4 + 2], kk.z, pk); pk = fmaf(s[4 * j4 + 3], kk.w, pk);
            pq = fmaf(s[4 * j4], qq.x, pq); pq = fmaf(s[4 * j4 + 1], qq.y, pq);
            pq = fmaf(s[4 * j4 + 2], qq.z, pq); pq = fmaf(s[4 * j4 + 3], qq.w, pq);
        }
        part[kq * 128 + v] = pk;
        part[512 + kq * 128 + v] = pq;
        __syncthreads();
        const float wv = (part[v] + part[128 + v]) + (part[256 + v] + part[384 + v]);
        const float sq = (part[512 + v] + part[640 + v]) + (part[768 + v] + part[896 + v]);
        const float kqd = (xs[b * 4] + xs[b * 4 + 1]) + (xs[b * 4 + 2] + xs[b * 4 + 3]);
        const float u = xs[8 + b] * (in[384 + v] - wv);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
            const float4 kk = kv[j4];
            s[4 * j4] = fmaf(kk.x, u, s[4 * j4]); s[4 * j4 + 1] = fmaf(kk.y, u, s[4 * j4 + 1]);
            s[4 * j4 + 2] = fmaf(kk.z, u, s[4 * j4 + 2]); s[4 * j4 + 3] = fmaf(kk.w, u, s[4 * j4 + 3]);
        }
        if (kq == 0) p.o[((size_t)tg * p.H + h) * VD + v] = __float2bfloat16_rn(p.scale * (sq + u * kqd));
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) P[(32 * kq + j) * FB_LD + v] = s[j];
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(NT, 1) prefill_tc_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lq = warp & 3;     // TMEM lane quarter this warp may access
    const int cq = warp >> 2;    // column quarter (0..3)
    float *beta_s = reinterpret_cast<float *>(sm + SM_BETA);
    float *gam_s = reinterpret_cast<float *>(sm + SM_GAM);
    float *As = reinterpret_cast<float *>(sm + SCR_A);
    float *Rws = reinterpret_cast<float *>(sm + SCR_RW);   // per-warp R scratch of the solve
    float *Ts = reinterpret_cast<float *>(sm + SCR_T);
    const uint32_t bar_qkg = sbase + SM_BAR, bar_v = sbase + SM_BAR + 8,
                   bar_mma = sbase + SM_BAR + 16, bar_st = sbase + SM_BAR + 24,
                   bar_p = sbase + SM_BAR + 32;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + SM_MISC);
    int *flags = reinterpret_cast<int *>(sm + SM_MISC + 4);

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
        mbar_init(bar_qkg, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_st, 1);
        mbar_init(bar_p, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *flags = 0;
        // the initial state, by four tensor copies into the staging tile
        if (si >= 0) {
            mbar_expect_tx(bar_st, STATE_ELEMS * sizeof(float));
            for (int j = 0; j < 4; ++j) tma_load_2d(sbase + STG + j * 16384, &p.tpool, bar_st, 32 * j, (si * p.H + h) * KD);
        }
        // the first chunk's raw tiles, issued before anything else so that they
        // land while TMEM is allocated and the state is loaded
        if (nchunks > 0 && !p.skip_first_load) {
            mbar_expect_tx(bar_qkg, 3 * 16384);
            for (int b = 0; b < 2; ++b) {
                tma_load_3d(sbase + RAW_Q + b * 8192, &p.tq, bar_qkg, 64 * b, h, bos);
                tma_load_3d(sbase + RAW_K + b * 8192, &p.tk, bar_qkg, 64 * b, h, bos);
                tma_load_3d(sbase + RAW_G + b * 8192, &p.tg, bar_qkg, 64 * b, h, bos);
            }
        }
        if (nchunks > 0) {
            mbar_expect_tx(bar_v, 16384);
            for (int b = 0; b < 2; ++b)
                tma_load_3d(sbase + RAW_V + b * 8192, &p.tv, bar_v, 64 * b, h, bos);
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
    const uint64_t wait_ns = p.wait_ns ? p.wait_ns : WAIT_NS;


    // ---- initial state: row k = 32*lq + lane, columns 32*cq .. 32*cq+31 ---
    const int srow = 32 * lq + lane;
    float *stg = reinterpret_cast<float *>(sm + STG);
    float S[32];
    if (si >= 0) {   // uniform across the CTA
        if (tid == 0 && !barrier_wait_for(bar_st, 0, wait_ns)) atomicOr(flags, FLAG_TIMEOUT);
        __syncthreads();
        const float *box = stg + cq * (KD * 32);   // columns 32 cq .. 32 cq + 31
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 t = *reinterpret_cast<const float4 *>(box + srow * 32 + ((j ^ (srow & 7)) << 2));
            S[4 * j] = t.x; S[4 * j + 1] = t.y; S[4 * j + 2] = t.z; S[4 * j + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) S[j] = 0.f;
    }
    __syncthreads();   // the staging tile is read before the S0 tile over it is written
    // a state beyond fp16 sends the next chunk down the recurrent path
    bool fb_next = !(absmax(S, 32) <= FP16_LIMIT);
#pragma unroll
    for (int j = 0; j < 4; ++j) store_f16(sm + OP_S, chunk_off(srow, 32 * cq + 8 * j, 128), S + 8 * j);

    const float LOG2E = 1.4426950408889634f;
    // beta of the chunk about to be processed, loaded one chunk ahead.  The raw
    // bf16 bits stay in a register and are converted only when the next chunk
    // stores them, so no thread waits for this load inside the chunk; a token
    // past the sequence loads its sequence's first beta and stores 0.
    const unsigned short *beta_bits = reinterpret_cast<const unsigned short *>(p.beta);
    unsigned short beta_raw = 0;
    bool beta_ok = false;
    if (tid < C && nchunks > 0) {
        beta_ok = tid < eos - bos;
        beta_raw = __ldg(beta_bits + (size_t)(beta_ok ? bos + tid : bos) * p.H + h);
    }
    constexpr uint32_t ID_G1 = idesc(128, 64, 0, 0, 2);
    constexpr uint32_t ID_P = idesc(128, 128, 0, 1, 0);
    constexpr uint32_t ID_U = idesc(128, 128, 0, 1, 0);
    constexpr uint32_t ID_G4A = idesc(128, 128, 0, 1, 0);
    constexpr uint32_t ID_G4B = idesc(128, 128, 1, 1, 0);
    // This thread's share of the raw q, k, gk tiles, taken into registers while
    // the previous chunk's G4 runs (for chunk 0: here).  Warp w owns key
    // channels 8w .. 8w+7; lane l owns rows 2l and 2l + 1, taken in the order
    // rA, rB: lanes with bit 2 set take the odd row first, so that the 8 lanes
    // of each quarter-warp cover all 8 positions of the 128-byte swizzle in
    // every load and in every store of the prep phase.
    uint4 wqA, wqB, wkA, wkB, wgA, wgB;
    auto load_raw = [&]() {
        const int ch = 8 * warp, sw = (lane >> 2) & 1;
        const int rA = 2 * lane + sw, rB = 2 * lane + 1 - sw;
        wqA = *reinterpret_cast<const uint4 *>(sm + RAW_Q + chunk_off(rA, ch, 64));
        wqB = *reinterpret_cast<const uint4 *>(sm + RAW_Q + chunk_off(rB, ch, 64));
        wkA = *reinterpret_cast<const uint4 *>(sm + RAW_K + chunk_off(rA, ch, 64));
        wkB = *reinterpret_cast<const uint4 *>(sm + RAW_K + chunk_off(rB, ch, 64));
        wgA = *reinterpret_cast<const uint4 *>(sm + RAW_G + chunk_off(rA, ch, 64));
        wgB = *reinterpret_cast<const uint4 *>(sm + RAW_G + chunk_off(rB, ch, 64));
    };
    // the exact state after (m + 1) * ckpt_chunks full chunks, once chunk c is done
    auto store_ckpt = [&](int c) {
        const int m = (c + 1) / max(p.ckpt_chunks, 1) - 1;
        if (nck > 0 && (c + 1) % p.ckpt_chunks == 0 && m < nck) {
            const int cs = p.ckpt_slots[(size_t)n * p.max_ckpts + m];
            if (cs >= 0) {
                float4 *dst = reinterpret_cast<float4 *>(
                    p.pool + ((size_t)cs * p.H + h) * STATE_ELEMS + (size_t)srow * VD + 32 * cq);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    __stcs(dst + j, make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]));
            }
        }
    };
    if (nchunks > 0 && !barrier_wait_for(bar_qkg, 0, wait_ns)) atomicOr(flags, FLAG_TIMEOUT);
    load_raw();
    __syncthreads();   // the raw tiles may now be overwritten
    bool aborted = (*flags & FLAG_TIMEOUT) != 0;
    bool fb_prev = false;   // the previous chunk took the recurrent path (its o is written)
    uint32_t nmma = 0;      // commits of bar_mma waited for so far: the parity of the next
    uint32_t np = 0;        // P products issued so far (one commit of bar_p each)
    for (int c = 0; c < nchunks && !aborted; ++c) {
        const int t0 = bos + c * C;
        const int L = min(C, eos - t0);
        const uint32_t par = (uint32_t)(c & 1);

        // (1) beta of this chunk into shared memory; the next chunk's is loaded
        if (tid < C) {
            beta_s[tid] = beta_ok ? __uint_as_float((uint32_t)beta_raw << 16) : 0.f;
            const int tn = t0 + C + tid;
            beta_ok = c + 1 < nchunks && tn < eos;
            beta_raw = __ldg(beta_bits + (size_t)(beta_ok ? tn : bos) * p.H + h);
        }

        // (2) cumulative decays and the operand tiles
        bool bad;
        // FULL: all 64 rows are tokens of the sequence (no row masks)
        auto prep = [&](auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            const int ch = 8 * warp, sw = (lane >> 2) & 1;
            const int rA = 2 * lane + sw, rB = 2 * lane + 1 - sw;
            float gA[8], gB[8];
            unpack_bf16(wgA, gA);
            unpack_bf16(wgB, gB);
            const bool vA = FULL || rA < L, vB = FULL || rB < L;
            // G at rows 2l and 2l+1: inclusive warp scan of the row-pair sums
            float gref[8], glast[8];
            float gmax = 0.f, qkmax = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float a = vA ? gA[i] : 0.f, b = vB ? gB[i] : 0.f;
                gmax = maxnan3(gmax, a, b);
                float s2 = a + b;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float t = __shfl_up_sync(0xffffffffu, s2, off);
                    if (lane >= off) s2 += t;
                }
                const float odd = sw ? a : b;   // the term of row 2l + 1
                gA[i] = sw ? s2 : s2 - odd;
                gB[i] = sw ? s2 - odd : s2;
                gref[i] = __shfl_sync(0xffffffffu, s2, 15);    // G at row 31
                glast[i] = __shfl_sync(0xffffffffu, s2, 31);   // G at row 63 (= last valid row)
            }
            // With every gk <= 0 (checked: gmax) G never increases down the rows,
            // and a sum of non-positive terms never increases under rounding
            // either, so |G_r - G_ref| is largest at the first or the last row:
            // at most -G_ref (the first row's G is <= 0) or G_ref - G_L.  A
            // one-nat margin covers the rounding of the scan; NaN fails the check.
            float egr[8], elr[8], gr2[8];   // per channel: exp(G_ref), exp(G_L - G_ref), G_ref log2(e)
            float dmax = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                dmax = maxnan3(dmax, -gref[i], gref[i] - glast[i]);
                gr2[i] = gref[i] * LOG2E;
                egr[i] = ex2(gr2[i]);
                elr[i] = ex2((glast[i] - gref[i]) * LOG2E);
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int r = half ? rB : rA;
                const bool valid = half ? vB : vA;
                const float *g = half ? gB : gA;
                float qq[8], kk[8];
                unpack_bf16(half ? wqB : wqA, qq);
                unpack_bf16(half ? wkB : wkA, kk);
                float kf[8], kb[8], kt[8], ke[8], qr[8], qt[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float q_ = valid ? qq[i] : 0.f, k_ = valid ? kk[i] : 0.f;
                    const float d = fmaf(g[i], LOG2E, -gr2[i]);   // (G_r - G_ref) log2(e)
                    qkmax = maxnan3(qkmax, fabsf(q_), fabsf(k_));
                    const float ef = ex2(d);                 // exp(G_r - G_ref)
                    const float eb = ex2(-d);                // exp(G_ref - G_r)
                    kf[i] = k_ * ef;
                    kb[i] = k_ * eb;
                    qr[i] = q_ * ef;
                    kt[i] = kf[i] * egr[i];                  // k exp(G_r)
                    qt[i] = qr[i] * egr[i];                  // q exp(G_r)
                    ke[i] = kb[i] * elr[i];                  // k exp(G_L - G_r)
                }
                store_f32x8(sm, OP_A1, r, ch, 128, kf);
                store_f32x8(sm, OP_A1, 64 + r, ch, 128, qr);
                store_f32x8(sm, OP_B1, r, ch, 64, kb);
                store_f16(sm, OP_A3 + chunk_off(r, ch, 128), kt);
                store_f16(sm, OP_KE + chunk_off(r, ch, 64), ke);
                store_f16(sm, OP_A3 + chunk_off(64 + r, ch, 128), qt);
            }
            bad = !(dmax <= D_LIMIT - 1.f) || !(qkmax <= QK_LIMIT) || !(gmax <= 0.f);
            if (lane == 31) {
#pragma unroll
                for (int i = 0; i < 8; ++i) gam_s[(c & 1) * 128 + ch + i] = expf(glast[i]);
            }
        };
        if (L == C) prep(std::integral_constant<bool, true>());
        else prep(std::integral_constant<bool, false>());
        fence_proxy_async();
        // Every check of a chunk is decided before its state update; a chunk
        // outside the operand formats leaves the tensor-core path for the
        // recurrence.  raw_next / o_prev / v_next record which hand-offs of the
        // chunk (next raw q, k, gk; the previous chunk's O; next v) are done.
        bool fb = __syncthreads_or(bad || fb_next);
        fb_next = false;
        bool raw_next = false, o_prev = false, v_next = false;

        const uint32_t pcol = TM_P + 128u * par, pcol_prev = TM_P + 128u * (par ^ 1u);
        const uint32_t ppar = np & 1u;   // parity of this chunk's P commit
        const bool p_issued = !fb;
        if (!fb) {
        ++np;
        // (3) G1 on TF32: [Kf; Qr] Kb^T (16 steps of K = 8); then P = [K~; Q~] S0
        //     (8 steps of K = 16) into this chunk's P columns.  P does not depend
        //     on the triangular solve, so it runs while the Gram matrix is read
        //     out and inverted.
        // G1 and P come from two threads (each commit tracks its own thread's
        // MMAs), so that thread 0 waits for G1 while P is still being issued.
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 16; ++s)
                mma_tf32(tmem, sdesc(sbase + OP_A1 + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024),
                         sdesc(sbase + OP_B1 + (s >> 2) * 8192 + (s & 3) * 32, 16, 1024), ID_G1, s > 0);
            mma_commit(bar_mma);
        } else if (tid == 32) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma(tmem + pcol, sdesc(sbase + OP_A3 + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024),
                    sdesc(sbase + OP_S + s * 2048, 16384, 1024), ID_P, s > 0);
            mma_commit(bar_p);
        }

        // (4) A -> fp32 scratch (strictly lower, x beta_r); Aqk -> fp16 rows
        //     128..191 of TBZ (lower incl. diagonal); then prefetch the next
        //     chunk's q, k, gk into R1 (G1 has consumed it)
        mma_wait_all(bar_mma, (nmma++) & 1u, flags, wait_ns);
        raw_next = true;
        if (tid == 0 && c + 1 < nchunks) {
            mbar_expect_tx(bar_qkg, 3 * 16384);
            for (int b = 0; b < 2; ++b) {
                tma_load_3d(sbase + RAW_Q + b * 8192, &p.tq, bar_qkg, 64 * b, h, t0 + C);
                tma_load_3d(sbase + RAW_K + b * 8192, &p.tk, bar_qkg, 64 * b, h, t0 + C);
                tma_load_3d(sbase + RAW_G + b * 8192, &p.tg, bar_qkg, 64 * b, h, t0 + C);
            }
        }
        float aqm = 0.f;
        {
            uint32_t r[16];
            KDA_TMEM_LD16(tmem + ((uint32_t)(32 * lq) << 16) + 16 * cq, r);
            const int row = 32 * (lq & 1) + lane;   // 0..63 within A or Aqk
            float v[16];
            if (lq < 2) {
                const float b = beta_s[row];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    v[j] = (16 * cq + j < row) ? __uint_as_float(r[j]) * b : 0.f;
                float4 *dst = reinterpret_cast<float4 *>(As + row * AS + 16 * cq);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = (16 * cq + j <= row) ? __uint_as_float(r[j]) : 0.f;
                aqm = absmax(v, 16);
                store_f16(sm, OP_TBZ + (uint32_t)(64 + row) * 128 + ((((2 * cq) ^ row) & 7) << 4), v);
                store_f16(sm, OP_TBZ + (uint32_t)(64 + row) * 128 + ((((2 * cq + 1) ^ row) & 7) << 4),
                          v + 8);
            }
        }
        tc_fence_before();
        fb = __syncthreads_or(!(aqm <= FP16_LIMIT));
        }
        if (!fb) {
        // (5) T = (I + A)^-1 in 16 x 16 blocks: diagonal blocks T_II by forward
        //     substitution (warps 2-3), then block columns (solve_block_column,
        //     warps 0-5); T Diag(b) goes to TBZ in fp16.  During the diagonal
        //     phase warps 6, 7, 10, 11, 14, 15 write out the previous chunk's O, and
        //     the eight warps of sub-partitions 0 and 1 (TMEM lanes 0..63) read
        //     K~ S0 out of P and turn v into V' = V - K~ S0 (fp16, in place), so
        //     that the block columns run with nothing else beside them.
        float xm = 0.f;   // magnitude of this thread's fp16 operands (T Diag(b) or V')
        if (lq < 2) {
            // sub-partitions 0 and 1 (TMEM lanes 0..63): zero the blocks of T Diag(b)
            // above the diagonal, then V' = V - K~ S0 for token row 32 lq + lane,
            // value channels 32 cq .. 32 cq + 31
            const int t = 64 * cq + 32 * lq + lane;   // 0 .. 255
            if (t < 96) {   // 6 upper blocks x 16 rows, two 16-byte chunks each
                const int blk = t >> 4, r = t & 15;
                const int I = (blk < 3) ? 0 : (blk < 5 ? 1 : 2);
                const int J = (blk < 3) ? blk + 1 : (blk < 5 ? blk - 1 : 3);
                const int rr = 16 * I + r;
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int cchunk = 2 * J + h2;
                    *reinterpret_cast<uint4 *>(sm + OP_TBZ + rr * 128 + (((cchunk ^ rr) & 7) << 4)) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            const int row = 32 * lq + lane;
            if (!barrier_wait_for(bar_p, ppar, wait_ns) || !barrier_wait_for(bar_v, par, wait_ns))
                atomicOr(flags, FLAG_TIMEOUT);
            tc_fence_after();
            uint32_t r[32];
            KDA_TMEM_LD32(tmem + ((uint32_t)(32 * lq) << 16) + pcol + 32 * cq, r);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t off = RAW_V + chunk_off(row, 32 * cq + 8 * j, 64);
                float vv[8];
                unpack_bf16(*reinterpret_cast<const uint4 *>(sm + off), vv);
#pragma unroll
                for (int e = 0; e < 8; ++e) vv[e] = row < L ? vv[e] - __uint_as_float(r[8 * j + e]) : 0.f;
                xm = maxnan(xm, absmax(vv, 8));
                store_f16(sm, off, vv);
            }
            tc_fence_before();
        } else if (warp == 2 || warp == 3) {
            // diagonal blocks: one block per half-warp, lane = column
            const int I = 2 * (warp - 2) + (lane >> 4), col = lane & 15;
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
            const int c = 16 * I + col;
            const float bc = beta_s[c];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int rr = 16 * I + r;
                Ts[rr * 64 + tsw(r, c)] = x[r];
                const float tv = x[r] * bc;
                xm = maxnan(xm, fabsf(tv));
                *reinterpret_cast<__half *>(sm + OP_TBZ + rr * 128 + ((((c >> 3) ^ rr) & 7) << 4) +
                                            (c & 7) * 2) = __float2half_rn(tv);
            }
        } else if (warp >= 6 && c > 0 && !fb_prev) {
            // the previous chunk's O by tensor stores (32 x 32 boxes): warps 6 and 7
            // take column quarters 0 and 1, warps 10, 11 quarter 2, warps 14, 15 quarter 3
            const int q0 = warp < 8 ? 0 : (warp < 12 ? 2 : 3), nq = warp < 8 ? 2 : 1;
#pragma unroll 1
            for (int q = q0; q < q0 + nq; ++q) store_o_tma(p, sm, sbase, tmem, pcol_prev, lq, q, lane, t0 - C, h);
            tc_fence_before();
        }
        o_prev = true;
        __syncthreads();
        // block columns J = 0, 1, 2 on warps (0, 1), (2, 3), (4, 5): one warp-level
        // tensor unit per sub-partition and chain, as far as it goes
        if (warp < 2) xm = maxnan(xm, solve_block_column<0>(As, Ts, Rws + warp * 16 * RW, lane, sm + OP_TBZ, beta_s, warp & 1));
        else if (warp < 4) xm = maxnan(xm, solve_block_column<1>(As, Ts, Rws + warp * 16 * RW, lane, sm + OP_TBZ, beta_s, warp & 1));
        else if (warp < 6) xm = maxnan(xm, solve_block_column<2>(As, Ts, Rws + warp * 16 * RW, lane, sm + OP_TBZ, beta_s, warp & 1));
        if (warp >= 6 && lq >= 2 && lane == 0 && c > 0 && !fb_prev) tma_store_wait_read();   // the O boxes are read
        fence_proxy_async();
        fb = __syncthreads_or(!(xm <= FP16_LIMIT));
        if (*flags & FLAG_TIMEOUT) { aborted = true; break; }
        }
        if (!fb) {
        // (6) U = [T Diag(b); Aqk] V' (rows 0-63 kept)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma(tmem, sdesc(sbase + OP_TBZ + s * 32, 16, 1024), sdesc(sbase + RAW_V + s * 2048, 8192, 1024),
                    ID_U, s > 0);
            mma_commit(bar_mma);
        }
        mma_wait_all(bar_mma, (nmma++) & 1u, flags, wait_ns);
        // (7) U -> fp16 MN-major [token][v]; prefetch the next v (U consumed V')
        v_next = true;
        if (tid == 0 && c + 1 < nchunks) {
            mbar_expect_tx(bar_v, 16384);
            for (int b = 0; b < 2; ++b)
                tma_load_3d(sbase + RAW_V + b * 8192, &p.tv, bar_v, 64 * b, h, t0 + C);
        }
        float um = 0.f;
        if (lq < 2) {
            uint32_t r[32];
            KDA_TMEM_LD32(tmem + ((uint32_t)(32 * lq) << 16) + 32 * cq, r);
            const int row = 32 * lq + lane;
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
            um = absmax(v, 32);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                store_f16(sm, OP_U + chunk_off(row, 32 * cq + 8 * j, 64), v + 8 * j);
        }
        fence_proxy_async();
        tc_fence_before();
        fb = __syncthreads_or(!(um <= FP16_LIMIT));
        }
        if (!fb) {
        // (8) G4a: [T Diag(b); Aqk] x U onto P (rows 64..127: Q~ S0 becomes O);
        //     G4b: K_end^T x U into cols 0..127
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t b = sdesc(sbase + OP_U + s * 2048, 8192, 1024);
                mma(tmem + pcol, sdesc(sbase + OP_TBZ + s * 32, 16, 1024), b, ID_G4A, 1);
                mma(tmem, sdesc(sbase + OP_KE + s * 2048, 8192, 1024), b, ID_G4B, s > 0);
            }
            mma_commit(bar_mma);
        }
        // the next chunk's raw tiles (prefetched after G1) into registers; the
        // barrier of the G4 wait then frees them for the next prep.  After the
        // last chunk the shared-memory reads still run (their values go unused)
        // so that these registers are never live across a whole chunk.
        if (c + 1 < nchunks && !barrier_wait_for(bar_qkg, par ^ 1u, wait_ns)) atomicOr(flags, FLAG_TIMEOUT);
        load_raw();
        mma_wait_all(bar_mma, (nmma++) & 1u, flags, wait_ns);
        if (*flags & FLAG_TIMEOUT) { aborted = true; break; }
        // (9) the state update (O is written out during the next chunk's solve)
        {
            // two 16-column reads keep the next chunk's raw tiles in registers
            const float gm = gam_s[(c & 1) * 128 + srow];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t r[16];
                KDA_TMEM_LD16(tmem + ((uint32_t)(32 * lq) << 16) + 32 * cq + 16 * hh, r);
#pragma unroll
                for (int j = 0; j < 16; ++j) S[16 * hh + j] = fmaf(gm, S[16 * hh + j], __uint_as_float(r[j]));
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    store_f16(sm, OP_S + chunk_off(srow, 32 * cq + 16 * hh + 8 * j, 128), S + 16 * hh + 8 * j);
            }
            fb_next = !(absmax(S, 32) <= FP16_LIMIT);
            store_ckpt(c);
        }
        // No block barrier here: each warp goes on to the next chunk's loads
        // and scan.  The next chunk's first barrier orders these TMEM reads
        // before G1 overwrites the columns, and these S stores before P reads
        // them (they reach the MMA's proxy through the fence below).  gam_s is
        // double-buffered by chunk parity; nothing else this epilogue reads is
        // written before that barrier.  O stays in this chunk's P columns until
        // the next chunk's solve.
        fence_proxy_async();
        tc_fence_before();
        } else {
            // ---- the chunk by the recurrence, from S (the state entering it) ----
            if (tid == 0) {
                if (!raw_next && c + 1 < nchunks) {   // R1's tiles are unused: the next raw q, k, gk
                    mbar_expect_tx(bar_qkg, 3 * 16384);
                    for (int b = 0; b < 2; ++b) {
                        tma_load_3d(sbase + RAW_Q + b * 8192, &p.tq, bar_qkg, 64 * b, h, t0 + C);
                        tma_load_3d(sbase + RAW_K + b * 8192, &p.tk, bar_qkg, 64 * b, h, t0 + C);
                        tma_load_3d(sbase + RAW_G + b * 8192, &p.tg, bar_qkg, 64 * b, h, t0 + C);
                    }
                }
                if (!v_next) {   // this chunk's v (unused) has landed; then the next v
                    if (!barrier_wait_for(bar_v, par, wait_ns)) atomicOr(flags, FLAG_TIMEOUT);
                    if (c + 1 < nchunks) {
                        mbar_expect_tx(bar_v, 16384);
                        for (int b = 0; b < 2; ++b)
                            tma_load_3d(sbase + RAW_V + b * 8192, &p.tv, bar_v, 64 * b, h, t0 + C);
                    }
                }
            }
            // P, if issued, reads the tiles the staged state is written over
            if (tid == 0 && p_issued && !barrier_wait_for(bar_p, ppar, wait_ns)) atomicOr(flags, FLAG_TIMEOUT);
            if (!o_prev && c > 0 && !fb_prev && lq >= 2) {   // the previous chunk's O, still in TMEM
                tc_fence_after();
                store_o(p, tmem, pcol_prev, lq, cq, lane, t0 - C, C, h);
            }
            __syncthreads();
            float *P = reinterpret_cast<float *>(sm + STG);
#pragma unroll
            for (int j = 0; j < 32; ++j) P[srow * FB_LD + 32 * cq + j] = S[j];
            __syncthreads();
            chunk_recurrent(p, sm, P, t0, L, h);
            __syncthreads();
#pragma unroll
            for (int j = 0; j < 32; ++j) S[j] = P[srow * FB_LD + 32 * cq + j];
            if (c + 1 < nchunks && !barrier_wait_for(bar_qkg, par ^ 1u, wait_ns)) atomicOr(flags, FLAG_TIMEOUT);
            load_raw();
            tc_fence_before();
            __syncthreads();   // the staged state is read before the tiles over it are written
            if (*flags & FLAG_TIMEOUT) { aborted = true; break; }
#pragma unroll
            for (int j = 0; j < 4; ++j) store_f16(sm + OP_S, chunk_off(srow, 32 * cq + 8 * j, 128), S + 8 * j);
            fb_next = !(absmax(S, 32) <= FP16_LIMIT);
            store_ckpt(c);
            fence_proxy_async();
        }
        fb_prev = fb;
    }
    __syncthreads();
    if (*flags & FLAG_TIMEOUT) aborted = true;
    if (!aborted && nchunks > 0 && lq >= 2 && !fb_prev) {
        tc_fence_after();
        const int tl = bos + (nchunks - 1) * C;
        store_o(p, tmem, TM_P + 128u * ((nchunks - 1) & 1), lq, cq, lane, tl, eos - tl, h);
    }

    if (aborted) {
        if (tid == 0) {
            report(p.err, DEVERR_TIMEOUT);
            // the self-test's unit gave up before its first v was consumed: let
            // that copy land (bounded) before the CTA's shared memory is released
            if (p.skip_first_load && nchunks > 0) barrier_wait_for(bar_v, 0, wait_ns);
        }
    } else {   // uniform; no copy or MMA is in flight, all of shared memory is free
#pragma unroll
        for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4 *>(stg + srow * VD + 4 * ((8 * cq + j) ^ (srow & 7))) =
                make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
        __syncthreads();
        float4 *dst = reinterpret_cast<float4 *>(p.pool + ((size_t)so * p.H + h) * STATE_ELEMS);
        float4 *d2 = ss >= 0 ? reinterpret_cast<float4 *>(p.pool + ((size_t)ss * p.H + h) * STATE_ELEMS) : nullptr;
        float4 t[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = i * NT + tid, r = e >> 5, c4 = e & 31;
            t[i] = *reinterpret_cast<const float4 *>(stg + r * VD + 4 * (c4 ^ (r & 7)));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            __stcs(dst + i * NT + tid, t[i]);
            if (d2) __stcs(d2 + i * NT + tid, t[i]);
        }
    }
    if (lq >= 2 && lane == 0) tma_store_wait_all();
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

// [T][H][128] bf16 viewed as a 3-D tensor {128, H, T}; boxes of bc channels x 1 head x bt tokens.
bool make_map(CUtensorMap *m, const void *base, int H, int T, cuuint32_t bc = 64, cuuint32_t bt = C,
              CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};
    cuuint32_t box[3] = {bc, 1, bt};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The state pool as a 2-D fp32 tensor [num_slots * H * 128 rows][128 columns],
// boxes of 32 columns x 128 rows (a head's state is four boxes), 128-byte swizzle.
bool make_pool_map(CUtensorMap *m, const float *pool, int num_slots, int H) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t rows = (cuuint64_t)num_slots * (cuuint64_t)H * KD;
    if (rows == 0 || rows > 0x7fffffffull) return false;   // row coordinates are 32-bit
    cuuint64_t dims[2] = {VD, rows};
    cuuint64_t strides[1] = {VD * sizeof(float)};
    cuuint32_t box[2] = {32, KD};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(pool), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

cudaError_t launch_prefill_chunked(const PrefillArgs &a, cudaStream_t s) {
    using namespace tc;
    Params p;   // ~9 KB, copied into the launch parameters
    memset(&p, 0, sizeof(p));
    if (a.T_total > 0) {
        if (!make_map(&p.tq, a.q, a.H, a.T_total) || !make_map(&p.tk, a.k, a.H, a.T_total) ||
            !make_map(&p.tg, a.gk, a.H, a.T_total) || !make_map(&p.tv, a.v, a.H, a.T_total) ||
            !make_map(&p.to, a.o, a.H, a.T_total, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    }
    if (!make_pool_map(&p.tpool, a.pool, a.num_slots, a.H)) return cudaErrorInvalidValue;
    p.N = a.N; p.T_total = a.T_total; p.H = a.H; p.num_slots = a.num_slots;
    p.beta = (const __nv_bfloat16 *)a.beta; p.cu = a.cu; p.pool = a.pool;
    p.init_slot = a.init_slot; p.out_slot = a.out_slot; p.snap_slot = a.snap_slot;
    p.o = (__nv_bfloat16 *)a.o; p.scale = a.scale; p.err = a.err;
    p.ckpt_chunks = a.ckpt_interval / C; p.max_ckpts = a.max_ckpts; p.ckpt_slots = a.ckpt_slots;
    p.q = (const __nv_bfloat16 *)a.q; p.k = (const __nv_bfloat16 *)a.k;
    p.gk = (const __nv_bfloat16 *)a.gk; p.v = (const __nv_bfloat16 *)a.v;
    p.wait_ns = a.wait_ns; p.skip_first_load = a.skip_first_load;
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
