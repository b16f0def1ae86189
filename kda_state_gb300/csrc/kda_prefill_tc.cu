// Chunked KDA prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One 256-thread CTA per (sequence, head) unit walks the sequence in chunks of
// C = 32 tokens; two units share an SM (109 KB of shared memory and 256 TMEM
// columns each), so that one unit's tensor-core and memory waits are covered
// by the other's CUDA-core work.  The fp32 128 x 128 state lives in TMEM,
// transposed (lane v, column k), for the whole sequence.  This follows the
// layout the pages give for the CuTe rewrite of FlashKDA (chunk 32, one CTA per
// (sequence, head), state in TMEM, longest sequences first: Kimi K3 on B200
// deployment notes, timeline entry "FlashKDA"); the chunk algebra, the operand
// formats and the schedule below are this kernel's own.
//
// Chunk algebra (unrolling the recurrence
//     S_t = (I - b_t k_t k_t^T) Diag(exp(gk_t)) S_{t-1} + b_t k_t v_t^T,  o_t = S_t^T q_t
// over a chunk).  G_r = sum_{j<=r} gk_j per key channel (rows r of the chunk),
// S the state entering it, and (row r scaled per channel)
//     K~ = K . exp(G),  Q~ = Q . exp(G),  Kb = K . exp(-G):
//     A   = tril_-1(Diag(b) K~ Kb^T),   Aqk = tril(Q~ Kb^T),   T = (I + A)^-1
//     P   = [Q~; K~] S                  (Q~ S and K~ S in one product)
//     U   = T Diag(b) (V - K~ S)
//     O   = Q~ S + Aqk U
//     S_L = Diag(exp(G_L)) (S + Kb^T U)
// so the Gram operands are also the operands of P and of the state update.
// Every product runs in TF32 (8-bit exponent), so one reference row (the
// chunk start) serves the whole chunk while its decay stays within 60 nats.
//
// Per chunk (every product kind::tf32, fp32 accumulators in TMEM):
//   G1  [Q~; K~] (64 x 128, smem) x Kb^T                 -> TMEM, M = 64: Aqk, A
//   P   S^T (TMEM, A operand) x [Q~; K~]^T (smem)        -> TMEM cols 128..191
//   U   V'^T (TMEM) x (T Diag(b))^T (smem)               -> TMEM cols 224..255
//   X|O U^T (TMEM) x [Kb^T; Aqk]^T (smem, 160 rows), added onto
//       [S^T | Q~ S]                                     -> TMEM cols 0..159
// (an MMA of N up to 128 costs the same as one of N = 32, and so does N =
// 160: O rides on the state update)
// and at the end of the chunk one pass over TMEM writes O out and scales X by
// exp(G_L) into the next chunk's state.  The CUDA cores do the cumulative
// decays and exponentials (prep), the 32 x 32 unit-lower-triangular inverse
// (8 x 8 substitutions and an 8 x 8 product per diagonal 16 x 16 block,
// warp-level TF32 MMAs off it), V' = V - K~ S in TMEM, and the read-outs.  The next chunk's prep runs while
// this chunk's U, O and state-update products are on the tensor cores.
// Kb and Aqk are rounded to TF32 to nearest by the CUDA cores that write them;
// K~, Q~, V' and T Diag(b) are written unrounded, and they and the TMEM
// operands S and U are truncated to TF32 by the tensor core.  A CPU model of
// this data flow (the product roundings included) gives about 6e-3 x RMS on o
// and 7e-3 on the state on the workload's inputs; Kb truncated as well would
// take the state past 1e-2.
//
// Exactness over the whole input domain: a chunk whose factors could leave
// fp32 range in the products (a decay above 60 nats over the chunk, a positive
// gk, |q| or |k| above 256, |T Diag(b)| |V'| above 1e6, a NaN) is done by the
// recurrence token by token in fp32 on the CUDA cores, from the state in TMEM
// (the products read it but never write it before the checks are decided).
//
// All waits are bounded (barrier_wait_for, with a per-launch limit); a wait
// that gives up reports KDA_DEVERR_TIMEOUT, frees TMEM and abandons the unit
// without writing its slots.  Raw q, k, gk tiles arrive by TMA into the Gram
// operand tile as soon as P has consumed it, v into its own tile once V' is
// formed; the state enters and leaves TMEM through registers with coalesced
// global accesses.
#include <cuda.h>

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

constexpr int C = 32;      // chunk length
constexpr int NT = 256;    // threads per CTA
constexpr int AS = 36;     // row stride (floats) of the fp32 A scratch

// Shared-memory map (byte offsets from a 1024-aligned base).  fp32 operand
// tiles are K-major with the 128-byte swizzle, 32 channels (128 B) per box.
// The producer warps (0-3) write [Q~; K~], Kb, Kb^T, A, Aqk, T Diag(b) and the
// decay factors; the consumer warps (4-7) own v, the state and the recurrent
// path's scratch.  T Diag(b) and the decay factors, read across the two
// groups one chunk apart, are kept by chunk parity; Aqk and Kb^T are single,
// rewritten only after the consumer has finished the chunk before.
constexpr uint32_t OP_QR = 0;          // [Q~; K~]: 64 rows x 128 ch, 4 boxes of 8 KB
constexpr uint32_t RAW_Q = 0;          // raw bf16 tiles (TMA, 32 tokens x 128 ch, two
constexpr uint32_t RAW_K = 8192;       //  64-channel boxes of 4 KB) of the next chunk,
constexpr uint32_t RAW_G = 16384;      //  landing over [Q~; K~] once G1 and P have read it
constexpr uint32_t OP_KB = 32768;      // Kb: 32 rows x 128 ch, 4 boxes of 4 KB (B of G1)
constexpr uint32_t OP_KBT = 49152;     // Kb^T: 128 rows (k) x 32 tokens, one box (B of the update)
constexpr uint32_t OP_AQ = 65536;      // Aqk: 32 rows (r) x 32 tokens, right after Kb^T: rows 128..159 of the
                                       // update's B operand [Kb^T; Aqk] (N = 160: X^T and O^T in one product)
constexpr uint32_t OP_TB = 73728;      // T Diag(b) by chunk parity: 2 x (32 rows (r) x 32 tokens) (B of U)
constexpr uint32_t RAW_V = 81920;      // raw bf16 v (TMA), 2 boxes of 4 KB
constexpr uint32_t OP_OST = 90112;     // o of a full chunk (bf16, 2 boxes of 64 ch x 32 tokens, SW128) for its tensor store
constexpr uint32_t SCR_A = 98304;      // fp32 Diag(b) K~ Kb^T [32][AS]; A is its strictly lower part
constexpr uint32_t SCR_T = SCR_A + 32 * AS * 4;   // fp32 T of the diagonal blocks [32][TS]
constexpr int TS = 20;                             // its row stride (floats)
constexpr uint32_t SCR_R = SCR_T + 32 * TS * 4;    // fp32 R = A_10 T_00 [16][TS]
constexpr uint32_t FB_IN = SCR_R + 16 * TS * 4;    // recurrent path: 2 x {alpha, k, q, v}[128] fp32
constexpr uint32_t FB_X = FB_IN + 4096;            // recurrent path: [2][4] k.q partials, [2] beta
constexpr uint32_t SM_BETA = FB_X + 64;            // fp32 [32]
constexpr uint32_t SM_ELR = SM_BETA + 128;         // fp32 [2][128] exp(G_L) by chunk parity
constexpr uint32_t SM_TOT = SM_ELR + 1024;         // fp32 [4][128] row-octet sums of gk
constexpr uint32_t SM_ZERO = SM_TOT + 2048;        // 16 zero bytes (the raw tile of a row past the sequence)
constexpr uint32_t SM_FLAG = SM_ZERO + 64;         // [2] int recurrent-path verdicts, [2][2] max |T Diag(b)|, [4] max |V'|
constexpr uint32_t SM_BAR = SM_FLAG + 64;          // 9 mbarriers
constexpr uint32_t SM_MISC = SM_BAR + 128;         // TMEM base
constexpr uint32_t SMEM_USED = SM_MISC + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // + alignment slack
static_assert(SCR_A % 16 == 0 && SCR_T % 16 == 0 && SCR_R % 16 == 0 && FB_IN % 16 == 0, "scratch misaligned");
static_assert(OP_OST % 1024 == 0, "the o staging tile must be 1024-aligned for its 128-byte swizzle");
static_assert(SM_ELR % 16 == 0 && SM_TOT % 16 == 0, "factor arrays misaligned");
static_assert(RAW_G + 8192 <= OP_KB, "raw tiles overflow the Gram operand tile");
static_assert(OP_TB % 1024 == 0 && OP_AQ % 1024 == 0 && OP_KBT % 1024 == 0 && RAW_V % 1024 == 0, "operand tiles misaligned");
static_assert(OP_AQ == OP_KBT + 128 * 128, "Aqk must follow Kb^T: one B operand of 160 rows");
static_assert(2 * (SMEM_BYTES + 1024) <= 233472, "two CTAs must fit one SM");

// TMEM columns (256 per CTA, two CTAs per SM)
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t TM_X = 0;     // the state, transposed: lane v, column k
constexpr uint32_t TM_P = 128;   // P^T: columns 128..159 Q~ S -> O^T (right after X^T); 160..191 K~ S -> V'^T
constexpr uint32_t TM_O = TM_P;       // O^T
constexpr uint32_t TM_V = TM_P + 32;  // V'^T
constexpr uint32_t TM_G = 192;   // the Gram product (M = 64 layout), 32 columns
constexpr uint32_t TM_U = 224;   // U^T, 32 columns

constexpr uint64_t WAIT_NS = 2000000000ull;   // bounded waits: 2 s
constexpr unsigned K_LIMIT_BITS = 0x4380u;    // |k| bound of the tensor-core path: 256 as bf16 bits
constexpr float D_LIMIT = 60.f;               // decay over a chunk (natural log)
constexpr float U_LIMIT = 1.0e6f;             // max |T Diag(b)| x max |V'|

struct Params {
    CUtensorMap tq, tk, tg, tv, to;   // [T][H][128] bf16: boxes of 64 channels x 1 head x 32 tokens
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
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// Bulk tensor store of a shared-memory box; completes in this thread's bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// This thread's bulk stores have read their shared-memory source.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// This thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Named barrier of `count` threads (whole warps).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also ORs a predicate over its threads.
__device__ __forceinline__ int named_or(uint32_t id, uint32_t count, int pred) {
    int r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
        " selp.s32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"(pred), "r"(id), "r"(count)
        : "memory");
    return r;
}
// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor: fp32 accumulate, TF32 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D (TMEM) (+)= A (shared memory) x B (shared memory)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc));
}
// D (TMEM) (+)= A (TMEM, lane = row, column = K) x B (shared memory)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
        "r"(a), "l"(b), "r"(id), "r"(acc));
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
// TMEM stores complete inside their asm statement (the wait is part of it).
#define KDA_TMEM_ST32(taddr, r)                                                                   \
    asm volatile(                                                                                 \
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"  \
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"    \
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),                                            \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),   \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),        \
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),      \
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),      \
        "r"(r[29]), "r"(r[30]), "r"(r[31])                                                        \
        : "memory")

#define KDA_TMEM_ST16(taddr, r)                                                                   \
    asm volatile(                                                                                 \
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"  \
        "%13,%14,%15,%16};\n"                                                                    \
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),                                            \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),   \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),        \
        "r"(r[15])                                                                                \
        : "memory")

// Byte offset of the 16-byte chunk holding fp32 columns col..col+3 (col % 4 ==
// 0) of a tile of `rows` rows x 128 fp32 columns stored as four boxes of 32
// columns (rows x 128 B each, 128-byte swizzle: chunk index XOR row % 8).  This
// is the canonical K-major SW128 operand layout for 32-bit elements.
__device__ __forceinline__ uint32_t off32(int row, int col, int rows) {
    return (uint32_t)((col >> 5) * rows * 128 + row * 128 + ((((col >> 2) & 7) ^ (row & 7)) << 4));
}
// Byte offset of bf16 element (row, col) of a raw TMA tile: two boxes of 64
// channels, rows x 128 B each, 128-byte swizzle.
__device__ __forceinline__ uint32_t raw_off(int row, int col, int rows) {
    return (uint32_t)((col >> 6) * rows * 128 + row * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4) +
                      (col & 7) * 2);
}
// fp32 -> tf32 (round to nearest, ties away), kept in an fp32 register.
__device__ __forceinline__ float tf32r(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}
__device__ __forceinline__ float4 tf32r4(float a, float b, float c, float d) {
    return make_float4(tf32r(a), tf32r(b), tf32r(c), tf32r(d));
}
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
// 2^x on the special-function unit (one MUFU op; relative error ~2^-22, below
// the TF32 rounding of the operands it feeds).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// max(a, b, c), NaN if any is NaN (one three-input instruction on sm_100+).
__device__ __forceinline__ float maxnan3(float a, float b, float c) {
    float d;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ void mma_m16n8k8(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9},"
        " {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// fp32 element (r, c) of a 32 x 32 K-major operand tile (one box, 128-byte rows)
__device__ __forceinline__ uint32_t off_sq(int r, int c) {
    return (uint32_t)(r * 128 + ((((c >> 2) ^ r) & 7) << 4) + (c & 3) * 4);
}

// ---------------------------------------------------------------------------
// 32 x 32 unit-lower-triangular inverse T = (I + A)^-1 by two warps (I = 0, 1), and
// T Diag(beta) into the B tile of U (its upper-right block stays zero from
// the unit's set-up).  A is the strictly lower part of fp32 [32][AS] (rows
// scaled by beta; nothing on or above the diagonal is read).  Warp I inverts
// the 16 x 16 diagonal block I in two levels: lanes 0-15 invert its two 8 x 8
// diagonal blocks by column-oriented forward substitution (lane = column),
// then the whole warp forms the lower-left 8 x 8 block as
//     T_(1,0) = -T_(1,1) (A_(1,0) T_(0,0))
// (two columns a lane, through an 8 x 8 scratch in qs).  Warp I = 0 then forms
// R = A_10 T_00 of the 16 x 16 blocks, and after a two-warp barrier each warp
// forms one half of
//     T_10 = -T_11 R
// (warp-level m16n8k8 TF32 MMAs).  The upper-right 8 x 8 of each diagonal
// block of T stays zero from the unit's set-up.  Returns this warp's largest
// |T Diag(beta)| (NaN if any entry is NaN) in every lane.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float solve32(uint8_t *sm, uint8_t *tb, const float *beta, float *qs, int I, int lane) {
    const float *As = reinterpret_cast<const float *>(sm + SCR_A);
    float *Ts = reinterpret_cast<float *>(sm + SCR_T);
    float *Rs = reinterpret_cast<float *>(sm + SCR_R);
    float tmax = 0.f;
    if (lane < 16) {
        const int b = lane >> 3, c = lane & 7, r0 = 16 * I + 8 * b;
        const float *Ab = As + r0 * AS + r0;
        float4 lo[8], hi[8];
#pragma unroll
        for (int r = 1; r < 8; ++r) {
            lo[r] = *reinterpret_cast<const float4 *>(Ab + r * AS);
            if (r > 4) hi[r] = *reinterpret_cast<const float4 *>(Ab + r * AS + 4);
        }
        float x[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < 7; ++j) {
#pragma unroll
            for (int r = j + 1; r < 8; ++r) {
                const float4 &q4 = j < 4 ? lo[r] : hi[r];
                const float e = (j & 3) == 0 ? q4.x : (j & 3) == 1 ? q4.y : (j & 3) == 2 ? q4.z : q4.w;
                x[r] = fmaf(-e, x[j], x[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) Ts[(r0 + r) * TS + 8 * b + c] = x[r];
    }
    __syncwarp();
    {
        // the lower-left 8 x 8 block of diagonal block I: lane = (row rl, columns c0, c0 + 1)
        const int rl = lane >> 2, c0 = 2 * (lane & 3);
        const float4 a0 = *reinterpret_cast<const float4 *>(As + (16 * I + 8 + rl) * AS + 16 * I);
        const float4 a1 = *reinterpret_cast<const float4 *>(As + (16 * I + 8 + rl) * AS + 16 * I + 4);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        float2 rv = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float2 t = *reinterpret_cast<const float2 *>(Ts + (16 * I + j) * TS + c0);
            rv.x = fmaf(av[j], t.x, rv.x);
            rv.y = fmaf(av[j], t.y, rv.y);
        }
        *reinterpret_cast<float2 *>(qs + rl * 8 + c0) = rv;
        __syncwarp();
        const float4 u0 = *reinterpret_cast<const float4 *>(Ts + (16 * I + 8 + rl) * TS + 8);
        const float4 u1 = *reinterpret_cast<const float4 *>(Ts + (16 * I + 8 + rl) * TS + 12);
        const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        float2 tv = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float2 r2 = *reinterpret_cast<const float2 *>(qs + j * 8 + c0);
            tv.x = fmaf(-uv[j], r2.x, tv.x);
            tv.y = fmaf(-uv[j], r2.y, tv.y);
        }
        *reinterpret_cast<float2 *>(Ts + (16 * I + 8 + rl) * TS + c0) = tv;
    }
    __syncwarp();
    {
        // T Diag(b) of diagonal block I: lane = (row lane / 2, 8 columns)
        const int rr = 16 * I + (lane >> 1), h8 = 8 * (lane & 1), cc = 16 * I + h8;
        const float4 t0 = *reinterpret_cast<const float4 *>(Ts + rr * TS + h8);
        const float4 t1 = *reinterpret_cast<const float4 *>(Ts + rr * TS + h8 + 4);
        const float4 b0 = *reinterpret_cast<const float4 *>(beta + cc);
        const float4 b1 = *reinterpret_cast<const float4 *>(beta + cc + 4);
        const float4 v0 = make_float4(t0.x * b0.x, t0.y * b0.y, t0.z * b0.z, t0.w * b0.w);
        const float4 v1 = make_float4(t1.x * b1.x, t1.y * b1.y, t1.z * b1.z, t1.w * b1.w);
        tmax = maxnan3(maxnan3(fabsf(v0.x), fabsf(v0.y), fabsf(v0.z)), maxnan3(fabsf(v0.w), fabsf(v1.x), fabsf(v1.y)),
                       maxnan3(fabsf(v1.z), fabsf(v1.w), 0.f));
        *reinterpret_cast<float4 *>(tb + off_sq(rr, cc)) = v0;
        *reinterpret_cast<float4 *>(tb + off_sq(rr, cc + 4)) = v1;
    }
    const int g = lane >> 2, t4 = lane & 3;
    if (I == 0) {
        // R = A_10 T_00 (rows 16..31, columns 0..15 of A)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const float *ar = As + (16 + g) * AS + 8 * ks + t4;
                const uint32_t a[4] = {to_tf32(ar[0]), to_tf32(ar[8 * AS]), to_tf32(ar[4]), to_tf32(ar[8 * AS + 4])};
                const uint32_t b[2] = {to_tf32(Ts[(8 * ks + t4) * TS + 8 * nt + g]),
                                       to_tf32(Ts[(8 * ks + t4 + 4) * TS + 8 * nt + g])};
                mma_m16n8k8(d, a, b);
            }
            Rs[g * TS + 8 * nt + 2 * t4] = d[0];
            Rs[g * TS + 8 * nt + 2 * t4 + 1] = d[1];
            Rs[(g + 8) * TS + 8 * nt + 2 * t4] = d[2];
            Rs[(g + 8) * TS + 8 * nt + 2 * t4 + 1] = d[3];
        }
    }
    named_sync(3, 64);   // R (warp I = 0) and T_11 (warp I = 1) complete
    // T_10 = -T_11 R, columns 8 I .. 8 I + 7 by warp I; T Diag(b) of the block
    {
        const int nt = I;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const float *tr = Ts + (16 + g) * TS + 8 * ks + t4;
            const uint32_t a[4] = {to_tf32(tr[0]), to_tf32(tr[8 * TS]), to_tf32(tr[4]), to_tf32(tr[8 * TS + 4])};
            const uint32_t b[2] = {to_tf32(Rs[(8 * ks + t4) * TS + 8 * nt + g]),
                                   to_tf32(Rs[(8 * ks + t4 + 4) * TS + 8 * nt + g])};
            mma_m16n8k8(d, a, b);
        }
        const int c = 8 * nt + 2 * t4;
        const float b0 = beta[c], b1 = beta[c + 1];
        const float2 lo = make_float2(-d[0] * b0, -d[1] * b1);
        const float2 hi = make_float2(-d[2] * b0, -d[3] * b1);
        tmax = maxnan3(tmax, maxnan3(fabsf(lo.x), fabsf(lo.y), fabsf(hi.x)), fabsf(hi.y));
        *reinterpret_cast<float2 *>(tb + off_sq(16 + g, c)) = lo;
        *reinterpret_cast<float2 *>(tb + off_sq(24 + g, c)) = hi;
    }
    fence_proxy_async();   // T Diag(b) is read by the tensor cores
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tmax = maxnan3(tmax, __shfl_xor_sync(0xffffffffu, tmax, off), 0.f);
    return tmax;
}

// ---------------------------------------------------------------------------
// The recurrence over one chunk on the CUDA cores, in fp32, by the 128
// consumer threads on the transposed state in TMEM: thread v (TMEM lane v)
// owns column v of S (all 128 rows, moved through registers 32 at a time).
// Per token the inputs are staged (alpha = exp(gk), k, q, v, beta;
// double-buffered by token parity); each thread decays its column and forms
// (S'^T k)[v] and (S'^T q)[v], then applies u = beta (v - S'^T k),
// S += k u^T and o = scale (S'^T q + u (k . q)).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void chunk_recurrent(const Params &p, uint8_t *sm, uint32_t lane_base, int v, int t0,
                                                int L, int h) {
    const int lane = v & 31, wq = v >> 5;
    float *xs = reinterpret_cast<float *>(sm + FB_X);     // [2][4] k.q partials, [2] beta
#pragma unroll 1
    for (int tk = 0; tk < L; ++tk) {
        const int tg = t0 + tk, b = tk & 1;
        float *in = reinterpret_cast<float *>(sm + FB_IN + b * 2048);   // alpha, k, q, v
        const size_t row = ((size_t)tg * p.H + h) * KD;
        const float kk = __bfloat162float(p.k[row + v]), qq = __bfloat162float(p.q[row + v]);
        in[v] = expf(__bfloat162float(p.gk[row + v]));
        in[128 + v] = kk;
        in[256 + v] = qq;
        in[384 + v] = __bfloat162float(p.v[row + v]);
        float x = kk * qq;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        if (lane == 0) xs[b * 4 + wq] = x;
        if (v == 0) xs[8 + b] = __bfloat162float(p.beta[(size_t)tg * p.H + h]);
        named_sync(2, 128);
        float pk = 0.f, pq = 0.f;
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
            uint32_t r[32];
            KDA_TMEM_LD32(lane_base + TM_X + 32 * g, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float sd = __uint_as_float(r[e]) * in[32 * g + e];
                pk = fmaf(sd, in[128 + 32 * g + e], pk);
                pq = fmaf(sd, in[256 + 32 * g + e], pq);
                r[e] = __float_as_uint(sd);
            }
            KDA_TMEM_ST32(lane_base + TM_X + 32 * g, r);
        }
        const float kqd = (xs[b * 4] + xs[b * 4 + 1]) + (xs[b * 4 + 2] + xs[b * 4 + 3]);
        const float u = xs[8 + b] * (in[384 + v] - pk);
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
            uint32_t r[32];
            KDA_TMEM_LD32(lane_base + TM_X + 32 * g, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(fmaf(in[128 + 32 * g + e], u, __uint_as_float(r[e])));
            KDA_TMEM_ST32(lane_base + TM_X + 32 * g, r);
        }
        p.o[((size_t)tg * p.H + h) * VD + v] = __float2bfloat16_rn(p.scale * (pq + u * kqd));
    }
}

// The state S[k][v] = X^T[v][k] from TMEM to a pool slot: consumer thread v
// stores column v (all 128 rows; coalesced over v).
__device__ __forceinline__ void store_state(float *dst, uint32_t lane_base, int v) {
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
        uint32_t r[32];
        KDA_TMEM_LD32(lane_base + TM_X + 32 * g, r);
#pragma unroll
        for (int e = 0; e < 32; ++e) __stcs(dst + (size_t)(32 * g + e) * VD + v, __uint_as_float(r[e]));
    }
}

// V' = V - K~ S for 16 tokens of this thread's value column, in place in TMEM
// (columns taddr .. taddr + 15); vrow is the column's bytes in token row 0 of
// the raw v tile (rows 128 B apart, 16-byte chunk index XOR the row).  With
// MASK, tokens from lh on are past the sequence and give 0.  vm collects the
// largest |V'| (NaN if any is NaN).
template <bool MASK>
__device__ __forceinline__ void vprime_half(const uint8_t *vrow, int cv, uint32_t taddr, int lh, float &vm) {
    uint32_t r[16];
    KDA_TMEM_LD16(taddr, r);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        float vp[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const uint16_t bits = *reinterpret_cast<const uint16_t *>(vrow + (i + e) * 128 + (((cv ^ (i + e)) & 7) << 4));
            vp[e] = __uint_as_float((uint32_t)bits << 16) - __uint_as_float(r[i + e]);
            if (MASK && i + e >= lh) vp[e] = 0.f;
            r[i + e] = __float_as_uint(vp[e]);
        }
        vm = maxnan3(vm, fabsf(vp[0]), fabsf(vp[1]));
    }
    KDA_TMEM_ST16(taddr, r);
}

// ---------------------------------------------------------------------------
// the kernel
//
// Producer warps 0-3, per chunk j: wait for the raw tiles; prep (cumulative
// decays, exponentials, [Q~; K~], Kb, exp(G_L)); signal "tiles"; G1 (thread 0)
// beside Kb^T (warps 1-3, once the consumer is done with chunk j - 1); A read
// out and T Diag(b) (warps 2-3) beside Aqk read out (warps 0-1); signal "solve".
// Consumer warps 4-7, per chunk j: wait for "tiles"; P; once P and G1 have
// read [Q~; K~], request the next raw tiles; V'; wait for "solve"; U, then the
// state update with O; O out and the state scaled by exp(G_L); signal "done".
// The producer thus prepares chunk j + 1 while the consumer runs chunk j.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(NT, 2) prefill_tc_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lq = warp & 3;         // TMEM lane quarter this warp may access
    float *beta_s = reinterpret_cast<float *>(sm + SM_BETA);
    float *elr = reinterpret_cast<float *>(sm + SM_ELR);
    float *tot = reinterpret_cast<float *>(sm + SM_TOT);
    float *As = reinterpret_cast<float *>(sm + SCR_A);
    int *fbf = reinterpret_cast<int *>(sm + SM_FLAG);                 // [2] recurrent-path verdict by chunk parity
    float *tbmax = reinterpret_cast<float *>(sm + SM_FLAG + 8);       // [2][2] max |T Diag(b)| by parity, warp
    float *vmaxs = reinterpret_cast<float *>(sm + SM_FLAG + 24);      // [4] max |V'| by consumer warp
    const uint32_t bar_raw = sbase + SM_BAR, bar_v = bar_raw + 8, bar_g1 = bar_raw + 16, bar_p = bar_raw + 24,
                   bar_u = bar_raw + 32, bar_ou = bar_raw + 40, bar_tiles = bar_raw + 48,
                   bar_tb = bar_raw + 56, bar_done = bar_raw + 64;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + SM_MISC);
    int tmo = 0;   // this thread gave up on a wait

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
    // the entering state (64 KB) into L2 now: the consumer reads it into TMEM
    // after the set-up, in four dependent rounds
    if (si >= 0 && tid >= 128 && tid < 132)
        prefetch_l2(p.pool + ((size_t)si * p.H + h) * STATE_ELEMS + (tid - 128) * (STATE_ELEMS / 4), STATE_ELEMS);

    // ---- set-up -----------------------------------------------------------
    auto load_qkg = [&](int tok) {
        mbar_expect_tx(bar_raw, 3 * 8192);
        for (int b = 0; b < 2; ++b) {
            tma_load_3d(sbase + RAW_Q + b * 4096, &p.tq, bar_raw, 64 * b, h, tok);
            tma_load_3d(sbase + RAW_K + b * 4096, &p.tk, bar_raw, 64 * b, h, tok);
            tma_load_3d(sbase + RAW_G + b * 4096, &p.tg, bar_raw, 64 * b, h, tok);
        }
    };
    auto load_v = [&](int tok) {
        mbar_expect_tx(bar_v, 8192);
        for (int b = 0; b < 2; ++b) tma_load_3d(sbase + RAW_V + b * 4096, &p.tv, bar_v, 64 * b, h, tok);
    };
    if (tid == 0) {
        for (int b = 0; b < 6; ++b) mbar_init(bar_raw + 8 * b, 1);
        for (int b = 6; b < 9; ++b) mbar_init(bar_raw + 8 * b, 4);   // one arrival per warp of a group
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (nchunks > 0 && !p.skip_first_load) load_qkg(bos);
        if (nchunks > 0) load_v(bos);
    }
    // the upper-right blocks (rows 0..15, columns 16..31) of both T Diag(b)
    // tiles and the zero row stay zero: thread t clears rows (t / 16) % 8 and
    // that + 8, column 16 + t % 16, of tile t / 128
    {
        uint8_t *tbz = sm + OP_TB + (tid >> 7) * 4096;
        const int r0 = (tid >> 4) & 7, col = 16 + (tid & 15);
        *reinterpret_cast<float *>(tbz + off_sq(r0, col)) = 0.f;
        *reinterpret_cast<float *>(tbz + off_sq(r0 + 8, col)) = 0.f;
    }
    if (tid < 4) reinterpret_cast<uint32_t *>(sm + SM_ZERO)[tid] = 0u;
    // the upper-right 8 x 8 of each diagonal 16 x 16 block of T stays zero
    if (tid < 128) reinterpret_cast<float *>(sm + SCR_T)[(16 * (tid >> 6) + ((tid >> 3) & 7)) * TS + 8 + (tid & 7)] = 0.f;
    fence_proxy_async();
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
    const uint32_t lane_base = tmem + ((uint32_t)(32 * lq) << 16);
    const uint64_t wait_ns = p.wait_ns ? p.wait_ns : WAIT_NS;
    // one arrival for the warp, after every lane's earlier accesses (the warp
    // barrier orders them before lane 0's release)
    // one lane of the warp waits; the warp barrier then orders the other
    // lanes' accesses after that wait
    auto warp_wait = [&](uint32_t bar, uint32_t parity) -> bool {
        int ok = 1;
        if (lane == 0) ok = barrier_wait_for(bar, parity, wait_ns);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        return ok != 0;
    };
    auto warp_arrive = [&](uint32_t bar) {
        __syncwarp();
        if (lane == 0) barrier_arrive(bar);
    };
    const float LOG2E = 1.4426950408889634f;
    constexpr uint32_t ID_G1 = idesc_tf32(64, 32);
    constexpr uint32_t ID_P = idesc_tf32(128, 64);
    constexpr uint32_t ID_N32 = idesc_tf32(128, 32);
    constexpr uint32_t ID_XO = idesc_tf32(128, 160);
    bool aborted = false;

    if (warp < 4) {
        // =================== producer: warps 0-3 ===================
        // beta of the chunk about to be prepared, loaded one chunk ahead as raw
        // bf16 bits; a token past the sequence loads its sequence's first beta
        // and stores 0.
        const unsigned short *beta_bits = reinterpret_cast<const unsigned short *>(p.beta);
        unsigned short beta_raw = 0;
        bool beta_ok = false;
        if (tid < C && nchunks > 0) {
            beta_ok = tid < eos - bos;
            beta_raw = __ldg(beta_bits + (size_t)(beta_ok ? bos + tid : bos) * p.H + h);
        }
        // prep mapping: warp = row octet o (rows 8 o + 4 rg + i, i < 4), lane =
        // (row group rg, channel group cg): channels 4 cg + 64 hf + j (j < 4, hf < 2)
        const int o8 = warp, rg = lane >> 4, cg = lane & 15;
        uint32_t n_g = 0;   // chunks whose G1 was issued
        for (int cc = 0; cc < nchunks; ++cc) {
            const int t0 = bos + cc * C;
            const int L = min(C, eos - t0);
            const int pc = cc & 1;
            if (tid < C) {
                beta_s[tid] = beta_ok ? __uint_as_float((uint32_t)beta_raw << 16) : 0.f;
                const int tn = t0 + C + tid;
                beta_ok = cc + 1 < nchunks && tn < eos;
                beta_raw = __ldg(beta_bits + (size_t)(beta_ok ? tn : bos) * p.H + h);
            }
            // (1) the raw tiles: one lane of each warp waits; the warp barrier
            //     then orders the other lanes' reads after that wait
            {
                int ok = 1;
                if (lane == 0) ok = barrier_wait_for(bar_raw, (uint32_t)pc, wait_ns);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                __syncwarp();
                if (!ok) tmo = 1;
            }
            // (2) prep.  q, k stay packed (bf16 pairs); a row past the sequence
            //     reads the zero row.  Every raw value is read before the barrier
            //     after which the operand tiles are written over them.
            float gv[2][4][4];
            float glo[2][4];   // the octet's row-group-0 sums, folded into the offsets by row group 1
            uint2 wq[2][4], wk[2][4];
            // checks on the raw bf16 bits, two at a time: the largest |k| as an
            // unsigned magnitude (a NaN is above every finite value), the largest
            // gk as a signed 16-bit integer (> 0 only for a positive gk or a NaN
            // with the sign clear; other NaNs reach the decay check through G)
            unsigned kbits = 0u;
            int gbits = (int)0x80008000u;
            // rows past the sequence (a partial chunk only) read the zero row
            auto load_rows = [&](int hf, bool full) {
                const int k0 = 4 * cg + 64 * hf;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 8 * o8 + 4 * rg + i;
                    const uint32_t ro = raw_off(r, k0, C);
                    const bool valid = full || r < L;
                    wq[hf][i] = *reinterpret_cast<const uint2 *>(sm + (valid ? RAW_Q + ro : SM_ZERO));
                    wk[hf][i] = *reinterpret_cast<const uint2 *>(sm + (valid ? RAW_K + ro : SM_ZERO));
                    const uint2 wg = *reinterpret_cast<const uint2 *>(sm + (valid ? RAW_G + ro : SM_ZERO));
                    gv[hf][i][0] = bf16_lo(wg.x); gv[hf][i][1] = bf16_hi(wg.x);
                    gv[hf][i][2] = bf16_lo(wg.y); gv[hf][i][3] = bf16_hi(wg.y);
                    gbits = __vmaxs2(gbits, __vmaxs2((int)wg.x, (int)wg.y));
                    kbits = __vmaxu2(kbits, __vmaxu2(wk[hf][i].x & 0x7FFF7FFFu, wk[hf][i].y & 0x7FFF7FFFu));
                }
            };
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int k0 = 4 * cg + 64 * hf;
                if (L == C) load_rows(hf, true);
                else load_rows(hf, false);
                // inclusive prefix over the thread's 4 rows; row group 1 of the
                // octet (lanes 16-31) adds row group 0's sums (lanes l ^ 16)
                // through its offsets
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int i = 1; i < 4; ++i) gv[hf][i][j] += gv[hf][i - 1][j];
                    const float lo = __shfl_xor_sync(0xffffffffu, gv[hf][3][j], 16);
                    glo[hf][j] = rg ? lo : 0.f;
                }
                if (rg)
                    *reinterpret_cast<float4 *>(tot + o8 * 128 + k0) =
                        make_float4(gv[hf][3][0] + glo[hf][0], gv[hf][3][1] + glo[hf][1], gv[hf][3][2] + glo[hf][2],
                                    gv[hf][3][3] + glo[hf][3]);
            }
            named_sync(1, 128);   // octet sums visible; every raw tile read
            float dmax = 0.f;   // largest decay over the chunk, log2 units (G is non-increasing)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int k0 = 4 * cg + 64 * hf;
                const float4 T0 = *reinterpret_cast<const float4 *>(tot + k0);
                const float4 T1 = *reinterpret_cast<const float4 *>(tot + 128 + k0);
                const float4 T2 = *reinterpret_cast<const float4 *>(tot + 256 + k0);
                const float4 T3 = *reinterpret_cast<const float4 *>(tot + 384 + k0);
                const float t0a[4] = {T0.x, T0.y, T0.z, T0.w}, t1a[4] = {T1.x, T1.y, T1.z, T1.w};
                const float t2a[4] = {T2.x, T2.y, T2.z, T2.w}, t3a[4] = {T3.x, T3.y, T3.z, T3.w};
                float cj[4];   // G_r log2(e) = G'_r log2(e) + cj, G'_r the thread-local prefix
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float g01 = t0a[j] + t1a[j], g012 = g01 + t2a[j];
                    const float pre = o8 == 0 ? 0.f : (o8 == 1 ? t0a[j] : (o8 == 2 ? g01 : g012));
                    cj[j] = (pre + glo[hf][j]) * LOG2E;
                    const float gl2 = (g012 + t3a[j]) * LOG2E;   // G_L log2(e)
                    dmax = maxnan3(dmax, -gl2, 0.f);
                    if (o8 == 0 && rg == 0) elr[pc * 128 + k0 + j] = ex2(gl2);   // exp(G_L)
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 8 * o8 + 4 * rg + i;
                    float2 ef[2], eb[2];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float d = fmaf(gv[hf][i][j], LOG2E, cj[j]);   // G_r log2(e)
                        (j & 1 ? ef[j >> 1].y : ef[j >> 1].x) = ex2(d);
                        (j & 1 ? eb[j >> 1].y : eb[j >> 1].x) = ex2(-d);
                    }
                    const float2 q01 = make_float2(bf16_lo(wq[hf][i].x), bf16_hi(wq[hf][i].x));
                    const float2 q23 = make_float2(bf16_lo(wq[hf][i].y), bf16_hi(wq[hf][i].y));
                    const float2 k01 = make_float2(bf16_lo(wk[hf][i].x), bf16_hi(wk[hf][i].x));
                    const float2 k23 = make_float2(bf16_lo(wk[hf][i].y), bf16_hi(wk[hf][i].y));
                    const float2 kt01 = __fmul2_rn(k01, ef[0]), kt23 = __fmul2_rn(k23, ef[1]);
                    const float2 qt01 = __fmul2_rn(q01, ef[0]), qt23 = __fmul2_rn(q23, ef[1]);
                    const float2 kb01 = __fmul2_rn(k01, eb[0]), kb23 = __fmul2_rn(k23, eb[1]);
                    *reinterpret_cast<float4 *>(sm + OP_QR + off32(32 + r, k0, 64)) = make_float4(kt01.x, kt01.y, kt23.x, kt23.y);
                    *reinterpret_cast<float4 *>(sm + OP_QR + off32(r, k0, 64)) =
                        make_float4(qt01.x, qt01.y, qt23.x, qt23.y);
                    *reinterpret_cast<float4 *>(sm + OP_KB + off32(r, k0, 32)) = tf32r4(kb01.x, kb01.y, kb23.x, kb23.y);
                }
            }
            fence_proxy_async();   // the tiles are read by the tensor cores
            const int gtop = max((int)(short)(gbits & 0xFFFF), (int)(short)((unsigned)gbits >> 16));
            const unsigned ktop = max(kbits & 0xFFFFu, kbits >> 16);
            const int bad = !(dmax <= D_LIMIT * LOG2E) || gtop > 0 || ktop > K_LIMIT_BITS;
            if (named_or(1, 128, tmo)) { aborted = true; break; }
            const int fb1 = named_or(1, 128, bad);
            if (tid == 0) fbf[pc] = fb1;
            warp_arrive(bar_tiles);   // (3) chunk cc's tiles (and its verdict) for the consumer
            // (4) G1 = [Q~; K~] Kb^T (M = 64) by thread 0, while warps 1-3 rebuild
            //     Kb^T from Kb once the consumer has finished chunk cc - 1 (its
            //     update read the previous Kb^T)
            if (warp == 0) {
                if (!fb1 && lane == 0) {
                    tc_fence_after();
                    const uint64_t da = sdesc(sbase + OP_QR, 16, 1024), db = sdesc(sbase + OP_KB, 16, 1024);
#pragma unroll
                    for (int s = 0; s < 16; ++s)
                        mma_ss(tmem + TM_G, da + (uint64_t)(((s >> 2) * 8192 + (s & 3) * 32) >> 4),
                               db + (uint64_t)(((s >> 2) * 4096 + (s & 3) * 32) >> 4), ID_G1, s > 0);
                    mma_commit(bar_g1);
                    if (!barrier_wait_for(bar_g1, n_g & 1u, wait_ns)) tmo = 1;
                }
            } else {
                if (cc > 0 && !warp_wait(bar_done, (uint32_t)((cc - 1) & 1))) tmo = 1;
                // 4 x 4 blocks (tokens 4 l8.., channels 4 kq..), eight lanes of a
                // phase on one diagonal: the loads and the stores each meet
                // eight different 16-byte bank groups
                for (int bk = tid - 32; bk < 256; bk += 96) {
                    const int l8 = bk & 7, kq = ((bk >> 3) + l8) & 31;
                    float4 kr[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        kr[i] = *reinterpret_cast<const float4 *>(sm + OP_KB + off32(4 * l8 + i, 4 * kq, 32));
                    uint8_t *dst = sm + OP_KBT + 4 * kq * 128;
                    const int sw = 4 * (kq & 1);
                    *reinterpret_cast<float4 *>(dst + 0 * 128 + ((l8 ^ (sw + 0)) << 4)) = make_float4(kr[0].x, kr[1].x, kr[2].x, kr[3].x);
                    *reinterpret_cast<float4 *>(dst + 1 * 128 + ((l8 ^ (sw + 1)) << 4)) = make_float4(kr[0].y, kr[1].y, kr[2].y, kr[3].y);
                    *reinterpret_cast<float4 *>(dst + 2 * 128 + ((l8 ^ (sw + 2)) << 4)) = make_float4(kr[0].z, kr[1].z, kr[2].z, kr[3].z);
                    *reinterpret_cast<float4 *>(dst + 3 * 128 + ((l8 ^ (sw + 3)) << 4)) = make_float4(kr[0].w, kr[1].w, kr[2].w, kr[3].w);
                }
                fence_proxy_async();   // Kb^T is read by the tensor cores
            }
            named_sync(1, 128);   // G1 done; Kb^T rebuilt
            if (!fb1) {
                // (5) A, Aqk read out; T Diag(b)
                ++n_g;
                tc_fence_after();
                uint32_t r[32];
                KDA_TMEM_LD32(lane_base + TM_G, r);   // M = 64: row r in lane 32 (r / 16) + r % 16
                if (lane < 16) {
                    const int row = 16 * (lq & 1) + lane;
                    if (lq >= 2) {
                        // the whole row, scaled by beta: the inverse reads only
                        // the strictly lower part
                        const float b = beta_s[row];
                        float4 *dst = reinterpret_cast<float4 *>(As + row * AS);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float2 lo = __fmul2_rn(make_float2(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1])),
                                                         make_float2(b, b));
                            const float2 hi = __fmul2_rn(make_float2(__uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])),
                                                         make_float2(b, b));
                            dst[j] = make_float4(lo.x, lo.y, hi.x, hi.y);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float a4[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) a4[e] = (4 * j + e <= row) ? __uint_as_float(r[4 * j + e]) : 0.f;
                            *reinterpret_cast<float4 *>(sm + OP_AQ + off_sq(row, 4 * j)) =
                                tf32r4(a4[0], a4[1], a4[2], a4[3]);
                        }
                    }
                }
                fence_proxy_async();   // Aqk is read by the tensor cores
                tc_fence_before();
                // warps 2-3 read A out of TMEM and invert I + A at once; warps 0-1
                // read Aqk out beside them
                if (warp >= 2) {
                    named_sync(3, 64);   // A complete
                    const float tmx = solve32(sm, sm + OP_TB + pc * 4096, beta_s, tot + 64 * (warp - 2), warp - 2, lane);   // tot: free here
                    if (lane == 0) tbmax[pc * 2 + warp - 2] = tmx;
                }
            }
            fence_proxy_async();
            tc_fence_before();
            warp_arrive(bar_tb);   // (6) T Diag(b), Aqk, Kb^T of chunk cc for the consumer
            if (named_or(1, 128, tmo)) { aborted = true; break; }
        }
    } else {
        // =================== consumer: warps 4-7 ===================
        const int v = tid - 128;          // this thread's TMEM lane = value channel
        const bool leader = v == 0;
        // the initial state (column v, all rows) into TMEM through registers
        {
            const float *s0 = si >= 0 ? p.pool + ((size_t)si * p.H + h) * STATE_ELEMS + v : nullptr;
#pragma unroll 1
            for (int g = 0; g < 4; ++g) {
                uint32_t st0[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) st0[e] = s0 ? __float_as_uint(__ldcs(s0 + (size_t)(32 * g + e) * VD)) : 0u;
                KDA_TMEM_ST32(lane_base + TM_X + 32 * g, st0);
            }
        }
        uint32_t n_p = 0, n_u = 0;   // chunks whose P / U were issued
        // O of the previous tensor-core chunk, held in registers (bf16 pairs,
        // rows 2i and 2i + 1 of column v) so that it leaves while the next
        // chunk's P runs: a full chunk through the staging tile and two tensor
        // stores, a partial one by direct stores
        uint32_t opk[16];
        bool o_pend = false;
        int o_t0 = 0, o_L = 0;
        auto flush_o = [&]() {
            if (!o_pend) return;
            o_pend = false;
            if (o_L == C) {
                if (leader) bulk_wait_read();   // the previous tensor store has read the staging tile
                named_sync(2, 128);
                const uint32_t ob = OP_OST + (v >> 6) * (C * 128) + (v & 7) * 2;
                const int cv = (v >> 3) & 7;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const uint16_t bits = (uint16_t)(i & 1 ? opk[i >> 1] >> 16 : opk[i >> 1] & 0xFFFFu);
                    *reinterpret_cast<uint16_t *>(sm + ob + i * 128 + (((cv ^ i) & 7) << 4)) = bits;
                }
                fence_proxy_async();
                named_sync(2, 128);
                if (leader) {
                    tma_store_3d(&p.to, sbase + OP_OST, 0, h, o_t0);
                    tma_store_3d(&p.to, sbase + OP_OST + C * 128, 64, h, o_t0);
                    bulk_commit();
                }
            } else {
                unsigned short *dst = reinterpret_cast<unsigned short *>(p.o) + ((size_t)o_t0 * p.H + h) * VD + v;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < o_L) dst[(size_t)i * p.H * VD] = (unsigned short)(i & 1 ? opk[i >> 1] >> 16 : opk[i >> 1] & 0xFFFFu);
            }
        };
        for (int c = 0; c < nchunks; ++c) {
            const int t0 = bos + c * C;
            const int L = min(C, eos - t0);
            const uint32_t par = (uint32_t)(c & 1);
            // (1) chunk c's tiles and the producer's verdict
            if (leader && !barrier_wait_for(bar_tiles, par, wait_ns)) tmo = 1;
            if (named_or(2, 128, tmo)) { aborted = true; break; }
            const int fb1 = fbf[par];
            bool tc_path = false;
            if (!fb1) {
                const uint32_t ppar = n_p & 1u;
                ++n_p;
                // (2) P^T = S^T [Q~; K~]^T (A from TMEM); once P and G1 have read
                //     [Q~; K~], the next raw tiles are requested over it
                if (leader) {
                    tc_fence_after();
                    const uint64_t da = sdesc(sbase + OP_QR, 16, 1024);
#pragma unroll
                    for (int s = 0; s < 16; ++s)
                        mma_ts(tmem + TM_P, tmem + TM_X + 8 * s, da + (uint64_t)(((s >> 2) * 8192 + (s & 3) * 32) >> 4),
                               ID_P, s > 0);
                    mma_commit(bar_p);
                }
                flush_o();   // the previous chunk's O, while P runs
                if (leader) {
                    if (!barrier_wait_for(bar_p, ppar, wait_ns) || !barrier_wait_for(bar_g1, ppar, wait_ns) ||
                        !barrier_wait_for(bar_v, par, wait_ns))
                        tmo = 1;
                    else if (c + 1 < nchunks)
                        load_qkg(t0 + C);
                }
                named_sync(2, 128);
                tc_fence_after();
                // (3) V' = V - K~ S in place of K~ S (columns 128..159), one token per column
                {
                    const uint32_t vb = RAW_V + (v >> 6) * (C * 128) + (v & 7) * 2;
                    const int cv = (v >> 3) & 7;
                    float vm = 0.f;
                    // rows past the sequence (a partial chunk only) are zero
                    if (L == C) {
#pragma unroll 1
                        for (int hf = 0; hf < 2; ++hf) vprime_half<false>(sm + vb + 16 * hf * 128, cv, lane_base + TM_V + 16 * hf, 16, vm);
                    } else {
#pragma unroll 1
                        for (int hf = 0; hf < 2; ++hf) vprime_half<true>(sm + vb + 16 * hf * 128, cv, lane_base + TM_V + 16 * hf, L - 16 * hf, vm);
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) vm = maxnan3(vm, __shfl_xor_sync(0xffffffffu, vm, off), 0.f);
                    if (lane == 0) vmaxs[lq] = vm;
                }
                fence_proxy_async();   // the raw v reads precede the next v's TMA
                tc_fence_before();
                // (4) T Diag(b), Aqk, Kb^T of chunk c
                if (leader && !barrier_wait_for(bar_tb, par, wait_ns)) tmo = 1;
                if (named_or(2, 128, tmo)) { aborted = true; break; }
                const float vmx = maxnan3(maxnan3(vmaxs[0], vmaxs[1], vmaxs[2]), vmaxs[3], 0.f);
                tc_path = maxnan3(tbmax[2 * par], tbmax[2 * par + 1], 0.f) * vmx <= U_LIMIT;   // false on a NaN
                if (tc_path) {
                    const uint32_t upar = n_u & 1u;
                    ++n_u;
                    // (5) U^T = V'^T (T Diag(b))^T; then O^T += U^T Aqk^T and X^T += U^T Kb
                    if (leader) {
                        tc_fence_after();
                        const uint64_t dtb = sdesc(sbase + OP_TB + par * 4096, 16, 1024);
#pragma unroll
                        for (int s = 0; s < 4; ++s)
                            mma_ts(tmem + TM_U, tmem + TM_V + 8 * s, dtb + (uint64_t)(2 * s), ID_N32, s > 0);
                        mma_commit(bar_u);
                        if (c + 1 < nchunks) load_v(t0 + C);
                        const uint64_t dkt = sdesc(sbase + OP_KBT, 16, 1024);   // [Kb^T; Aqk]: 160 rows
                        if (barrier_wait_for(bar_u, upar, wait_ns)) {
                            tc_fence_after();
#pragma unroll
                            for (int s = 0; s < 4; ++s)   // [X^T | O^T] += U^T [Kb^T; Aqk]^T
                                mma_ts(tmem + TM_X, tmem + TM_U + 8 * s, dkt + (uint64_t)(2 * s), ID_XO, 1);
                            mma_commit(bar_ou);
                            if (!barrier_wait_for(bar_ou, upar, wait_ns)) tmo = 1;
                        } else {
                            tmo = 1;
                        }
                    }
                    if (named_or(2, 128, tmo)) { aborted = true; break; }
                    tc_fence_after();
                }
            } else if (leader && !barrier_wait_for(bar_tb, par, wait_ns)) {   // keep the phases in step
                tmo = 1;
            }
            // the checkpoint slot this chunk closes, if any
            const int m = (c + 1) / max(p.ckpt_chunks, 1) - 1;
            float *ckd = nullptr;
            if (nck > 0 && (c + 1) % p.ckpt_chunks == 0 && m < nck) {
                const int cs = p.ckpt_slots[(size_t)n * p.max_ckpts + m];
                if (cs >= 0) ckd = p.pool + ((size_t)cs * p.H + h) * STATE_ELEMS;
            }
            if (tc_path) {
                // (6) O of the chunk into registers (it leaves during the next
                //     chunk's P); then the next chunk's state S = Diag(exp(G_L)) X
                //     (and a checkpoint of it)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t r[16];
                    KDA_TMEM_LD16(lane_base + TM_O + 16 * hf, r);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float2 os = __fmul2_rn(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                                                     make_float2(p.scale, p.scale));
                        opk[8 * hf + i] = pack_bf16x2(os.x, os.y);
                    }
                }
                o_pend = true;
                o_t0 = t0;
                o_L = L;
                const float *f = elr + par * 128;
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    uint32_t r[32];
                    KDA_TMEM_LD32(lane_base + TM_X + 32 * g, r);
                    const float4 *f4 = reinterpret_cast<const float4 *>(f + 32 * g);
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 fv = f4[e4];
                        const float2 a = __fmul2_rn(make_float2(__uint_as_float(r[4 * e4]), __uint_as_float(r[4 * e4 + 1])),
                                                    make_float2(fv.x, fv.y));
                        const float2 b = __fmul2_rn(make_float2(__uint_as_float(r[4 * e4 + 2]), __uint_as_float(r[4 * e4 + 3])),
                                                    make_float2(fv.z, fv.w));
                        r[4 * e4] = __float_as_uint(a.x); r[4 * e4 + 1] = __float_as_uint(a.y);
                        r[4 * e4 + 2] = __float_as_uint(b.x); r[4 * e4 + 3] = __float_as_uint(b.y);
                    }
                    KDA_TMEM_ST32(lane_base + TM_X + 32 * g, r);
                    if (ckd) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) __stcs(ckd + (size_t)(32 * g + e) * VD + v, __uint_as_float(r[e]));
                    }
                }
            } else {
                // ---- the chunk by the recurrence, from the state in TMEM ----
                if (leader) {
                    if (fb1 && c + 1 < nchunks) load_qkg(t0 + C);   // [Q~; K~] is not read by an MMA
                    if (fb1 && !barrier_wait_for(bar_v, par, wait_ns)) tmo = 1;
                    if (c + 1 < nchunks) load_v(t0 + C);
                }
                if (named_or(2, 128, tmo)) { aborted = true; break; }
                flush_o();
                tc_fence_after();
                chunk_recurrent(p, sm, lane_base, v, t0, L, h);
                if (ckd) store_state(ckd, lane_base, v);
            }
            tc_fence_before();
            warp_arrive(bar_done);   // (7) chunk c is done: its tiles and parity buffers may be reused
        }
        if (!aborted) flush_o();
        if (leader) bulk_wait_all();   // every o tensor store is complete
        // the final state, unless a wait gave up
        if (!aborted) {
            tc_fence_after();
            store_state(p.pool + ((size_t)so * p.H + h) * STATE_ELEMS, lane_base, v);
            if (ss >= 0) store_state(p.pool + ((size_t)ss * p.H + h) * STATE_ELEMS, lane_base, v);
        }
    }
    if (__syncthreads_or(aborted || tmo)) {
        if (tid == 0) {
            report(p.err, DEVERR_TIMEOUT);
            // the self-test's unit gave up before its first v was consumed: let
            // that copy land (bounded) before the CTA's shared memory is released
            if (p.skip_first_load && nchunks > 0) barrier_wait_for(bar_v, 0, wait_ns);
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

// [T][H][128] bf16 viewed as a 3-D tensor {128, H, T}; boxes of 64 channels x
// 1 head x C tokens, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, int H, int T) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};
    cuuint32_t box[3] = {64, 1, C};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

cudaError_t launch_prefill_chunked(const PrefillArgs &a, cudaStream_t s) {
    using namespace tc;
    Params p;   // ~8.5 KB, copied into the launch parameters
    memset(&p, 0, sizeof(p));
    if (a.T_total > 0) {
        if (!make_map(&p.tq, a.q, a.H, a.T_total) || !make_map(&p.tk, a.k, a.H, a.T_total) ||
            !make_map(&p.tg, a.gk, a.H, a.T_total) || !make_map(&p.tv, a.v, a.H, a.T_total) ||
            !make_map(&p.to, a.o, a.H, a.T_total))
            return cudaErrorInvalidValue;
    }
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
    e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<<<(unsigned)(a.N * a.H), NT, SMEM_BYTES, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
