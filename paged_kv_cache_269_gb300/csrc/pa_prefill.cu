// pa_prefill.cu -- paged prefill on the tcgen05 tensor cores (sm_103a).
//
// What it computes: for each sequence s, the last q_len_s tokens of its
// context are queries; query i at position p = ctx_s - q_len_s + i attends,
// causally, to keys 0 .. p of that sequence, whose K/V sit in the paged cache
// ("vLLM 2026 推理引擎全解：从 PagedAttention 到分离式 Prefill", §1.3 -- prefill
// processes the prompt's tokens together and is compute-bound; §1.1 for the
// attention; §2.1-§2.2 for the block table).
//
// How: this is the one dense contraction of the paged cache, so it runs on
// the 5th-generation tensor cores with every accumulator in tensor memory.
//  * Persistent: one CTA per SM takes work items -- (pair of 128-query
//    tiles, sequence, head), heaviest first -- from an atomic counter.
//  * Warp 8 (TMA): publishes each item to the other roles through a
//    two-slot ring, loads its two Q tiles once and, per tile of 64 keys, the
//    four 16-token K and V blocks named by the block table as 2-D tensor-map
//    boxes (64 dims x 16 tokens) that land directly in the 128-byte-swizzled
//    operand layouts; three stages each for K and V.  Rows of an item's last
//    V tile past its last key are zeroed before use (a zero weight times a
//    NaN from an unused slot would still be NaN).
//  * Warps 9-12 issue the tensor-core products, one thread each, so four
//    instruction streams keep the tensor core busy (one thread's stream
//    alone is limited by the issue latency of each tcgen05.mma):
//      warps 9, 10: S_t = Q_t K^T (M 128, N 64, K 128) for query tile t, into
//        one of two tensor-memory S/P buffers, ahead of the softmax, once the
//        P V product that last read the buffer is complete;
//      warps 11, 12: once softmax t has published P_t, O_t += P_hi V +
//        P_lo V (M 128, N 128, K 64; P read from tensor memory, V as an
//        MN-major operand).
//  * Warps 0-3 / 4-7 (softmax of query tile 0 / 1): thread = query row (the
//    tensor-memory lane of an M = 128 accumulator).  It reads its 64 scores,
//    masks the causal boundary, and turns them into weights 2^(x - m + 6) in
//    fp32, where x is the score in the log2 domain and m a running maximum
//    that is only raised when a tile's maximum exceeds it by more than 8 (so
//    weights stay below 2^14, inside fp16's range); raising it rescales O_t
//    in tensor memory once the previous P V product is done.  The weights are
//    first taken against the running maximum; only when a row sum exceeds
//    2^14 (always on a query tile's first key tile) are the scores read again
//    and the tile's maximum found first.  The weights go
//    back into the same tensor-memory columns as a 16-bit pair P_hi + P_lo
//    (P_hi the weight rounded to the format, P_lo the rounded remainder),
//    which carries about 22 bits, so small outputs meet the same relative
//    bound as decode.  The row sum stays in fp32; the epilogue divides O_t
//    by it.
//  * Tensor-memory columns: S/P buffers of tile t at 128 t and 128 t + 64,
//    O_0 at 256, O_1 at 384 (the whole of the SM's tensor memory).
//  * Every wait is bounded; tensor memory is released on every path.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kD = 128;             // head_dim
constexpr int kBM = 128;            // query rows per tile (MMA M)
constexpr int kTiles = 2;           // query tiles per CTA
constexpr int kBN = 64;             // keys per tile
constexpr int kB = 16;              // block_size
constexpr int kBlocksPerTile = kBN / kB;
constexpr int kStages = 3;          // K and V ring depth
constexpr int kSBufs = 2;           // S/P buffers per query tile
constexpr int kThreads = 512;       // 2 x 4 softmax warps; TMA warp, 4 MMA-issuing warps, 3 idle
constexpr int kTmaWarp = 8;
constexpr int kSWarp0 = 9;          // issues query tile 0's S products; warp 10 tile 1's
constexpr int kPvWarp0 = 11;        // issues query tile 0's P V products; warp 12 tile 1's
// Register split: launched at 128 per thread (512 threads), the two
// producer warpgroups (warps 8-15) give registers up to the two softmax
// warpgroups; the four shares must fit the block's launch allotment of
// 4 x 128 per lane.  At 56 the producer roles compile without spills (at 48
// the TMA and MMA loops spilled a few words).
#ifndef PA_PREFILL_REGS_SOFTMAX
#define PA_PREFILL_REGS_SOFTMAX 200
#endif
#ifndef PA_PREFILL_REGS_OTHER
#define PA_PREFILL_REGS_OTHER 56
#endif
constexpr int kRegsSoftmax = PA_PREFILL_REGS_SOFTMAX;
constexpr int kRegsOther = PA_PREFILL_REGS_OTHER;
static_assert(2 * kRegsSoftmax + 2 * kRegsOther <= 4 * 128, "register split exceeds the launch");
static_assert(kRegsSoftmax % 8 == 0 && kRegsOther % 8 == 0 && kRegsOther >= 24, "bad split");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;      // S/P buffer b of tile t: columns 128 t + 64 b .. + 63
constexpr uint32_t kTmemO = 256;    // O_t: columns 256 + 128 t .. 256 + 128 t + 127
constexpr float kRescaleLog2 = 8.f; // raise the running maximum only past this margin
constexpr float kBiasLog2 = 6.f;    // weights are 2^(x - m + 6): at most 2^14

// shared memory layout (bytes; tiles 1024-aligned for the 128B swizzle)
constexpr int kHalfQ = kBM * 128;              // one 64-dim half of a Q tile
constexpr int kTileQ = 2 * kHalfQ;             // 32 KiB
constexpr int kHalfKV = kBN * 128;             // one 64-dim half of a K or V tile
constexpr int kTileKV = 2 * kHalfKV;           // 16 KiB
constexpr int OFF_Q = 0;                       // [tile][half][128 rows][128 B]
constexpr int OFF_K = OFF_Q + kTiles * kTileQ; // [stage][half][64 keys][128 B]
constexpr int OFF_V = OFF_K + kStages * kTileKV;
constexpr int OFF_BAR = OFF_V + kStages * kTileKV;
enum Bar {
    Q_FULL = 0,
    Q_EMPTY = 1,         // every S product of the item complete, one arrival per S thread
    K_FULL = 2,          // [stage]
    K_EMPTY = 5,         // [stage], one arrival per S thread
    V_FULL = 8,          // [stage]
    V_EMPTY = 11,        // [stage], one arrival per P V thread
    V_ZERO = 14,         // an item's last V tile loaded and its tail rows cleared
    ZERO_SEEN = 15,      // both P V threads have passed the item's V_ZERO
    S_FULL = 16,         // [tile][buffer]
    P_FULL = 20,         // [tile][buffer], one arrival per softmax warp
    PV_DONE = 24,        // [tile][buffer]: the P V product reading the buffer is complete
    O_FULL = 28,         // [tile]
    O_EMPTY = 30,        // [tile], the epilogue has read O_t (one arrival per softmax warp)
    MMA_DONE = 32,       // [issuing thread]
    ITEM_FULL = 36,      // [slot] of the work-item ring
    ITEM_EMPTY = 38,     // [slot]: the 4 MMA threads and the 8 softmax warps
    kNumBars = 40
};
// K_EMPTY and Q_EMPTY take one arrival from each S thread, V_EMPTY and
// ZERO_SEEN one from each P V thread; a thread arrives on an EMPTY barrier
// only after waiting for the matching FULL phase, so an arrival can never
// count toward an earlier phase.  The per-buffer barriers (S_FULL, P_FULL,
// PV_DONE) never run more than one phase ahead of their waiters, so a parity
// wait cannot alias.  V_ZERO could (a short item's V tiles can all be loaded
// while the P V threads still work on the previous item), so the TMA warp
// completes it for item k only after ZERO_SEEN shows both P V threads past it
// for item k - 1.
constexpr int OFF_TMEM = OFF_BAR + kNumBars * 8;
constexpr int OFF_FLAG = OFF_TMEM + 8;
constexpr int OFF_ITEM = OFF_FLAG + 8;              // int[2]
constexpr int kSmemBytes = OFF_ITEM + 8 + 1024;  // + alignment slack

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
    d |= static_cast<uint64_t>(1) << 46;   // descriptor version
    d |= static_cast<uint64_t>(2) << 61;   // 128-byte swizzle
    return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, A/B fp16 or bf16,
// A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), M = 128.
__host__ __device__ constexpr uint32_t instr_desc(bool bf16, bool b_mn, int n) {
    return (1u << 4) | (static_cast<uint32_t>(bf16) << 7) | (static_cast<uint32_t>(bf16) << 10) |
           (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(kBM >> 4) << 24);
}

// D (tensor memory) [+]= A (shared memory) * B (shared memory)
__device__ __forceinline__ void mma_ss(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                       bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1 : 0));
}

// D (tensor memory) [+]= A (tensor memory: row = lane, two 16-bit elements
// per 32-bit column, lower k in the low half) * B (shared memory)
__device__ __forceinline__ void mma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b,
                                       uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(b), "r"(idesc), "r"(accumulate ? 1 : 0));
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive 32-bit columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t addr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(addr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 / 32 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t addr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(addr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t addr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(addr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x by the hardware approximation (ex2.approx.ftz.f32: 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pair arithmetic (one instruction for two lanes of data).
__device__ __forceinline__ void fma2(float &d0, float &d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
    asm("{\n\t.reg .b64 a, b, c, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void sub2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "sub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// max of three
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *tm, int x, int y, int z,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// The weight pair (P_hi, P_lo) of two consecutive keys, packed as the MMA
// reads A from tensor memory (lower key in the low half).  P_hi = the weight
// rounded to the 16-bit format, P_lo = the remainder p - P_hi (exact in
// fp32) rounded to the format.  PA_PREFILL_SPLIT_RN=0 takes P_hi by cutting
// the fp32 mantissa instead (one more integer op per weight).
#ifndef PA_PREFILL_SPLIT_RN
#define PA_PREFILL_SPLIT_RN 1
#endif
struct F16T {
    static constexpr bool kBf16 = false;
    __device__ static __forceinline__ void split2(float p0, float p1, uint32_t &hi, uint32_t &lo) {
#if PA_PREFILL_SPLIT_RN
        // P_hi = p rounded to fp16, widened back exactly; P_lo = the rounded
        // remainder
        const __half2 h = __floats2half2_rn(p0, p1);
        const float2 hf = __half22float2(h);
        float l0, l1;
        sub2(l0, l1, p0, p1, hf.x, hf.y);
#else
        const float h0 = __uint_as_float(__float_as_uint(p0) & 0xFFFFE000u);
        const float h1 = __uint_as_float(__float_as_uint(p1) & 0xFFFFE000u);
        float l0, l1;
        sub2(l0, l1, p0, p1, h0, h1);
        const __half2 h = __floats2half2_rn(h0, h1);
#endif
        const __half2 l = __floats2half2_rn(l0, l1);
        hi = *reinterpret_cast<const uint32_t *>(&h);
        lo = *reinterpret_cast<const uint32_t *>(&l);
    }
    __device__ static __forceinline__ uint16_t round(float x) {
        const __half h = __float2half_rn(x);
        return *reinterpret_cast<const uint16_t *>(&h);
    }
};
struct BF16T {
    static constexpr bool kBf16 = true;
    __device__ static __forceinline__ void split2(float p0, float p1, uint32_t &hi, uint32_t &lo) {
#if PA_PREFILL_SPLIT_RN
        const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
        hi = *reinterpret_cast<const uint32_t *>(&h);
        float l0, l1;
        sub2(l0, l1, p0, p1, __uint_as_float(hi << 16), __uint_as_float(hi & 0xFFFF0000u));
#else
        const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
        hi = __byte_perm(b0, b1, 0x7632);   // upper halves: the truncated bf16 values
        float l0, l1;
        sub2(l0, l1, p0, p1, __uint_as_float(b0 & 0xFFFF0000u), __uint_as_float(b1 & 0xFFFF0000u));
#endif
        const __nv_bfloat162 l = __floats2bfloat162_rn(l0, l1);
        lo = *reinterpret_cast<const uint32_t *>(&l);
    }
    __device__ static __forceinline__ uint16_t round(float x) {
        const __nv_bfloat16 b = __float2bfloat16_rn(x);
        return *reinterpret_cast<const uint16_t *>(&b);
    }
};

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// One work item: a pair of query tiles of one (sequence, head).
struct Item {
    int s, h, row0, q_first, q_len, ctx, ntiles, kmax, nkt;
    int table_row;   // block-table row of the keys
};

// Work item w, heaviest pairs (latest positions) first: w = (level, s, h)
// with pair = num_pairs - 1 - level.  Returns false for an empty item (the
// sequence has no query rows in that pair) or, with `check`, for a sequence
// whose lengths are inconsistent (recorded in the error word).
// kShared: shared-prefix mode (a compile-time variant of the kernel, so the
// causal kernel carries none of its tests).
template <bool kShared>
__device__ __forceinline__ bool item_geometry(const PrefillArgs &a, int w, bool check, Item &it) {
    const int sh = a.num_seqs * a.num_heads;
    const int level = w / sh;
    const int rem = w - level * sh;
    it.s = rem / a.num_heads;
    it.h = rem - it.s * a.num_heads;
    const int pair = a.num_pairs - 1 - level;
    it.q_first = __ldg(a.query_start + it.s);
    const int q_end = __ldg(a.query_start + it.s + 1);
    // rows outside [0, total_q) (the difference taken without overflow)
    const bool rows_bad = it.q_first < 0 || q_end < it.q_first || q_end > a.total_q;
    it.q_len = rows_bad ? 0 : q_end - it.q_first;
    it.row0 = pair * kTiles * kBM;
    if constexpr (kShared) {
        // shared-prefix mode: s is a group of decode rows, all of which see
        // the whole prefix through the group's first row's table.  A
        // malformed group is skipped here; the plan kernel reports it and
        // leaves its rows to the decode kernel.
        const int pb = __ldg(a.group_prefix_blocks + it.s);
        if (rows_bad || it.q_len == 0 || it.row0 >= it.q_len || pb <= 0 ||
            pb > a.max_blocks_per_seq)
            return false;
        it.ctx = pb * kB;
        it.table_row = it.q_first;
        it.ntiles = it.q_len - it.row0 > kBM ? 2 : 1;
        it.kmax = it.ctx;
        it.nkt = (it.kmax + kBN - 1) / kBN;
        return true;
    }
    it.ctx = __ldg(a.context_lens + it.s);
    it.table_row = it.s;
    // query rows past num_pairs * 256 (max_query_len understated) would never be
    // computed: reported once per sequence
    if (check && it.h == 0 && it.row0 == 0 && it.q_len > a.num_pairs * kTiles * kBM)
        atomicOr(a.err, PA_DEVERR_CONTEXT);
    if (!rows_bad && (it.q_len == 0 || it.row0 >= it.q_len)) return false;
    if (rows_bad || it.ctx > a.max_blocks_per_seq * kB || it.q_len > it.ctx) {
        if (check && it.h == 0 && it.row0 == 0) atomicOr(a.err, PA_DEVERR_CONTEXT);
        return false;
    }
    it.ntiles = it.q_len - it.row0 > kBM ? 2 : 1;
    const int rows_last = min(kBM, it.q_len - it.row0 - (it.ntiles - 1) * kBM);
    it.kmax = it.ctx - it.q_len + it.row0 + (it.ntiles - 1) * kBM + rows_last;
    it.nkt = (it.kmax + kBN - 1) / kBN;
    return true;
}

// key tiles needed by query tile t of an item (0 if the tile is idle)
template <bool kShared>
__device__ __forceinline__ int tile_key_tiles(const Item &it, int t) {
    if (t >= it.ntiles) return 0;
    if constexpr (kShared) return it.nkt;
    const int rows_t = min(kBM, it.q_len - it.row0 - t * kBM);
    return (it.ctx - it.q_len + it.row0 + t * kBM + rows_t + kBN - 1) / kBN;
}

template <typename E, bool kShared>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + OFF_TMEM);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_FLAG);
    volatile int *item_ring = reinterpret_cast<volatile int *>(smem + OFF_ITEM);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int H = a.num_heads;
    const int num_items = a.num_pairs * a.num_seqs * a.num_heads;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t count = 1;
            if ((i >= P_FULL && i < P_FULL + 4) || i == O_EMPTY || i == O_EMPTY + 1)
                count = 4;                       // one arrival per softmax warp
            else if (i == ITEM_EMPTY || i == ITEM_EMPTY + 1)
                count = 12;                      // the 4 MMA threads and the 8 softmax warps
            else if ((i >= K_EMPTY && i < K_EMPTY + kStages) ||
                     (i >= V_EMPTY && i < V_EMPTY + kStages) || i == Q_EMPTY || i == ZERO_SEEN)
                count = 2;                       // the 2 S threads / the 2 P V threads
            mbar_init(&bar[i], count);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(const_cast<uint32_t *>(tmem_slot))),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // global memory written by the previous kernel on the stream is read only
    // after this point
    grid_dependency_wait();
    allow_dependents_to_launch();

    if (warp >= 8) {
      // the register split is made at the top of each warpgroup's branch, so
      // the compiler allocates each role against its own limit
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
      if (warp == kTmaWarp) {
        // ------------------------------------------------------------ TMA
        // Takes items from the queue, publishes them to the other roles
        // through a two-slot ring, and loads their Q, K and V.
        uint32_t gk = 0, gv = 0;   // K / V tiles issued, over all items
        int k = 0;           // items published
        int q_loads = 0;     // Q loads issued
        bool ok = true;
        for (;;) {
            int w = 0;
            Item it;
            for (;;) {       // next non-empty item, or the end of the queue
                if (lane == 0) w = static_cast<int>(atomicAdd(a.counters, 1u));
                w = __shfl_sync(0xffffffffu, w, 0);
                if (w >= num_items) break;
                if (item_geometry<kShared>(a, w, lane == 0, it)) break;
            }
            const bool done = w >= num_items;
            const int slot = k % 2;
            ok = warp_all(mbar_wait(&bar[ITEM_EMPTY + slot], ((k / 2) & 1) ^ 1, abort_flag, a.err));
            if (!ok) break;
            if (lane == 0) {
                item_ring[slot] = done ? -1 : w;
                mbar_arrive(&bar[ITEM_FULL + slot]);   // release: the slot is visible
            }
            if (done) break;
            // Q: the previous item's S products must all have been issued and done
            if (k > 0) {
                ok = warp_all(mbar_wait(&bar[Q_EMPTY], (k - 1) & 1, abort_flag, a.err));
                if (!ok) break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar[Q_FULL], it.ntiles * kTileQ);
                for (int t = 0; t < it.ntiles; ++t)
                    for (int half = 0; half < 2; ++half)
                        tma_load_3d(smem + OFF_Q + t * kTileQ + half * kHalfQ, &tm_q, half * 64,
                                    it.h, it.q_first + it.row0 + t * kBM, &bar[Q_FULL]);
            }
            ++q_loads;
            const int nblk_needed = (it.kmax + kB - 1) / kB;
            const int32_t *table = a.block_tables + static_cast<size_t>(it.table_row) * a.max_blocks_per_seq;
            for (int j = 0; j < it.nkt && ok; ++j) {
                const int st = gk % kStages;
                const uint32_t ph = (gk / kStages) & 1;
                // physical blocks of this key tile: lane i < 4 looks up block i
                int phys = -1;
                const int b = j * kBlocksPerTile + lane;
                if (lane < kBlocksPerTile && b < nblk_needed) {
                    const int p = __ldg(table + b);
                    if (static_cast<unsigned>(p) < static_cast<unsigned>(a.num_blocks))
                        phys = p;
                    else
                        atomicOr(a.err, PA_DEVERR_TABLE);
                }
                const unsigned valid_mask = __ballot_sync(0xffffffffu, phys >= 0);
                const uint32_t bytes = __popc(valid_mask) * 2u * kB * 128u;
                const int y = (phys * H + it.h) * kB;
                ok = warp_all(mbar_wait(&bar[K_EMPTY + st], ph ^ 1, abort_flag, a.err));
                if (!ok) break;
                if (lane == 0) mbar_arrive_expect_tx(&bar[K_FULL + st], bytes);
                __syncwarp();
                if (phys >= 0) {
                    uint8_t *dst = smem + OFF_K + st * kTileKV + lane * (kB * 128);
                    tma_load_2d(dst, &tm_k, 0, y, &bar[K_FULL + st]);
                    tma_load_2d(dst + kHalfKV, &tm_k, 64, y, &bar[K_FULL + st]);
                }
                ++gk;
                ok = warp_all(mbar_wait(&bar[V_EMPTY + st], ph ^ 1, abort_flag, a.err));
                if (!ok) break;
                if (lane == 0) mbar_arrive_expect_tx(&bar[V_FULL + st], bytes);
                __syncwarp();
                if (phys >= 0) {
                    uint8_t *dst = smem + OFF_V + st * kTileKV + lane * (kB * 128);
                    tma_load_2d(dst, &tm_v, 0, y, &bar[V_FULL + st]);
                    tma_load_2d(dst + kHalfKV, &tm_v, 64, y, &bar[V_FULL + st]);
                }
                ++gv;
                if (j == it.nkt - 1) {
                    // clear V rows kmax .. end of the tile once the loads have
                    // landed (and the P V threads are past the previous item's)
                    ok = warp_all(mbar_wait(&bar[V_FULL + st], ph, abort_flag, a.err));
                    if (ok && k > 0)
                        ok = warp_all(mbar_wait(&bar[ZERO_SEEN], (k - 1) & 1, abort_flag, a.err));
                    if (!ok) break;
                    const int first_zero = it.kmax - j * kBN;
                    uint8_t *vt = smem + OFF_V + st * kTileKV;
                    for (int idx = lane; idx < (kBN - first_zero) * 16; idx += 32) {
                        const int key = first_zero + idx / 16, half = (idx / 8) % 2, c = idx % 8;
                        *reinterpret_cast<uint4 *>(vt + half * kHalfKV + key * 128 + c * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[V_ZERO]);
                }
            }
            if (!ok) break;
            ++k;
        }
        if (lane == 0) {
            if (!ok) {  // let every copy already issued land
                if (q_loads > 0) mbar_wait_drain(&bar[Q_FULL], (q_loads - 1) & 1);
                for (uint32_t i = gk > kStages ? gk - kStages : 0; i < gk; ++i)
                    mbar_wait_drain(&bar[K_FULL + i % kStages], (i / kStages) & 1);
                for (uint32_t i = gv > kStages ? gv - kStages : 0; i < gv; ++i)
                    mbar_wait_drain(&bar[V_FULL + i % kStages], (i / kStages) & 1);
            }
            // the last CTA to leave the queue leaves both counters at zero for
            // the next launch
            __threadfence();
            if (atomicAdd(a.counters + 1, 1u) == gridDim.x - 1) {
                atomicExch(a.counters, 0u);
                atomicExch(a.counters + 1, 0u);
            }
        }
        __syncwarp();
      } else if (warp == kSWarp0 || warp == kSWarp0 + 1) {
        // ------------------------------------------------------------ S
        // One thread per query tile t: S_t(n) = Q_t K^T into buffer n % 2,
        // once the P V product that last read that buffer (number n - 2) is
        // complete; the buffers let S run two key tiles ahead of the
        // softmax.  Every K tile of an item receives one EMPTY arrival from
        // each of the two threads.
        if (lane == 0) {
            const int t = warp - kSWarp0;
            constexpr uint32_t idesc_s = instr_desc(E::kBf16, false, kBN);
            const uint32_t q_addr = smem_addr(smem + OFF_Q) + t * kTileQ;
            const uint32_t k_addr = smem_addr(smem + OFF_K);
            uint32_t g = 0;      // K tiles consumed, over all items
            uint32_t ns = 0;     // S products issued
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int slot = k % 2;
                ok = mbar_wait(&bar[ITEM_FULL + slot], (k / 2) & 1, abort_flag, a.err);
                if (!ok) break;
                const int w = item_ring[slot];
                mbar_arrive(&bar[ITEM_EMPTY + slot]);
                if (w < 0) break;
                Item it;
                item_geometry<kShared>(a, w, false, it);
                const int nk = tile_key_tiles<kShared>(it, t);
                ok = mbar_wait(&bar[Q_FULL], k & 1, abort_flag, a.err);
                if (ok && nk == 0) mbar_arrive(&bar[Q_EMPTY]);   // this query tile is idle
                for (int j = 0; j < it.nkt && ok; ++j, ++g) {
                    const int st = g % kStages;
                    ok = mbar_wait(&bar[K_FULL + st], (g / kStages) & 1, abort_flag, a.err);
                    if (!ok) break;
                    if (j >= nk) {
                        mbar_arrive(&bar[K_EMPTY + st]);
                        continue;
                    }
                    const uint32_t buf = ns % kSBufs;
                    if (ns >= kSBufs)   // the buffer's previous reader
                        ok = mbar_wait(&bar[PV_DONE + t * kSBufs + buf], ((ns - kSBufs) / kSBufs) & 1,
                                       abort_flag, a.err);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t tm_s = tmem + kTmemS + t * 128 + buf * 64;
#pragma unroll
                    for (int ks = 0; ks < kD / 16; ++ks) {  // over the 128 dims
                        const int half = ks / 4, kk = ks % 4;
                        mma_ss(tm_s, smem_desc(q_addr + half * kHalfQ + kk * 32, 16, 1024),
                               smem_desc(k_addr + st * kTileKV + half * kHalfKV + kk * 32, 16, 1024),
                               idesc_s, ks > 0);
                    }
                    mma_commit(&bar[S_FULL + t * kSBufs + buf]);
                    ++ns;
                    mma_commit(&bar[K_EMPTY + st]);
                    if (j == nk - 1) mma_commit(&bar[Q_EMPTY]);   // this tile's last S
                }
            }
            // make sure none of this thread's products is still running when
            // the CTA releases TMEM
            mma_commit(&bar[MMA_DONE + t]);
            mbar_wait_drain(&bar[MMA_DONE + t], 0);
        }
        __syncwarp();
      } else if (warp == kPvWarp0 || warp == kPvWarp0 + 1) {
        // ------------------------------------------------------------ P V
        // One thread per query tile t: O_t += P_hi V + P_lo V for each key
        // tile, once softmax t has published P_t.  Every V tile of an item
        // receives one EMPTY arrival from each of the two threads.
        if (lane == 0) {
            const int t = warp - kPvWarp0;
            constexpr uint32_t idesc_pv = instr_desc(E::kBf16, true, kD);
            const uint32_t v_addr = smem_addr(smem + OFF_V);
            const uint32_t tm_s = tmem + kTmemS + t * 128;   // + 64 b for buffer b
            const uint32_t tm_o = tmem + kTmemO + t * 128;
            uint32_t g = 0;      // V tiles consumed, over all items
            uint32_t np = 0;     // P_t tiles consumed (buffer = np % 2)
            uint32_t oc = 0;     // items in which this query tile was active
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int slot = k % 2;
                ok = mbar_wait(&bar[ITEM_FULL + slot], (k / 2) & 1, abort_flag, a.err);
                if (!ok) break;
                const int w = item_ring[slot];
                mbar_arrive(&bar[ITEM_EMPTY + slot]);
                if (w < 0) break;
                Item it;
                item_geometry<kShared>(a, w, false, it);
                const int nk = tile_key_tiles<kShared>(it, t);
                for (int j = 0; j < it.nkt && ok; ++j, ++g) {
                    const int st = g % kStages;
                    const bool last = j == it.nkt - 1;
                    ok = last ? mbar_wait(&bar[V_ZERO], k & 1, abort_flag, a.err)
                              : mbar_wait(&bar[V_FULL + st], (g / kStages) & 1, abort_flag, a.err);
                    if (!ok) break;
                    if (last) mbar_arrive(&bar[ZERO_SEEN]);
                    if (j < nk) {
                        const uint32_t buf = np % kSBufs;
                        ok = mbar_wait(&bar[P_FULL + t * kSBufs + buf], (np / kSBufs) & 1, abort_flag,
                                       a.err);
                        // O_t still holds the previous item's result until its
                        // epilogue has read it
                        if (ok && j == 0 && oc > 0)
                            ok = mbar_wait(&bar[O_EMPTY + t], (oc - 1) & 1, abort_flag, a.err);
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int pass = 0; pass < 2; ++pass)  // O_t += P_hi V + P_lo V
#pragma unroll
                            for (int ks = 0; ks < kBN / 16; ++ks)
                                mma_ts(tm_o, tm_s + buf * 64 + pass * 32 + ks * 8,
                                       smem_desc(v_addr + st * kTileKV + ks * 2048, kHalfKV, 1024),
                                       idesc_pv, j > 0 || pass > 0 || ks > 0);
                        mma_commit(&bar[PV_DONE + t * kSBufs + buf]);
                        mma_commit(&bar[V_EMPTY + st]);
                        ++np;
                        if (j == nk - 1) mma_commit(&bar[O_FULL + t]);
                    } else {
                        mbar_arrive(&bar[V_EMPTY + st]);
                    }
                }
                if (nk > 0) ++oc;
            }
            mma_commit(&bar[MMA_DONE + 2 + t]);
            mbar_wait_drain(&bar[MMA_DONE + 2 + t], 0);
        }
        __syncwarp();
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ------------------------------------------------------------ softmax
        const int t = warp / 4;                      // query tile of this warpgroup
        const int r = (warp % 4) * 32 + lane;        // row within the tile = TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
        const uint32_t s_col = lane_base + kTmemS + t * 128;   // + 64 b for buffer b
        const uint32_t o_col = lane_base + kTmemO + t * 128;
        const float c = a.scale_log2;
        const bool scale_pos = c > 0.f;
        const float cm = scale_pos ? c : 1.f;   // multiplier left for the exponent
        uint32_t n = 0;                         // S tiles consumed (buffer = n % 2)
        uint32_t o_cnt = 0;                     // O_FULL phases consumed
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int slot = k % 2;
            ok = warp_all(mbar_wait(&bar[ITEM_FULL + slot], (k / 2) & 1, abort_flag, a.err));
            if (!ok) break;
            const int w = item_ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[ITEM_EMPTY + slot]);
            if (w < 0) break;
            Item it;
            item_geometry<kShared>(a, w, false, it);
            if (t >= it.ntiles) continue;
            const int rows_t = min(kBM, it.q_len - it.row0 - t * kBM);
            // key position of the row (every row sits past the whole prefix
            // in shared-prefix mode)
            const int first_pos = kShared ? it.ctx - 1 : it.ctx - it.q_len + it.row0 + t * kBM;
            const int my_nkt = tile_key_tiles<kShared>(it, t);
            const int pos = r < rows_t ? (kShared ? first_pos : first_pos + r) : -1;   // -1: padding row, all masked
            const int warp_min_pos = __reduce_min_sync(0xffffffffu, pos);
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < my_nkt && ok; ++j, ++n) {
                const uint32_t buf = n % kSBufs;
                ok = warp_all(mbar_wait(&bar[S_FULL + t * kSBufs + buf], (n / kSBufs) & 1, abort_flag,
                                        a.err));
                if (!ok) break;
                tc_fence_after();
                const uint32_t sb = s_col + buf * 64;
                float x[kBN];
                // the tile's scores, in the log2 domain for a non-positive
                // scale (for a positive one the scale is folded into the
                // exponent's FMA), causally masked (key j*64 + i is visible to
                // this row iff i <= pos - j*64)
                auto load_scores = [&]() {
                    uint32_t u[kBN];
#pragma unroll
                    for (int q2 = 0; q2 < kBN / 32; ++q2)
                        tmem_ld32_nowait(sb + q2 * 32, *reinterpret_cast<uint32_t(*)[32]>(&u[q2 * 32]));
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < kBN; ++i) x[i] = __uint_as_float(u[i]);
                    if (!scale_pos) {
#pragma unroll
                        for (int i = 0; i < kBN; ++i) x[i] *= c;
                    }
                    if (j * kBN + kBN - 1 > warp_min_pos) {
                        const int lim = pos - j * kBN;
#pragma unroll
                        for (int i = 0; i < kBN; ++i) x[i] = i <= lim ? x[i] : -INFINITY;
                    }
                };
                // x <- 2^(x cm + bias) in place; returns the row sum
                auto exponentiate = [&](float bias) {
                    float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int i = 0; i < kBN; i += 8) {
#pragma unroll
                        for (int q = 0; q < 8; q += 2) {
                            fma2(x[i + q], x[i + q + 1], x[i + q], x[i + q + 1], cm, cm, bias, bias);
                            x[i + q] = fast_exp2(x[i + q]);
                            x[i + q + 1] = fast_exp2(x[i + q + 1]);
                            add2(sum[q], sum[q + 1], sum[q], sum[q + 1], x[i + q], x[i + q + 1]);
                        }
                    }
                    add2(sum[0], sum[1], sum[0], sum[1], sum[2], sum[3]);
                    add2(sum[4], sum[5], sum[4], sum[5], sum[6], sum[7]);
                    add2(sum[0], sum[1], sum[0], sum[1], sum[4], sum[5]);
                    return sum[0] + sum[1];
                };
                load_scores();
                // Optimistic pass: weights against the running maximum.  A row
                // sum of at most 2^14 proves that no weight exceeds 2^14, i.e.
                // that the tile's maximum does not exceed the running one by
                // more than the margin, so the maximum stays and no max pass is
                // needed.  Otherwise (always on a query tile's first key tile)
                // the scores are read again -- P has not overwritten them yet
                // -- and the maximum is taken first.
                float m_new = m_used, alpha = 1.f, tile_sum = 0.f;
                bool exact = !warp_all(m_used != -INFINITY);
                if (!exact) {
                    tile_sum = exponentiate(kBiasLog2 - m_used);
                    exact = !warp_all(tile_sum <= 16384.f);
                    if (exact) load_scores();
                }
                if (exact) {
                    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int i = 0; i < kBN; i += 8)
#pragma unroll
                        for (int q = 0; q < 4; ++q) mx[q] = max3(mx[q], x[i + 2 * q], x[i + 2 * q + 1]);
                    const float m_tile = max3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * cm;
                    if (m_tile > m_used + kRescaleLog2) m_new = m_tile;
                    alpha = m_new == m_used ? 1.f : fast_exp2(m_used - m_new);
                    tile_sum = exponentiate(m_new == -INFINITY ? 0.f : kBiasLog2 - m_new);
                }
                l = l * alpha + tile_sum;
                m_used = m_new;
                // P_t into the buffer: P_hi at +0..31, P_lo at +32..63
#pragma unroll
                for (int q2 = 0; q2 < kBN / 32; ++q2) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        E::split2(x[q2 * 32 + 2 * e], x[q2 * 32 + 2 * e + 1], hi[e], lo[e]);
                    tmem_st16(sb + q2 * 16, hi);
                    tmem_st16(sb + 32 + q2 * 16, lo);
                }
                // a raised maximum rescales O_t once the previous tile's P V
                // product (the last update of O_t) is complete
                if (j > 0 && !warp_all(alpha == 1.f)) {
                    const uint32_t pb = (n - 1) % kSBufs;
                    ok = warp_all(mbar_wait(&bar[PV_DONE + t * kSBufs + pb], ((n - 1) / kSBufs) & 1,
                                            abort_flag, a.err));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t ov[32];
                        tmem_ld32_nowait(o_col + q4 * 32, ov);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st32(o_col + q4 * 32, ov);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[P_FULL + t * kSBufs + buf]);
            }
            if (!ok) break;
            // epilogue: read O_t, hand its columns back to the MMA warp, then
            // normalise and store
            ok = warp_all(mbar_wait(&bar[O_FULL + t], o_cnt & 1, abort_flag, a.err));
            ++o_cnt;
            if (!ok) break;
            tc_fence_after();
            uint32_t ov[kD];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                tmem_ld32_nowait(o_col + q4 * 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[q4 * 32]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[O_EMPTY + t]);
            if (kShared && r < rows_t) {
                // a decode partial for row s: the weights were 2^(x - (m - 6))
                const size_t pidx =
                    (static_cast<size_t>(it.q_first + it.row0 + t * kBM + r) * H + it.h) * a.max_parts;
                reinterpret_cast<float2 *>(a.part_ml)[pidx] = make_float2(m_used - kBiasLog2, l);
                float4 *dst = reinterpret_cast<float4 *>(a.part_acc + pidx * kD);
#pragma unroll
                for (int c4 = 0; c4 < kD / 4; ++c4)
                    dst[c4] = make_float4(__uint_as_float(ov[4 * c4]), __uint_as_float(ov[4 * c4 + 1]),
                                          __uint_as_float(ov[4 * c4 + 2]), __uint_as_float(ov[4 * c4 + 3]));
            } else if (r < rows_t) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                uint16_t *dst =
                    a.out + (static_cast<size_t>(it.q_first + it.row0 + t * kBM + r) * H + it.h) * kD;
#pragma unroll
                for (int c8 = 0; c8 < kD / 8; ++c8) {
                    uint16_t v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = E::round(__uint_as_float(ov[c8 * 8 + e]) * inv);
                    *reinterpret_cast<uint4 *>(dst + c8 * 8) = *reinterpret_cast<const uint4 *>(v);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
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

bool encode(CUtensorMap *tm, bool bf16, const void *base, int rank, const cuuint64_t *dims,
            const cuuint64_t *strides, const cuuint32_t *box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(tm, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
              rank, const_cast<void *>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace

bool prefill_supported(int dtype, int head_dim, int block_size) {
    return (dtype == PA_DTYPE_F16 || dtype == PA_DTYPE_BF16) && head_dim == kD && block_size == kB;
}

cudaError_t launch_prefill(const PrefillArgs &args, const void *q, const void *k_cache,
                           const void *v_cache, int dtype, int num_sms, cudaStream_t stream) {
    const bool bf16 = dtype == PA_DTYPE_BF16;
    const int H = args.num_heads;
    CUtensorMap tm_q, tm_k, tm_v;
    const cuuint64_t q_dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H),
                                  static_cast<cuuint64_t>(args.total_q)};
    const cuuint64_t q_strides[2] = {static_cast<cuuint64_t>(kD) * 2,
                                     static_cast<cuuint64_t>(H) * kD * 2};
    const cuuint32_t q_box[3] = {64, 1, kBM};
    const cuuint64_t kv_dims[2] = {static_cast<cuuint64_t>(kD),
                                   static_cast<cuuint64_t>(args.num_blocks) * H * kB};
    const cuuint64_t kv_strides[1] = {static_cast<cuuint64_t>(kD) * 2};
    const cuuint32_t kv_box[2] = {64, kB};
    if (!encode(&tm_q, bf16, q, 3, q_dims, q_strides, q_box) ||
        !encode(&tm_k, bf16, k_cache, 2, kv_dims, kv_strides, kv_box) ||
        !encode(&tm_v, bf16, v_cache, 2, kv_dims, kv_strides, kv_box))
        return cudaErrorInvalidValue;
    const bool shared = args.group_prefix_blocks != nullptr;
    const void *kernels[2][2] = {
        {reinterpret_cast<const void *>(&prefill_kernel<F16T, false>),
         reinterpret_cast<const void *>(&prefill_kernel<F16T, true>)},
        {reinterpret_cast<const void *>(&prefill_kernel<BF16T, false>),
         reinterpret_cast<const void *>(&prefill_kernel<BF16T, true>)}};
    const void *kernel = kernels[bf16 ? 1 : 0][shared ? 1 : 0];
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    {
        static std::mutex mu;
        static bool ready[64][4] = {};   // per kernel variant
        const int which = (bf16 ? 2 : 0) + (shared ? 1 : 0);
        std::lock_guard<std::mutex> lock(mu);
        if (!ready[device][which]) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemBytes);
            if (e != cudaSuccess) return e;
            ready[device][which] = true;
        }
    }
    void *params[] = {&tm_q, &tm_k, &tm_v, const_cast<PrefillArgs *>(&args)};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    // persistent: one CTA per SM (the shared memory allows no second one)
    const long long items = static_cast<long long>(args.num_pairs) * args.num_seqs * H;
    cfg.gridDim = dim3(static_cast<unsigned>(items < num_sms ? items : num_sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, kernel, params);
}

}  // namespace pa
