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
// the 5th-generation tensor cores with accumulators in tensor memory.
//  * One CTA per (tile of 128 queries, head, sequence); six warps.
//  * Warp 4 (TMA): loads the Q tile once and, per tile of 64 keys, the four
//    16-token K and V blocks named by the block table, each as two 2-D
//    tensor-map boxes (64 dims x 16 tokens) that land directly in the
//    128-byte-swizzled operand layouts; double-buffered.
//  * Warp 5 (MMA): S = Q K^T (M 128, N 64, K 128) into TMEM columns 0-63;
//    after the softmax warps publish P, PV = P_hi V + P_lo V (M 128, N 128,
//    K 64, V as an MN-major operand) into TMEM columns 128-255.
//  * Warps 0-3 (softmax): thread t owns query row t (the TMEM lane layout of
//    an M = 128 accumulator), reads its 64 scores with tcgen05.ld, masks the
//    causal and context boundary, keeps the running max / sum in fp32 and
//    the output row in registers (rescaled each tile), and writes P to
//    shared memory as a 16-bit pair P_hi + P_lo (P_lo = P - P_hi), which
//    keeps P exact to about 22 bits so small outputs meet the same relative
//    bound as decode.  Rows of V past the last key are zeroed before use
//    (a zero weight times a NaN would still be NaN).
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
constexpr int kBM = 128;            // query rows per CTA (MMA M)
constexpr int kBN = 64;             // keys per tile
constexpr int kB = 16;              // block_size
constexpr int kBlocksPerTile = kBN / kB;
constexpr int kStages = 2;
constexpr int kThreads = 192;       // 4 softmax warps + TMA warp + MMA warp
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemS = 0;      // S: columns 0-63
constexpr uint32_t kTmemPV = 128;   // PV: columns 128-255

// shared memory layout (bytes; tiles 1024-aligned for the 128B swizzle)
constexpr int kHalfRowsQ = kBM * 128;          // one 64-dim half of Q: 128 rows x 128 B
constexpr int OFF_Q = 0;                       // [2 halves][128 rows][128 B]
constexpr int kTileKV = 2 * kBN * 128;         // K or V tile: 2 halves x 64 keys x 128 B
constexpr int OFF_K = OFF_Q + 2 * kHalfRowsQ;  // [stage][half][64 keys][128 B]
constexpr int OFF_V = OFF_K + kStages * kTileKV;
constexpr int kTileP = kBM * 128;              // P: 128 rows x 64 keys x 2 B
constexpr int OFF_PHI = OFF_V + kStages * kTileKV;
constexpr int OFF_PLO = OFF_PHI + kTileP;
constexpr int OFF_BAR = OFF_PLO + kTileP;
constexpr int kNumBars = 12;
constexpr int OFF_TMEM = OFF_BAR + kNumBars * 8;
constexpr int OFF_FLAG = OFF_TMEM + 8;
constexpr int kSmemBytes = OFF_FLAG + 8 + 1024;  // + alignment slack

enum Bar { Q_FULL = 0, K_FULL = 1, V_FULL = 3, KV_EMPTY = 5, S_FULL = 7, S_EMPTY = 8, P_FULL = 9,
           PV_FULL = 10, MMA_DONE = 11 };

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

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                        bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1 : 0));
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

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t addr, float (&v)[32]) {
    uint32_t r[32];
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
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
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

struct F16T {
    static constexpr bool kBf16 = false;
    __device__ static __forceinline__ uint16_t round(float x) {
        const __half h = __float2half_rn(x);
        return *reinterpret_cast<const uint16_t *>(&h);
    }
    __device__ static __forceinline__ float widen(uint16_t b) {
        return __half2float(*reinterpret_cast<const __half *>(&b));
    }
};
struct BF16T {
    static constexpr bool kBf16 = true;
    __device__ static __forceinline__ uint16_t round(float x) {
        const __nv_bfloat16 b = __float2bfloat16_rn(x);
        return *reinterpret_cast<const uint16_t *>(&b);
    }
    __device__ static __forceinline__ float widen(uint16_t b) {
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
};

template <typename E>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + OFF_TMEM);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_FLAG);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int s = blockIdx.z, h = blockIdx.y, qt = blockIdx.x;
    const int H = a.num_heads;

    grid_dependency_wait();
    allow_dependents_to_launch();
    const int q_first = a.query_start[s];
    const int q_len = a.query_start[s + 1] - q_first;
    int ctx = a.context_lens[s];
    const int row0 = qt * kBM;
    if (q_len <= 0 || row0 >= q_len) return;  // nothing for this CTA (before any set-up)
    if (ctx > a.max_blocks_per_seq * kB || q_len > ctx || q_first < 0 ||
        q_first + q_len > a.total_q) {
        if (threadIdx.x == 0) atomicOr(a.err, PA_DEVERR_CONTEXT);
        return;
    }
    const int rows = min(kBM, q_len - row0);
    const int first_pos = ctx - q_len + row0;     // position of tile row 0
    const int kmax = first_pos + rows;            // keys 0 .. kmax-1 are needed
    const int nkt = (kmax + kBN - 1) / kBN;       // key tiles
    const int nblk_needed = (kmax + kB - 1) / kB;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i)
            mbar_init(&bar[i], i == S_EMPTY ? 4       // one arrival per softmax warp
                               : i == P_FULL ? 128   // every softmax thread
                                             : 1);
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

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ TMA
        uint32_t issued = 0;  // key tiles issued
        bool ok = true;
        if (lane == 0) {
            mbar_arrive_expect_tx(&bar[Q_FULL], 2 * kHalfRowsQ);
            tma_load_3d(smem + OFF_Q, &tm_q, 0, h, q_first + row0, &bar[Q_FULL]);
            tma_load_3d(smem + OFF_Q + kHalfRowsQ, &tm_q, 64, h, q_first + row0, &bar[Q_FULL]);
            const int32_t *table = a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq;
            for (int j = 0; j < nkt; ++j) {
                const int st = j % kStages;
                if (!mbar_wait(&bar[KV_EMPTY + st], ((j / kStages) & 1) ^ 1, abort_flag, a.err)) {
                    ok = false;
                    break;
                }
                int phys[kBlocksPerTile];
                int nvalid = 0;
#pragma unroll
                for (int i = 0; i < kBlocksPerTile; ++i) {
                    const int b = j * kBlocksPerTile + i;
                    phys[i] = -1;
                    if (b < nblk_needed) {
                        const int p = __ldg(table + b);
                        if (static_cast<unsigned>(p) < static_cast<unsigned>(a.num_blocks)) {
                            phys[i] = p;
                            ++nvalid;
                        } else {
                            atomicOr(a.err, PA_DEVERR_TABLE);
                        }
                    }
                }
                uint8_t *kdst = smem + OFF_K + st * kTileKV;
                uint8_t *vdst = smem + OFF_V + st * kTileKV;
                mbar_arrive_expect_tx(&bar[K_FULL + st], nvalid * 2 * kB * 128);
                mbar_arrive_expect_tx(&bar[V_FULL + st], nvalid * 2 * kB * 128);
#pragma unroll
                for (int i = 0; i < kBlocksPerTile; ++i) {
                    if (phys[i] < 0) continue;
                    const int y = (phys[i] * H + h) * kB;
                    for (int half = 0; half < 2; ++half) {
                        const int off = half * (kBN * 128) + i * (kB * 128);
                        tma_load_2d(kdst + off, &tm_k, half * 64, y, &bar[K_FULL + st]);
                        tma_load_2d(vdst + off, &tm_v, half * 64, y, &bar[V_FULL + st]);
                    }
                }
                ++issued;
            }
            if (!ok) {  // let every copy already issued land
                mbar_wait_drain(&bar[Q_FULL], 0);
                for (uint32_t j = issued > kStages ? issued - kStages : 0; j < issued; ++j) {
                    mbar_wait_drain(&bar[K_FULL + j % kStages], (j / kStages) & 1);
                    mbar_wait_drain(&bar[V_FULL + j % kStages], (j / kStages) & 1);
                }
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idesc_s = instr_desc(E::kBf16, false, kBN);
            constexpr uint32_t idesc_pv = instr_desc(E::kBf16, true, kD);
            const uint32_t q_addr = smem_addr(smem + OFF_Q);
            bool ok = mbar_wait(&bar[Q_FULL], 0, abort_flag, a.err);
            int committed = 0;
            for (int j = 0; j < nkt && ok; ++j) {
                const int st = j % kStages;
                ok = mbar_wait(&bar[K_FULL + st], (j / kStages) & 1, abort_flag, a.err);
                if (ok && j > 0) ok = mbar_wait(&bar[S_EMPTY], (j - 1) & 1, abort_flag, a.err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t k_addr = smem_addr(smem + OFF_K + st * kTileKV);
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {  // S = Q K^T over the 128 dims
                    const int half = ks / 4, kk = ks % 4;
                    mma_f16(tmem + kTmemS,
                            smem_desc(q_addr + half * kHalfRowsQ + kk * 32, 16, 1024),
                            smem_desc(k_addr + half * (kBN * 128) + kk * 32, 16, 1024), idesc_s,
                            ks > 0);
                }
                mma_commit(&bar[S_FULL]);
                ok = mbar_wait(&bar[P_FULL], j & 1, abort_flag, a.err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t v_addr = smem_addr(smem + OFF_V + st * kTileKV);
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {  // PV = P_hi V + P_lo V
                    const uint32_t p_addr = smem_addr(smem + (pass ? OFF_PLO : OFF_PHI));
#pragma unroll
                    for (int ks = 0; ks < kBN / 16; ++ks)
                        mma_f16(tmem + kTmemPV, smem_desc(p_addr + ks * 32, 16, 1024),
                                smem_desc(v_addr + ks * 2048, kBN * 128, 1024), idesc_pv,
                                pass > 0 || ks > 0);
                }
                mma_commit(&bar[PV_FULL]);
                mma_commit(&bar[KV_EMPTY + st]);
                ++committed;
            }
            // make sure no MMA is still running when the CTA releases TMEM
            mma_commit(&bar[MMA_DONE]);
            mbar_wait_drain(&bar[MMA_DONE], 0);
            (void)committed;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int r = threadIdx.x;                 // query row of this thread
        const bool row_valid = r < rows;
        const int pos = first_pos + r;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        float run_max = -INFINITY, run_sum = 0.f, alpha_prev = 0.f;
        float o[kD];
#pragma unroll
        for (int d = 0; d < kD; ++d) o[d] = 0.f;
        bool ok = true;
        uint8_t *phi = smem + OFF_PHI + r * 128;
        uint8_t *plo = smem + OFF_PLO + r * 128;
        for (int j = 0; j < nkt && ok; ++j) {
            const int st = j % kStages;
            ok = __all_sync(0xffffffffu, mbar_wait(&bar[S_FULL], j & 1, abort_flag, a.err));
            if (!ok) break;
            tc_fence_after();
            float sc[kBN];
            tmem_ld32(lane_base + kTmemS, *reinterpret_cast<float(*)[32]>(&sc[0]));
            tmem_ld32(lane_base + kTmemS + 32, *reinterpret_cast<float(*)[32]>(&sc[32]));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[S_EMPTY]);
            // causal + context mask, scale into the log2 domain, online softmax
            float tile_max = -INFINITY;
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
                const int key = j * kBN + c;
                sc[c] = (row_valid && key <= pos) ? sc[c] * a.scale_log2 : -INFINITY;
                tile_max = fmaxf(tile_max, sc[c]);
            }
            const float new_max = fmaxf(run_max, tile_max);
            const float ref = new_max == -INFINITY ? 0.f : new_max;
            const float alpha = exp2f(run_max - ref);
            float psum = 0.f;
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
                sc[c] = exp2f(sc[c] - ref);
                psum += sc[c];
            }
            run_sum = run_sum * alpha + psum;
            run_max = new_max;
            // fold in the previous tile's P V (its weights used the previous max)
            if (j > 0) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&bar[PV_FULL], (j - 1) & 1, abort_flag, a.err));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < kD; c0 += 32) {
                    float pv[32];
                    tmem_ld32(lane_base + kTmemPV + c0, pv);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[c0 + i] = fmaf(o[c0 + i], alpha_prev, pv[i]);
                }
            }
            alpha_prev = alpha;
            // P = P_hi + P_lo as two 16-bit K-major rows (128-byte swizzle)
#pragma unroll
            for (int c8 = 0; c8 < kBN / 8; ++c8) {
                uint16_t hi[8], lo[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float p = sc[c8 * 8 + e];
                    hi[e] = E::round(p);
                    lo[e] = E::round(p - E::widen(hi[e]));
                }
                const int chunk = (c8 ^ (r & 7)) * 16;
                *reinterpret_cast<uint4 *>(phi + chunk) = *reinterpret_cast<const uint4 *>(hi);
                *reinterpret_cast<uint4 *>(plo + chunk) = *reinterpret_cast<const uint4 *>(lo);
            }
            // V must have landed; past the last key its rows are zeroed
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bar[V_FULL + st], (j / kStages) & 1, abort_flag, a.err));
            if (!ok) break;
            if (j == nkt - 1) {
                const int first_zero = kmax - j * kBN;       // tile-local key
                const int nzero = kBN - first_zero;          // rows to clear
                uint8_t *vt = smem + OFF_V + st * kTileKV;
                for (int idx = threadIdx.x; idx < nzero * 2 * 8; idx += 128) {
                    const int key = first_zero + idx / 16;
                    const int half = (idx / 8) % 2, chunk = idx % 8;
                    *reinterpret_cast<uint4 *>(vt + half * (kBN * 128) + (key / 8) * 1024 +
                                               (key % 8) * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc_fence_before();
            mbar_arrive(&bar[P_FULL]);
        }
        if (ok)
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bar[PV_FULL], (nkt - 1) & 1, abort_flag, a.err));
        if (ok) {
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < kD; c0 += 32) {
                float pv[32];
                tmem_ld32(lane_base + kTmemPV + c0, pv);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[c0 + i] = fmaf(o[c0 + i], alpha_prev, pv[i]);
            }
            if (row_valid) {
                const float inv = run_sum > 0.f ? 1.f / run_sum : 0.f;
                uint16_t *dst = a.out + (static_cast<size_t>(q_first + row0 + r) * H + h) * kD;
#pragma unroll
                for (int c8 = 0; c8 < kD / 8; ++c8) {
                    uint16_t v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = E::round(o[c8 * 8 + e] * inv);
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
                           const void *v_cache, int dtype, int max_query_len,
                           cudaStream_t stream) {
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
    const void *kernel = bf16 ? reinterpret_cast<const void *>(&prefill_kernel<BF16T>)
                              : reinterpret_cast<const void *>(&prefill_kernel<F16T>);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    {
        static std::mutex mu;
        static bool ready[64][2] = {};
        std::lock_guard<std::mutex> lock(mu);
        if (!ready[device][bf16 ? 1 : 0]) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemBytes);
            if (e != cudaSuccess) return e;
            ready[device][bf16 ? 1 : 0] = true;
        }
    }
    void *params[] = {&tm_q, &tm_k, &tm_v, const_cast<PrefillArgs *>(&args)};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((max_query_len + kBM - 1) / kBM),
                       static_cast<unsigned>(H), static_cast<unsigned>(args.num_seqs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, kernel, params);
}

}  // namespace pa
