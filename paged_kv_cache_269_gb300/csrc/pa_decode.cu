// pa_decode.cu -- paged-attention decode kernel for GB300 (sm_103a).
//
// What it computes: for every sequence s and head h,
//   out[s,h,:] = sum_t softmax_t(scale * q[s,h,:] . K_t) V_t,  t < ctx_s,
// where K_t / V_t is row t % B of physical block block_tables[s][t / B]
// ("vLLM 2026 推理引擎全解：从 PagedAttention 到分离式 Prefill", §1.1 for the
// attention, §2.1-§2.2 for the block table; mjmagnets.cn vLLM tutorial, §2.2:
// the operator gathers the K/V blocks through the table, then computes).
//
// How (a GB300 design, not the pages' sketch):
//  * Work unit = (sequence, head, partition of tiles_per_unit KV blocks).
//    A persistent grid (CTAs per SM x SMs) pulls units from a device-wide
//    atomic queue.  Units are ordered sequence-major, then partition, with the
//    head fastest, so CTAs running at the same time read neighbouring 4 KiB
//    head tiles of the same physical blocks and the same shared-prefix blocks.
//  * Warp specialisation.  One producer warp reads each unit's block-table
//    slice with one coalesced load and streams whole K and V tiles (B x D
//    fp16, contiguous in the [N, H, B, D] layout) into a ring of shared-memory
//    stages with the bulk asynchronous copy engine (cp.async.bulk, completion
//    on an mbarrier).  NC consumer warps take the unit's tiles round-robin.
//  * Per tile, a consumer warp computes the q.k scores with 16-byte shared
//    loads and xor-shuffle reductions, updates a running max / sum softmax in
//    fp32 (the FlashAttention-style page-by-page computation the pages
//    describe, "vLLM 2026 推理引擎全解", §2.2), and accumulates p * V in fp32.
//  * At the end of a unit the NC warps' (max, sum, acc) states are merged in
//    shared memory by one warp.  A unit covering the whole context writes the
//    fp16 output directly.  Otherwise it writes its partial to the workspace
//    and takes a ticket; the last partition of a (sequence, head) to finish
//    combines all partials and writes the output (split-context reduce in the
//    same launch, no second kernel).
//  * No tensor cores: single-query decode is a bandwidth-bound GEMV.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr unsigned kFull = 0xffffffffu;

constexpr int clamp_int(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

// Launch-shape constants, overridable at build time for tuning sweeps.
// Several small CTAs per SM, each with its own producer warp, keep more
// copies in flight than one large CTA: on the LLaMA-7B batch, 4 consumer
// warps with a 40 KiB ring (4 CTAs per SM) ran 1.7x faster than 16 consumer
// warps with a 176 KiB ring (1 CTA per SM).  Two descriptor slots instead of
// four free the shared memory for a sixth ring stage at 4 CTAs per SM.
#ifndef PA_DECODE_CONSUMER_WARPS
#define PA_DECODE_CONSUMER_WARPS 4
#endif
#ifndef PA_DECODE_STAGE_KIB
#define PA_DECODE_STAGE_KIB 48
#endif
// Ring budgets of two small-tile shapes, from a sweep of 32, 40 and 48 KiB:
// D 64 x B 8 at 40 KiB fits four CTAs per SM (56 registers, no spill) instead
// of three (+0.3 %), D 64 x B 16 gains 0.5 % at 32 KiB; every other shape is
// best at 48 KiB (D 128 x B 8 lost 1 % at 32).
#ifndef PA_DECODE_STAGE_KIB_D64_B8
#define PA_DECODE_STAGE_KIB_D64_B8 40
#endif
#ifndef PA_DECODE_STAGE_KIB_D64_B16
#define PA_DECODE_STAGE_KIB_D64_B16 32
#endif
__host__ __device__ constexpr int stage_budget_kib(int head_dim, int block_size) {
    return head_dim == 64 && block_size == 8    ? PA_DECODE_STAGE_KIB_D64_B8
           : head_dim == 64 && block_size == 16 ? PA_DECODE_STAGE_KIB_D64_B16
                                                : PA_DECODE_STAGE_KIB;
}
#ifndef PA_DECODE_MAX_STAGES
#define PA_DECODE_MAX_STAGES 16
#endif

#ifndef PA_DECODE_MIXED_FMA
#define PA_DECODE_MIXED_FMA 1
#endif
#ifndef PA_DECODE_DESC_SLOTS
#define PA_DECODE_DESC_SLOTS 2
#endif

// Heads per work unit by tile size (B x D x 2 bytes), overridable at build
// time.  In the [N, H, B, D] layout the tiles of heads h .. h + HG - 1 of one
// block are one contiguous run, so a unit of HG heads moves each block's K
// (and V) with one bulk copy of HG tiles and reads its table slice once.
// Measured on a LLaMA-shaped batch (H x D = 4096), fraction of the copy rate
// with one head per unit -> the group below: 1 KiB tiles (D 64 x B 8) 0.835
// -> 0.885 with 4 heads; 2 KiB (D 64 x B 16, D 128 x B 8) 0.930 -> 0.975 and
// 0.937 -> 0.960 with 2; 4 KiB tiles of D 64 x B 32 and D 256 x B 8 0.968 ->
// 0.981 and 0.960 -> 0.970 with 2, while D 128 x B 16 lost 0.6 % with 2 and
// keeps one head per unit.
#ifndef PA_DECODE_HG_1K
#define PA_DECODE_HG_1K 4
#endif
#ifndef PA_DECODE_HG_2K
#define PA_DECODE_HG_2K 2
#endif
#ifndef PA_DECODE_HG_4K
#define PA_DECODE_HG_4K 2
#endif
#ifndef PA_DECODE_HG_D128_B16
#define PA_DECODE_HG_D128_B16 1
#endif

__host__ __device__ constexpr int preferred_heads(int head_dim, int block_size) {
    return (head_dim == 128 && block_size == 16) ? PA_DECODE_HG_D128_B16
           : block_size * head_dim * 2 <= 1024 ? PA_DECODE_HG_1K
           : block_size * head_dim * 2 <= 2048 ? PA_DECODE_HG_2K
           : block_size * head_dim * 2 <= 4096 ? PA_DECODE_HG_4K : 1;
}

// Consumer warps per CTA.  1 KiB tiles (D 64 x B 8) leave each warp little
// work per barrier and hand-off, and more warps per CTA hide that: 8 consumer
// warps took that shape from 0.885 to 0.945 of the copy rate, while every
// other shape lost 1-17 % with 8 (fewer CTAs, hence fewer producers, per SM).
#ifndef PA_DECODE_NC_1K
#define PA_DECODE_NC_1K 8
#endif
__host__ __device__ constexpr int consumer_warps(int head_dim, int block_size) {
    return block_size * head_dim * 2 <= 1024 ? PA_DECODE_NC_1K : PA_DECODE_CONSUMER_WARPS;
}

template <int D, int B, int HG = 1>
struct Cfg {
    static_assert(D == 64 || D == 128 || D == 256, "head_dim");
    static_assert(B == 8 || B == 16 || B == 32, "block_size");
    static_assert(HG == 1 || HG == 2 || HG == 4, "heads per unit");
    static constexpr int NC = consumer_warps(D, B);     // consumer warps
    static_assert(NC % HG == 0, "each head of a unit gets the same number of warps");
    static constexpr int THREADS = (NC + 1) * 32;     // + one producer warp
    static constexpr int TILE_BYTES = B * D * 2;      // one K (or V) tile, fp16
    // Blocks per ring stage: with one head per unit, tiles under 2 KiB (D 64 x
    // B 8) are grouped four blocks to a stage, so that one barrier, tag and
    // hand-off carries 4 KiB of K and of V; every other shape, and every unit
    // of several heads, keeps one block per stage.
    static constexpr int R = (HG == 1 && TILE_BYTES < 2048) ? 4096 / TILE_BYTES : 1;
    static_assert(32 % R == 0, "a stage never straddles a 32-entry table slice");
    // [K: R blocks x HG heads][V: the same]
    static constexpr int STAGE_BYTES = 2 * R * HG * TILE_BYTES;
    static constexpr int STAGE_BUDGET = stage_budget_kib(D, B) * 1024;
    // At least 4 stages, unless a 4-stage ring of very large tiles would
    // exceed twice the budget (D 256 x B 32: 128 KiB, one CTA per SM); then
    // 3 stages, so that two CTAs fit (0.91 -> 0.985 of the copy rate there,
    // while 3 stages cost 2 % on the 16 KiB tiles).
    // (the ring holds at most PA_DECODE_MAX_STAGES blocks)
    static constexpr int NS_WANT =
        clamp_int(STAGE_BUDGET / STAGE_BYTES, 4, PA_DECODE_MAX_STAGES / R);
    static constexpr int NS = NS_WANT * STAGE_BYTES > 2 * STAGE_BUDGET
                                  ? clamp_int(2 * STAGE_BUDGET / STAGE_BYTES, 3, PA_DECODE_MAX_STAGES)
                                  : NS_WANT;
    static constexpr int ND = PA_DECODE_DESC_SLOTS;   // unit descriptor slots
    // q.k layout: LPT lanes per token, 8 dims (16 bytes) per lane.
    static constexpr int LPT = D / 8;
    static constexpr int TPR = 32 / LPT;              // tokens per row group
    static constexpr int RG = B / TPR;                // row groups per tile
    static_assert(RG * TPR == B, "tile rows");
    // p.V layout: DPL dims per lane.
    static constexpr int DPL = D / 32;

    static constexpr int OFF_STAGES = 0;
    static constexpr int OFF_DESC_Q = NS * STAGE_BYTES;
    static constexpr int OFF_MERGE_ACC = OFF_DESC_Q + ND * HG * D * 2;
    static constexpr int OFF_MERGE_ML = OFF_MERGE_ACC + ND * NC * D * 4;
    static constexpr int OFF_PROBS = OFF_MERGE_ML + ND * NC * 8;
    static constexpr int OFF_META = OFF_PROBS + NC * B * 4;
    static constexpr int META_INTS = 8;
    static constexpr int OFF_STAGE_OK = OFF_META + ND * META_INTS * 4;
    static constexpr int OFF_STAGE_TAG = OFF_STAGE_OK + NS * 4;
    static constexpr int OFF_BARS = (OFF_STAGE_TAG + NS * 4 + 7) / 8 * 8;
    static constexpr int NUM_BARS = 2 * NS + 3 * ND;
    static constexpr int OFF_FLAGS = OFF_BARS + NUM_BARS * 8;
    static constexpr int OFF_SEQ = OFF_FLAGS + 16;    // prefix[S + 1], ctx[S] (+ shared-prefix state)
    static constexpr int DEFER = 8;                   // deferred prefix merges per consumer warp
    static constexpr int KEYS = 32;                   // unit-length classes of the work order

    // CTAs per SM the shared-memory footprint allows (228 KiB per SM, 1 KiB
    // reserved per CTA, room for 1024 sequences); the launch bound caps the
    // registers so that as many CTAs fit.
    static constexpr int MIN_BLOCKS = clamp_int(228 * 1024 / (OFF_SEQ + 8 * 1024 + 1024), 1, 8);

    // Plain mode keeps, per sequence, its partition count (as a prefix) and
    // context length (chunk_shift 0), or one partition count per chunk of
    // 2^chunk_shift sequences.  Shared-prefix mode (num_groups >= 0) adds each
    // sequence's first block and place in the work order, the group starts,
    // the order's length classes, and the deferred-merge lists (kept small:
    // at S = 128 four CTAs per SM still fit).
    __host__ __device__ static size_t seq_ints(int num_seqs, int num_groups, int chunk_shift) {
        const size_t S = static_cast<size_t>(num_seqs);
        const size_t chunks = chunk_shift == 0 ? 0 : ((S + (size_t{1} << chunk_shift) - 1) >> chunk_shift);
        if (num_groups >= 0) {
            const size_t groups = 2 * static_cast<size_t>(num_groups) + 1;
            return chunk_shift == 0 ? 4 * S + 1 + groups + KEYS : chunks + 1 + groups;
        }
        return chunk_shift == 0 ? 2 * S + 1 : chunks + 1;
    }
    static size_t smem_bytes(int num_seqs, int num_groups, int chunk_shift) {
        size_t n = static_cast<size_t>(OFF_SEQ) + seq_ints(num_seqs, num_groups, chunk_shift) * 4;
        if (num_groups >= 0) n = (n + 7) / 8 * 8 + static_cast<size_t>(NC) * DEFER * 8;
        return n;
    }
};

__device__ __forceinline__ float2 h2f(uint32_t bits) {
    __half2 h = *reinterpret_cast<const __half2 *>(&bits);
    return __half22float2(h);
}

// The 16-bit element types of q, the caches and the output.
struct F16 {
    static constexpr bool kBf16 = false;
    __device__ static __forceinline__ float2 pair(uint32_t bits) { return h2f(bits); }
    __device__ static __forceinline__ uint16_t round(float x) {
        const __half h = __float2half_rn(x);
        return *reinterpret_cast<const uint16_t *>(&h);
    }
};
struct BF16 {
    static constexpr bool kBf16 = true;
    // bf16 is the top half of an fp32: widening is a shift
    __device__ static __forceinline__ float2 pair(uint32_t bits) {
        return make_float2(__uint_as_float(bits << 16), __uint_as_float(bits & 0xffff0000u));
    }
    __device__ static __forceinline__ uint16_t round(float x) {
        const __nv_bfloat16 b = __float2bfloat16_rn(x);
        return *reinterpret_cast<const uint16_t *>(&b);
    }
};

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// Partial q.k over this lane's 8 dims of one K row (16 bytes).
template <typename E>
__device__ __forceinline__ float dot8(const uint4 kv, const uint4 qh, const float (&qf)[8]) {
#if PA_DECODE_MIXED_FMA
    // A product of two 16-bit floats is exact in fp32, so fusing the
    // conversion into the FMA gives the same result as converting first.
    float dot = 0.f;
    const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
    const uint32_t qw[4] = {qh.x, qh.y, qh.z, qh.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (E::kBf16) {
            asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
                "mov.b32 {a0, a1}, %1;\n\t"
                "mov.b32 {b0, b1}, %2;\n\t"
                "fma.rn.f32.bf16 %0, a0, b0, %0;\n\t"
                "fma.rn.f32.bf16 %0, a1, b1, %0;\n\t}"
                : "+f"(dot)
                : "r"(kw[i]), "r"(qw[i]));
        } else {
            asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
                "mov.b32 {a0, a1}, %1;\n\t"
                "mov.b32 {b0, b1}, %2;\n\t"
                "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
                "fma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
                : "+f"(dot)
                : "r"(kw[i]), "r"(qw[i]));
        }
    }
    return dot;
#else
    (void)qh;
    const float2 k0 = E::pair(kv.x), k1 = E::pair(kv.y), k2 = E::pair(kv.z), k3 = E::pair(kv.w);
    float dot = qf[0] * k0.x;
    dot = fmaf(qf[1], k0.y, dot);
    dot = fmaf(qf[2], k1.x, dot);
    dot = fmaf(qf[3], k1.y, dot);
    dot = fmaf(qf[4], k2.x, dot);
    dot = fmaf(qf[5], k2.y, dot);
    dot = fmaf(qf[6], k3.x, dot);
    dot = fmaf(qf[7], k3.y, dot);
    return dot;
#endif
}

// The lazily raised softmax reference may lag the running maximum by up to
// this much (log2 units): weights stay at most 2^8 before a rescale.
constexpr float kLazyLog2 = 8.f;

// Lanes holding copies of the same row after consume_tile's reduce-scatter.
template <int D, int B>
__host__ __device__ constexpr int row_copies() {
    using C = Cfg<D, B>;
    return C::LPT >> ilog2(C::RG < C::LPT ? C::RG : C::LPT);
}

// The warp's sum of a per-lane row quantity (each row counted once).
template <int D, int B>
__device__ __forceinline__ float warp_row_sum(float v) {
#pragma unroll
    for (int o = 16; o >= row_copies<D, B>(); o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// One KV tile of one unit, processed by one warp.
template <typename E, int D, int B>
__device__ __forceinline__ void consume_tile(const uint8_t *ktile, const uint8_t *vtile,
                                             const uint4 qh, const float (&qf)[8],
                                             float scale_log2, int nvalid, float &run_max,
                                             float &run_sum, float (&acc)[Cfg<D, B>::DPL],
                                             float *probs, int lane) {
    using C = Cfg<D, B>;
    const int c = lane % C::LPT;   // 16-byte column of the row
    const int tr = lane / C::LPT;  // token within the row group

    // partial dot products over this lane's 8 dims, one per row group
    float sc[C::RG];
    const uint4 *K4 = reinterpret_cast<const uint4 *>(ktile);
#pragma unroll
    for (int r = 0; r < C::RG; ++r) sc[r] = dot8<E>(K4[(r * C::TPR + tr) * C::LPT + c], qh, qf);

    // Reduce-scatter across the LPT lanes of a token.  Each halving step swaps
    // half of a lane's remaining partial sums with the lane `o` apart and adds
    // the half it keeps, so after H steps a lane holds RG / 2^H rows summed
    // over 2^H lanes (rows base .. base + V - 1); the lane bits still unsummed
    // are finished with plain butterflies, after which those lanes hold equal
    // copies.  This needs RG - 1 + log2 shuffles instead of RG * log2(LPT).
    constexpr int H = ilog2(C::RG < C::LPT ? C::RG : C::LPT);
    constexpr int V = C::RG >> H;
    constexpr int DUP = C::LPT >> H;  // lanes holding the same rows
    int base = 0;
#pragma unroll
    for (int step = 0; step < H; ++step) {
        const int o = C::LPT >> (step + 1);
        const int half = (C::RG >> step) / 2;
        const bool upper = (c & o) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
            const float send = upper ? sc[j] : sc[j + half];
            const float keep = upper ? sc[j + half] : sc[j];
            sc[j] = keep + __shfl_xor_sync(kFull, send, o);
        }
        base += upper ? half : 0;
    }
#pragma unroll
    for (int o = DUP / 2; o >= 1; o >>= 1) {
#pragma unroll
        for (int j = 0; j < V; ++j) sc[j] += __shfl_xor_sync(kFull, sc[j], o);
    }

    // scale into the log2 domain, mask the tokens past the context
    float lane_max = -INFINITY;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int t = (base + j) * C::TPR + tr;
        sc[j] = (t < nvalid) ? sc[j] * scale_log2 : -INFINITY;
        lane_max = fmaxf(lane_max, sc[j]);
    }

    // Online softmax with a lazily raised reference.  The weights are taken
    // against run_max while no score of the tile exceeds it by more than
    // kLazyLog2 (so no weight exceeds 2^kLazyLog2); only a tile that does
    // reduces its maximum across the warp and rescales the state.  Every
    // weight and the sum share one reference, so the normalised result is
    // the same.  run_sum holds this lane's rows only; warp_row_sum adds the
    // lanes up once the unit is done.
    if (__any_sync(kFull, lane_max > run_max + kLazyLog2)) {
        float tile_max = lane_max;
#pragma unroll
        for (int o = 16; o >= DUP; o >>= 1)
            tile_max = fmaxf(tile_max, __shfl_xor_sync(kFull, tile_max, o));
        const float new_max = fmaxf(run_max, tile_max);
        const float alpha = exp2f(run_max - new_max);
        run_sum *= alpha;
#pragma unroll
        for (int i = 0; i < C::DPL; ++i) acc[i] *= alpha;
        run_max = new_max;
    }
#pragma unroll
    for (int j = 0; j < V; ++j) {
        sc[j] = exp2f(sc[j] - run_max);
        run_sum += sc[j];
    }

    // publish the B probabilities to the whole warp (one writer per token)
    if ((c & (DUP - 1)) == 0) {
#pragma unroll
        for (int j = 0; j < V; ++j) probs[(base + j) * C::TPR + tr] = sc[j];
    }
    __syncwarp();

    // p.V: this lane owns dims [lane * DPL, lane * DPL + DPL)
    const uint8_t *vrow = vtile + lane * C::DPL * 2;
    auto accumulate_row = [&](int t) {
        const float p = probs[t];
        const uint8_t *src = vrow + t * D * 2;
        if constexpr (C::DPL == 2) {
            const float2 v = E::pair(*reinterpret_cast<const uint32_t *>(src));
            acc[0] = fmaf(p, v.x, acc[0]);
            acc[1] = fmaf(p, v.y, acc[1]);
        } else if constexpr (C::DPL == 4) {
            const uint2 raw = *reinterpret_cast<const uint2 *>(src);
            const float2 v0 = E::pair(raw.x), v1 = E::pair(raw.y);
            acc[0] = fmaf(p, v0.x, acc[0]);
            acc[1] = fmaf(p, v0.y, acc[1]);
            acc[2] = fmaf(p, v1.x, acc[2]);
            acc[3] = fmaf(p, v1.y, acc[3]);
        } else {
            const uint4 raw = *reinterpret_cast<const uint4 *>(src);
            const float2 v0 = E::pair(raw.x), v1 = E::pair(raw.y), v2 = E::pair(raw.z),
                         v3 = E::pair(raw.w);
            acc[0] = fmaf(p, v0.x, acc[0]);
            acc[1] = fmaf(p, v0.y, acc[1]);
            acc[2] = fmaf(p, v1.x, acc[2]);
            acc[3] = fmaf(p, v1.y, acc[3]);
            acc[4] = fmaf(p, v2.x, acc[4]);
            acc[5] = fmaf(p, v2.y, acc[5]);
            acc[6] = fmaf(p, v3.x, acc[6]);
            acc[7] = fmaf(p, v3.y, acc[7]);
        }
    };
    if (nvalid == B) {
#pragma unroll
        for (int t = 0; t < B; ++t) accumulate_row(t);
    } else {
        // rows past the context may hold anything (even NaN): skip, never
        // multiply them by a zero weight
#pragma unroll
        for (int t = 0; t < B; ++t)
            if (t < nvalid) accumulate_row(t);
    }
    __syncwarp();  // probs is rewritten by the next tile
}

template <typename E, int DPL>
__device__ __forceinline__ void store_out(uint16_t *dst, const float (&v)[DPL], float inv) {
    uint16_t h[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) h[i] = E::round(v[i] * inv);
    if constexpr (DPL == 2) {
        *reinterpret_cast<uint32_t *>(dst) = *reinterpret_cast<const uint32_t *>(h);
    } else if constexpr (DPL == 4) {
        *reinterpret_cast<uint2 *>(dst) = *reinterpret_cast<const uint2 *>(h);
    } else {
        *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(h);
    }
}

template <int DPL>
__device__ __forceinline__ void load_f32(const float *src, float (&v)[DPL], bool bypass_l1) {
#pragma unroll
    for (int i = 0; i < DPL; i += 2) {
        const float2 x = bypass_l1 ? __ldcg(reinterpret_cast<const float2 *>(src + i))
                                   : *reinterpret_cast<const float2 *>(src + i);
        v[i] = x.x;
        v[i + 1] = x.y;
    }
}

template <int DPL>
__device__ __forceinline__ void store_f32(float *dst, const float (&v)[DPL]) {
#pragma unroll
    for (int i = 0; i < DPL; i += 2)
        *reinterpret_cast<float2 *>(dst + i) = make_float2(v[i], v[i + 1]);
}

// One warp: out[s, h] from partials begin .. end - 1 of (s, h) = sh in the
// workspace, (max, sum) pairs and unnormalised outputs written by other CTAs
// or launches (read through L2).
template <typename E, int D, int DPL>
__device__ __forceinline__ void combine_partials(const DecodeArgs &a, size_t sh, int begin,
                                                 int end, int lane) {
    const float2 *pml = reinterpret_cast<const float2 *>(a.part_ml) + sh * a.max_parts;
    const float *pacc = a.part_acc + sh * a.max_parts * D + lane * DPL;
    float GM = -INFINITY;
    for (int i = begin + lane; i < end; i += 32) GM = fmaxf(GM, __ldcg(pml + i).x);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) GM = fmaxf(GM, __shfl_xor_sync(kFull, GM, off));
    float GL = 0.f;
    float go[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) go[e] = 0.f;
#pragma unroll 4
    for (int i = begin; i < end; ++i) {
        const float2 ml = __ldcg(pml + i);
        float v[DPL];
        load_f32<DPL>(pacc + static_cast<size_t>(i) * D, v, true);
        const float f = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - GM);
        GL = fmaf(f, ml.y, GL);
#pragma unroll
        for (int e = 0; e < DPL; ++e) go[e] = fmaf(f, v[e], go[e]);
    }
    store_out<E, DPL>(a.out + sh * D + lane * DPL, go, GL > 0.f ? 1.f / GL : 0.f);
}

template <typename E, int D, int B, int HG>
__global__ void __launch_bounds__(Cfg<D, B, HG>::THREADS, Cfg<D, B, HG>::MIN_BLOCKS)
    decode_kernel(const DecodeArgs a) {
    using C = Cfg<D, B, HG>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BARS);
    uint64_t *empty = full + C::NS;
    uint64_t *desc_full = empty + C::NS;
    uint64_t *desc_empty = desc_full + C::ND;
    uint64_t *merge_full = desc_empty + C::ND;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_FLAGS);
    int *meta = reinterpret_cast<int *>(smem + C::OFF_META);
    int *stage_ok = reinterpret_cast<int *>(smem + C::OFF_STAGE_OK);
    // stage_tag[st] = index of the last tile the producer issued into stage st.
    // Different consumer warps use successive fills of one stage, so a warp may
    // reach a stage before the previous fill has landed; waiting for the tag
    // first guarantees that the fill before the awaited one has completed,
    // which keeps the mbarrier parity wait unambiguous.
    volatile uint32_t *stage_tag = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_STAGE_TAG);
    float *merge_acc = reinterpret_cast<float *>(smem + C::OFF_MERGE_ACC);
    float2 *merge_ml = reinterpret_cast<float2 *>(smem + C::OFF_MERGE_ML);
    uint16_t *desc_q = reinterpret_cast<uint16_t *>(smem + C::OFF_DESC_Q);
    const int S = a.num_seqs;
    const int H = a.num_heads;
    int *prefix = reinterpret_cast<int *>(smem + C::OFF_SEQ);  // [S + 1]
    int *ctx_of = prefix + S + 1;                              // [S]
    // Shared-prefix mode.  start_of[s]: the leading blocks of s that the
    // prefix kernel's partial (slot 0) may cover, provided s's table starts
    // like that of its group's first sequence (the producer checks this per
    // unit); this kernel covers the rest.
    const bool shared = a.group_start != nullptr;
    const int G = shared ? a.num_groups : 0;
    int *start_of = ctx_of + S;                                // [S]
    int *order = start_of + S;                                 // [S] work order: position -> s
    // Chunked mode (CS > 0): prefix[c] counts the partitions of the sequences
    // before chunk c (chunks of 2^CS sequences); no per-sequence array is
    // kept, and in shared-prefix mode the group arrays follow the prefix.
    const int CS = a.chunk_shift;
    const int nch = CS > 0 ? static_cast<int>((static_cast<long long>(S) + (1 << CS) - 1) >> CS) : 0;
    int *gstart = CS > 0 ? prefix + nch + 1 : order + S;      // [G + 1]
    int *gpre = gstart + G + 1;                                // [G]
    int *classes = gpre + G;                                   // [KEYS] (exact mode)
    uint2 *defer = reinterpret_cast<uint2 *>(
        smem + (C::OFF_SEQ + C::seq_ints(S, G, CS) * 4 + 7) / 8 * 8);   // [NC][DEFER]

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int TPU = a.tiles_per_unit;

    // ---- prologue: barriers, per-sequence context lengths and unit counts
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], HG);   // one arrival per warp reading the stage
            stage_tag[i] = 0xffffffffu;
        }
        for (int i = 0; i < C::ND; ++i) {
            mbar_init(&desc_full[i], 1);
            mbar_init(&desc_empty[i], C::NC);
            mbar_init(&merge_full[i], C::NC);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    // Everything above touched shared memory only; inputs may still be being
    // written by the previous kernel on the stream (e.g. reshape_and_cache).
    // After the shared-prefix kernel, which waited for them before letting
    // this one launch, only its partials are outstanding: the wait moves to
    // where they are read (and to the end).
    if (!shared) grid_dependency_wait();
    allow_dependents_to_launch();
    // the producer's first unit, grabbed now so that the grab's round trip
    // overlaps the prologue (every earlier call on the stream, which resets
    // the queue at its end, is complete here)
    uint32_t first_grab = 0;
    if (warp == C::NC && lane == 0) first_grab = atomicAdd(&a.counters[0], 1u);
    const int ctx_cap = a.max_blocks_per_seq * B;
    bool malformed = false;
    if (shared) {
        // one round of global loads: the group arrays and the lengths, each
        // thread's loads all issued before any is stored
        const int n_in = max(G + 1, CS == 0 ? S : 0);
        for (int i = threadIdx.x; i < n_in; i += blockDim.x) {
            const int gs_i = i <= G ? __ldg(a.group_start + i) : 0;
            const int gp_i = i < G ? __ldg(a.group_prefix_blocks + i) : 0;
            const int c_i = CS == 0 && i < S ? a.context_lens[i] : 0;
            if (i <= G) gstart[i] = gs_i;
            if (i < G) gpre[i] = gp_i;
            if (CS == 0 && i < S) ctx_of[i] = c_i;
        }
        __syncthreads();
        // the group arrays: non-decreasing within [0, S], P_g within the table
        bool bad = false;
        for (int g = threadIdx.x; g <= G; g += blockDim.x) {
            const int lo = gstart[g];
            bad = bad || lo < 0 || lo > S;
            if (g < G) bad = bad || gstart[g + 1] < lo || gpre[g] < 0 || gpre[g] > a.max_blocks_per_seq;
        }
        malformed = __syncthreads_or(bad) != 0;
        if (malformed && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.err, PA_DEVERR_PREFIX);
    }
    // partitions of a remainder of nb blocks; an empty context still takes
    // one unit, which writes its zero output row
    auto parts_of = [&](int nb) { return nb == 0 ? 1 : (nb + TPU - 1) / TPU; };
    // Shared-prefix mode: the leading blocks of s that the prefix kernel's
    // partial (slot 0) may cover, from its group, given its context length as
    // passed (the producer still checks s's table against the group's first
    // sequence per unit); 0 outside every group.
    auto member_first = [&](int s, int c_in, bool report) {
        int first = 0;
        if (!malformed && G > 0 && gstart[0] <= s) {
            int lo = 0, hi = G - 1;   // the last group starting at or before s
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (gstart[mid] <= s) lo = mid; else hi = mid - 1;
            }
            const int pb = gpre[lo];
            if (s < gstart[lo + 1] && pb > 0) {
                // rows the prefix kernel covers, whose context holds the prefix
                if (c_in >= pb * B && c_in <= ctx_cap && s - gstart[lo] < a.rows_cap)
                    first = pb;
                else if (report)
                    atomicOr(a.err, PA_DEVERR_PREFIX);
            }
        }
        return first;
    };
    if (CS > 0) {   // one warp per chunk: its sequences' partition counts, summed
        const int nwarps = static_cast<int>(blockDim.x / 32);
        for (int c = warp; c < nch; c += nwarps) {
            int cnt = 0;
            for (int i = lane; i < (1 << CS); i += 32) {
                const int s = (c << CS) + i;
                if (s >= S) break;
                const int x_in = a.context_lens[s];
                int x = x_in;
                if (x < 0 || x > ctx_cap) {
                    atomicOr(a.err, PA_DEVERR_CONTEXT);
                    x = x < 0 ? 0 : ctx_cap;
                }
                const int first = shared ? member_first(s, x_in, blockIdx.x == 0) : 0;
                cnt += parts_of((x + B - 1) / B - first);
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) cnt += __shfl_xor_sync(kFull, cnt, off);
            if (lane == 0) prefix[c + 1] = cnt;
        }
    }
    for (int s = threadIdx.x; s < (CS > 0 ? 0 : S); s += blockDim.x) {
        const int c_in = shared ? ctx_of[s] : a.context_lens[s];
        int c = c_in;
        if (c < 0 || c > ctx_cap) {
            atomicOr(a.err, PA_DEVERR_CONTEXT);
            c = c < 0 ? 0 : ctx_cap;
        }
        const int nblk = (c + B - 1) / B;
        int first = 0;
        if (shared) {
            first = member_first(s, c_in, blockIdx.x == 0);
            start_of[s] = first;
        }
        const int rest = nblk - first;
        ctx_of[s] = c;
        if (!shared) prefix[s + 1] = rest == 0 ? 1 : (rest + TPU - 1) / TPU;  // partitions of s
    }
    __syncthreads();
    // Work order, shared-prefix mode: longest first unit first (a stable
    // counting sort, descending, over KEYS length classes), so that the queue
    // ends on short units.  Plain decode keeps sequence order (its concurrent
    // CTAs then share the L2 lines of common blocks); here the common blocks
    // are the prefix kernel's.  Every CTA derives the same order: class sizes,
    // then placement in sequence order within a class.
    static_assert(C::KEYS == 32, "one length class per lane");
    auto key_of = [&](int s) {
        const int rest = (ctx_of[s] + B - 1) / B - start_of[s];
        return min(rest, TPU) * (C::KEYS - 1) / TPU;
    };
    // All warps sort, one chunk of 32 sequences each, with per-chunk class
    // sizes kept in the merge buffer (unused until the first unit ends); a
    // batch whose sizes do not fit there is sorted by one warp.
    const int nch32 = (S + 31) / 32;
    const bool wide_sort = shared && CS == 0 && nch32 * C::KEYS <= C::ND * C::NC * D;
    if (wide_sort) {
        int *first_of = reinterpret_cast<int *>(merge_acc);   // [nch32][KEYS]
        const int nwarps = static_cast<int>(blockDim.x / 32);
        for (int c = warp; c < nch32; c += nwarps) {   // the classes' sizes in chunk c
            const int s = c * 32 + lane;
            first_of[c * C::KEYS + lane] = 0;
            __syncwarp();
            const unsigned active = __ballot_sync(kFull, s < S);
            if (s < S) {
                const int k = key_of(s);
                const unsigned peers = __match_any_sync(active, k);
                if (lane == __ffs(peers) - 1) first_of[c * C::KEYS + k] = __popc(peers);
            }
            __syncwarp();
        }
        __syncthreads();
        if (warp == 0) {
            // first place of (class k, chunk c): the classes longer than k,
            // then class k in the chunks before c; lane 0 holds the longest
            const int k = C::KEYS - 1 - lane;
            int total = 0;
            for (int c = 0; c < nch32; ++c) total += first_of[c * C::KEYS + k];
            int v = total;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(kFull, v, off);
                if (lane >= off) v += y;
            }
            int place = v - total;
            for (int c = 0; c < nch32; ++c) {
                const int n = first_of[c * C::KEYS + k];
                first_of[c * C::KEYS + k] = place;
                place += n;
            }
        }
        __syncthreads();
        for (int c = warp; c < nch32; c += nwarps) {   // placement
            const int s = c * 32 + lane;
            const unsigned active = __ballot_sync(kFull, s < S);
            if (s < S) {
                const int k = key_of(s);
                const unsigned peers = __match_any_sync(active, k);
                order[first_of[c * C::KEYS + k] + __popc(peers & ((1u << lane) - 1u))] = s;
            }
        }
        __syncthreads();
    } else if (shared && CS == 0 && warp == C::NC) {
        classes[lane] = 0;
        __syncwarp();
        for (int s = lane; s < S; s += 32) atomicAdd(&classes[key_of(s)], 1);
        __syncwarp();
        {   // first place of class k: the sizes of the classes above it
            const int k = C::KEYS - 1 - lane;
            const int n = classes[k];
            int v = n;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(kFull, v, off);
                if (lane >= off) v += y;
            }
            __syncwarp();
            classes[k] = v - n;
        }
        __syncwarp();
        for (int base = 0; base < S; base += 32) {
            const int s = base + lane;
            const unsigned active = __ballot_sync(kFull, s < S);
            if (s < S) {
                const int k = key_of(s);
                const unsigned peers = __match_any_sync(active, k);
                order[classes[k] + __popc(peers & ((1u << lane) - 1u))] = s;
                __syncwarp(active);
                if (lane == __ffs(peers) - 1) classes[k] += __popc(peers);
            }
            __syncwarp();
        }
    }
    // entries of the prefix: one per sequence, or one per chunk
    const int NE = CS > 0 ? nch : S;
    if (warp == C::NC) {  // exclusive prefix over the order of partition counts
        int running = 0;
        for (int base = 0; base < NE; base += 32) {
            const int s = base + lane;
            int v = 0;
            if (s < NE && shared && CS == 0) {   // partitions of the sequence in place s
                const int r = order[s];
                const int rest = (ctx_of[r] + B - 1) / B - start_of[r];
                v = rest == 0 ? 1 : (rest + TPU - 1) / TPU;
            } else if (s < NE) {
                v = prefix[s + 1];
            }
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(kFull, v, off);
                if (lane >= off) v += y;
            }
            if (s < NE) prefix[s + 1] = running + v;
            running += __shfl_sync(kFull, v, 31);
        }
        if (lane == 0) prefix[0] = 0;
    }
    __syncthreads();

    // units: (entry of the order, partition, group of HG heads), heads fastest
    const int HGR = H / HG;   // head groups (the host launches HG > 1 only if HG divides H)
    const uint32_t num_units = static_cast<uint32_t>(prefix[NE]) * static_cast<uint32_t>(HGR);

    if (warp == C::NC) {
        // ================= producer warp =================
        uint32_t kq = 0;  // tiles issued
        uint32_t dq = 0;  // unit descriptors issued
        bool ok = true;
        uint32_t pending = first_grab;
        while (true) {
            const uint32_t u = __shfl_sync(kFull, pending, 0);
            if (u >= num_units) break;
            if (lane == 0) pending = atomicAdd(&a.counters[0], 1u);  // prefetch the next grab
            const int g = static_cast<int>(u / HGR);
            const int h = static_cast<int>(u - static_cast<uint32_t>(g) * HGR) * HG;   // first head
            int lo = 0, hi = NE - 1;  // entry i with prefix[i] <= g < prefix[i + 1]
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (prefix[mid] <= g) lo = mid; else hi = mid - 1;
            }
            int s, p, np, ctx, first = 0;
            if (CS == 0) {
                s = shared ? order[lo] : lo;
                p = g - prefix[lo];
                np = prefix[lo + 1] - prefix[lo];
                ctx = ctx_of[s];
                if (shared) first = start_of[s];
            } else {
                // chunk lo: each lane takes 2^(CS-5) consecutive sequences,
                // a warp scan of their partition counts finds the lane whose
                // range holds partition `rem` of the chunk, and that lane
                // walks its sequences to the one that holds it
                const int rem = g - prefix[lo];
                const int per_lane = 1 << (CS - 5);
                const int sb = (lo << CS) + lane * per_lane;
                // partitions of sequence q (and its prefix blocks, shared mode)
                auto seq_parts = [&](int q, int &c, int &f) {
                    const int x_in = __ldg(a.context_lens + q);
                    c = min(max(x_in, 0), ctx_cap);
                    f = shared ? member_first(q, x_in, false) : 0;
                    return parts_of((c + B - 1) / B - f);
                };
                int tot = 0;
                for (int i = 0; i < per_lane; ++i) {
                    if (sb + i >= S) break;
                    int c, f;
                    tot += seq_parts(sb + i, c, f);
                }
                int inc = tot;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(kFull, inc, off);
                    if (lane >= off) inc += y;
                }
                const unsigned hit = __ballot_sync(kFull, inc > rem);
                if (hit == 0) {   // only if the lengths changed during the launch
                    if (lane == 0) atomicOr(a.err, PA_DEVERR_CONTEXT);
                    continue;
                }
                const int L = __ffs(hit) - 1;
                int fs = -1, fp = 0, fnp = 1, fctx = 0, ffirst = 0;
                if (lane == L) {
                    int r = rem - (inc - tot);
                    for (int i = 0; i < per_lane && sb + i < S; ++i) {
                        int c, f;
                        const int n = seq_parts(sb + i, c, f);
                        if (r < n) { fs = sb + i; fp = r; fnp = n; fctx = c; ffirst = f; break; }
                        r -= n;
                    }
                }
                s = __shfl_sync(kFull, fs, L);
                p = __shfl_sync(kFull, fp, L);
                np = __shfl_sync(kFull, fnp, L);
                ctx = __shfl_sync(kFull, fctx, L);
                first = __shfl_sync(kFull, ffirst, L);
                if (s < 0) {
                    if (lane == 0) atomicOr(a.err, PA_DEVERR_CONTEXT);
                    continue;
                }
            }
            const int nblk = (ctx + B - 1) / B;
            bool pre = first > 0;
            int leader = s;
            if (pre) {   // the group's first sequence: the last group start at or before s
                int glo = 0, ghi = G - 1;
                while (glo < ghi) {
                    const int mid = (glo + ghi + 1) >> 1;
                    if (gstart[mid] <= s) glo = mid; else ghi = mid - 1;
                }
                leader = gstart[glo];
            }
            const int32_t *srow = a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq;
            // the first table slice, loaded as it is if the prefix partial
            // applies, together with the check below
            int t0 = (pre || p > 0) ? first + p * TPU : 0;
            int nt = max(0, min(nblk, first + (p + 1) * TPU) - t0);
            int phys_first = lane < min(nt, 32) ? __ldg(srow + t0 + lane) : 0;
            if (pre && leader != s) {
                // the prefix partial is s's only if s's first blocks are its
                // group's; otherwise the first partition takes them on
                const int32_t *lead =
                    a.block_tables + static_cast<size_t>(leader) * a.max_blocks_per_seq;
                bool same = true;
                for (int b = lane; b < first; b += 32) same = same && __ldg(srow + b) == __ldg(lead + b);
                pre = __all_sync(kFull, same);
                if (!pre && lane == 0 && h == 0 && p == 0) atomicOr(a.err, PA_DEVERR_PREFIX);
                if (!pre && p == 0) {   // the first partition starts at block 0 after all
                    t0 = 0;
                    nt = max(0, min(nblk, first + TPU));
                    phys_first = lane < min(nt, 32) ? __ldg(srow + lane) : 0;
                }
            }

            const int slot = static_cast<int>(dq % C::ND);
            bool w_ok = mbar_wait(&desc_empty[slot], ((dq / C::ND) & 1u) ^ 1u, abort_flag, a.err);
            if (!__all_sync(kFull, w_ok)) { ok = false; break; }
            if (lane == 0) {
                int *m = meta + slot * C::META_INTS;
                m[0] = s; m[1] = h; m[2] = p; m[3] = nt; m[4] = ctx; m[5] = np;
                m[6] = t0; m[7] = pre ? 1 : 0;
                // the queries of heads h .. h + HG - 1: one contiguous run
                mbar_arrive_expect_tx(&desc_full[slot], HG * D * 2);
                bulk_copy_g2s(desc_q + slot * HG * D, a.q + (static_cast<size_t>(s) * H + h) * D,
                              HG * D * 2, &desc_full[slot]);
            }
            ++dq;

            const int32_t *row = srow + t0;
            for (int j0 = 0; j0 < nt && ok; j0 += 32) {
                const int n = min(32, nt - j0);
                const int phys_lane =
                    j0 == 0 ? phys_first : (lane < n ? __ldg(row + j0 + lane) : 0);
                if constexpr (C::R == 1) {
                    for (int jj = 0; jj < n; ++jj) {
                        const int phys = __shfl_sync(kFull, phys_lane, jj);
                        const int st = static_cast<int>(kq % C::NS);
                        w_ok = mbar_wait(&empty[st], ((kq / C::NS) & 1u) ^ 1u, abort_flag, a.err);
                        if (!__all_sync(kFull, w_ok)) { ok = false; break; }
                        if (lane == 0) {
                            const bool in_pool = static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks);
                            stage_ok[st] = in_pool ? 1 : 0;
                            stage_tag[st] = kq;
                            if (in_pool) {
                                // heads h .. h + HG - 1 of the block: HG adjacent tiles
                                const size_t off = (static_cast<size_t>(phys) * H + h) * (B * D);
                                uint8_t *dst = smem + C::OFF_STAGES + st * C::STAGE_BYTES;
                                mbar_arrive_expect_tx(&full[st], 2 * HG * C::TILE_BYTES);
                                bulk_copy_g2s(dst, a.k_cache + off, HG * C::TILE_BYTES, &full[st]);
                                bulk_copy_g2s(dst + HG * C::TILE_BYTES, a.v_cache + off,
                                              HG * C::TILE_BYTES, &full[st]);
                            } else {
                                atomicOr(a.err, PA_DEVERR_TABLE);
                                mbar_arrive(&full[st]);
                            }
                        }
                        ++kq;
                    }
                } else {
                    for (int jj = 0; jj < n; jj += C::R) {   // one stage: blocks jj .. jj + R - 1
                        int phys[C::R];
#pragma unroll
                        for (int r = 0; r < C::R; ++r) phys[r] = __shfl_sync(kFull, phys_lane, jj + r);
                        const int st = static_cast<int>(kq % C::NS);
                        w_ok = mbar_wait(&empty[st], ((kq / C::NS) & 1u) ^ 1u, abort_flag, a.err);
                        if (!__all_sync(kFull, w_ok)) { ok = false; break; }
                        if (lane == 0) {
                            // bit r: block jj + r exists and is in the pool (copied)
                            uint32_t mask = 0;
#pragma unroll
                            for (int r = 0; r < C::R; ++r) {
                                if (jj + r >= n) break;
                                if (static_cast<unsigned>(phys[r]) < static_cast<unsigned>(a.num_blocks))
                                    mask |= 1u << r;
                                else
                                    atomicOr(a.err, PA_DEVERR_TABLE);
                            }
                            stage_ok[st] = static_cast<int>(mask);
                            stage_tag[st] = kq;
                            if (mask) {
                                uint8_t *dst = smem + C::OFF_STAGES + st * C::STAGE_BYTES;
                                mbar_arrive_expect_tx(&full[st], 2 * C::TILE_BYTES * __popc(mask));
#pragma unroll
                                for (int r = 0; r < C::R; ++r) {
                                    if (!(mask & (1u << r))) continue;
                                    const size_t off = (static_cast<size_t>(phys[r]) * H + h) * (B * D);
                                    bulk_copy_g2s(dst + r * C::TILE_BYTES, a.k_cache + off, C::TILE_BYTES,
                                                  &full[st]);
                                    bulk_copy_g2s(dst + (C::R + r) * C::TILE_BYTES, a.v_cache + off,
                                                  C::TILE_BYTES, &full[st]);
                                }
                            } else {
                                mbar_arrive(&full[st]);
                            }
                        }
                        ++kq;
                    }
                }
            }
            if (!ok) break;
        }
        if (ok) {  // tell the consumers there is no more work
            const int slot = static_cast<int>(dq % C::ND);
            const bool w_ok = mbar_wait(&desc_empty[slot], ((dq / C::ND) & 1u) ^ 1u, abort_flag, a.err);
            if (__all_sync(kFull, w_ok)) {
                if (lane == 0) {
                    meta[slot * C::META_INTS] = -1;
                    mbar_arrive(&desc_full[slot]);
                }
                ++dq;
            } else {
                ok = false;
            }
        }
        if (lane == 0) {
            if (ok) {
                // The last CTA to finish resets the work queue for the next call.
                __threadfence();
                const uint32_t done = atomicAdd(&a.counters[1], 1u);
                if (done == gridDim.x - 1) {
                    __threadfence();
                    atomicExch(&a.counters[0], 0u);
                    atomicExch(&a.counters[1], 0u);
                }
            } else {
                // Let every copy already issued land before the CTA exits.
                for (uint32_t k = kq > C::NS ? kq - C::NS : 0; k < kq; ++k)
                    mbar_wait_drain(&full[k % C::NS], (k / C::NS) & 1u);
                for (uint32_t d = dq > C::ND ? dq - C::ND : 0; d < dq; ++d)
                    mbar_wait_drain(&desc_full[d % C::ND], (d / C::ND) & 1u);
            }
        }
        // this grid must not complete before the shared-prefix kernel it
        // reads from (a later kernel that waits for this one relies on it)
        if (shared) grid_dependency_wait();
        return;
    }

    // ================= consumer warps =================
    const int w = warp;
    float *probs = reinterpret_cast<float *>(smem + C::OFF_PROBS) + w * B;
    uint32_t kq = 0, dq = 0;
    int ndefer = 0;   // this warp's deferred prefix merges
    while (true) {
        const int slot = static_cast<int>(dq % C::ND);
        bool w_ok = mbar_wait(&desc_full[slot], (dq / C::ND) & 1u, abort_flag, a.err);
        if (!__all_sync(kFull, w_ok)) return;
        const int *m = meta + slot * C::META_INTS;
        const int s = m[0];
        if (s < 0) break;
        // this warp's head: gw-th of the unit's HG heads; its blocks are
        // every (NC / HG)-th one from w / HG
        const int gw = w % HG;
        const int h = m[1] + gw, p = m[2], nt = m[3], ctx = m[4], np = m[5], t0 = m[6];
        // with a shared prefix, slot 0 of (s, h) holds the prefix kernel's partial
        const int pre = m[7];

        float qf[8];
        const uint4 qraw = *reinterpret_cast<const uint4 *>(desc_q + (slot * HG + gw) * D +
                                                            (lane % C::LPT) * 8);
        {
            const float2 q0 = E::pair(qraw.x), q1 = E::pair(qraw.y), q2 = E::pair(qraw.z),
                         q3 = E::pair(qraw.w);
            qf[0] = q0.x; qf[1] = q0.y; qf[2] = q1.x; qf[3] = q1.y;
            qf[4] = q2.x; qf[5] = q2.y; qf[6] = q3.x; qf[7] = q3.y;
        }
        float run_max = -INFINITY, run_sum = 0.f;
        float acc[C::DPL];
#pragma unroll
        for (int i = 0; i < C::DPL; ++i) acc[i] = 0.f;

        if constexpr (C::R == 1) {
            for (int j = w / HG; j < nt; j += C::NC / HG) {
                const uint32_t k = kq + j;
                const int st = static_cast<int>(k % C::NS);
                w_ok = wait_value(&stage_tag[st], k, abort_flag, a.err) &&
                       mbar_wait(&full[st], (k / C::NS) & 1u, abort_flag, a.err);
                if (!__all_sync(kFull, w_ok)) return;
                if (stage_ok[st]) {
                    const int tok0 = (t0 + j) * B;
                    const int nvalid = min(B, ctx - tok0);
                    const uint8_t *ktile =
                        smem + C::OFF_STAGES + st * C::STAGE_BYTES + gw * C::TILE_BYTES;
                    consume_tile<E, D, B>(ktile, ktile + HG * C::TILE_BYTES, qraw, qf,
                                          a.scale_log2, nvalid, run_max, run_sum, acc, probs, lane);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
            kq += nt;
        } else {
            const int nstages = (nt + C::R - 1) / C::R;   // ring stages of this unit
            for (int j = w; j < nstages; j += C::NC) {
                const uint32_t k = kq + j;
                const int st = static_cast<int>(k % C::NS);
                w_ok = wait_value(&stage_tag[st], k, abort_flag, a.err) &&
                       mbar_wait(&full[st], (k / C::NS) & 1u, abort_flag, a.err);
                if (!__all_sync(kFull, w_ok)) return;
                const uint32_t mask = static_cast<uint32_t>(stage_ok[st]);
                const uint8_t *stage = smem + C::OFF_STAGES + st * C::STAGE_BYTES;
#pragma unroll
                for (int r = 0; r < C::R; ++r) {
                    if (!(mask & (1u << r))) continue;   // past the unit, or outside the pool
                    const int tok0 = (t0 + j * C::R + r) * B;
                    const int nvalid = min(B, ctx - tok0);
                    consume_tile<E, D, B>(stage + r * C::TILE_BYTES,
                                          stage + (C::R + r) * C::TILE_BYTES, qraw, qf,
                                          a.scale_log2, nvalid, run_max, run_sum, acc, probs, lane);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
            kq += nstages;
        }

        // hand this warp's state to the unit's owner warp
        store_f32<C::DPL>(merge_acc + (slot * C::NC + w) * D + lane * C::DPL, acc);
        run_sum = warp_row_sum<D, B>(run_sum);
        if (lane == 0) merge_ml[slot * C::NC + w] = make_float2(run_max, run_sum);
        __syncwarp();
        if (lane == 0) mbar_arrive(&merge_full[slot]);

        // one owner per head of the unit: it merges the NC / HG warps that
        // read that head (warps gw, gw + HG, ...), rotating with the unit
        constexpr int WPH = C::NC / HG;   // warps per head
        const int owner_rank = static_cast<int>(dq % WPH);
        if (w / HG == owner_rank) {
            w_ok = mbar_wait(&merge_full[slot], (dq / C::ND) & 1u, abort_flag, a.err);
            if (!__all_sync(kFull, w_ok)) return;
            float M = -INFINITY;
#pragma unroll
            for (int k = 0; k < WPH; ++k) M = fmaxf(M, merge_ml[slot * C::NC + k * HG + gw].x);
            float L = 0.f;
            float o[C::DPL];
#pragma unroll
            for (int i = 0; i < C::DPL; ++i) o[i] = 0.f;
#pragma unroll
            for (int k = 0; k < WPH; ++k) {
                const int i = k * HG + gw;
                const float2 ml = merge_ml[slot * C::NC + i];
                if (ml.x == -INFINITY) continue;  // a warp with no tile of this unit
                const float f = exp2f(ml.x - M);
                L = fmaf(f, ml.y, L);
                float v[C::DPL];
                load_f32<C::DPL>(merge_acc + (slot * C::NC + i) * D + lane * C::DPL, v, false);
#pragma unroll
                for (int e = 0; e < C::DPL; ++e) o[e] = fmaf(f, v[e], o[e]);
            }
            const size_t sh = static_cast<size_t>(s) * H + h;
            if (np == 1 && !pre) {
                store_out<E, C::DPL>(a.out + sh * D + lane * C::DPL, o, L > 0.f ? 1.f / L : 0.f);
            } else {
                // a partial.  In shared-prefix mode slot 0 is the prefix
                // kernel's alone (it may be writing it now, for any row of a
                // group, even one this kernel decodes in full).
                const int base = shared ? 1 : 0;
                const size_t pidx = sh * a.max_parts + p + base;
                if (lane == 0) reinterpret_cast<float2 *>(a.part_ml)[pidx] = make_float2(M, L);
                store_f32<C::DPL>(a.part_acc + pidx * D + lane * C::DPL, o);
                bool last = true;
                if (np > 1) {
                    __threadfence();
                    __syncwarp();
                    uint32_t ticket = 0;
                    if (lane == 0) ticket = atomicAdd(&a.counters[2 + sh], 1u);
                    ticket = __shfl_sync(kFull, ticket, 0);
                    last = ticket == static_cast<uint32_t>(np - 1);
                    if (last) {
                        __threadfence();
                        if (lane == 0) atomicExch(&a.counters[2 + sh], 0u);  // ready for the next call
                    }
                }
                if (last) {
                    // the last partition of (s, h) combines all partials.  The
                    // prefix partial comes from the previous launch: that
                    // combine waits until this warp has no unit left, when the
                    // prefix kernel has long finished.
                    const int end = np + base;
                    if (!pre) {
                        combine_partials<E, D, C::DPL>(a, sh, base, end, lane);
                    } else if (ndefer < C::DEFER) {
                        if (lane == 0)
                            defer[w * C::DEFER + ndefer] =
                                make_uint2(static_cast<uint32_t>(sh), static_cast<uint32_t>(end));
                        ++ndefer;
                    } else {
                        grid_dependency_wait();
                        combine_partials<E, D, C::DPL>(a, sh, 0, end, lane);
                    }
                }
            }
            __syncwarp();
        }
        if (lane == 0) mbar_arrive(&desc_empty[slot]);
        ++dq;
    }
    if (ndefer > 0) {   // the deferred prefix merges
        grid_dependency_wait();
        __syncwarp();
        for (int i = 0; i < ndefer; ++i) {
            const uint2 e = defer[w * C::DEFER + i];
            combine_partials<E, D, C::DPL>(a, e.x, 0, static_cast<int>(e.y), lane);
        }
    }
}

struct Variant {
    int dtype, head_dim, block_size, hg;
    const void *kernel;
    int threads;
    size_t (*smem_bytes)(int, int, int);
};

template <typename E, int D, int B, int HG>
Variant make_variant() {
    return Variant{E::kBf16 ? PA_DTYPE_BF16 : PA_DTYPE_F16, D, B, HG,
                   reinterpret_cast<const void *>(&decode_kernel<E, D, B, HG>),
                   Cfg<D, B, HG>::THREADS, &Cfg<D, B, HG>::smem_bytes};
}

// Two kernels per shape: one head per unit, and the preferred head group
// (the same kernel again when that is one head).
template <typename E, int D, int B>
void add_shape(Variant *v) {
    v[0] = make_variant<E, D, B, 1>();
    v[1] = make_variant<E, D, B, preferred_heads(D, B)>();
}

template <typename E>
void add_variants(Variant *v) {
    add_shape<E, 64, 8>(v + 0);   add_shape<E, 64, 16>(v + 2);   add_shape<E, 64, 32>(v + 4);
    add_shape<E, 128, 8>(v + 6);  add_shape<E, 128, 16>(v + 8);  add_shape<E, 128, 32>(v + 10);
    add_shape<E, 256, 8>(v + 12); add_shape<E, 256, 16>(v + 14); add_shape<E, 256, 32>(v + 16);
}

constexpr int kNumVariants = 36;

const Variant *variants() {
    static Variant table[kNumVariants];
    static bool filled = [] {
        add_variants<F16>(table);
        add_variants<BF16>(table + 18);
        return true;
    }();
    (void)filled;
    return table;
}

// The kernel for a shape: the preferred head group when it divides the head
// count, else one head per unit.
const Variant *find_variant(int dtype, int head_dim, int block_size, int num_heads) {
    const Variant *t = variants();
    for (int i = 0; i < kNumVariants; i += 2)
        if (t[i].dtype == dtype && t[i].head_dim == head_dim && t[i].block_size == block_size)
            return (num_heads > 0 && num_heads % t[i + 1].hg == 0) ? &t[i + 1] : &t[i];
    return nullptr;
}

// Largest dynamic shared memory a CTA may opt into, per device (set by
// prepare_decode_kernels before any launch on that device).
constexpr int kMaxDevices = 64;
int g_max_dynamic_smem[kMaxDevices] = {0};

// Launch shape of one decode: the sequence-state layout, its shared memory
// and the CTAs per SM it allows.  The last shape computed per device and
// variant is kept, so repeated calls with the same batch (and groups) query
// the occupancy calculator once.
struct Shape {
    int num_seqs = -1, num_groups = -2, chunk_shift = 0, per_sm = 0;
    size_t smem = 0;
};
Shape g_last_shape[kMaxDevices][kNumVariants];
std::mutex g_shape_mutex;

cudaError_t occupancy(const Variant *v, size_t smem, int *per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, v->kernel, v->threads, smem);
}

// Per-sequence state (chunk_shift 0) while it leaves the CTAs per SM at what
// the fixed footprint (and the group arrays) alone allow; otherwise the
// smallest chunk of 2^c sequences (c >= 5) that does, or one chunk for the
// whole batch.  num_groups < 0: plain mode.
cudaError_t decode_shape(const Variant *v, int device, int num_seqs, int num_groups, Shape *out) {
    const int vi = static_cast<int>(v - variants());
    {
        std::lock_guard<std::mutex> lock(g_shape_mutex);
        const Shape &c = g_last_shape[device][vi];
        if (c.num_seqs == num_seqs && c.num_groups == num_groups) {
            *out = c;
            return cudaSuccess;
        }
    }
    int best = 0;
    const size_t least = v->smem_bytes(1, num_groups, 30);
    if (least > static_cast<size_t>(g_max_dynamic_smem[device])) return cudaErrorInvalidConfiguration;
    cudaError_t e = occupancy(v, least, &best);
    if (e != cudaSuccess) return e;
    Shape sh;
    sh.num_seqs = num_seqs;
    sh.num_groups = num_groups;
    for (int cs = 0;; cs = cs == 0 ? 5 : cs + 1) {
        sh.chunk_shift = cs;
        sh.smem = v->smem_bytes(num_seqs, num_groups, cs);
        const bool one_chunk = cs >= 30 || (cs > 0 && (num_seqs >> cs) == 0);
        if (sh.smem > static_cast<size_t>(g_max_dynamic_smem[device])) {
            if (one_chunk) return cudaErrorInvalidConfiguration;
            continue;
        }
        e = occupancy(v, sh.smem, &sh.per_sm);
        if (e != cudaSuccess) return e;
        if (sh.per_sm >= best || one_chunk) break;
    }
    if (sh.per_sm < 1) return cudaErrorInvalidConfiguration;
    std::lock_guard<std::mutex> lock(g_shape_mutex);
    g_last_shape[device][vi] = sh;
    *out = sh;
    return cudaSuccess;
}

}  // namespace

bool decode_variant_supported(int dtype, int head_dim, int block_size) {
    return find_variant(dtype, head_dim, block_size, 1) != nullptr;
}

cudaError_t prepare_decode_kernels(int device) {
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess) return e;
    const Variant *t = variants();
    for (int i = 0; i < kNumVariants; ++i) {
        e = cudaFuncSetAttribute(t[i].kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        if (e != cudaSuccess) return e;
    }
    g_max_dynamic_smem[device] = optin;
    return cudaSuccess;
}

bool decode_fits(int dtype, int head_dim, int block_size, int num_heads, int num_seqs,
                 int num_groups) {
    const Variant *v = find_variant(dtype, head_dim, block_size, num_heads);
    int device = 0;
    if (!v || cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
        return false;
    // some layout fits unless the group arrays alone exceed the shared memory
    Shape sh;
    return decode_shape(v, device, num_seqs, num_groups, &sh) == cudaSuccess;
}

cudaError_t launch_decode(const DecodeArgs &args, int dtype, int head_dim, int block_size,
                          int num_sms, cudaStream_t stream) {
    const Variant *v = find_variant(dtype, head_dim, block_size, args.num_heads);
    if (!v) return cudaErrorInvalidValue;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    DecodeArgs la = args;
    Shape sh;
    e = decode_shape(v, device, args.num_seqs, args.group_start != nullptr ? args.num_groups : -1,
                     &sh);
    if (e != cudaSuccess) return e;
    la.chunk_shift = sh.chunk_shift;
    const size_t smem = sh.smem;
    const int per_sm = sh.per_sm;
    // Persistent grid; never more CTAs than the most work units there can be.
    const long long max_units = static_cast<long long>(args.num_seqs) * args.num_heads * args.max_parts;
    long long grid = static_cast<long long>(per_sm) * num_sms;
    if (grid > max_units) grid = max_units;
    if (grid < 1) grid = 1;
    void *params[] = {&la};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(v->threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, v->kernel, params);
}

}  // namespace pa
