// pa_blocks.cu -- table-driven copies of whole KV blocks between two pools.
//
// The pages describe two block moves of the KV cache manager: blocks that
// several requests share through reference counts, so a request that must
// change one gets its own copy; and blocks swapped out to CPU memory when GPU
// memory runs short, then swapped back in (doramagic.ai vLLM manual,
// "内存管理策略": 层级淘汰 to CPU memory; "BlockPool 组件": GPU/CPU block
// state tracking and reference counts; "共享机制").  Both are one operation:
// copy block src -> block dst, K and V, every head, between a source pool and
// a destination pool, each either device memory or host memory the GPU can
// address (pinned or registered).
//
// A pure copy, bound by the slower of the two memories.  A pair's K block then
// V block (H * B * D * 2 bytes each, contiguous in the [N, H, B, D] layout)
// are split into segments of 4 x 256 16-byte chunks; a CTA copies one
// segment of a pair, its threads taking consecutive chunks, so every load and
// store is coalesced and each thread has four loads in flight.  The source
// and destination pools may be the same memory (copy-on-write), so the
// pointers are not declared non-aliasing.  Block ids are checked against both
// pools; an id out of range skips that pair and sets PA_DEVERR_TABLE.
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // 16-byte chunks per thread per segment
constexpr int kSegmentChunks = kThreads * kUnroll;

// grid.x: segments of one pair's K-then-V chunks; grid.y: pairs (strided).
__global__ void __launch_bounds__(kThreads) copy_blocks_kernel(
    const uint4 *src_k, const uint4 *src_v, uint4 *dst_k, uint4 *dst_v,
    const int32_t *__restrict__ block_pairs, int32_t num_pairs,
    int32_t chunks_per_block, int32_t src_num_blocks, int32_t dst_num_blocks,
    unsigned int *err) {
    allow_dependents_to_launch();
    grid_dependency_wait();
    const int32_t first = blockIdx.x * kSegmentChunks + threadIdx.x;
    for (int32_t pair = blockIdx.y; pair < num_pairs; pair += gridDim.y) {
        const int32_t src = __ldg(block_pairs + 2 * static_cast<size_t>(pair));
        const int32_t dst = __ldg(block_pairs + 2 * static_cast<size_t>(pair) + 1);
        if (static_cast<unsigned>(src) >= static_cast<unsigned>(src_num_blocks) ||
            static_cast<unsigned>(dst) >= static_cast<unsigned>(dst_num_blocks)) {
            if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err, PA_DEVERR_TABLE);
            continue;
        }
        const size_t from = static_cast<size_t>(src) * chunks_per_block;
        const size_t to = static_cast<size_t>(dst) * chunks_per_block;
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {  // all loads first, then all stores
            const int32_t c = first + u * kThreads;
            if (c < 2 * chunks_per_block)
                v[u] = c < chunks_per_block ? src_k[from + c] : src_v[from + (c - chunks_per_block)];
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int32_t c = first + u * kThreads;
            if (c < 2 * chunks_per_block) {
                if (c < chunks_per_block)
                    dst_k[to + c] = v[u];
                else
                    dst_v[to + (c - chunks_per_block)] = v[u];
            }
        }
    }
}

}  // namespace

cudaError_t launch_copy_blocks(const uint16_t *src_k, const uint16_t *src_v, uint16_t *dst_k,
                               uint16_t *dst_v, const int32_t *block_pairs, int32_t num_pairs,
                               int32_t num_heads, int32_t head_dim, int32_t block_size,
                               int32_t src_num_blocks, int32_t dst_num_blocks, int /*num_sms*/,
                               unsigned int *err, cudaStream_t stream) {
    const long long chunks = static_cast<long long>(num_heads) * block_size * head_dim / 8;
    if (num_pairs == 0 || chunks == 0) return cudaSuccess;
    if (2 * chunks > 0x7fffffffLL - kSegmentChunks) return cudaErrorInvalidValue;
    const int32_t chunks_per_block = static_cast<int32_t>(chunks);
    const unsigned segments =
        static_cast<unsigned>((2 * chunks + kSegmentChunks - 1) / kSegmentChunks);
    const unsigned pairs_y = static_cast<unsigned>(num_pairs < 65535 ? num_pairs : 65535);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(segments, pairs_y);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, copy_blocks_kernel, reinterpret_cast<const uint4 *>(src_k),
                              reinterpret_cast<const uint4 *>(src_v),
                              reinterpret_cast<uint4 *>(dst_k), reinterpret_cast<uint4 *>(dst_v),
                              block_pairs, num_pairs, chunks_per_block, src_num_blocks,
                              dst_num_blocks, err);
}

}  // namespace pa
