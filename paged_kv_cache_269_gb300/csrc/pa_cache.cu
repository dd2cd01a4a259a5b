// pa_cache.cu -- reshape_and_cache: store each new token's K and V in its slot.
//
// The pages say the K and V of past tokens are cached in HBM and each newly
// generated token is appended ("vLLM 2026 推理引擎全解：从 PagedAttention 到分离式
// Prefill", §1.1; doramagic.ai vLLM manual, "KVCacheManager 缓存管理").  Slot
// encoding (slot = physical_block * B + offset, negative = skip) is this
// library's reading.
//
// Launched with programmatic dependent launch: it may become resident while the
// previous decode on the stream drains, and waits for it before touching the
// caches.
//
// A pure copy: one thread moves 16 bytes (8 fp16 values) of one (token, head)
// row of K and the same of V; a warp covers whole 256-byte rows, so loads and
// stores are fully coalesced.  The work is a few MiB per decode step, so the
// kernel is launch-bound; it uses a grid-stride loop capped at a few waves.
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, uint4 *__restrict__ k_cache,
    uint4 *__restrict__ v_cache, const int32_t *__restrict__ slot_mapping, int32_t num_tokens,
    int32_t num_heads, int32_t chunks_per_row, int32_t block_size, long long pool_slots,
    unsigned int *err) {
    // The previous kernel on the stream may still be reading the caches.
    allow_dependents_to_launch();
    grid_dependency_wait();
    const long long total = static_cast<long long>(num_tokens) * num_heads * chunks_per_row;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += stride) {
        const int c = static_cast<int>(idx % chunks_per_row);
        const long long row = idx / chunks_per_row;  // token * H + head
        const int h = static_cast<int>(row % num_heads);
        const long long i = row / num_heads;
        const int32_t slot = __ldg(slot_mapping + i);
        if (slot < 0) continue;
        if (slot >= pool_slots) {
            if (h == 0 && c == 0) atomicOr(err, PA_DEVERR_SLOT);
            continue;
        }
        const long long blk = slot / block_size;
        const int off = slot % block_size;
        const size_t dst =
            ((static_cast<size_t>(blk) * num_heads + h) * block_size + off) * chunks_per_row + c;
        k_cache[dst] = __ldg(k + idx);
        v_cache[dst] = __ldg(v + idx);
    }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const uint16_t *k, const uint16_t *v, uint16_t *k_cache,
                                     uint16_t *v_cache, const int32_t *slot_mapping,
                                     int32_t num_tokens, int32_t num_heads, int32_t head_dim,
                                     int32_t block_size, int32_t num_blocks, unsigned int *err,
                                     cudaStream_t stream) {
    const int chunks = head_dim / 8;
    const long long total = static_cast<long long>(num_tokens) * num_heads * chunks;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    if (blocks > 65535) blocks = 65535;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, reshape_and_cache_kernel,
                              reinterpret_cast<const uint4 *>(k), reinterpret_cast<const uint4 *>(v),
                              reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache),
                              slot_mapping, num_tokens, num_heads, chunks, block_size,
                              static_cast<long long>(num_blocks) * block_size, err);
}

}  // namespace pa
