// pa_static.cu -- pa_decode_static: paged-attention decode that allocates
// no device memory.
//
// Who needs this: a caller that cannot let a library call cudaMalloc.  Typical
// cases are a serving process that reserves almost all device memory for its
// KV-block pool at start-up and forbids allocations afterwards (a late
// cudaMalloc would fail or eat into the pool), a latency-critical decode loop
// that must never stall on cudaMalloc / cudaFree (both can synchronise the
// whole device), and a plugin running inside a host program whose allocator it
// does not own.  Such a caller passes only its inputs and outputs; the
// counters and partial results the split-context decode needs live in the
// fixed array below instead of a caller-provided or stream-allocated
// workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds PA_STATIC_SCRATCH_BYTES of it until the process exits.  In
// host code its name is only a host-side stand-in, so the device address is
// looked up with cudaGetSymbolAddress, once per device, on the first call made
// while that device is current, and cached for the life of the process (a
// cudaDeviceReset invalidates it, as it does every per-device address the
// library caches).  Argument checks all run before that look-up, so a call
// that is rejected launches nothing.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr size_t kScratchBytes = PA_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Shared by every call on a device; keeps whatever the last call left in it.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
unsigned char *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device (looked up once).
int scratch_address(unsigned char **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return record_cuda_error(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return record_cuda_error(e);
        g_scratch_ptr[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

size_t round_up_256(size_t x) { return (x + 255) / 256 * 256; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pa

extern "C" int pa_decode_static(void *out, const void *q, const void *k_cache,
                                const void *v_cache, const int32_t *block_tables,
                                const int32_t *context_lens, float scale,
                                int32_t max_blocks_per_seq, const pa_dims *dims, void *stream) {
    using namespace pa;
    const size_t size_error = static_cast<size_t>(-1);
    if (!dims) return PA_ERR_NULL;
    // Every check that needs no GPU comes first, in pa_decode_ws's order, so
    // that a rejected call neither touches the device nor queues anything.
    const size_t counters = pa_decode_counters_bytes(dims);
    if (counters == 0) {
        // invalid dims: let the regular checks report the exact reason
        return pa_decode_ws(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                            max_blocks_per_seq, dims, 0, nullptr, 0, nullptr, 0, stream);
    }
    if (max_blocks_per_seq <= 0) return PA_ERR_SHAPE;
    size_t partials = pa_decode_workspace_bytes(dims, max_blocks_per_seq, 0);
    if (partials == size_error) return PA_ERR_SHAPE;
    if (dims->num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_NULL;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_ALIGN;
    if (!isfinite(scale)) return PA_ERR_SHAPE;
    const size_t counters_region = round_up_256(counters);
    if (counters_region > kScratchBytes) return PA_ERR_WORKSPACE;  // too many (seq, head) pairs

    // Partition length: the library default if its partial results fit next
    // to the counters, else doubled until they fit; a single pass over each
    // context (no partials at all) always fits.
    const long long single_pass = static_cast<long long>(max_blocks_per_seq) * dims->block_size;
    int32_t partition = 0;
    long long tokens = 512;
    while (counters_region + partials > kScratchBytes) {
        if (tokens >= single_pass || tokens > 0x40000000LL) tokens = single_pass;
        partition = static_cast<int32_t>(tokens);
        partials = pa_decode_workspace_bytes(dims, max_blocks_per_seq, partition);
        if (partials == size_error) return PA_ERR_SHAPE;
        if (tokens == single_pass) break;
        tokens *= 2;
    }
    if (counters_region + partials > kScratchBytes) return PA_ERR_WORKSPACE;

    unsigned char *scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != PA_OK) return rc;
    // The counters must start at zero; the array holds whatever the last call
    // (possibly one that failed part-way) left there.
    cudaError_t e = cudaMemsetAsync(scratch, 0, counters, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return record_cuda_error(e);
    return pa_decode_ws(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                        max_blocks_per_seq, dims, partition,
                        partials ? scratch + counters_region : nullptr, partials,
                        reinterpret_cast<uint32_t *>(scratch), counters, stream);
}
