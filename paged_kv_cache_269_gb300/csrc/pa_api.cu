// pa_api.cu -- the C ABI of libpa (declared in include/pa.h).
//
// Host-side argument checking, per-device set-up, workspace sizing and the
// launches.  Every entry point returns a pa_status; nothing here throws,
// aborts or synchronises except pa_device_errors.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace pa {

// The device error word: kernels OR PA_DEVERR_* bits into it.
__device__ unsigned int g_device_error_word = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kDefaultPartitionTokens = 512;
constexpr int kVersion = 10000;  // 1.0.0

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    unsigned int *err = nullptr;  // device address of g_device_error_word
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
thread_local int t_last_cuda_error = 0;

int fail_cuda(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return PA_ERR_CUDA;
}

// Set up the current device once: SM count, error-word address, kernel
// attributes.  Returns PA_OK and the state, or PA_ERR_CUDA.
int current_device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return fail_cuda(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &st = g_devices[dev];
    if (!st.ready) {
        e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail_cuda(e);
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_device_error_word);
        if (e != cudaSuccess) return fail_cuda(e);
        st.err = static_cast<unsigned int *>(addr);
        e = prepare_decode_kernels(dev);
        if (e != cudaSuccess) return fail_cuda(e);
        st.ready = true;
    }
    *out = &st;
    return PA_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared checks of pa_dims.  need_seqs: num_seqs is used by the call.
int check_dims(const pa_dims *dims, bool need_seqs) {
    if (!dims) return PA_ERR_NULL;
    if (dims->num_heads <= 0 || dims->head_dim <= 0 || dims->block_size <= 0 ||
        dims->num_blocks <= 0)
        return PA_ERR_SHAPE;
    if (need_seqs && dims->num_seqs < 0) return PA_ERR_SHAPE;
    if (!decode_variant_supported(dims->dtype, dims->head_dim, dims->block_size))
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// Tiles per unit and number of partitions for a partition length.
int partition_plan(const pa_dims *dims, int32_t max_blocks_per_seq, int32_t partition_tokens,
                   int32_t *tiles_per_unit, int32_t *max_parts) {
    if (max_blocks_per_seq <= 0) return PA_ERR_SHAPE;
    const int B = dims->block_size;
    if (static_cast<long long>(max_blocks_per_seq) * B > 0x7fffffffLL) return PA_ERR_SHAPE;
    int32_t tokens = partition_tokens == 0 ? kDefaultPartitionTokens : partition_tokens;
    if (tokens < 0 || tokens % B != 0 || tokens == 0) return PA_ERR_SHAPE;
    int32_t tpu = tokens / B;
    if (tpu > max_blocks_per_seq) tpu = max_blocks_per_seq;
    *tiles_per_unit = tpu;
    *max_parts = (max_blocks_per_seq + tpu - 1) / tpu;
    // the work-queue index (sequence, partition, head) must fit in 32 bits
    const long long units = static_cast<long long>(dims->num_seqs) * dims->num_heads * *max_parts;
    if (units >= 0xffffffffLL - (1LL << 20)) return PA_ERR_SHAPE;
    return PA_OK;
}

// PA_OK if the current device can read and write `p` in a kernel: device
// memory of this device, managed memory, pinned or registered host memory,
// or any host memory when the device has coherent access to pageable memory.
int check_device_addressable(const void *p, int device) {
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();  // the failed query leaves a (non-sticky) error behind
        return PA_ERR_UNSUPPORTED;
    }
    switch (attr.type) {
        case cudaMemoryTypeDevice:
            return attr.device == device ? PA_OK : PA_ERR_UNSUPPORTED;
        case cudaMemoryTypeManaged:
        case cudaMemoryTypeHost:
            return PA_OK;
        default: {
            int pageable = 0;
            e = cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, device);
            return (e == cudaSuccess && pageable) ? PA_OK : PA_ERR_UNSUPPORTED;
        }
    }
}

// Buffers of a shared-prefix decode.  Counters (zero on entry and exit):
// the decode kernel's, then the prefix kernel's two (in 256 bytes).
// Workspace (no initialisation): the decode partials with one more slot per
// (sequence, head), slot 0, for the prefix partial.
struct SharedLayout {
    WorkspaceLayout dec;
    int32_t tiles_per_unit, max_parts;
    size_t prefix_counters_off, counters_bytes, workspace_bytes;
};

int shared_layout(const pa_dims *dims, int32_t max_blocks_per_seq, int32_t partition_tokens,
                  SharedLayout *out) {
    SharedLayout l;
    int rc = partition_plan(dims, max_blocks_per_seq, partition_tokens, &l.tiles_per_unit,
                            &l.max_parts);
    if (rc != PA_OK) return rc;
    l.max_parts += 1;
    workspace_layout(dims->num_seqs, dims->num_heads, dims->head_dim, l.max_parts, &l.dec);
    l.prefix_counters_off = l.dec.counters_bytes;
    l.counters_bytes = l.prefix_counters_off + 256;
    l.workspace_bytes = l.dec.workspace_bytes;
    *out = l;
    return PA_OK;
}

}  // namespace

int record_cuda_error(cudaError_t e) { return fail_cuda(e); }

int current_device_info(unsigned int **err, int *num_sms) {
    DeviceState *st = nullptr;
    const int rc = current_device_state(&st);
    if (rc != PA_OK) return rc;
    *err = st->err;
    *num_sms = st->num_sms;
    return PA_OK;
}

void workspace_layout(int32_t num_seqs, int32_t num_heads, int32_t head_dim, int32_t max_parts,
                      WorkspaceLayout *out) {
    const size_t pairs = static_cast<size_t>(num_seqs) * static_cast<size_t>(num_heads);
    const size_t parts = max_parts > 1 ? pairs * static_cast<size_t>(max_parts) : 0;
    WorkspaceLayout l;
    l.counters_bytes = round_up((2 + pairs) * sizeof(uint32_t), 256);
    l.ml_off = 0;
    l.ml_bytes = round_up(parts * 2 * sizeof(float), 256);
    l.acc_off = l.ml_off + l.ml_bytes;
    l.acc_bytes = round_up(parts * static_cast<size_t>(head_dim) * sizeof(float), 256);
    l.workspace_bytes = l.acc_off + l.acc_bytes;
    *out = l;
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                         const int32_t *slot_mapping, int32_t num_tokens, const pa_dims *dims,
                         void *stream) {
    int rc = check_dims(dims, false);
    if (rc != PA_OK) return rc;
    if (num_tokens < 0) return PA_ERR_SHAPE;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_NULL;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PA_ERR_ALIGN;
    if (static_cast<long long>(dims->num_blocks) * dims->block_size > 0x7fffffffLL)
        return PA_ERR_SHAPE;
    DeviceState *st = nullptr;
    rc = current_device_state(&st);
    if (rc != PA_OK) return rc;
    cudaError_t e = launch_reshape_and_cache(
        static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(v),
        static_cast<uint16_t *>(k_cache), static_cast<uint16_t *>(v_cache), slot_mapping,
        num_tokens, dims->num_heads, dims->head_dim, dims->block_size, dims->num_blocks, st->err,
        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : fail_cuda(e);
}

int pa_copy_blocks(const void *src_k, const void *src_v, int32_t src_num_blocks, void *dst_k,
                   void *dst_v, int32_t dst_num_blocks, const int32_t *block_pairs,
                   int32_t num_pairs, const pa_dims *dims, void *stream) {
    if (!dims) return PA_ERR_NULL;
    if (dims->num_heads <= 0 || dims->head_dim <= 0 || dims->block_size <= 0 || num_pairs < 0 ||
        src_num_blocks <= 0 || dst_num_blocks <= 0)
        return PA_ERR_SHAPE;
    if (!decode_variant_supported(dims->dtype, dims->head_dim, dims->block_size))
        return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !block_pairs) return PA_ERR_NULL;
    if (!aligned(src_k, 16) || !aligned(src_v, 16) || !aligned(dst_k, 16) || !aligned(dst_v, 16) ||
        !aligned(block_pairs, 4))
        return PA_ERR_ALIGN;
    DeviceState *st = nullptr;
    int rc = current_device_state(&st);
    if (rc != PA_OK) return rc;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    for (const void *p : {src_k, src_v, static_cast<const void *>(dst_k),
                          static_cast<const void *>(dst_v),
                          static_cast<const void *>(block_pairs)}) {
        rc = check_device_addressable(p, dev);
        if (rc != PA_OK) return rc;
    }
    e = launch_copy_blocks(static_cast<const uint16_t *>(src_k), static_cast<const uint16_t *>(src_v),
                           static_cast<uint16_t *>(dst_k), static_cast<uint16_t *>(dst_v),
                           block_pairs, num_pairs, dims->num_heads, dims->head_dim,
                           dims->block_size, src_num_blocks, dst_num_blocks, st->num_sms, st->err,
                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : fail_cuda(e);
}

int pa_prefill_ws(void *out, const void *q, const void *k_cache, const void *v_cache,
                  const int32_t *block_tables, const int32_t *context_lens,
                  const int32_t *query_start, int32_t total_query_tokens, int32_t max_query_len,
                  float scale, int32_t max_blocks_per_seq, const pa_dims *dims,
                  uint32_t *counters, size_t counters_bytes, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != PA_OK) return rc;
    if (!prefill_supported(dims->dtype, dims->head_dim, dims->block_size)) return PA_ERR_UNSUPPORTED;
    if (total_query_tokens < 0 || max_query_len < 0 || max_blocks_per_seq <= 0) return PA_ERR_SHAPE;
    if (dims->num_seqs == 0 || total_query_tokens == 0 || max_query_len == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start ||
        !counters)
        return PA_ERR_NULL;
    if (counters_bytes < PA_PREFILL_COUNTERS_BYTES) return PA_ERR_WORKSPACE;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(counters, 4))
        return PA_ERR_ALIGN;
    if (!isfinite(scale)) return PA_ERR_SHAPE;
    // tensor-map coordinates are 32-bit: every cache row and query row must fit
    const long long pairs = (static_cast<long long>(max_query_len) + 255) / 256;
    if (static_cast<long long>(dims->num_blocks) * dims->num_heads * dims->block_size > 0x7fffffffLL ||
        static_cast<long long>(max_blocks_per_seq) * dims->block_size > 0x7fffffffLL ||
        pairs * dims->num_seqs * dims->num_heads > 0x7fffffffLL)
        return PA_ERR_SHAPE;
    unsigned int *err = nullptr;
    int sms = 0;
    rc = current_device_info(&err, &sms);
    if (rc != PA_OK) return rc;
    PrefillArgs a;
    a.out = static_cast<uint16_t *>(out);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start = query_start;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    a.num_seqs = dims->num_seqs;
    a.num_heads = dims->num_heads;
    a.num_blocks = dims->num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.total_q = total_query_tokens;
    a.num_pairs = static_cast<int32_t>(pairs);
    a.counters = counters;
    a.err = err;
    a.group_prefix_blocks = nullptr;
    a.part_ml = nullptr;
    a.part_acc = nullptr;
    a.max_parts = 0;
    const cudaError_t e = launch_prefill(a, q, k_cache, v_cache, dims->dtype, sms,
                                         static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue) return PA_ERR_UNSUPPORTED;  // tensor maps could not be made
    return e == cudaSuccess ? PA_OK : fail_cuda(e);
}

int pa_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
               const int32_t *block_tables, const int32_t *context_lens,
               const int32_t *query_start, int32_t total_query_tokens, int32_t max_query_len,
               float scale, int32_t max_blocks_per_seq, const pa_dims *dims, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != PA_OK) return rc;
    if (!prefill_supported(dims->dtype, dims->head_dim, dims->block_size)) return PA_ERR_UNSUPPORTED;
    if (total_query_tokens < 0 || max_query_len < 0 || max_blocks_per_seq <= 0) return PA_ERR_SHAPE;
    if (dims->num_seqs == 0 || total_query_tokens == 0 || max_query_len == 0) return PA_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *buf = nullptr;
    cudaError_t e = cudaMallocAsync(&buf, PA_PREFILL_COUNTERS_BYTES, s);
    if (e != cudaSuccess) return fail_cuda(e);
    e = cudaMemsetAsync(buf, 0, PA_PREFILL_COUNTERS_BYTES, s);
    if (e != cudaSuccess) {
        cudaFreeAsync(buf, s);
        return fail_cuda(e);
    }
    rc = pa_prefill_ws(out, q, k_cache, v_cache, block_tables, context_lens, query_start,
                       total_query_tokens, max_query_len, scale, max_blocks_per_seq, dims,
                       static_cast<uint32_t *>(buf), PA_PREFILL_COUNTERS_BYTES, stream);
    e = cudaFreeAsync(buf, s);
    if (rc != PA_OK) return rc;
    return e == cudaSuccess ? PA_OK : fail_cuda(e);
}

size_t pa_decode_workspace_bytes(const pa_dims *dims, int32_t max_blocks_per_seq,
                                 int32_t partition_tokens) {
    if (check_dims(dims, true) != PA_OK) return static_cast<size_t>(-1);
    int32_t tpu = 0, parts = 0;
    if (partition_plan(dims, max_blocks_per_seq, partition_tokens, &tpu, &parts) != PA_OK)
        return static_cast<size_t>(-1);
    WorkspaceLayout l;
    workspace_layout(dims->num_seqs, dims->num_heads, dims->head_dim, parts, &l);
    return l.workspace_bytes;
}

size_t pa_decode_counters_bytes(const pa_dims *dims) {
    if (check_dims(dims, true) != PA_OK) return 0;
    WorkspaceLayout l;
    workspace_layout(dims->num_seqs, dims->num_heads, dims->head_dim, 1, &l);
    return l.counters_bytes;
}

int pa_decode_ws(void *out, const void *q, const void *k_cache, const void *v_cache,
                 const int32_t *block_tables, const int32_t *context_lens, float scale,
                 int32_t max_blocks_per_seq, const pa_dims *dims, int32_t partition_tokens,
                 void *workspace, size_t workspace_bytes, uint32_t *counters,
                 size_t counters_bytes, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != PA_OK) return rc;
    int32_t tpu = 0, parts = 0;
    rc = partition_plan(dims, max_blocks_per_seq, partition_tokens, &tpu, &parts);
    if (rc != PA_OK) return rc;
    if (dims->num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_NULL;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PA_ERR_ALIGN;
    if (!isfinite(scale)) return PA_ERR_SHAPE;
    WorkspaceLayout l;
    workspace_layout(dims->num_seqs, dims->num_heads, dims->head_dim, parts, &l);
    if (!counters || counters_bytes < l.counters_bytes || !aligned(counters, 4))
        return PA_ERR_WORKSPACE;
    if (l.workspace_bytes > 0 &&
        (!workspace || workspace_bytes < l.workspace_bytes || !aligned(workspace, 16)))
        return PA_ERR_WORKSPACE;

    DeviceState *st = nullptr;
    rc = current_device_state(&st);
    if (rc != PA_OK) return rc;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    DecodeArgs a;
    a.out = static_cast<uint16_t *>(out);
    a.q = static_cast<const uint16_t *>(q);
    a.k_cache = static_cast<const uint16_t *>(k_cache);
    a.v_cache = static_cast<const uint16_t *>(v_cache);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    a.num_seqs = dims->num_seqs;
    a.num_heads = dims->num_heads;
    a.num_blocks = dims->num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.tiles_per_unit = tpu;
    a.max_parts = parts;
    a.counters = counters;
    a.part_ml = parts > 1 ? reinterpret_cast<float *>(ws + l.ml_off) : nullptr;
    a.part_acc = parts > 1 ? reinterpret_cast<float *>(ws + l.acc_off) : nullptr;
    a.err = st->err;
    a.group_start = nullptr;
    a.group_prefix_blocks = nullptr;
    a.num_groups = 0;
    a.rows_cap = 0;
    a.chunk_shift = 0;
    cudaError_t e = launch_decode(a, dims->dtype, dims->head_dim, dims->block_size, st->num_sms,
                                  static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidConfiguration) return PA_ERR_UNSUPPORTED;  // too many sequences
    return e == cudaSuccess ? PA_OK : fail_cuda(e);
}

int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, const int32_t *context_lens, float scale,
              int32_t max_blocks_per_seq, const pa_dims *dims, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != PA_OK) return rc;
    int32_t tpu = 0, parts = 0;
    rc = partition_plan(dims, max_blocks_per_seq, 0, &tpu, &parts);
    if (rc != PA_OK) return rc;
    if (dims->num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_NULL;
    WorkspaceLayout l;
    workspace_layout(dims->num_seqs, dims->num_heads, dims->head_dim, parts, &l);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceState *st = nullptr;
    rc = current_device_state(&st);
    if (rc != PA_OK) return rc;
    // one allocation: counters first, then the partial-result workspace
    void *buf = nullptr;
    cudaError_t e = cudaMallocAsync(&buf, l.counters_bytes + l.workspace_bytes, s);
    if (e != cudaSuccess) return fail_cuda(e);
    e = cudaMemsetAsync(buf, 0, l.counters_bytes, s);
    if (e != cudaSuccess) {
        cudaFreeAsync(buf, s);
        return fail_cuda(e);
    }
    uint8_t *base = static_cast<uint8_t *>(buf);
    rc = pa_decode_ws(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                      max_blocks_per_seq, dims, 0, l.workspace_bytes ? base + l.counters_bytes : nullptr,
                      l.workspace_bytes, reinterpret_cast<uint32_t *>(base), l.counters_bytes,
                      stream);
    e = cudaFreeAsync(buf, s);
    if (rc != PA_OK) return rc;
    return e == cudaSuccess ? PA_OK : fail_cuda(e);
}

size_t pa_decode_shared_prefix_workspace_bytes(const pa_dims *dims, int32_t max_blocks_per_seq,
                                               int32_t partition_tokens) {
    if (check_dims(dims, true) != PA_OK) return static_cast<size_t>(-1);
    SharedLayout l;
    if (shared_layout(dims, max_blocks_per_seq, partition_tokens, &l) != PA_OK)
        return static_cast<size_t>(-1);
    return l.workspace_bytes;
}

size_t pa_decode_shared_prefix_counters_bytes(const pa_dims *dims) {
    if (check_dims(dims, true) != PA_OK) return 0;
    SharedLayout l;
    if (shared_layout(dims, 1, 0, &l) != PA_OK) return 0;
    return l.counters_bytes;
}

int pa_decode_shared_prefix_ws(void *out, const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens,
                               float scale, int32_t max_blocks_per_seq, const pa_dims *dims,
                               const int32_t *group_start, const int32_t *group_prefix_blocks,
                               int32_t num_groups, int32_t max_group_size,
                               int32_t partition_tokens, void *workspace, size_t workspace_bytes,
                               uint32_t *counters, size_t counters_bytes, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != PA_OK) return rc;
    if (!prefill_supported(dims->dtype, dims->head_dim, dims->block_size)) return PA_ERR_UNSUPPORTED;
    if (num_groups < 0 || max_group_size < 0) return PA_ERR_SHAPE;
    SharedLayout l;
    rc = shared_layout(dims, max_blocks_per_seq, partition_tokens, &l);
    if (rc != PA_OK) return rc;
    if (dims->num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_NULL;
    const bool groups = num_groups > 0 && max_group_size > 0;
    if (groups && (!group_start || !group_prefix_blocks)) return PA_ERR_NULL;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PA_ERR_ALIGN;
    if (!isfinite(scale)) return PA_ERR_SHAPE;
    // the prefix kernel's tensor-map coordinates and work items are 32-bit
    const long long pairs = (static_cast<long long>(max_group_size) + 255) / 256;
    if (static_cast<long long>(dims->num_blocks) * dims->num_heads * dims->block_size > 0x7fffffffLL ||
        pairs * num_groups * dims->num_heads > 0x7fffffffLL)
        return PA_ERR_SHAPE;
    if (!counters || counters_bytes < l.counters_bytes || !aligned(counters, 4))
        return PA_ERR_WORKSPACE;
    if (!workspace || workspace_bytes < l.workspace_bytes || !aligned(workspace, 16))
        return PA_ERR_WORKSPACE;

    DeviceState *st = nullptr;
    rc = current_device_state(&st);
    if (rc != PA_OK) return rc;
    // checked before the prefix kernel writes anything into the counters
    if (!decode_fits(dims->dtype, dims->head_dim, dims->block_size, dims->num_heads,
                     dims->num_seqs, groups ? num_groups : -1))
        return PA_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *ctr = reinterpret_cast<uint8_t *>(counters);
    float *part_ml = reinterpret_cast<float *>(ws + l.dec.ml_off);
    float *part_acc = reinterpret_cast<float *>(ws + l.dec.acc_off);
    const float scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);

    if (groups) {
        PrefillArgs p;
        p.out = nullptr;
        p.block_tables = block_tables;
        p.context_lens = context_lens;
        p.query_start = group_start;
        p.scale_log2 = scale_log2;
        p.num_seqs = num_groups;
        p.num_heads = dims->num_heads;
        p.num_blocks = dims->num_blocks;
        p.max_blocks_per_seq = max_blocks_per_seq;
        p.total_q = dims->num_seqs;
        p.num_pairs = static_cast<int32_t>(pairs);
        p.counters = reinterpret_cast<uint32_t *>(ctr + l.prefix_counters_off);
        p.err = st->err;
        p.group_prefix_blocks = group_prefix_blocks;
        p.part_ml = part_ml;
        p.part_acc = part_acc;
        p.max_parts = l.max_parts;
        const cudaError_t e = launch_prefill(p, q, k_cache, v_cache, dims->dtype, st->num_sms, s);
        if (e == cudaErrorInvalidValue) return PA_ERR_UNSUPPORTED;  // tensor maps could not be made
        if (e != cudaSuccess) return fail_cuda(e);
    }
    DecodeArgs a;
    a.out = static_cast<uint16_t *>(out);
    a.q = static_cast<const uint16_t *>(q);
    a.k_cache = static_cast<const uint16_t *>(k_cache);
    a.v_cache = static_cast<const uint16_t *>(v_cache);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.scale_log2 = scale_log2;
    a.num_seqs = dims->num_seqs;
    a.num_heads = dims->num_heads;
    a.num_blocks = dims->num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.tiles_per_unit = l.tiles_per_unit;
    a.max_parts = l.max_parts;
    a.counters = counters;
    a.part_ml = part_ml;
    a.part_acc = part_acc;
    a.err = st->err;
    a.group_start = groups ? group_start : nullptr;
    a.group_prefix_blocks = groups ? group_prefix_blocks : nullptr;
    a.num_groups = groups ? num_groups : 0;
    a.rows_cap = static_cast<int32_t>(pairs * 256 > 0x7fffffffLL ? 0x7fffffffLL : pairs * 256);
    a.chunk_shift = 0;
    const cudaError_t e = launch_decode(a, dims->dtype, dims->head_dim, dims->block_size,
                                        st->num_sms, s);
    if (e == cudaErrorInvalidConfiguration) return PA_ERR_UNSUPPORTED;  // too many sequences
    return e == cudaSuccess ? PA_OK : fail_cuda(e);
}

int pa_decode_shared_prefix(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *context_lens, float scale,
                            int32_t max_blocks_per_seq, const pa_dims *dims,
                            const int32_t *group_start, const int32_t *group_prefix_blocks,
                            int32_t num_groups, int32_t max_group_size, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != PA_OK) return rc;
    if (!prefill_supported(dims->dtype, dims->head_dim, dims->block_size)) return PA_ERR_UNSUPPORTED;
    SharedLayout l;
    rc = shared_layout(dims, max_blocks_per_seq, 0, &l);
    if (rc != PA_OK) return rc;
    if (dims->num_seqs == 0) return PA_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceState *st = nullptr;
    rc = current_device_state(&st);
    if (rc != PA_OK) return rc;
    void *buf = nullptr;
    cudaError_t e = cudaMallocAsync(&buf, l.counters_bytes + l.workspace_bytes, s);
    if (e != cudaSuccess) return fail_cuda(e);
    e = cudaMemsetAsync(buf, 0, l.counters_bytes, s);
    if (e != cudaSuccess) {
        cudaFreeAsync(buf, s);
        return fail_cuda(e);
    }
    uint8_t *base = static_cast<uint8_t *>(buf);
    rc = pa_decode_shared_prefix_ws(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                    max_blocks_per_seq, dims, group_start, group_prefix_blocks,
                                    num_groups, max_group_size, 0, base + l.counters_bytes,
                                    l.workspace_bytes, reinterpret_cast<uint32_t *>(base),
                                    l.counters_bytes, stream);
    e = cudaFreeAsync(buf, s);
    if (rc != PA_OK) return rc;
    return e == cudaSuccess ? PA_OK : fail_cuda(e);
}

int pa_selftest_wait_timeout(int32_t *results, void *stream) {
    if (!results) return PA_ERR_NULL;
    DeviceState *st = nullptr;
    int rc = current_device_state(&st);
    if (rc != PA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int *dres = nullptr;
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void **>(&dres), 3 * sizeof(int), s);
    if (e != cudaSuccess) return fail_cuda(e);
    e = cudaMemsetAsync(dres, 0xff, 3 * sizeof(int), s);
    if (e == cudaSuccess) e = launch_wait_timeout_selftest(st->err, dres, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(results, dres, 3 * sizeof(int), cudaMemcpyDeviceToHost, s);
    const cudaError_t ef = cudaFreeAsync(dres, s);
    if (e == cudaSuccess) e = ef;
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? PA_OK : fail_cuda(e);
}

int pa_device_errors(void *stream, uint32_t *flags) {
    if (!flags) return PA_ERR_NULL;
    DeviceState *st = nullptr;
    int rc = current_device_state(&st);
    if (rc != PA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&word, st->err, sizeof(word), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(st->err, 0, sizeof(unsigned int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail_cuda(e);
    *flags = word;
    return PA_OK;
}

const char *pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_NULL: return "a required pointer is NULL";
        case PA_ERR_SHAPE: return "invalid size";
        case PA_ERR_UNSUPPORTED: return "unsupported head_dim, block_size or batch size";
        case PA_ERR_ALIGN: return "fp16 pointer not 16-byte aligned";
        case PA_ERR_WORKSPACE: return "workspace or counter buffer missing, too small or misaligned";
        case PA_ERR_CUDA: return "CUDA runtime error";
        case PA_ERR_OUT_OF_BLOCKS: return "KV cache exhausted: no free block";
        default: return "unknown status";
    }
}

int pa_last_cuda_error(void) { return t_last_cuda_error; }

int pa_version(void) { return kVersion; }

}  // extern "C"
