// pa_internal.h -- declarations shared by the translation units of libpa.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// Arguments of one decode launch (device pointers unless noted).
struct DecodeArgs {
    uint16_t *out;                 // fp16 or bf16 [S, H, D]
    const uint16_t *q;             // [S, H, D]
    const uint16_t *k_cache;       // [N, H, B, D]
    const uint16_t *v_cache;       // [N, H, B, D]
    const int32_t *block_tables;   // [S, max_blocks_per_seq]
    const int32_t *context_lens;   // [S]
    float scale_log2;              // softmax scale * log2(e)
    int32_t num_seqs;
    int32_t num_heads;
    int32_t num_blocks;
    int32_t max_blocks_per_seq;
    int32_t tiles_per_unit;        // KV blocks per partition (work unit)
    int32_t max_parts;             // ceil(max_blocks_per_seq / tiles_per_unit)
    float *part_ml;                // [S * H * max_parts * 2]: (running max, sum) per partition
    float *part_acc;               // [S * H * max_parts * D]: unnormalised partial outputs
    uint32_t *counters;            // [2 + S * H]: work queue, finished CTAs, per-(s,h) tickets
    unsigned int *err;             // device error word
    // Shared-prefix mode (group_start != nullptr): the prefix kernel, the
    // previous launch on the stream, has written slot 0 of the partials of
    // every row of each well-formed group with P_g > 0 (rows past rows_cap
    // excepted).  This kernel covers the rest of each sequence that may use
    // it and merges the two after waiting for the prefix kernel; the inputs
    // were complete before that kernel let this one launch.
    const int32_t *group_start;          // [num_groups + 1]
    const int32_t *group_prefix_blocks;  // [num_groups]
    int32_t num_groups;
    int32_t rows_cap;                    // rows per group the prefix kernel computes
    // Set by launch_decode (plain mode only).  0: every CTA keeps each
    // sequence's partition count and context length in shared memory.  c > 0:
    // it keeps one partition count per chunk of 2^c sequences (c >= 5), and
    // the producer warp resolves a unit's sequence from one coalesced load of
    // its chunk's context lengths, so large batches keep the CTAs per SM.
    int32_t chunk_shift;
};

// Sizes of the two caller buffers of pa_decode_ws.
//   counters: [2 + S * H] uint32 (queue head, finished CTAs, per-(s,h) tickets)
//   workspace: partial (max, sum) pairs [S * H * max_parts * 2] floats, then
//              partial outputs [S * H * max_parts * D] floats; empty when
//              max_parts == 1.
struct WorkspaceLayout {
    size_t counters_bytes;
    size_t ml_off, ml_bytes;
    size_t acc_off, acc_bytes;
    size_t workspace_bytes;
};

void workspace_layout(int32_t num_seqs, int32_t num_heads, int32_t head_dim, int32_t max_parts,
                      WorkspaceLayout *out);

cudaError_t launch_copy_blocks(const uint16_t *src_k, const uint16_t *src_v, uint16_t *dst_k,
                               uint16_t *dst_v, const int32_t *block_pairs, int32_t num_pairs,
                               int32_t num_heads, int32_t head_dim, int32_t block_size,
                               int32_t src_num_blocks, int32_t dst_num_blocks, int num_sms,
                               unsigned int *err, cudaStream_t stream);

// Arguments of one prefill launch (device pointers unless noted).
struct PrefillArgs {
    uint16_t *out;                 // [total_q, H, D]
    const int32_t *block_tables;   // [S, max_blocks_per_seq]
    const int32_t *context_lens;   // [S]
    const int32_t *query_start;    // [S + 1]
    float scale_log2;
    int32_t num_seqs;
    int32_t num_heads;
    int32_t num_blocks;
    int32_t max_blocks_per_seq;
    int32_t total_q;
    int32_t num_pairs;             // ceil(max_query_len / 256): pairs of 128-row tiles
    uint32_t *counters;            // [2]: next work item, CTAs done; zero on entry and exit
    unsigned int *err;
    // Shared-prefix mode (group_prefix_blocks != nullptr).  The "sequences"
    // are num_seqs groups of decode sequences: group g holds decode rows
    // query_start[g] .. query_start[g + 1] - 1 (total_q = the decode batch),
    // which share their first group_prefix_blocks[g] table entries.  Every
    // row attends to all of those prefix keys (no causal mask), the table row
    // read is the group's first sequence, and the result is written as a
    // decode partial -- (max, sum) and the unnormalised output -- into slot 0
    // of the row's partials.  block_tables is the decode batch's.
    const int32_t *group_prefix_blocks;
    float *part_ml;                // [S * H * max_parts * 2]
    float *part_acc;               // [S * H * max_parts * D]
    int32_t max_parts;
};


bool prefill_supported(int dtype, int head_dim, int block_size);
cudaError_t launch_prefill(const PrefillArgs &args, const void *q, const void *k_cache,
                           const void *v_cache, int dtype, int num_sms, cudaStream_t stream);

// One CTA whose bounded waits must all run out (pa_selftest.cu); result[3].
cudaError_t launch_wait_timeout_selftest(unsigned int *err, int *result, cudaStream_t stream);

// SM count and device error word of the current device (set up on first use).
int current_device_info(unsigned int **err, int *num_sms);

// Record a CUDA error for pa_last_cuda_error() and return PA_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// Kernel launchers (pa_decode.cu / pa_cache.cu).  They return a cudaError_t.
// `num_sms` sizes the persistent decode grid.
cudaError_t launch_decode(const DecodeArgs &args, int dtype, int head_dim, int block_size,
                          int num_sms, cudaStream_t stream);
bool decode_variant_supported(int dtype, int head_dim, int block_size);
// Whether a decode launch of num_seqs sequences (and num_groups shared-prefix
// groups; -1 for none) fits the current device's shared memory (after
// prepare_decode_kernels).
bool decode_fits(int dtype, int head_dim, int block_size, int num_heads, int num_seqs,
                 int num_groups);
cudaError_t prepare_decode_kernels(int device);

cudaError_t launch_reshape_and_cache(const uint16_t *k, const uint16_t *v, uint16_t *k_cache,
                                     uint16_t *v_cache, const int32_t *slot_mapping,
                                     int32_t num_tokens, int32_t num_heads, int32_t head_dim,
                                     int32_t block_size, int32_t num_blocks, unsigned int *err,
                                     cudaStream_t stream);

}  // namespace pa
