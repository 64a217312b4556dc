// ns_internal.h -- host-side launchers shared between the C-ABI file and the
// kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include "ns_paged.h"

namespace ns {

cudaError_t launch_kv_append(const void *k, const void *v, const int64_t *slot_mapping, void *k_pool,
                             void *v_pool, int num_tokens, int num_kv_heads, int head_dim, int block_size,
                             long long num_blocks, unsigned *status, cudaStream_t stream);

// q8_0 append: quantise each new token's K/V rows and scatter codes and scales.
cudaError_t launch_kv_append_q8(const void *k, const void *v, const int64_t *slot_mapping, void *k_codes,
                                void *k_scales, void *v_codes, void *v_scales, int num_tokens, int num_kv_heads,
                                int block_size, long long num_blocks, ns_dtype dtype, unsigned *status,
                                cudaStream_t stream);

// Query spans -> per-row table row and key count (prefill through the decode
// walk).  Rows of spans with at least `tc_min_span` tokens (tc_min_span > 0)
// are marked for the tensor-core kernel: table row -1, key count 0.
cudaError_t launch_span_rows(const int32_t *query_start_loc, const int32_t *context_lens,
                             int num_seqs, int total_rows, int tc_min_span, int32_t *row_seq,
                             int32_t *row_len, unsigned *status, cudaStream_t stream);

// Address of the device status word on device `dev` (current), or nullptr.
unsigned *device_status_word(int dev);

struct DecodeParams;

// Launch the split-KV decode kernel with num_ctas CTAs, or with the resident
// CTAs of device `dev` when num_ctas is 0.
ns_status launch_decode(const DecodeParams &P, ns_dtype dtype, int block_size, int num_ctas,
                        cudaStream_t stream, int dev, bool q8 = false, int head_dim = 64);

// Chunked prefill of every span of two or more tokens on the tcgen05 tensor cores.
// after_walk: the kernel just before it on the stream is this call's span walk
// (whose results it does not read), so it may be launched to overlap it.
bool tc_prefill_supported(int block_size, int group);
cudaError_t launch_tc_prefill(const void *q, const int32_t *query_start_loc, const void *k_pool,
                              const void *v_pool, const int32_t *block_tables,
                              const int32_t *context_lens, int num_seqs, int total_q_tokens,
                              int num_q_heads, int num_kv_heads, int block_size, float scale,
                              void *out, int max_blocks_per_seq, long long num_blocks, ns_dtype dtype,
                              int min_span, int head_dim, unsigned *status, bool after_walk,
                              cudaStream_t stream);

}  // namespace ns
