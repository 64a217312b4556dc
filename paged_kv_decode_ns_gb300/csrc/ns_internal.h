// ns_internal.h -- host-side launchers shared between the C-ABI file and the
// kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include "ns_paged.h"

namespace ns {

cudaError_t launch_kv_append(const void *k, const void *v, const int64_t *slot_mapping, void *k_pool,
                             void *v_pool, int num_tokens, int num_kv_heads, int block_size,
                             long long num_blocks, unsigned *status, cudaStream_t stream);

// Query spans -> per-row table row and key count (prefill through the decode walk).
cudaError_t launch_span_rows(const int32_t *query_start_loc, const int32_t *context_lens,
                             int num_seqs, int total_rows, int32_t *row_seq, int32_t *row_len,
                             unsigned *status, cudaStream_t stream);

}  // namespace ns
