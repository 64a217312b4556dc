// span_rows.cu -- map query rows of chunked-prefill spans to their sequence.
//
// Query token i of a span of n tokens in a sequence of L tokens sits at
// position L - n + i and sees keys 0 .. L - n + i: the cached prefix plus
// causal within the chunk (Inference Engineering Day 12 short, "What is
// chunked prefill within vLLM").  This kernel writes, per query row, the
// sequence whose block table it walks and its key count L - n + i + 1, so the
// split-KV decode walk can serve the rows.  Rows of spans long enough for the
// tensor-core kernel get table row -1 and are left to that kernel.
#include "ns_common.cuh"
#include "ns_internal.h"

namespace ns {

__global__ void span_rows_kernel(const int32_t *__restrict__ qsl, const int32_t *__restrict__ lens,
                                 int num_seqs, int total_rows, int tc_min_span,
                                 int32_t *__restrict__ row_seq, int32_t *__restrict__ row_len,
                                 unsigned *status)
{
    const int v = blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= total_rows)
        return;
    // largest s with qsl[s] <= v (qsl is nondecreasing)
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(qsl + mid) <= v)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int s = lo;
    const int first = __ldg(qsl + s), next = __ldg(qsl + s + 1);
    const int n = next - first;
    const int L = __ldg(lens + s);
    int keys = L - n + (v - first) + 1;
    if (v < first || v >= next || n > L || first < 0) {
        raise_status(status, NS_DEV_BAD_QUERY_SPAN);
        keys = 0;
    }
    const bool tensor_core = tc_min_span > 0 && n >= tc_min_span;
    row_seq[v] = tensor_core ? -1 : s;
    row_len[v] = tensor_core ? 0 : keys;
}

cudaError_t launch_span_rows(const int32_t *query_start_loc, const int32_t *context_lens,
                             int num_seqs, int total_rows, int tc_min_span, int32_t *row_seq,
                             int32_t *row_len, unsigned *status, cudaStream_t stream)
{
    if (total_rows <= 0)
        return cudaSuccess;
    const int threads = 256;
    span_rows_kernel<<<(total_rows + threads - 1) / threads, threads, 0, stream>>>(
        query_start_loc, context_lens, num_seqs, total_rows, tc_min_span, row_seq, row_len, status);
    return cudaGetLastError();
}

}  // namespace ns
