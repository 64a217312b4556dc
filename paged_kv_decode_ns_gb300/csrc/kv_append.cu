// kv_append.cu -- scatter the step's new tokens into their pool slots.
//
// Each step stores its tokens' new K/V rows in the cache (Inference
// Engineering Day 11 short, "How does vLLM work"); in the paged layout (nanoserve project page, "What I built") slot s of a token is
// block s / bs, offset s % bs.  A bit-exact copy: one thread moves 16 bytes,
// eight threads move one 64-element head row, so both the reads of the new
// rows and the writes into the pool are whole 128-byte lines.
#include "ns_common.cuh"
#include "ns_internal.h"

namespace ns {

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4 *__restrict__ k,
                                                        const uint4 *__restrict__ v,
                                                        const int64_t *__restrict__ slot_mapping,
                                                        uint4 *__restrict__ k_pool,
                                                        uint4 *__restrict__ v_pool, long long n_chunks,
                                                        int num_kv_heads, int block_size,
                                                        long long num_slots, unsigned *status)
{
    constexpr int kChunksPerRow = kRowBytes / 16;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_chunks; i += stride) {
        const long long row = i / kChunksPerRow;  // (token, kv head)
        const int chunk = (int)(i % kChunksPerRow);
        const long long t = row / num_kv_heads;
        const int h = (int)(row % num_kv_heads);
        const long long slot = __ldg(slot_mapping + t);
        if (slot < 0)
            continue;
        if (slot >= num_slots) {
            if (h == 0 && chunk == 0)
                raise_status(status, NS_DEV_BAD_SLOT);
            continue;
        }
        const long long blk = slot / block_size, off = slot % block_size;
        const long long dst = ((blk * num_kv_heads + h) * block_size + off) * kChunksPerRow + chunk;
        k_pool[dst] = __ldg(k + i);
        v_pool[dst] = __ldg(v + i);
    }
}

cudaError_t launch_kv_append(const void *k, const void *v, const int64_t *slot_mapping, void *k_pool,
                             void *v_pool, int num_tokens, int num_kv_heads, int block_size,
                             long long num_blocks, unsigned *status, cudaStream_t stream)
{
    const long long n_chunks = (long long)num_tokens * num_kv_heads * (kRowBytes / 16);
    if (n_chunks == 0)
        return cudaSuccess;
    const int threads = 256;
    long long blocks = (n_chunks + threads - 1) / threads;
    if (blocks > 65535)
        blocks = 65535;
    kv_append_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping,
        static_cast<uint4 *>(k_pool), static_cast<uint4 *>(v_pool), n_chunks, num_kv_heads,
        block_size, num_blocks * block_size, status);
    return cudaGetLastError();
}

}  // namespace ns
