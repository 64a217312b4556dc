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
                                                        long long num_slots, unsigned *status,
                                                        int chunks_per_row)
{
    const int kChunksPerRow = chunks_per_row;  // 16-byte chunks of a head row
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

// q8_0 append: eight threads per (token, kv head) row, thread i holding
// elements 8i..8i+7 of K and of V; four threads make a 32-element block.  The
// block's scale d = max|x| / 127 and every code rint(x * (1/d)) (ties to even,
// clamped to +-127) are rounded to fp32 at each step, and d is stored as fp16
// (nearest even, saturating): the decisions the CPU oracle takes.  The threads
// of a block always run together (whole rows per warp), so a row that is
// skipped still takes part in the shuffles.
template <typename T>
__device__ __forceinline__ void q8_quantize8(const uint4 w, uint2 &codes, uint16_t &d16)
{
    const float2 x0 = unpack2<T>(w.x), x1 = unpack2<T>(w.y), x2 = unpack2<T>(w.z), x3 = unpack2<T>(w.w);
    const float x[8] = {x0.x, x0.y, x1.x, x1.y, x2.x, x2.y, x3.x, x3.y};
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        amax = fmaxf(amax, fabsf(x[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = __fdiv_rn(amax, 127.f);
    const float inv = d > 0.f ? __fdiv_rn(1.f, d) : 0.f;
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int code = max(-127, min(127, __float2int_rn(__fmul_rn(x[i], inv))));
        packed[i >> 2] |= (uint32_t)(code & 0xff) << (8 * (i & 3));
    }
    codes = make_uint2(packed[0], packed[1]);
    d16 = __half_as_ushort(__float2half_rn(fminf(d, 65504.f)));
}

template <typename T>
__global__ void __launch_bounds__(256) kv_append_q8_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                           const int64_t *__restrict__ slot_mapping,
                                                           uint2 *__restrict__ k_codes, uint16_t *__restrict__ k_scales,
                                                           uint2 *__restrict__ v_codes, uint16_t *__restrict__ v_scales,
                                                           long long n_chunks, int num_kv_heads, int block_size,
                                                           long long num_slots, unsigned *status)
{
    constexpr int kChunksPerRow = kHeadDim / 8;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long base = (long long)blockIdx.x * blockDim.x; base < n_chunks; base += stride) {
        const long long i = base + threadIdx.x;
        const bool on = i < n_chunks;
        const long long row = on ? i / kChunksPerRow : 0;  // (token, kv head)
        const int chunk = (int)(i % kChunksPerRow);
        const long long t = row / num_kv_heads;
        const int h = (int)(row % num_kv_heads);
        const long long slot = on ? __ldg(slot_mapping + t) : -1;
        const uint4 kw = on ? __ldg(k + i) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 vw = on ? __ldg(v + i) : make_uint4(0u, 0u, 0u, 0u);
        uint2 kc, vc;
        uint16_t kd, vd;
        q8_quantize8<T>(kw, kc, kd);
        q8_quantize8<T>(vw, vc, vd);
        if (slot < 0)
            continue;
        if (slot >= num_slots) {
            if (h == 0 && chunk == 0)
                raise_status(status, NS_DEV_BAD_SLOT);
            continue;
        }
        const long long blk = slot / block_size, off = slot % block_size;
        const long long prow = (blk * num_kv_heads + h) * block_size + off;
        k_codes[prow * kChunksPerRow + chunk] = kc;
        v_codes[prow * kChunksPerRow + chunk] = vc;
        if ((chunk & 3) == 0) {
            k_scales[prow * 2 + (chunk >> 2)] = kd;
            v_scales[prow * 2 + (chunk >> 2)] = vd;
        }
    }
}

cudaError_t launch_kv_append_q8(const void *k, const void *v, const int64_t *slot_mapping, void *k_codes,
                                void *k_scales, void *v_codes, void *v_scales, int num_tokens, int num_kv_heads,
                                int block_size, long long num_blocks, ns_dtype dtype, unsigned *status,
                                cudaStream_t stream)
{
    const long long n_chunks = (long long)num_tokens * num_kv_heads * (kHeadDim / 8);
    if (n_chunks == 0)
        return cudaSuccess;
    const int threads = 256;
    long long blocks = (n_chunks + threads - 1) / threads;
    if (blocks > 65535)
        blocks = 65535;
    auto kern = dtype == NS_BF16 ? kv_append_q8_kernel<BF16> : kv_append_q8_kernel<F16>;
    kern<<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, static_cast<uint2 *>(k_codes),
        static_cast<uint16_t *>(k_scales), static_cast<uint2 *>(v_codes), static_cast<uint16_t *>(v_scales),
        n_chunks, num_kv_heads, block_size, num_blocks * block_size, status);
    return cudaGetLastError();
}

cudaError_t launch_kv_append(const void *k, const void *v, const int64_t *slot_mapping, void *k_pool,
                             void *v_pool, int num_tokens, int num_kv_heads, int head_dim, int block_size,
                             long long num_blocks, unsigned *status, cudaStream_t stream)
{
    const int chunks_per_row = head_dim * 2 / 16;
    const long long n_chunks = (long long)num_tokens * num_kv_heads * chunks_per_row;
    if (n_chunks == 0)
        return cudaSuccess;
    const int threads = 256;
    long long blocks = (n_chunks + threads - 1) / threads;
    if (blocks > 65535)
        blocks = 65535;
    kv_append_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping,
        static_cast<uint4 *>(k_pool), static_cast<uint4 *>(v_pool), n_chunks, num_kv_heads,
        block_size, num_blocks * block_size, status, chunks_per_row);
    return cudaGetLastError();
}

}  // namespace ns
