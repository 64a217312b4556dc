// paged_decode_launch.cuh -- host launch of the decode kernel for one element
// type and block size (included by the per-type instantiation files).
#pragma once

#include "paged_decode.cuh"

namespace ns {

constexpr int kDecodeWarps = 4;  // consumer warps per CTA (one block each per stage)

// Shared-memory ring depth: about 64 KB of K/V staging per CTA.
constexpr int decode_stages(int BS)
{
    return (65536 / (kDecodeWarps * 2 * BS * kRowBytes)) < 2 ? 2
           : (65536 / (kDecodeWarps * 2 * BS * kRowBytes)) > 8
               ? 8
               : (65536 / (kDecodeWarps * 2 * BS * kRowBytes));
}

template <typename T, int BS>
struct DecodeKernel {
    static constexpr int NW = kDecodeWarps;
    static constexpr int STAGES = decode_stages(BS);
    static constexpr int THREADS = (NW + 1) * 32;
    static constexpr size_t SMEM = sizeof(DecodeSmem<BS, NW, STAGES>);
    static void (*fn())(const DecodeParams) { return paged_decode_kernel<T, BS, NW, STAGES>; }

    static cudaError_t prepare()
    {
        // Opt in to more than 48 KB of dynamic shared memory (per device; cheap to repeat).
        static int done_mask = 0;
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return e;
        if (dev < 31 && (done_mask >> dev) & 1)
            return cudaSuccess;
        e = cudaFuncSetAttribute(fn(), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
        if (e == cudaSuccess && dev < 31)
            __atomic_fetch_or(&done_mask, 1 << dev, __ATOMIC_RELAXED);
        return e;
    }
};

template <typename T, int BS>
cudaError_t launch_paged_decode(const DecodeParams &P, int num_ctas, cudaStream_t stream)
{
    using K = DecodeKernel<T, BS>;
    cudaError_t e = K::prepare();
    if (e != cudaSuccess)
        return e;
    K::fn()<<<num_ctas, K::THREADS, K::SMEM, stream>>>(P);
    return cudaGetLastError();
}

template <typename T, int BS>
int decode_ctas_per_sm()
{
    using K = DecodeKernel<T, BS>;
    if (K::prepare() != cudaSuccess)
        return 1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, K::fn(), K::THREADS, K::SMEM) != cudaSuccess || n < 1)
        return 1;
    return n;
}

#define NS_INSTANTIATE_DECODE(T, BS)                                                               \
    template cudaError_t launch_paged_decode<T, BS>(const DecodeParams &, int, cudaStream_t);      \
    template int decode_ctas_per_sm<T, BS>();

}  // namespace ns
