// paged_decode_launch.cuh -- host launch of the decode kernel for one element
// type, block size and group size (included by the instantiation files).
#pragma once

#include "paged_decode.cuh"

namespace ns {

template <typename T, int BS, int G, bool Q8, int D, bool TWO = false, int VU = 0>
struct DecodeKernel {
    static constexpr int S = decode_stages<BS, G, Q8, D>();
    static_assert(sizeof(DecodeSmem<BS, G, S, Q8, D>) <= kMaxDynSmem, "decode shared memory");
    static constexpr int THREADS = kDecodeThreads;  // consumers + producer warpgroup
    static constexpr size_t SMEM = sizeof(DecodeSmem<BS, G, S, Q8, D>);
    static void (*fn())(const DecodeParams) { return paged_decode_kernel<T, BS, G, S, Q8, D, TWO, VU>; }

    static cudaError_t prepare()
    {
        // Opt in to more than 48 KB of dynamic shared memory (per device).
        static int done_mask = 0;
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return e;
        if (dev < 31 && ((__atomic_load_n(&done_mask, __ATOMIC_RELAXED) >> dev) & 1))
            return cudaSuccess;
        // The warpgroups trade registers with setmaxnreg; the trade balances
        // only at exactly kLaunchRegs registers a thread, so refuse any other.
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, fn());
        if (e != cudaSuccess)
            return e;
        if (fa.numRegs != kLaunchRegs)
            return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(fn(), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
        if (e == cudaSuccess && dev < 31)
            __atomic_fetch_or(&done_mask, 1 << dev, __ATOMIC_RELAXED);
        return e;
    }
};

template <typename T, int BS, int G, bool Q8, int D, bool TWO, int VU>
cudaError_t launch_paged_decode(const DecodeParams &P, int num_ctas, cudaStream_t stream)
{
    using K = DecodeKernel<T, BS, G, Q8, D, TWO, VU>;
    cudaError_t e = K::prepare();
    if (e != cudaSuccess)
        return e;
    if (!P.overlap) {
        K::fn()<<<num_ctas, K::THREADS, K::SMEM, stream>>>(P);
        return cudaGetLastError();
    }
    // programmatic dependent launch: may start while the previous grid drains
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_ctas);
    cfg.blockDim = dim3(K::THREADS);
    cfg.dynamicSmemBytes = K::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, K::fn(), P);
}

template <typename T, int BS, int G, bool Q8, int D>
int decode_ctas_per_sm()
{
    using K = DecodeKernel<T, BS, G, Q8, D>;
    if (K::prepare() != cudaSuccess)
        return 1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, K::fn(), K::THREADS, K::SMEM) != cudaSuccess || n < 1)
        return 1;
    return n;
}

#define NS_INSTANTIATE_DECODE_G(T, BS, G, Q8, D)                                                    \
    template cudaError_t launch_paged_decode<T, BS, G, Q8, D>(const DecodeParams &, int, cudaStream_t); \
    template int decode_ctas_per_sm<T, BS, G, Q8, D>();

#define NS_INSTANTIATE_DECODE_QD(T, BS, Q8, D)                                                     \
    NS_INSTANTIATE_DECODE_G(T, BS, 1, Q8, D)                                                       \
    NS_INSTANTIATE_DECODE_G(T, BS, 2, Q8, D)                                                       \
    NS_INSTANTIATE_DECODE_G(T, BS, 3, Q8, D)                                                       \
    NS_INSTANTIATE_DECODE_G(T, BS, 4, Q8, D)                                                       \
    NS_INSTANTIATE_DECODE_G(T, BS, 5, Q8, D)                                                       \
    NS_INSTANTIATE_DECODE_G(T, BS, 6, Q8, D)                                                       \
    NS_INSTANTIATE_DECODE_G(T, BS, 7, Q8, D)                                                       \
    NS_INSTANTIATE_DECODE_G(T, BS, 8, Q8, D)

#define NS_INSTANTIATE_DECODE(T, BS) NS_INSTANTIATE_DECODE_QD(T, BS, false, 64)

// Two-level merge kernels (16-bit pools, head_dim 64).
#define NS_INSTANTIATE_DECODE_TWO_G(T, BS, G) \
    template cudaError_t launch_paged_decode<T, BS, G, false, 64, true>(const DecodeParams &, int, cudaStream_t);
#define NS_INSTANTIATE_DECODE_TWO(T, BS)  \
    NS_INSTANTIATE_DECODE_TWO_G(T, BS, 1) \
    NS_INSTANTIATE_DECODE_TWO_G(T, BS, 2) \
    NS_INSTANTIATE_DECODE_TWO_G(T, BS, 3) \
    NS_INSTANTIATE_DECODE_TWO_G(T, BS, 4) \
    NS_INSTANTIATE_DECODE_TWO_G(T, BS, 5) \
    NS_INSTANTIATE_DECODE_TWO_G(T, BS, 6) \
    NS_INSTANTIATE_DECODE_TWO_G(T, BS, 7) \
    NS_INSTANTIATE_DECODE_TWO_G(T, BS, 8)
#define NS_INSTANTIATE_DECODE_Q(T, BS, Q8) NS_INSTANTIATE_DECODE_QD(T, BS, Q8, 64)

// Short-walk kernels (16-bit pools, head_dim 64): the values pass unrolled
// kShortWalkValuesUnroll row groups a trip, for less code to fetch when each
// worker runs few steps.
#define NS_INSTANTIATE_DECODE_SHORT_G(T, BS, G)                                                    \
    template cudaError_t launch_paged_decode<T, BS, G, false, 64, false, kShortWalkValuesUnroll>( \
        const DecodeParams &, int, cudaStream_t);
#define NS_INSTANTIATE_DECODE_SHORT(T, BS)  \
    NS_INSTANTIATE_DECODE_SHORT_G(T, BS, 1) \
    NS_INSTANTIATE_DECODE_SHORT_G(T, BS, 2) \
    NS_INSTANTIATE_DECODE_SHORT_G(T, BS, 3) \
    NS_INSTANTIATE_DECODE_SHORT_G(T, BS, 4) \
    NS_INSTANTIATE_DECODE_SHORT_G(T, BS, 5) \
    NS_INSTANTIATE_DECODE_SHORT_G(T, BS, 6) \
    NS_INSTANTIATE_DECODE_SHORT_G(T, BS, 7) \
    NS_INSTANTIATE_DECODE_SHORT_G(T, BS, 8)

}  // namespace ns
