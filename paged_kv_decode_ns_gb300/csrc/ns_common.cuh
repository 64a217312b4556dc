// ns_common.cuh -- device helpers shared by the sm_103a kernels of the
// paged-KV library: mbarrier waits with a time limit, TMA bulk copies,
// fp16/bf16 unpacking, packed fp32 arithmetic and the device status word.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ns_paged.h"

namespace ns {

constexpr int kHeadDim = 64;          // supported head_dim
constexpr int kMaxGroup = 8;          // query heads per KV head, at most
constexpr int kRowBytes = kHeadDim * 2;  // one token row of one head (fp16/bf16)

// Wall-clock limit of every wait inside a kernel (nanoseconds).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

struct F16 {
    static constexpr ns_dtype code = NS_F16;
};
struct BF16 {
    static constexpr ns_dtype code = NS_BF16;
};

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void raise_status(unsigned *status, unsigned bits)
{
    atomicOr(status, bits);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Generic-proxy accesses to shared memory are ordered with later async-proxy
// (TMA / tensor core) accesses to it.
__device__ __forceinline__ void fence_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Warpgroup-wide register reallocation (every warp of the warpgroup executes it).
template <int N>
__device__ __forceinline__ void regs_grow()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_shrink()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Programmatic dependent launch: wait for the previous grid on the stream
// (complete, memory visible) / let the next one be scheduled.  Both are
// no-ops for a grid launched without the programmatic attribute.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier among `threads` threads (a multiple of 32) of the CTA on barrier `id`
// (1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_barrier_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ int ld_acquire_cta(const int *p)
{
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_cta(int *p, int v)
{
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

// Non-blocking: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; false after
// limit_ns of waiting (the caller then reports NS_DEV_WAIT_TIMEOUT).
// try_wait may hold the thread inside the instruction for a window the
// hardware picks (microseconds); a limit shorter than the default polls with
// the non-blocking test instead, so that the limit itself is what expires.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs)
{
    if (limit_ns < kWaitLimitNs) {
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_test(bar, parity))
            if (global_timer_ns() - t0 > limit_ns)
                return false;
        return true;
    }
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (global_timer_ns() - t0 > limit_ns)
            return false;
    }
}

// ---------------------------------------------------------------------------
// TMA bulk copy global -> shared (contiguous bytes, 16-byte aligned, size a
// multiple of 16), completing on an mbarrier.  The L2 policy marks the
// streamed K/V as evict-first so they do not push out reused data.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                          uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes"
        " [%0], [%1], %2, [%3];" ::"r"(smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// ---------------------------------------------------------------------------
// Element unpacking: a 32-bit word holding two 16-bit elements -> two floats
// (exact for every finite value).
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w);

template <>
__device__ __forceinline__ float2 unpack2<BF16>(uint32_t w)
{
    // bf16 is the upper half of a binary32.  Byte permutes (ALU pipe) rather
    // than a shift, which may be issued on the FMA pipe that the packed FMAs
    // keep busy (measured 1% faster on the batch-256 decode).
    uint32_t lo, hi;
    asm("prmt.b32 %0, %1, 0, 0x1044;" : "=r"(lo) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0x3244;" : "=r"(hi) : "r"(w));
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}

template <>
__device__ __forceinline__ float2 unpack2<F16>(uint32_t w)
{
    __half2 h;
    *reinterpret_cast<uint32_t *>(&h) = w;
    return __half22float2(h);
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);

template <>
__device__ __forceinline__ uint32_t pack2<BF16>(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <>
__device__ __forceinline__ uint32_t pack2<F16>(float a, float b)
{
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <typename T>
__device__ __forceinline__ uint16_t pack1(float a);

template <>
__device__ __forceinline__ uint16_t pack1<BF16>(float a)
{
    __nv_bfloat16 h = __float2bfloat16_rn(a);
    return *reinterpret_cast<uint16_t *>(&h);
}

template <>
__device__ __forceinline__ uint16_t pack1<F16>(float a)
{
    __half h = __float2half_rn(a);
    return *reinterpret_cast<uint16_t *>(&h);
}

// Packed fp32 (two lanes per instruction on sm_100-class GPUs).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 lds128(const void *p)
{
    return *reinterpret_cast<const uint4 *>(p);
}

}  // namespace ns
