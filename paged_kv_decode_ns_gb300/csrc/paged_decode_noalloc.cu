// paged_decode_noalloc.cu -- the split-KV decode with library-owned scratch,
// for callers that cannot allocate device memory.
//
// ns_paged_attn_decode needs a caller-provided workspace (split-KV partial
// records, one arrival counter per (sequence, kv head) and a plan record).
// Some callers cannot call cudaMalloc or a caching allocator: plugins
// embedded in a host runtime that owns every device allocation, and serving
// loops that forbid allocation after start-up.  This file gives them
// ns_paged_attn_decode_noalloc, which runs the same kernel (and grid) over a
// fixed-size scratch array that lives in the library image itself.
//
// The scratch is a file-scope __device__ array: every GPU that loads the
// library holds it (about 8.7 MB) until the process exits.  Host code cannot
// use the array's name as a device address, so the first call on each device
// asks the runtime for that device's address (cudaGetSymbolAddress) with the
// device current, checks the result and caches it.  Every call shares the one
// array: calls that
// overlap on the GPU (two streams, two threads) race and give wrong results.
// The arrival counters must start at zero, so each call clears them with
// cudaMemsetAsync on its own stream before the kernel; the partial records need
// no clearing.
#include <atomic>
#include <cmath>
#include <cstring>

#include "ns_internal.h"
#include "paged_decode.cuh"

namespace {

constexpr size_t kPlanBytes = 256;
constexpr size_t kCounterBytes = (size_t)NS_NOALLOC_MAX_PAIRS * sizeof(int32_t);
constexpr size_t kPartialBytes = (size_t)ns::kMaxWorkers * 2 * ns::slot_floats(64) * sizeof(float);
constexpr size_t kScratchBytes = kPlanBytes + kCounterBytes + kPartialBytes;

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<unsigned char *> g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on device `dev` (which must be current).
unsigned char *scratch_address(int dev)
{
    unsigned char *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess || a == nullptr)
            return nullptr;
        p = static_cast<unsigned char *>(a);
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace

extern "C" ns_status ns_paged_attn_decode_noalloc(const void *q, const void *k_pool,
                                                  const void *v_pool, const int32_t *block_tables,
                                                  const int32_t *context_lens, int num_seqs,
                                                  int num_q_heads, int num_kv_heads, int head_dim,
                                                  int block_size, float scale, void *out,
                                                  ns_stream_t stream, int max_blocks_per_seq,
                                                  int64_t num_blocks, ns_dtype dtype)
{
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0)
        return NS_ERR_INVALID_ARG;
    if (dtype != NS_F16 && dtype != NS_BF16)
        return NS_ERR_UNSUPPORTED;
    if (head_dim != ns::kHeadDim ||
        (block_size != 4 && block_size != 8 && block_size != 16 && block_size != 32) ||
        num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > ns::kMaxGroup)
        return NS_ERR_UNSUPPORTED;
    // the scratch array holds one arrival counter per (sequence, kv head)
    if ((long long)num_seqs * num_kv_heads > NS_NOALLOC_MAX_PAIRS)
        return NS_ERR_UNSUPPORTED;
    if (num_seqs == 0)
        return NS_OK;
    const auto aligned = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out)
        return NS_ERR_INVALID_ARG;
    if (!aligned(q) || !aligned(k_pool) || !aligned(v_pool) || !aligned(out))
        return NS_ERR_INVALID_ARG;
    if (max_blocks_per_seq < 1 || num_blocks < 1 || !std::isfinite(scale))
        return NS_ERR_INVALID_ARG;
    if (!ns::split_fits(num_seqs, num_kv_heads, max_blocks_per_seq))
        return NS_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return NS_ERR_CUDA;
    unsigned char *scratch = scratch_address(dev);
    unsigned *status = ns::device_status_word(dev);
    if (scratch == nullptr || status == nullptr)
        return NS_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int *counters = reinterpret_cast<int *>(scratch + kPlanBytes);
    if (cudaMemsetAsync(counters, 0, (size_t)num_seqs * num_kv_heads * sizeof(int32_t), st) !=
        cudaSuccess)
        return NS_ERR_CUDA;

    ns::DecodeParams P;
    std::memset(&P, 0, sizeof(P));
    P.q = static_cast<const uint16_t *>(q);
    P.k_pool = static_cast<const uint16_t *>(k_pool);
    P.v_pool = static_cast<const uint16_t *>(v_pool);
    P.block_tables = block_tables;
    P.context_lens = context_lens;
    P.out = static_cast<uint16_t *>(out);
    P.num_seqs = num_seqs;
    P.num_q_heads = num_q_heads;
    P.num_kv_heads = num_kv_heads;
    P.group = num_q_heads / num_kv_heads;
    P.max_blocks_per_seq = max_blocks_per_seq;
    P.num_blocks = num_blocks;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.counters = counters;
    P.partials = reinterpret_cast<float *>(scratch + kPlanBytes + kCounterBytes);
    P.plan = reinterpret_cast<ns_decode_plan *>(scratch);
    P.status = status;
    P.min_blocks_per_cta = ns::kDefaultMinBlocksPerCta;
    P.whole_sequences = 0;
    P.auto_policy = 1;
    P.wait_limit_ns = ns::kWaitLimitNs;
    P.kv_sub = 1;  // groups of at most ns::kMaxGroup heads only

    return ns::launch_decode(P, dtype, block_size, 0, st, dev);
}
