// ns_api.cu -- the C ABI (include/ns_paged.h): argument checks, workspace
// layout, kernel dispatch and the device status word.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "ns_internal.h"
#include "paged_decode.cuh"

namespace {

// OR of NS_DEV_* bits raised by the kernels (one word per device).
__device__ unsigned int g_device_status;

constexpr int kMaxDevices = 64;
constexpr int kMaxLargeGroup = 64;  // query heads per kv head (above ns::kMaxGroup: virtual kv heads)
std::atomic<unsigned *> g_status_ptr[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_ctas_per_sm[kMaxDevices][2][4][ns::kMaxGroup];
std::atomic<int> g_ctas_per_sm_q8[kMaxDevices][2][ns::kMaxGroup];
std::atomic<int> g_ctas_per_sm_d128[kMaxDevices][2][ns::kMaxGroup];

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int bs_index(int bs)
{
    switch (bs) {
    case 4: return 0;
    case 8: return 1;
    case 16: return 2;
    case 32: return 3;
    default: return -1;
    }
}

cudaError_t current_device(int *dev)
{
    cudaError_t e = cudaGetDevice(dev);
    if (e == cudaSuccess && (*dev < 0 || *dev >= kMaxDevices))
        e = cudaErrorInvalidDevice;
    return e;
}

unsigned *status_word(int dev)
{
    unsigned *p = g_status_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_device_status) != cudaSuccess)
            return nullptr;
        p = static_cast<unsigned *>(a);
        g_status_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

int sm_count(int dev)
{
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

template <typename T, int BS>
cudaError_t dispatch_decode_g(int g, const ns::DecodeParams &P, int ctas, cudaStream_t s)
{
    switch (g) {
    case 1: return ns::launch_paged_decode<T, BS, 1>(P, ctas, s);
    case 2: return ns::launch_paged_decode<T, BS, 2>(P, ctas, s);
    case 3: return ns::launch_paged_decode<T, BS, 3>(P, ctas, s);
    case 4: return ns::launch_paged_decode<T, BS, 4>(P, ctas, s);
    case 5: return ns::launch_paged_decode<T, BS, 5>(P, ctas, s);
    case 6: return ns::launch_paged_decode<T, BS, 6>(P, ctas, s);
    case 7: return ns::launch_paged_decode<T, BS, 7>(P, ctas, s);
    default: return ns::launch_paged_decode<T, BS, 8>(P, ctas, s);
    }
}

// Two-level merge kernels: block size 16, head_dim 64, 16-bit pools.
template <typename T>
cudaError_t dispatch_decode_two(int g, const ns::DecodeParams &P, int ctas, cudaStream_t s)
{
    switch (g) {
    case 1: return ns::launch_paged_decode<T, 16, 1, false, 64, true>(P, ctas, s);
    case 2: return ns::launch_paged_decode<T, 16, 2, false, 64, true>(P, ctas, s);
    case 3: return ns::launch_paged_decode<T, 16, 3, false, 64, true>(P, ctas, s);
    case 4: return ns::launch_paged_decode<T, 16, 4, false, 64, true>(P, ctas, s);
    case 5: return ns::launch_paged_decode<T, 16, 5, false, 64, true>(P, ctas, s);
    case 6: return ns::launch_paged_decode<T, 16, 6, false, 64, true>(P, ctas, s);
    case 7: return ns::launch_paged_decode<T, 16, 7, false, 64, true>(P, ctas, s);
    default: return ns::launch_paged_decode<T, 16, 8, false, 64, true>(P, ctas, s);
    }
}

// Short-walk kernels: block size 16, head_dim 64, 16-bit pools.
template <typename T>
cudaError_t dispatch_decode_short(int g, const ns::DecodeParams &P, int ctas, cudaStream_t s)
{
    constexpr int VU = ns::kShortWalkValuesUnroll;
    switch (g) {
    case 1: return ns::launch_paged_decode<T, 16, 1, false, 64, false, VU>(P, ctas, s);
    case 2: return ns::launch_paged_decode<T, 16, 2, false, 64, false, VU>(P, ctas, s);
    case 3: return ns::launch_paged_decode<T, 16, 3, false, 64, false, VU>(P, ctas, s);
    case 4: return ns::launch_paged_decode<T, 16, 4, false, 64, false, VU>(P, ctas, s);
    case 5: return ns::launch_paged_decode<T, 16, 5, false, 64, false, VU>(P, ctas, s);
    case 6: return ns::launch_paged_decode<T, 16, 6, false, 64, false, VU>(P, ctas, s);
    case 7: return ns::launch_paged_decode<T, 16, 7, false, 64, false, VU>(P, ctas, s);
    default: return ns::launch_paged_decode<T, 16, 8, false, 64, false, VU>(P, ctas, s);
    }
}

template <typename T>
cudaError_t dispatch_decode(int bs, int g, const ns::DecodeParams &P, int ctas, cudaStream_t s)
{
    switch (bs) {
    case 4: return dispatch_decode_g<T, 4>(g, P, ctas, s);
    case 8: return dispatch_decode_g<T, 8>(g, P, ctas, s);
    case 16: return dispatch_decode_g<T, 16>(g, P, ctas, s);
    default: return dispatch_decode_g<T, 32>(g, P, ctas, s);
    }
}

template <typename T, int BS>
int ctas_per_sm_g(int g)
{
    switch (g) {
    case 1: return ns::decode_ctas_per_sm<T, BS, 1>();
    case 2: return ns::decode_ctas_per_sm<T, BS, 2>();
    case 3: return ns::decode_ctas_per_sm<T, BS, 3>();
    case 4: return ns::decode_ctas_per_sm<T, BS, 4>();
    case 5: return ns::decode_ctas_per_sm<T, BS, 5>();
    case 6: return ns::decode_ctas_per_sm<T, BS, 6>();
    case 7: return ns::decode_ctas_per_sm<T, BS, 7>();
    default: return ns::decode_ctas_per_sm<T, BS, 8>();
    }
}

// head_dim 128: block size 16, 16-bit pools.
template <typename T>
cudaError_t dispatch_decode_d128(int g, const ns::DecodeParams &P, int ctas, cudaStream_t s)
{
    switch (g) {
    case 1: return ns::launch_paged_decode<T, 16, 1, false, 128>(P, ctas, s);
    case 2: return ns::launch_paged_decode<T, 16, 2, false, 128>(P, ctas, s);
    case 3: return ns::launch_paged_decode<T, 16, 3, false, 128>(P, ctas, s);
    case 4: return ns::launch_paged_decode<T, 16, 4, false, 128>(P, ctas, s);
    case 5: return ns::launch_paged_decode<T, 16, 5, false, 128>(P, ctas, s);
    case 6: return ns::launch_paged_decode<T, 16, 6, false, 128>(P, ctas, s);
    case 7: return ns::launch_paged_decode<T, 16, 7, false, 128>(P, ctas, s);
    default: return ns::launch_paged_decode<T, 16, 8, false, 128>(P, ctas, s);
    }
}

template <typename T>
int ctas_per_sm_d128(int g)
{
    switch (g) {
    case 1: return ns::decode_ctas_per_sm<T, 16, 1, false, 128>();
    case 2: return ns::decode_ctas_per_sm<T, 16, 2, false, 128>();
    case 3: return ns::decode_ctas_per_sm<T, 16, 3, false, 128>();
    case 4: return ns::decode_ctas_per_sm<T, 16, 4, false, 128>();
    case 5: return ns::decode_ctas_per_sm<T, 16, 5, false, 128>();
    case 6: return ns::decode_ctas_per_sm<T, 16, 6, false, 128>();
    case 7: return ns::decode_ctas_per_sm<T, 16, 7, false, 128>();
    default: return ns::decode_ctas_per_sm<T, 16, 8, false, 128>();
    }
}

// q8_0 pools: block size 16 only.
template <typename T>
cudaError_t dispatch_decode_q8(int g, const ns::DecodeParams &P, int ctas, cudaStream_t s)
{
    switch (g) {
    case 1: return ns::launch_paged_decode<T, 16, 1, true>(P, ctas, s);
    case 2: return ns::launch_paged_decode<T, 16, 2, true>(P, ctas, s);
    case 3: return ns::launch_paged_decode<T, 16, 3, true>(P, ctas, s);
    case 4: return ns::launch_paged_decode<T, 16, 4, true>(P, ctas, s);
    case 5: return ns::launch_paged_decode<T, 16, 5, true>(P, ctas, s);
    case 6: return ns::launch_paged_decode<T, 16, 6, true>(P, ctas, s);
    case 7: return ns::launch_paged_decode<T, 16, 7, true>(P, ctas, s);
    default: return ns::launch_paged_decode<T, 16, 8, true>(P, ctas, s);
    }
}

template <typename T>
int ctas_per_sm_q8(int g)
{
    switch (g) {
    case 1: return ns::decode_ctas_per_sm<T, 16, 1, true>();
    case 2: return ns::decode_ctas_per_sm<T, 16, 2, true>();
    case 3: return ns::decode_ctas_per_sm<T, 16, 3, true>();
    case 4: return ns::decode_ctas_per_sm<T, 16, 4, true>();
    case 5: return ns::decode_ctas_per_sm<T, 16, 5, true>();
    case 6: return ns::decode_ctas_per_sm<T, 16, 6, true>();
    case 7: return ns::decode_ctas_per_sm<T, 16, 7, true>();
    default: return ns::decode_ctas_per_sm<T, 16, 8, true>();
    }
}

template <typename T>
int dispatch_ctas_per_sm(int bs, int g)
{
    switch (bs) {
    case 4: return ctas_per_sm_g<T, 4>(g);
    case 8: return ctas_per_sm_g<T, 8>(g);
    case 16: return ctas_per_sm_g<T, 16>(g);
    default: return ctas_per_sm_g<T, 32>(g);
    }
}

int resident_ctas(int dev, ns_dtype dt, int bs, int g, bool q8, int head_dim)
{
    const int t = dt == NS_BF16 ? 1 : 0;
    std::atomic<int> &slot = q8 ? g_ctas_per_sm_q8[dev][t][g - 1]
                             : head_dim == 128 ? g_ctas_per_sm_d128[dev][t][g - 1]
                                               : g_ctas_per_sm[dev][t][bs_index(bs)][g - 1];
    int n = slot.load(std::memory_order_relaxed);
    if (n <= 0) {
        if (q8)
            n = dt == NS_BF16 ? ctas_per_sm_q8<ns::BF16>(g) : ctas_per_sm_q8<ns::F16>(g);
        else if (head_dim == 128)
            n = dt == NS_BF16 ? ctas_per_sm_d128<ns::BF16>(g) : ctas_per_sm_d128<ns::F16>(g);
        else
            n = dt == NS_BF16 ? dispatch_ctas_per_sm<ns::BF16>(bs, g) : dispatch_ctas_per_sm<ns::F16>(bs, g);
        slot.store(n, std::memory_order_relaxed);
    }
    long long total = (long long)n * sm_count(dev);
    return (int)(total > NS_MAX_CTAS ? NS_MAX_CTAS : total);
}

// Workspace layout (byte offsets), for up to `rows` query rows.
struct WsLayout {
    size_t plan, counters, partials, row_seq, row_len, total;
};

// Groups of more than kMaxGroup query heads run as kv_sub groups of G / kv_sub
// heads each (virtual kv heads over the same pool head); 0 when G cannot be
// cut so (G not a multiple of ceil(G / kMaxGroup)), 1 for G <= kMaxGroup.
int kv_sub(int num_q_heads, int num_kv_heads)
{
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return 1;
    const int g = num_q_heads / num_kv_heads;
    const int sub = (g + ns::kMaxGroup - 1) / ns::kMaxGroup;
    return g % sub == 0 ? sub : 0;
}

WsLayout ws_layout(long long rows, int num_kv_heads, int head_dim)
{
    WsLayout L;
    L.plan = 0;
    L.counters = 256;
    L.partials = L.counters + align256((size_t)rows * num_kv_heads * sizeof(int32_t));
    L.row_seq = L.partials + align256((size_t)ns::kMaxWorkers * 2 * ns::slot_floats(head_dim) * sizeof(float));
    L.row_len = L.row_seq + align256((size_t)rows * sizeof(int32_t));
    L.total = L.row_len + align256((size_t)rows * sizeof(int32_t));
    return L;
}

ns_status check_shapes(int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       ns_dtype dtype)
{
    if (num_q_heads <= 0 || num_kv_heads <= 0)
        return NS_ERR_INVALID_ARG;
    if (dtype != NS_F16 && dtype != NS_BF16)
        return NS_ERR_UNSUPPORTED;
    if ((head_dim != 64 && head_dim != 128) || bs_index(block_size) < 0)
        return NS_ERR_UNSUPPORTED;
    if (head_dim == 128 && block_size != 16)
        return NS_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > kMaxLargeGroup ||
        kv_sub(num_q_heads, num_kv_heads) == 0)
        return NS_ERR_UNSUPPORTED;
    return NS_OK;
}

struct DecodeCall {
    const void *q;
    const void *k_pool;
    const void *v_pool;
    const int32_t *block_tables;
    const int32_t *lens;       // per row
    const int32_t *table_row;  // nullptr: identity
    int rows;
    int num_q_heads, num_kv_heads, block_size;
    float scale;
    void *out;
    cudaStream_t stream;
    int max_blocks_per_seq;
    long long num_blocks;
    ns_dtype dtype;
    void *workspace;
    const ns_decode_config *cfg;
    const void *k_new, *v_new;
    const int64_t *slot_mapping;
    bool pack = false;  // keep the workers on the fewest CTAs (another kernel waits for the SMs)
    bool fixed_split = false;  // default blocks per worker, no automatic finer cut
    int max_ctas = 0;          // > 0: at most this many CTAs (fewer than one per SM)
    // q8_0 pools (k_pool and v_pool unused then)
    bool q8 = false;
    const void *k_codes = nullptr, *k_scales = nullptr, *v_codes = nullptr, *v_scales = nullptr;
    int head_dim = 64;
};

ns_status run_decode(const DecodeCall &c, int dev)
{
    unsigned *status = status_word(dev);
    if (status == nullptr)
        return NS_ERR_CUDA;
    const int sub = kv_sub(c.num_q_heads, c.num_kv_heads);
    const WsLayout L = ws_layout(c.rows, c.num_kv_heads * sub, c.head_dim);
    char *ws = static_cast<char *>(c.workspace);

    ns::DecodeParams P;
    std::memset(&P, 0, sizeof(P));
    P.q = static_cast<const uint16_t *>(c.q);
    P.k_pool = static_cast<const uint16_t *>(c.k_pool);
    P.v_pool = static_cast<const uint16_t *>(c.v_pool);
    P.block_tables = c.block_tables;
    P.context_lens = c.lens;
    P.table_row = c.table_row;
    P.out = static_cast<uint16_t *>(c.out);
    P.k_new = static_cast<const uint16_t *>(c.k_new);
    P.v_new = static_cast<const uint16_t *>(c.v_new);
    P.slot_mapping = c.slot_mapping;
    P.k_pool_w = const_cast<uint16_t *>(static_cast<const uint16_t *>(c.k_pool));
    P.v_pool_w = const_cast<uint16_t *>(static_cast<const uint16_t *>(c.v_pool));
    P.num_seqs = c.rows;
    P.num_q_heads = c.num_q_heads;
    P.num_kv_heads = c.num_kv_heads * sub;  // virtual kv heads
    P.group = c.num_q_heads / P.num_kv_heads;
    P.kv_sub = sub;
    P.max_blocks_per_seq = c.max_blocks_per_seq;
    P.num_blocks = c.num_blocks;
    P.scale_log2 = c.scale * 1.4426950408889634f;
    P.counters = reinterpret_cast<int *>(ws + L.counters);
    P.partials = reinterpret_cast<float *>(ws + L.partials);
    P.plan = reinterpret_cast<ns_decode_plan *>(ws + L.plan);
    P.status = status;
    P.min_blocks_per_cta = (c.cfg && c.cfg->min_blocks_per_cta > 0) ? c.cfg->min_blocks_per_cta
                                                                     : ns::kDefaultMinBlocksPerCta;
    P.whole_sequences = (c.cfg && c.cfg->whole_sequences) ? 1 : 0;
    P.overlap = (c.cfg && c.cfg->overlap_prologue) ? 1 : 0;
    P.pack = c.pack ? 1 : 0;
    P.wait_limit_ns = (c.cfg && c.cfg->wait_limit_ns > 0) ? (unsigned long long)c.cfg->wait_limit_ns
                                                           : ns::kWaitLimitNs;
    P.merge_levels = c.cfg ? c.cfg->merge_levels : 0;
    P.k_codes = static_cast<const int8_t *>(c.k_codes);
    P.v_codes = static_cast<const int8_t *>(c.v_codes);
    P.k_scales = static_cast<const uint16_t *>(c.k_scales);
    P.v_scales = static_cast<const uint16_t *>(c.v_scales);
    P.auto_policy = (!c.fixed_split && (c.cfg == nullptr || (c.cfg->num_ctas == 0 && c.cfg->min_blocks_per_cta == 0 &&
                                                             c.cfg->whole_sequences == 0)))
                        ? 1
                        : 0;

    int num_ctas = c.cfg ? c.cfg->num_ctas : 0;
    if (num_ctas == 0 && c.max_ctas > 0) {
        num_ctas = std::min(c.max_ctas, resident_ctas(dev, c.dtype, c.block_size, P.group, c.q8, c.head_dim));
    }
    return ns::launch_decode(P, c.dtype, c.block_size, num_ctas, c.stream, dev, c.q8, c.head_dim);
}

ns_status check_decode_args(const void *q, const void *k_pool, const void *v_pool,
                            const int32_t *block_tables, const int32_t *context_lens, int rows,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            float scale, void *out, int max_blocks_per_seq, int64_t num_blocks,
                            ns_dtype dtype, void *workspace, size_t workspace_bytes,
                            const ns_decode_config *cfg)
{
    if (rows < 0)
        return NS_ERR_INVALID_ARG;
    const ns_status s = check_shapes(num_q_heads, num_kv_heads, head_dim, block_size, dtype);
    if (s != NS_OK)
        return s;
    if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out || !workspace)
        return NS_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
        !aligned16(workspace))
        return NS_ERR_INVALID_ARG;
    if (max_blocks_per_seq < 1 || num_blocks < 1 || !std::isfinite(scale))
        return NS_ERR_INVALID_ARG;
    if (!ns::split_fits(rows, (long long)num_kv_heads * kv_sub(num_q_heads, num_kv_heads), max_blocks_per_seq))
        return NS_ERR_UNSUPPORTED;
    if (workspace_bytes < ns_paged_attn_workspace_bytes(rows, num_q_heads, num_kv_heads, head_dim))
        return NS_ERR_INVALID_ARG;
    if (cfg && (cfg->num_ctas < 0 || cfg->num_ctas > NS_MAX_CTAS || cfg->min_blocks_per_cta < 0 ||
                cfg->wait_limit_ns < 0 || cfg->merge_levels < 0 || cfg->merge_levels > 2))
        return NS_ERR_INVALID_ARG;
    return NS_OK;
}

}  // namespace

namespace ns {

ns_status launch_decode(const DecodeParams &P, ns_dtype dtype, int block_size, int num_ctas,
                        cudaStream_t stream, int dev, bool q8, int head_dim)
{
    const int g = P.group;
    int ctas = num_ctas > 0 ? num_ctas : resident_ctas(dev, dtype, block_size, g, q8, head_dim);
    if (ctas > NS_MAX_CTAS)
        ctas = NS_MAX_CTAS;
    // Two-level merges where a cut pair has many pieces in each CTA: few
    // pairs for the CTAs' warps (at least 32 warps a pair) that could fill
    // them (the pairs' table rows span at least a block a warp).
    bool two = false, shortw = false;
    if (head_dim == 64 && !q8 && block_size == 16) {
        const long long pairs = (long long)P.num_seqs * P.num_kv_heads, warps = (long long)ctas * kConsumerWarps;
        two = P.merge_levels == 2 ||
              (P.merge_levels == 0 && pairs * 32 <= warps && pairs * P.max_blocks_per_seq >= warps);
        // Short walks: when the pairs' table rows bound every worker's share at
        // 16 blocks (8 steps), the kernel with the values pass looped.
        shortw = !two && pairs * (P.max_blocks_per_seq + kPieceCost) <= 16 * warps;
    }
    cudaError_t e;
    if (two)
        e = dtype == NS_BF16 ? dispatch_decode_two<BF16>(g, P, ctas, stream) : dispatch_decode_two<F16>(g, P, ctas, stream);
    else if (head_dim == 128)
        e = dtype == NS_BF16 ? dispatch_decode_d128<BF16>(g, P, ctas, stream)
                             : dispatch_decode_d128<F16>(g, P, ctas, stream);
    else if (q8)
        e = dtype == NS_BF16 ? dispatch_decode_q8<BF16>(g, P, ctas, stream) : dispatch_decode_q8<F16>(g, P, ctas, stream);
    else if (shortw)
        e = dtype == NS_BF16 ? dispatch_decode_short<BF16>(g, P, ctas, stream)
                             : dispatch_decode_short<F16>(g, P, ctas, stream);
    else
        e = dtype == NS_BF16 ? dispatch_decode<BF16>(block_size, g, P, ctas, stream)
                             : dispatch_decode<F16>(block_size, g, P, ctas, stream);
    return e == cudaSuccess ? NS_OK : NS_ERR_CUDA;
}

}  // namespace ns

unsigned *ns::device_status_word(int dev)
{
    return (dev >= 0 && dev < kMaxDevices) ? status_word(dev) : nullptr;
}

namespace {

ns_status decode_q8_0(const void *q, const void *k_new, const void *v_new, const int64_t *slot_mapping,
                      const void *k_codes, const void *k_scales, const void *v_codes, const void *v_scales,
                      const int32_t *block_tables, const int32_t *context_lens, int num_seqs, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size, float scale, void *out,
                      ns_stream_t stream, int max_blocks_per_seq, int64_t num_blocks, ns_dtype dtype,
                      void *workspace, size_t workspace_bytes, const ns_decode_config *cfg)
{
    if (!k_codes || !k_scales || !v_codes || !v_scales)
        return NS_ERR_INVALID_ARG;
    const ns_status s = check_decode_args(q, k_codes, v_codes, block_tables, context_lens, num_seqs, num_q_heads,
                                          num_kv_heads, head_dim, block_size, scale, out, max_blocks_per_seq,
                                          num_blocks, dtype, workspace, workspace_bytes, cfg);
    if (s != NS_OK)
        return s;
    if (block_size != 16 || head_dim != 64)
        return NS_ERR_UNSUPPORTED;
    if (!aligned16(k_scales) || !aligned16(v_scales))
        return NS_ERR_INVALID_ARG;
    if (num_seqs == 0)
        return NS_OK;
    if (k_new && (!v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new)))
        return NS_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != cudaSuccess)
        return NS_ERR_CUDA;
    DecodeCall c{q, nullptr, nullptr, block_tables, context_lens, nullptr, num_seqs, num_q_heads, num_kv_heads,
                 block_size, scale, out, reinterpret_cast<cudaStream_t>(stream), max_blocks_per_seq, num_blocks,
                 dtype, workspace, cfg, k_new, v_new, k_new ? slot_mapping : nullptr};
    c.q8 = true;
    c.head_dim = head_dim;
    c.k_codes = k_codes;
    c.k_scales = k_scales;
    c.v_codes = v_codes;
    c.v_scales = v_scales;
    return run_decode(c, dev);
}

}  // namespace

extern "C" {

const char *ns_status_string(ns_status status)
{
    switch (status) {
    case NS_OK: return "NS_OK";
    case NS_ERR_INVALID_ARG: return "NS_ERR_INVALID_ARG: invalid argument";
    case NS_ERR_UNSUPPORTED: return "NS_ERR_UNSUPPORTED: shape or type not supported";
    case NS_ERR_CUDA: return "NS_ERR_CUDA: CUDA call or launch failed";
    case NS_ERR_DEVICE: return "NS_ERR_DEVICE: a kernel raised a device status bit";
    default: return "unknown ns_status";
    }
}

int ns_version(void) { return 100; }

ns_status ns_kv_append(const void *k, const void *v, const int64_t *slot_mapping, void *k_pool,
                       void *v_pool, int num_tokens, int num_kv_heads, int head_dim,
                       int block_size, int64_t num_blocks, ns_dtype dtype, ns_stream_t stream)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks < 1)
        return NS_ERR_INVALID_ARG;
    if (dtype != NS_F16 && dtype != NS_BF16)
        return NS_ERR_UNSUPPORTED;
    if ((head_dim != 64 && head_dim != 128) || bs_index(block_size) < 0)
        return NS_ERR_UNSUPPORTED;
    if (head_dim == 128 && block_size != 16)
        return NS_ERR_UNSUPPORTED;
    if (num_tokens == 0)
        return NS_OK;
    if (!k || !v || !slot_mapping || !k_pool || !v_pool)
        return NS_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool))
        return NS_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != cudaSuccess)
        return NS_ERR_CUDA;
    unsigned *status = status_word(dev);
    if (status == nullptr)
        return NS_ERR_CUDA;
    const cudaError_t e = ns::launch_kv_append(k, v, slot_mapping, k_pool, v_pool, num_tokens,
                                               num_kv_heads, head_dim, block_size, num_blocks, status,
                                               reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NS_OK : NS_ERR_CUDA;
}

size_t ns_paged_attn_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim)
{
    (void)num_q_heads;
    if (num_seqs < 0 || num_kv_heads <= 0)
        return 0;
    const int sub = kv_sub(num_q_heads, num_kv_heads);
    return ws_layout(num_seqs, num_kv_heads * (sub > 0 ? sub : 1), head_dim == 128 ? 128 : 64).total;
}

ns_status ns_paged_attn_workspace_init(void *workspace, size_t workspace_bytes, ns_stream_t stream)
{
    if (!workspace)
        return NS_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? NS_OK
               : NS_ERR_CUDA;
}

ns_status ns_paged_attn_decode_ex(const void *q, const void *k_pool, const void *v_pool,
                                  const int32_t *block_tables, const int32_t *context_lens,
                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, float scale, void *out, ns_stream_t stream,
                                  int max_blocks_per_seq, int64_t num_blocks, ns_dtype dtype,
                                  void *workspace, size_t workspace_bytes,
                                  const ns_decode_config *cfg)
{
    const ns_status s = check_decode_args(q, k_pool, v_pool, block_tables, context_lens, num_seqs,
                                          num_q_heads, num_kv_heads, head_dim, block_size, scale,
                                          out, max_blocks_per_seq, num_blocks, dtype, workspace,
                                          workspace_bytes, cfg);
    if (s != NS_OK)
        return s;
    if (num_seqs == 0)
        return NS_OK;
    int dev = 0;
    if (current_device(&dev) != cudaSuccess)
        return NS_ERR_CUDA;
    DecodeCall c{q, k_pool, v_pool, block_tables, context_lens, nullptr, num_seqs, num_q_heads,
                 num_kv_heads, block_size, scale, out, reinterpret_cast<cudaStream_t>(stream),
                 max_blocks_per_seq, num_blocks, dtype, workspace, cfg, nullptr, nullptr, nullptr};
    c.head_dim = head_dim;
    return run_decode(c, dev);
}

ns_status ns_paged_attn_decode(const void *q, const void *k_pool, const void *v_pool,
                               const int32_t *block_tables, const int32_t *context_lens,
                               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, float scale, void *out, ns_stream_t stream,
                               int max_blocks_per_seq, int64_t num_blocks, ns_dtype dtype,
                               void *workspace, size_t workspace_bytes)
{
    return ns_paged_attn_decode_ex(q, k_pool, v_pool, block_tables, context_lens, num_seqs,
                                   num_q_heads, num_kv_heads, head_dim, block_size, scale, out,
                                   stream, max_blocks_per_seq, num_blocks, dtype, workspace,
                                   workspace_bytes, nullptr);
}

ns_status ns_kv_append_paged_attn_decode(const void *q, const void *k_new, const void *v_new,
                                         const int64_t *slot_mapping, void *k_pool,
                                         void *v_pool, const int32_t *block_tables,
                                         const int32_t *context_lens, int num_seqs,
                                         int num_q_heads, int num_kv_heads, int head_dim,
                                         int block_size, float scale, void *out,
                                         ns_stream_t stream, int max_blocks_per_seq,
                                         int64_t num_blocks, ns_dtype dtype, void *workspace,
                                         size_t workspace_bytes)
{
    return ns_kv_append_paged_attn_decode_ex(q, k_new, v_new, slot_mapping, k_pool, v_pool,
                                             block_tables, context_lens, num_seqs, num_q_heads,
                                             num_kv_heads, head_dim, block_size, scale, out, stream,
                                             max_blocks_per_seq, num_blocks, dtype, workspace,
                                             workspace_bytes, nullptr);
}

ns_status ns_kv_append_paged_attn_decode_ex(const void *q, const void *k_new, const void *v_new,
                                            const int64_t *slot_mapping, void *k_pool,
                                            void *v_pool, const int32_t *block_tables,
                                            const int32_t *context_lens, int num_seqs,
                                            int num_q_heads, int num_kv_heads, int head_dim,
                                            int block_size, float scale, void *out,
                                            ns_stream_t stream, int max_blocks_per_seq,
                                            int64_t num_blocks, ns_dtype dtype, void *workspace,
                                            size_t workspace_bytes, const ns_decode_config *cfg)
{
    const ns_status s = check_decode_args(q, k_pool, v_pool, block_tables, context_lens, num_seqs,
                                          num_q_heads, num_kv_heads, head_dim, block_size, scale,
                                          out, max_blocks_per_seq, num_blocks, dtype, workspace,
                                          workspace_bytes, cfg);
    if (s != NS_OK)
        return s;
    if (num_seqs == 0)
        return NS_OK;
    if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new))
        return NS_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != cudaSuccess)
        return NS_ERR_CUDA;
    DecodeCall c{q, k_pool, v_pool, block_tables, context_lens, nullptr, num_seqs, num_q_heads,
                 num_kv_heads, block_size, scale, out, reinterpret_cast<cudaStream_t>(stream),
                 max_blocks_per_seq, num_blocks, dtype, workspace, cfg, k_new, v_new,
                 slot_mapping};
    c.head_dim = head_dim;
    return run_decode(c, dev);
}

ns_status ns_read_decode_plan(const void *workspace, ns_decode_plan *plan, ns_stream_t stream)
{
    if (!workspace || !plan)
        return NS_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(plan, workspace, sizeof(ns_decode_plan), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return NS_ERR_CUDA;
    return NS_OK;
}

ns_status ns_paged_attn_prefill_ex(const void *q, const int32_t *query_start_loc,
                                   const void *k_pool, const void *v_pool,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   int num_seqs, int total_q_tokens, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size, float scale,
                                   void *out, ns_stream_t stream, int max_blocks_per_seq,
                                   int64_t num_blocks, ns_dtype dtype, void *workspace,
                                   size_t workspace_bytes, const ns_prefill_config *cfg)
{
    if (num_seqs < 0 || total_q_tokens < 0 || !query_start_loc)
        return NS_ERR_INVALID_ARG;
    const ns_status s = check_decode_args(q, k_pool, v_pool, block_tables, context_lens,
                                          total_q_tokens, num_q_heads, num_kv_heads, head_dim,
                                          block_size, scale, out, max_blocks_per_seq, num_blocks,
                                          dtype, workspace, workspace_bytes, nullptr);
    if (s != NS_OK)
        return s;
    if (total_q_tokens == 0 || num_seqs == 0)
        return NS_OK;
    int dev = 0;
    if (current_device(&dev) != cudaSuccess)
        return NS_ERR_CUDA;
    unsigned *status = status_word(dev);
    if (status == nullptr)
        return NS_ERR_CUDA;
    const WsLayout L = ws_layout(total_q_tokens, num_kv_heads * kv_sub(num_q_heads, num_kv_heads), head_dim);
    char *ws = static_cast<char *>(workspace);
    int32_t *row_seq = reinterpret_cast<int32_t *>(ws + L.row_seq);
    int32_t *row_len = reinterpret_cast<int32_t *>(ws + L.row_len);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int tc_min = cfg && cfg->tensor_core_min_span != 0 ? cfg->tensor_core_min_span : 2;
    // Automatic: with no more query tokens than spans, every span has one token
    // unless some are empty, so all rows take the split-KV walk (a longer span
    // beside empty ones as well) and no tensor-core kernel is launched (4
    // single-token spans: 18.4 -> 17.6 us a call, batch 32 24.4 -> 23.2).
    if (!(cfg && cfg->tensor_core_min_span != 0) && total_q_tokens <= num_seqs)
        tc_min = 0;
    if (tc_min < 0 || (head_dim == 128 && block_size != 16) ||
        !ns::tc_prefill_supported(block_size, num_q_heads / num_kv_heads) ||
        (long long)num_blocks * num_kv_heads * block_size > 0x7fffffffLL)
        tc_min = 0;
    const int phases = cfg && cfg->phases != 0 ? cfg->phases : (NS_PREFILL_WALK | NS_PREFILL_TENSOR_CORE);
    if (phases & NS_PREFILL_WALK) {
        if (ns::launch_span_rows(query_start_loc, context_lens, num_seqs, total_q_tokens, tc_min,
                                 row_seq, row_len, status, st) != cudaSuccess)
            return NS_ERR_CUDA;
        DecodeCall c{q, k_pool, v_pool, block_tables, row_len, row_seq, total_q_tokens, num_q_heads,
                     num_kv_heads, block_size, scale, out, st, max_blocks_per_seq, num_blocks, dtype,
                     workspace, nullptr, nullptr, nullptr, nullptr};
        c.head_dim = head_dim;
        // With more query tokens than spans, some span has two or more and the
        // tensor-core kernel after the walk has work: the walk then packs its
        // workers on the fewest CTAs (the tensor-core kernel takes the SMs its
        // idle CTAs leave) and keeps the default blocks per worker. The
        // automatic finer cut spreads a few live rows over every warp of the
        // grid, which holds all SMs and cuts a long row into so many pieces that
        // its merge is the walk's tail (16 decode rows of 103-4096 tokens beside
        // two 512-token chunks: the call 55.3 -> 49.2 us). Otherwise every span
        // has one token (or some are empty) and the walk is split as a decode
        // step is.
        c.pack = total_q_tokens > num_seqs && tc_min != 0 && (phases & NS_PREFILL_TENSOR_CORE) != 0;
        c.fixed_split = c.pack;
        // Its grid is at most one CTA (8 workers) per (span, kv head) pair, so
        // that the tensor-core kernel has the other SMs from the start instead
        // of waiting for idle walk CTAs to leave (the same call: 49.2 -> 43.1
        // us; 32, 48 and 64 walk CTAs alike, 96 47.1 us).
        if (c.pack)
            c.max_ctas = (int)std::min<long long>(
                NS_MAX_CTAS, std::max<long long>(8, (long long)num_seqs * num_kv_heads *
                                                        kv_sub(num_q_heads, num_kv_heads)));
        const ns_status r = run_decode(c, dev);
        if (r != NS_OK)
            return r;
    }
    if (tc_min == 0 || !(phases & NS_PREFILL_TENSOR_CORE))
        return NS_OK;
    return ns::launch_tc_prefill(q, query_start_loc, k_pool, v_pool, block_tables, context_lens,
                                 num_seqs, total_q_tokens, num_q_heads, num_kv_heads, block_size,
                                 scale, out, max_blocks_per_seq, num_blocks, dtype, tc_min, head_dim, status,
                                 (phases & NS_PREFILL_WALK) != 0, st) == cudaSuccess
               ? NS_OK
               : NS_ERR_CUDA;
}

ns_status ns_paged_attn_prefill(const void *q, const int32_t *query_start_loc, const void *k_pool,
                                const void *v_pool, const int32_t *block_tables,
                                const int32_t *context_lens, int num_seqs, int total_q_tokens,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                float scale, void *out, ns_stream_t stream, int max_blocks_per_seq,
                                int64_t num_blocks, ns_dtype dtype, void *workspace,
                                size_t workspace_bytes)
{
    return ns_paged_attn_prefill_ex(q, query_start_loc, k_pool, v_pool, block_tables, context_lens,
                                    num_seqs, total_q_tokens, num_q_heads, num_kv_heads, head_dim,
                                    block_size, scale, out, stream, max_blocks_per_seq, num_blocks,
                                    dtype, workspace, workspace_bytes, nullptr);
}

ns_status ns_kv_append_q8_0(const void *k, const void *v, const int64_t *slot_mapping, void *k_codes,
                            void *k_scales, void *v_codes, void *v_scales, int num_tokens, int num_kv_heads,
                            int head_dim, int block_size, int64_t num_blocks, ns_dtype dtype, ns_stream_t stream)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks < 1)
        return NS_ERR_INVALID_ARG;
    if (dtype != NS_F16 && dtype != NS_BF16)
        return NS_ERR_UNSUPPORTED;
    if (head_dim != ns::kHeadDim || bs_index(block_size) < 0)
        return NS_ERR_UNSUPPORTED;
    if (num_tokens == 0)
        return NS_OK;
    if (!k || !v || !slot_mapping || !k_codes || !k_scales || !v_codes || !v_scales)
        return NS_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_codes) || !aligned16(k_scales) || !aligned16(v_codes) ||
        !aligned16(v_scales))
        return NS_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != cudaSuccess)
        return NS_ERR_CUDA;
    unsigned *status = status_word(dev);
    if (status == nullptr)
        return NS_ERR_CUDA;
    return ns::launch_kv_append_q8(k, v, slot_mapping, k_codes, k_scales, v_codes, v_scales, num_tokens,
                                   num_kv_heads, block_size, num_blocks, dtype, status,
                                   reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? NS_OK
               : NS_ERR_CUDA;
}


ns_status ns_paged_attn_decode_q8_0(const void *q, const void *k_codes, const void *k_scales,
                                   const void *v_codes, const void *v_scales, const int32_t *block_tables,
                                   const int32_t *context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size, float scale, void *out, ns_stream_t stream,
                                   int max_blocks_per_seq, int64_t num_blocks, ns_dtype dtype, void *workspace,
                                   size_t workspace_bytes)
{
    return decode_q8_0(q, nullptr, nullptr, nullptr, k_codes, k_scales, v_codes, v_scales, block_tables,
                       context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, scale, out,
                       stream, max_blocks_per_seq, num_blocks, dtype, workspace, workspace_bytes, nullptr);
}

ns_status ns_kv_append_paged_attn_decode_q8_0(const void *q, const void *k_new, const void *v_new,
                                             const int64_t *slot_mapping, void *k_codes, void *k_scales,
                                             void *v_codes, void *v_scales, const int32_t *block_tables,
                                             const int32_t *context_lens, int num_seqs, int num_q_heads,
                                             int num_kv_heads, int head_dim, int block_size, float scale,
                                             void *out, ns_stream_t stream, int max_blocks_per_seq,
                                             int64_t num_blocks, ns_dtype dtype, void *workspace,
                                             size_t workspace_bytes)
{
    if (!k_new)
        return NS_ERR_INVALID_ARG;
    return decode_q8_0(q, k_new, v_new, slot_mapping, k_codes, k_scales, v_codes, v_scales, block_tables,
                       context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, scale, out,
                       stream, max_blocks_per_seq, num_blocks, dtype, workspace, workspace_bytes, nullptr);
}

ns_status ns_get_device_status(ns_stream_t stream, uint32_t *bits, int clear)
{
    if (!bits)
        return NS_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != cudaSuccess)
        return NS_ERR_CUDA;
    unsigned *p = status_word(dev);
    if (p == nullptr)
        return NS_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned v = 0;
    if (cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return NS_ERR_CUDA;
    if (clear && cudaMemsetAsync(p, 0, sizeof(unsigned), s) != cudaSuccess)
        return NS_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return NS_ERR_CUDA;
    *bits = v;
    return NS_OK;
}

}  // extern "C"
