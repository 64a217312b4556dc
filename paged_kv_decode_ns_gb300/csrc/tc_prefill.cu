// tc_prefill.cu -- chunked-prefill attention on the tcgen05 tensor cores.
//
// What it computes (Inference Engineering Day 12 short, "What is chunked
// prefill within vLLM"; nanoserve project page, "What I built"): query token i
// of a span of n tokens in a sequence of L tokens sits at position L-n+i and
// attends to keys 0..L-n+i -- the cached prefix plus causally within the
// chunk -- through the sequence's block table.
//
// Work unit: (span, kv head, query tile).  A query tile is QT tokens x G query
// heads of one GQA group packed into M = QT*G <= 128 rows (row r = token r/G,
// head r%G), so every K/V tile is loaded once for all heads of the group.
//
//   warp 9   producer: TMA 3D load of the Q tile; per 128-key tile, one TMA 2D
//            load per pool block for K and for V (128-byte swizzle), into a
//            4-stage ring, the next tile's block-table entries read ahead;
//   warp 8   allocates 512 TMEM columns; lane 0 issues the score products
//              S[128x128] = Q K^T   (4 steps of K=16, A and B K-major)
//            as soon as the softmax has read the previous S;
//   warp 10  lane 0 issues the value products
//              O_h[128x64] += P_h V_h (4 steps of K=16 per key half h,
//                                    P read from TMEM, V MN-major)
//            from one of two P buffers, so that neither kind of product
//            waits behind the other's issue (a tile's 8 value products take
//            ~0.7 us to issue, against ~0.15 us for its 4 score products);
//   warps 0-7 softmax: thread t owns row t % 128 (TMEM lane) and key columns
//            64 h .. 64 h + 63 of each tile, h = t / 128.  Each key half has
//            its own running max (moving lazily, by more than 8 in log2 units),
//            sum and O accumulator (TMEM), so the halves never wait on each
//            other; it reads its half of the S row, masks keys past its
//            position, writes its half of P as packed fp16/bf16 pairs into
//            the P columns of TMEM (the A operand of the PV product) and
//            rescales its O when its max moved.  At the end the two halves of a row are merged by
//            log-sum-exp and each writes half of the output row.  (One
//            warpgroup for all 128 columns took ~1.5 us of ~1.9 us per tile.)
// Values of keys past the context are zeroed in shared memory before the PV
// product, so undefined (even NaN) pool slots never reach the accumulator.
#include <algorithm>
#include <cstddef>
#include <cudaTypedefs.h>

#include "ns_internal.h"
#include "tcgen05.cuh"

namespace ns {

namespace {

constexpr int kRows = 128;       // MMA M
constexpr int kTmemCols = 512;
constexpr int kRegionBytes = 128;     // 64 elements of a row: one 128-byte swizzle span
constexpr int kSoftmaxThreads = 256;  // two warpgroups: the two key halves of each tile

// Geometry by head dim D.  A row of D elements is D/64 regions of 64; each
// region of a Q, K or V tile is its own 128-byte-swizzled panel in shared
// memory, loaded by its own TMA box.  D 64: 128-key tiles, 4 stages; D 128:
// 64-key tiles and 3 stages, so that shared memory and TMEM fit.
// TMEM columns: S [0, KT); O of key half h [KT + D h, KT + D (h+1)); P of
// tile j in buffer b = j mod 2, part p, key half h: [KT + 2D + NP KT/2 b +
// KT/2 p + KT/4 h, + KT/4) (two 16-bit values a column; NP parts).
template <int D>
struct TcGeo {
    static constexpr int KT = D == 64 ? 128 : 64;  // keys per K/V tile
    static constexpr int REG = D / 64;             // regions of a row
    static constexpr int HALF = KT / 2;            // key columns per softmax thread
    static constexpr int STAGES = D == 64 ? 4 : 3; // K/V tiles in flight (D 64: 3 measured 4% slower, 5 alike)
    static constexpr int TMEM_O = KT;
    static constexpr int TMEM_P = KT + 2 * D;
    static constexpr int ROW_BYTES = 2 * D;
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
};
constexpr int kMmaWarp = 8;            // score products; TMEM allocation
constexpr int kProducerWarp = 9;
constexpr int kPvWarp = 10;            // value products
constexpr int kThreads = 352;          // warps 0-7 softmax, 8 and 10 MMA, 9 producer
constexpr float kSlack = 8.0f;   // lazy rescale: the max moves by more than this (log2 units)
// Every exponential runs on the MUFU pipe: an FMA-pipe polynomial for half of
// them measured 12% slower (its instructions cost more than MUFU).

struct PrefillParams {
    const int32_t *qsl;
    const int32_t *context_lens;
    const int32_t *block_tables;
    uint16_t *out;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int qt;  // tokens per query tile
    int min_span;  // spans of at least this many query tokens run here
    int max_blocks_per_seq;
    long long num_blocks;
    float scale_log2;
    unsigned *status;
};

// P goes to the tensor core as fp16/bf16.  For bf16 one rounding (2^-9
// relative) is too coarse, so P is split into P_hi + P_lo (both bf16, about
// 16 bits together) and multiplied by V twice.
template <typename T>
struct PParts {
    static constexpr int N = T::code == NS_BF16 ? 2 : 1;
};

// NP (the P parts, 1 or 2) sizes no member: P lives in TMEM.
template <int NP, int D>
struct alignas(1024) PrefillSmem {
    using GG = TcGeo<D>;
    uint8_t q[GG::REG][kRows * kRegionBytes];
    uint8_t k[GG::STAGES][GG::REG][GG::KT * kRegionBytes];
    uint8_t v[GG::STAGES][GG::REG][GG::KT * kRegionBytes];
    uint64_t q_full;
    uint64_t kv_full[GG::STAGES];
    uint64_t kv_empty[GG::STAGES];
    uint64_t s_full;
    uint64_t s_free;
    uint64_t p_full;
    uint64_t o_done[2];  // value products of the tiles that used P buffer b done
    // the two softmax halves of a row exchange their maxima and sums once,
    // at the end, through these
    uint64_t xbar;
    float xm[2][kRows];  // [half][row]
    float xl[2][kRows];
    // rank 1's unnormalised rows, written remotely into rank 0 with 16-byte stores
    alignas(16) float rem_o[kRows][D];
    float rem_m[kRows];
    float rem_l[kRows];
    uint64_t rem_bar;
    uint32_t tmem_base;
    uint32_t loaded[GG::STAGES];  // bit i: block i of the tile was loaded
    int u_s, u_h, u_i0, u_n, u_L, u_tiles, u_ok;
    int u_j0, u_nt;  // this CTA's key tiles: u_j0, u_j0 + 2, ... (u_nt of them)
};

// Vector (16-byte) and mbarrier (8-byte) accesses need these alignments.
using Smem164 = PrefillSmem<1, 64>;
using Smem264 = PrefillSmem<2, 64>;
using Smem1128 = PrefillSmem<1, 128>;
using Smem2128 = PrefillSmem<2, 128>;
static_assert(offsetof(Smem164, rem_o) % 16 == 0 && offsetof(Smem264, rem_o) % 16 == 0 &&
                  offsetof(Smem1128, rem_o) % 16 == 0 && offsetof(Smem2128, rem_o) % 16 == 0,
              "remote 16-byte stores into rem_o");
static_assert(offsetof(Smem164, q_full) % 8 == 0 && offsetof(Smem264, rem_bar) % 8 == 0 &&
                  offsetof(Smem1128, q_full) % 8 == 0 && offsetof(Smem2128, rem_bar) % 8 == 0,
              "mbarriers are 8-byte aligned");
// every swizzled panel starts on a 1024-byte boundary
static_assert(offsetof(Smem1128, k) % 1024 == 0 && offsetof(Smem1128, v) % 1024 == 0 &&
                  offsetof(Smem164, k) % 1024 == 0 && offsetof(Smem164, v) % 1024 == 0 &&
                  (TcGeo<128>::KT * kRegionBytes) % 1024 == 0,
              "128-byte swizzle panels are 1024-byte aligned");

template <int NP, int D>
constexpr size_t smem_bytes()
{
    return sizeof(PrefillSmem<NP, D>) + 1024;  // + alignment slack
}

static_assert(smem_bytes<1, 64>() <= 227 * 1024 && smem_bytes<2, 64>() <= 227 * 1024 &&
                  smem_bytes<1, 128>() <= 227 * 1024 && smem_bytes<2, 128>() <= 227 * 1024,
              "prefill shared memory");

template <int NP, int D>
__device__ __forceinline__ PrefillSmem<NP, D> &smem_of(unsigned char *raw)
{
    const uintptr_t a = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023);
    return *reinterpret_cast<PrefillSmem<NP, D> *>(a);
}

// Find this CTA's unit.  Units are enumerated spans last-to-first (later
// chunks sit on longer prefixes), query tiles last-to-first, then kv heads.
template <class Smem>
__device__ void find_unit(const PrefillParams &P, Smem &sm, int lane)
{
    const long long u = blockIdx.x >> 1;  // one unit per 2-CTA cluster
    long long base = 0;
    int found = 0;
    for (int s0 = P.num_seqs - 1; s0 >= 0 && !found; s0 -= 32) {
        const int s = s0 - lane;
        int tiles = 0;
        if (s >= 0) {
            const int n = __ldg(P.qsl + s + 1) - __ldg(P.qsl + s);
            tiles = n >= P.min_span ? (n + P.qt - 1) / P.qt : 0;
        }
        long long w = (long long)tiles * P.num_kv_heads;
        long long incl = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        const long long excl = base + incl - w;
        const bool mine = w > 0 && u >= excl && u < excl + w;
        const unsigned who = __ballot_sync(0xffffffffu, mine);
        if (who) {
            found = 1;
            if (mine) {
                const long long r = u - excl;
                const int tile_rev = (int)(r / P.num_kv_heads);
                const int h = (int)(r % P.num_kv_heads);
                const int n = __ldg(P.qsl + s + 1) - __ldg(P.qsl + s);
                const int ntiles = (n + P.qt - 1) / P.qt;
                const int tile = ntiles - 1 - tile_rev;
                sm.u_s = s;
                sm.u_h = h;
                sm.u_i0 = tile * P.qt;
                sm.u_n = n;
                sm.u_L = __ldg(P.context_lens + s);
                sm.u_ok = 1;
            }
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0 && !found)
        sm.u_ok = -1;  // no unit for this CTA
}

// P of a softmax thread's key half into TMEM: 32 columns (D 64) or 16 (D 128).
__device__ __forceinline__ void store_p(uint32_t addr, const uint32_t (&v)[32]) { tc::tmem_st32(addr, v); }
__device__ __forceinline__ void store_p(uint32_t addr, const uint32_t (&v)[16]) { tc::tmem_st16(addr, v); }

template <typename T, int BS, int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillParams P)
{
    constexpr int NP = PParts<T>::N;
    using GG = TcGeo<D>;
    constexpr int kKT = GG::KT, kHalf = GG::HALF, kStages = GG::STAGES, kRowBytes = GG::ROW_BYTES;
    constexpr int kTmemO = GG::TMEM_O, kTmemP = GG::TMEM_P, REG = GG::REG;
    constexpr int OC = D / 2;  // output columns of a softmax thread
    static_assert(kTmemP + 2 * NP * (kKT / 2) <= kTmemCols, "two P buffers fit in TMEM");
    extern __shared__ unsigned char smem_raw[];
    PrefillSmem<NP, D> &sm = smem_of<NP, D>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = P.group;

    if (warp == kProducerWarp) {
        find_unit(P, sm, lane);
        __syncwarp();
        if (lane == 0 && sm.u_ok == 1) {
            const int n = sm.u_n;
            int L = sm.u_L;
            const long long cap = (long long)P.max_blocks_per_seq * BS;
            if (L < n || n < 1 || L < 0) {
                raise_status(P.status, NS_DEV_BAD_QUERY_SPAN);
                sm.u_ok = 0;
            } else if (L > cap) {
                raise_status(P.status, NS_DEV_BAD_CONTEXT_LEN);
                sm.u_ok = 0;
            } else {
                const int last_tok = min(sm.u_i0 + P.qt, n) - 1;
                const long long keys = (long long)(L - n) + last_tok + 1;
                const int tiles = (int)((keys + kKT - 1) / kKT);
                // the two CTAs of the cluster take alternate key tiles (even,
                // odd), so that the masked tiles at the diagonal are shared
                // (measured against first and second halves: 37.6-37.9 ->
                // 36.9 us on the mixed chunked-prefill step)
                const int half = (tiles + 1) / 2;
                const bool second = tc::cluster_rank() != 0;
                sm.u_tiles = tiles;
                sm.u_j0 = second ? 1 : 0;
                sm.u_nt = second ? tiles - half : half;
            }
        }
    }
    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.kv_full[i], 1);
            mbar_init(&sm.kv_empty[i], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_free, kSoftmaxThreads);
        mbar_init(&sm.p_full, kSoftmaxThreads);
        mbar_init(&sm.o_done[0], 1);
        mbar_init(&sm.o_done[1], 1);
        mbar_init(&sm.xbar, kSoftmaxThreads);
        mbar_init(&sm.rem_bar, kSoftmaxThreads);
        mbar_init_fence();
    }
    __syncthreads();
    if (sm.u_ok != 1)
        return;  // both CTAs of the cluster see the same unit and leave together
    tc::cluster_sync();  // rank 0's barriers are initialised before rank 1 can arrive on them
    const uint32_t rank = tc::cluster_rank();
    // Rows of the Q tile the TMA box does not cover are zeroed once.
    if (warp < 4 && (int)threadIdx.x >= P.qt * G) {
#pragma unroll
        for (int g = 0; g < REG; ++g)
#pragma unroll
            for (int b = 0; b < kRegionBytes; b += 16)
                *reinterpret_cast<uint4 *>(sm.q[g] + threadIdx.x * kRegionBytes + b) = make_uint4(0, 0, 0, 0);
        tc::fence_async_smem();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(&sm.tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    const int s = sm.u_s, h = sm.u_h, i0 = sm.u_i0, n = sm.u_n, L = sm.u_L;
    const int tiles = sm.u_nt;   // this CTA's key tiles ...
    const int j0 = sm.u_j0;      // ... every other one from key tile j0
    const int prefix = L - n;
    const uint32_t tmem = sm.tmem_base;
    const int ab_fmt = T::code == NS_BF16 ? 1 : 0;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && tiles > 0) {
            tc::prefetch_tensormap(&tm_q);
            tc::prefetch_tensormap(&tm_k);
            tc::prefetch_tensormap(&tm_v);
            mbar_arrive_expect_tx(&sm.q_full, (uint32_t)(P.qt * G * kRowBytes));
#pragma unroll
            for (int g = 0; g < REG; ++g)
                tc::tma_load_3d(sm.q[g], &tm_q, g * 64, h * G, __ldg(P.qsl + s) + i0, &sm.q_full);
        }
        constexpr int kBlocksPerTile = kKT / BS;
        const int nb_seq = (L + BS - 1) / BS;
        // lane i < kBlocksPerTile: the table entry of block i of key tile j
        // (-1 past the sequence); tile j+1's entry loads while tile j's
        // slot is awaited, so no copy waits on a table read
        auto table_entry = [&](int j) {
            const int blk = (j0 + 2 * j) * kBlocksPerTile + lane;
            return (lane < kBlocksPerTile && j < tiles && blk < nb_seq)
                       ? __ldg(P.block_tables + (long long)s * P.max_blocks_per_seq + blk)
                       : -1;
        };
        bool ok = true;
        int issued = 0;
        int next_phys = table_entry(0);
        for (int j = 0; ok && j < tiles; ++j) {
            const int stage = j % kStages;
            const uint32_t par = ((uint32_t)(j / kStages) & 1u) ^ 1u;
            int phys = next_phys;
            next_phys = table_entry(j + 1);
            const int blk = (j0 + 2 * j) * kBlocksPerTile + lane;
            if (lane < kBlocksPerTile && blk < nb_seq && (phys < 0 || (long long)phys >= P.num_blocks)) {
                raise_status(P.status, NS_DEV_BAD_BLOCK_ID);
                phys = -1;
            }
            const unsigned mask = __ballot_sync(0xffffffffu, phys >= 0);
            if (lane == 0) {
                if (!mbar_wait(&sm.kv_empty[stage], par)) {
                    raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
                    ok = false;
                } else {
                    sm.loaded[stage] = mask;
                    mbar_arrive_expect_tx(&sm.kv_full[stage],
                                          (uint32_t)__popc(mask) * 2u * BS * kRowBytes);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (ok && phys >= 0) {
                const int row = (int)(((long long)phys * P.num_kv_heads + h) * BS);
#pragma unroll
                for (int g = 0; g < REG; ++g) {
                    tc::tma_load_2d(sm.k[stage][g] + lane * BS * kRegionBytes, &tm_k, g * 64, row, &sm.kv_full[stage]);
                    tc::tma_load_2d(sm.v[stage][g] + lane * BS * kRegionBytes, &tm_v, g * 64, row, &sm.kv_full[stage]);
                }
            }
            if (ok)
                issued = j + 1;
        }
        // Never leave while copies may still land in this CTA's shared memory.
        if (lane == 0 && tiles > 0) {
            bool drained = mbar_wait(&sm.q_full, 0);
            for (int k = 1; drained && k <= kStages && k <= issued; ++k) {
                const int j = issued - k;
                drained = mbar_wait(&sm.kv_full[j % kStages], (uint32_t)(j / kStages) & 1u);
            }
            if (!drained)
                raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ score products
        if (lane == 0 && tiles > 0) {
            const uint32_t idesc_s = tc::idesc_f16(kRows, kKT, ab_fmt, false);
            const uint32_t q_addr = smem_addr(sm.q[0]);  // region g at + g * kRows * kRegionBytes
            // S_j = Q K_j^T into TMEM columns [0, 128), once K_j has landed
            // and the softmax has read S_{j-1}
            bool ok = mbar_wait(&sm.q_full, 0);
            for (int j = 0; ok && j < tiles; ++j) {
                ok = mbar_wait(&sm.kv_full[j % kStages], (uint32_t)(j / kStages) & 1u) &&
                     (j == 0 || mbar_wait(&sm.s_free, (uint32_t)(j - 1) & 1u));
                if (!ok)
                    break;
                tc::fence_after_sync();
                const uint32_t k_addr = smem_addr(sm.k[j % kStages][0]);  // region g at + g * kKT * kRegionBytes
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // dims 16 kk ..: region kk / 4, 32 bytes a step inside it
                    const int g = kk >> 2;
                    tc::mma_ss(tmem, tc::desc_sw128(q_addr + g * kRows * kRegionBytes + (kk & 3) * 32),
                               tc::desc_sw128(k_addr + g * kKT * kRegionBytes + (kk & 3) * 32), idesc_s,
                               kk > 0 ? 1u : 0u);
                }
                tc::mma_commit(&sm.s_full);
            }
            if (!ok)
                raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------------ value products
        if (lane == 0 && tiles > 0) {
            const uint32_t idesc_o = tc::idesc_f16(kRows, 64, ab_fmt, true);  // one region of O per product
            bool ok = true;
            for (int j = 0; ok && j < tiles; ++j) {
                // P_j is in TMEM buffer j mod 2 (and V_j landed before S_j was computed)
                ok = mbar_wait(&sm.p_full, (uint32_t)j & 1u);
                if (!ok)
                    break;
                tc::fence_after_sync();
                const uint32_t v_addr = smem_addr(sm.v[j % kStages][0]);  // region g at + g * kKT * kRegionBytes
                const uint32_t p_buf = kTmemP + (uint32_t)(j & 1) * (NP * kKT / 2);
#pragma unroll
                for (int part = 0; part < NP; ++part)
#pragma unroll
                    for (int kk = 0; kk < kKT / 16; ++kk) {
                        // keys 16 kk ..: key half kk / KH accumulates into its own O,
                        // one product per 64-dim region of V
                        constexpr int KH = kHalf / 16;
                        const int hh = kk / KH, ki = kk % KH;
                        const uint32_t p_cols = p_buf + part * (kKT / 2) + hh * (kHalf / 2) + ki * 8;
#pragma unroll
                        for (int g = 0; g < REG; ++g)
                            tc::mma_ts(tmem + kTmemO + hh * D + g * 64, tmem + p_cols,
                                       tc::desc_sw128(v_addr + g * kKT * kRegionBytes + kk * 16 * kRegionBytes),
                                       idesc_o, (j > 0 || part > 0 || ki > 0) ? 1u : 0u);
                    }
                tc::mma_commit(&sm.o_done[j & 1]);
                tc::mma_commit(&sm.kv_empty[j % kStages]);
            }
            if (!ok)
                raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int r = threadIdx.x & (kRows - 1);  // row == TMEM lane
        const int hf = threadIdx.x / kRows;       // 0: key columns 0..63, 1: 64..127
        const int c0 = hf * kHalf;
        const int tok = r / G;
        const bool row_ok = r < P.qt * G && i0 + tok < n;
        const int pos = row_ok ? prefix + i0 + tok : -1;
        const int pos_lo = prefix + i0;  // smallest position in the tile
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        float m = -INFINITY, l = 0.f;  // this key half's running max and sum
        bool ok = true;
        for (int j = 0; j < tiles; ++j) {
            const int stage = j % kStages;
            if (!mbar_wait(&sm.s_full, (uint32_t)j & 1u)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            float sv[kHalf];
#pragma unroll
            for (int c = 0; c < kHalf / 32; ++c)
                tc::tmem_ld32(lane_addr + c0 + c * 32, *reinterpret_cast<float(*)[32]>(&sv[c * 32]));
            tc::tmem_ld_wait();
            tc::fence_before_sync();
            mbar_arrive(&sm.s_free);

            const int tbase = (j0 + 2 * j) * kKT;  // first key of the tile
            const int kbase = tbase + c0;      // first key of this half
            const bool masked = tbase + kKT - 1 > pos_lo;
            // four independent running maxima (no long dependent chain)
            float tm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (masked) {
#pragma unroll
                for (int c = 0; c < kHalf; ++c) {
                    sv[c] = (kbase + c <= pos) ? sv[c] : -INFINITY;
                    tm[c & 3] = fmaxf(tm[c & 3], sv[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < kHalf; ++c)
                    tm[c & 3] = fmaxf(tm[c & 3], sv[c]);
            }
            float tmax = fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3]));
            tmax *= P.scale_log2;  // scale > 0 keeps the order
            float m_new = m;
            if (tmax > m + kSlack)
                m_new = tmax;
            const float alpha = fast_exp2(m - m_new);
            const bool rescale = (m_new != m) && j > 0;
            l *= (m_new != m) ? alpha : 1.f;
            m = m_new;

            uint32_t pk[kHalf / 2];
            // pairs of columns in packed fp32 (scale and shift, sums); two
            // independent partial sums
            const float2 sc2 = make_float2(P.scale_log2, P.scale_log2);
            const float2 nm2 = make_float2(-m, -m);
            float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int c = 0; c < kHalf; c += 2) {
                const float2 z = ffma2(make_float2(sv[c], sv[c + 1]), sc2, nm2);
                float p0 = fast_exp2(z.x);
                float p1 = fast_exp2(z.y);
                if (masked) {
                    p0 = sv[c] > -INFINITY ? p0 : 0.f;
                    p1 = sv[c + 1] > -INFINITY ? p1 : 0.f;
                }
                ls2[(c >> 1) & 1] = fadd2(ls2[(c >> 1) & 1], make_float2(p0, p1));
                pk[c >> 1] = pack2<T>(p0, p1);
                if (NP == 2) {
                    // keep the rounding residue of P for the second product
                    const float2 hi = unpack2<T>(pk[c >> 1]);
                    sv[c] = p0 - hi.x;
                    sv[c + 1] = p1 - hi.y;
                }
            }
            l += (ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y);

            // P buffer j mod 2 is free once the value products of tile j-2
            // are done; O may be rescaled once those of tile j-1 are (a
            // commit covers every product issued before it)
            const bool any_rescale = __any_sync(0xffffffffu, rescale);
            if (any_rescale ? (j > 0 && !mbar_wait(&sm.o_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u))
                            : (j > 1 && !mbar_wait(&sm.o_done[j & 1], (uint32_t)((j - 2) >> 1) & 1u))) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            if (any_rescale) {
                // this key half's O row
                const float a = rescale ? alpha : 1.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float ov[32];
                    tc::tmem_ld32(lane_addr + kTmemO + hf * D + c * 32, ov);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        ov[e] *= a;
                    tc::tmem_st32(lane_addr + kTmemO + hf * D + c * 32, ov);
                }
                tc::tmem_st_wait();
            }
            // P row r, this half's keys c0 .. c0 + 63: column c holds keys
            // c0 + 2c (low half) and c0 + 2c + 1
            const uint32_t p_buf = kTmemP + (uint32_t)(j & 1) * (NP * kKT / 2);
            store_p(lane_addr + p_buf + hf * (kHalf / 2), pk);
            if (NP == 2) {
                uint32_t pl[kHalf / 2];
#pragma unroll
                for (int c = 0; c < kHalf / 2; ++c)
                    pl[c] = pack2<T>(sv[2 * c], sv[2 * c + 1]);
                store_p(lane_addr + p_buf + (NP - 1) * (kKT / 2) + hf * (kHalf / 2), pl);
            }
            // Values of keys past the context, or of blocks that were not
            // loaded, must be zero: P is zero there but 0 * NaN is not.  This
            // half clears bytes 64 hf .. 64 hf + 63 of value row r.
            if (masked || sm.loaded[stage] != (1u << (kKT / BS)) - 1u) {
                if (!mbar_wait(&sm.kv_full[stage], (uint32_t)(j / kStages) & 1u)) {
                    ok = false;
                    break;
                }
                const int key = tbase + r;
                const bool blk_loaded = r < kKT && ((sm.loaded[stage] >> (r / BS)) & 1u);
                if (r < kKT && (key >= L || !blk_loaded)) {
                    // this half's share of the row: bytes 64 hf.. of its one
                    // region (D 64), or region hf (D 128)
                    uint8_t *row = REG == 1 ? sm.v[stage][0] + r * kRegionBytes + hf * (kRegionBytes / 2)
                                            : sm.v[stage][hf] + r * kRegionBytes;
#pragma unroll
                    for (int b = 0; b < kRowBytes / 2; b += 16)
                        *reinterpret_cast<uint4 *>(row + b) = make_uint4(0, 0, 0, 0);
                }
            }
            tc::tmem_st_wait();
            tc::fence_async_smem();
            tc::fence_before_sync();
            mbar_arrive(&sm.p_full);
        }
        // ---- epilogue: merge the row's two key halves (log-sum-exp), then this
        // CTA's unnormalised output columns 32 hf .. 32 hf + 31 (zero when it had no tile)
        sm.xm[hf][r] = m;
        sm.xl[hf][r] = l;
        mbar_arrive(&sm.xbar);
        float ov[OC];
        float fa = 0.f, fb = 0.f;  // factors of key halves 0 and 1
        if (ok && mbar_wait(&sm.xbar, 0)) {
            const float ma = sm.xm[0][r], mb = sm.xm[1][r];
            const float M = fmaxf(ma, mb);
            fa = (ma > -INFINITY) ? fast_exp2(ma - M) : 0.f;
            fb = (mb > -INFINITY) ? fast_exp2(mb - M) : 0.f;
            l = fa * sm.xl[0][r] + fb * sm.xl[1][r];
            m = M;
        } else {
            ok = false;
        }
        if (ok && tiles > 0) {
            ok = mbar_wait(&sm.o_done[(tiles - 1) & 1], (uint32_t)((tiles - 1) >> 1) & 1u);
            if (ok) {
                tc::fence_after_sync();
#pragma unroll
                for (int ch = 0; ch < OC / 32; ++ch) {
                    float oa[32], ob[32];
                    tc::tmem_ld32(lane_addr + kTmemO + hf * OC + ch * 32, oa);
                    tc::tmem_ld32(lane_addr + kTmemO + D + hf * OC + ch * 32, ob);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        ov[ch * 32 + c] = fmaf(fa, oa[c], fb * ob[c]);
                }
            }
        }
        if (!ok || tiles == 0) {
#pragma unroll
            for (int c = 0; c < OC; ++c)
                ov[c] = 0.f;
        }
        if (!ok)
            raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
        if (rank != 0) {
            // rank 1: hand (max, sum, half rows) to rank 0 through distributed shared memory
            const uint32_t dst = tc::map_to_rank(&sm.rem_o[r][hf * OC], 0);
#pragma unroll
            for (int c = 0; c < OC; c += 4)
                tc::st_cluster_v4(dst + c * 4, ov[c], ov[c + 1], ov[c + 2], ov[c + 3]);
            if (hf == 0) {
                tc::st_cluster_f32(tc::map_to_rank(&sm.rem_m[r], 0), m);
                tc::st_cluster_f32(tc::map_to_rank(&sm.rem_l[r], 0), l);
            }
            tc::mbar_arrive_remote(tc::map_to_rank(&sm.rem_bar, 0));
        } else if (tc::mbar_wait_cluster(&sm.rem_bar, 0)) {
            // rank 0: log-sum-exp merge of the two key halves, then O / l
            const float m1 = sm.rem_m[r], l1 = sm.rem_l[r];
            const float M = fmaxf(m, m1);
            const float f0 = (m > -INFINITY) ? fast_exp2(m - M) : 0.f;
            const float f1 = (m1 > -INFINITY) ? fast_exp2(m1 - M) : 0.f;
            if (row_ok) {
                const float inv = 1.f / (f0 * l + f1 * l1);
                const float a0 = f0 * inv, a1 = f1 * inv;
                const long long tok_g = __ldg(P.qsl + s) + i0 + tok;
                uint16_t *o = P.out + (tok_g * P.num_q_heads + (long long)h * G + (r % G)) * D + hf * OC;
                const float *o1 = &sm.rem_o[r][hf * OC];
#pragma unroll
                for (int c = 0; c < OC; c += 8) {
                    uint4 w;
                    w.x = pack2<T>(fmaf(ov[c], a0, o1[c] * a1), fmaf(ov[c + 1], a0, o1[c + 1] * a1));
                    w.y = pack2<T>(fmaf(ov[c + 2], a0, o1[c + 2] * a1), fmaf(ov[c + 3], a0, o1[c + 3] * a1));
                    w.z = pack2<T>(fmaf(ov[c + 4], a0, o1[c + 4] * a1), fmaf(ov[c + 5], a0, o1[c + 5] * a1));
                    w.w = pack2<T>(fmaf(ov[c + 6], a0, o1[c + 6] * a1), fmaf(ov[c + 7], a0, o1[c + 7] * a1));
                    *reinterpret_cast<uint4 *>(o + c) = w;
                }
            }
        } else {
            raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    // Neither CTA leaves while the other may still touch its shared memory
    // (rank 1's remote stores land before it reaches this barrier, also when
    // rank 0 gave up waiting for them).
    tc::cluster_sync();
}

}  // namespace

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch.
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

static bool encode(CUtensorMap *map, ns_dtype dt, int rank, const void *base, const cuuint64_t *dims,
                   const cuuint64_t *strides, const cuuint32_t *box)
{
    auto fn = encode_fn();
    if (fn == nullptr)
        return false;
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, dt == NS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tc_prefill_supported(int block_size, int group)
{
    return (block_size == 16 || block_size == 32) && group >= 1 && group <= kMaxGroup;
}

template <typename T, int BS, int D>
static cudaError_t launch_tc(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const PrefillParams &P, int grid, bool overlap, cudaStream_t stream)
{
    static int done_mask = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (!(dev < 31 && ((done_mask >> dev) & 1))) {
        e = cudaFuncSetAttribute(tc_prefill_kernel<T, BS, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes<PParts<T>::N, D>());
        if (e != cudaSuccess)
            return e;
        if (dev < 31)
            __atomic_fetch_or(&done_mask, 1 << dev, __ATOMIC_RELAXED);
    }
    if (!overlap) {
        tc_prefill_kernel<T, BS, D><<<grid, kThreads, smem_bytes<PParts<T>::N, D>(), stream>>>(tq, tk, tv, P);
        return cudaGetLastError();
    }
    // programmatic dependent of the kernel before it (the span walk of the same
    // call, whose results this kernel does not read): it may start as soon as
    // SMs free up, with no wait
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes<PParts<T>::N, D>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_prefill_kernel<T, BS, D>, tq, tk, tv, P);
}

cudaError_t launch_tc_prefill(const void *q, const int32_t *query_start_loc, const void *k_pool,
                              const void *v_pool, const int32_t *block_tables,
                              const int32_t *context_lens, int num_seqs, int total_q_tokens,
                              int num_q_heads, int num_kv_heads, int block_size, float scale,
                              void *out, int max_blocks_per_seq, long long num_blocks, ns_dtype dtype,
                              int min_span, int head_dim, unsigned *status, bool after_walk,
                              cudaStream_t stream)
{
    const int G = num_q_heads / num_kv_heads;
    const int qt = kRows / G;
    if (min_span < 1 || (head_dim != 64 && head_dim != 128))
        return cudaErrorInvalidValue;
    const int row_bytes = 2 * head_dim;
    CUtensorMap tq, tk, tv;
    {
        // boxes of 64 elements (one 128-byte swizzle span); a 128-element row is two
        const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_q_heads, (cuuint64_t)total_q_tokens};
        const cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)num_q_heads * row_bytes};
        const cuuint32_t box[3] = {64u, (cuuint32_t)G, (cuuint32_t)qt};
        if (!encode(&tq, dtype, 3, q, dims, strides, box))
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t rows = (cuuint64_t)num_blocks * num_kv_heads * block_size;
        const cuuint64_t dims[2] = {(cuuint64_t)head_dim, rows};
        const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
        const cuuint32_t box[2] = {64u, (cuuint32_t)block_size};
        if (!encode(&tk, dtype, 2, k_pool, dims, strides, box) ||
            !encode(&tv, dtype, 2, v_pool, dims, strides, box))
            return cudaErrorInvalidValue;
    }
    PrefillParams P;
    P.qsl = query_start_loc;
    P.context_lens = context_lens;
    P.block_tables = block_tables;
    P.out = static_cast<uint16_t *>(out);
    P.num_seqs = num_seqs;
    P.num_q_heads = num_q_heads;
    P.num_kv_heads = num_kv_heads;
    P.group = G;
    P.qt = qt;
    P.min_span = min_span;
    P.max_blocks_per_seq = max_blocks_per_seq;
    P.num_blocks = num_blocks;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.status = status;
    // an upper bound on the units (2 CTAs each): a span of n >= min_span
    // tokens has ceil(n / qt) query tiles, and there are at most
    // min(num_seqs, T / min_span) such spans; CTA pairs without a unit exit at once
    const long long spans = std::min<long long>(num_seqs, total_q_tokens / min_span);
    const long long units = (long long)num_kv_heads * ((total_q_tokens + qt - 1) / qt + spans);
    const int grid = (int)(2 * units > 0x7ffffffe ? 0x7ffffffe : 2 * units);
    if (grid == 0)
        return cudaSuccess;
    if (head_dim == 128)  // block size 16 only
        return dtype == NS_BF16 ? launch_tc<BF16, 16, 128>(tq, tk, tv, P, grid, after_walk, stream)
                                : launch_tc<F16, 16, 128>(tq, tk, tv, P, grid, after_walk, stream);
    if (dtype == NS_BF16)
        return block_size == 16 ? launch_tc<BF16, 16, 64>(tq, tk, tv, P, grid, after_walk, stream)
                                : launch_tc<BF16, 32, 64>(tq, tk, tv, P, grid, after_walk, stream);
    return block_size == 16 ? launch_tc<F16, 16, 64>(tq, tk, tv, P, grid, after_walk, stream)
                            : launch_tc<F16, 32, 64>(tq, tk, tv, P, grid, after_walk, stream);
}

}  // namespace ns
