// tc_decode.cu -- split-KV paged-attention decode on the tcgen05 tensor cores
// (block sizes 16 and 32).
//
// What it computes is the decode step of the nanoserve project page ("What I
// built": paged-attention decode with online softmax over each sequence's
// block table): out[s][j] = softmax_p(scale * q[s][j] . K_s[p]) . V_s[p] for
// every query head j of every sequence s, split across CTAs and merged by
// log-sum-exp as in the flash-decoding arm of the build log (Day 74 post).
// The split, the partial records and their merge are those of the CUDA-core
// decode kernel (paged_decode.cuh); this file replaces its inner loop.
//
// How.  A GQA group has G <= 8 query heads sharing one kv head, so one decode
// step of one (sequence, kv head) is two thin matrix products per tile of 128
// keys: S^T = K Q^T (128 keys x 8 heads) and O += P V (8 heads x 64 dims).
// Both run on the tensor core with operands in shared memory and fp32
// accumulators in TMEM:
//  * S^T: A = the K tile (M = 128 keys, K-major, 128-byte swizzle as TMA lays
//    it down), B = the group's Q rows (N = 16: 8 rows, the row-group stride
//    0 repeats them), D = 16 TMEM columns; lane t of TMEM holds key t's 8
//    scores, so each softmax thread owns one key and its softmax is 8
//    exponentials with no cross-thread work.
//  * O_w += P_w V_w for each of the 4 softmax warps w separately: A = warp
//    w's 32 columns of P (8 head rows, row-group stride 0, so the 128 D rows
//    repeat the 8 heads), B = the V tile (MN-major), D = 64 TMEM columns of
//    warp w.  Each warp keeps its own running max, so warps never wait on
//    each other inside a piece; their 4 partial results are merged when a
//    piece ends.
// Warp roles (192 threads, one CTA per SM): warps 0-3 softmax (thread =
// key), warp 4 issues the MMAs, warp 5 issues the TMA loads of whole KV blocks
// into a 4-stage ring (1 block = 1 box of the pool's 3-D tensor map, L2
// evict-first).  The MMA order per tile g is S_{g+1} then PV_g, so the
// softmax of a tile overlaps the tensor core and the copies of later tiles.
// Every wait is bounded (NS_DEV_WAIT_TIMEOUT, then an orderly wind-down).
#include <cstddef>
#include <cudaTypedefs.h>

#include "ns_internal.h"
#include "paged_decode.cuh"
#include "tcgen05.cuh"

namespace ns {
namespace {

constexpr int kTileKeys = 128;    // keys per tile = MMA M
constexpr int kTcStages = 4;      // K/V tiles in flight
constexpr int kSoftWarps = 4;
constexpr int kTcDecThreads = 192;
constexpr int kTmemAlloc = 512;   // one CTA per SM: the whole TMEM
constexpr int kSCols = 16;        // S^T buffer b: columns [16b, 16b + 16)
constexpr int kOCol0 = 64;        // O of softmax warp w: columns [64 + 64w, 128 + 64w)
constexpr int kQRows = 8;

// P in fp16 is one operand; bf16 P is split into hi + lo parts (about 16
// bits together), each multiplied by V.
template <typename T>
struct PSplit {
    static constexpr int N = T::code == NS_BF16 ? 2 : 1;
};

template <int NP>
struct alignas(1024) TcDecodeSmem {
    // 1024-byte aligned operand tiles first (128-byte swizzle atoms)
    uint8_t k[kTcStages][kTileKeys * 128];
    uint8_t v[kTcStages][kTileKeys * 128];
    uint8_t q[2][kQRows * 128];      // the group's Q rows, per piece parity
    uint8_t p[NP][2][kQRows * 128];  // P: [part][keys 0..63 | 64..127], 8 head rows
    float cm[2][kSoftWarps][kMaxGroup];  // per-warp results at a piece end, per piece parity
    float cl[2][kSoftWarps][kMaxGroup];
    float co[2][kSoftWarps][kMaxGroup][kHeadDim];
    uint64_t kv_full[kTcStages], kv_empty[kTcStages];
    uint64_t q_full[2], q_empty[2];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full[kSoftWarps], o_done[kSoftWarps];
    uint64_t mma_idle;
    uint64_t cons;  // rendezvous of the 128 softmax threads
    uint32_t tmem_base;
    uint32_t loaded[kTcStages];  // bit b: block b of the tile was loaded
    // split plan (decode_prologue) and piece walk state
    long long scan[32];
    int maxnb[32];
    long long b0, b1, total, start_off;
    int start_s, g_eff, merge_prev, abort_flag;
    int plan_split, plan_maxp;
    int whole;
};

static_assert(offsetof(TcDecodeSmem<2>, q) % 1024 == 0 && offsetof(TcDecodeSmem<2>, p) % 1024 == 0,
              "swizzle atoms are 1024-byte aligned");
static_assert(offsetof(TcDecodeSmem<1>, q) % 1024 == 0 && offsetof(TcDecodeSmem<1>, p) % 1024 == 0,
              "swizzle atoms are 1024-byte aligned");
static_assert(offsetof(TcDecodeSmem<2>, co) % 16 == 0 && offsetof(TcDecodeSmem<2>, kv_full) % 8 == 0,
              "vector and mbarrier alignment");
static_assert(offsetof(TcDecodeSmem<1>, co) % 16 == 0 && offsetof(TcDecodeSmem<1>, kv_full) % 8 == 0,
              "vector and mbarrier alignment");

template <int NP>
constexpr size_t tc_decode_smem_bytes()
{
    return sizeof(TcDecodeSmem<NP>) + 1024;  // + alignment slack
}

// Tiles of a piece of nb blocks.
template <int BS>
__device__ __forceinline__ int tiles_of(const PieceWalk &w)
{
    constexpr int TB = kTileKeys / BS;
    return (w.hi - w.lo + TB - 1) / TB;
}

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ---------------------------------------------------------------------------
// Producer (warp 5): Q rows of each piece, then the K and V blocks of its
// tiles, one block per lane.  With a fused append, the lane holding a pair's
// last block first writes the new token into its pool slot.
// ---------------------------------------------------------------------------
template <typename T, int BS, int NP>
__device__ void tc_producer(const DecodeParams &P, TcDecodeSmem<NP> &sm, const CUtensorMap *tm_q,
                            const CUtensorMap *tm_k, const CUtensorMap *tm_v, int lane)
{
    constexpr int TB = kTileKeys / BS;
    const int G = P.group;
    const uint64_t pol = l2_evict_first_policy();
    if (lane == 0) {
        tc::prefetch_tensormap(tm_q);
        tc::prefetch_tensormap(tm_k);
        tc::prefetch_tensormap(tm_v);
    }
    PieceWalk w;
    walk_init(P, sm, w);
    int g = 0, k = 0;
    int q_issued = 0;
    bool ok = true;
    while (ok && walk_next<BS>(P, w)) {
        if (lane == 0) {
            if (!wait_or_abort(&sm.q_empty[k & 1], ((uint32_t)(k >> 1) & 1u) ^ 1u, &sm.abort_flag)) {
                ok = false;
            } else {
                mbar_arrive_expect_tx(&sm.q_full[k & 1], (uint32_t)G * kRowBytes);
                const long long row = (long long)w.ps * P.num_q_heads + (long long)w.ph * G;
                tc::tma_load_2d(sm.q[k & 1], tm_q, 0, (int)row, &sm.q_full[k & 1]);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok)
            break;
        q_issued = k + 1;
        const long long trow = P.table_row != nullptr ? __ldg(P.table_row + w.ps) : w.ps;
        const int nt = tiles_of<BS>(w);
        long long new_slot = -1;
        if (P.k_new != nullptr && w.hi == w.pnb && lane == (w.pnb - 1 - w.lo) % TB)
            new_slot = __ldg(P.slot_mapping + w.ps);
        for (int j = 0; j < nt; ++j, ++g) {
            const int st = g % kTcStages;
            const int blk = w.lo + j * TB + lane;
            int phys = -1;
            if (lane < TB && blk < w.hi) {
                phys = __ldg(P.block_tables + trow * P.max_blocks_per_seq + blk);
                if (phys < 0 || (long long)phys >= P.num_blocks) {
                    raise_status(P.status, NS_DEV_BAD_BLOCK_ID);
                    phys = -1;
                }
            }
            const unsigned mask = __ballot_sync(0xffffffffu, phys >= 0);
            if (lane == 0) {
                if (!wait_or_abort(&sm.kv_empty[st], ((uint32_t)(g / kTcStages) & 1u) ^ 1u, &sm.abort_flag)) {
                    ok = false;
                } else {
                    sm.loaded[st] = mask;
                    mbar_arrive_expect_tx(&sm.kv_full[st], (uint32_t)__popc(mask) * 2u * BS * kRowBytes);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok)
                break;
            if (phys >= 0) {
                if (P.k_new != nullptr && blk == w.pnb - 1) {
                    // fused append: the new token goes to its slot before the block is read
                    const long long want = (long long)phys * BS + (w.pL - 1) % BS;
                    if (new_slot != want)
                        raise_status(P.status, NS_DEV_FUSED_SLOT);
                    if (new_slot >= P.num_blocks * BS) {
                        raise_status(P.status, NS_DEV_BAD_SLOT);
                    } else if (new_slot >= 0) {
                        const long long dst =
                            (((new_slot / BS) * P.num_kv_heads + w.ph) * BS + new_slot % BS) * kHeadDim;
                        const long long src = ((long long)w.ps * P.num_kv_heads + w.ph) * kHeadDim;
#pragma unroll
                        for (int c = 0; c < kHeadDim; c += 8) {
                            *reinterpret_cast<uint4 *>(P.k_pool_w + dst + c) =
                                __ldg(reinterpret_cast<const uint4 *>(P.k_new + src + c));
                            *reinterpret_cast<uint4 *>(P.v_pool_w + dst + c) =
                                __ldg(reinterpret_cast<const uint4 *>(P.v_new + src + c));
                        }
                        // the generic-proxy stores above are ordered before the TMA reads below
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                    }
                }
                tc::tma_load_3d_hint(sm.k[st] + lane * BS * kRowBytes, tm_k, 0, w.ph * BS, phys,
                                     &sm.kv_full[st], pol);
                tc::tma_load_3d_hint(sm.v[st] + lane * BS * kRowBytes, tm_v, 0, w.ph * BS, phys,
                                     &sm.kv_full[st], pol);
            }
        }
        ++k;
    }
    if (!ok)
        set_abort(P, sm);
    // Never leave while copies may still land in this CTA's shared memory.
    if (lane == 0) {
        bool drained = true;
        for (int kk = (q_issued > 2 ? q_issued - 2 : 0); drained && kk < q_issued; ++kk)
            drained = mbar_wait(&sm.q_full[kk & 1], (uint32_t)(kk >> 1) & 1u);
        for (int gg = (g > kTcStages ? g - kTcStages : 0); drained && gg < g; ++gg)
            drained = mbar_wait(&sm.kv_full[gg % kTcStages], (uint32_t)(gg / kTcStages) & 1u);
        if (!drained)
            raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// MMA issuer (warp 4, one lane).
// ---------------------------------------------------------------------------
struct TileCursor {
    PieceWalk w;
    int k = -1;   // piece index
    int j = 0;    // tile inside the piece
    int nt = 0;   // tiles of the piece
    bool valid = false;
};

template <int BS>
__device__ __forceinline__ void cursor_next(const DecodeParams &P, TileCursor &c)
{
    if (c.valid && c.j + 1 < c.nt) {
        ++c.j;
        return;
    }
    c.valid = walk_next<BS>(P, c.w);
    if (c.valid) {
        ++c.k;
        c.j = 0;
        c.nt = tiles_of<BS>(c.w);
    }
}

template <typename T, int BS, int NP>
__device__ void tc_mma(const DecodeParams &P, TcDecodeSmem<NP> &sm, uint32_t tmem)
{
    const int ab_fmt = T::code == NS_BF16 ? 1 : 0;
    const uint32_t idesc_s = tc::idesc_f16(kTileKeys, 16, ab_fmt, false);
    const uint32_t idesc_o = tc::idesc_f16(kTileKeys, kHeadDim, ab_fmt, true);
    TileCursor cur;
    walk_init(P, sm, cur.w);
    cursor_next<BS>(P, cur);
    bool ok = true;
    int g = 0;

    // S^T of tile gg (cursor c) into S buffer gg & 1
    auto issue_s = [&](const TileCursor &c, int gg) -> bool {
        const int st = gg % kTcStages;
        if (c.j == 0 && !wait_or_abort(&sm.q_full[c.k & 1], (uint32_t)(c.k >> 1) & 1u, &sm.abort_flag))
            return false;
        if (!wait_or_abort(&sm.kv_full[st], (uint32_t)(gg / kTcStages) & 1u, &sm.abort_flag))
            return false;
        if (!wait_or_abort(&sm.s_free[gg & 1], ((uint32_t)(gg >> 1) & 1u) ^ 1u, &sm.abort_flag))
            return false;
        tc::fence_after_sync();
        const uint32_t k_addr = smem_addr(sm.k[st]);
        const uint32_t q_addr = smem_addr(sm.q[c.k & 1]);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk)
            tc::mma_ss(tmem + (gg & 1) * kSCols, tc::desc_sw128(k_addr + kk * 32),
                       tc::desc_sw128_rows(q_addr + kk * 32, 0), idesc_s, kk > 0 ? 1u : 0u);
        tc::mma_commit(&sm.s_full[gg & 1]);
        if (c.j + 1 == c.nt)
            tc::mma_commit(&sm.q_empty[c.k & 1]);  // the piece's Q rows are free once these finish
        return true;
    };

    if (cur.valid)
        ok = issue_s(cur, 0);
    while (ok && cur.valid) {
        TileCursor nxt = cur;
        cursor_next<BS>(P, nxt);
        if (nxt.valid && !(ok = issue_s(nxt, g + 1)))
            break;
        // PV of tile g, warp by warp as their P columns arrive
        const int st = g % kTcStages;
        const uint32_t v_addr = smem_addr(sm.v[st]);
        for (int w = 0; w < kSoftWarps && ok; ++w) {
            if (!wait_or_abort(&sm.p_full[w], (uint32_t)g & 1u, &sm.abort_flag)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
#pragma unroll
            for (int part = 0; part < NP; ++part)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int kk = 2 * w + h;  // 16 keys: rows 16kk.. of V, columns 16kk.. of P
                    const uint32_t p_addr = smem_addr(sm.p[part][kk >> 2]) + (kk & 3) * 32;
                    tc::mma_ss(tmem + kOCol0 + w * kHeadDim, tc::desc_sw128_rows(p_addr, 0),
                               tc::desc_sw128(v_addr + kk * 16 * kRowBytes), idesc_o,
                               (cur.j > 0 || part > 0 || h > 0) ? 1u : 0u);
                }
            tc::mma_commit(&sm.o_done[w]);
        }
        if (!ok)
            break;
        tc::mma_commit(&sm.kv_empty[st]);
        cur = nxt;
        ++g;
    }
    if (!ok)
        set_abort(P, sm);
    // every MMA issued so far has finished before TMEM or shared memory is released
    tc::mma_commit(&sm.mma_idle);
    if (!mbar_wait(&sm.mma_idle, 0))
        raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Softmax warps 0-3: thread t owns key t of every tile.
// ---------------------------------------------------------------------------
template <typename T, int BS, int NP>
__device__ bool tc_piece_end(const DecodeParams &P, TcDecodeSmem<NP> &sm, const PieceWalk &pc, int k,
                             const float (&m)[kMaxGroup], const float (&l)[kMaxGroup], uint32_t tmem,
                             int warp, int lane, uint32_t &phase)
{
    const int G = P.group;
    const int tid = threadIdx.x;
    const int cb = k & 1;
    // this warp's O rows: TMEM lanes 32w + j (j < 8) hold head j
    float ov[kHeadDim];
    const uint32_t oaddr = tmem + ((uint32_t)(warp * 32) << 16) + kOCol0 + warp * kHeadDim;
    tc::tmem_ld32(oaddr, *reinterpret_cast<float(*)[32]>(&ov[0]));
    tc::tmem_ld32(oaddr + 32, *reinterpret_cast<float(*)[32]>(&ov[32]));
    tc::tmem_ld_wait();
    tc::fence_before_sync();
#pragma unroll
    for (int j = 0; j < kMaxGroup; ++j) {
        if (j < G) {
            const float ls = warp_sum(l[j]);
            if (lane == 0) {
                sm.cm[cb][warp][j] = m[j];
                sm.cl[cb][warp][j] = ls;
            }
        }
    }
    if (lane < G) {
#pragma unroll
        for (int d = 0; d < kHeadDim; d += 4)
            *reinterpret_cast<float4 *>(&sm.co[cb][warp][lane][d]) =
                make_float4(ov[d], ov[d + 1], ov[d + 2], ov[d + 3]);
    }
    if (!cta_sync(P, sm, phase))
        return false;

    // combine the 4 warps: thread t -> head t/16, dims 4(t%16)..+3
    const int jh = tid >> 4, d0 = (tid & 15) * 4;
    float M = -INFINITY, Ls = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (jh < G) {
#pragma unroll
        for (int w = 0; w < kSoftWarps; ++w)
            M = fmaxf(M, sm.cm[cb][w][jh]);
#pragma unroll
        for (int w = 0; w < kSoftWarps; ++w) {
            const float mw = sm.cm[cb][w][jh];
            const float f = (mw > -INFINITY) ? fast_exp2(mw - M) : 0.f;
            const float4 a = *reinterpret_cast<const float4 *>(&sm.co[cb][w][jh][d0]);
            Ls += f * sm.cl[cb][w][jh];
            o.x += f * a.x;
            o.y += f * a.y;
            o.z += f * a.z;
            o.w += f * a.w;
        }
    }
    const int s = pc.ps, h = pc.ph;
    const long long out_row = ((long long)s * P.num_q_heads + (long long)h * G) * kHeadDim;
    if (pc.flags & kFlagWhole) {
        if (jh < G) {
            const float inv = 1.f / Ls;
            uint2 wv;
            wv.x = pack2<T>(o.x * inv, o.y * inv);
            wv.y = pack2<T>(o.z * inv, o.w * inv);
            *reinterpret_cast<uint2 *>(P.out + out_row + jh * kHeadDim + d0) = wv;
        }
        return true;
    }

    // partial piece: record, arrival count, merge by the CTA that completes the pair
    const int which = (pc.flags & kFlagWhich1) ? 1 : 0;
    float *slot = P.partials + ((long long)blockIdx.x * 2 + which) * kSlotFloats;
    if (jh < G) {
        __stcg(reinterpret_cast<float4 *>(slot + 2 * kMaxGroup + jh * kHeadDim + d0), o);
        if (d0 == 0) {
            __stcg(slot + jh, M);
            __stcg(slot + kMaxGroup + jh, Ls);
        }
    }
    __threadfence();
    if (!cta_sync(P, sm, phase))
        return false;
    const long long B = sm.total, Gc = sm.g_eff;
    const long long c0 = cta_of(pc.pstart, B, Gc);
    const long long c1 = cta_of(pc.pstart + pc.pnb - 1, B, Gc);
    const int pair = s * P.num_kv_heads + h;
    if (tid == 0) {
        __threadfence();
        sm.merge_prev = atomicAdd(P.counters + pair, 1);
    }
    if (!cta_sync(P, sm, phase))
        return false;
    if (sm.merge_prev == (int)(c1 - c0)) {
        __threadfence();
        merge_pieces<T>(P, c0, c1, range_begin(c0, B, Gc) != pc.pstart, out_row, G, tid,
                        kSoftWarps * 32);
        if (tid == 0)
            P.counters[pair] = 0;
    }
    return true;
}

template <typename T, int BS, int NP>
__device__ void tc_softmax(const DecodeParams &P, TcDecodeSmem<NP> &sm, uint32_t tmem, int warp, int lane)
{
    constexpr int TB = kTileKeys / BS;
    const int G = P.group;
    const int t = threadIdx.x;  // key of the tile == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    PieceWalk pc;
    walk_init(P, sm, pc);
    int g = 0, k = 0;
    uint32_t phase = 0;
    bool ok = true;
    while (ok && walk_next<BS>(P, pc)) {
        float m[kMaxGroup], l[kMaxGroup];
#pragma unroll
        for (int j = 0; j < kMaxGroup; ++j) {
            m[j] = -INFINITY;
            l[j] = 0.f;
        }
        const int nt = tiles_of<BS>(pc);
        for (int jt = 0; jt < nt; ++jt, ++g) {
            const int sb = g & 1, st = g % kTcStages;
            if (!wait_or_abort(&sm.s_full[sb], (uint32_t)(g >> 1) & 1u, &sm.abort_flag) ||
                !wait_or_abort(&sm.kv_full[st], (uint32_t)(g / kTcStages) & 1u, &sm.abort_flag)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            float sv[8];
            tc::tmem_ld8(lane_base + sb * kSCols, sv);
            tc::tmem_ld_wait();
            tc::fence_before_sync();
            mbar_arrive(&sm.s_free[sb]);

            const int blk = pc.lo + jt * TB + t / BS;
            const int pos = blk * BS + (t % BS);
            const bool valid = blk < pc.hi && pos < pc.pL && ((sm.loaded[st] >> (t / BS)) & 1u);
            float z[kMaxGroup];
            bool grow = false;
#pragma unroll
            for (int j = 0; j < kMaxGroup; ++j) {
                z[j] = valid ? sv[j] * P.scale_log2 : -INFINITY;
                grow |= (j < G) && (z[j] > m[j] + kRescaleSlack);
            }
            bool rescale = false;
            float alpha_row = 1.f;  // factor of this lane's O row (head lane % 8)
            if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                for (int j = 0; j < kMaxGroup; ++j) {
                    if (j < G) {
                        const float tm = warp_max(z[j]);
                        if (tm > m[j] + kRescaleSlack) {
                            // from -inf the factor is 0 (nothing accumulated yet)
                            const float a = fast_exp2(m[j] - tm);
                            l[j] *= a;
                            if ((lane & 7) == j)
                                alpha_row = a;
                            rescale |= m[j] > -INFINITY;
                            m[j] = tm;
                        }
                    }
                }
            }
            float p[kMaxGroup];
#pragma unroll
            for (int j = 0; j < kMaxGroup; ++j) {
                p[j] = (valid && j < G) ? fast_exp2(z[j] - m[j]) : 0.f;
                l[j] += p[j];
            }
            // P and O of this warp are free once the PV of the previous tile finished
            if (g > 0 && !wait_or_abort(&sm.o_done[warp], (uint32_t)(g - 1) & 1u, &sm.abort_flag)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            if (jt > 0 && __any_sync(0xffffffffu, rescale)) {
                const uint32_t oaddr = lane_base + kOCol0 + warp * kHeadDim;
#pragma unroll
                for (int c = 0; c < kHeadDim; c += 32) {
                    float ov[32];
                    tc::tmem_ld32(oaddr + c, ov);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        ov[e] *= alpha_row;
                    tc::tmem_st32(oaddr + c, ov);
                }
                tc::tmem_st_wait();
            }
            // P[head j][key t]: panel t/64, row j, 16-byte chunk ((t%64)/8) ^ j, element t%8
            {
                const int pn = t >> 6;
                const int ch = (t & 63) >> 3;
#pragma unroll
                for (int j = 0; j < kMaxGroup; ++j) {
                    if (j < G) {
                        const int off = j * 128 + ((ch ^ j) << 4) + (t & 7) * 2;
                        const uint16_t hi = pack1<T>(p[j]);
                        *reinterpret_cast<uint16_t *>(sm.p[0][pn] + off) = hi;
                        if (NP == 2) {
                            const float hv = __uint_as_float((uint32_t)hi << 16);
                            *reinterpret_cast<uint16_t *>(sm.p[NP - 1][pn] + off) = pack1<T>(p[j] - hv);
                        }
                    }
                }
            }
            // a key past the context or in a block not loaded has P = 0, but
            // 0 * NaN is NaN: its V row is zeroed
            if (!valid) {
#pragma unroll
                for (int b = 0; b < kRowBytes; b += 16)
                    *reinterpret_cast<uint4 *>(sm.v[st] + t * kRowBytes + b) = make_uint4(0, 0, 0, 0);
            }
            fence_async_smem();
            tc::fence_before_sync();
            mbar_arrive(&sm.p_full[warp]);
        }
        if (!ok)
            break;
        // the last PV of the piece has finished before its O is read
        if (!wait_or_abort(&sm.o_done[warp], (uint32_t)(g - 1) & 1u, &sm.abort_flag)) {
            ok = false;
            break;
        }
        tc::fence_after_sync();
        ok = tc_piece_end<T, BS, NP>(P, sm, pc, k, m, l, tmem, warp, lane, phase);
        ++k;
    }
    if (!ok)
        set_abort(P, sm);
}

template <typename T, int BS>
__global__ void __launch_bounds__(kTcDecThreads, 1)
    tc_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const DecodeParams P)
{
    constexpr int NP = PSplit<T>::N;
    extern __shared__ unsigned char smem_raw[];
    const uintptr_t a = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    TcDecodeSmem<NP> &sm = *reinterpret_cast<TcDecodeSmem<NP> *>(a);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(&sm.kv_full[i], 1);
            mbar_init(&sm.kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.q_full[i], 1);
            mbar_init(&sm.q_empty[i], 1);
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.s_free[i], kSoftWarps * 32);
        }
        for (int w = 0; w < kSoftWarps; ++w) {
            mbar_init(&sm.p_full[w], 32);
            mbar_init(&sm.o_done[w], 1);
        }
        mbar_init(&sm.mma_idle, 1);
        mbar_init(&sm.cons, kSoftWarps * 32);
        mbar_init_fence();
    }
    // Q rows >= G (the TMA box covers G rows) and P rows >= G stay zero.
    {
        uint4 *z0 = reinterpret_cast<uint4 *>(sm.q);
        constexpr int n = (int)(sizeof(sm.q) + sizeof(sm.p)) / 16;  // q and p are adjacent
        static_assert(offsetof(TcDecodeSmem<NP>, p) == offsetof(TcDecodeSmem<NP>, q) + sizeof(sm.q),
                      "q and p are adjacent");
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            z0[i] = make_uint4(0, 0, 0, 0);
        fence_async_smem();
    }
    if (!decode_prologue<TcDecodeSmem<NP>, BS>(P, sm))
        return;  // no work: every thread of the CTA leaves here, before TMEM is allocated

    if (warp == 4) {
        tc::tmem_alloc(&sm.tmem_base, kTmemAlloc);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 5) {
        tc_producer<T, BS, NP>(P, sm, &tm_q, &tm_k, &tm_v, lane);
    } else if (warp == 4) {
        if (lane == 0)
            tc_mma<T, BS, NP>(P, sm, tmem);
        __syncwarp();
    } else {
        tc_softmax<T, BS, NP>(P, sm, tmem, warp, lane);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 4) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemAlloc);
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
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

bool encode_sw128(CUtensorMap *map, ns_dtype dt, int rank, const void *base, const cuuint64_t *dims,
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

template <typename T, int BS>
struct TcDecodeKernel {
    static constexpr size_t SMEM = tc_decode_smem_bytes<PSplit<T>::N>();
    static cudaError_t prepare()
    {
        static int done_mask = 0;
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return e;
        if (dev < 31 && ((__atomic_load_n(&done_mask, __ATOMIC_RELAXED) >> dev) & 1))
            return cudaSuccess;
        e = cudaFuncSetAttribute(tc_decode_kernel<T, BS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
        if (e == cudaSuccess && dev < 31)
            __atomic_fetch_or(&done_mask, 1 << dev, __ATOMIC_RELAXED);
        return e;
    }
    static cudaError_t launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                              const DecodeParams &P, int ctas, cudaStream_t stream)
    {
        cudaError_t e = prepare();
        if (e != cudaSuccess)
            return e;
        tc_decode_kernel<T, BS><<<ctas, kTcDecThreads, SMEM, stream>>>(tq, tk, tv, P);
        return cudaGetLastError();
    }
    static int ctas_per_sm()
    {
        if (prepare() != cudaSuccess)
            return 1;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tc_decode_kernel<T, BS>, kTcDecThreads, SMEM) !=
                cudaSuccess ||
            n < 1)
            return 1;
        return n;
    }
};

}  // namespace

bool tc_decode_supported(int block_size, int group)
{
    return (block_size == 16 || block_size == 32) && group >= 1 && group <= kMaxGroup;
}

int tc_decode_ctas_per_sm(ns_dtype dtype, int block_size)
{
    if (dtype == NS_BF16)
        return block_size == 16 ? TcDecodeKernel<BF16, 16>::ctas_per_sm() : TcDecodeKernel<BF16, 32>::ctas_per_sm();
    return block_size == 16 ? TcDecodeKernel<F16, 16>::ctas_per_sm() : TcDecodeKernel<F16, 32>::ctas_per_sm();
}

cudaError_t launch_tc_decode(const DecodeParams &P, ns_dtype dtype, int block_size, int num_ctas,
                             cudaStream_t stream)
{
    const int G = P.group;
    CUtensorMap tq, tk, tv;
    {
        // q as rows of 64: [rows * num_q_heads][64]; a box is the G rows of one group
        const long long rows = (long long)P.num_seqs * P.num_q_heads;
        const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)(rows > 0 ? rows : 1)};
        const cuuint64_t strides[1] = {(cuuint64_t)kRowBytes};
        const cuuint32_t box[2] = {(cuuint32_t)kHeadDim, (cuuint32_t)G};
        if (!encode_sw128(&tq, dtype, 2, P.q, dims, strides, box))
            return cudaErrorInvalidValue;
    }
    {
        // pool as [num_blocks][num_kv_heads * bs][64]; a box is one (block, kv head)
        const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)P.num_kv_heads * block_size,
                                    (cuuint64_t)P.num_blocks};
        const cuuint64_t strides[2] = {(cuuint64_t)kRowBytes,
                                       (cuuint64_t)P.num_kv_heads * block_size * kRowBytes};
        const cuuint32_t box[3] = {(cuuint32_t)kHeadDim, (cuuint32_t)block_size, 1};
        if (!encode_sw128(&tk, dtype, 3, P.k_pool, dims, strides, box) ||
            !encode_sw128(&tv, dtype, 3, P.v_pool, dims, strides, box))
            return cudaErrorInvalidValue;
    }
    if (dtype == NS_BF16)
        return block_size == 16 ? TcDecodeKernel<BF16, 16>::launch(tq, tk, tv, P, num_ctas, stream)
                                : TcDecodeKernel<BF16, 32>::launch(tq, tk, tv, P, num_ctas, stream);
    return block_size == 16 ? TcDecodeKernel<F16, 16>::launch(tq, tk, tv, P, num_ctas, stream)
                            : TcDecodeKernel<F16, 32>::launch(tq, tk, tv, P, num_ctas, stream);
}

}  // namespace ns
