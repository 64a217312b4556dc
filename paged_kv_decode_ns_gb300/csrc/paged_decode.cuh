// paged_decode.cuh -- split-KV paged-attention decode for sm_103a.
//
// What it computes: for every sequence s and query head j (kv head h =
// j / group), out[s][j] = softmax_p(scale * q[s][j] . K_s[p]) . V_s[p] over
// the L_s tokens found through the sequence's block table (nanoserve project
// page, "What I built": fused paged-attention decode with online softmax over
// the block table).  Long walks are split across CTAs and merged by
// log-sum-exp (the flash-decoding split arm of the nanoserve build log, Day
// 74 post).
//
// How (GB300-first design, not the pages' Triton kernel):
//  * Persistent grid.  The KV blocks of all (sequence, kv head) pairs are laid
//    end to end; CTA c of G takes blocks [c*B/G, (c+1)*B/G), so every CTA
//    gets the same number of blocks whatever the length mix.  A pair cut by a
//    CTA boundary yields partial (max, sum, unnormalised output) records; the
//    CTA that finishes a pair's last piece merges them (log-sum-exp) and
//    writes the output.  G is chosen on the device from the real lengths.
//  * Per-warp TMA rings.  Each of the 4 warps of a CTA takes every 4th block
//    of a piece and keeps its own S-slot ring of shared memory fed by TMA bulk
//    copies (cp.async.bulk) of whole (block, kv head) K and V chunks --
//    block_size*128 contiguous bytes each -- issued S blocks ahead of use and
//    completed on the slot's mbarrier.  No warp waits on another warp's
//    progress except at the merge at the end of a piece.
//  * Lane layout.  Lane (r, c) = (lane>>3, lane&7) owns dims 8c..8c+7 of token
//    rows r, r+4, r+8, ... of its block, for all G query heads of the GQA
//    group, so one 16-byte shared load feeds every head.  Dot products run on
//    packed fp32 FMA (two per instruction).  The partial sums of a token are
//    combined by a shuffle reduce-scatter over the row's 8 lanes; the heads
//    are padded to a power of two N and slot i of lane c holds head
//    i ^ (c >> (3 - log2 N)), so the halving steps need no lane-dependent
//    selects and lane c ends with head c >> (3 - log2 N).  All token rows of a
//    block are scored before any softmax work, so the shuffle chains of the
//    rows overlap.
//  * Online softmax per (row, head) in log2 units with lazy rescaling: the
//    running max moves only when a score exceeds it by more than
//    kRescaleSlack, and the result is exact because sum and accumulator share
//    the stale max.
//  * Every wait is bounded; a timeout sets NS_DEV_WAIT_TIMEOUT and the CTA
//    winds down (warps meet through an mbarrier with a bounded wait, never
//    through bar.sync, so a warp that leaves early cannot hang the others),
//    waiting -- again bounded -- for its own copies in flight before it exits.
#pragma once

#include "ns_common.cuh"

namespace ns {

// Partial record of one piece of a (sequence, kv head): M[8] (running max,
// log2 units), L[8] (sum of 2^(z-M)), acc[8][64] (unnormalised output).
constexpr int kSlotFloats = 2 * kMaxGroup + kMaxGroup * kHeadDim;
constexpr float kRescaleSlack = 8.0f;
constexpr int kDecodeWarps = 4;
constexpr int kDefaultMinBlocksPerCta = 32;

struct DecodeParams {
    const uint16_t *q;
    const uint16_t *k_pool;
    const uint16_t *v_pool;
    const int32_t *block_tables;
    const int32_t *context_lens;  // keys of each row (decode: of each sequence)
    const int32_t *table_row;     // nullptr: row i uses table row i; else table_row[i]
    uint16_t *out;
    // fused append (k_new == nullptr when not fused)
    const uint16_t *k_new;
    const uint16_t *v_new;
    const int64_t *slot_mapping;
    uint16_t *k_pool_w;
    uint16_t *v_pool_w;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int max_blocks_per_seq;
    long long num_blocks;
    float scale_log2;  // scale * log2(e)
    int *counters;     // [num_seqs * num_kv_heads], zero between calls
    float *partials;   // [NS_MAX_CTAS][2][kSlotFloats]
    ns_decode_plan *plan;
    unsigned *status;
    int min_blocks_per_cta;
    int whole_sequences;
    int auto_policy;  // no override given: the device may deal whole pairs instead of splitting
};

enum : int {
    kFlagWhole = 4,    // the piece is the whole (sequence, kv head)
    kFlagWhich1 = 16,  // partial piece stored in the CTA's second slot
};

// Reduce-scatter slots: the G heads of a group padded to a power of two.
template <int G>
struct HeadSlots {
    static constexpr int N = G <= 1 ? 1 : (G <= 2 ? 2 : (G <= 4 ? 4 : 8));
    static constexpr int LOG = N == 1 ? 0 : (N == 2 ? 1 : (N == 4 ? 2 : 3));
    static constexpr int SHIFT = 3 - LOG;  // lane c holds head c >> SHIFT
};

// Bytes of K/V each warp keeps in flight (its ring); a build-time tuning knob.
#ifndef NS_DECODE_RING_BYTES
#define NS_DECODE_RING_BYTES 16384
#endif

// Ring depth per warp: NS_DECODE_RING_BYTES of K/V per warp, 2 to 8 slots.
constexpr int decode_stages(int BS)
{
    return (NS_DECODE_RING_BYTES / (BS * 2 * kRowBytes)) < 2 ? 2
           : (NS_DECODE_RING_BYTES / (BS * 2 * kRowBytes)) > 8 ? 8
                                                                : (NS_DECODE_RING_BYTES / (BS * 2 * kRowBytes));
}

template <int BS, int G, int S>
struct DecodeSmem {
    uint16_t k[kDecodeWarps][S][BS * kHeadDim];
    uint16_t v[kDecodeWarps][S][BS * kHeadDim];
    uint16_t q[kDecodeWarps][S][G * kHeadDim];
    uint16_t knew[kDecodeWarps][S][kHeadDim];
    uint16_t vnew[kDecodeWarps][S][kHeadDim];
    float2 p[kDecodeWarps][BS][8];  // (p, p) per [token][head]
    float mrow[kDecodeWarps][4][8];
    float lrow[kDecodeWarps][4][8];
    float acc[kDecodeWarps][G][kHeadDim];
    float mfin[8];
    float lfin[8];
    long long new_slot[kDecodeWarps][S];  // fused append: slot of the new token, or -1
    uint64_t full[kDecodeWarps][S];
    uint64_t cons;  // rendezvous of the 4 warps
    long long scan[32];
    int maxnb[32];
    long long b0, b1, total, start_off;
    int start_s, g_eff, merge_prev, abort_flag;
    int plan_split, plan_maxp;
    int whole;  // 1: whole (sequence, kv head) pairs dealt round-robin, no split
};

__device__ __forceinline__ int nblocks_of(int L, int BS) { return (L + BS - 1) / BS; }

// Context length of row s, clamped to what the table can address.
__device__ __forceinline__ int clamped_len(const DecodeParams &P, int s, int BS, bool report)
{
    int L = __ldg(P.context_lens + s);
    const long long cap = (long long)P.max_blocks_per_seq * BS;
    if (L < 0 || L > cap) {
        if (report)
            raise_status(P.status, NS_DEV_BAD_CONTEXT_LEN);
        L = L < 0 ? 0 : (int)cap;
    }
    return L;
}

// First CTA whose block range contains global block b:  b0(c) = c*B/G.
__device__ __forceinline__ long long cta_of(long long b, long long B, long long G)
{
    return ((b + 1) * G - 1) / B;
}

__device__ __forceinline__ long long range_begin(long long c, long long B, long long G)
{
    return c * B / G;
}

// Bounded wait that also gives up when another warp has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (global_timer_ns() - t0 > kWaitLimitNs)
            return false;
    }
}

template <class Smem>
__device__ __forceinline__ void set_abort(const DecodeParams &P, Smem &sm)
{
    *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
    raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
}

// Rendezvous of all threads of the CTA (4 warps x 32 arrivals per phase).
template <class Smem>
__device__ __forceinline__ bool cta_sync(const DecodeParams &P, Smem &sm, uint32_t &phase)
{
    mbar_arrive(&sm.cons);
    const bool ok = wait_or_abort(&sm.cons, phase, &sm.abort_flag);
    phase ^= 1u;
    if (!ok)
        set_abort(P, sm);
    return ok;
}

// ---------------------------------------------------------------------------
// Walk over the pieces of this CTA: in split mode the runs of one (sequence,
// kv head) pair inside [b0, b1); with whole_sequences the pairs
// blockIdx.x, blockIdx.x + gridDim.x, ...  Every warp runs the same walk.
// ---------------------------------------------------------------------------
struct PieceWalk {
    long long pos, end, soff;
    int s, h, L, nb;
    bool first;
    bool whole;
    // the current piece
    int ps, ph, pL, pnb, lo, hi, flags;
    long long pstart;
};

template <class Smem>
__device__ __forceinline__ void walk_init(const DecodeParams &P, const Smem &sm, PieceWalk &w)
{
    w.whole = sm.whole != 0;
    if (w.whole) {
        w.pos = blockIdx.x;
        w.end = (long long)P.num_seqs * P.num_kv_heads;
    } else {
        w.pos = sm.b0;
        w.end = sm.b1;
    }
    w.soff = sm.start_off;
    w.s = sm.start_s;
    w.h = 0;
    w.L = -1;
    w.nb = 0;
    w.first = true;
}

template <int BS>
__device__ __forceinline__ bool walk_next(const DecodeParams &P, PieceWalk &w)
{
    const int Hkv = P.num_kv_heads;
    if (w.whole) {
        while (w.pos < w.end) {
            const long long pair = w.pos;
            w.pos += gridDim.x;
            const int s = (int)(pair / Hkv);
            const int L = clamped_len(P, s, BS, false);
            const int nb = nblocks_of(L, BS);
            if (nb == 0)
                continue;
            w.ps = s;
            w.ph = (int)(pair % Hkv);
            w.pL = L;
            w.pnb = nb;
            w.lo = 0;
            w.hi = nb;
            w.flags = kFlagWhole;
            w.pstart = -1;
            return true;
        }
        return false;
    }
    while (w.pos < w.end && w.s < P.num_seqs) {
        if (w.L < 0) {
            w.L = clamped_len(P, w.s, BS, false);
            w.nb = nblocks_of(w.L, BS);
            w.h = 0;
        }
        if (w.h >= Hkv) {
            w.soff += (long long)Hkv * w.nb;
            ++w.s;
            w.L = -1;
            continue;
        }
        const long long pstart = w.soff + (long long)w.h * w.nb;
        const long long pend = pstart + w.nb;
        const int h = w.h++;
        if (pend <= w.pos)
            continue;
        w.ps = w.s;
        w.ph = h;
        w.pL = w.L;
        w.pnb = w.nb;
        w.lo = (int)(w.pos - pstart);
        w.hi = (int)(min(w.end, pend) - pstart);
        const bool whole = (w.lo == 0 && w.hi == w.nb);
        w.flags = whole ? kFlagWhole : (w.first ? 0 : kFlagWhich1);
        w.first = false;
        w.pstart = pstart;
        w.pos = pstart + w.hi;
        return true;
    }
    return false;
}

// ---------------------------------------------------------------------------
// Issue side of a warp's ring: walks the same pieces as the consumer and
// issues the TMA copies of this warp's blocks, up to S blocks ahead.
// ---------------------------------------------------------------------------
template <typename T, int BS, int G, int S>
struct Issuer {
    PieceWalk w;
    int i;             // this warp's next block index inside the piece
    bool has;          // a piece is open
    bool done;
    int issued;        // blocks issued so far
    int tab_first;     // first block of the cached table chunk (-1: none)
    int tab_val;       // lane l: phys block of tab_first + 4*l (-1: invalid)
    long long slot_v;  // fused: slot_mapping of the piece's sequence
    uint64_t policy;

    __device__ void init(const DecodeParams &P, const DecodeSmem<BS, G, S> &sm)
    {
        walk_init(P, sm, w);
        i = 0;
        has = false;
        done = false;
        issued = 0;
        tab_first = -1;
        tab_val = -1;
        slot_v = -1;
        policy = l2_evict_first_policy();
    }

    // Issue this warp's next block; false when the walk is exhausted.
    __device__ bool issue_one(const DecodeParams &P, DecodeSmem<BS, G, S> &sm, int warp, int lane)
    {
        int blk;
        while (true) {
            if (!has) {
                if (!walk_next<BS>(P, w)) {
                    done = true;
                    return false;
                }
                has = true;
                i = 0;
                tab_first = -1;
                if (P.k_new != nullptr && w.hi == w.pnb)
                    slot_v = __ldg(P.slot_mapping + w.ps);  // read early, used at the last block
            }
            blk = w.lo + warp + kDecodeWarps * i;
            if (blk < w.hi)
                break;
            has = false;
        }
        if (tab_first < 0 || blk >= tab_first + kDecodeWarps * 32) {
            tab_first = blk;
            const int b = blk + kDecodeWarps * lane;
            tab_val = -1;
            if (b < w.hi) {
                const long long trow = P.table_row != nullptr ? __ldg(P.table_row + w.ps) : w.ps;
                const int v = __ldg(P.block_tables + trow * P.max_blocks_per_seq + b);
                if (v < 0 || (long long)v >= P.num_blocks)
                    raise_status(P.status, NS_DEV_BAD_BLOCK_ID);
                else
                    tab_val = v;
            }
        }
        const int phys = __shfl_sync(0xffffffffu, tab_val, (blk - tab_first) / kDecodeWarps);
        const int slot = issued % S;
        const bool first_of_mine = (i == 0);
        const bool last_of_seq = P.k_new != nullptr && blk == w.pnb - 1;
        const uint32_t bytes = (phys >= 0 ? 2u * BS * kRowBytes : 0u) +
                               (first_of_mine ? (uint32_t)G * kRowBytes : 0u) +
                               (last_of_seq ? 2u * kRowBytes : 0u);
        __syncwarp();  // every lane is done reading this slot's previous contents
        if (lane == 0) {
            long long ns = -1;
            if (last_of_seq) {
                ns = slot_v;
                const long long want = (long long)phys * BS + (w.pL - 1) % BS;
                if (ns != want || phys < 0)
                    raise_status(P.status, NS_DEV_FUSED_SLOT);
                if (ns >= P.num_blocks * BS) {
                    raise_status(P.status, NS_DEV_BAD_SLOT);
                    ns = -1;
                }
            }
            sm.new_slot[warp][slot] = ns;
            fence_async_smem();  // generic-proxy reads of the slot before the async-proxy refill
            uint64_t *bar = &sm.full[warp][slot];
            if (bytes == 0) {
                mbar_arrive(bar);
            } else {
                mbar_arrive_expect_tx(bar, bytes);
                if (phys >= 0) {
                    const long long off = ((long long)phys * P.num_kv_heads + w.ph) * BS * kHeadDim;
                    bulk_load(sm.k[warp][slot], P.k_pool + off, BS * kRowBytes, bar, policy);
                    bulk_load(sm.v[warp][slot], P.v_pool + off, BS * kRowBytes, bar, policy);
                }
                if (first_of_mine) {
                    const long long qoff = ((long long)w.ps * P.num_q_heads + (long long)w.ph * G) * kHeadDim;
                    bulk_load(sm.q[warp][slot], P.q + qoff, G * kRowBytes, bar);
                }
                if (last_of_seq) {
                    const long long noff = ((long long)w.ps * P.num_kv_heads + w.ph) * kHeadDim;
                    bulk_load(sm.knew[warp][slot], P.k_new + noff, kRowBytes, bar);
                    bulk_load(sm.vnew[warp][slot], P.v_new + noff, kRowBytes, bar);
                }
            }
        }
        __syncwarp();
        ++issued;
        ++i;
        return true;
    }
};

// ---------------------------------------------------------------------------
// One block of BS tokens for one warp.  LAST: the sequence's last block
// (tokens >= valid are masked; with a fused append, token t_new comes from
// the new-token buffers instead of the pool copy).
// ---------------------------------------------------------------------------
template <typename T, int BS, int G, bool LAST>
__device__ __forceinline__ void process_block(const uint16_t *__restrict__ kb,
                                              const uint16_t *__restrict__ vb, int valid, int t_new,
                                              const uint16_t *knew, const uint16_t *vnew,
                                              const float2 (&q2)[HeadSlots<G>::N][4],
                                              float2 (&acc)[G][4], float &m_run, float &l_run,
                                              float2 *pbuf, int lane)
{
    constexpr int NS = HeadSlots<G>::N;
    constexpr int SHIFT = HeadSlots<G>::SHIFT;
    constexpr int STEPS = BS / 4;
    const int c = lane & 7;
    const int r = lane >> 3;

    // ---- scores of all token rows of the block
    float z[STEPS];
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
        const int t = st * 4 + r;
        uint4 kw = lds128(kb + t * kHeadDim + c * 8);
        if (LAST && t == t_new)
            kw = lds128(knew + c * 8);
        const float2 k0 = unpack2<T>(kw.x), k1 = unpack2<T>(kw.y);
        const float2 k2 = unpack2<T>(kw.z), k3 = unpack2<T>(kw.w);
        // breadth-first over the head slots: NS independent chains between
        // each dependent step
        float2 a[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i)
            a[i] = fmul2(q2[i][0], k0);
#pragma unroll
        for (int i = 0; i < NS; ++i)
            a[i] = ffma2(q2[i][1], k1, a[i]);
#pragma unroll
        for (int i = 0; i < NS; ++i)
            a[i] = ffma2(q2[i][2], k2, a[i]);
#pragma unroll
        for (int i = 0; i < NS; ++i)
            a[i] = ffma2(q2[i][3], k3, a[i]);
        float part[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i)
            part[i] = a[i].x + a[i].y;
        // halving steps (lane masks 4, 2, 1 from the top), then the lanes that
        // share a head sum what is left
#pragma unroll
        for (int n = NS, m = 4; n > 1; n >>= 1, m >>= 1) {
#pragma unroll
            for (int i = 0; i < n / 2; ++i)
                part[i] += __shfl_xor_sync(0xffffffffu, part[i + n / 2], m);
        }
        float zz = part[0];
#pragma unroll
        for (int m = 4 >> HeadSlots<G>::LOG; m >= 1; m >>= 1)
            zz += __shfl_xor_sync(0xffffffffu, zz, m);
        z[st] = (LAST && t >= valid) ? -INFINITY : zz;
    }

    // ---- online softmax over this lane's rows, lazily rescaled
    float zmax = z[0];
#pragma unroll
    for (int st = 1; st < STEPS; ++st)
        zmax = fmaxf(zmax, z[st]);
    const bool grow = zmax > m_run + kRescaleSlack;
    if (__any_sync(0xffffffffu, grow)) {
        // 1 for lanes whose max stays (also at -inf: -inf - -inf would be NaN); 0 from -inf
        const float alpha = grow ? fast_exp2(m_run - zmax) : 1.f;
        if (grow)
            m_run = zmax;
        l_run *= alpha;
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const float aj = __shfl_sync(0xffffffffu, alpha, (lane & ~7) | (j << SHIFT));
            const float2 a2 = make_float2(aj, aj);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                acc[j][k] = fmul2(acc[j][k], a2);
        }
    }
    float p[STEPS];
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
        p[st] = fast_exp2(z[st] - m_run);
        if (LAST && !(z[st] > -INFINITY))
            p[st] = 0.f;
        l_run += p[st];
    }

    // ---- share p of (token, head) with the row (lanes that share a head
    // write the same value; a padding head lands in an unused slot)
#pragma unroll
    for (int st = 0; st < STEPS; ++st)
        pbuf[(st * 4 + r) * 8 + (c >> SHIFT)] = make_float2(p[st], p[st]);
    __syncwarp();

    // ---- values
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
        const int t = st * 4 + r;
        uint4 vw = lds128(vb + t * kHeadDim + c * 8);
        if (LAST && t == t_new)
            vw = lds128(vnew + c * 8);
        float2 v0 = unpack2<T>(vw.x), v1 = unpack2<T>(vw.y);
        float2 v2 = unpack2<T>(vw.z), v3 = unpack2<T>(vw.w);
        if (LAST && t >= valid)
            v0 = v1 = v2 = v3 = make_float2(0.f, 0.f);
        const float4 *prow = reinterpret_cast<const float4 *>(pbuf + t * 8);
        float4 pp[(G + 1) / 2];
#pragma unroll
        for (int i = 0; i < (G + 1) / 2; ++i)
            pp[i] = prow[i];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const float2 pj = (j & 1) ? make_float2(pp[j >> 1].z, pp[j >> 1].w)
                                      : make_float2(pp[j >> 1].x, pp[j >> 1].y);
            acc[j][0] = ffma2(pj, v0, acc[j][0]);
            acc[j][1] = ffma2(pj, v1, acc[j][1]);
            acc[j][2] = ffma2(pj, v2, acc[j][2]);
            acc[j][3] = ffma2(pj, v3, acc[j][3]);
        }
    }
    __syncwarp();  // the next block rewrites pbuf
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge of the partial records of one (sequence, kv head) pair,
// pieces c0..c1 (the first in its CTA's second slot when c0_second), written
// to out[out_row + j*64 + d] for the G heads.  Threads tid = 0..NT-1 of the
// calling CTA share the G*64 outputs.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ void merge_pieces(const DecodeParams &P, long long c0, long long c1,
                                             bool c0_second, long long out_row, int G, int tid, int NT)
{
    const int npieces = (int)(c1 - c0 + 1);
    constexpr int U = 8;  // records read per round, so their latencies overlap
    for (int idx = tid; idx < G * kHeadDim; idx += NT) {
        const int j = idx >> 6;
        float M = -INFINITY;
        for (int k0 = 0; k0 < npieces; k0 += U) {
            float mk[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = k0 + u;
                const long long cc = c0 + k;
                const int wh = (k == 0 && c0_second) ? 1 : 0;
                mk[u] = k < npieces ? __ldcg(P.partials + (cc * 2 + wh) * kSlotFloats + j) : -INFINITY;
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                M = fmaxf(M, mk[u]);
        }
        float Ls = 0.f, o = 0.f;
        for (int k0 = 0; k0 < npieces; k0 += U) {
            float mk[U], lk[U], ak[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = k0 + u;
                const long long cc = c0 + k;
                const int wh = (k == 0 && c0_second) ? 1 : 0;
                const float *sl = P.partials + (cc * 2 + wh) * kSlotFloats;
                const bool in = k < npieces;
                mk[u] = in ? __ldcg(sl + j) : -INFINITY;
                lk[u] = in ? __ldcg(sl + kMaxGroup + j) : 0.f;
                ak[u] = in ? __ldcg(sl + 2 * kMaxGroup + idx) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float f = (mk[u] > -INFINITY) ? fast_exp2(mk[u] - M) : 0.f;
                Ls += f * lk[u];
                o += f * ak[u];
            }
        }
        P.out[out_row + idx] = pack1<T>(o / Ls);
    }
}

// ---------------------------------------------------------------------------
// End of a piece: merge the 4 rows x 4 warps, then write the output (whole
// pair) or a partial record and, if this CTA completes the pair, merge every
// piece.  Returns false if a rendezvous gave up.
// ---------------------------------------------------------------------------
template <typename T, int BS, int G, int S>
__device__ bool piece_epilogue(const DecodeParams &P, DecodeSmem<BS, G, S> &sm,
                               const PieceWalk &pc, float2 (&acc)[G][4], float m_run, float l_run,
                               int warp, int lane, uint32_t &phase)
{
    constexpr int SHIFT = HeadSlots<G>::SHIFT;
    constexpr int NT = kDecodeWarps * 32;
    const int c = lane & 7;
    const int r = lane >> 3;
    const int tid = warp * 32 + lane;

    if ((c & ((1 << SHIFT) - 1)) == 0 && (c >> SHIFT) < G) {
        sm.mrow[warp][r][c >> SHIFT] = m_run;
        sm.lrow[warp][r][c >> SHIFT] = l_run;
    }
    if (!cta_sync(P, sm, phase))
        return false;
    if (tid < G) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr)
                M = fmaxf(M, sm.mrow[w][rr][tid]);
        float Ls = 0.f;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const float m = sm.mrow[w][rr][tid];
                if (m > -INFINITY)
                    Ls += sm.lrow[w][rr][tid] * fast_exp2(m - M);
            }
        sm.mfin[tid] = M;
        sm.lfin[tid] = Ls;
    }
    if (!cta_sync(P, sm, phase))
        return false;
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const float mj = sm.mrow[warp][r][j];
        const float f = (mj > -INFINITY) ? fast_exp2(mj - sm.mfin[j]) : 0.f;
        const float2 f2 = make_float2(f, f);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float2 a = fmul2(acc[j][k], f2);
            a.x += __shfl_xor_sync(0xffffffffu, a.x, 8);
            a.y += __shfl_xor_sync(0xffffffffu, a.y, 8);
            a.x += __shfl_xor_sync(0xffffffffu, a.x, 16);
            a.y += __shfl_xor_sync(0xffffffffu, a.y, 16);
            if (r == 0)
                *reinterpret_cast<float2 *>(&sm.acc[warp][j][c * 8 + 2 * k]) = a;
        }
    }
    if (!cta_sync(P, sm, phase))
        return false;

    const int s = pc.ps, h = pc.ph;
    const long long out_row = ((long long)s * P.num_q_heads + (long long)h * G) * kHeadDim;
    if (pc.flags & kFlagWhole) {
        for (int idx = tid; idx < G * kHeadDim; idx += NT) {
            const int j = idx >> 6, d = idx & 63;
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < kDecodeWarps; ++w)
                o += sm.acc[w][j][d];
            P.out[out_row + idx] = pack1<T>(o / sm.lfin[j]);
        }
        return cta_sync(P, sm, phase);
    }

    // ---- partial piece: store the record, count arrivals, merge if last.
    const int which = (pc.flags & kFlagWhich1) ? 1 : 0;
    float *slot = P.partials + ((long long)blockIdx.x * 2 + which) * kSlotFloats;
    for (int idx = tid; idx < G * kHeadDim; idx += NT) {
        const int j = idx >> 6, d = idx & 63;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w)
            o += sm.acc[w][j][d];
        __stcg(slot + 2 * kMaxGroup + idx, o);
    }
    if (tid < G) {
        __stcg(slot + tid, sm.mfin[tid]);
        __stcg(slot + kMaxGroup + tid, sm.lfin[tid]);
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
        merge_pieces<T>(P, c0, c1, range_begin(c0, B, Gc) != pc.pstart, out_row, G, tid, NT);
        if (tid == 0)
            P.counters[pair] = 0;
    }
    return cta_sync(P, sm, phase);
}

// ---------------------------------------------------------------------------
// One warp: consume its blocks piece by piece, keeping its ring S blocks ahead.
// ---------------------------------------------------------------------------
template <typename T, int BS, int G, int S>
__device__ void decode_warp(const DecodeParams &P, DecodeSmem<BS, G, S> &sm, int warp, int lane)
{
    constexpr int NS = HeadSlots<G>::N;
    constexpr int SHIFT = HeadSlots<G>::SHIFT;
    const int c = lane & 7;
    float2 q2[NS][4];
    float2 acc[G][4];
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t phase = 0;
#pragma unroll
    for (int i = 0; i < NS; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            q2[i][k] = make_float2(0.f, 0.f);

    Issuer<T, BS, G, S> is;
    is.init(P, sm);
    while (is.issued < S && is.issue_one(P, sm, warp, lane)) {
    }

    PieceWalk pc;
    walk_init(P, sm, pc);
    int consumed = 0;
    bool ok = true;
    while (ok && walk_next<BS>(P, pc)) {
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                acc[j][k] = make_float2(0.f, 0.f);
        m_run = -INFINITY;
        l_run = 0.f;
        for (int blk = pc.lo + warp; blk < pc.hi; blk += kDecodeWarps) {
            while (!is.done && is.issued < consumed + S)
                is.issue_one(P, sm, warp, lane);
            const int slot = consumed % S;
            if (!wait_or_abort(&sm.full[warp][slot], (uint32_t)(consumed / S) & 1u, &sm.abort_flag)) {
                set_abort(P, sm);
                ok = false;
                break;
            }
            if (blk == pc.lo + warp) {
                const uint16_t *qs = sm.q[warp][slot];
#pragma unroll
                for (int i = 0; i < NS; ++i) {
                    const int head = i ^ (c >> SHIFT);
                    if (head < G) {
                        const uint4 w = lds128(qs + head * kHeadDim + c * 8);
                        const float2 sc = make_float2(P.scale_log2, P.scale_log2);
                        q2[i][0] = fmul2(unpack2<T>(w.x), sc);
                        q2[i][1] = fmul2(unpack2<T>(w.y), sc);
                        q2[i][2] = fmul2(unpack2<T>(w.z), sc);
                        q2[i][3] = fmul2(unpack2<T>(w.w), sc);
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            q2[i][k] = make_float2(0.f, 0.f);
                    }
                }
            }
            float2 *pbuf = &sm.p[warp][0][0];
            if (blk == pc.pnb - 1) {
                const int valid = pc.pL - blk * BS;
                const int t_new = P.k_new != nullptr ? valid - 1 : -1;
                process_block<T, BS, G, true>(sm.k[warp][slot], sm.v[warp][slot], valid, t_new,
                                              sm.knew[warp][slot], sm.vnew[warp][slot], q2, acc,
                                              m_run, l_run, pbuf, lane);
                const long long ns = sm.new_slot[warp][slot];
                // fused append: the lanes of the new token's row write it to its slot
                if (P.k_new != nullptr && ns >= 0 && (t_new & 3) == (lane >> 3)) {
                    const long long dst =
                        (((ns / BS) * P.num_kv_heads + pc.ph) * BS + ns % BS) * kHeadDim + c * 8;
                    *reinterpret_cast<uint4 *>(P.k_pool_w + dst) = lds128(sm.knew[warp][slot] + c * 8);
                    *reinterpret_cast<uint4 *>(P.v_pool_w + dst) = lds128(sm.vnew[warp][slot] + c * 8);
                }
            } else {
                process_block<T, BS, G, false>(sm.k[warp][slot], sm.v[warp][slot], BS, -1, nullptr,
                                               nullptr, q2, acc, m_run, l_run, pbuf, lane);
            }
            ++consumed;
        }
        if (ok)
            ok = piece_epilogue<T, BS, G, S>(P, sm, pc, acc, m_run, l_run, warp, lane, phase);
    }
    // Never leave with copies still landing in this warp's slots.
    if (!ok && lane == 0) {
        for (int k = consumed; k < is.issued; ++k)
            if (!mbar_wait(&sm.full[warp][k % S], (uint32_t)(k / S) & 1u)) {
                raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
                break;
            }
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// Prologue: total work, active CTAs, this CTA's range and starting pair.
// Returns false if this CTA has no work.
// ---------------------------------------------------------------------------
template <class Smem, int BS>
__device__ bool decode_prologue(const DecodeParams &P, Smem &sm)
{
    constexpr int NT = kDecodeWarps * 32;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int Hkv = P.num_kv_heads;
    const int per = (P.num_seqs + NT - 1) / NT;
    const int s_lo = min(P.num_seqs, tid * per);
    const int s_hi = min(P.num_seqs, s_lo + per);
    const bool report = blockIdx.x == 0;

    long long mine = 0;
    int my_maxnb = 0;
    for (int s = s_lo; s < s_hi; ++s) {
        const int L = clamped_len(P, s, BS, report);
        mine += (long long)Hkv * nblocks_of(L, BS);
        my_maxnb = max(my_maxnb, nblocks_of(L, BS));
        if (L == 0 && (s % (int)gridDim.x) == (int)blockIdx.x &&
            (P.table_row == nullptr || __ldg(P.table_row + s) >= 0)) {
            uint16_t *o = P.out + (long long)s * P.num_q_heads * kHeadDim;
            for (int i = 0; i < P.num_q_heads * kHeadDim; ++i)
                o[i] = 0;
        }
    }
    // block-wide exclusive scan of `mine`
    long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    int wmax = my_maxnb;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
    if (lane == 31)
        sm.scan[warp] = incl;
    if (lane == 0)
        sm.maxnb[warp] = wmax;
    if (tid == 0)
        sm.abort_flag = 0;
    __syncthreads();
    long long before = 0, total = 0;
    int maxnb = 0;
    for (int w = 0; w < kDecodeWarps; ++w) {
        if (w < warp)
            before += sm.scan[w];
        total += sm.scan[w];
        maxnb = max(maxnb, sm.maxnb[w]);
    }
    const long long excl = before + incl - mine;

    // Split policy from the real lengths and batch size: an even split over
    // G CTAs unless no pair is longer than twice the even share, in which
    // case whole pairs dealt round-robin need no merge at all.
    const long long minb = P.min_blocks_per_cta > 0 ? P.min_blocks_per_cta : 1;
    long long G = (total + minb - 1) / minb;
    if (G > (long long)gridDim.x)
        G = gridDim.x;
    if (G < 1)
        G = 1;
    const long long pairs = (long long)P.num_seqs * Hkv;
    const bool whole = P.whole_sequences ||
                       (P.auto_policy && total > 0 &&
                        (long long)maxnb <= 2 * ((total + G - 1) / G) && pairs <= (long long)gridDim.x);
    if (whole)
        G = gridDim.x;
    const long long c = blockIdx.x;
    const long long b0 = range_begin(c, total, G);
    const long long b1 = range_begin(c + 1, total, G);
    if (tid == 0) {
        sm.whole = whole ? 1 : 0;
        sm.total = total;
        sm.g_eff = (int)G;
        sm.b0 = b0;
        sm.b1 = b1;
        sm.start_s = P.num_seqs;
        sm.start_off = total;
        sm.plan_split = 0;
        sm.plan_maxp = 1;
    }
    __syncthreads();
    if (!whole && c < G && mine > 0 && b0 >= excl && b0 < excl + mine) {
        long long cum = excl;
        for (int s = s_lo; s < s_hi; ++s) {
            const long long w = (long long)Hkv * nblocks_of(clamped_len(P, s, BS, false), BS);
            if (b0 < cum + w) {
                sm.start_s = s;
                sm.start_off = cum;
                break;
            }
            cum += w;
        }
    }
    if (blockIdx.x == 0 && !whole && total > 0) {
        long long cum = excl;
        int split = 0, maxp = 1;
        for (int s = s_lo; s < s_hi; ++s) {
            const int nb = nblocks_of(clamped_len(P, s, BS, false), BS);
            for (int h = 0; h < Hkv && nb > 0; ++h) {
                const long long ps = cum + (long long)h * nb;
                const long long np = cta_of(ps + nb - 1, total, G) - cta_of(ps, total, G) + 1;
                split += np > 1;
                maxp = max(maxp, (int)np);
            }
            cum += (long long)Hkv * nb;
        }
        atomicAdd(&sm.plan_split, split);
        atomicMax(&sm.plan_maxp, maxp);
    }
    __syncthreads();
    if (blockIdx.x == 0 && tid == 0) {
        ns_decode_plan pl;
        pl.ctas_launched = gridDim.x;
        pl.ctas_active = whole ? (int)min((long long)gridDim.x, pairs) : (int)G;
        pl.total_blocks = total;
        pl.split_pairs = whole ? 0 : sm.plan_split;
        pl.max_pieces = whole ? 1 : sm.plan_maxp;
        pl.whole_sequences = whole ? 1 : 0;
        for (int i = 0; i < 9; ++i)
            pl.reserved[i] = 0;
        *P.plan = pl;
    }
    if (whole)
        return c < pairs;
    return c < G && b0 < b1;
}

// CTAs per SM the register allocation is sized for; a build-time tuning knob.
#ifndef NS_DECODE_MIN_CTAS
#define NS_DECODE_MIN_CTAS 2
#endif

template <typename T, int BS, int G, int S>
__global__ void __launch_bounds__(kDecodeWarps * 32, NS_DECODE_MIN_CTAS) paged_decode_kernel(const DecodeParams P)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<DecodeSmem<BS, G, S> *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int w = 0; w < kDecodeWarps; ++w)
            for (int i = 0; i < S; ++i)
                mbar_init(&sm.full[w][i], 1);
        mbar_init(&sm.cons, kDecodeWarps * 32);
        mbar_init_fence();
    }
    if (!decode_prologue<DecodeSmem<BS, G, S>, BS>(P, sm))
        return;
    decode_warp<T, BS, G, S>(P, sm, warp, lane);
}

// Host-side launch helpers (defined in the per-type instantiation files).
template <typename T, int BS, int G>
cudaError_t launch_paged_decode(const DecodeParams &P, int num_ctas, cudaStream_t stream);

template <typename T, int BS, int G>
int decode_ctas_per_sm();

}  // namespace ns
