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
//  * Warp specialisation.  One producer warp walks the block table and
//    issues TMA bulk copies (cp.async.bulk) of whole (block, kv head) K and V
//    chunks -- block_size*128 contiguous bytes each -- into a STAGES-deep
//    shared-memory ring completed by mbarriers.  NW consumer warps each take
//    one block of a stage.
//  * Consumer lane layout.  Lane (r, c) = (lane>>3, lane&7) owns dims
//    8c..8c+7 of token rows r, r+4, r+8, ... of its block, for all query heads
//    of the GQA group, so one 16-byte shared load feeds every head.  Dot
//    products run on packed fp32 FMA (two per instruction); the 8 partial
//    sums of a token are combined by a 3-step shuffle reduce-scatter that
//    leaves lane c with the score of head c (slot i of lane c holds head
//    i^c, so no lane-dependent selects are needed).  Online softmax per
//    (row, head) with lazy rescaling: the running max moves only when a score
//    exceeds it by more than kRescaleSlack (log2 units), and the result is
//    exact because sum and accumulator share the stale max.
//  * Every wait is bounded; a timeout sets NS_DEV_WAIT_TIMEOUT and the CTA
//    winds down (consumer warps synchronise through an mbarrier with a
//    bounded wait, never through bar.sync, so a warp that leaves early cannot
//    hang the others).
#pragma once

#include "ns_common.cuh"

namespace ns {

// Partial record of one piece of a (sequence, kv head): M[8] (running max,
// log2 units), L[8] (sum of 2^(z-M)), acc[8][64] (unnormalised output).
constexpr int kSlotFloats = 2 * kMaxGroup + kMaxGroup * kHeadDim;
constexpr float kRescaleSlack = 8.0f;

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
};

enum : int {
    kFlagStart = 1,    // first stage of a piece: load q, reset state
    kFlagEnd = 2,      // last stage of a piece: merge warps, write
    kFlagWhole = 4,    // the piece is the whole (sequence, kv head)
    kFlagDone = 8,     // no more work
    kFlagWhich1 = 16,  // partial piece stored in the CTA's second slot
};

struct StageMeta {
    int s, h, blk0, nblk, L, flags;
    int pair_nblk, pad;
    long long pair_start;
    long long new_slot;  // fused: slot of the new token (-1: none)
};

template <int BS, int NW, int STAGES>
struct DecodeSmem {
    uint16_t k[STAGES][NW][BS * kHeadDim];
    uint16_t v[STAGES][NW][BS * kHeadDim];
    uint16_t q[STAGES][kMaxGroup * kHeadDim];
    uint16_t knew[STAGES][kHeadDim];
    uint16_t vnew[STAGES][kHeadDim];
    float2 p[NW][2][4][8];  // (p, p) per [buffer][row][head]
    float mrow[NW][4][8];
    float lrow[NW][4][8];
    float acc[NW][kMaxGroup][kHeadDim];
    float mfin[8];
    float lfin[8];
    StageMeta meta[STAGES];
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t cons;  // consumer-warp rendezvous
    long long scan[32];
    long long b0, b1, total, start_off;
    int start_s, g_eff, merge_prev, abort_flag;
    int plan_split, plan_maxp;
};

__device__ __forceinline__ int nblocks_of(int L, int BS) { return (L + BS - 1) / BS; }

// Context length of sequence s, clamped to what the table can address.
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

template <int BS, int NW, int STAGES>
__device__ __forceinline__ void set_abort(const DecodeParams &P, DecodeSmem<BS, NW, STAGES> &sm)
{
    *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
    raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
}

// Rendezvous of all consumer threads (NW*32 arrivals per phase).
template <int BS, int NW, int STAGES>
__device__ __forceinline__ bool consumer_sync(const DecodeParams &P, DecodeSmem<BS, NW, STAGES> &sm,
                                              uint32_t &phase)
{
    mbar_arrive(&sm.cons);
    const bool ok = wait_or_abort(&sm.cons, phase, &sm.abort_flag);
    phase ^= 1u;
    if (!ok)
        set_abort(P, sm);
    return ok;
}

// ---------------------------------------------------------------------------
// One block of BS tokens for one warp.  LAST: the sequence's last block
// (tokens >= valid are masked; with a fused append, token t_new comes from
// the new-token buffers instead of the pool copy).
// ---------------------------------------------------------------------------
template <typename T, int BS, bool LAST>
__device__ __forceinline__ void process_block(const uint16_t *__restrict__ kb,
                                              const uint16_t *__restrict__ vb, int valid, int t_new,
                                              const uint16_t *knew, const uint16_t *vnew,
                                              const float2 (&q2)[8][4], float2 (&acc)[8][4],
                                              float &m_run, float &l_run, float2 *pbuf, int G,
                                              int lane)
{
    const int c = lane & 7;
    const int r = lane >> 3;
#pragma unroll
    for (int st = 0; st < BS / 4; ++st) {
        const int t = st * 4 + r;
        // ---- scores: partial dot over this lane's 8 dims for all 8 head slots
        uint4 kw = lds128(kb + t * kHeadDim + c * 8);
        if (LAST && t == t_new)
            kw = lds128(knew + c * 8);
        const float2 k0 = unpack2<T>(kw.x), k1 = unpack2<T>(kw.y);
        const float2 k2 = unpack2<T>(kw.z), k3 = unpack2<T>(kw.w);
        float part[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float2 a = fmul2(q2[i][0], k0);
            a = ffma2(q2[i][1], k1, a);
            a = ffma2(q2[i][2], k2, a);
            a = ffma2(q2[i][3], k3, a);
            part[i] = a.x + a.y;
        }
        // reduce-scatter across the row's 8 lanes -> lane c holds head c
#pragma unroll
        for (int i = 0; i < 4; ++i)
            part[i] += __shfl_xor_sync(0xffffffffu, part[i + 4], 4);
#pragma unroll
        for (int i = 0; i < 2; ++i)
            part[i] += __shfl_xor_sync(0xffffffffu, part[i + 2], 2);
        float z = part[0] + __shfl_xor_sync(0xffffffffu, part[1], 1);
        if (LAST && t >= valid)
            z = -INFINITY;

        // ---- online softmax with lazy rescaling
        const bool grow = z > m_run + kRescaleSlack;
        if (__any_sync(0xffffffffu, grow)) {
            const float m_new = grow ? z : m_run;
            // 1 for lanes whose max stays (also at -inf: -inf - -inf would be NaN); 0 from -inf
            const float alpha = grow ? fast_exp2(m_run - z) : 1.f;
            l_run *= alpha;
            m_run = m_new;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float aj = __shfl_sync(0xffffffffu, alpha, (lane & ~7) | j);
                if (j < G) {
                    const float2 a2 = make_float2(aj, aj);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        acc[j][k] = fmul2(acc[j][k], a2);
                }
            }
        }
        float p = fast_exp2(z - m_run);
        if (LAST && !(z > -INFINITY))
            p = 0.f;
        l_run += p;

        // ---- share p of (token t, head c) with the row
        float2 *pb = pbuf + (st & 1) * 32;
        pb[r * 8 + c] = make_float2(p, p);
        __syncwarp();

        // ---- values
        uint4 vw = lds128(vb + t * kHeadDim + c * 8);
        if (LAST && t == t_new)
            vw = lds128(vnew + c * 8);
        float2 v0 = unpack2<T>(vw.x), v1 = unpack2<T>(vw.y);
        float2 v2 = unpack2<T>(vw.z), v3 = unpack2<T>(vw.w);
        if (LAST && t >= valid) {
            v0 = v1 = v2 = v3 = make_float2(0.f, 0.f);
        }
        const float4 *prow = reinterpret_cast<const float4 *>(pb + r * 8);
        float4 pp[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            pp[i] = prow[i];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < G) {
                const float2 pj = (j & 1) ? make_float2(pp[j >> 1].z, pp[j >> 1].w)
                                          : make_float2(pp[j >> 1].x, pp[j >> 1].y);
                acc[j][0] = ffma2(pj, v0, acc[j][0]);
                acc[j][1] = ffma2(pj, v1, acc[j][1]);
                acc[j][2] = ffma2(pj, v2, acc[j][2]);
                acc[j][3] = ffma2(pj, v3, acc[j][3]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// End of a piece: merge the 4 rows x NW warps, then write the output (whole
// pair) or a partial record and, if this CTA completes the pair, merge every
// piece.  Returns false if a rendezvous gave up.
// ---------------------------------------------------------------------------
template <typename T, int BS, int NW, int STAGES>
__device__ bool piece_epilogue(const DecodeParams &P, DecodeSmem<BS, NW, STAGES> &sm,
                               const StageMeta &meta, float2 (&acc)[8][4], float m_run,
                               float l_run, int warp, int lane, uint32_t &phase)
{
    const int c = lane & 7;
    const int r = lane >> 3;
    const int G = P.group;
    const int tid = warp * 32 + lane;
    constexpr int NT = NW * 32;

    sm.mrow[warp][r][c] = m_run;
    sm.lrow[warp][r][c] = l_run;
    if (!consumer_sync(P, sm, phase))
        return false;
    if (tid < 8) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr)
                M = fmaxf(M, sm.mrow[w][rr][tid]);
        float Ls = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const float m = sm.mrow[w][rr][tid];
                if (m > -INFINITY)
                    Ls += sm.lrow[w][rr][tid] * fast_exp2(m - M);
            }
        sm.mfin[tid] = M;
        sm.lfin[tid] = Ls;
    }
    if (!consumer_sync(P, sm, phase))
        return false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j < G) {
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
    }
    if (!consumer_sync(P, sm, phase))
        return false;

    const int s = meta.s, h = meta.h;
    const long long out_row = ((long long)s * P.num_q_heads + (long long)h * G) * kHeadDim;
    if (meta.flags & kFlagWhole) {
        for (int idx = tid; idx < G * kHeadDim; idx += NT) {
            const int j = idx >> 6, d = idx & 63;
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w)
                o += sm.acc[w][j][d];
            P.out[out_row + idx] = pack1<T>(o / sm.lfin[j]);
        }
        return consumer_sync(P, sm, phase);
    }

    // ---- partial piece: store the record, count arrivals, merge if last.
    const int which = (meta.flags & kFlagWhich1) ? 1 : 0;
    float *slot = P.partials + ((long long)blockIdx.x * 2 + which) * kSlotFloats;
    for (int idx = tid; idx < G * kHeadDim; idx += NT) {
        const int j = idx >> 6, d = idx & 63;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w)
            o += sm.acc[w][j][d];
        __stcg(slot + 2 * kMaxGroup + idx, o);
    }
    if (tid < G) {
        __stcg(slot + tid, sm.mfin[tid]);
        __stcg(slot + kMaxGroup + tid, sm.lfin[tid]);
    }
    __threadfence();
    if (!consumer_sync(P, sm, phase))
        return false;
    const long long B = sm.total, Gc = sm.g_eff;
    const long long c0 = cta_of(meta.pair_start, B, Gc);
    const long long c1 = cta_of(meta.pair_start + meta.pair_nblk - 1, B, Gc);
    const int pair = s * P.num_kv_heads + h;
    if (tid == 0) {
        __threadfence();
        sm.merge_prev = atomicAdd(P.counters + pair, 1);
    }
    if (!consumer_sync(P, sm, phase))
        return false;
    if (sm.merge_prev == (int)(c1 - c0)) {
        __threadfence();
        const bool c0_second = range_begin(c0, B, Gc) != meta.pair_start;
        for (int idx = tid; idx < G * kHeadDim; idx += NT) {
            const int j = idx >> 6;
            float M = -INFINITY;
            for (long long cc = c0; cc <= c1; ++cc) {
                const int wh = (cc == c0 && c0_second) ? 1 : 0;
                const float *sl = P.partials + (cc * 2 + wh) * kSlotFloats;
                M = fmaxf(M, __ldcg(sl + j));
            }
            float Ls = 0.f, o = 0.f;
            for (long long cc = c0; cc <= c1; ++cc) {
                const int wh = (cc == c0 && c0_second) ? 1 : 0;
                const float *sl = P.partials + (cc * 2 + wh) * kSlotFloats;
                const float m = __ldcg(sl + j);
                const float f = (m > -INFINITY) ? fast_exp2(m - M) : 0.f;
                Ls += f * __ldcg(sl + kMaxGroup + j);
                o += f * __ldcg(sl + 2 * kMaxGroup + idx);
            }
            P.out[out_row + idx] = pack1<T>(o / Ls);
        }
        if (tid == 0)
            P.counters[pair] = 0;
    }
    return consumer_sync(P, sm, phase);
}

// ---------------------------------------------------------------------------
// Consumer warps.
// ---------------------------------------------------------------------------
template <typename T, int BS, int NW, int STAGES>
__device__ void decode_consumer(const DecodeParams &P, DecodeSmem<BS, NW, STAGES> &sm, int warp,
                                int lane)
{
    const int c = lane & 7;
    const int G = P.group;
    float2 q2[8][4];
    float2 acc[8][4];
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t phase = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            q2[j][k] = make_float2(0.f, 0.f);
            acc[j][k] = make_float2(0.f, 0.f);
        }

    for (int it = 0;; ++it) {
        const int stage = it % STAGES;
        const uint32_t par = (uint32_t)(it / STAGES) & 1u;
        if (!wait_or_abort(&sm.full[stage], par, &sm.abort_flag)) {
            set_abort(P, sm);
            return;
        }
        const StageMeta &meta = sm.meta[stage];  // stays valid until this warp arrives on empty
        const int flags = meta.flags;
        if (flags & kFlagDone)
            return;
        if (flags & kFlagStart) {
            const uint16_t *qs = sm.q[stage];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int head = i ^ c;
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
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    acc[j][k] = make_float2(0.f, 0.f);
            m_run = -INFINITY;
            l_run = 0.f;
        }
        if (warp < meta.nblk) {
            const int blk = meta.blk0 + warp;
            const int nb = nblocks_of(meta.L, BS);
            float2 *pbuf = &sm.p[warp][0][0][0];
            if (blk == nb - 1) {
                const int valid = meta.L - blk * BS;
                const int t_new = P.k_new != nullptr ? valid - 1 : -1;
                process_block<T, BS, true>(sm.k[stage][warp], sm.v[stage][warp], valid, t_new,
                                           sm.knew[stage], sm.vnew[stage], q2, acc, m_run, l_run,
                                           pbuf, G, lane);
                // fused append: the lanes of the new token's row write it to its slot
                if (P.k_new != nullptr && meta.new_slot >= 0 && (t_new & 3) == (lane >> 3)) {
                    const long long slot = meta.new_slot;
                    const long long blkid = slot / BS, off = slot % BS;
                    const long long dst =
                        ((blkid * P.num_kv_heads + meta.h) * BS + off) * kHeadDim + c * 8;
                    *reinterpret_cast<uint4 *>(P.k_pool_w + dst) = lds128(sm.knew[stage] + c * 8);
                    *reinterpret_cast<uint4 *>(P.v_pool_w + dst) = lds128(sm.vnew[stage] + c * 8);
                }
            } else {
                process_block<T, BS, false>(sm.k[stage][warp], sm.v[stage][warp], BS, -1, nullptr,
                                            nullptr, q2, acc, m_run, l_run, pbuf, G, lane);
            }
        }
        if (flags & kFlagEnd) {
            if (!piece_epilogue<T, BS, NW, STAGES>(P, sm, meta, acc, m_run, l_run, warp, lane,
                                                   phase))
                return;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sm.empty[stage]);
    }
}

// ---------------------------------------------------------------------------
// Producer warp.
// ---------------------------------------------------------------------------
template <typename T, int BS, int NW, int STAGES>
struct Producer {
    const DecodeParams &P;
    DecodeSmem<BS, NW, STAGES> &sm;
    int lane;
    int it;
    uint64_t policy;

    // Issue the stages of piece [lo, hi) of pair (s, h).  False on abort.
    __device__ bool piece(int s, int h, int L, int lo, int hi, int flags, long long pair_start,
                          int pair_nblk)
    {
        const int G = P.group;
        const int nb = pair_nblk;
        long long new_slot = -1;
        const bool fused = P.k_new != nullptr;
        for (int base = lo; base < hi; base += 32) {
            const int n32 = min(32, hi - base);
            int phys = -1;
            const long long trow = P.table_row != nullptr ? __ldg(P.table_row + s) : s;
            if (lane < n32) {
                phys = __ldg(P.block_tables + trow * P.max_blocks_per_seq + base + lane);
                if (phys < 0 || (long long)phys >= P.num_blocks) {
                    raise_status(P.status, NS_DEV_BAD_BLOCK_ID);
                    phys = -1;
                }
            }
            const unsigned valid_mask = __ballot_sync(0xffffffffu, phys >= 0);
            if (fused && base + n32 == nb) {
                // the chunk holds the sequence's last block: check the new slot
                const int last_phys = __shfl_sync(0xffffffffu, phys, n32 - 1);
                if (lane == 0) {
                    long long sl = __ldg(P.slot_mapping + s);
                    const long long want = (long long)last_phys * BS + (L - 1) % BS;
                    if (sl != want || last_phys < 0)
                        raise_status(P.status, NS_DEV_FUSED_SLOT);
                    if (sl >= P.num_blocks * BS) {
                        raise_status(P.status, NS_DEV_BAD_SLOT);
                        sl = -1;
                    }
                    new_slot = sl;
                }
                new_slot = __shfl_sync(0xffffffffu, new_slot, 0);
            }
            for (int sub = 0; sub < n32; sub += NW) {
                const int n = min(NW, n32 - sub);
                const int blk0 = base + sub;
                const int stage = it % STAGES;
                const uint32_t par = ((uint32_t)(it / STAGES) & 1u) ^ 1u;
                if (!wait_or_abort(&sm.empty[stage], par, &sm.abort_flag)) {
                    set_abort(P, sm);
                    return false;
                }
                const bool start = blk0 == lo;
                const bool end = blk0 + n == hi;
                const bool has_last = fused && (blk0 + n == nb);
                const unsigned mine = (valid_mask >> sub) & ((1u << n) - 1u);
                const uint32_t bytes = (uint32_t)__popc(mine) * 2u * BS * kRowBytes +
                                       (start ? (uint32_t)G * kRowBytes : 0u) +
                                       (has_last ? 2u * kRowBytes : 0u);
                if (lane == 0) {
                    StageMeta &m = sm.meta[stage];
                    m.s = s;
                    m.h = h;
                    m.blk0 = blk0;
                    m.nblk = n;
                    m.L = L;
                    m.flags = flags | (start ? kFlagStart : 0) | (end ? kFlagEnd : 0);
                    m.pair_nblk = pair_nblk;
                    m.pair_start = pair_start;
                    m.new_slot = has_last ? new_slot : -1;
                    mbar_arrive_expect_tx(&sm.full[stage], bytes);
                }
                __syncwarp();
                const int my_phys = __shfl_sync(0xffffffffu, phys, (sub + lane) & 31);
                if (lane < n && my_phys >= 0) {
                    const long long off = ((long long)my_phys * P.num_kv_heads + h) * BS * kHeadDim;
                    bulk_load(sm.k[stage][lane], P.k_pool + off, BS * kRowBytes, &sm.full[stage],
                              policy);
                    bulk_load(sm.v[stage][lane], P.v_pool + off, BS * kRowBytes, &sm.full[stage],
                              policy);
                }
                if (start && lane == 31) {
                    const long long qoff = ((long long)s * P.num_q_heads + (long long)h * G) * kHeadDim;
                    bulk_load(sm.q[stage], P.q + qoff, G * kRowBytes, &sm.full[stage]);
                }
                if (has_last && lane == 30) {
                    const long long noff = ((long long)s * P.num_kv_heads + h) * kHeadDim;
                    bulk_load(sm.knew[stage], P.k_new + noff, kRowBytes, &sm.full[stage]);
                    bulk_load(sm.vnew[stage], P.v_new + noff, kRowBytes, &sm.full[stage]);
                }
                ++it;
            }
        }
        return true;
    }
};

template <typename T, int BS, int NW, int STAGES>
__device__ void decode_producer(const DecodeParams &P, DecodeSmem<BS, NW, STAGES> &sm, int lane)
{
    Producer<T, BS, NW, STAGES> pr{P, sm, lane, 0, l2_evict_first_policy()};
    bool ok = true;
    if (P.whole_sequences) {
        const long long pairs = (long long)P.num_seqs * P.num_kv_heads;
        for (long long pair = blockIdx.x; ok && pair < pairs; pair += gridDim.x) {
            const int s = (int)(pair / P.num_kv_heads);
            const int h = (int)(pair % P.num_kv_heads);
            const int L = clamped_len(P, s, BS, false);
            const int nb = nblocks_of(L, BS);
            if (nb == 0)
                continue;
            ok = pr.piece(s, h, L, 0, nb, kFlagWhole, -1, nb);
        }
    } else {
        long long pos = sm.b0;
        const long long end = sm.b1;
        int s = sm.start_s;
        long long soff = sm.start_off;
        bool first = true;
        while (ok && pos < end && s < P.num_seqs) {
            const int L = clamped_len(P, s, BS, false);
            const int nb = nblocks_of(L, BS);
            for (int h = 0; ok && h < P.num_kv_heads && pos < end; ++h) {
                const long long pstart = soff + (long long)h * nb;
                const long long pend = pstart + nb;
                if (pend <= pos)
                    continue;
                const int lo = (int)(pos - pstart);
                const int hi = (int)(min(end, pend) - pstart);
                const bool whole = (lo == 0 && hi == nb);
                const int flags = whole ? kFlagWhole : (first ? 0 : kFlagWhich1);
                first = false;
                ok = pr.piece(s, h, L, lo, hi, flags, pstart, nb);
                pos = pstart + hi;
            }
            soff += (long long)P.num_kv_heads * nb;
            ++s;
        }
    }
    bool done_issued = false;
    if (ok) {
        const int stage = pr.it % STAGES;
        const uint32_t par = ((uint32_t)(pr.it / STAGES) & 1u) ^ 1u;
        if (wait_or_abort(&sm.empty[stage], par, &sm.abort_flag)) {
            if (lane == 0) {
                sm.meta[stage].flags = kFlagDone;
                mbar_arrive(&sm.full[stage]);
            }
            done_issued = true;
        } else {
            set_abort(P, sm);
        }
    }
    // After an abort, never leave with bulk copies still landing in this
    // CTA's shared memory.  (Once the done stage is issued the consumers
    // themselves wait for every copy before they finish.)
    if (!done_issued && lane == 0) {
        const int issued = pr.it;
        for (int k = 1; k <= STAGES && k <= issued; ++k) {
            const int i = issued - k;
            if (!mbar_wait(&sm.full[i % STAGES], (uint32_t)(i / STAGES) & 1u)) {
                raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
                break;
            }
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// Prologue: total work, active CTAs, this CTA's range and starting pair.
// Returns false if this CTA has no work.
// ---------------------------------------------------------------------------
template <typename T, int BS, int NW, int STAGES>
__device__ bool decode_prologue(const DecodeParams &P, DecodeSmem<BS, NW, STAGES> &sm)
{
    constexpr int NT = (NW + 1) * 32;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int Hkv = P.num_kv_heads;
    const int per = (P.num_seqs + NT - 1) / NT;
    const int s_lo = min(P.num_seqs, tid * per);
    const int s_hi = min(P.num_seqs, s_lo + per);
    const bool report = blockIdx.x == 0;

    long long mine = 0;
    for (int s = s_lo; s < s_hi; ++s) {
        const int L = clamped_len(P, s, BS, report);
        mine += (long long)Hkv * nblocks_of(L, BS);
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
    if (lane == 31)
        sm.scan[warp] = incl;
    if (tid == 0)
        sm.abort_flag = 0;
    __syncthreads();
    long long before = 0, total = 0;
    for (int w = 0; w < NW + 1; ++w) {
        if (w < warp)
            before += sm.scan[w];
        total += sm.scan[w];
    }
    const long long excl = before + incl - mine;

    long long G;
    if (P.whole_sequences) {
        G = gridDim.x;
    } else {
        const long long minb = P.min_blocks_per_cta > 0 ? P.min_blocks_per_cta : 1;
        G = (total + minb - 1) / minb;
        if (G > (long long)gridDim.x)
            G = gridDim.x;
        if (G < 1)
            G = 1;
    }
    const long long c = blockIdx.x;
    const long long b0 = range_begin(c, total, G);
    const long long b1 = range_begin(c + 1, total, G);
    if (tid == 0) {
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
    if (!P.whole_sequences && c < G && mine > 0 && b0 >= excl && b0 < excl + mine) {
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
    if (blockIdx.x == 0 && !P.whole_sequences && total > 0) {
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
        pl.ctas_active = P.whole_sequences ? (int)min((long long)gridDim.x,
                                                      (long long)P.num_seqs * Hkv)
                                           : (int)G;
        pl.total_blocks = total;
        pl.split_pairs = P.whole_sequences ? 0 : sm.plan_split;
        pl.max_pieces = P.whole_sequences ? 1 : sm.plan_maxp;
        pl.whole_sequences = P.whole_sequences ? 1 : 0;
        for (int i = 0; i < 9; ++i)
            pl.reserved[i] = 0;
        *P.plan = pl;
    }
    if (P.whole_sequences)
        return true;
    return c < G && b0 < b1;
}

template <typename T, int BS, int NW, int STAGES>
__global__ void __launch_bounds__((NW + 1) * 32, 2) paged_decode_kernel(const DecodeParams P)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<DecodeSmem<BS, NW, STAGES> *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], NW);
        }
        mbar_init(&sm.cons, NW * 32);
        mbar_init_fence();
    }
    if (!decode_prologue<T, BS, NW, STAGES>(P, sm))
        return;
    if (warp == NW)
        decode_producer<T, BS, NW, STAGES>(P, sm, lane);
    else
        decode_consumer<T, BS, NW, STAGES>(P, sm, warp, lane);
}

// Host-side launch helpers (defined in the per-type instantiation files).
template <typename T, int BS>
cudaError_t launch_paged_decode(const DecodeParams &P, int num_ctas, cudaStream_t stream);

template <typename T, int BS>
int decode_ctas_per_sm();

}  // namespace ns
