// paged_decode.cuh -- split-KV paged-attention decode for sm_103a (CUDA cores).
//
// What it computes: for every sequence s and query head j (kv head h =
// j / group), out[s][j] = softmax_p(scale * q[s][j] . K_s[p]) . V_s[p] over
// the L_s tokens found through the sequence's block table (nanoserve project
// page, "What I built": fused paged-attention decode with online softmax over
// the block table).  Long walks are split and the parts merged by
// log-sum-exp (the flash-decoding split arm of the nanoserve build log, Day
// 74 post).
//
// How (GB300-first design, not the pages' Triton kernel):
//  * Workers are warps.  The KV blocks of all (sequence, kv head) pairs are
//    laid end to end (each pair counted kPieceCost blocks longer) and worker
//    c of Gw takes an equal run of them, so every warp gets the same share
//    whatever the length mix, and no warp ever waits on another: a pair cut
//    by a worker boundary yields a partial (max, sum, unnormalised output)
//    record written by the warp alone; at the end of its ring the warp
//    counts its records, and the warp whose count completes a pair queues
//    its log-sum-exp merge, which the CTA's idle warps run in parts of 1-8
//    query heads.  Gw is chosen on the device from the real lengths and the
//    batch (read_split); when no pair is long, whole pairs are dealt
//    round-robin and nothing is merged.
//  * Per-warp TMA rings, fed by a producer warpgroup.  Each consumer warp
//    streams its range through its own ring of S slots of TOK tokens (32 at
//    head_dim 64, 16 at 128): TMA bulk copies (cp.async.bulk) of the K and V
//    rows of TOK/bs whole blocks, issued S steps ahead of use, L2
//    evict-first, completed on the slot's mbarrier.  The first step of a
//    piece also brings the group's q rows, and with a fused append the step
//    that holds the new token brings its K/V rows.  Block-table entries are
//    read one step ahead.
//  * Lane layout (head_dim 64).  Lane (r, c) = (lane>>3, lane&7) owns dims
//    8c..8c+7 of token rows r, r+4, ..., r+28 of a step, for all G query
//    heads of the GQA group, so one 16-byte shared load feeds every head.
//    Scores run on packed fp32 FMA with two heads per instruction (q held as
//    head pairs); the partial sums of a token are combined by a shuffle
//    reduce-scatter over the row's lanes; the heads are padded to a power
//    of two N and slot i of lane c holds head i ^ (c >> (3 - log2 N)), so
//    the halving steps need no lane-dependent selects and lane c ends with
//    head c >> (3 - log2 N).  At head_dim 128 a row spans 16 lanes.
//  * Online softmax per (row group, head) in log2 units with lazy
//    rescaling: the running max moves only when a score exceeds it by more
//    than kRescaleSlack, and the result is exact because sum and accumulator
//    share the stale max.
//  * q8_0 pools (Q8): a step carries each row's int8 codes and fp16 block
//    scales; codes convert exactly to fp32 and the scales apply per
//    32-element block; the fused append quantises the new token.
//  * Every wait is bounded; a timeout sets NS_DEV_WAIT_TIMEOUT and the warp
//    stops, waiting -- again bounded -- for its own copies in flight.
#pragma once

#include "ns_common.cuh"

namespace ns {

// Partial record of one piece of a (sequence, kv head): M[8] (running max,
// log2 units), L[8] (sum of 2^(z-M)), acc[8][64] (unnormalised output).
// Geometry of the decode for head dim D: a token row of one head spans COLS
// lanes of 8 elements; a warp holds ROWS rows at once (a row group); a ring
// step is 8 row groups, TOK tokens.  D 64: 8 lanes, 4 rows, 32 tokens; D 128:
// 16 lanes, 2 rows, 16 tokens, so that registers and ring bytes per step stay
// the same.  A partial record is M[8], L[8], acc[8][D].
template <int D>
struct Geo {
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static constexpr int COLS = D / 8;
    static constexpr int LOGC = D == 64 ? 3 : 4;
    static constexpr int ROWS = 32 / COLS;
    static constexpr int TOK = 8 * ROWS;
    static constexpr int ROW_BYTES = 2 * D;
    static constexpr int SLOT_FLOATS = 2 * kMaxGroup + kMaxGroup * D;
};
// Floats of a partial record for a runtime head dim (host side).
__host__ __device__ constexpr int slot_floats(int head_dim) { return 2 * kMaxGroup + kMaxGroup * head_dim; }
constexpr float kRescaleSlack = 8.0f;
// One CTA per SM: two consumer warpgroups (8 warps, one worker each) and a
// producer warpgroup.  (Measured alternative: 12 consumers, two per ring
// splitting the query heads, issued 22% more instructions and ran slower.)
constexpr int kConsumerWarps = 8;
// Row groups (4 tokens each) whose scores are computed together: 2 measured
// 1.3% faster than 1 and 4 on the batch-256 decode.
constexpr int kQkRows = 2;
// Row groups of the values pass a trip in the short-walk kernels, which the
// host takes when no worker can have more than a few steps: less code to
// fetch (batch 32 19.56 -> 18.98 us, 4 sequences 13.41 -> 13.10), where batch
// 256 ran slower with it (57.6 -> 59.3 us) and keeps the whole unroll.
constexpr int kShortWalkValuesUnroll = 4;
constexpr int kZeroElems = 2048;       // 16-bit zeros: the largest step of K or V rows
constexpr int kMaxWorkers = 2048;      // split workers (each has two record slots)
constexpr int kDefaultMinBlocksPerCta = 64;  // spread over a CTA's workers
constexpr int kLensCache = 256;        // context lengths kept in shared memory
// Split cost of a (sequence, kv head) pair beyond its blocks: the even split
// counts kPieceCost virtual blocks at the start of every pair, so a worker
// whose range crosses many pair boundaries (a piece end, a partial last
// step, an arrival count and perhaps a merge each) gets fewer real blocks.
// (2, 3 and 4 measured alike on the batch-256 decode; 1 and 6 slower.)
constexpr int kPieceCost = 4;
// Pieces the automatic split aims at for the longest pair when the batch is
// small, and the pairs per warp below which every warp takes a range
// (measured against 8 blocks a worker: the 4-sequence step 16.4 -> 13.3 us,
// batch 32 20.5 -> 20.2 us, 8 x 4096 tokens 23.2 -> 21.5 us).
constexpr int kAutoPieces = 32;

// Length of a pair in the split's coordinates (0 for a pair with no block).
__host__ __device__ __forceinline__ int pair_span(int nb) { return nb > 0 ? nb + kPieceCost : 0; }

// The split's coordinates are 32-bit: a call fits when its pairs, each at
// most max_blocks_per_seq + kPieceCost long, add up to at most INT32_MAX.
inline bool split_fits(long long rows, long long num_kv_heads, long long max_blocks_per_seq)
{
    return rows * num_kv_heads * (max_blocks_per_seq + kPieceCost) <= 0x7fffffffLL;
}

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
    // q8_0 pools (the Q8 kernels): int8 codes [NB][Hkv][bs][64] and fp16
    // scales [NB][Hkv][bs][2], one scale per 32 consecutive elements of a row
    const int8_t *k_codes;
    const int8_t *v_codes;
    const uint16_t *k_scales;
    const uint16_t *v_scales;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int max_blocks_per_seq;
    long long num_blocks;
    float scale_log2;  // scale * log2(e)
    int *counters;     // [num_seqs * num_kv_heads], zero between calls
    float *partials;   // [kMaxWorkers][2][Geo<D>::SLOT_FLOATS]
    ns_decode_plan *plan;
    unsigned *status;
    int min_blocks_per_cta;
    int whole_sequences;
    int auto_policy;  // no override given: the device may deal whole pairs instead of splitting
    int overlap;      // launched as a programmatic dependent: wait for the previous grid (see the prologue)
    int pack;         // number workers CTA-major even when only some have work
    unsigned long long wait_limit_ns;  // consumers' waits for a ring step (the producer's own drain keeps kWaitLimitNs)
    // A group of more than 8 query heads runs as kv_sub groups of group / kv_sub
    // heads: num_kv_heads and group above count these virtual kv heads, and
    // virtual head h reads the pools' (and the new K/V's) head h / kv_sub.
    int kv_sub;
    int merge_levels;  // host: 0 automatic, 1 or 2 forced (the kernel instantiation follows it)
};

// The pools' kv heads, and the pools' head of virtual kv head h.
__device__ __forceinline__ int pool_heads(const DecodeParams &P) { return P.num_kv_heads / max(P.kv_sub, 1); }
__device__ __forceinline__ int pool_head(const DecodeParams &P, int h) { return h / max(P.kv_sub, 1); }
// Whether virtual kv head h stores the new token into the pools (one of each
// pool head's virtual heads does).
__device__ __forceinline__ bool stores_new_token(const DecodeParams &P, int h) { return h % max(P.kv_sub, 1) == 0; }

// Source of the zero-filled rows of a step (32 rows of 64 elements).
static __device__ __align__(128) uint16_t g_zero_rows[kZeroElems];

// Merges queued by consumers and run by the consumers whose rings are done.
// A ring holds at most two partial pieces (the first and last of its range),
// so at most 2 x 8 merges fall to one CTA.  A merge is cut into parts of hpp
// query heads each, so that several warps can share a long one; a part is
// taken by advancing the cursor head = job * kMergeParts + part.
constexpr int kMergeQueue = 32;
constexpr int kMergeParts = 16;
struct MergeJob {
    long long c0, c1, out_row;
    int pair, c0_second;  // c0_second: bit 0 the first record is in c0's second slot; kJobPerCta
    int hpp, nparts;      // query heads per part, parts
};
constexpr int kJobPerCta = 2;  // a two-level merge over one record per CTA
struct MergeQueue {
    MergeJob job[kMergeQueue];
    int ready[kMergeQueue];
    int tail;  // entries taken by producers of jobs
    int head;  // cursor of the next part to run
    int done;  // consumer warps finished
};

// Thread block: the consumer warpgroups and one producer warpgroup; the
// registers a thread gets at launch, then the shares setmaxnreg moves to.
constexpr int kDecodeThreads = (kConsumerWarps + 4) * 32;
constexpr int kLaunchRegs = 65536 / kDecodeThreads / 8 * 8;  // 168 for 8 consumers
// Producer back-off when no slot is free (ns; the rings hold 3 steps): 200 and
// 1000 measured alike.
constexpr unsigned kProducerIdleNs = 500;
// The producer warpgroup's registers (the consumers get the rest of the
// launch allocation).
constexpr int kProducerRegs = 88;
constexpr int kConsumerRegs = (kLaunchRegs * kDecodeThreads - kProducerRegs * 128) / (kConsumerWarps * 32) / 8 * 8;
static_assert(kConsumerWarps % 4 == 0, "consumer warpgroups");
static_assert(kConsumerRegs * kConsumerWarps * 32 + kProducerRegs * 128 <= kLaunchRegs * kDecodeThreads,
              "register shares exceed the launch allocation");

// Reduce-scatter slots: the G heads of a group padded to a power of two.
// PSTRIDE: floats per token row of the p buffer, at least 4 so that rows
// stay 16-byte aligned for the float4 loads of the values pass.
template <int G>
struct HeadSlots {
    static constexpr int N = G <= 1 ? 1 : (G <= 2 ? 2 : (G <= 4 ? 4 : 8));
    static constexpr int LOG = N == 1 ? 0 : (N == 2 ? 1 : (N == 4 ? 2 : 3));
    static constexpr int PSTRIDE = N < 4 ? 4 : N;
};

// A consumer lane's query registers (pre-scaled by scale * log2 e), for the
// lane's 8 dims 8c..8c+7:
//  * two or more head slots: head pairs, q2[m*8 + d] = (q[slot 2m][8c+d],
//    q[slot 2m+1][8c+d]), so one packed FMA serves two heads;
//  * one head slot: dim pairs, q2[k] = (q[8c+2k], q[8c+2k+1]).
template <int G>
struct QRegs {
    static constexpr int N = HeadSlots<G>::N * 4;
};

// Rings (workers) of a CTA and how producer lanes serve them: lane i of
// producer warp p serves ring i * PW + p, so that rings 0..PW-1 (the only
// ones with work when few workers are active) each have a warp of their own.
template <int G>
struct DecodeShape {
    static constexpr int NG = kConsumerWarps;  // rings = workers per CTA
    static constexpr int SERVED = (NG + 3) / 4;  // two rings per producer warp: three measured slower
    static constexpr int PW = (NG + SERVED - 1) / SERVED;  // producer warps
    static constexpr int PSTRIDE = HeadSlots<G>::PSTRIDE;  // p buffer row of a warp
    static_assert(PW <= 4 && PW * SERVED == NG, "producer lanes");
};

enum : int {
    kFlagWhole = 4,    // the piece is the whole (sequence, kv head)
    kFlagWhich1 = 16,  // partial piece stored in the worker's second record slot
    kFlagNewTok = 64,  // fused append: this step holds the new token
};

// What the producer tells a consumer about one ring slot.
struct alignas(16) SlotMeta {
    int ps, ph, pL, flags;      // the pair; piece flags (kFlag*)
    int pspan, step, nsteps;    // nsteps: steps of the piece; 0 = a piece with no key
                                // (record only); -1 = no more work
    int t_new;                  // fused append: the new token's row in the step
    long long pstart;           // the pair's place in the split
    long long new_slot;         // fused append: checked pool slot, or -1
    uint32_t vmask;             // bit t: token t of the step is a key
    int pad[3];
};

__device__ __forceinline__ void put_meta(SlotMeta &mt, int ps, int ph, int pL, int flags, int pspan, int step,
                                         int nsteps, int t_new, long long pstart, long long new_slot,
                                         uint32_t vmask)
{
    int4 *v = reinterpret_cast<int4 *>(&mt);
    v[0] = make_int4(ps, ph, pL, flags);
    v[1] = make_int4(pspan, step, nsteps, t_new);
    *reinterpret_cast<longlong2 *>(&mt.pstart) = make_longlong2(pstart, new_slot);
    mt.vmask = vmask;
}

// The fields of a piece that its end needs.
struct PieceRef {
    int ps, ph, flags, pspan, pstart;
};



// One ring slot: K and V rows of one 32-token step and the q rows that ride
// with a piece's first step.  With a fused append the new token's K/V are
// copied straight into their row of the step.
template <int G, bool Q8, int D>
struct DecodeSlot {
    uint16_t k[Geo<D>::TOK * D];
    uint16_t v[Geo<D>::TOK * D];
    uint16_t q[G * D];
};

// q8_0 pools: a step holds each row's 64 int8 codes and 2 fp16 scales, and the
// new token's 16-bit K/V rows (fused append), which the consumer quantises.
constexpr int kQ8Block = 32;                        // elements per scale
constexpr int kQ8Scales = kHeadDim / kQ8Block;      // scales per row
constexpr int kQ8CodeRow = kHeadDim;                // bytes of a row's codes
constexpr int kQ8ScaleRow = kQ8Scales * 2;          // bytes of a row's scales
template <int G>
struct DecodeSlot<G, true, 64> {
    int8_t k[Geo<64>::TOK * kHeadDim];
    int8_t v[Geo<64>::TOK * kHeadDim];
    uint16_t ks[Geo<64>::TOK * kQ8Scales];
    uint16_t vs[Geo<64>::TOK * kQ8Scales];
    uint16_t q[G * kHeadDim];
    uint16_t knew[kHeadDim];
    uint16_t vnew[kHeadDim];
};

template <int BS, int G, int S, bool Q8 = false, int D = 64>
struct DecodeSmem {
    static constexpr int NG = DecodeShape<G>::NG;
    DecodeSlot<G, Q8, D> ring[NG][S];
    float p[kConsumerWarps][Geo<D>::TOK][DecodeShape<G>::PSTRIDE];  // p per consumer warp [token][head]
    SlotMeta meta[NG][S];
    uint64_t full[NG][S];                    // producer -> consumers: the step has landed
    uint64_t empty[NG][S];                   // consumers -> producer: the slot may be refilled
    static constexpr int STAGES = S;
    // prologue scan of the split coordinates (pair blocks plus piece costs):
    // per warp its total, largest pair and live pairs; per thread its
    // exclusive offset inside its warp
    int wtot[kDecodeThreads / 32];
    int wmax[kDecodeThreads / 32];
    int wpairs[kDecodeThreads / 32];
    int toff[kDecodeThreads];
    MergeQueue mq;
    int lens[kLensCache];                    // clamped context lengths of rows 0..kLensCache-1
    int abort_flag;  // set by a warp that gave up waiting
    int plan_split, plan_maxp;
    // two-level merges: pieces of a cut pair in this CTA that have arrived,
    // by the pair's first worker in the CTA
    int cta_count[kConsumerWarps];
};

// Slots per ring: as many (up to four) as fit in a CTA's shared memory.
constexpr size_t kMaxDynSmem = 227 * 1024;
template <int BS, int G, bool Q8 = false, int D = 64>
constexpr int decode_stages()
{
    return sizeof(DecodeSmem<BS, G, 4, Q8, D>) <= kMaxDynSmem   ? 4
           : sizeof(DecodeSmem<BS, G, 3, Q8, D>) <= kMaxDynSmem ? 3
                                                                 : 2;
}

__device__ __forceinline__ int nblocks_of(int L, int BS) { return (L + BS - 1) / BS; }

// Worker number of ring `ring` of this CTA (ng rings).  When only some workers have
// work (wmajor), warp-major, so that they are spread over every SM before any
// SM gets two; when all have work, CTA-major, so that the warps of a CTA walk
// neighbouring runs of the same sequences.
__device__ __forceinline__ int worker_id(int ring, bool wmajor, int ng)
{
    return wmajor ? ring * (int)gridDim.x + (int)blockIdx.x : (int)blockIdx.x * ng + ring;
}

// The split of the KV work over the workers.  Every CTA computes the same one
// from the context lengths.  The pairs' blocks (each pair counted kPieceCost
// blocks longer) are laid end to end and cut into gw ranges; the
// coordinates are 32-bit because the host refuses calls whose
// pairs * (max_blocks_per_seq + kPieceCost) exceed INT32_MAX.
struct Split {
    int total;        // blocks plus piece costs over all (sequence, kv head) pairs
    int gw;           // split workers
    int q, r;         // total = q * gw + r: workers c < r hold q + 1 blocks, the rest q
    int live_pairs;   // pairs with at least one key
    bool whole;       // whole pairs dealt round-robin, nothing merged
    bool wmajor;      // workers numbered warp-major
};

// First block of worker c's range.
__device__ __forceinline__ int range_begin(int c, int q, int r) { return c * q + min(c, r); }

// The worker whose range holds block b (0 <= b < total).
__device__ __forceinline__ int worker_of(int b, int q, int r)
{
    const int big = r * (q + 1);
    return b < big ? b / (q + 1) : r + (b - big) / q;
}

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


// ---------------------------------------------------------------------------
// Walk over the pieces of one worker: in split mode the runs of one
// (sequence, kv head) pair inside [b0, b1); with whole pairs the pairs
// w, w + stride, w + 2 stride, ...
// ---------------------------------------------------------------------------
struct PieceWalk {
    const int *lens;  // shared-memory copy of the first kLensCache clamped lengths
    int pos, end, soff, stride;
    int s, h, L, nb;
    bool first;
    bool whole;
    // the current piece: real blocks [lo, hi) of pair (ps, ph); pstart and
    // pspan place the whole pair in the split's coordinates
    int ps, ph, pL, pnb, lo, hi, flags, pspan;
    int pstart;
};

template <int BS>
__device__ __forceinline__ int len_at(const DecodeParams &P, const PieceWalk &w, int s)
{
    return s < kLensCache ? w.lens[s] : clamped_len(P, s, BS, false);
}

// Start of worker wk's walk.  Split mode: the range [b0, b1) and the
// sequence that holds b0, found from the prologue scan (the warp, then the
// thread chunk by binary search, then the chunk's sequences).  Whole mode:
// pairs wk, wk + stride, ...
template <int BS, class Smem>
__device__ __forceinline__ void walk_init(const DecodeParams &P, const Smem &sm, const Split &sp, int wk,
                                          PieceWalk &w)
{
    constexpr int NWARPS = kDecodeThreads / 32;
    const int Hkv = P.num_kv_heads;
    w.lens = sm.lens;
    w.whole = sp.whole;
    w.first = true;
    w.h = 0;
    w.L = -1;
    w.nb = 0;
    w.s = P.num_seqs;
    w.soff = 0;
    w.stride = 0;
    w.pos = w.end = 0;
    if (sp.whole) {
        w.pos = wk;
        w.stride = (int)gridDim.x * Smem::NG;
        w.end = P.num_seqs * Hkv;
        return;
    }
    if (wk >= sp.gw)
        return;
    const int b0 = range_begin(wk, sp.q, sp.r), b1 = range_begin(wk + 1, sp.q, sp.r);
    w.pos = b0;
    w.end = b1;
    if (b1 <= b0)
        return;
    int base = 0, ws = 0;
    for (; ws < NWARPS - 1; ++ws) {
        const int t = sm.wtot[ws];
        if (base + t > b0)
            break;
        base += t;
    }
    int lo = 0, hi = 31;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (base + sm.toff[ws * 32 + mid] <= b0)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int t = ws * 32 + lo;
    const int per = (P.num_seqs + kDecodeThreads - 1) / kDecodeThreads;
    int s = min(P.num_seqs, t * per);
    int soff = base + sm.toff[t];
    while (s < P.num_seqs) {  // whole sequences before b0
        const int n = Hkv * pair_span(nblocks_of(len_at<BS>(P, w, s), BS));
        if (soff + n > b0)
            break;
        soff += n;
        ++s;
    }
    w.s = s;
    w.soff = soff;
}

template <int BS>
__device__ __forceinline__ bool walk_next(const DecodeParams &P, PieceWalk &w)
{
    const int Hkv = P.num_kv_heads;
    if (w.whole) {
        while (w.pos < w.end) {
            const int pair = w.pos;
            w.pos += w.stride;
            const int s = pair / Hkv;
            const int L = len_at<BS>(P, w, s);
            const int nb = nblocks_of(L, BS);
            if (nb == 0)
                continue;
            w.ps = s;
            w.ph = pair % Hkv;
            w.pL = L;
            w.pnb = nb;
            w.lo = 0;
            w.hi = nb;
            w.flags = kFlagWhole;
            w.pstart = -1;
            w.pspan = pair_span(nb);
            return true;
        }
        return false;
    }
    while (w.pos < w.end && w.s < P.num_seqs) {
        if (w.L < 0) {
            w.L = len_at<BS>(P, w, w.s);
            w.nb = nblocks_of(w.L, BS);
            w.h = 0;
        }
        const int span = pair_span(w.nb);
        if (w.h >= Hkv) {
            w.soff += Hkv * span;
            ++w.s;
            w.L = -1;
            continue;
        }
        const int pstart = w.soff + w.h * span;
        const int pend = pstart + span;
        const int h = w.h++;
        if (pend <= w.pos)
            continue;
        const int lo_v = w.pos - pstart;
        const int hi_v = min(w.end, pend) - pstart;
        w.ps = w.s;
        w.ph = h;
        w.pL = w.L;
        w.pnb = w.nb;
        w.lo = max(lo_v - kPieceCost, 0);  // the virtual blocks hold no keys
        w.hi = max(hi_v - kPieceCost, 0);
        const bool whole = (lo_v == 0 && hi_v == span);
        w.flags = whole ? kFlagWhole : (w.first ? 0 : kFlagWhich1);
        w.first = false;
        w.pstart = pstart;
        w.pspan = span;
        w.pos = pstart + hi_v;
        return true;
    }
    return false;
}

// One past the last key of a piece (inside the pair).
template <int BS>
__device__ __forceinline__ int piece_end_token(const PieceWalk &w)
{
    return min(w.hi * BS, w.pL);
}

// Steps (TOK-token ring slots) of a piece: step i covers keys
// lo*bs + TOK*i .. lo*bs + TOK*i + TOK-1 of the pair, i.e. TOK/bs whole blocks.
template <int BS, int TOK>
__device__ __forceinline__ int steps_of(const PieceWalk &w)
{
    return max(0, (piece_end_token<BS>(w) - w.lo * BS + TOK - 1) / TOK);
}

// First token (inside the pair) of step i of the piece.
template <int BS, int TOK>
__device__ __forceinline__ int step_token0(const PieceWalk &w, int i)
{
    return w.lo * BS + i * TOK;
}

// ---------------------------------------------------------------------------
// One 32-token step for one warp.  Tokens of the step that are not keys
// (bit t of vmask clear) get score -inf, so p = 0; their rows in the slot are
// zero-filled by the producer, so p * v adds nothing.
// ---------------------------------------------------------------------------
// A row's 8 elements of this lane (dims 8c..8c+7) from a ring slot, as four
// fp32 pairs, and (q8_0) the row's scale for those dims.  16-bit pools: the
// elements themselves, scale 1.  q8_0: the codes, converted exactly (a code
// byte, offset by 128, is placed in the mantissa of 2^23 and 2^23 + 128 is
// subtracted), and the fp16 scale of the 32-element block.
template <typename T, int G, bool Q8, int D>
struct RowLoad;

template <typename T, int G, int D>
struct RowLoad<T, G, false, D> {
    static __device__ __forceinline__ void k(const DecodeSlot<G, false, D> &sl, int row, int c, float2 (&x)[4], float &d)
    {
        const uint4 w = lds128(sl.k + row * D + c * 8);
        x[0] = unpack2<T>(w.x);
        x[1] = unpack2<T>(w.y);
        x[2] = unpack2<T>(w.z);
        x[3] = unpack2<T>(w.w);
        d = 1.f;
    }
    static __device__ __forceinline__ void v(const DecodeSlot<G, false, D> &sl, int row, int c, float2 (&x)[4], float &d)
    {
        const uint4 w = lds128(sl.v + row * D + c * 8);
        x[0] = unpack2<T>(w.x);
        x[1] = unpack2<T>(w.y);
        x[2] = unpack2<T>(w.z);
        x[3] = unpack2<T>(w.w);
        d = 1.f;
    }
};

__device__ __forceinline__ float2 q8_code_pair(uint32_t biased, int k)
{
    const float2 f = make_float2(__int_as_float(__byte_perm(biased, 0x4B000000u, 0x7540u + k)),
                                 __int_as_float(__byte_perm(biased, 0x4B000000u, 0x7541u + k)));
    return fadd2(f, make_float2(-8388736.0f, -8388736.0f));
}

template <typename T, int G>
struct RowLoad<T, G, true, 64> {
    static __device__ __forceinline__ void load(const int8_t *codes, const uint16_t *scales, int row, int c,
                                                float2 (&x)[4], float &d)
    {
        const uint2 w = *reinterpret_cast<const uint2 *>(codes + row * kQ8CodeRow + c * 8);
        const uint32_t lo = w.x ^ 0x80808080u, hi = w.y ^ 0x80808080u;
        x[0] = q8_code_pair(lo, 0);
        x[1] = q8_code_pair(lo, 2);
        x[2] = q8_code_pair(hi, 0);
        x[3] = q8_code_pair(hi, 2);
        d = __half2float(__ushort_as_half(scales[row * kQ8Scales + (c >> 2)]));
    }
    static __device__ __forceinline__ void k(const DecodeSlot<G, true, 64> &sl, int row, int c, float2 (&x)[4], float &d)
    {
        load(sl.k, sl.ks, row, c, x, d);
    }
    static __device__ __forceinline__ void v(const DecodeSlot<G, true, 64> &sl, int row, int c, float2 (&x)[4], float &d)
    {
        load(sl.v, sl.vs, row, c, x, d);
    }
};

// VU: row groups of the values pass unrolled per trip (0: all of them).
template <typename T, int G, bool Q8, int D, int VU = 0>
__device__ __forceinline__ void process_step(const DecodeSlot<G, Q8, D> &sl, uint32_t vmask,
                                             const float2 (&q2)[QRegs<G>::N],
                                             float2 (&acc)[G][4], float &m_run, float &l_run,
                                             float *pbuf, int lane)
{
    using GD = Geo<D>;
    constexpr int NS = HeadSlots<G>::N;
    constexpr int SHIFT = GD::LOGC - HeadSlots<G>::LOG;  // lane c holds head c >> SHIFT
    constexpr int STEPS = GD::TOK / GD::ROWS;            // row groups of a step
    const int c = lane & (GD::COLS - 1);
    const int r = lane >> GD::LOGC;

    // ---- scores of all token rows of the step, kQkRows row groups at a
    // time (their FMA chains and shuffle levels interleave)
    static_assert(STEPS % kQkRows == 0, "row groups per round");
    float z[STEPS];
#pragma unroll
    for (int st = 0; st < STEPS; st += kQkRows) {
        float zz[kQkRows];
        if constexpr (NS >= 2) {
            // Head pairs: a[u][m] holds this lane's partial dot products of
            // head slots 2m and 2m+1 (its 8 dims), one packed FMA per key
            // element for two heads, so no horizontal add is needed.
            constexpr int NP = NS / 2;
            float2 a[kQkRows][NP];
#pragma unroll
            for (int u = 0; u < kQkRows; ++u) {
                float2 kx[4];  // dims 2e, 2e+1 of the lane's 8
                float kd;
                RowLoad<T, G, Q8, D>::k(sl, (st + u) * GD::ROWS + r, c, kx, kd);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 k0 = make_float2(kx[e].x, kx[e].x), k1 = make_float2(kx[e].y, kx[e].y);
#pragma unroll
                    for (int m = 0; m < NP; ++m) {
                        a[u][m] = e == 0 ? fmul2(q2[m * 8], k0) : ffma2(q2[m * 8 + 2 * e], k0, a[u][m]);
                        a[u][m] = ffma2(q2[m * 8 + 2 * e + 1], k1, a[u][m]);
                    }
                }
                if constexpr (Q8) {  // the row's scale for this lane's dims, before lanes combine
#pragma unroll
                    for (int m = 0; m < NP; ++m)
                        a[u][m] = fmul2(a[u][m], make_float2(kd, kd));
                }
            }
            // Reduce-scatter over the row's COLS lanes: whole pairs are halved
            // (lane masks COLS/2, COLS/4, ...) while more than one is left,
            // the last pair is split at the next mask, and lanes that still
            // share a head (fewer slots than lanes) sum what is left.
            int msk = GD::COLS / 2;
#pragma unroll
            for (int n = NP; n > 1; n >>= 1, msk >>= 1)
#pragma unroll
                for (int i = 0; i < n / 2; ++i)
#pragma unroll
                    for (int u = 0; u < kQkRows; ++u) {
                        const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, a[u][i + n / 2].x, msk),
                                                     __shfl_xor_sync(0xffffffffu, a[u][i + n / 2].y, msk));
                        a[u][i] = fadd2(a[u][i], o);
                    }
#pragma unroll
            for (int u = 0; u < kQkRows; ++u)
                zz[u] = a[u][0].x + __shfl_xor_sync(0xffffffffu, a[u][0].y, msk);
#pragma unroll
            for (int m = msk >> 1; m >= 1; m >>= 1)
#pragma unroll
                for (int u = 0; u < kQkRows; ++u)
                    zz[u] += __shfl_xor_sync(0xffffffffu, zz[u], m);
        } else {
            // One head: dim pairs, then a sum over the row's COLS lanes.
#pragma unroll
            for (int u = 0; u < kQkRows; ++u) {
                float2 kx[4];
                float kd;
                RowLoad<T, G, Q8, D>::k(sl, (st + u) * GD::ROWS + r, c, kx, kd);
                float2 a = fmul2(q2[0], kx[0]);
                a = ffma2(q2[1], kx[1], a);
                a = ffma2(q2[2], kx[2], a);
                a = ffma2(q2[3], kx[3], a);
                zz[u] = a.x + a.y;
                if constexpr (Q8)
                    zz[u] *= kd;
            }
#pragma unroll
            for (int m = GD::COLS / 2; m >= 1; m >>= 1)
#pragma unroll
                for (int u = 0; u < kQkRows; ++u)
                    zz[u] += __shfl_xor_sync(0xffffffffu, zz[u], m);
        }
#pragma unroll
        for (int u = 0; u < kQkRows; ++u) {
            const int t = (st + u) * GD::ROWS + r;
            z[st + u] = !((vmask >> t) & 1u) ? -INFINITY : zz[u];
        }
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
            const float aj = __shfl_sync(0xffffffffu, alpha, (lane & ~(GD::COLS - 1)) | (j << SHIFT));
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
        if (!(z[st] > -INFINITY))
            p[st] = 0.f;
        l_run += p[st];
    }

    // ---- share p of (token, head) with the row (lanes that share a head
    // write the same value; a padding head lands in an unused slot)
#pragma unroll
    for (int st = 0; st < STEPS; ++st)
        pbuf[(st * GD::ROWS + r) * HeadSlots<G>::PSTRIDE + (c >> SHIFT)] = p[st];
    __syncwarp();

    // ---- values
#pragma unroll (VU == 0 ? STEPS : VU)
    for (int st = 0; st < STEPS; ++st) {
        const int t = st * GD::ROWS + r;
        float2 vx[4];
        float vd;
        RowLoad<T, G, Q8, D>::v(sl, t, c, vx, vd);
        if constexpr (Q8) {
            // a row that holds no key has p = 0 and zero codes, but its pool
            // scale may be anything: use 0
            const float d = ((vmask >> t) & 1u) ? vd : 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                vx[k] = fmul2(vx[k], make_float2(d, d));
        }
        const float2 v0 = vx[0], v1 = vx[1], v2 = vx[2], v3 = vx[3];
        const float4 *prow = reinterpret_cast<const float4 *>(pbuf + t * HeadSlots<G>::PSTRIDE);
        float4 pp[(G + 3) / 4];
#pragma unroll
        for (int i = 0; i < (G + 3) / 4; ++i)
            pp[i] = prow[i];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const float4 &q4 = pp[j >> 2];
            const float pv = (j & 3) == 0 ? q4.x : (j & 3) == 1 ? q4.y : (j & 3) == 2 ? q4.z : q4.w;
            const float2 pj = make_float2(pv, pv);
            acc[j][0] = ffma2(pj, v0, acc[j][0]);
            acc[j][1] = ffma2(pj, v1, acc[j][1]);
            acc[j][2] = ffma2(pj, v2, acc[j][2]);
            acc[j][3] = ffma2(pj, v3, acc[j][3]);
        }
    }
    __syncwarp();  // the next step rewrites pbuf
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge of the partial records of one (sequence, kv head) pair:
// pieces c0..c1 (the first in its worker's second record slot when
// c0_second).  One warp merges one part, query heads h0..h0+HPP-1 of the
// group, and writes out[out_row + j*D + d] for those heads.  Parts of 1 or 2
// heads (many pieces): a head's row of one piece is D/4 float4s, one per
// lane, so a warp reads PPR = 128/D rows at once (lane l: row l / (D/4),
// dims 4(l mod D/4)..+3).  A chunk of CH pieces is loaded at once -- lane k
// also loads piece k's maxima and sums -- so that a chunk costs one round
// trip to L2; chunks are merged online (a chunk with a larger maximum
// rescales what came before).  Parts of 4 or 8 heads (few pieces) take
// merge_part_lanes, where no value crosses lanes.
// ---------------------------------------------------------------------------
constexpr int kMergeLoads = 24;  // float4 loads in flight per lane (16 and 32 measured slower)
template <int D>
struct MergeGeo {
    static constexpr int LPP = D / 4;                 // lanes of one (head, piece) row
    static constexpr int PPR = 32 / LPP;              // rows a warp reads at once
    static constexpr int BUDGET = kMergeLoads * PPR;  // (head, piece) rows in flight
};

// Query heads per part for a merge of n pieces: the most heads whose rows of
// all n pieces fit in one chunk (1 when even one head's do not).
template <int D>
__device__ __forceinline__ int merge_heads_per_part(int n)
{
    constexpr int B = MergeGeo<D>::BUDGET;
    return n <= B / 8 ? 8 : n <= B / 4 ? 4 : n <= B / 2 ? 2 : 1;
}

template <int D>
__device__ __forceinline__ const float *piece_record(const DecodeParams &P, int c0, int k, bool c0_second)
{
    const int wh = (k == 0 && c0_second) ? 1 : 0;
    return P.partials + ((long long)(c0 + k) * 2 + wh) * Geo<D>::SLOT_FLOATS;
}

// Records of a two-level merge: record 0 is worker c0's; record k >= 1 is in
// the first slot of the first worker of the k-th CTA after c0's, where the
// CTA's pieces of the pair were combined (c1 - c0 + 1 counts the records).
template <int D>
__device__ __forceinline__ const float *cta_record(const DecodeParams &P, int c0, int k, bool c0_second)
{
    constexpr int NG = kConsumerWarps;
    const int wk = k == 0 ? c0 : (c0 / NG + k) * NG;
    const int wh = (k == 0 && c0_second) ? 1 : 0;
    return P.partials + ((long long)wk * 2 + wh) * Geo<D>::SLOT_FLOATS;
}

template <int D, bool PER_CTA>
__device__ __forceinline__ const float *record_at(const DecodeParams &P, int c0, int k, bool c0_second)
{
    if constexpr (PER_CTA)
        return cta_record<D>(P, c0, k, c0_second);
    else
        return piece_record<D>(P, c0, k, c0_second);
}

template <typename T, int D, int HPP, bool PER_CTA = false>
__device__ void merge_part(const DecodeParams &P, int c0, int c1, bool c0_second, long long out_row, int h0, int G,
                           int lane)
{
    using MG = MergeGeo<D>;
    constexpr int CH = MG::BUDGET / HPP < 64 ? MG::BUDGET / HPP : 64;  // pieces per chunk
    constexpr int NJ = CH / MG::PPR;                                     // loads per head and lane
    constexpr int U = (CH + 31) / 32;                                    // pieces per lane (maxima, sums)
    const int sub = lane / MG::LPP, dd = 4 * (lane % MG::LPP);
    const int npieces = c1 - c0 + 1;
    float mr[HPP], lr[HPP];
    float4 o[HPP];
#pragma unroll
    for (int i = 0; i < HPP; ++i) {
        mr[i] = -INFINITY;
        lr[i] = 0.f;
        o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int k0 = 0; k0 < npieces; k0 += CH) {
        const int nk = min(CH, npieces - k0);
        // lane l holds the maxima and sums of pieces l, l + 32, ...
        float mk[U][HPP], lk[U][HPP];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int i = 0; i < HPP; ++i) {
                mk[u][i] = -INFINITY;
                lk[u][i] = 0.f;
                if (lane + 32 * u < nk && h0 + i < G) {
                    const float *r = record_at<D, PER_CTA>(P, c0, k0 + lane + 32 * u, c0_second);
                    mk[u][i] = __ldcg(r + h0 + i);
                    lk[u][i] = __ldcg(r + kMaxGroup + h0 + i);
                }
            }
        float4 a[HPP][NJ];
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int k = j * MG::PPR + sub;
            const float *r = record_at<D, PER_CTA>(P, c0, k0 + (k < nk ? k : 0), c0_second) + 2 * kMaxGroup + dd;
#pragma unroll
            for (int i = 0; i < HPP; ++i)
                a[i][j] = (k < nk && h0 + i < G) ? __ldcg(reinterpret_cast<const float4 *>(r + (h0 + i) * D))
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < HPP; ++i) {
            float n = mk[0][i];
#pragma unroll
            for (int u = 1; u < U; ++u)
                n = fmaxf(n, mk[u][i]);
#pragma unroll
            for (int o2 = 16; o2 >= 1; o2 >>= 1)
                n = fmaxf(n, __shfl_xor_sync(0xffffffffu, n, o2));
            n = fmaxf(n, mr[i]);
            // weights of what came before and of this lane's pieces (0 for an empty one)
            const float sc = mr[i] > -INFINITY ? fast_exp2(mr[i] - n) : 0.f;
            float f[U], w = 0.f;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                f[u] = mk[u][i] > -INFINITY ? fast_exp2(mk[u][i] - n) : 0.f;
                w += f[u] * lk[u][i];
            }
#pragma unroll
            for (int o2 = 16; o2 >= 1; o2 >>= 1)
                w += __shfl_xor_sync(0xffffffffu, w, o2);
            lr[i] = lr[i] * sc + w;
            mr[i] = n;
            o[i].x *= sc;
            o[i].y *= sc;
            o[i].z *= sc;
            o[i].w *= sc;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                // piece j * PPR + sub: lane (j * PPR) % 32 + sub, copy (j * PPR) / 32
                const float fk = __shfl_sync(0xffffffffu, f[(j * MG::PPR) / 32], (j * MG::PPR) % 32 + sub);
                o[i].x = fmaf(fk, a[i][j].x, o[i].x);
                o[i].y = fmaf(fk, a[i][j].y, o[i].y);
                o[i].z = fmaf(fk, a[i][j].z, o[i].z);
                o[i].w = fmaf(fk, a[i][j].w, o[i].w);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < HPP; ++i) {
        // the PPR rows of a lane column hold different pieces: add them
#pragma unroll
        for (int m = MG::LPP; m < 32; m <<= 1) {
            o[i].x += __shfl_xor_sync(0xffffffffu, o[i].x, m);
            o[i].y += __shfl_xor_sync(0xffffffffu, o[i].y, m);
            o[i].z += __shfl_xor_sync(0xffffffffu, o[i].z, m);
            o[i].w += __shfl_xor_sync(0xffffffffu, o[i].w, m);
        }
        if (lane < MG::LPP && h0 + i < G) {
            const float inv = 1.f / lr[i];
            uint2 w;
            w.x = pack2<T>(o[i].x * inv, o[i].y * inv);
            w.y = pack2<T>(o[i].z * inv, o[i].w * inv);
            *reinterpret_cast<uint2 *>(P.out + out_row + (h0 + i) * D + dd) = w;
        }
    }
}

// A part of HPP >= 4 heads: lane l merges head h0 + l / (32 / HPP), DPL
// consecutive dims, over all pieces itself -- it loads each piece's maximum
// and sum of its head and its dims' rows (a chunk of CH pieces per round
// trip), so that no value crosses lanes.  REC: the result is a partial
// record (maxima, sums, unnormalised rows) at rec, which may be one of the
// records read, rather than the output.
template <typename T, int D, int HPP, bool PER_CTA = false, bool REC = false>
__device__ void merge_part_lanes(const DecodeParams &P, int c0, int c1, bool c0_second, long long out_row, int h0,
                                 int G, int lane, float *rec = nullptr)
{
    constexpr int LPH = 32 / HPP;             // lanes per head
    constexpr int DPL = D / LPH;              // dims per lane
    constexpr int NV = DPL / 4;               // float4 of a piece's row per lane
    constexpr int CH = kMergeLoads * 4 / DPL;  // pieces per chunk
    static_assert(NV >= 1 && CH >= 1, "merge geometry");
    const int head = h0 + lane / LPH;
    const bool live = head < G;
    const int d0 = (lane % LPH) * DPL;
    const int npieces = c1 - c0 + 1;
    float m = -INFINITY, w = 0.f;
    float4 o[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v)
        o[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < npieces; k0 += CH) {
        const int nk = min(CH, npieces - k0);
        float mk[CH], lk[CH];
        float4 a[CH][NV];
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            mk[k] = -INFINITY;
            lk[k] = 0.f;
#pragma unroll
            for (int v = 0; v < NV; ++v)
                a[k][v] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < nk && live) {
                const float *r = record_at<D, PER_CTA>(P, c0, k0 + k, c0_second);
                mk[k] = __ldcg(r + head);
                lk[k] = __ldcg(r + kMaxGroup + head);
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    a[k][v] = __ldcg(reinterpret_cast<const float4 *>(r + 2 * kMaxGroup + head * D + d0 + 4 * v));
            }
        }
        float mn = m;
#pragma unroll
        for (int k = 0; k < CH; ++k)
            mn = fmaxf(mn, mk[k]);
        const float sc = m > -INFINITY ? fast_exp2(m - mn) : 0.f;
        w *= sc;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            o[v].x *= sc;
            o[v].y *= sc;
            o[v].z *= sc;
            o[v].w *= sc;
        }
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const float f = mk[k] > -INFINITY ? fast_exp2(mk[k] - mn) : 0.f;
            w = fmaf(f, lk[k], w);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                o[v].x = fmaf(f, a[k][v].x, o[v].x);
                o[v].y = fmaf(f, a[k][v].y, o[v].y);
                o[v].z = fmaf(f, a[k][v].z, o[v].z);
                o[v].w = fmaf(f, a[k][v].w, o[v].w);
            }
        }
        m = mn;
    }
    if constexpr (REC) {
        __syncwarp();  // every lane has read its rows before any is overwritten
        if (live) {
            if (lane % LPH == 0) {
                __stcg(rec + head, m);
                __stcg(rec + kMaxGroup + head, w);
            }
#pragma unroll
            for (int v = 0; v < NV; ++v)
                __stcg(reinterpret_cast<float4 *>(rec + 2 * kMaxGroup + head * D + d0 + 4 * v), o[v]);
        }
        return;
    }
    if (live) {
        const float inv = 1.f / w;
        uint16_t *dst = P.out + out_row + (long long)head * D + d0;
#pragma unroll
        for (int v = 0; v < NV; v += 2) {
            uint4 u;
            u.x = pack2<T>(o[v].x * inv, o[v].y * inv);
            u.y = pack2<T>(o[v].z * inv, o[v].w * inv);
            if (v + 1 < NV) {
                u.z = pack2<T>(o[v + 1].x * inv, o[v + 1].y * inv);
                u.w = pack2<T>(o[v + 1].z * inv, o[v + 1].w * inv);
                *reinterpret_cast<uint4 *>(dst + 4 * v) = u;
            } else {
                *reinterpret_cast<uint2 *>(dst + 4 * v) = make_uint2(u.x, u.y);
            }
        }
    }
}

// The partial records a warp has stored but not yet counted (at most two: the
// first and the last piece of its range).  Their arrivals are counted at the
// end of the ring, behind one fence: a pair's merge cannot start before the
// last piece of its other workers' ranges anyway.
struct PendingMerge {
    int n;
    int pair0, pspan0, pstart0;
    int pair1, pspan1, pstart1;
};

// Queue the merge of `pair` when this warp's arrival was the last (prev =
// the count before it).
template <typename T, int D>
__device__ __forceinline__ void queue_if_last(const DecodeParams &P, int pair, int pspan, int pstart, int prev,
                                              int q, int r, int G, MergeQueue &mq, int lane)
{
    const int c0 = worker_of(pstart, q, r);
    const int c1 = worker_of(pstart + pspan - 1, q, r);
    if (prev != c1 - c0)
        return;
    // every piece has arrived: lane 0's acquiring count ordered the other
    // pieces' records before the hand-off (the release of the queue entry)
    const int s = pair / P.num_kv_heads, h = pair % P.num_kv_heads;
    const long long out_row = ((long long)s * P.num_q_heads + (long long)h * G) * D;
    const bool c0_second = range_begin(c0, q, r) != pstart;
    int idx = kMergeQueue;
    if (lane == 0)
        idx = atomicAdd(&mq.tail, 1);
    idx = __shfl_sync(0xffffffffu, idx, 0);
    // A ring holds at most two partial pieces, so a CTA queues at most
    // 2 x 8 merges and the queue cannot fill; the check guards the bound.
    if (idx >= kMergeQueue) {
        if (lane == 0)
            raise_status(P.status, NS_DEV_MERGE_QUEUE);
    } else if (lane == 0) {
        MergeJob &j = mq.job[idx];
        j.c0 = c0;
        j.c1 = c1;
        j.out_row = out_row;
        j.pair = pair;
        j.c0_second = c0_second ? 1 : 0;
        j.hpp = merge_heads_per_part<D>(c1 - c0 + 1);
        j.nparts = (G + j.hpp - 1) / j.hpp;
        st_release_cta(&mq.ready[idx], 1);
    }
}

// Count this warp's stored records and queue the merges it completes.
template <typename T, int D>
__device__ __forceinline__ void count_arrivals(const DecodeParams &P, PendingMerge &pm, int q, int r, int G,
                                               MergeQueue &mq, int lane)
{
    if (pm.n == 0)
        return;
    __threadfence();  // the records before their counts
    // Acquire-release counts: the last arrival's acquire orders the other
    // pieces' records (each published by its warp's fence before its count)
    // before the merge's hand-off (measured against a relaxed add and a
    // second fence: 4 sequences 13.75 -> 13.29 us, the others alike).
    int prev0 = 0, prev1 = 0;
    if (lane == 0) {
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev0) : "l"(P.counters + pm.pair0) : "memory");
        if (pm.n > 1)
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev1) : "l"(P.counters + pm.pair1) : "memory");
    }
    prev0 = __shfl_sync(0xffffffffu, prev0, 0);
    prev1 = __shfl_sync(0xffffffffu, prev1, 0);
    queue_if_last<T, D>(P, pm.pair0, pm.pspan0, pm.pstart0, prev0, q, r, G, mq, lane);
    if (pm.n > 1)
        queue_if_last<T, D>(P, pm.pair1, pm.pspan1, pm.pstart1, prev1, q, r, G, mq, lane);
    pm.n = 0;
}

// ---------------------------------------------------------------------------
// Two-level merges (kernels instantiated with TWO, chosen by the host when
// few pairs are cut over many workers numbered CTA-major, so that each pair
// has many pieces in each CTA).  A pair cut into at least kTwoLevelPieces
// pieces is merged in two levels: its pieces inside one CTA are counted in
// shared memory and combined by the last of them into one record (into the
// output when the CTA holds every piece); the CTA records are then counted
// in global memory and merged as one-level pairs are.  Other pairs merge in
// one level.
// ---------------------------------------------------------------------------
constexpr int kTwoLevelPieces = 16;

// Queue the merge of `pair` over records c0..c1 (flags: kJob* bits); the
// caller's fence orders every record before the hand-off.
template <typename T, int D>
__device__ __forceinline__ void queue_job(const DecodeParams &P, int pair, int c0, int c1, int flags, int G,
                                          MergeQueue &mq, int lane)
{
    const int s = pair / P.num_kv_heads, h = pair % P.num_kv_heads;
    const long long out_row = ((long long)s * P.num_q_heads + (long long)h * G) * D;
    int idx = kMergeQueue;
    if (lane == 0)
        idx = atomicAdd(&mq.tail, 1);
    idx = __shfl_sync(0xffffffffu, idx, 0);
    if (idx >= kMergeQueue) {
        if (lane == 0)
            raise_status(P.status, NS_DEV_MERGE_QUEUE);
    } else if (lane == 0) {
        MergeJob &j = mq.job[idx];
        j.c0 = c0;
        j.c1 = c1;
        j.out_row = out_row;
        j.pair = pair;
        j.c0_second = flags;
        j.hpp = merge_heads_per_part<D>(c1 - c0 + 1);
        j.nparts = (G + j.hpp - 1) / j.hpp;
        st_release_cta(&mq.ready[idx], 1);
    }
}

// One pending record: the pair, its workers c0..c1, lo..hi of them in this
// CTA, and whether it merges in two levels.
struct Arrival {
    int pair, c0, c1, lo, hi;
    bool sec, two;
};

__device__ __forceinline__ Arrival arrival_of(int pair, int pspan, int pstart, const Split &sp)
{
    constexpr int NG = kConsumerWarps;
    Arrival a;
    a.pair = pair;
    a.c0 = worker_of(pstart, sp.q, sp.r);
    a.c1 = worker_of(pstart + pspan - 1, sp.q, sp.r);
    a.sec = range_begin(a.c0, sp.q, sp.r) != pstart;
    const int wlo = (int)blockIdx.x * NG;
    a.lo = max(a.c0, wlo);
    a.hi = min(a.c1, wlo + NG - 1);
    a.two = !sp.wmajor && a.c1 - a.c0 + 1 >= kTwoLevelPieces && a.hi > a.lo;
    return a;
}

// After the count (prev: the count before this arrival): queue the merge
// when this was the last arrival, or, in two levels, combine this CTA's
// pieces when this was the last of them.
template <typename T, int D>
__device__ __forceinline__ void arrive_two(const DecodeParams &P, const Arrival &a, int prev, int G,
                                           MergeQueue &mq, int lane)
{
    constexpr int NG = kConsumerWarps;
    int n = a.c1 - a.c0 + 1, flags = a.sec ? 1 : 0;
    if (a.two) {
        if (prev != a.hi - a.lo)
            return;  // another warp of this CTA combines
        __threadfence_block();  // the other warps' records, counted before this one
        const bool lsec = a.lo == a.c0 && a.sec;
        const int nc = a.c1 / NG - a.c0 / NG + 1;
        if (nc == 1) {
            const int s = a.pair / P.num_kv_heads, h = a.pair % P.num_kv_heads;
            merge_part_lanes<T, D, 8>(P, a.lo, a.hi, lsec, ((long long)s * P.num_q_heads + (long long)h * G) * D, 0,
                                      G, lane);
            return;
        }
        // the CTA record replaces the record of the pair's first worker here
        float *rec = const_cast<float *>(piece_record<D>(P, a.lo, 0, lsec));
        merge_part_lanes<T, D, 8, false, true>(P, a.lo, a.hi, lsec, 0, 0, G, lane, rec);
        __threadfence();  // the CTA record before its count
        prev = 0;
        if (lane == 0)
            prev = atomicAdd(P.counters + a.pair, 1);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        n = nc;
        flags |= kJobPerCta;
    }
    if (prev != n - 1)
        return;
    __threadfence();  // every record before the hand-off to whichever warp runs the merge
    queue_job<T, D>(P, a.pair, a.c0, a.c0 + n - 1, flags, G, mq, lane);
}

template <typename T, int D>
__device__ __forceinline__ void count_arrivals_two(const DecodeParams &P, PendingMerge &pm, const Split &sp, int G,
                                                   MergeQueue &mq, int *cta_count, int lane)
{
    if (pm.n == 0)
        return;
    constexpr int NG = kConsumerWarps;
    const Arrival a0 = arrival_of(pm.pair0, pm.pspan0, pm.pstart0, sp);
    const Arrival a1 = pm.n > 1 ? arrival_of(pm.pair1, pm.pspan1, pm.pstart1, sp) : a0;
    // the records before their counts (a count in this CTA needs CTA scope only)
    if (!a0.two || (pm.n > 1 && !a1.two))
        __threadfence();
    else
        __threadfence_block();
    const int wlo = (int)blockIdx.x * NG;
    int prev0 = 0, prev1 = 0;
    if (lane == 0) {
        prev0 = a0.two ? atomicAdd(cta_count + (a0.lo - wlo), 1) : atomicAdd(P.counters + a0.pair, 1);
        if (pm.n > 1)
            prev1 = a1.two ? atomicAdd(cta_count + (a1.lo - wlo), 1) : atomicAdd(P.counters + a1.pair, 1);
    }
    prev0 = __shfl_sync(0xffffffffu, prev0, 0);
    prev1 = __shfl_sync(0xffffffffu, prev1, 0);
    arrive_two<T, D>(P, a0, prev0, G, mq, lane);
    if (pm.n > 1)
        arrive_two<T, D>(P, a1, prev1, G, mq, lane);
    pm.n = 0;
}

// Take the next part of a queued merge: lane 0's cursor value (broadcast),
// -1 when every queued part is taken, -2 when a reserved entry was not
// filled in time.
__device__ __forceinline__ bool merge_ready_wait(MergeQueue &mq, int job)
{
    const unsigned long long t0 = global_timer_ns();
    while (ld_acquire_cta(&mq.ready[job]) == 0)
        if (global_timer_ns() - t0 > kWaitLimitNs)
            return false;
    return true;
}

__device__ __forceinline__ int merge_pop(MergeQueue &mq, int lane)
{
    int got = -1;
    if (lane == 0) {
        while (true) {
            const int c = ld_acquire_cta(&mq.head);
            const int job = c / kMergeParts, part = c % kMergeParts;
            if (job >= min(ld_acquire_cta(&mq.tail), kMergeQueue))
                break;
            if (!merge_ready_wait(mq, job)) {  // its parts are known once it is filled
                got = -2;
                break;
            }
            const int next = part + 1 < mq.job[job].nparts ? c + 1 : (job + 1) * kMergeParts;
            if (atomicCAS(&mq.head, c, next) == c) {
                got = c;
                break;
            }
        }
    }
    return __shfl_sync(0xffffffffu, got, 0);
}

// Run part `c % kMergeParts` of queued merge `c / kMergeParts` (filled: the
// pop waited for it).
template <typename T, int D, bool TWO = false>
__device__ __forceinline__ void merge_run(const DecodeParams &P, MergeQueue &mq, int c, int G, int lane)
{
    const int job = c / kMergeParts, part = c % kMergeParts;
    const MergeJob j = mq.job[job];
    const int c0 = (int)j.c0, c1 = (int)j.c1, h0 = part * j.hpp;
    if constexpr (TWO) {
        const bool second = (j.c0_second & 1) != 0;
        if (j.c0_second & kJobPerCta) {
            switch (j.hpp) {
            case 8: merge_part_lanes<T, D, 8, true>(P, c0, c1, second, j.out_row, h0, G, lane); break;
            case 4: merge_part_lanes<T, D, 4, true>(P, c0, c1, second, j.out_row, h0, G, lane); break;
            case 2: merge_part<T, D, 2, true>(P, c0, c1, second, j.out_row, h0, G, lane); break;
            default: merge_part<T, D, 1, true>(P, c0, c1, second, j.out_row, h0, G, lane); break;
            }
        } else {
            switch (j.hpp) {
            case 8: merge_part_lanes<T, D, 8>(P, c0, c1, second, j.out_row, h0, G, lane); break;
            case 4: merge_part_lanes<T, D, 4>(P, c0, c1, second, j.out_row, h0, G, lane); break;
            case 2: merge_part<T, D, 2>(P, c0, c1, second, j.out_row, h0, G, lane); break;
            default: merge_part<T, D, 1>(P, c0, c1, second, j.out_row, h0, G, lane); break;
            }
        }
        if (lane == 0 && part == 0)
            P.counters[j.pair] = 0;
        return;
    }
    const bool second = j.c0_second != 0;
    switch (j.hpp) {
    case 8: merge_part_lanes<T, D, 8>(P, c0, c1, second, j.out_row, h0, G, lane); break;
    case 4: merge_part_lanes<T, D, 4>(P, c0, c1, second, j.out_row, h0, G, lane); break;
    case 2: merge_part<T, D, 2>(P, c0, c1, second, j.out_row, h0, G, lane); break;
    default: merge_part<T, D, 1>(P, c0, c1, second, j.out_row, h0, G, lane); break;
    }
    if (lane == 0 && part == 0)
        P.counters[j.pair] = 0;
}

// ---------------------------------------------------------------------------
// End of a piece for one warp: combine the row groups (shuffles), then
// write the output (whole pair) or the partial record, whose arrival is
// counted at the end of the ring (count_arrivals), so that the warp waits
// neither for a fence nor for an atomic here.
// ---------------------------------------------------------------------------
template <typename T, int BS, int G, int D>
__device__ void piece_end(const DecodeParams &P, const PieceRef &pc, int worker, int q, int r,
                          float2 (&acc)[G][4], float m_run, float l_run, int lane, PendingMerge &pm,
                          MergeQueue &mq)
{
    using GD = Geo<D>;
    constexpr int SHIFT = GD::LOGC - HeadSlots<G>::LOG;
    const int c = lane & (GD::COLS - 1);
    // lane (r, c) with (c & ((1 << SHIFT) - 1)) == 0 owns (row group r, head c >> SHIFT);
    // the row groups' lanes are lane ^ COLS, lane ^ 2 COLS, ...
    float M = m_run;
#pragma unroll
    for (int m = GD::COLS; m < 32; m <<= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
    const float f = (m_run > -INFINITY) ? fast_exp2(m_run - M) : 0.f;
    float Ls = f * l_run;
#pragma unroll
    for (int m = GD::COLS; m < 32; m <<= 1)
        Ls += __shfl_xor_sync(0xffffffffu, Ls, m);
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const float fj = __shfl_sync(0xffffffffu, f, (lane & ~(GD::COLS - 1)) | (j << SHIFT));
        const float2 f2 = make_float2(fj, fj);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float2 a = fmul2(acc[j][k], f2);
#pragma unroll
            for (int m = GD::COLS; m < 32; m <<= 1) {
                a.x += __shfl_xor_sync(0xffffffffu, a.x, m);
                a.y += __shfl_xor_sync(0xffffffffu, a.y, m);
            }
            acc[j][k] = a;
        }
    }
    // every lane now holds, for dims 8c..8c+7: the merged acc of this warp's
    // heads; head j's max and sum are in lane (j << SHIFT)
    const int s = pc.ps, h = pc.ph;
    const long long out_row = ((long long)s * P.num_q_heads + (long long)h * G) * D;
    constexpr unsigned kRowLanes = GD::COLS == 32 ? 0xffffffffu : ((1u << GD::COLS) - 1u);
    if (pc.flags & kFlagWhole) {
        if (lane < GD::COLS) {
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const float inv = 1.f / __shfl_sync(kRowLanes, Ls, j << SHIFT);
                uint4 w;
                w.x = pack2<T>(acc[j][0].x * inv, acc[j][0].y * inv);
                w.y = pack2<T>(acc[j][1].x * inv, acc[j][1].y * inv);
                w.z = pack2<T>(acc[j][2].x * inv, acc[j][2].y * inv);
                w.w = pack2<T>(acc[j][3].x * inv, acc[j][3].y * inv);
                *reinterpret_cast<uint4 *>(P.out + out_row + j * D + c * 8) = w;
            }
        }
        return;
    }

    // ---- partial piece: store the record, count arrivals, merge if last.
    const int which = (pc.flags & kFlagWhich1) ? 1 : 0;
    float *rec = P.partials + ((long long)worker * 2 + which) * GD::SLOT_FLOATS;
    if (lane < GD::COLS) {
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float *a = rec + 2 * kMaxGroup + j * D + c * 8;
            __stcg(reinterpret_cast<float4 *>(a), make_float4(acc[j][0].x, acc[j][0].y, acc[j][1].x, acc[j][1].y));
            __stcg(reinterpret_cast<float4 *>(a + 4), make_float4(acc[j][2].x, acc[j][2].y, acc[j][3].x, acc[j][3].y));
        }
        if ((c & ((1 << SHIFT) - 1)) == 0 && (c >> SHIFT) < G) {
            __stcg(rec + (c >> SHIFT), M);
            __stcg(rec + kMaxGroup + (c >> SHIFT), Ls);
        }
    }
    const int pair = s * P.num_kv_heads + h;
    if (pm.n == 0) {
        pm.pair0 = pair;
        pm.pspan0 = pc.pspan;
        pm.pstart0 = pc.pstart;
    } else {
        pm.pair1 = pair;
        pm.pspan1 = pc.pspan;
        pm.pstart1 = pc.pstart;
    }
    ++pm.n;
}

// Table row, first-step table entries and slot_mapping entry of a piece.
template <int BS, int KB>
__device__ __forceinline__ void piece_prefetch(const DecodeParams &P, const PieceWalk &pc, long long &trow,
                                               int (&phys)[KB], long long &slot)
{
    trow = P.table_row != nullptr ? __ldg(P.table_row + pc.ps) : pc.ps;
    slot = (P.k_new != nullptr && pc.hi == pc.pnb) ? __ldg(P.slot_mapping + pc.ps) : -1;
#pragma unroll
    for (int u = 0; u < KB; ++u)
        phys[u] = pc.lo + u < pc.hi ? __ldg(P.block_tables + trow * P.max_blocks_per_seq + pc.lo + u) : -1;
}

// ---------------------------------------------------------------------------
// Producer warps: lane i of producer warp p serves ring (worker)
// w = i * PW + p.  It walks w's pieces one piece ahead, reads the
// block-table entries of each step one step ahead, and issues the TMA copies
// of the next step into w's ring as soon as its consumers free a slot, with
// the step's description (piece, valid keys, fused slot) in the slot's
// SlotMeta.  Consumers then hold no walk or issue state: their registers go
// to the scores and accumulators.
// ---------------------------------------------------------------------------
template <typename T, int BS, int G, int S, bool Q8, int D>
__device__ void decode_producer(const DecodeParams &P, DecodeSmem<BS, G, S, Q8, D> &sm, const Split &sp,
                                int pwarp, int lane)
{
    constexpr int TOK = Geo<D>::TOK;       // tokens per step
    constexpr int KB = TOK / BS;           // blocks per step
    constexpr uint32_t kRowB16 = Geo<D>::ROW_BYTES;  // a 16-bit row
    constexpr int SERVED = DecodeShape<G>::SERVED;
    const int w = (lane < SERVED ? lane : 0) * DecodeShape<G>::PW + pwarp;
    const uint64_t pol = l2_evict_first_policy();
    bool done = lane >= SERVED;
    // `walk` runs one piece ahead of `cur`: the table entries of the next
    // piece's first step (and its slot_mapping entry) load while the current
    // piece streams.
    PieceWalk walk;
    walk_init<BS>(P, sm, sp, worker_id(w, sp.wmajor, DecodeShape<G>::NG), walk);
    long long a_trow = 0, a_slot = -1;
    int aphys[KB];
    bool ahead = !done && walk_next<BS>(P, walk);
    if (ahead)
        piece_prefetch<BS, KB>(P, walk, a_trow, aphys, a_slot);
    PieceWalk cur;
    bool has = false;
    int step = 0, nsteps = 0, issued = 0;
    long long trow = 0, slot_v = -1;
    int nphys[KB];  // raw table entries of the next step
    bool ok = true;
    unsigned long long idle_since = 0;
    bool idle = false;
    // The lanes go round in step: each round, every lane whose next slot is
    // free fills it; a round where no lane could sleeps briefly.
    while (__any_sync(0xffffffffu, !done)) {
        const int slot = issued % S;
        const bool ready = !done && mbar_test(&sm.empty[w][slot], ((uint32_t)(issued / S) & 1u) ^ 1u);
        if (__ballot_sync(0xffffffffu, ready) == 0) {
            const bool abort = *reinterpret_cast<volatile int *>(&sm.abort_flag) != 0;
            const unsigned long long now = global_timer_ns();
            if (!idle) {
                idle = true;
                idle_since = now;
            }
            if (__any_sync(0xffffffffu, abort || now - idle_since > kWaitLimitNs)) {
                ok = false;
                break;
            }
            __nanosleep(kProducerIdleNs);
            continue;
        }
        idle = false;
        if (!ready)
            continue;
        // launched as a programmatic dependent: the copies touch q, the pools
        // and the new K/V, which the previous grid may still be writing
        if (P.overlap && issued == 0)
            grid_dependency_wait();
        SlotMeta &mt = sm.meta[w][slot];
        DecodeSlot<G, Q8, D> &sl = sm.ring[w][slot];
        uint64_t *bar = &sm.full[w][slot];
        if (!has || step >= nsteps) {
            if (!ahead) {
                mt.nsteps = -1;  // no more work for this ring
                mbar_arrive(bar);
                ++issued;
                done = true;
                continue;
            }
            cur = walk;
            has = true;
            step = 0;
            nsteps = steps_of<BS, TOK>(cur);
            trow = a_trow;
            slot_v = a_slot;
#pragma unroll
            for (int u = 0; u < KB; ++u)
                nphys[u] = aphys[u];
            ahead = walk_next<BS>(P, walk);
            if (ahead)
                piece_prefetch<BS, KB>(P, walk, a_trow, aphys, a_slot);
            if (nsteps == 0) {
                // only virtual blocks of the pair: the consumers write an empty record
                put_meta(mt, cur.ps, cur.ph, cur.pL, cur.flags, cur.pspan, 0, 0, 0, cur.pstart, -1, 0u);
                mbar_arrive(bar);
                ++issued;
                has = false;
                continue;
            }
        }
        // this step's blocks: KB whole blocks from `first`
        const int first = cur.lo + step * KB;
        int phys[KB];
        unsigned loaded = 0;
#pragma unroll
        for (int u = 0; u < KB; ++u) {
            phys[u] = nphys[u];
            if (first + u < cur.hi && (phys[u] < 0 || (long long)phys[u] >= P.num_blocks)) {
                raise_status(P.status, NS_DEV_BAD_BLOCK_ID);
                phys[u] = -1;
            }
            if (first + u >= cur.hi)
                phys[u] = -1;
            loaded |= (phys[u] >= 0 ? 1u : 0u) << u;
        }
        if (step + 1 < nsteps) {
#pragma unroll
            for (int u = 0; u < KB; ++u)
                nphys[u] = first + KB + u < cur.hi
                               ? __ldg(P.block_tables + trow * P.max_blocks_per_seq + first + KB + u)
                               : -1;
        }
        const int tok0 = step_token0<BS, TOK>(cur, step);
        const int nval = min(TOK, piece_end_token<BS>(cur) - tok0);  // >= 1
        uint32_t vm = nval >= 32 ? 0xffffffffu : ((1u << nval) - 1u);
        if (KB > 1) {
            uint32_t bm = 0;
#pragma unroll
            for (int u = 0; u < KB; ++u)
                if ((loaded >> u) & 1u)
                    bm |= (BS >= 32 ? 0xffffffffu : ((1u << BS) - 1u)) << (u * BS);
            vm &= bm;
        } else if (!(loaded & 1u)) {
            vm = 0;
        }
        const bool first_step = step == 0;
        const bool new_tok = P.k_new != nullptr && cur.hi == cur.pnb && step == nsteps - 1;
        long long ns = -1;
        // fused append: block u_last of the step holds position L-1; only its
        // rows before r_new come from the pool, row r_new is the new token
        int u_last = -1, r_new = 0;
        if (new_tok) {
            // the pool slot of position L-1 must be the one slot_mapping names
            u_last = (cur.pL - 1) / BS - first;
            r_new = (cur.pL - 1) % BS;
            int phys_last = -1;
#pragma unroll
            for (int u = 0; u < KB; ++u)
                phys_last = u == u_last ? phys[u] : phys_last;
            const long long want = (long long)phys_last * BS + (cur.pL - 1) % BS;
            ns = slot_v;
            if (ns != want || phys_last < 0)
                raise_status(P.status, NS_DEV_FUSED_SLOT);
            if (ns >= P.num_blocks * BS) {
                raise_status(P.status, NS_DEV_BAD_SLOT);
                ns = -1;
            }
        }
        put_meta(mt, cur.ps, cur.ph, cur.pL, cur.flags | (new_tok ? kFlagNewTok : 0), cur.pspan, step, nsteps,
                 (cur.pL - 1) - tok0, cur.pstart, ns, vm);
        // Rows of each block: the first rows[u] come from the pool; in the new
        // token's block row r_new comes from k_new/v_new; every other row is
        // zero-filled, so that each row of the slot is finite and a masked
        // token (p = 0) adds nothing.  Zero ranges: [rows, za) and [zb, BS).
        // (q8_0: the codes likewise; the scales of a loaded block are copied
        // whole, a 16-byte multiple, and the consumer ignores those of rows
        // without a key; the new token's rows land in the slot's staging rows
        // and the consumer quantises them into row r_new.)
        const int pend_tok = piece_end_token<BS>(cur);
        constexpr uint32_t kRowB = Q8 ? (uint32_t)kQ8CodeRow : kRowB16;
        int rows[KB], za[KB], zb[KB];
        uint32_t bytes = (first_step ? (uint32_t)G * kRowB16 : 0u) + (new_tok ? 2u * kRowB16 : 0u);
#pragma unroll
        for (int u = 0; u < KB; ++u) {
            const int keys = min(max(pend_tok - (tok0 + u * BS), 0), BS);
            rows[u] = phys[u] < 0 ? 0 : (u == u_last ? r_new : keys);
            za[u] = u == u_last ? r_new : BS;      // zero rows [rows, za)
            zb[u] = u == u_last ? r_new + 1 : BS;  // and [zb, BS)
            bytes += 2u * (uint32_t)(rows[u] + (za[u] - rows[u]) + (BS - zb[u])) * kRowB;
            if (Q8)
                bytes += 2u * (uint32_t)(BS * kQ8ScaleRow);
        }
        if (bytes == 0)
            mbar_arrive(bar);
        else
            mbar_arrive_expect_tx(bar, bytes);
        const int pool_h = pool_head(P, cur.ph), pool_hkv = pool_heads(P);
#pragma unroll
        for (int u = 0; u < KB; ++u) {
            const long long row0 = ((long long)phys[u] * pool_hkv + pool_h) * BS;  // pool row of the block
            if constexpr (!Q8) {
                if (rows[u] > 0) {
                    bulk_load(sl.k + u * BS * D, P.k_pool + row0 * D, rows[u] * kRowB16, bar, pol);
                    bulk_load(sl.v + u * BS * D, P.v_pool + row0 * D, rows[u] * kRowB16, bar, pol);
                }
            } else {
                if (rows[u] > 0) {
                    bulk_load(sl.k + u * BS * D, P.k_codes + row0 * kQ8CodeRow, rows[u] * kQ8CodeRow, bar, pol);
                    bulk_load(sl.v + u * BS * D, P.v_codes + row0 * kQ8CodeRow, rows[u] * kQ8CodeRow, bar, pol);
                }
                if (phys[u] >= 0) {
                    bulk_load(sl.ks + u * BS * kQ8Scales, P.k_scales + row0 * kQ8Scales, BS * kQ8ScaleRow, bar, pol);
                    bulk_load(sl.vs + u * BS * kQ8Scales, P.v_scales + row0 * kQ8Scales, BS * kQ8ScaleRow, bar, pol);
                } else {
                    bulk_load(sl.ks + u * BS * kQ8Scales, g_zero_rows, BS * kQ8ScaleRow, bar);
                    bulk_load(sl.vs + u * BS * kQ8Scales, g_zero_rows, BS * kQ8ScaleRow, bar);
                }
            }
            if (za[u] > rows[u]) {
                const uint32_t n = (uint32_t)(za[u] - rows[u]) * kRowB;
                bulk_load(sl.k + (u * BS + rows[u]) * D, g_zero_rows, n, bar);
                bulk_load(sl.v + (u * BS + rows[u]) * D, g_zero_rows, n, bar);
            }
            if (zb[u] < BS) {
                const uint32_t n = (uint32_t)(BS - zb[u]) * kRowB;
                bulk_load(sl.k + (u * BS + zb[u]) * D, g_zero_rows, n, bar);
                bulk_load(sl.v + (u * BS + zb[u]) * D, g_zero_rows, n, bar);
            }
        }
        if (first_step) {
            const long long qoff = ((long long)cur.ps * P.num_q_heads + (long long)cur.ph * G) * D;
            bulk_load(sl.q, P.q + qoff, G * kRowB16, bar);
        }
        if (new_tok) {
            const long long noff = ((long long)cur.ps * pool_hkv + pool_h) * D;
            if constexpr (!Q8) {
                const int t_new = (cur.pL - 1) - tok0;
                bulk_load(sl.k + t_new * D, P.k_new + noff, kRowB16, bar);
                bulk_load(sl.v + t_new * D, P.v_new + noff, kRowB16, bar);
            } else {
                bulk_load(sl.knew, P.k_new + noff, kRowB16, bar);
                bulk_load(sl.vnew, P.v_new + noff, kRowB16, bar);
            }
        }
        ++issued;
        ++step;
    }
    if (lane >= SERVED)
        return;
    if (!ok) {
        *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
        raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
    }
    // Never leave with copies still landing in this consumer's slots.
    for (int k = (issued > S ? issued - S : 0); k < issued; ++k)
        if (!mbar_wait(&sm.full[w][k % S], (uint32_t)(k / S) & 1u)) {
            raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
            break;
        }
}

// ---------------------------------------------------------------------------
// Consumer warp: the G heads of ring `ring`.  Takes the
// ring's slots in order, computes each step, and at the end of each piece
// writes the output or its part of a partial record; then frees the slot
// (its empty barrier).
// ---------------------------------------------------------------------------
// q8_0 quantisation of the new token's K (lanes 0-7) and V (lanes 8-15) rows,
// staged in the slot as 16-bit rows, into row t of the slot and, for a valid
// slot, into the pool.  A block of 32 elements is four lanes' eight: its
// scale d = max|x| / 127 and every code rint(x * (1/d)) (ties to even,
// clamped to +-127) are rounded to fp32 at each step, and d is stored as
// fp16 (nearest even, saturating), the decisions the CPU oracle takes.
template <typename T, int BS, int G>
__device__ __forceinline__ void quantize_new_row(const DecodeParams &P, DecodeSlot<G, true, 64> &sl, int t,
                                                 long long new_slot, int ph, int lane)
{
    const int cc = lane & 7;
    const bool isv = (lane & 8) != 0;
    const uint4 w = lds128((isv ? sl.vnew : sl.knew) + cc * 8);
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
    const uint16_t d16 = __half_as_ushort(__float2half_rn(fminf(d, 65504.f)));
    if (lane < 16) {
        int8_t *row = (isv ? sl.v : sl.k) + t * kQ8CodeRow + cc * 8;
        *reinterpret_cast<uint2 *>(row) = make_uint2(packed[0], packed[1]);
        if ((cc & 3) == 0)
            (isv ? sl.vs : sl.ks)[t * kQ8Scales + (cc >> 2)] = d16;
        if (new_slot >= 0 && stores_new_token(P, ph)) {
            const long long prow = ((new_slot / BS) * pool_heads(P) + pool_head(P, ph)) * BS + new_slot % BS;
            int8_t *codes = const_cast<int8_t *>(isv ? P.v_codes : P.k_codes);
            uint16_t *scales = const_cast<uint16_t *>(isv ? P.v_scales : P.k_scales);
            *reinterpret_cast<uint2 *>(codes + prow * kQ8CodeRow + cc * 8) = make_uint2(packed[0], packed[1]);
            if ((cc & 3) == 0)
                scales[prow * kQ8Scales + (cc >> 2)] = d16;
        }
    }
    __syncwarp();
}

template <typename T, int BS, int G, int S, bool Q8, int D, bool TWO, int VU>
__device__ void decode_consumer(const DecodeParams &P, DecodeSmem<BS, G, S, Q8, D> &sm, const Split &sp,
                                int ring, int warp, int lane)
{
    using GD = Geo<D>;
    constexpr int NS = HeadSlots<G>::N;
    constexpr int SHIFT = GD::LOGC - HeadSlots<G>::LOG;
    const int c = lane & (GD::COLS - 1);
    const int worker = worker_id(ring, sp.wmajor, DecodeShape<G>::NG);
    const int q = sp.q, r = sp.r;
    float2 q2[QRegs<G>::N];
    float2 acc[G][4];
    float m_run = -INFINITY, l_run = 0.f;
#pragma unroll
    for (int i = 0; i < QRegs<G>::N; ++i)
        q2[i] = make_float2(0.f, 0.f);
    float *pbuf = &sm.p[warp][0][0];
    PendingMerge pm;
    pm.n = 0;
    int slot = 0;
    uint32_t phase = 0;
    bool ok = true;
    // One piece per outer iteration; its steps run in a tight inner loop, so
    // the per-piece work (query load, record or output) stays off the
    // per-step path.
    while (ok) {
        if (!mbar_wait(&sm.full[ring][slot], phase, P.wait_limit_ns)) {
            ok = false;
            break;
        }
        const int4 m0 = *reinterpret_cast<const int4 *>(&sm.meta[ring][slot].ps);     // ps, ph, pL, flags
        const int4 m1 = *reinterpret_cast<const int4 *>(&sm.meta[ring][slot].pspan);  // pspan, step, nsteps, t_new
        const int nsteps = m1.z;
        if (nsteps < 0)
            break;  // no more work
        const PieceRef pr{m0.x, m0.y, m0.w, m1.x, (int)sm.meta[ring][slot].pstart};
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                acc[j][k] = make_float2(0.f, 0.f);
        m_run = -INFINITY;
        l_run = 0.f;
        if (nsteps > 0) {
            // slot i holds head i ^ (c >> SHIFT); slots past the group are 0.
            // The raw 16-bit words of the slots are paired first (byte
            // permutes), so that each register pair is one packed product.
            const uint16_t *qs = sm.ring[ring][slot].q;
            const float2 sc = make_float2(P.scale_log2, P.scale_log2);
            uint32_t wq[NS][4];
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                const int head = i ^ (c >> SHIFT);
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (head < G)
                    w = lds128(qs + head * D + c * 8);
                wq[i][0] = w.x;
                wq[i][1] = w.y;
                wq[i][2] = w.z;
                wq[i][3] = w.w;
            }
            if constexpr (NS >= 2) {
#pragma unroll
                for (int m = 0; m < NS / 2; ++m)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // dims 2k, 2k+1 of slots 2m, 2m+1
                        q2[m * 8 + 2 * k] = fmul2(unpack2<T>(__byte_perm(wq[2 * m][k], wq[2 * m + 1][k], 0x5410)), sc);
                        q2[m * 8 + 2 * k + 1] =
                            fmul2(unpack2<T>(__byte_perm(wq[2 * m][k], wq[2 * m + 1][k], 0x7632)), sc);
                    }
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    q2[k] = fmul2(unpack2<T>(wq[0][k]), sc);
            }
        }
        for (int step = 0;;) {
            if (nsteps > 0) {
                const SlotMeta &mt = sm.meta[ring][slot];
                DecodeSlot<G, Q8, D> &sl = sm.ring[ring][slot];
                // fused append (the piece's last step): the new token's K/V
                // landed in the slot; this warp also writes them to the pool
                // slot the producer checked (q8_0: quantised first)
                if (step == nsteps - 1 && (mt.flags & kFlagNewTok)) {
                    if constexpr (!Q8) {
                        if (lane < 2 * GD::COLS && mt.new_slot >= 0 && stores_new_token(P, mt.ph)) {
                            const bool isv = lane >= GD::COLS;
                            const int cc = lane & (GD::COLS - 1);
                            const uint4 val = lds128((isv ? sl.v : sl.k) + mt.t_new * D + cc * 8);
                            const long long ns = mt.new_slot;
                            const long long dst =
                                (((ns / BS) * pool_heads(P) + pool_head(P, mt.ph)) * BS + ns % BS) * D + cc * 8;
                            *reinterpret_cast<uint4 *>((isv ? P.v_pool_w : P.k_pool_w) + dst) = val;
                        }
                    } else {
                        quantize_new_row<T, BS, G>(P, sl, mt.t_new, mt.new_slot, mt.ph, lane);
                    }
                }
                // one step path for full and partial steps: a second, unmasked
                // copy measured 4% slower (instruction-fetch stalls)
                process_step<T, G, Q8, D, VU>(sl, mt.vmask, q2, acc, m_run, l_run, pbuf, lane);
            }
            // The slot is only read (the async proxy alone writes it), so the
            // barrier's release/acquire orders these reads before the refill.
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.empty[ring][slot]);
            if (++slot == S) {
                slot = 0;
                phase ^= 1u;
            }
            if (++step >= nsteps)
                break;
            if (!mbar_wait(&sm.full[ring][slot], phase, P.wait_limit_ns)) {
                ok = false;
                break;
            }
        }
        if (ok)
            piece_end<T, BS, G, D>(P, pr, worker, q, r, acc, m_run, l_run, lane, pm, sm.mq);
    }
    if (!ok) {
        *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
        raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
    }
    if (ok) {
        if constexpr (TWO)
            count_arrivals_two<T, D>(P, pm, sp, G, sm.mq, sm.cta_count, lane);
        else
            count_arrivals<T, D>(P, pm, q, r, G, sm.mq, lane);
    }
    __syncwarp();
    if (lane == 0) {
        __threadfence_block();  // this warp's queued jobs before its count
        atomicAdd(&sm.mq.done, 1);
    }
    if (!ok)
        return;
    // Run merge parts until every ring of the CTA has ended (no job can
    // come after that) and the queue is empty: the parts of a long merge
    // spread over the warps that are idle by then.
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        int all = 0, late = 0;
        if (lane == 0) {
            all = ld_acquire_cta(&sm.mq.done) >= DecodeShape<G>::NG;
            late = global_timer_ns() - t0 > kWaitLimitNs;
        }
        all = __shfl_sync(0xffffffffu, all, 0);
        late = __shfl_sync(0xffffffffu, late, 0);
        const int c = merge_pop(sm.mq, lane);
        if (c >= 0) {
            merge_run<T, D, TWO>(P, sm.mq, c, G, lane);
            continue;
        }
        if (c == -2 || late) {
            if (lane == 0)
                raise_status(P.status, NS_DEV_WAIT_TIMEOUT);
            break;
        }
        if (all)
            break;
        __nanosleep(200);
    }
}

// ---------------------------------------------------------------------------
// Prologue (every thread, one barrier): the ring barriers, the context
// lengths of this thread's chunk of sequences, and a block-wide scan of their
// split coordinates.  Each thread then derives the split itself (read_split)
// and each producer lane its own range (walk_init).
// ---------------------------------------------------------------------------
template <class Smem, int BS>
__device__ void decode_prologue(const DecodeParams &P, Smem &sm)
{
    constexpr int NT = kDecodeThreads;
    constexpr int NG = Smem::NG;
    constexpr int S = Smem::STAGES;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    if (tid < 2 * NG * S) {
        const int i = tid % (NG * S);
        mbar_init(tid < NG * S ? &sm.full[i / S][i % S] : &sm.empty[i / S][i % S], 1);
        mbar_init_fence();
    }
    const int per = (P.num_seqs + NT - 1) / NT;
    const int s_lo = min(P.num_seqs, tid * per);
    const int s_hi = min(P.num_seqs, s_lo + per);
    const bool report = blockIdx.x == 0;
    int mine = 0, my_maxnb = 0, my_pairs = 0;
    for (int s = s_lo; s < s_hi; ++s) {
        const int L = clamped_len(P, s, BS, report);
        if (s < kLensCache)
            sm.lens[s] = L;
        const int nb = nblocks_of(L, BS);
        mine += P.num_kv_heads * pair_span(nb);
        my_maxnb = max(my_maxnb, nb);
        my_pairs += L > 0 ? P.num_kv_heads : 0;
    }
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    sm.toff[tid] = incl - mine;
    int wmax = my_maxnb, wpairs = my_pairs;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
        wpairs += __shfl_xor_sync(0xffffffffu, wpairs, o);
    }
    if (lane == 31)
        sm.wtot[warp] = incl;
    if (lane == 0) {
        sm.wmax[warp] = wmax;
        sm.wpairs[warp] = wpairs;
    }
    if (tid < kMergeQueue)
        sm.mq.ready[tid] = 0;
    if (tid < kConsumerWarps)
        sm.cta_count[tid] = 0;
    if (tid == 0) {
        sm.mq.tail = 0;
        sm.mq.head = 0;
        sm.mq.done = 0;
        sm.abort_flag = 0;
        sm.plan_split = 0;
        sm.plan_maxp = 1;
    }
    __syncthreads();
}

// The split, from the prologue scan.  An even split over gw workers (each at
// least min_blocks_per_cta / NG blocks) unless no pair is longer than twice
// the even share and every pair can have its own worker: then whole pairs
// dealt round-robin need no merge at all.
template <class Smem>
__device__ __forceinline__ Split read_split(const DecodeParams &P, const Smem &sm)
{
    constexpr int NWARPS = kDecodeThreads / 32;
    constexpr int NG = Smem::NG;
    Split sp;
    int total = 0, live = 0, maxnb = 0;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) {
        total += sm.wtot[w];
        live += sm.wpairs[w];
        maxnb = max(maxnb, sm.wmax[w]);
    }
    const int W = (int)gridDim.x * NG;
    unsigned per_worker = (unsigned)max(1, (P.min_blocks_per_cta + NG - 1) / NG);
    // Automatic policy: no more blocks a worker than keep the longest pair
    // in about kAutoPieces pieces, so that short steps use more workers
    // (cut finer: more pieces, but each merge part still loads in one round
    // trip); with at most W / kAutoPieces live pairs, every warp.
    if (P.auto_policy) {
        per_worker = min(per_worker, (unsigned)max(1, (maxnb + kPieceCost + kAutoPieces - 1) / kAutoPieces));
        if (live * kAutoPieces <= W)
            per_worker = 1;
    }
    int gw = (int)(((unsigned)total + per_worker - 1u) / per_worker);
    gw = min(gw, min(W, kMaxWorkers));
    gw = max(1, min(gw, total));  // no empty ranges: every worker between a pair's first and last holds a piece
    sp.total = total;
    sp.live_pairs = live;
    sp.gw = gw;
    sp.q = total / gw;
    sp.r = total % gw;
    const int pairs = P.num_seqs * P.num_kv_heads;
    const int share = (int)(((unsigned)total + (unsigned)gw - 1u) / (unsigned)gw);
    sp.whole = P.whole_sequences || (P.auto_policy && total > 0 && maxnb <= 2 * share && pairs <= W);
    sp.wmajor = !P.pack && (sp.whole ? pairs < W : gw < W);
    return sp;
}

// Side work of the consumer warps while the first steps are in flight: rows
// of sequences with no key get zeros (CTA s mod grid writes row s), and CTA 0
// records the plan (workers, pairs cut across workers, most pieces of one pair).
template <class Smem, int BS, int D>
__device__ void decode_side_work(const DecodeParams &P, Smem &sm, const Split &sp, int levels)
{
    constexpr int NT = kDecodeThreads;
    constexpr int NC = kConsumerWarps * 32;
    constexpr int NG = Smem::NG;
    const int tid = threadIdx.x;
    const int per = (P.num_seqs + NT - 1) / NT;
    const int Hkv = P.num_kv_heads;
    int split = 0, maxp = 1;
    for (int t = tid; t < NT; t += NC) {
        const int s_lo = min(P.num_seqs, t * per);
        const int s_hi = min(P.num_seqs, s_lo + per);
        int cum = 0;
        if (blockIdx.x == 0 && !sp.whole) {
            for (int w = 0; w < (t >> 5); ++w)
                cum += sm.wtot[w];
            cum += sm.toff[t];
        }
        for (int s = s_lo; s < s_hi; ++s) {
            const int L = s < kLensCache ? sm.lens[s] : clamped_len(P, s, BS, false);
            if (L == 0 && (s % (int)gridDim.x) == (int)blockIdx.x &&
                (P.table_row == nullptr || __ldg(P.table_row + s) >= 0)) {
                uint16_t *o = P.out + (long long)s * P.num_q_heads * D;
                for (int i = 0; i < P.num_q_heads * D; ++i)
                    o[i] = 0;
            }
            const int nb = nblocks_of(L, BS);
            const int span = pair_span(nb);
            if (blockIdx.x == 0 && !sp.whole && nb > 0) {
                for (int h = 0; h < Hkv; ++h) {
                    const int ps = cum + h * span;
                    const int np = worker_of(ps + span - 1, sp.q, sp.r) - worker_of(ps, sp.q, sp.r) + 1;
                    split += np > 1;
                    maxp = max(maxp, np);
                }
            }
            cum += Hkv * span;
        }
    }
    if (blockIdx.x != 0)
        return;
    atomicAdd(&sm.plan_split, split);
    atomicMax(&sm.plan_maxp, maxp);
    named_barrier_sync(1, NC);  // the consumer warps of CTA 0
    if (tid == 0) {
        ns_decode_plan pl;
        const int W = (int)gridDim.x * NG;
        const int pairs = P.num_seqs * Hkv;
        const int wact = sp.whole ? min(W, pairs) : sp.gw;
        pl.ctas_launched = gridDim.x;
        pl.ctas_active = sp.wmajor ? min((int)gridDim.x, wact) : (wact + NG - 1) / NG;
        pl.total_blocks = (long long)sp.total - (long long)kPieceCost * sp.live_pairs;  // real blocks
        pl.split_pairs = sp.whole ? 0 : sm.plan_split;
        pl.max_pieces = sp.whole ? 1 : sm.plan_maxp;
        pl.whole_sequences = sp.whole ? 1 : 0;
        pl.workers_active = wact;
        pl.merge_levels = levels;
        for (int i = 0; i < 7; ++i)
            pl.reserved[i] = 0;
        *P.plan = pl;
    }
}

template <typename T, int BS, int G, int S, bool Q8, int D, bool TWO = false, int VU = 0>
__global__ void __launch_bounds__(kDecodeThreads, 1) paged_decode_kernel(const DecodeParams P)
{
    using Smem = DecodeSmem<BS, G, S, Q8, D>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    using Shape = DecodeShape<G>;
    // the next grid on the stream may be scheduled on SMs this one frees
    // (only when it was launched as a programmatic dependent)
    grid_launch_dependents();
    decode_prologue<Smem, BS>(P, sm);
    const Split sp = read_split(P, sm);
    // Registers move from the producer warpgroup to the consumer warpgroups;
    // the shares add up to the launch allocation.
    if (warp < kConsumerWarps) {
        regs_grow<kConsumerRegs>();
        // launched as a programmatic dependent: the side work writes the
        // output and the plan, which the previous grid may still be using
        if (P.overlap)
            grid_dependency_wait();
        decode_side_work<Smem, BS, D>(P, sm, sp, TWO ? 2 : 1);
        decode_consumer<T, BS, G, S, Q8, D, TWO, VU>(P, sm, sp, warp, warp, lane);
    } else {
        regs_shrink<kProducerRegs>();
        if (warp - kConsumerWarps < Shape::PW)
            decode_producer<T, BS, G, S, Q8, D>(P, sm, sp, warp - kConsumerWarps, lane);
    }
}

// Host-side launch helpers (defined in the per-type instantiation files).
// Q8: the pools are q8_0 codes and scales (DecodeParams.k_codes ...); D: head dim;
// TWO: two-level merges; VU: the values pass's unroll (0: whole).
template <typename T, int BS, int G, bool Q8 = false, int D = 64, bool TWO = false, int VU = 0>
cudaError_t launch_paged_decode(const DecodeParams &P, int num_ctas, cudaStream_t stream);

template <typename T, int BS, int G, bool Q8 = false, int D = 64>
int decode_ctas_per_sm();

}  // namespace ns
