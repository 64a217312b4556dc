/*
 * ns_paged.h -- C ABI of the GB300 (sm_103a) paged-KV attention library.
 *
 * The library is the data-parallel hot path of a nanoserve-style LLM server:
 * every query head of every running sequence walks its block table over a
 * paged K/V pool with online softmax (nanoserve project page, "What I built":
 * paged KV cache with block tables; fused paged-attention decode kernel with
 * online softmax over the block table), after the step's new K/V rows have
 * been written to their pool slots (Inference Engineering Day 11 short, "How
 * does vLLM work": the engine's cache update of each step).  Long
 * contexts are split across CTAs and merged by log-sum-exp, the flash-decoding
 * split arm of the nanoserve author's build log (Day 74 post).  A chunked
 * prefill variant takes a span of query tokens per sequence (nanoserve project
 * page, "What I built", continuous batching bullet: chunked prefill;
 * Inference Engineering Day 12 short, "What is chunked prefill within vLLM").
 *
 * ---------------------------------------------------------------------------
 * Conventions shared by every entry point
 * ---------------------------------------------------------------------------
 *  Pointers     Every tensor argument is a DEVICE pointer on the current CUDA
 *               device, 16-byte aligned, dense (row-major, no padding) unless
 *               a stride argument says otherwise.  The caller owns and
 *               allocates every buffer; the library allocates nothing and
 *               frees nothing.
 *  Streams      Work is enqueued on `stream` (NULL = the legacy default
 *               stream) and the call returns without synchronising.  Inputs
 *               must stay valid until the work completes.
 *  Elements     K, V, q and out are fp16 or bf16 (`ns_dtype`), all of one type.
 *  Shapes       head_dim is 64, or 128 with block_size 16 (the q8_0 pools
 *               and the allocation-free entry point take 64).
 *               num_q_heads must be a multiple of num_kv_heads; query head
 *               j reads KV head j / G, G = num_q_heads / num_kv_heads.  G is
 *               at most 8, or up to 64 when it is a multiple of
 *               n = ceil(G / 8): such a group runs as n groups of G / n heads
 *               over the same KV head (the tensor-core prefill and the
 *               allocation-free entry point take G <= 8; larger groups'
 *               spans take the split-KV walk).  block_size must be 4, 8, 16
 *               or 32.
 *  Pool layout  k_pool and v_pool are [num_blocks][num_kv_heads][block_size]
 *               [head_dim]: one (block, kv head) is block_size*head_dim
 *               contiguous elements.  Token slot s lives in block
 *               s / block_size at offset s % block_size.
 *  Tables       block_tables is int32 [num_seqs][max_blocks_per_seq]; entry
 *               [s][i] is the pool block holding tokens i*block_size ..
 *               (i+1)*block_size-1 of sequence s.  Only the first
 *               ceil(context_lens[s] / block_size) entries of a row are read.
 *               context_lens is int32 [num_seqs] and counts the tokens in the
 *               pool INCLUDING this step's new ones.
 *  Errors       Argument checks run on the host before anything is enqueued
 *               and return a negative ns_status; nothing is launched then.  A
 *               failed launch returns NS_ERR_CUDA.  Checks that need device
 *               data (block ids inside the pool, lengths that fit the table,
 *               slots inside the pool) run inside the kernels on every call:
 *               a bad unit is skipped (never read or written out of bounds)
 *               and a bit is OR-ed into the device status word, which
 *               ns_get_device_status() returns.  No kernel traps or aborts.
 *  Waits        Every wait inside a kernel is bounded (about one second);
 *               on expiry the kernel sets NS_DEV_WAIT_TIMEOUT and returns.
 */
#ifndef NS_PAGED_H
#define NS_PAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *ns_stream_t;

typedef enum ns_status {
    NS_OK = 0,
    NS_ERR_INVALID_ARG = -1,   /* null pointer, misalignment, negative size, too-small buffer */
    NS_ERR_UNSUPPORTED = -2,   /* a shape or type outside the supported set above */
    NS_ERR_CUDA = -3,          /* a CUDA runtime call or a launch failed */
    NS_ERR_DEVICE = -4         /* ns_get_device_status found a device-side status bit */
} ns_status;

typedef enum ns_dtype { NS_F16 = 0, NS_BF16 = 1 } ns_dtype;

/* Device status bits (ns_get_device_status). */
#define NS_DEV_BAD_BLOCK_ID 0x1u     /* a block table entry outside [0, num_blocks) */
#define NS_DEV_BAD_CONTEXT_LEN 0x2u  /* context_len < 0 or > max_blocks_per_seq*block_size */
#define NS_DEV_BAD_SLOT 0x4u         /* a slot_mapping entry >= num_blocks*block_size */
#define NS_DEV_WAIT_TIMEOUT 0x8u     /* a bounded wait inside a kernel expired */
#define NS_DEV_FUSED_SLOT 0x10u      /* fused append: slot is not the slot of position L-1 */
#define NS_DEV_BAD_QUERY_SPAN 0x20u  /* prefill: query span longer than the context, or negative */
#define NS_DEV_MERGE_QUEUE 0x40u     /* decode: a CTA's merge queue overflowed (a merge was skipped) */

/* Human-readable name of a status code (static string). */
const char *ns_status_string(ns_status status);

/* Library version, major*10000 + minor*100 + patch. */
int ns_version(void);

/*
 * ns_kv_append -- write the step's new tokens into their pool slots.
 *
 * Definition (Inference Engineering Day 11 short, "How does vLLM work": each
 * step stores its tokens' new K/V rows in the cache; paged layout from the
 * nanoserve project page, "What I built"):
 *   for every token t with slot_mapping[t] >= 0 and every kv head h:
 *     k_pool[slot/bs][h][slot%bs][:] = k[t][h][:]   (same for v)
 * A bit-exact copy.  A negative slot marks a padding token and is skipped.
 *
 *   k, v          [num_tokens][num_kv_heads][head_dim] elements (read)
 *   slot_mapping  int64 [num_tokens] (read)
 *   k_pool/v_pool [num_blocks][num_kv_heads][block_size][head_dim] (written)
 * Slots >= num_blocks*block_size are skipped and set NS_DEV_BAD_SLOT.  Two
 * tokens with the same slot race (one of them wins).  num_tokens == 0 is a
 * no-op.
 */
ns_status ns_kv_append(const void *k, const void *v, const int64_t *slot_mapping,
                       void *k_pool, void *v_pool, int num_tokens, int num_kv_heads,
                       int head_dim, int block_size, int64_t num_blocks, ns_dtype dtype,
                       ns_stream_t stream);

/*
 * Workspace for the attention entry points: split-KV partial results
 * (fp32 running max, running sum and unnormalised output of each piece of a
 * sequence that was cut across workers: about 8.7 MB for head_dim 64, 17 MB
 * for 128), one arrival counter per (sequence, kv head) and a small plan
 * record.  Size it with ns_paged_attn_workspace_bytes for the largest
 * num_seqs and the head_dim you will pass.  It must be zero-filled once before
 * first use (ns_paged_attn_workspace_init or cudaMemsetAsync); every call
 * that completes without a device status bit leaves it ready for the next
 * call.  Two calls that share a workspace must not run concurrently.
 */
size_t ns_paged_attn_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim);

/* cudaMemsetAsync(workspace, 0, workspace_bytes, stream). */
ns_status ns_paged_attn_workspace_init(void *workspace, size_t workspace_bytes,
                                       ns_stream_t stream);

/*
 * ns_paged_attn_decode -- one decode step of paged attention.
 *
 * Definition (nanoserve project page, "What I built": fused paged-attention
 * decode with online softmax over the block table).  For every sequence s,
 * query head j, with h = j / (num_q_heads/num_kv_heads) and L = context_lens[s]:
 *   z_p   = scale * sum_d q[s][j][d] * K_s[p][d],    p = 0 .. L-1
 *   out[s][j][:] = sum_p softmax(z)_p * V_s[p][:]
 * where K_s[p] = k_pool[block_tables[s][p/bs]][h][p%bs].  A sequence with
 * L == 0 gets out = 0.  Arithmetic is fp32 with the output rounded to the
 * element type; the result matches the exact value within the tolerance of
 * the test suite, not bit for bit.
 *
 *   q            [num_seqs][num_q_heads][head_dim] (read)
 *   out          [num_seqs][num_q_heads][head_dim] (written)
 *   max_blocks_per_seq  row stride of block_tables (entries)
 *   num_blocks   pool size in blocks (block ids are checked against it)
 *   scale        softmax scale, usually 1/sqrt(head_dim)
 *   workspace    see ns_paged_attn_workspace_bytes (read and written)
 *
 * The work is spread evenly over a persistent grid: the KV blocks of all
 * (sequence, kv head) pairs are laid end to end and each CTA takes an equal
 * run of them, so a long context is split across CTAs (flash-decoding style)
 * and its partial results are merged by log-sum-exp.  How many CTAs run is
 * decided on the device from the actual context lengths and batch size.
 */
ns_status ns_paged_attn_decode(const void *q, const void *k_pool, const void *v_pool,
                               const int32_t *block_tables, const int32_t *context_lens,
                               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, float scale, void *out, ns_stream_t stream,
                               int max_blocks_per_seq, int64_t num_blocks, ns_dtype dtype,
                               void *workspace, size_t workspace_bytes);

/*
 * Policy overrides for the split-KV decode (tests and measurements).
 *   num_ctas            0 = auto (resident CTAs on this GPU); else the grid size
 *                       (1 .. NS_MAX_CTAS)
 *   min_blocks_per_cta  0 = auto; fewer workers (warps, 8 per CTA) are used
 *                       when the total work would give each less than an
 *                       eighth of this many KV blocks
 *   whole_sequences     nonzero = never split a (sequence, kv head): worker w
 *                       of W takes pairs w, w+W, w+2W, ... (no merge step)
 *   overlap_prologue    nonzero = launch as a programmatic dependent of the
 *                       kernel before it on the stream (CUDA programmatic
 *                       dependent launch): the decode may start while that
 *                       kernel drains, reads context_lens and block_tables,
 *                       then waits for it to finish before it touches q, the
 *                       pools, k_new/v_new, slot_mapping, out or the
 *                       workspace.  The caller guarantees that the kernel just
 *                       before it on the stream does not write context_lens or
 *                       block_tables.  It also lets the kernel after it start
 *                       early.  Not a policy override: the split stays automatic.
 *   wait_limit_ns       0 = default (about one second); else the limit, in ns, of
 *                       each wait of a computing warp for its next K/V step.  On
 *                       expiry the kernel sets NS_DEV_WAIT_TIMEOUT, stops issuing
 *                       copies, waits (with the default limit) for the copies it
 *                       has in flight and returns; the outputs of that call are
 *                       undefined and the workspace must be zero-filled again
 *                       (ns_paged_attn_workspace_init) before its next use.  For
 *                       testing the failure path: a limit shorter than a copy's
 *                       latency makes every call time out.
 *   merge_levels        0 = automatic; 1 = every cut pair merges its pieces'
 *                       records in one step; 2 = a pair cut into 16 or more
 *                       pieces first combines its pieces inside each CTA
 *                       (block size 16, head_dim 64, 16-bit pools; elsewhere
 *                       ignored).  Automatic takes 2 there when the pairs are
 *                       few for the CTAs' warps (32 or more warps a pair) and
 *                       their table rows span the warps; the single-token
 *                       rows of a prefill call choose the same way.  The
 *                       result is the same up to rounding order.
 *   reserved            must be 0.
 */
#define NS_MAX_CTAS 1024
typedef struct ns_decode_config {
    int num_ctas;
    int min_blocks_per_cta;
    int whole_sequences;
    int overlap_prologue;
    int wait_limit_ns;
    int merge_levels;
    int reserved[2];
} ns_decode_config;

/* ns_paged_attn_decode with policy overrides (cfg may be NULL = auto). */
ns_status ns_paged_attn_decode_ex(const void *q, const void *k_pool, const void *v_pool,
                                  const int32_t *block_tables, const int32_t *context_lens,
                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, float scale, void *out, ns_stream_t stream,
                                  int max_blocks_per_seq, int64_t num_blocks, ns_dtype dtype,
                                  void *workspace, size_t workspace_bytes,
                                  const ns_decode_config *cfg);

/*
 * ns_kv_append_paged_attn_decode -- ns_kv_append of one new token per
 * sequence followed by ns_paged_attn_decode, in one kernel.
 *
 *   k_new, v_new  [num_seqs][num_kv_heads][head_dim] (read): token s is the
 *                 new token of sequence s, at position context_lens[s]-1
 *   slot_mapping  int64 [num_seqs]: must be the slot of that position,
 *                 block_tables[s][(L-1)/bs]*bs + (L-1)%bs
 * The result equals the two calls in order: the pool slot is written and the
 * attention includes the new token.  The CTA that owns a sequence's last
 * block takes the new K/V from k_new/v_new (never from the pool slot it is
 * writing), so nothing reads the slot while it is written.  A slot that is
 * not the slot of position L-1 sets NS_DEV_FUSED_SLOT (the slot is still
 * written; the attention still uses the new token at position L-1).
 */
ns_status ns_kv_append_paged_attn_decode(const void *q, const void *k_new, const void *v_new,
                                         const int64_t *slot_mapping, void *k_pool,
                                         void *v_pool, const int32_t *block_tables,
                                         const int32_t *context_lens, int num_seqs,
                                         int num_q_heads, int num_kv_heads, int head_dim,
                                         int block_size, float scale, void *out,
                                         ns_stream_t stream, int max_blocks_per_seq,
                                         int64_t num_blocks, ns_dtype dtype, void *workspace,
                                         size_t workspace_bytes);

/* ns_kv_append_paged_attn_decode with policy overrides (cfg may be NULL = auto). */
ns_status ns_kv_append_paged_attn_decode_ex(const void *q, const void *k_new, const void *v_new,
                                            const int64_t *slot_mapping, void *k_pool,
                                            void *v_pool, const int32_t *block_tables,
                                            const int32_t *context_lens, int num_seqs,
                                            int num_q_heads, int num_kv_heads, int head_dim,
                                            int block_size, float scale, void *out,
                                            ns_stream_t stream, int max_blocks_per_seq,
                                            int64_t num_blocks, ns_dtype dtype, void *workspace,
                                            size_t workspace_bytes, const ns_decode_config *cfg);

/*
 * Plan record the decode kernels leave at the start of the workspace (CTA 0
 * writes it during every call).  It shows which split the device chose.  The
 * unit of work is a worker: one warp of a CTA (8 workers per CTA).
 *   ctas_launched   grid size
 *   ctas_active     CTAs with at least one worker that received work
 *   total_blocks    KV blocks over all (sequence, kv head) pairs
 *   split_pairs     (sequence, kv head) pairs cut across two or more workers
 *   max_pieces      most workers sharing one pair
 *   whole_sequences 1 when the no-split policy ran
 *   workers_active  workers that received work
 */
typedef struct ns_decode_plan {
    int32_t ctas_launched;
    int32_t ctas_active;
    int64_t total_blocks;
    int32_t split_pairs;
    int32_t max_pieces;
    int32_t whole_sequences;
    int32_t workers_active;
    int32_t merge_levels;  /* 1 or 2: the merge the kernel was built for (see merge_levels above) */
    int32_t reserved[7];
} ns_decode_plan;

/* Copy the plan record out of `workspace` (synchronises `stream`). */
ns_status ns_read_decode_plan(const void *workspace, ns_decode_plan *plan, ns_stream_t stream);

/*
 * ns_paged_attn_prefill -- chunked-prefill attention over query spans.
 *
 * Definition (Inference Engineering Day 12 short, "What is chunked prefill
 * within vLLM": a chunk's K/V are written into blocks and the chunk attends
 * to everything already cached; nanoserve project page, "What I built").
 * Sequence s owns query rows query_start_loc[s] .. query_start_loc[s+1]-1;
 * with n = query_start_loc[s+1]-query_start_loc[s] and L = context_lens[s],
 * row i sits at position L-n+i and sees keys p <= L-n+i (cached prefix plus
 * causal within the span).  The span's own K/V must already be in the pool
 * (ns_kv_append first).  A span of one row is a decode step.
 *
 *   q               [total_q_tokens][num_q_heads][head_dim] (read)
 *   query_start_loc int32 [num_seqs+1], nondecreasing, [0] == 0,
 *                   [num_seqs] == total_q_tokens (read)
 *   out             [total_q_tokens][num_q_heads][head_dim] (written)
 * Spans of two or more rows run on the tcgen05 tensor cores when block_size
 * is 16 or 32: query-key and probability-value products take fp16/bf16
 * operands with fp32 accumulation (the probabilities are rounded to the
 * element type before the second product).  Single-row spans, and every span
 * for other block sizes, take the split-KV decode walk.  The workspace is
 * sized with ns_paged_attn_workspace_bytes(total_q_tokens, ...).
 */
ns_status ns_paged_attn_prefill(const void *q, const int32_t *query_start_loc,
                                const void *k_pool, const void *v_pool,
                                const int32_t *block_tables, const int32_t *context_lens,
                                int num_seqs, int total_q_tokens, int num_q_heads,
                                int num_kv_heads, int head_dim, int block_size, float scale,
                                void *out, ns_stream_t stream, int max_blocks_per_seq,
                                int64_t num_blocks, ns_dtype dtype, void *workspace,
                                size_t workspace_bytes);

/*
 * Policy overrides for the chunked prefill (tests and measurements).
 *   tensor_core_min_span  0 = auto: spans of 2 or more query tokens run on the
 *                         tensor cores when block_size is 16 or 32, unless the
 *                         call has no more query tokens than spans (then every
 *                         row takes the split-KV walk); a positive
 *                         value raises that threshold; -1 = never (every row
 *                         takes the split-KV decode walk)
 *   phases                0 = everything; else a mask of the parts to run
 *                         (NS_PREFILL_WALK: the split-KV walk over the rows it
 *                         owns, NS_PREFILL_TENSOR_CORE: the tensor-core spans),
 *                         so each part can be timed on its own
 */
#define NS_PREFILL_WALK 1
#define NS_PREFILL_TENSOR_CORE 2
typedef struct ns_prefill_config {
    int tensor_core_min_span;
    int phases;
    int reserved[6];
} ns_prefill_config;

/* ns_paged_attn_prefill with policy overrides (cfg may be NULL = auto). */
ns_status ns_paged_attn_prefill_ex(const void *q, const int32_t *query_start_loc,
                                   const void *k_pool, const void *v_pool,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   int num_seqs, int total_q_tokens, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size, float scale,
                                   void *out, ns_stream_t stream, int max_blocks_per_seq,
                                   int64_t num_blocks, ns_dtype dtype, void *workspace,
                                   size_t workspace_bytes, const ns_prefill_config *cfg);

/*
 * ns_paged_attn_decode_noalloc -- ns_paged_attn_decode for callers that
 * cannot allocate device memory.
 *
 * The pages describe no such entry point; it serves callers that may not
 * call cudaMalloc or a caching allocator at all: plugins inside a host
 * runtime that owns every device allocation, and serving loops that must not
 * allocate once they run.  It takes the same inputs and output as
 * ns_paged_attn_decode (same checks, same result) but no workspace: the split
 * partial records, arrival counters and plan record live in a scratch array
 * compiled into the library (about 8.7 MB, held by every GPU that loads the
 * library until the process exits).
 *   - num_seqs * num_kv_heads must not exceed NS_NOALLOC_MAX_PAIRS; larger
 *     calls return NS_ERR_UNSUPPORTED and launch nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.
 *   - Every call clears the arrival counters it needs (cudaMemsetAsync on
 *     `stream`) before its kernel; it allocates and frees nothing.
 *   - All calls share the one array: calls that overlap on the GPU (two
 *     streams, two threads) race and give wrong results.
 */
#define NS_NOALLOC_MAX_PAIRS 16384
ns_status ns_paged_attn_decode_noalloc(const void *q, const void *k_pool, const void *v_pool,
                                       const int32_t *block_tables, const int32_t *context_lens,
                                       int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, float scale, void *out,
                                       ns_stream_t stream, int max_blocks_per_seq,
                                       int64_t num_blocks, ns_dtype dtype);

/*
 * 8-bit (q8_0) KV cache.  The video-shorts aggregator page's post on serving
 * a 26B model on one 24 GB GPU ("q8 kv cache") keeps K and V in llama.cpp's
 * q8_0 format, 8 bits instead of 16, dequantised on the fly by every
 * attention step.  The pages name the format without defining it; the reading
 * taken here is the q8_0 block format:
 *   - a block is 32 consecutive elements of one token's head row (a 64-wide
 *     row holds two);
 *   - its scale d = max|x| / 127 in fp32, stored as fp16 (nearest even,
 *     saturating at 65504); an all-zero block has d = 0;
 *   - code = rint(x * (1/d)) with both products rounded to fp32, ties to even,
 *     clamped to [-127, 127]; the code q stands for fp16(d) * q.
 * Pools: k_codes, v_codes int8 [num_blocks][num_kv_heads][block_size][64];
 * k_scales, v_scales fp16 [num_blocks][num_kv_heads][block_size][2] (the
 * scale of elements 0-31, then of 32-63).  All four 16-byte aligned.
 */

/*
 * ns_kv_append_q8_0 -- ns_kv_append into a q8_0 pool: each new token's K and
 * V rows (fp16 or bf16, [num_tokens][num_kv_heads][64]) are quantised as
 * above and their codes and scales written at slot_mapping (negative: skipped;
 * outside the pool: skipped, NS_DEV_BAD_SLOT).  The codes and scales match the
 * q8_0 definition bit for bit.  block_size 4, 8, 16 or 32.
 */
ns_status ns_kv_append_q8_0(const void *k, const void *v, const int64_t *slot_mapping,
                            void *k_codes, void *k_scales, void *v_codes, void *v_scales,
                            int num_tokens, int num_kv_heads, int head_dim, int block_size,
                            int64_t num_blocks, ns_dtype dtype, ns_stream_t stream);

/*
 * ns_paged_attn_decode_q8_0 -- ns_paged_attn_decode over a q8_0 pool: the
 * same definition with K_s[p] and V_s[p] the dequantised rows
 * (fp16(d) * code).  q and out are fp16 or bf16 (dtype); the arithmetic is
 * fp32.  block_size must be 16.  Same workspace, split and merge as the
 * 16-bit decode; the copies move 64 code bytes and 4 scale bytes per row
 * instead of 128.
 */
ns_status ns_paged_attn_decode_q8_0(const void *q, const void *k_codes, const void *k_scales,
                                   const void *v_codes, const void *v_scales,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, float scale, void *out, ns_stream_t stream,
                                   int max_blocks_per_seq, int64_t num_blocks, ns_dtype dtype,
                                   void *workspace, size_t workspace_bytes);

/*
 * ns_kv_append_paged_attn_decode_q8_0 -- ns_kv_append_q8_0 of one new token
 * per sequence followed by ns_paged_attn_decode_q8_0, in one kernel (the q8_0
 * form of ns_kv_append_paged_attn_decode: the same slot rule and status
 * bits).  The attention sees the new token quantised, as the two calls would.
 */
ns_status ns_kv_append_paged_attn_decode_q8_0(const void *q, const void *k_new, const void *v_new,
                                             const int64_t *slot_mapping, void *k_codes,
                                             void *k_scales, void *v_codes, void *v_scales,
                                             const int32_t *block_tables,
                                             const int32_t *context_lens, int num_seqs,
                                             int num_q_heads, int num_kv_heads, int head_dim,
                                             int block_size, float scale, void *out,
                                             ns_stream_t stream, int max_blocks_per_seq,
                                             int64_t num_blocks, ns_dtype dtype, void *workspace,
                                             size_t workspace_bytes);

/*
 * Device status word of the current device: OR of NS_DEV_* bits raised by
 * kernels since the last clear.  Synchronises `stream`, copies the word to
 * *bits, and zeroes it when `clear` is nonzero.  Returns NS_OK (whatever the
 * bits) or NS_ERR_CUDA.
 */
ns_status ns_get_device_status(ns_stream_t stream, uint32_t *bits, int clear);

#ifdef __cplusplus
}
#endif

#endif /* NS_PAGED_H */
