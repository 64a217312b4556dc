"""Seeded synthetic inputs for the paged-KV hot path.

This module builds the inputs of one serving step -- context lengths, a
block-table KV pool, query rows, the step's new K/V tokens and their slots --
and nothing else.  It holds none of the attention arithmetic: both the CUDA
path and the CPU oracle consume what it returns, so the two see identical
bytes.

Provenance of the shapes and distributions:
  * the paged KV cache with a block allocator and per-sequence block tables,
    waste under one block per sequence (nanoserve project page, "What I built",
    paged KV cache bullet);
  * lognormal request lengths (nanoserve project page, "What I built",
    benchmark harness bullet);
  * Qwen2.5-0.5B attention geometry, fp16 (nanoserve project page, "What the
    numbers don't say"): 14 query heads, 2 KV heads, head_dim 64;
  * chunked prefill writes a prompt chunk by chunk into fixed-size blocks
    (Inference Engineering Day 12 short, "What is chunked prefill within
    vLLM": 8-token chunks into 4-token blocks occupy 2, then 4 blocks).

Element values are stored as raw 16-bit patterns (``uint16``) of fp16 or
bf16.  Values are N(0, 1) drawn in float32 and rounded to the element type
with round-to-nearest-even.

Draw order for every workload (one ``numpy.random.Generator``): lengths,
block permutation, q, pool K, pool V, new K, new V.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

F16 = "f16"
BF16 = "bf16"
DTYPES = (F16, BF16)

# Bit patterns used to poison slots that hold no live token.
NAN_BITS = {F16: 0x7E00, BF16: 0x7FC0}


def float_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to fp16 / bf16 (nearest-even); return raw bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        u = x.view(np.uint32).astype(np.uint64)
        r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        return r.astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def _randn_bits(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    chunk = 1 << 24
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        out[lo:hi] = float_to_bits(rng.standard_normal(hi - lo, dtype=np.float32), dtype)
    return out.reshape(shape)


def blocks_needed(length: int, block_size: int) -> int:
    """Blocks a sequence of ``length`` tokens occupies: ceil(length / block_size)."""
    return -(-int(length) // int(block_size))


def lognormal_lengths(rng: np.random.Generator, n: int, median: float, sigma: float,
                      max_len: int, min_len: int = 1) -> np.ndarray:
    """Request lengths L = clip(rint(exp(N(ln median, sigma))), min_len, max_len)."""
    z = rng.normal(math.log(median), sigma, size=n)
    return np.clip(np.rint(np.exp(z)), min_len, max_len).astype(np.int32)


@dataclasses.dataclass
class PagedStep:
    """One step of the hot path: append the new tokens, then attend.

    Shapes (S sequences, T query/new tokens, NB pool blocks):
      context_lens     int32  [S]     tokens per sequence AFTER this step's append
      query_lens       int32  [S]     query tokens of each sequence (1 = decode)
      query_start_loc  int32  [S+1]   prefix sums of query_lens
      block_tables     int32  [S, max_blocks_per_seq]; entries past
                                      ceil(L/bs) hold -1
      k_pool, v_pool   uint16 [NB, Hkv, bs, D]   pool BEFORE the append
      q                uint16 [T, Hq, D]
      k_new, v_new     uint16 [T, Hkv, D]        this step's tokens
      slot_mapping     int64  [T]     slot = block_id * bs + offset of each new
                                      token; token i of sequence s sits at
                                      position context_lens[s] - query_lens[s] + i
    """

    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    context_lens: np.ndarray
    query_lens: np.ndarray
    query_start_loc: np.ndarray
    block_tables: np.ndarray
    num_blocks: int
    k_pool: np.ndarray
    v_pool: np.ndarray
    q: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    slot_mapping: np.ndarray

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def is_decode(self) -> bool:
        return bool(np.all(self.query_lens == 1))

    def kv_row_bytes(self, kv: str = "native") -> int:
        """Bytes of one token's K (or V) row of one kv head in the pool: 2 per
        element for the 16-bit pools; for q8_0 one code per element plus an
        fp16 scale per 32 elements."""
        if kv == "q8_0":
            return self.head_dim + 2 * (self.head_dim // 32)
        return 2 * self.head_dim

    def kv_read_bytes(self, kv: str = "native") -> int:
        """K and V bytes one attention pass over every context reads."""
        return int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads * 2 * self.kv_row_bytes(kv)

    def algorithmic_bytes(self, with_append: bool = True, kv: str = "native") -> int:
        """Bytes the step must move at minimum (each input read once, output written once).

        K/V of every context token + q in + out + the block-table entries in
        use + context lengths (+ new K/V read, pool slots written and slots read
        when the append is part of the step).  ``kv`` is the pool format.
        """
        esz = 2
        b = self.kv_read_bytes(kv)
        b += 2 * self.num_tokens * self.num_q_heads * self.head_dim * esz
        nb = sum(blocks_needed(L, self.block_size) for L in self.context_lens)
        b += 4 * nb + 4 * self.num_seqs
        if not self.is_decode:
            b += 4 * (self.num_seqs + 1)
        if with_append:
            new_rows = self.num_kv_heads * self.head_dim * esz * 2      # K and V read (16-bit)
            pool_rows = self.num_kv_heads * self.kv_row_bytes(kv) * 2   # K and V written
            b += self.num_tokens * (new_rows + pool_rows + 8)
        return int(b)


def make_step(rng: np.random.Generator, context_lens, query_lens, *, dtype: str,
              num_q_heads: int = 14, num_kv_heads: int = 2, head_dim: int = 64,
              block_size: int = 16, scale: float | None = None,
              num_blocks: int | None = None, free_frac: float = 0.10,
              max_blocks_per_seq: int | None = None, poison_unused: bool = False,
              name: str = "step") -> PagedStep:
    """Build a step from lengths already drawn from ``rng``.

    The toy allocator takes a seeded permutation of the pool's block ids and
    hands each sequence the next ceil(L/bs) ids in order, so every sequence
    wastes fewer than ``block_size`` slots.  ``num_blocks`` defaults to the
    blocks in use plus ``free_frac`` of them (rounded up) left free.
    """
    if dtype not in DTYPES:
        raise ValueError(dtype)
    context_lens = np.asarray(context_lens, dtype=np.int32)
    query_lens = np.asarray(query_lens, dtype=np.int32)
    S = context_lens.shape[0]
    if query_lens.shape != (S,):
        raise ValueError("query_lens must have one entry per sequence")
    if np.any(query_lens < 0) or np.any(query_lens > context_lens):
        raise ValueError("need 0 <= query_len <= context_len")
    nbs = np.array([blocks_needed(L, block_size) for L in context_lens], dtype=np.int64)
    used = int(nbs.sum())
    if num_blocks is None:
        num_blocks = used + int(math.ceil(free_frac * used))
    if num_blocks < used:
        raise ValueError("pool too small")
    mbps = int(max_blocks_per_seq if max_blocks_per_seq is not None else max(1, int(nbs.max(initial=1))))
    if mbps < int(nbs.max(initial=0)):
        raise ValueError("max_blocks_per_seq too small")

    perm = rng.permutation(num_blocks).astype(np.int32)
    block_tables = np.full((S, mbps), -1, dtype=np.int32)
    off = 0
    for s in range(S):
        n = int(nbs[s])
        block_tables[s, :n] = perm[off:off + n]
        off += n

    T = int(query_lens.sum())
    qsl = np.zeros(S + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(query_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)

    q = _randn_bits(rng, (T, num_q_heads, head_dim), dtype)
    k_pool = _randn_bits(rng, (num_blocks, num_kv_heads, block_size, head_dim), dtype)
    v_pool = _randn_bits(rng, (num_blocks, num_kv_heads, block_size, head_dim), dtype)
    k_new = _randn_bits(rng, (T, num_kv_heads, head_dim), dtype)
    v_new = _randn_bits(rng, (T, num_kv_heads, head_dim), dtype)

    slot_mapping = np.empty(T, dtype=np.int64)
    for s in range(S):
        first = int(context_lens[s] - query_lens[s])
        for i in range(int(query_lens[s])):
            p = first + i
            slot_mapping[qsl[s] + i] = int(block_tables[s, p // block_size]) * block_size + p % block_size

    if poison_unused:
        live = np.zeros((num_blocks, block_size), dtype=bool)
        for s in range(S):
            L = int(context_lens[s])
            for p in range(L - int(query_lens[s])):  # tokens already cached
                live[block_tables[s, p // block_size], p % block_size] = True
        nan = np.uint16(NAN_BITS[dtype])
        k_pool.transpose(0, 2, 1, 3)[~live] = nan   # [NB, bs, Hkv, D] view
        v_pool.transpose(0, 2, 1, 3)[~live] = nan

    return PagedStep(name=name, dtype=dtype, num_q_heads=num_q_heads,
                     num_kv_heads=num_kv_heads, head_dim=head_dim,
                     block_size=block_size, scale=float(scale),
                     context_lens=context_lens, query_lens=query_lens,
                     query_start_loc=qsl, block_tables=block_tables,
                     num_blocks=int(num_blocks), k_pool=k_pool, v_pool=v_pool,
                     q=q, k_new=k_new, v_new=v_new, slot_mapping=slot_mapping)


# --------------------------------------------------------------------------
# The five workloads (Qwen2.5-0.5B attention geometry: 14 q / 2 kv heads,
# head_dim 64, block_size 16, scale 1/8).  Seeds are 1000 + workload number.
# --------------------------------------------------------------------------

def tiny_decode(seed: int = 1001, **kw) -> PagedStep:
    """Decode step, 4 sequences of {1, 17, 64, 200} tokens, fp16, 32-block pool."""
    rng = np.random.default_rng(seed)
    lens = np.array([1, 17, 64, 200], dtype=np.int32)
    kw.setdefault("dtype", F16)
    kw.setdefault("num_blocks", 32)
    return make_step(rng, lens, np.ones(4, np.int32), name="tiny_decode_4seq", **kw)


def lognormal_decode(num_seqs: int, median: float, sigma: float, max_len: int,
                     dtype: str, seed: int, name: str, **kw) -> PagedStep:
    rng = np.random.default_rng(seed)
    lens = lognormal_lengths(rng, num_seqs, median, sigma, max_len)
    return make_step(rng, lens, np.ones(num_seqs, np.int32), dtype=dtype, name=name, **kw)


def decode_batch32(seed: int = 1002, **kw) -> PagedStep:
    """Decode step, 32 sequences, lengths lognormal(median 512, sigma 1.0) in [1, 4096], fp16."""
    return lognormal_decode(32, 512, 1.0, 4096, kw.pop("dtype", F16), seed,
                            "decode_b32_ln512", **kw)


def long_context_decode(seed: int = 1003, **kw) -> PagedStep:
    """Decode step, 8 sequences of 4096 tokens, fp16."""
    rng = np.random.default_rng(seed)
    lens = np.full(8, 4096, dtype=np.int32)
    kw.setdefault("dtype", F16)
    return make_step(rng, lens, np.ones(8, np.int32), name="decode_b8_ctx4096", **kw)


def decode_batch256(seed: int = 1004, **kw) -> PagedStep:
    """Continuous-batching decode step, 256 sequences, lognormal(median 1024, sigma 1.2) in [1, 8192], bf16."""
    return lognormal_decode(256, 1024, 1.2, 8192, kw.pop("dtype", BF16), seed,
                            "decode_b256_ln1024", **kw)


def mixed_chunked_prefill(seed: int = 1005, **kw) -> PagedStep:
    """16 decode sequences (lognormal median 768, sigma 1.0, in [1, 4096]) then
    two 512-token prefill chunks over cached prefixes of 1500 and 3000 tokens, fp16."""
    rng = np.random.default_rng(seed)
    dec = lognormal_lengths(rng, 16, 768, 1.0, 4096)
    lens = np.concatenate([dec, np.array([1500 + 512, 3000 + 512], dtype=np.int32)])
    qlens = np.concatenate([np.ones(16, np.int32), np.array([512, 512], np.int32)])
    kw.setdefault("dtype", F16)
    return make_step(rng, lens, qlens, name="mixed_16dec_2x512chunk", **kw)


# Attention layers of the Qwen2.5-0.5B stack (the pages' model): every layer
# has its own K/V pool and its own q / new K / new V, while the block tables,
# lengths and slots are the sequences' and so the same in every layer.
QWEN25_05B_LAYERS = 24


def layer_steps(st: PagedStep, num_layers: int, seed: int = 7000) -> list:
    """``num_layers`` steps sharing ``st``'s block tables, lengths and slots;
    layer 0 is ``st`` itself, layer l > 0 draws fresh pools, q and new K/V
    (seeded, standard normal, rounded to the step's type)."""
    out = [st]
    for layer in range(1, num_layers):
        rng = np.random.default_rng(seed + layer)
        out.append(dataclasses.replace(
            st, name=f"{st.name}_layer{layer}",
            q=_randn_bits(rng, st.q.shape, st.dtype),
            k_pool=_randn_bits(rng, st.k_pool.shape, st.dtype),
            v_pool=_randn_bits(rng, st.v_pool.shape, st.dtype),
            k_new=_randn_bits(rng, st.k_new.shape, st.dtype),
            v_new=_randn_bits(rng, st.v_new.shape, st.dtype)))
    return out


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "decode_b32": decode_batch32,
    "long_context_decode": long_context_decode,
    "decode_b256": decode_batch256,
    "mixed_chunked_prefill": mixed_chunked_prefill,
}


def chunked_prompt_steps(rng: np.random.Generator, prompt_len: int, chunk: int, *,
                         dtype: str, block_size: int = 4, num_q_heads: int = 2,
                         num_kv_heads: int = 1, head_dim: int = 64,
                         num_blocks: int | None = None):
    """A prompt written into the pool whole, and the same prompt written in chunks.

    Returns ``(whole, chunks, k_tok, v_tok, q_tok)``.  ``whole`` is one
    PagedStep with the full prompt as one query span; ``chunks`` is a list of
    PagedSteps, chunk c carrying prompt tokens [c*chunk, (c+1)*chunk) as its
    query span over the prefix written by the earlier chunks.  All steps share
    one block table (the allocator's ids for the full prompt) and the same
    token values, so appending the chunks in order must leave the same pool
    as appending the whole prompt at once.
    """
    nb_total = blocks_needed(prompt_len, block_size)
    if num_blocks is None:
        num_blocks = nb_total + 3
    perm = rng.permutation(num_blocks).astype(np.int32)
    table = np.full((1, nb_total), -1, dtype=np.int32)
    table[0, :] = perm[:nb_total]
    q_tok = _randn_bits(rng, (prompt_len, num_q_heads, head_dim), dtype)
    k_tok = _randn_bits(rng, (prompt_len, num_kv_heads, head_dim), dtype)
    v_tok = _randn_bits(rng, (prompt_len, num_kv_heads, head_dim), dtype)
    empty = np.full((num_blocks, num_kv_heads, block_size, head_dim), NAN_BITS[dtype], np.uint16)

    def step(lo, hi, name):
        slots = np.array([int(table[0, p // block_size]) * block_size + p % block_size
                          for p in range(lo, hi)], dtype=np.int64)
        return PagedStep(name=name, dtype=dtype, num_q_heads=num_q_heads,
                         num_kv_heads=num_kv_heads, head_dim=head_dim,
                         block_size=block_size, scale=1.0 / math.sqrt(head_dim),
                         context_lens=np.array([hi], np.int32),
                         query_lens=np.array([hi - lo], np.int32),
                         query_start_loc=np.array([0, hi - lo], np.int32),
                         block_tables=table.copy(), num_blocks=num_blocks,
                         k_pool=empty.copy(), v_pool=empty.copy(),
                         q=q_tok[lo:hi].copy(), k_new=k_tok[lo:hi].copy(),
                         v_new=v_tok[lo:hi].copy(), slot_mapping=slots)

    whole = step(0, prompt_len, "whole_prompt")
    chunks = [step(lo, min(prompt_len, lo + chunk), f"chunk{c}")
              for c, lo in enumerate(range(0, prompt_len, chunk))]
    return whole, chunks, k_tok, v_tok, q_tok
