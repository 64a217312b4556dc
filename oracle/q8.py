"""8-bit (q8_0) KV cache: quantisation, dequantisation, append and paged
decode attention over a q8_0 pool -- TEST INFRASTRUCTURE ONLY.

The same rule holds as for the rest of this package: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and reference arm
may import it; the product path never does, and it imports nothing from the
product package.  Plain numpy.

What it follows: the video-shorts page's post on serving Gemma 4 26B A4B on
one 24 GB GPU with an 8-bit KV cache ("q8 kv cache"): llama.cpp's q8_0 cache
type for K and V stores the cache in 8 bits instead of 16 and dequantises it
on the fly in every attention step.  The pages name the format but do not
define it.  The reading taken here is the q8_0 block format:

* a block is 32 consecutive elements of one token's head row, so a 64-wide
  head row holds two blocks;
* the block's scale is d = max|x| / 127, computed in fp32 -- the precision in
  which a GPU quantiser takes the same decision, so that both sides pick the
  same integer codes -- and stored rounded to fp16 (nearest even, saturating
  at the largest finite fp16);
* each code is x * (1/d), both steps rounded to fp32, then rounded to the
  nearest integer with ties to even and clamped to [-127, 127]; an all-zero
  block has d = 0 and all codes 0;
* a code q stands for the value fp16(d) * q.

Attention over a q8_0 pool is the plain definition of the 16-bit oracle with
the dequantised K and V in place of the 16-bit ones: gather through the block
table, scores in fp64, softmax with the maximum subtracted, weighted sum of V.

Pool layout (a reading, chosen so that one (block, kv head) is one contiguous
chunk of codes and one of scales): codes int8 [num_blocks][Hkv][bs][D], scales
fp16 [num_blocks][Hkv][bs][D / 32].
"""
from __future__ import annotations

import numpy as np

QK = 32          # elements per q8_0 block
QMAX = 127       # largest code magnitude
F16_MAX = 65504.0


def quantize_q8_0(x):
    """Quantise rows x [..., D] (D a multiple of 32) to q8_0.

    Returns (codes int8 [..., D], scales float16 [..., D / 32]).  Follows the
    block format read from the video-shorts page's q8 KV-cache post (module
    docstring): fp32 scale and codes, ties to even, fp16 stored scale.
    """
    xf = np.asarray(x, dtype=np.float32)
    D = xf.shape[-1]
    if D % QK:
        raise ValueError("row length must be a multiple of 32")
    blk = xf.reshape(xf.shape[:-1] + (D // QK, QK))
    amax = np.max(np.abs(blk), axis=-1)                    # exact in fp32
    d = (amax / np.float32(QMAX)).astype(np.float32)       # fp32, nearest
    inv = np.zeros_like(d)
    nz = d > 0
    inv[nz] = np.float32(1.0) / d[nz]                      # fp32, nearest
    prod = (blk * inv[..., None]).astype(np.float32)       # fp32, nearest
    codes = np.clip(np.rint(prod), -QMAX, QMAX).astype(np.int8)  # ties to even
    scales = np.minimum(d, np.float32(F16_MAX)).astype(np.float16)
    return codes.reshape(xf.shape), scales


def dequantize_q8_0(codes, scales):
    """Values of q8_0 rows: codes int8 [..., D], scales fp16 [..., D / 32] ->
    float64 [..., D], each code times its block's stored fp16 scale (exact in
    fp64)."""
    c = np.asarray(codes, dtype=np.int8)
    D = c.shape[-1]
    blk = c.reshape(c.shape[:-1] + (D // QK, QK)).astype(np.float64)
    out = blk * np.asarray(scales, dtype=np.float16).astype(np.float64)[..., None]
    return out.reshape(c.shape)


def append_q8_0(k, v, slot_mapping, k_codes, k_scales, v_codes, v_scales):
    """Quantise each new token's K and V rows [T, Hkv, D] and write them into
    the q8_0 pools at slot // bs, slot % bs (every kv head); a negative slot
    marks padding and is skipped.  The KV-append step of the paged cache
    (Inference Engineering Day 11 short, "How does vLLM work"), with the
    8-bit cache of the video-shorts page's q8 post.  Pools are updated in place."""
    bs = k_codes.shape[2]
    kc, ks = quantize_q8_0(k)
    vc, vs = quantize_q8_0(v)
    for t, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        b, o = divmod(int(slot), bs)
        k_codes[b, :, o, :] = kc[t]
        k_scales[b, :, o, :] = ks[t]
        v_codes[b, :, o, :] = vc[t]
        v_scales[b, :, o, :] = vs[t]


def paged_decode_q8_0(q, k_codes, k_scales, v_codes, v_scales, block_tables, context_lens,
                      scale):
    """Decode attention over a q8_0 pool, in fp64.

    q: float values [S, Hq, D]; query head j reads kv head j // (Hq / Hkv).
    Sequence s attends to its positions 0..L_s-1, position p at block
    block_tables[s][p // bs], offset p % bs (nanoserve project page, "What I
    built": the paged KV cache and the decode that walks each sequence's block
    table with online softmax -- evaluated here directly, which online
    softmax reformulates exactly).  A sequence with L = 0 gives zeros.
    """
    q = np.asarray(q, dtype=np.float64)
    S, Hq, D = q.shape
    Hkv, bs = k_codes.shape[1], k_codes.shape[2]
    G = Hq // Hkv
    out = np.zeros((S, Hq, D))
    for s in range(S):
        L = int(context_lens[s])
        if L <= 0:
            continue
        pos = np.arange(L)
        blk = np.asarray(block_tables[s])[pos // bs]
        off = pos % bs
        for h in range(Hkv):
            K = dequantize_q8_0(k_codes[blk, h, off], k_scales[blk, h, off])   # [L, D]
            V = dequantize_q8_0(v_codes[blk, h, off], v_scales[blk, h, off])
            for j in range(h * G, (h + 1) * G):
                z = scale * (K @ q[s, j])
                w = np.exp(z - z.max())
                out[s, j] = (w / w.sum()) @ V
    return out
