"""Pins for the fp64 oracle: checks that tie it to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` handle and raises
AssertionError when the oracle disagrees with
  * a library routine (numpy's float16 decoding, the float32 bit layout of
    bf16, torch's fp64 scaled_dot_product_attention),
  * an independent brute-force implementation on contiguous (unpaged) data,
  * an invariant the pages fix (block-id permutation, chunked versus whole
    writes with 8-token chunks into 4-token blocks, context length 1 returns V,
    constant V returns that constant).
They are small so that ``tests/test_oracle_mutants.py`` can run the whole set
against every mistake it plants in a copy of the oracle.
"""
from __future__ import annotations

import math

import numpy as np

from paged_kv_decode_ns_gb300 import workloads as wl


# ---------------------------------------------------------------------------
# independent helpers (numpy only)
# ---------------------------------------------------------------------------

def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Decode raw fp16 / bf16 bit patterns with library views."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == wl.F16:
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def contiguous_attention(qf, Kf, Vf, scale, positions):
    """Brute-force attention on contiguous K/V of one sequence.

    qf [R, Hq, D], Kf/Vf [L, Hkv, D]; query row r sees keys 0..positions[r].
    Query heads map to KV heads by repeating each KV head Hq/Hkv times
    (np.repeat), the grouped-query convention.
    """
    R, Hq, D = qf.shape
    Hkv = Kf.shape[1]
    Kr = np.repeat(Kf, Hq // Hkv, axis=1)   # [L, Hq, D]
    Vr = np.repeat(Vf, Hq // Hkv, axis=1)
    out = np.zeros((R, Hq, D))
    for r in range(R):
        n = positions[r] + 1
        if n <= 0:
            continue
        z = np.einsum("jd,pjd->jp", qf[r], Kr[:n]) * scale
        z = z - z.max(axis=1, keepdims=True)
        w = np.exp(z)
        w /= w.sum(axis=1, keepdims=True)
        out[r] = np.einsum("jp,pjd->jd", w, Vr[:n])
    return out


def make_tiny(rng, lens, qlens, *, hq=4, hkv=2, d=16, bs=4, dtype=wl.F16, spare=3,
              garbage=True):
    """Random paged case built by scattering contiguous per-sequence K/V.

    Returns a dict with the paged inputs and, per sequence, the contiguous
    K/V values they were scattered from.
    """
    lens = [int(x) for x in lens]
    qlens = [int(x) for x in qlens]
    nbs = [wl.blocks_needed(L, bs) for L in lens]
    nblocks = sum(nbs) + spare
    mbps = max(1, max(nbs))
    perm = rng.permutation(nblocks)
    bt = np.full((len(lens), mbps), -1, np.int32)
    off = 0
    for s, n in enumerate(nbs):
        bt[s, :n] = perm[off:off + n]
        off += n
    rand = lambda shape: wl.float_to_bits(rng.standard_normal(shape).astype(np.float32), dtype)
    kp = rand((nblocks, hkv, bs, d)) if garbage else np.zeros((nblocks, hkv, bs, d), np.uint16)
    vp = rand((nblocks, hkv, bs, d)) if garbage else np.zeros((nblocks, hkv, bs, d), np.uint16)
    Ks, Vs = [], []
    for s, L in enumerate(lens):
        K = rand((L, hkv, d))
        V = rand((L, hkv, d))
        for p in range(L):
            kp[bt[s, p // bs], :, p % bs, :] = K[p]
            vp[bt[s, p // bs], :, p % bs, :] = V[p]
        Ks.append(K)
        Vs.append(V)
    T = sum(qlens)
    q = rand((T, hq, d))
    qsl = np.zeros(len(lens) + 1, np.int32)
    qsl[1:] = np.cumsum(qlens)
    return dict(dtype=dtype, q=q, k_pool=kp, v_pool=vp, block_tables=bt,
                context_lens=np.array(lens, np.int32), query_start_loc=qsl,
                qlens=qlens, Ks=Ks, Vs=Vs, hq=hq, hkv=hkv, d=d, bs=bs,
                scale=1.0 / math.sqrt(d))


def run_case(orc, c, decode=None):
    decode = all(x == 1 for x in c["qlens"]) if decode is None else decode
    return orc.paged_attention(c["dtype"], c["q"], c["k_pool"], c["v_pool"], c["block_tables"],
                               c["context_lens"], c["scale"],
                               query_start_loc=None if decode else c["query_start_loc"])


def brute_case(c):
    out = []
    for s, L in enumerate(c["context_lens"]):
        lo, hi = c["query_start_loc"][s], c["query_start_loc"][s + 1]
        qf = bits_to_f64(c["q"][lo:hi], c["dtype"])
        pos = [int(L) - (hi - lo) + i for i in range(hi - lo)]
        out.append(contiguous_attention(qf, bits_to_f64(c["Ks"][s], c["dtype"]),
                                        bits_to_f64(c["Vs"][s], c["dtype"]), c["scale"], pos))
    return np.concatenate(out, axis=0)


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_f16_decoder(orc):
    """Every binary16 bit pattern decodes as numpy's float16 does."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_double(int(b)) for b in bits[::7]])
    r = ref[::7]
    same = (got == r) | (np.isnan(got) & np.isnan(r))
    assert same.all(), f"f16 decode differs at {bits[::7][~same][:5]}"


def pin_bf16_decoder(orc):
    """Every bf16 bit pattern decodes as the upper half of a float32."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = np.array([orc.bf16_to_double(int(b)) for b in bits[::7]])
    r = ref[::7]
    same = (got == r) | (np.isnan(got) & np.isnan(r))
    assert same.all(), f"bf16 decode differs at {bits[::7][~same][:5]}"


def pin_append_scatter(orc):
    """kv_append equals a numpy fancy-index scatter; slot < 0 is skipped and
    untouched slots keep their sentinel."""
    rng = np.random.default_rng(7)
    nb, hkv, bs, d, T = 6, 3, 4, 8, 11
    kp = np.full((nb, hkv, bs, d), 0xABCD, np.uint16)
    vp = np.full((nb, hkv, bs, d), 0x1234, np.uint16)
    k = rng.integers(0, 1 << 16, (T, hkv, d), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, (T, hkv, d), dtype=np.uint16)
    slots = rng.choice(np.arange(1, nb * bs), T, replace=False).astype(np.int64)
    slots[5] = 0
    slots[3] = -1
    slots[8] = -7
    ko, vo = orc.kv_append(kp, vp, k, v, slots, bs)
    kr, vr = kp.copy(), vp.copy()
    keep = slots >= 0
    fk = kr.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d)
    fv = vr.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d)
    fk[slots[keep]] = k[keep]
    fv[slots[keep]] = v[keep]
    kr = fk.reshape(nb, bs, hkv, d).transpose(0, 2, 1, 3)
    vr = fv.reshape(nb, bs, hkv, d).transpose(0, 2, 1, 3)
    assert np.array_equal(ko, kr) and np.array_equal(vo, vr)


def pin_brute_force_decode(orc):
    """Decode through random block tables equals contiguous brute force (fp16 and bf16)."""
    for dtype, seed in ((wl.F16, 11), (wl.BF16, 12)):
        rng = np.random.default_rng(seed)
        c = make_tiny(rng, [1, 5, 9, 13], [1, 1, 1, 1], hq=6, hkv=2, d=16, bs=4, dtype=dtype)
        got = run_case(orc, c)
        ref = brute_case(c)
        assert np.max(np.abs(got - ref)) < 1e-12, np.max(np.abs(got - ref))


def pin_brute_force_prefill(orc):
    """Query spans (cached prefix + causal chunk) equal contiguous brute force."""
    rng = np.random.default_rng(13)
    c = make_tiny(rng, [7, 12, 3], [3, 5, 1], hq=4, hkv=1, d=8, bs=4)
    got = run_case(orc, c)
    ref = brute_case(c)
    assert np.max(np.abs(got - ref)) < 1e-12, np.max(np.abs(got - ref))


def pin_torch_sdpa(orc):
    """A prefill span equals torch's fp64 scaled_dot_product_attention with a
    prefix+causal mask (GQA via repeat_interleave)."""
    import torch
    rng = np.random.default_rng(17)
    L, qlen, hq, hkv, d = 19, 6, 6, 3, 16
    c = make_tiny(rng, [L], [qlen], hq=hq, hkv=hkv, d=d, bs=4)
    got = run_case(orc, c, decode=False)
    q = torch.from_numpy(bits_to_f64(c["q"], c["dtype"])).permute(1, 0, 2)[None]
    k = torch.from_numpy(bits_to_f64(c["Ks"][0], c["dtype"])).permute(1, 0, 2)
    v = torch.from_numpy(bits_to_f64(c["Vs"][0], c["dtype"])).permute(1, 0, 2)
    k = k.repeat_interleave(hq // hkv, dim=0)[None]
    v = v.repeat_interleave(hq // hkv, dim=0)[None]
    pos = torch.arange(L - qlen, L)[:, None]
    mask = torch.arange(L)[None, :] <= pos
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                           scale=c["scale"])
    ref = ref[0].permute(1, 0, 2).numpy()
    assert np.max(np.abs(got - ref)) < 1e-12, np.max(np.abs(got - ref))


def pin_sdpa_causal_empty_prefix(orc):
    """A chunk over an empty prefix is plain causal attention (is_causal=True)."""
    import torch
    rng = np.random.default_rng(19)
    c = make_tiny(rng, [10], [10], hq=2, hkv=2, d=8, bs=4)
    got = run_case(orc, c, decode=False)
    q = torch.from_numpy(bits_to_f64(c["q"], c["dtype"])).permute(1, 0, 2)[None]
    k = torch.from_numpy(bits_to_f64(c["Ks"][0], c["dtype"])).permute(1, 0, 2)[None]
    v = torch.from_numpy(bits_to_f64(c["Vs"][0], c["dtype"])).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                           scale=c["scale"])
    ref = ref[0].permute(1, 0, 2).numpy()
    assert np.max(np.abs(got - ref)) < 1e-12


def pin_block_permutation(orc):
    """Relabelling physical block ids (moving the pool contents with them)
    leaves the output bit-identical."""
    rng = np.random.default_rng(23)
    c = make_tiny(rng, [3, 8, 14], [1, 1, 1], hq=4, hkv=2, d=8, bs=4, spare=5)
    a = run_case(orc, c)
    nb = c["k_pool"].shape[0]
    pi = rng.permutation(nb)
    kp = np.empty_like(c["k_pool"])
    vp = np.empty_like(c["v_pool"])
    kp[pi] = c["k_pool"]
    vp[pi] = c["v_pool"]
    bt = np.where(c["block_tables"] >= 0, pi[np.maximum(c["block_tables"], 0)], -1).astype(np.int32)
    c2 = dict(c, k_pool=kp, v_pool=vp, block_tables=bt)
    b = run_case(orc, c2)
    assert np.array_equal(a, b)


def pin_context_one_returns_v(orc):
    """A sequence of one token returns that token's V exactly, for every head."""
    for dtype in (wl.F16, wl.BF16):
        rng = np.random.default_rng(29)
        c = make_tiny(rng, [1, 1, 6], [1, 1, 1], hq=4, hkv=2, d=8, bs=4, dtype=dtype)
        got = run_case(orc, c)
        for s in range(2):
            v = bits_to_f64(c["Vs"][s][0], dtype)            # [Hkv, D]
            assert np.array_equal(got[s], np.repeat(v, 2, axis=0))


def pin_constant_v(orc):
    """If every V row is the same vector c, the output is c (to 1e-15)."""
    rng = np.random.default_rng(31)
    c = make_tiny(rng, [5, 9, 16], [1, 1, 1], hq=4, hkv=2, d=8, bs=4)
    vec = wl.float_to_bits(rng.standard_normal((2, 8)).astype(np.float32), c["dtype"])
    c["v_pool"][:] = vec[None, :, None, :]
    got = run_case(orc, c)
    want = np.repeat(bits_to_f64(vec, c["dtype"]), 2, axis=0)
    for s in range(3):
        assert np.max(np.abs(got[s] - want)) <= 1e-15 * max(1.0, np.abs(want).max())


def _read_golden(name):
    import os
    vals = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                vals[line[0]] = [int(x) for x in line[1:]]
    return vals


GOLDEN_BLOCKS = _read_golden("chunked_prefill_blocks.txt")


def pin_chunked_vs_whole(orc):
    """A 16-token prompt appended in 8-token chunks into 4-token blocks leaves the
    same pool and the same outputs as appending it whole; 2 then 4 blocks are
    occupied after the first and second chunk."""
    rng = np.random.default_rng(37)
    chunk = GOLDEN_BLOCKS["chunk_tokens"][0]
    bs = GOLDEN_BLOCKS["block_size"][0]
    whole, chunks, *_ = wl.chunked_prompt_steps(rng, 2 * chunk, chunk, dtype=wl.F16, block_size=bs,
                                                num_q_heads=2, num_kv_heads=1, head_dim=8)
    kw, vw = orc.kv_append(whole.k_pool, whole.v_pool, whole.k_new, whole.v_new,
                           whole.slot_mapping, bs)
    ow = orc.paged_attention(wl.F16, whole.q, kw, vw, whole.block_tables, whole.context_lens,
                             whole.scale, query_start_loc=whole.query_start_loc)
    kc, vc = chunks[0].k_pool, chunks[0].v_pool
    outs, occupied = [], []
    nan = wl.NAN_BITS[wl.F16]
    for st in chunks:
        kc, vc = orc.kv_append(kc, vc, st.k_new, st.v_new, st.slot_mapping, bs)
        occupied.append(int(np.sum(np.any(kc != nan, axis=(1, 2, 3)))))
        outs.append(orc.paged_attention(wl.F16, st.q, kc, vc, st.block_tables, st.context_lens,
                                        st.scale, query_start_loc=st.query_start_loc))
    assert occupied == GOLDEN_BLOCKS["blocks_occupied_after_chunk"], occupied
    assert np.array_equal(kc, kw) and np.array_equal(vc, vw)
    assert np.array_equal(np.concatenate(outs), ow)


def pin_prefill_last_row_is_decode(orc):
    """The last row of a prefill span equals a decode step of the same sequence."""
    rng = np.random.default_rng(41)
    c = make_tiny(rng, [11], [4], hq=4, hkv=2, d=8, bs=4)
    pre = run_case(orc, c, decode=False)
    dec = orc.paged_attention(c["dtype"], c["q"][-1:], c["k_pool"], c["v_pool"],
                              c["block_tables"], c["context_lens"], c["scale"])
    assert np.array_equal(pre[-1], dec[0])


PINS = [pin_f16_decoder, pin_bf16_decoder, pin_append_scatter, pin_brute_force_decode,
        pin_brute_force_prefill, pin_torch_sdpa, pin_sdpa_causal_empty_prefix,
        pin_block_permutation, pin_context_one_returns_v, pin_constant_v,
        pin_chunked_vs_whole, pin_prefill_last_row_is_decode]


def failing_pins(orc):
    """Names of the pins ``orc`` fails (an exception counts as a failure)."""
    bad = []
    for pin in PINS:
        try:
            pin(orc)
        except Exception:  # noqa: BLE001 - any failure of a pin counts
            bad.append(pin.__name__)
    return bad
