"""Pins for the q8_0 (8-bit KV cache) oracle in ``oracle/q8.py``.

Each pin ties the oracle to something other than itself: closed forms of the
block format (an exact grid, an all-zero block, the block maximum's code,
ties, a scale that fp16 must round, worked out by hand), the rounding error
bound of any quantiser of that format, brute-force contiguous attention over
the dequantised values, and invariants the pages fix (block-id permutation,
a one-token context returns its V).  ``test_each_planted_mistake_fails_a_pin``
plants plausible mistakes in copies of the oracle and checks that every one is
caught.
"""
from __future__ import annotations

import math
import os
import types

import numpy as np
import pytest

from oracle import q8
from tests._pins import contiguous_attention

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "q8.py")


def independent_dequant(codes, scales):
    """codes int8 [..., D] x their block's fp16 scale, blocks of 32 (np.repeat)."""
    return codes.astype(np.float64) * np.repeat(scales.astype(np.float64), 32, axis=-1)


# ---------------------------------------------------------------------------
# format pins
# ---------------------------------------------------------------------------

def pin_exact_grid(m):
    """x = c * k with c a power of two and each block's max |k| = 127: the
    scale is c, the codes are k and dequantisation gives x back exactly."""
    rng = np.random.default_rng(11)
    c = 2.0 ** -5
    k = rng.integers(-127, 128, size=(6, 64))
    k[:, 3] = 127
    k[:, 40] = -127
    codes, scales = m.quantize_q8_0((c * k).astype(np.float32))
    assert scales.shape == (6, 2) and scales.dtype == np.float16
    assert codes.dtype == np.int8 and np.array_equal(codes.astype(np.int64), k)
    assert np.all(scales.astype(np.float64) == c)
    assert np.array_equal(m.dequantize_q8_0(codes, scales), c * k)


def pin_zero_block(m):
    """An all-zero block has scale 0 and codes 0; the other block is untouched by it."""
    x = np.zeros((1, 64), np.float32)
    x[0, 32:] = np.linspace(-1.0, 2.0, 32, dtype=np.float32)
    codes, scales = m.quantize_q8_0(x)
    assert scales[0, 0] == 0 and not np.any(codes[0, :32])
    assert scales[0, 1] > 0 and codes[0, 63] == 127
    assert not np.any(m.dequantize_q8_0(codes, scales)[0, :32])


def pin_block_max_code(m):
    """The element of largest magnitude in a block gets code +-127 with its sign."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((20, 64)).astype(np.float32)
    codes, _ = m.quantize_q8_0(x)
    for r in range(20):
        for b in range(2):
            blk = x[r, 32 * b:32 * b + 32]
            i = int(np.argmax(np.abs(blk)))
            assert int(codes[r, 32 * b + i]) == (127 if blk[i] > 0 else -127)


def pin_ties_to_even(m):
    """With max |x| = 127 the scale is 1, so x * (1/d) = x; halves round to even."""
    x = np.zeros((1, 64), np.float32)
    x[0, :8] = [127, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5]
    x[0, 32] = -127
    codes, scales = m.quantize_q8_0(x)
    assert np.all(scales.astype(np.float64) == 1.0)
    assert codes[0, :8].tolist() == [127, 0, 2, 2, 0, -2, -2, 4]


def pin_fp16_scale(m):
    """max |x| = 1: d = 1/127 = 0.0078740157..., between 2^-7 and 2^-6 where
    fp16 steps by 2^-17, so the stored scale is round(1032.06) / 2^17 =
    0.00787353515625 and the code 127 stands for 127 * that = 0.99993896484375."""
    x = np.zeros((1, 64), np.float32)
    x[0, 0] = 1.0
    x[0, 32] = -1.0
    codes, scales = m.quantize_q8_0(x)
    assert scales[0, 0].astype(np.float64) == 0.00787353515625
    assert codes[0, 0] == 127 and codes[0, 32] == -127
    deq = m.dequantize_q8_0(codes, scales)
    assert deq[0, 0] == 0.99993896484375 and deq[0, 32] == -0.99993896484375


def pin_error_bound(m):
    """|x - fp16(d) q| <= d (1/2 + 1e-4) + 127 |d - fp16(d)| per element, d the
    block's max |x| / 127 (the rounding bound of the format)."""
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((64, 64)) * rng.uniform(0.01, 100.0, size=(64, 1))).astype(np.float32)
    codes, scales = m.quantize_q8_0(x)
    deq = m.dequantize_q8_0(codes, scales)
    for b in range(2):
        blk = x[:, 32 * b:32 * b + 32].astype(np.float64)
        d = np.abs(blk).max(axis=1) / 127.0
        d16 = scales[:, b].astype(np.float64)
        bound = d * (0.5 + 1e-4) + 127.0 * np.abs(d - d16)
        err = np.abs(blk - deq[:, 32 * b:32 * b + 32]).max(axis=1)
        assert np.all(err <= bound), (err - bound).max()


def pin_append_scatter(m):
    """Each token's quantised rows land at slot // bs, slot % bs for every kv
    head; a negative slot is skipped; every other slot keeps its sentinel."""
    rng = np.random.default_rng(14)
    nb, hkv, bs, d = 4, 2, 4, 64
    kc = np.full((nb, hkv, bs, d), 99, np.int8)
    vc = np.full((nb, hkv, bs, d), 99, np.int8)
    ks = np.full((nb, hkv, bs, 2), 7.0, np.float16)
    vs = np.full((nb, hkv, bs, 2), 7.0, np.float16)
    slots = np.array([3, -1, 12, 0, 9], np.int64)
    k = rng.standard_normal((5, hkv, d)).astype(np.float32)
    v = rng.standard_normal((5, hkv, d)).astype(np.float32)
    m.append_q8_0(k, v, slots, kc, ks, vc, vs)
    want_kc, want_ks = m.quantize_q8_0(k)
    want_vc, want_vs = m.quantize_q8_0(v)
    written = set()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        b, o = divmod(int(s), bs)
        written.add((b, o))
        assert np.array_equal(kc[b, :, o], want_kc[t]) and np.array_equal(ks[b, :, o], want_ks[t])
        assert np.array_equal(vc[b, :, o], want_vc[t]) and np.array_equal(vs[b, :, o], want_vs[t])
    for b in range(nb):
        for o in range(bs):
            if (b, o) not in written:
                assert np.all(kc[b, :, o] == 99) and np.all(vc[b, :, o] == 99)
                assert np.all(ks[b, :, o] == 7.0) and np.all(vs[b, :, o] == 7.0)


# ---------------------------------------------------------------------------
# attention pins
# ---------------------------------------------------------------------------

def make_case(m, lens, seed, hq=4, hkv=2, bs=4):
    """A paged q8_0 case: random K/V per sequence appended through slots into
    pools of garbage codes and scales at permuted block ids."""
    rng = np.random.default_rng(seed)
    d = 64
    nbs = [(L + bs - 1) // bs for L in lens]
    nblocks = sum(nbs) + 3
    perm = rng.permutation(nblocks)
    tables = np.full((len(lens), max(1, max(nbs))), -1, np.int32)
    off = 0
    for s, n in enumerate(nbs):
        tables[s, :n] = perm[off:off + n]
        off += n
    kc = rng.integers(-127, 128, size=(nblocks, hkv, bs, d)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(nblocks, hkv, bs, d)).astype(np.int8)
    ks = rng.uniform(0.0, 1.0, size=(nblocks, hkv, bs, 2)).astype(np.float16)
    vs = rng.uniform(0.0, 1.0, size=(nblocks, hkv, bs, 2)).astype(np.float16)
    Ks, Vs, slots = [], [], []
    for s, L in enumerate(lens):
        Ks.append(rng.standard_normal((L, hkv, d)).astype(np.float32))
        Vs.append(rng.standard_normal((L, hkv, d)).astype(np.float32))
        slots += [int(tables[s, p // bs]) * bs + p % bs for p in range(L)]
    if slots:
        m.append_q8_0(np.concatenate(Ks), np.concatenate(Vs), np.array(slots, np.int64),
                      kc, ks, vc, vs)
    q = rng.standard_normal((len(lens), hq, d)).astype(np.float16).astype(np.float64)
    return dict(q=q, kc=kc, ks=ks, vc=vc, vs=vs, tables=tables, lens=np.array(lens, np.int32),
                Ks=Ks, Vs=Vs, scale=1.0 / math.sqrt(d), bs=bs)


def run(m, c):
    return m.paged_decode_q8_0(c["q"], c["kc"], c["ks"], c["vc"], c["vs"], c["tables"],
                               c["lens"], c["scale"])


def pin_brute_force_decode(m):
    """Paged q8_0 decode = brute-force attention on the contiguous dequantised K/V."""
    c = make_case(m, [1, 5, 17, 33], seed=15)
    out = run(m, c)
    for s, L in enumerate(c["lens"]):
        Kq = independent_dequant(*q8.quantize_q8_0(c["Ks"][s]))
        Vq = independent_dequant(*q8.quantize_q8_0(c["Vs"][s]))
        want = contiguous_attention(c["q"][s][None], Kq, Vq, c["scale"], [int(L) - 1])[0]
        assert np.abs(out[s] - want).max() <= 1e-12


def pin_block_permutation(m):
    """Relabelling the physical block ids (moving the pools with them) changes
    no output bit."""
    c = make_case(m, [7, 16, 29], seed=16)
    base = run(m, c)
    nb = c["kc"].shape[0]
    pi = np.random.default_rng(17).permutation(nb)
    moved = dict(c)
    for key in ("kc", "ks", "vc", "vs"):
        arr = np.empty_like(c[key])
        arr[pi] = c[key]
        moved[key] = arr
    moved["tables"] = np.where(c["tables"] >= 0, pi[np.maximum(c["tables"], 0)], -1).astype(np.int32)
    assert np.array_equal(run(m, moved), base)


def pin_context_one(m):
    """A one-token context returns that token's dequantised V exactly."""
    c = make_case(m, [1, 1], seed=18)
    out = run(m, c)
    hq, hkv = out.shape[1], c["Vs"][0].shape[1]
    for s in range(2):
        v = independent_dequant(*q8.quantize_q8_0(c["Vs"][s][0]))   # [Hkv, D]
        for j in range(hq):
            assert np.array_equal(out[s, j], v[j // (hq // hkv)])


PINS = [pin_exact_grid, pin_zero_block, pin_block_max_code, pin_ties_to_even, pin_fp16_scale,
        pin_error_bound, pin_append_scatter, pin_brute_force_decode, pin_block_permutation,
        pin_context_one]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_meets_pin(pin):
    pin(q8)


# ---------------------------------------------------------------------------
# planted mistakes
# ---------------------------------------------------------------------------

MUTANTS = {
    "scale over 128": ("amax / np.float32(QMAX)", "amax / np.float32(128)"),
    "one block per row": ("QK = 32 ", "QK = 64 "),
    "truncating codes": ("np.rint(prod)", "np.trunc(prod)"),
    "ties rounded up": ("np.rint(prod)", "np.floor(prod + np.float32(0.5))"),
    "dropped softmax scale": ("z = scale * (K @ q[s, j])", "z = (K @ q[s, j])"),
    "softmax sign": ("w = np.exp(z - z.max())", "w = np.exp(z.max() - z)"),
    "interleaved GQA groups": ("for j in range(h * G, (h + 1) * G):", "for j in range(h, Hq, Hkv):"),
    "block and offset swapped": ("blk = np.asarray(block_tables[s])[pos // bs]\n        off = pos % bs",
                                 "blk = np.asarray(block_tables[s])[pos % bs]\n        off = pos // bs"),
    "one position short": ("pos = np.arange(L)", "pos = np.arange(L - 1)"),
    "append offset swapped": ("b, o = divmod(int(slot), bs)", "o, b = divmod(int(slot), bs)"),
    "slot 0 taken as padding": ("if slot < 0:", "if slot <= 0:"),
    "K codes into V": ("v_codes[b, :, o, :] = vc[t]", "v_codes[b, :, o, :] = kc[t]"),
    "signed maximum for the scale": ("amax = np.max(np.abs(blk), axis=-1)", "amax = np.max(blk, axis=-1)"),
    "block scales swapped": ("np.asarray(scales, dtype=np.float16).astype(np.float64)[..., None]",
                             "np.asarray(scales, dtype=np.float16).astype(np.float64)[..., ::-1, None]"),
    "V read from the K pool": ("V = dequantize_q8_0(v_codes[blk, h, off], v_scales[blk, h, off])",
                               "V = dequantize_q8_0(k_codes[blk, h, off], k_scales[blk, h, off])"),
}


def load_variant(src_text):
    mod = types.ModuleType("q8_variant")
    exec(compile(src_text, "q8_variant", "exec"), mod.__dict__)
    return mod


def failing(mod):
    bad = []
    for pin in PINS:
        try:
            pin(mod)
        except Exception:  # noqa: BLE001 - any failure of a pin counts
            bad.append(pin.__name__)
    return bad


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_each_planted_mistake_fails_a_pin(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    assert failing(load_variant(src.replace(old, new))), f"mutant '{name}' passes every pin"


def test_unmodified_copy_fails_no_pin():
    assert failing(load_variant(open(SRC).read())) == []
