"""The seeded input generator: shapes, the allocator's bounded waste, the
pages' chunked-prefill block counts, determinism."""
import numpy as np
import pytest

from paged_kv_decode_ns_gb300 import workloads as wl


def _live_slots(st):
    """Set of (block, offset) slots holding a token of some sequence."""
    out = set()
    for s in range(st.num_seqs):
        for p in range(int(st.context_lens[s])):
            out.add((int(st.block_tables[s, p // st.block_size]), p % st.block_size))
    return out


@pytest.mark.parametrize("name", ["tiny_decode", "decode_b32", "long_context_decode",
                                  "mixed_chunked_prefill"])
def test_shapes_and_waste(name):
    st = wl.WORKLOADS[name]()
    S, bs = st.num_seqs, st.block_size
    assert st.q.shape == (st.num_tokens, 14, 64)
    assert st.k_pool.shape == (st.num_blocks, 2, bs, 64) == st.v_pool.shape
    assert st.k_new.shape == (st.num_tokens, 2, 64)
    used = st.block_tables[st.block_tables >= 0]
    # every block belongs to at most one sequence
    assert len(np.unique(used)) == used.size
    assert used.max() < st.num_blocks
    for s in range(S):
        L = int(st.context_lens[s])
        n = wl.blocks_needed(L, bs)
        assert np.all(st.block_tables[s, :n] >= 0) and np.all(st.block_tables[s, n:] == -1)
        # wasted slots stay below one block per sequence
        assert 0 <= n * bs - L < bs
    # each new token's slot is the slot of its position in its own table
    assert len(set(st.slot_mapping.tolist())) == st.num_tokens
    assert set((int(x) // bs, int(x) % bs) for x in st.slot_mapping) <= _live_slots(st)


def test_tiny_decode_matches_its_description():
    st = wl.tiny_decode()
    assert st.context_lens.tolist() == [1, 17, 64, 200]
    assert st.num_blocks == 32 and st.dtype == wl.F16 and st.scale == 0.125
    assert (st.block_tables >= 0).sum() == 1 + 2 + 4 + 13


def test_lognormal_lengths_distribution():
    rng = np.random.default_rng(0)
    L = wl.lognormal_lengths(rng, 200000, 1024, 1.2, 8192)
    assert L.min() >= 1 and L.max() <= 8192
    assert abs(np.median(L) - 1024) / 1024 < 0.02
    # P(L <= x) = Phi((ln x - ln 1024) / 1.2) below the clip
    from math import erf, log, sqrt
    for x in (64, 256, 4096):
        want = 0.5 * (1 + erf((log(x + 0.5) - log(1024)) / (1.2 * sqrt(2))))
        assert abs(np.mean(L <= x) - want) < 0.005, x
    # the clip at 8192 holds the whole upper tail
    want_tail = 0.5 * (1 - erf((log(8191.5) - log(1024)) / (1.2 * sqrt(2))))
    assert abs(np.mean(L == 8192) - want_tail) < 0.005


def test_mixed_step_spans():
    st = wl.mixed_chunked_prefill()
    assert st.num_seqs == 18
    assert st.query_lens.tolist() == [1] * 16 + [512, 512]
    assert st.context_lens[16:].tolist() == [2012, 3512]
    assert st.num_tokens == 16 + 1024
    assert st.query_start_loc[-1] == st.num_tokens


def test_deterministic():
    a, b = wl.decode_batch32(), wl.decode_batch32()
    for f in ("context_lens", "block_tables", "q", "k_pool", "v_pool", "slot_mapping"):
        assert np.array_equal(getattr(a, f), getattr(b, f))


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 3.0e38], np.float32)
    bits = wl.float_to_bits(x, wl.BF16)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    # 1+2^-8 is a tie between 1 and 1+2^-7: even mantissa (1.0) wins;
    # 1+3*2^-8 ties between 1+2^-7 and 1+2^-6: even (1+2^-6) wins.
    assert back.tolist()[:4] == [1.0, 1.0, 1.0 + 2**-6, -2.5]


def test_poisoned_pool_keeps_live_tokens():
    st = wl.tiny_decode(poison_unused=True)
    live = _live_slots(st)
    new = set((int(x) // 16, int(x) % 16) for x in st.slot_mapping)
    nan = wl.NAN_BITS[wl.F16]
    for b in range(st.num_blocks):
        for o in range(16):
            is_nan = bool(np.all(st.k_pool[b, :, o, :] == nan))
            assert is_nan == (((b, o) not in live) or ((b, o) in new))


def test_chunked_prompt_golden_block_counts():
    """Inference Engineering Day 12 short, "What is chunked prefill within vLLM":
    8-token chunks into 4-token blocks occupy 2, then 4 blocks."""
    import _pins
    g = _pins.GOLDEN_BLOCKS
    rng = np.random.default_rng(2)
    chunk, bs = g["chunk_tokens"][0], g["block_size"][0]
    whole, chunks, *_ = wl.chunked_prompt_steps(rng, 2 * chunk, chunk, dtype=wl.F16,
                                                block_size=bs)
    seen = set()
    counts = []
    for st in chunks:
        seen |= set(int(x) // bs for x in st.slot_mapping)
        counts.append(len(seen))
    assert counts == g["blocks_occupied_after_chunk"]
