"""GPU parity of chunked-prefill attention over query spans."""
import numpy as np
import pytest
import torch

import _gpu
from _gpu import DevStep, compare
from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_mixed_chunked_prefill_step(orc):
    """16 decode rows + two 512-token chunks over 1500 / 3000 cached tokens."""
    st = wl.mixed_chunked_prefill()
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = DevStep(st)
    d.append()
    out = d.prefill()
    torch.cuda.synchronize()
    assert np.array_equal(_gpu.to_bits(d.k_pool), kp)
    compare(out, ref, st.dtype, "mixed step")
    _gpu.assert_no_device_status()


def test_mixed_step_walk_keeps_default_blocks_per_worker(orc):
    """Beside tensor-core spans, the single-token rows' walk keeps the default
    8 blocks a worker (no finer automatic cut) on a grid of one CTA per
    (span, kv head) pair. Its workers fill the fewest CTAs, and the 4096-token
    row is cut into at most 34 pieces. The output still matches the oracle."""
    st = wl.mixed_chunked_prefill()
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = DevStep(st, k_pool=kp, v_pool=vp)
    out = d.prefill()
    torch.cuda.synchronize()
    compare(out, ref, st.dtype, "mixed step")
    _gpu.assert_no_device_status()
    plan = nb.ns_read_decode_plan(d.ws)
    dec = st.query_lens == 1
    nblocks = -(-st.context_lens[dec].astype(np.int64) // st.block_size)
    assert plan["total_blocks"] == st.num_kv_heads * nblocks.sum()
    virtual = st.num_kv_heads * (nblocks + 4).sum()  # 4 virtual blocks of split cost a pair
    workers = -(-virtual // 8)
    assert plan["whole_sequences"] == 0 and plan["workers_active"] == workers
    assert plan["ctas_active"] == -(-workers // 8)
    assert 2 <= plan["max_pieces"] <= -(-(nblocks.max() + 4) // 8) + 1
    # its grid: one CTA per (span, kv head) pair at most
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan["ctas_launched"] == min(sms, st.num_seqs * st.num_kv_heads)


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
@pytest.mark.parametrize("bs", [4, 16])
def test_spans_with_ragged_prefixes(dtype, bs, orc):
    rng = np.random.default_rng(bs)
    lens = np.array([1, 9, 40, 130, 77, 300], np.int32)
    qlens = np.array([1, 9, 13, 1, 64, 33], np.int32)
    st = wl.make_step(rng, lens, qlens, dtype=dtype, block_size=bs)
    ref, kp, vp = orc.step(st)
    d = DevStep(st)
    d.append()
    out = d.prefill()
    torch.cuda.synchronize()
    compare(out, ref, dtype, f"spans bs={bs}")
    _gpu.assert_no_device_status()


def test_chunked_writes_equal_whole_prompt(orc):
    """The chunked-prefill worked example (8-token chunks, 4-token blocks):
    appending the prompt chunk by chunk leaves the same pool as appending it
    whole, and each chunk's attention matches the oracle."""
    rng = np.random.default_rng(21)
    whole, chunks, *_ = wl.chunked_prompt_steps(rng, 64, 8, dtype=wl.F16, block_size=4,
                                                num_q_heads=14, num_kv_heads=2)
    dw = DevStep(whole)
    dw.append()
    ow = dw.prefill().clone()
    dc = DevStep(chunks[0])
    outs = []
    for st in chunks:
        dc.st = st
        dc.q = _gpu.to_dev(st.q, st.dtype)
        dc.k_new = _gpu.to_dev(st.k_new, st.dtype)
        dc.v_new = _gpu.to_dev(st.v_new, st.dtype)
        dc.slot_mapping = _gpu.dev_ints(st.slot_mapping, np.int64)
        dc.context_lens = _gpu.dev_ints(st.context_lens, np.int32)
        dc.query_start_loc = _gpu.dev_ints(st.query_start_loc, np.int32)
        dc.out = torch.empty_like(dc.q)
        dc.append()
        outs.append(dc.prefill().clone())
    torch.cuda.synchronize()
    # bit patterns (the never-written slots hold NaN, which == does not match)
    assert np.array_equal(_gpu.to_bits(dc.k_pool), _gpu.to_bits(dw.k_pool))
    assert np.array_equal(_gpu.to_bits(dc.v_pool), _gpu.to_bits(dw.v_pool))
    ref, *_ = orc.step(whole)
    compare(torch.cat(outs), ref, wl.F16, "chunked")
    compare(ow, ref, wl.F16, "whole")
    _gpu.assert_no_device_status()


def test_single_row_spans_equal_decode(orc):
    st = wl.decode_batch32()
    ref, kp, vp = orc.step(st)
    d = DevStep(st, k_pool=kp, v_pool=vp)
    a = d.decode().clone()
    b = d.prefill()
    torch.cuda.synchronize()
    compare(a, ref, st.dtype)
    compare(b, ref, st.dtype)


def test_bad_span_is_flagged():
    rng = np.random.default_rng(5)
    st = wl.make_step(rng, np.array([10, 10], np.int32), np.array([3, 2], np.int32),
                      dtype=wl.F16)
    d = DevStep(st)
    d.context_lens = _gpu.dev_ints(np.array([2, 10], np.int32), np.int32)  # span longer than context
    d.prefill()
    torch.cuda.synchronize()
    assert nb.ns_get_device_status(clear=True) & 0x20


def _prefill_cfg(min_span):
    c = nb.PrefillConfig()
    c.tensor_core_min_span = min_span
    return c


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("hq,hkv", [(14, 2), (8, 1), (4, 2), (2, 2), (16, 2)])
def test_tensor_core_spans(dtype, bs, hq, hkv, orc):
    """Spans of 2+ rows on the tcgen05 kernel: ragged prefixes, query tiles
    cut mid-span, key tiles cut mid-block, both element types."""
    rng = np.random.default_rng(100 + bs + hq)
    lens = np.array([2, 30, 150, 129, 400, 700], np.int32)
    qlens = np.array([2, 30, 19, 128, 37, 300], np.int32)
    st = wl.make_step(rng, lens, qlens, dtype=dtype, block_size=bs, num_q_heads=hq,
                      num_kv_heads=hkv, poison_unused=True)
    ref, kp, vp = orc.step(st)
    d = DevStep(st)
    d.append()
    out = d.prefill()
    torch.cuda.synchronize()
    compare(out, ref, dtype, f"tc bs={bs} Hq={hq} Hkv={hkv}")
    _gpu.assert_no_device_status()


def test_tensor_core_and_cuda_core_paths_agree(orc):
    st = wl.mixed_chunked_prefill()
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = DevStep(st, k_pool=kp, v_pool=vp)
    nb.ns_paged_attn_prefill(d.q, d.query_start_loc, d.k_pool, d.v_pool, d.block_tables,
                             d.context_lens, st.scale, d.out, d.ws, config=_prefill_cfg(-1))
    cuda_core = d.out.clone()
    nb.ns_paged_attn_prefill(d.q, d.query_start_loc, d.k_pool, d.v_pool, d.block_tables,
                             d.context_lens, st.scale, d.out, d.ws, config=_prefill_cfg(2))
    torch.cuda.synchronize()
    compare(cuda_core, ref, st.dtype, "cuda-core path")
    compare(d.out, ref, st.dtype, "tensor-core path")
    _gpu.assert_no_device_status()


@pytest.mark.parametrize("min_span", [5, 40])
def test_raised_tensor_core_threshold_partitions_the_rows(min_span, orc):
    """With tensor_core_min_span raised, spans below it are the walk's alone and
    spans at or above it the tensor-core kernel's alone: each phase run by
    itself leaves the other's rows untouched (still NaN), and both together
    match the oracle."""
    rng = np.random.default_rng(700 + min_span)
    lens = np.array([1, 3, 60, 5, 300, 45, 4], np.int32)
    qlens = np.array([1, 3, 40, 5, 100, 39, 2], np.int32)
    st = wl.make_step(rng, lens, qlens, dtype=wl.F16, poison_unused=True)
    ref, kp, vp = orc.step(st)
    d = DevStep(st, k_pool=kp, v_pool=vp)
    span_of_row = np.repeat(np.arange(len(qlens)), qlens)
    tc_rows = torch.from_numpy(qlens[span_of_row] >= min_span).to(d.out.device)
    for phase, mine in ((nb.NS_PREFILL_TENSOR_CORE, tc_rows), (nb.NS_PREFILL_WALK, ~tc_rows)):
        d.out.fill_(float("nan"))
        cfg = _prefill_cfg(min_span)
        cfg.phases = phase
        nb.ns_paged_attn_prefill(d.q, d.query_start_loc, d.k_pool, d.v_pool, d.block_tables,
                                 d.context_lens, st.scale, d.out, d.ws, config=cfg)
        torch.cuda.synchronize()
        written = ~torch.isnan(d.out.float()).flatten(1).any(dim=1)
        assert torch.equal(written, mine), f"phase {phase}: rows written {written.tolist()}"
    nb.ns_paged_attn_prefill(d.q, d.query_start_loc, d.k_pool, d.v_pool, d.block_tables,
                             d.context_lens, st.scale, d.out, d.ws, config=_prefill_cfg(min_span))
    torch.cuda.synchronize()
    compare(d.out, ref, st.dtype, f"min_span {min_span}")
    _gpu.assert_no_device_status()


def test_no_more_tokens_than_spans_all_on_the_walk(orc):
    """With as many query tokens as spans (one empty span, one of two tokens)
    every row takes the split-KV walk, the two-token span too: the output
    matches the oracle."""
    rng = np.random.default_rng(77)
    lens = np.array([7, 40, 20, 130, 3], np.int32)
    qlens = np.array([0, 2, 1, 1, 1], np.int32)
    st = wl.make_step(rng, lens, qlens, dtype=wl.F16, poison_unused=True)
    ref, kp, vp = orc.step(st)
    d = DevStep(st, k_pool=kp, v_pool=vp)
    out = d.prefill()
    torch.cuda.synchronize()
    compare(out, ref, st.dtype, "tokens <= spans")
    _gpu.assert_no_device_status()
