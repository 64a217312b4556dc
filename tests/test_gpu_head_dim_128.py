"""GPU parity at head_dim 128 (the decode kernel generalised beyond the
Qwen2.5-0.5B geometry of the pages' model: nanoserve project page, "What I
built", the fused paged-attention decode).

At head_dim 128 a token row spans 16 lanes and a ring step holds 16 tokens;
the decode, its fused append, the forced split policies and the chunked
prefill (whose spans take the split-KV walk) are compared with the fp64
oracle, which is generic in head_dim, within the 16-bit tolerance.
"""
import numpy as np
import pytest
import torch

import _gpu
from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CASES = [(4, 1, wl.BF16), (8, 1, wl.F16), (14, 2, wl.BF16), (16, 2, wl.F16)]


def _step(hq, hkv, dtype, seed, n=48, median=600.0, sigma=1.0, max_len=4096, query_lens=None):
    rng = np.random.default_rng(seed)
    lens = wl.lognormal_lengths(rng, n, median, sigma, max_len)
    ql = np.ones(n, np.int32) if query_lens is None else query_lens
    return wl.make_step(rng, lens, ql, dtype=dtype, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                        name=f"d128_{hq}_{hkv}_{dtype}")


@pytest.mark.parametrize("hq,hkv,dtype", CASES)
def test_d128_fused_append_decode_matches_oracle(hq, hkv, dtype, orc):
    st = _step(hq, hkv, dtype, 5100 + hq)
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = _gpu.DevStep(st)
    out = d.fused()
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    _gpu.compare(out, ref, st.dtype, st.name)
    assert np.array_equal(_gpu.to_bits(d.k_pool), kp)
    assert np.array_equal(_gpu.to_bits(d.v_pool), vp)


@pytest.mark.parametrize("hq,hkv,dtype", CASES[:2])
@pytest.mark.parametrize("cfg", [dict(whole_sequences=1), dict(num_ctas=3), dict(min_blocks_per_cta=1)])
def test_d128_append_then_decode_under_forced_policies(hq, hkv, dtype, cfg, orc):
    st = _step(hq, hkv, dtype, 5200 + hq, n=12, median=900.0)
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = _gpu.DevStep(st)
    d.append()
    out = d.decode(config=_gpu.config(**cfg))
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    _gpu.compare(out, ref, st.dtype, f"{st.name} {cfg}")
    assert np.array_equal(_gpu.to_bits(d.k_pool), kp)


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_d128_chunked_prefill_matches_oracle(dtype, orc):
    rng = np.random.default_rng(5300)
    lens = np.array([1, 60, 300, 1000, 17], np.int32)
    qlen = np.array([1, 24, 100, 64, 17], np.int32)
    st = wl.make_step(rng, lens, qlen, dtype=dtype, num_q_heads=8, num_kv_heads=2, head_dim=128,
                      name="d128_prefill")
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = _gpu.DevStep(st)
    d.append()
    out = d.prefill()
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    _gpu.compare(out, ref, st.dtype, "d128 prefill")


def test_d128_rejects_other_block_sizes():
    rng = np.random.default_rng(5400)
    st = wl.make_step(rng, np.array([5, 9], np.int32), np.ones(2, np.int32), dtype=wl.F16,
                      num_q_heads=4, num_kv_heads=1, head_dim=128, block_size=8)
    d = _gpu.DevStep(st)
    with pytest.raises(nb.NsError) as e:
        d.decode()
    assert e.value.status == -2


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (8, 1), (4, 1)])
def test_d128_tensor_core_spans(dtype, hq, hkv, orc):
    """Spans of 2+ rows on the tcgen05 kernel at head_dim 128 (64-key tiles,
    two 64-element regions a row): ragged prefixes, query tiles cut mid-span,
    key tiles cut mid-block, NaN in unused pool slots."""
    rng = np.random.default_rng(5500 + hq + hkv)
    lens = np.array([2, 30, 150, 129, 400, 700], np.int32)
    qlens = np.array([2, 30, 19, 128, 37, 300], np.int32)
    st = wl.make_step(rng, lens, qlens, dtype=dtype, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                      poison_unused=True, name="d128_tc")
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = _gpu.DevStep(st)
    d.append()
    out = d.prefill()
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    _gpu.compare(out, ref, st.dtype, f"d128 tc Hq={hq} Hkv={hkv}")


def test_d128_tensor_core_and_walk_agree(orc):
    rng = np.random.default_rng(5600)
    lens = np.array([1, 512 + 1500, 17, 512 + 900], np.int32)
    qlens = np.array([1, 512, 1, 512], np.int32)
    st = wl.make_step(rng, lens, qlens, dtype=wl.BF16, num_q_heads=8, num_kv_heads=2, head_dim=128,
                      name="d128_mixed")
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = _gpu.DevStep(st, k_pool=kp, v_pool=vp)
    outs = []
    for min_span in (-1, 2):
        cfg = nb.PrefillConfig()
        cfg.tensor_core_min_span = min_span
        nb.ns_paged_attn_prefill(d.q, d.query_start_loc, d.k_pool, d.v_pool, d.block_tables,
                                 d.context_lens, st.scale, d.out, d.ws, config=cfg)
        torch.cuda.synchronize()
        outs.append(d.out.clone())
    _gpu.compare(outs[0], ref, st.dtype, "d128 walk")
    _gpu.compare(outs[1], ref, st.dtype, "d128 tensor cores")
    _gpu.assert_no_device_status()
