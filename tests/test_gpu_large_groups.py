"""GPU parity for GQA groups of more than 8 query heads per kv head (the decode
generalised beyond the Qwen2.5-0.5B geometry: nanoserve project page, "What I
built", the fused paged-attention decode).

A group of G > 8 heads runs as n = ceil(G / 8) groups of G / n heads over the
same kv head; the pools, the fused append and the output are those of the
plain group, so the fp64 oracle (generic in the group) checks them directly.
"""
import numpy as np
import pytest
import torch

import _gpu
from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

# (q heads, kv heads, dtype): groups of 16 (2 x 8), 12 (2 x 6), 32 (4 x 8), 10 (2 x 5)
CASES = [(32, 2, wl.BF16), (12, 1, wl.F16), (32, 1, wl.F16), (20, 2, wl.BF16)]


def _step(hq, hkv, dtype, seed, n=40, median=700.0, query_lens=None):
    rng = np.random.default_rng(seed)
    lens = wl.lognormal_lengths(rng, n, median, 1.0, 4096)
    ql = np.ones(n, np.int32) if query_lens is None else query_lens
    return wl.make_step(rng, lens, ql, dtype=dtype, num_q_heads=hq, num_kv_heads=hkv,
                        name=f"group_{hq // hkv}_{dtype}")


@pytest.mark.parametrize("hq,hkv,dtype", CASES)
def test_large_group_fused_append_decode_matches_oracle(hq, hkv, dtype, orc):
    st = _step(hq, hkv, dtype, 6100 + hq)
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = _gpu.DevStep(st)
    out = d.fused()
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    _gpu.compare(out, ref, st.dtype, st.name)
    # the new token is stored once, bit-exact
    assert np.array_equal(_gpu.to_bits(d.k_pool), kp)
    assert np.array_equal(_gpu.to_bits(d.v_pool), vp)


@pytest.mark.parametrize("cfg", [dict(whole_sequences=1), dict(num_ctas=3), dict(min_blocks_per_cta=1)])
def test_large_group_under_forced_policies(cfg, orc):
    st = _step(32, 2, wl.F16, 6200, n=12, median=900.0)
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = _gpu.DevStep(st)
    d.append()
    out = d.decode(config=_gpu.config(**cfg))
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    _gpu.compare(out, ref, st.dtype, f"{st.name} {cfg}")


def test_large_group_prefill_takes_the_walk(orc):
    rng = np.random.default_rng(6300)
    lens = np.array([1, 60, 300, 17], np.int32)
    qlen = np.array([1, 24, 100, 17], np.int32)
    st = wl.make_step(rng, lens, qlen, dtype=wl.F16, num_q_heads=16, num_kv_heads=1, name="group_prefill")
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = _gpu.DevStep(st)
    d.append()
    out = d.prefill()
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    _gpu.compare(out, ref, st.dtype, "group 16 prefill")


def test_uneven_large_group_is_rejected():
    rng = np.random.default_rng(6400)
    st = wl.make_step(rng, np.array([5, 9], np.int32), np.ones(2, np.int32), dtype=wl.F16,
                      num_q_heads=9, num_kv_heads=1)
    d = _gpu.DevStep(st)
    with pytest.raises(nb.NsError) as e:
        d.decode()
    assert e.value.status == -2
