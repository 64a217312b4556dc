"""GPU parity of the append and the split-KV decode against the fp64 oracle."""
import numpy as np
import pytest
import torch

import _gpu
from _gpu import DevStep, compare, config
from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DECODE_WORKLOADS = ["tiny_decode", "decode_b32", "long_context_decode", "decode_b256"]


@pytest.fixture(scope="module")
def steps():
    return {}


def _get(steps, name, orc):
    if name not in steps:
        st = wl.WORKLOADS[name]()
        ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
        steps[name] = (st, ref, kp, vp)
    return steps[name]


@pytest.mark.parametrize("name", DECODE_WORKLOADS + ["mixed_chunked_prefill"])
def test_append_bit_exact(name, orc, steps):
    st, ref, kp, vp = _get(steps, name, orc)
    d = DevStep(st)
    d.append()
    torch.cuda.synchronize()
    assert np.array_equal(_gpu.to_bits(d.k_pool), kp)
    assert np.array_equal(_gpu.to_bits(d.v_pool), vp)
    _gpu.assert_no_device_status()


def test_append_skips_negative_and_flags_out_of_pool(orc):
    st = wl.tiny_decode()
    sm = st.slot_mapping.copy()
    sm[1] = -1
    sm[2] = st.num_blocks * st.block_size + 5  # beyond the pool
    kp, vp = orc.kv_append(st.k_pool, st.v_pool, st.k_new, st.v_new,
                           np.where(sm >= st.num_blocks * st.block_size, -1, sm), st.block_size)
    d = DevStep(st)
    d.slot_mapping = _gpu.dev_ints(sm, np.int64)
    d.append()
    torch.cuda.synchronize()
    assert np.array_equal(_gpu.to_bits(d.k_pool), kp)
    assert np.array_equal(_gpu.to_bits(d.v_pool), vp)
    assert nb.ns_get_device_status(clear=True) == 0x4


@pytest.mark.parametrize("name", DECODE_WORKLOADS)
def test_decode_matches_oracle(name, orc, steps):
    st, ref, kp, vp = _get(steps, name, orc)
    d = DevStep(st, k_pool=kp, v_pool=vp)
    out = d.decode()
    torch.cuda.synchronize()
    compare(out, ref, st.dtype, name)
    _gpu.assert_no_device_status()


@pytest.mark.parametrize("name", DECODE_WORKLOADS)
def test_fused_append_decode_matches_oracle(name, orc, steps):
    st, ref, kp, vp = _get(steps, name, orc)
    d = DevStep(st)
    out = d.fused()
    torch.cuda.synchronize()
    compare(out, ref, st.dtype, name + " fused")
    assert np.array_equal(_gpu.to_bits(d.k_pool), kp)
    assert np.array_equal(_gpu.to_bits(d.v_pool), vp)
    _gpu.assert_no_device_status()


@pytest.mark.parametrize("cfg", [dict(num_ctas=1), dict(num_ctas=2), dict(num_ctas=3),
                                 dict(num_ctas=7), dict(num_ctas=nb.NS_MAX_CTAS, min_blocks_per_cta=1),
                                 dict(min_blocks_per_cta=1), dict(whole_sequences=1),
                                 dict(num_ctas=5, whole_sequences=1)],
                         ids=lambda c: ",".join(f"{k}={v}" for k, v in c.items()))
@pytest.mark.parametrize("name", ["decode_b32", "long_context_decode", "tiny_decode"])
def test_forced_split_policies_agree(name, cfg, orc, steps):
    """Every split of the KV walk gives the oracle's result; the plan record
    shows that the split really happened (or did not, for whole sequences)."""
    st, ref, kp, vp = _get(steps, name, orc)
    d = DevStep(st, k_pool=kp, v_pool=vp)
    out = d.decode(config(**cfg))
    torch.cuda.synchronize()
    compare(out, ref, st.dtype, f"{name} {cfg}")
    plan = nb.ns_read_decode_plan(d.ws)
    total = sum(wl.blocks_needed(L, st.block_size) for L in st.context_lens) * st.num_kv_heads
    assert plan["total_blocks"] == total
    if cfg.get("whole_sequences"):
        assert plan["whole_sequences"] == 1 and plan["split_pairs"] == 0
    else:
        assert plan["whole_sequences"] == 0
        if plan["workers_active"] == 1:
            assert plan["split_pairs"] == 0
        # a worker is one warp: never more than the launched grid holds
        assert 1 <= plan["workers_active"] <= 12 * plan["ctas_launched"]
        if name == "long_context_decode" and plan["workers_active"] > 16:
            # 16 pairs of 256 blocks over more workers than pairs: every pair is cut
            assert plan["split_pairs"] == 16 and plan["max_pieces"] >= plan["workers_active"] // 16
    _gpu.assert_no_device_status()


def test_repeated_calls_reuse_workspace(orc, steps):
    """Split merges leave the workspace counters at zero for the next call."""
    st, ref, kp, vp = _get(steps, "long_context_decode", orc)
    d = DevStep(st, k_pool=kp, v_pool=vp)
    first = d.decode().clone()
    for _ in range(3):
        again = d.decode()
    torch.cuda.synchronize()
    assert torch.equal(first, again)
    compare(again, ref, st.dtype)
    _gpu.assert_no_device_status()
