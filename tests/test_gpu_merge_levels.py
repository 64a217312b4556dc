"""GPU parity of the two-level merge: a pair cut into many pieces first combines
its pieces inside each CTA (counted in shared memory), then the CTA records
are merged.  Both merges must give the oracle's result for every grid."""
import numpy as np
import pytest
import torch

import _gpu
from _gpu import DevStep, compare, config
from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def long_ctx(orc):
    st = wl.long_context_decode()
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    return st, ref, kp, vp


def _expected_levels(st, levels, plan):
    if levels:
        return levels
    pairs = st.num_seqs * st.num_kv_heads
    warps = plan["ctas_launched"] * 8
    return 2 if pairs * 32 <= warps and pairs * st.max_blocks_per_seq >= warps else 1


@pytest.mark.parametrize("levels", [0, 1, 2])
@pytest.mark.parametrize("cfg", [dict(), dict(num_ctas=5), dict(num_ctas=3, min_blocks_per_cta=1),
                                 dict(num_ctas=nb.NS_MAX_CTAS, min_blocks_per_cta=1)],
                         ids=lambda c: ",".join(f"{k}={v}" for k, v in c.items()) or "auto")
def test_long_context_merge_levels(levels, cfg, long_ctx):
    """8 sequences of 4096 tokens (16 pairs): every grid and merge depth
    matches the oracle, and the plan names the merge the kernel ran."""
    st, ref, kp, vp = long_ctx
    d = DevStep(st, k_pool=kp, v_pool=vp)
    c = config(**cfg)
    c.merge_levels = levels
    out = d.decode(c)
    torch.cuda.synchronize()
    compare(out, ref, st.dtype, f"levels={levels} {cfg}")
    plan = nb.ns_read_decode_plan(d.ws)
    assert plan["merge_levels"] == _expected_levels(st, levels, plan)
    if not cfg:
        # the default grid cuts each pair into more than 16 pieces
        assert plan["split_pairs"] == 16 and plan["max_pieces"] >= 16
    _gpu.assert_no_device_status()


def test_auto_two_level_on_long_context(long_ctx):
    """The automatic choice for this shape is the two-level merge, and a
    second call on the same workspace (counters reset) gives the same bits."""
    st, ref, kp, vp = long_ctx
    d = DevStep(st, k_pool=kp, v_pool=vp)
    first = d.decode().clone()
    again = d.decode()
    torch.cuda.synchronize()
    assert torch.equal(first, again)
    compare(again, ref, st.dtype)
    assert nb.ns_read_decode_plan(d.ws)["merge_levels"] == 2
    _gpu.assert_no_device_status()


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
@pytest.mark.parametrize("hq,hkv", [(2, 2), (8, 2), (14, 2), (16, 2)])
def test_two_level_groups(hq, hkv, dtype, orc):
    """Forced two-level merges at group sizes 1, 4, 7 and 8, with a ragged
    mix of lengths so that CTA boundaries fall inside pairs and some pairs
    stay below the two-level piece count."""
    rng = np.random.default_rng(31 + hq)
    lens = np.array([3000, 17, 1500, 2049, 1, 700], np.int32)
    st = wl.make_step(rng, lens, np.ones(len(lens), np.int32), dtype=dtype, num_q_heads=hq,
                      num_kv_heads=hkv, block_size=16)
    ref, kp, vp = orc.step(st)
    d = DevStep(st, k_pool=kp, v_pool=vp)
    c = config(min_blocks_per_cta=1)
    c.merge_levels = 2
    out = d.decode(c)
    torch.cuda.synchronize()
    compare(out, ref, st.dtype, f"G={hq // hkv} {dtype}")
    plan = nb.ns_read_decode_plan(d.ws)
    assert plan["merge_levels"] == 2 and plan["max_pieces"] >= 16
    _gpu.assert_no_device_status()


def test_merge_levels_out_of_range_refused():
    st = wl.tiny_decode()
    d = DevStep(st)
    c = config()
    c.merge_levels = 3
    with pytest.raises(nb.NsError):
        d.decode(c)


def test_long_context_through_prefill_two_level(long_ctx):
    """The same rows as single-token spans of a prefill call: the span walk
    takes the automatic split and the two-level merge, and matches the
    oracle."""
    st, ref, kp, vp = long_ctx
    d = DevStep(st, k_pool=kp, v_pool=vp)
    out = d.prefill()
    torch.cuda.synchronize()
    compare(out, ref, st.dtype, "prefill rows")
    plan = nb.ns_read_decode_plan(d.ws)
    assert plan["merge_levels"] == 2 and plan["max_pieces"] >= 16
    assert plan["workers_active"] == plan["ctas_launched"] * 8
    _gpu.assert_no_device_status()
