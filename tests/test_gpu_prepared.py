"""GPU: a prepared call (arguments checked and marshalled once) runs the same
kernels as the direct call: the same output bits and pool bits, on the
current stream or a given one, and the oracle's result."""
import numpy as np
import pytest
import torch

import _gpu
from _gpu import DevStep, compare
from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_prepared_fused_decode_equals_direct(orc):
    st = wl.decode_batch32()
    ref, kp, vp = orc.step(st)
    d = DevStep(st)
    direct = d.fused().clone()
    pool = _gpu.to_bits(d.k_pool)
    d2 = DevStep(st)
    pc = nb.prepare(nb.ns_kv_append_paged_attn_decode, d2.q, d2.k_new, d2.v_new, d2.slot_mapping,
                    d2.k_pool, d2.v_pool, d2.block_tables, d2.context_lens, st.scale, d2.out, d2.ws)
    s = torch.cuda.Stream()
    for stream in (None, s):
        d2.out.fill_(float("nan"))
        pc(stream)
        torch.cuda.synchronize()
        assert torch.equal(d2.out, direct)
    assert np.array_equal(_gpu.to_bits(d2.k_pool), pool)
    compare(d2.out, ref, st.dtype, "prepared")
    _gpu.assert_no_device_status()


def test_prepared_mixed_prefill_equals_direct(orc):
    st = wl.mixed_chunked_prefill()
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = DevStep(st, k_pool=kp, v_pool=vp)
    direct = d.prefill().clone()
    pc = nb.prepare(nb.ns_paged_attn_prefill, d.q, d.query_start_loc, d.k_pool, d.v_pool,
                    d.block_tables, d.context_lens, st.scale, d.out, d.ws)
    d.out.fill_(float("nan"))
    pc()
    torch.cuda.synchronize()
    assert torch.equal(d.out, direct)
    compare(d.out, ref, st.dtype, "prepared prefill")
    _gpu.assert_no_device_status()
