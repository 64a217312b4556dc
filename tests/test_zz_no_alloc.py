"""The allocation-free decode entry point, ns_paged_attn_decode_noalloc.

Some callers cannot allocate device memory: plugins that live inside a host
runtime which owns every device allocation, and serving loops that must not
allocate once they are running.  For them the library runs the split-KV
decode over scratch memory that is part of the library image instead of a
caller-provided workspace.  This file checks, through the C ABI, that two
calls in a row give the same bits as ns_paged_attn_decode with a workspace
(both run the same kernel on the same grid) and match the fp64 oracle within
the tolerance of the other parity tests.  It is collected last so that a
failure here cannot hide another test's result.
"""
import numpy as np
import pytest
import torch

import _gpu
from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _check_two_calls(st, d, ref):
    d.append()
    want = d.decode().clone()
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(d.q, float("nan"))
        nb.ns_paged_attn_decode_noalloc(d.q, d.k_pool, d.v_pool, d.block_tables, d.context_lens,
                                        st.scale, out)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), want.view(torch.int16))
        _gpu.compare(out, ref, st.dtype, st.name)
    _gpu.assert_no_device_status()


# all three workloads cut sequences across workers, so the scratch partial
# records and arrival counters are exercised
@pytest.mark.parametrize("name", ["decode_b32", "long_context_decode", "decode_b256"])
def test_noalloc_matches_workspace_entry_point_and_oracle(name, orc):
    st = wl.WORKLOADS[name]()
    ref, _, _ = orc.step(st, num_threads=max(1, orc.max_threads()))
    _check_two_calls(st, _gpu.DevStep(st), ref)


def test_noalloc_at_its_pair_limit(orc):
    """Exactly NS_NOALLOC_MAX_PAIRS (sequence, kv head) pairs: the last arrival
    counter of the scratch array is used and cleared."""
    S = nb.NS_NOALLOC_MAX_PAIRS // 2  # 2 kv heads per sequence
    rng = np.random.default_rng(4242)
    lens = rng.integers(1, 48, size=S).astype(np.int32)
    st = wl.make_step(rng, lens, np.ones(S, np.int32), dtype=wl.F16, name="noalloc_cap")
    ref, _, _ = orc.step(st, num_threads=max(1, orc.max_threads()))
    _check_two_calls(st, _gpu.DevStep(st), ref)


def test_noalloc_rejects_more_pairs_than_its_scratch_holds():
    S = nb.NS_NOALLOC_MAX_PAIRS // 2 + 1          # 2 kv heads per sequence
    q = torch.zeros(S, 14, 64, dtype=torch.float16, device="cuda")
    pool = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device="cuda")
    tables = torch.zeros(S, 1, dtype=torch.int32, device="cuda")
    lens = torch.ones(S, dtype=torch.int32, device="cuda")
    with pytest.raises(nb.NsError) as e:
        nb.ns_paged_attn_decode_noalloc(q, pool, pool, tables, lens, 0.125, torch.empty_like(q))
    assert e.value.status == -2


@pytest.mark.parametrize("scale", [float("inf"), float("-inf"), float("nan")])
def test_noalloc_rejects_a_scale_that_is_not_finite(scale):
    st = wl.tiny_decode()
    d = _gpu.DevStep(st)
    with pytest.raises(nb.NsError) as e:
        nb.ns_paged_attn_decode_noalloc(d.q, d.k_pool, d.v_pool, d.block_tables, d.context_lens,
                                        scale, d.out)
    assert e.value.status == -1
