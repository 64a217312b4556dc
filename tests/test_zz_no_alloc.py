"""The allocation-free decode entry point, ns_paged_attn_decode_noalloc.

Some callers cannot allocate device memory: code that runs while a CUDA graph
is being captured (an allocation cannot be captured), plugins that live inside
a host runtime which owns every device allocation, and serving loops that must
not allocate once they are running.  For them the library runs the split-KV
decode over scratch memory that is part of the library image instead of a
caller-provided workspace.  This file checks, through the C ABI, that two
calls in a row give the same result as ns_paged_attn_decode with a workspace,
within the tolerance of the other parity tests.  It is collected last so that
a failure here cannot hide another test's result.
"""
import numpy as np
import pytest
import torch

import _gpu
from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _close(got, want):
    g, w = _gpu.to_f64(got), _gpu.to_f64(want)
    max_abs = float(np.abs(g - w).max())
    rel = float(np.linalg.norm(g - w) / max(np.linalg.norm(w), 1e-30))
    assert max_abs <= _gpu.MAX_ABS and rel <= _gpu.REL_L2, (max_abs, rel)


# both workloads cut sequences across CTAs, so the scratch partial records
# and arrival counters are exercised
@pytest.mark.parametrize("name", ["decode_b32", "long_context_decode", "decode_b256"])
def test_noalloc_matches_workspace_entry_point(name):
    st = wl.WORKLOADS[name]()
    d = _gpu.DevStep(st)
    d.append()
    want = d.decode().clone()
    for _ in range(2):
        out = torch.full_like(d.q, float("nan"))
        nb.ns_paged_attn_decode_noalloc(d.q, d.k_pool, d.v_pool, d.block_tables, d.context_lens,
                                        st.scale, out)
        torch.cuda.synchronize()
        _close(out, want)
    _gpu.assert_no_device_status()


def test_noalloc_rejects_more_pairs_than_its_scratch_holds():
    S = nb.NS_NOALLOC_MAX_PAIRS // 2 + 1          # 2 kv heads per sequence
    q = torch.zeros(S, 14, 64, dtype=torch.float16, device="cuda")
    pool = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device="cuda")
    tables = torch.zeros(S, 1, dtype=torch.int32, device="cuda")
    lens = torch.ones(S, dtype=torch.int32, device="cuda")
    with pytest.raises(nb.NsError) as e:
        nb.ns_paged_attn_decode_noalloc(q, pool, pool, tables, lens, 0.125, torch.empty_like(q))
    assert e.value.status == -2
