"""The bounded-wait failure path of the split-KV decode.

Every wait inside the kernels has a time limit; when it runs out the kernel
sets NS_DEV_WAIT_TIMEOUT, stops issuing copies, waits for its own copies in
flight and returns, so that the context stays usable (failure detection: a
GPU wait that gives up and reports, never a trap or a hang).  The
test shortens the limit of the computing warps' waits for their next K/V
step (ns_decode_config.wait_limit_ns) below a copy's latency, so the wait
runs out on a real workload with nothing faulting, and checks that the call
returns, that the status bit is set, and that after the workspace is zeroed
again the next call with the default limit matches the oracle.
"""
import numpy as np
import pytest
import torch

import _gpu
from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

NS_DEV_WAIT_TIMEOUT = 0x8


def _zero(ws):
    st = nb.lib().ns_paged_attn_workspace_init(ws.data_ptr(), ws.numel(),
                                               torch.cuda.current_stream().cuda_stream)
    assert st == 0


@pytest.mark.parametrize("name", ["decode_b32", "decode_b256"])
def test_short_wait_limit_times_out_and_next_call_is_clean(name, orc):
    st = wl.WORKLOADS[name]()
    ref, kp, vp = orc.step(st, num_threads=max(1, orc.max_threads()))
    d = _gpu.DevStep(st)
    _gpu.assert_no_device_status()
    cfg = nb.DecodeConfig()
    cfg.wait_limit_ns = 200  # far below the ~1 us latency of a K/V copy
    for _ in range(2):
        _zero(d.ws)
        nb.ns_kv_append_paged_attn_decode(d.q, d.k_new, d.v_new, d.slot_mapping, d.k_pool, d.v_pool,
                                          d.block_tables, d.context_lens, st.scale, d.out, d.ws,
                                          config=cfg)
        torch.cuda.synchronize()  # the call returned: nothing waits past its limit
        bits = nb.ns_get_device_status(clear=True)
        assert bits & NS_DEV_WAIT_TIMEOUT, f"status 0x{bits:x}"
        assert not bits & ~NS_DEV_WAIT_TIMEOUT, f"unexpected status bits 0x{bits:x}"
    # a timed-out call may leave arrival counters behind: zero the workspace
    _zero(d.ws)
    out = d.fused()
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    _gpu.compare(out, ref, st.dtype, name)
    assert np.array_equal(_gpu.to_bits(d.k_pool), kp)
    assert np.array_equal(_gpu.to_bits(d.v_pool), vp)


def test_negative_wait_limit_is_rejected():
    st = wl.tiny_decode()
    d = _gpu.DevStep(st)
    cfg = nb.DecodeConfig()
    cfg.wait_limit_ns = -1
    with pytest.raises(nb.NsError) as e:
        d.decode(config=cfg)
    assert e.value.status == -1
