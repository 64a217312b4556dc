"""GPU parity of the q8_0 (8-bit) KV cache against its oracle (oracle/q8.py).

The video-shorts aggregator page's "q8 kv cache" post keeps K and V in
llama.cpp's q8_0 format and dequantises them in every attention step; the
block format read from it (32-element blocks, fp16 scale max|x|/127, codes
rounded to nearest even in fp32) is pinned in tests/test_oracle_q8.py.  Here
the CUDA path is compared with that oracle through the C ABI:
  * the append writes codes and scales bit for bit (plain and fused);
  * the decode over a q8_0 pool matches the oracle's fp64 attention over the
    dequantised pool within the 16-bit output tolerance of the other parity
    tests (max-abs 2e-3 beyond the output rounding, rel-L2 1e-3).
"""
import numpy as np
import pytest
import torch

import _gpu
from oracle import q8
from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def values(bits, dtype):
    """fp16 / bf16 bit patterns -> float32 values (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == wl.F16:
        return b.view(np.float16).astype(np.float32)
    return (b.astype(np.uint32) << 16).view(np.float32)


class Q8Step:
    """A decode step over a q8_0 pool: the 16-bit pool of `st` quantised, on the
    device, with the oracle's expected pools after the step's append."""

    def __init__(self, st):
        self.st = st
        kc, ks = q8.quantize_q8_0(values(st.k_pool, st.dtype))
        vc, vs = q8.quantize_q8_0(values(st.v_pool, st.dtype))
        self.pools0 = (kc, ks, vc, vs)
        self.want = [a.copy() for a in self.pools0]
        q8.append_q8_0(values(st.k_new, st.dtype), values(st.v_new, st.dtype), st.slot_mapping, *self.want)
        dev = "cuda"
        self.kc, self.ks, self.vc, self.vs = (torch.from_numpy(kc).to(dev), torch.from_numpy(ks).to(dev),
                                              torch.from_numpy(vc).to(dev), torch.from_numpy(vs).to(dev))
        self.d = _gpu.DevStep(st)

    def ref(self):
        st = self.st
        return q8.paged_decode_q8_0(values(st.q, st.dtype), *self.want, st.block_tables, st.context_lens,
                                    st.scale)

    def pools_equal(self):
        got = [t.cpu().numpy() for t in (self.kc, self.ks, self.vc, self.vs)]
        return all(np.array_equal(g.view(np.uint8) if g.dtype == np.int8 else g.view(np.uint16),
                                  w.view(np.uint8) if w.dtype == np.int8 else w.view(np.uint16))
                   for g, w in zip(got, self.want))


NAMES = ["tiny_decode", "decode_b32", "long_context_decode", "decode_b256"]


@pytest.mark.parametrize("name", NAMES)
def test_q8_append_is_bit_exact(name):
    s = Q8Step(wl.WORKLOADS[name]())
    d = s.d
    nb.ns_kv_append_q8_0(d.k_new, d.v_new, d.slot_mapping, s.kc, s.ks, s.vc, s.vs)
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    assert s.pools_equal()


@pytest.mark.parametrize("name", NAMES)
def test_q8_decode_matches_oracle(name):
    s = Q8Step(wl.WORKLOADS[name]())
    d = s.d
    nb.ns_kv_append_q8_0(d.k_new, d.v_new, d.slot_mapping, s.kc, s.ks, s.vc, s.vs)
    out = torch.full_like(d.q, float("nan"))
    nb.ns_paged_attn_decode_q8_0(d.q, s.kc, s.ks, s.vc, s.vs, d.block_tables, d.context_lens, s.st.scale,
                                 out, d.ws)
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    _gpu.compare(out, s.ref(), s.st.dtype, name)


@pytest.mark.parametrize("name", NAMES)
def test_q8_fused_append_decode_matches_oracle(name):
    s = Q8Step(wl.WORKLOADS[name]())
    d = s.d
    out = torch.full_like(d.q, float("nan"))
    nb.ns_kv_append_paged_attn_decode_q8_0(d.q, d.k_new, d.v_new, d.slot_mapping, s.kc, s.ks, s.vc, s.vs,
                                           d.block_tables, d.context_lens, s.st.scale, out, d.ws)
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    assert s.pools_equal()
    _gpu.compare(out, s.ref(), s.st.dtype, name)


def test_q8_context_one_returns_the_dequantised_value():
    """L = 1: the output is the new token's dequantised V, rounded once."""
    rng = np.random.default_rng(99)
    st = wl.make_step(rng, np.ones(6, np.int32), np.ones(6, np.int32), dtype=wl.BF16, name="q8_len1")
    s = Q8Step(st)
    d = s.d
    out = torch.empty_like(d.q)
    nb.ns_kv_append_paged_attn_decode_q8_0(d.q, d.k_new, d.v_new, d.slot_mapping, s.kc, s.ks, s.vc, s.vs,
                                           d.block_tables, d.context_lens, st.scale, out, d.ws)
    torch.cuda.synchronize()
    vc, vs = q8.quantize_q8_0(values(st.v_new, st.dtype))
    v = q8.dequantize_q8_0(vc, vs)                    # [S, Hkv, D]
    G = st.num_q_heads // st.num_kv_heads
    want = _gpu.round_to_dtype(np.repeat(v, G, axis=1), st.dtype)
    assert np.array_equal(_gpu.to_f64(out), want)


def test_q8_decode_rejects_other_block_sizes():
    st = wl.tiny_decode()
    s = Q8Step(st)
    d = s.d
    bad = lambda t: t.reshape(t.shape[0] * 2, t.shape[1], t.shape[2] // 2, t.shape[3])  # noqa: E731
    with pytest.raises(nb.NsError) as e:
        nb.ns_paged_attn_decode_q8_0(d.q, bad(s.kc), bad(s.ks), bad(s.vc), bad(s.vs), d.block_tables,
                                     d.context_lens, st.scale, torch.empty_like(d.q), d.ws)
    assert e.value.status == -2
