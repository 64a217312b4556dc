"""Prepared calls of the Python binding (host logic, no GPU): a prepared call
passes the library exactly the arguments the direct call passes, fills in
the stream per run, and keeps its tensors alive."""
import gc
import weakref

import pytest
import torch

from paged_kv_decode_ns_gb300 import binding as nb


class FakeLib:
    """Records every entry-point call; returns NS_OK."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if not name.startswith("ns_"):
            raise AttributeError(name)

        def fn(*args):
            self.calls.append((name, args))
            return nb.NS_OK
        return fn


@pytest.fixture
def fake(monkeypatch):
    lib = FakeLib()
    monkeypatch.setattr(nb, "lib", lambda: lib)
    # host tensors stand in for device ones: only their addresses are passed
    monkeypatch.setattr(nb, "_dev", lambda t, name, dtype=None: t.data_ptr())
    return lib


def _decode_inputs(S=3, hq=14, hkv=2, d=64, nbk=10, bs=16, maxb=4):
    h = torch.float16
    return dict(q=torch.zeros(S, hq, d, dtype=h), k_new=torch.zeros(S, hkv, d, dtype=h),
                v_new=torch.zeros(S, hkv, d, dtype=h), slot_mapping=torch.zeros(S, dtype=torch.int64),
                k_pool=torch.zeros(nbk, hkv, bs, d, dtype=h), v_pool=torch.zeros(nbk, hkv, bs, d, dtype=h),
                block_tables=torch.zeros(S, maxb, dtype=torch.int32),
                context_lens=torch.ones(S, dtype=torch.int32), scale=0.125,
                out=torch.zeros(S, hq, d, dtype=h), workspace=torch.zeros(4096, dtype=torch.uint8))


def test_prepared_fused_decode_passes_the_direct_arguments(fake):
    a = _decode_inputs()
    cfg = nb.DecodeConfig()
    cfg.merge_levels = 1
    nb.ns_kv_append_paged_attn_decode(**a, config=cfg, stream=1234)
    pc = nb.prepare(nb.ns_kv_append_paged_attn_decode, **a, config=cfg)
    assert len(fake.calls) == 1  # preparing calls nothing
    pc(stream=1234)
    pc(stream=99)
    (n0, direct), (n1, first), (n2, second) = fake.calls
    assert n0 == n1 == n2 == "ns_kv_append_paged_attn_decode_ex"
    assert len(direct) == len(first)
    for x, y in zip(direct, first):
        if isinstance(x, (int, float)) or x is None:
            assert x == y
        else:  # ctypes.byref of the same config
            assert ctypes_addr(x) == ctypes_addr(y)
    i = direct.index(1234)
    assert second[i] == 99 and second[:i] == first[:i]


def ctypes_addr(ref):
    import ctypes
    return ctypes.cast(ref, ctypes.c_void_p).value


def test_prepared_prefill_and_append(fake):
    S, hq, hkv, d, bs, nbk = 2, 14, 2, 64, 16, 8
    h = torch.float16
    q = torch.zeros(5, hq, d, dtype=h)
    kp, vp = torch.zeros(nbk, hkv, bs, d, dtype=h), torch.zeros(nbk, hkv, bs, d, dtype=h)
    qsl = torch.tensor([0, 1, 5], dtype=torch.int32)
    bt = torch.zeros(S, 4, dtype=torch.int32)
    cl = torch.tensor([3, 9], dtype=torch.int32)
    out, ws = torch.zeros_like(q), torch.zeros(4096, dtype=torch.uint8)
    pc = nb.prepare(nb.ns_paged_attn_prefill, q, qsl, kp, vp, bt, cl, 0.125, out, ws)
    pc(stream=7)
    nb.ns_paged_attn_prefill(q, qsl, kp, vp, bt, cl, 0.125, out, ws, stream=7)
    assert fake.calls[0] == fake.calls[1] and fake.calls[0][0] == "ns_paged_attn_prefill"
    k, v = torch.zeros(5, hkv, d, dtype=h), torch.zeros(5, hkv, d, dtype=h)
    slots = torch.arange(5, dtype=torch.int64)
    nb.prepare(nb.ns_kv_append, k, v, slots, kp, vp)(stream=7)
    nb.ns_kv_append(k, v, slots, kp, vp, stream=7)
    assert fake.calls[2] == fake.calls[3] and fake.calls[2][0] == "ns_kv_append"


def test_prepared_call_keeps_its_tensors(fake):
    a = _decode_inputs()
    ref = weakref.ref(a["out"])
    pc = nb.prepare(nb.ns_kv_append_paged_attn_decode, **a)
    del a
    gc.collect()
    assert ref() is not None
    del pc
    gc.collect()
    assert ref() is None


def test_prepare_checks_like_the_call_and_takes_no_stream(fake):
    a = _decode_inputs()
    bad = dict(a, k_new=torch.zeros(2, 2, 64, dtype=torch.float16))
    with pytest.raises(ValueError):
        nb.prepare(nb.ns_kv_append_paged_attn_decode, **bad)
    with pytest.raises(ValueError):
        nb.prepare(nb.ns_kv_append_paged_attn_decode, **a, stream=5)
    with pytest.raises(TypeError):
        nb.prepare(nb.ns_version)
    # a failed prepare leaves the binding calling the library again
    nb.ns_kv_append_paged_attn_decode(**a, stream=3)
    assert fake.calls[-1][0] == "ns_kv_append_paged_attn_decode_ex"


def test_prepared_q8_0_fused_decode(fake):
    S, hq, hkv, d, nbk, bs = 2, 14, 2, 64, 6, 16
    h = torch.float16
    q, out = torch.zeros(S, hq, d, dtype=h), torch.zeros(S, hq, d, dtype=h)
    kn, vn = torch.zeros(S, hkv, d, dtype=h), torch.zeros(S, hkv, d, dtype=h)
    slots = torch.zeros(S, dtype=torch.int64)
    kc, vc = (torch.zeros(nbk, hkv, bs, d, dtype=torch.int8) for _ in range(2))
    ks, vs = (torch.zeros(nbk, hkv, bs, d // 32, dtype=h) for _ in range(2))
    bt, cl = torch.zeros(S, 3, dtype=torch.int32), torch.ones(S, dtype=torch.int32)
    ws = torch.zeros(4096, dtype=torch.uint8)
    args = (q, kn, vn, slots, kc, ks, vc, vs, bt, cl, 0.125, out, ws)
    nb.ns_kv_append_paged_attn_decode_q8_0(*args, stream=11)
    nb.prepare(nb.ns_kv_append_paged_attn_decode_q8_0, *args)(stream=11)
    assert fake.calls[0] == fake.calls[1]
    assert fake.calls[0][0] == "ns_kv_append_paged_attn_decode_q8_0"
