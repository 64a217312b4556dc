"""GPU edge cases and the invariants the pages fix, through the C ABI."""
import numpy as np
import pytest
import torch

import _gpu
from _gpu import DevStep, compare, config
from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def make(lens, *, dtype=wl.F16, hq=14, hkv=2, bs=16, seed=0, **kw):
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int32)
    return wl.make_step(rng, lens, np.ones(len(lens), np.int32), dtype=dtype, num_q_heads=hq,
                        num_kv_heads=hkv, block_size=bs, **kw)


def run_decode(st, orc, cfg=None, fused=False):
    ref, kp, vp = orc.step(st)
    d = DevStep(st) if fused else DevStep(st, k_pool=kp, v_pool=vp)
    out = d.fused() if fused else d.decode(cfg)
    torch.cuda.synchronize()
    return d, out, ref, kp, vp


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
@pytest.mark.parametrize("bs", [4, 8, 16, 32])
def test_block_sizes_and_ragged_tails(bs, dtype, orc):
    st = make([1, bs - 1, bs, bs + 1, 3 * bs + 2, 200, 77], dtype=dtype, bs=bs, seed=bs)
    for fused in (False, True):
        d, out, ref, kp, vp = run_decode(st, orc, fused=fused)
        compare(out, ref, dtype, f"bs={bs} fused={fused}")
    _gpu.assert_no_device_status()


@pytest.mark.parametrize("hq,hkv", [(1, 1), (2, 1), (3, 1), (4, 2), (10, 2), (12, 2), (14, 2),
                                    (16, 2), (8, 8), (32, 4)])
def test_group_sizes(hq, hkv, orc):
    st = make([5, 40, 129, 300], hq=hq, hkv=hkv, seed=hq * 10 + hkv)
    d, out, ref, *_ = run_decode(st, orc)
    compare(out, ref, st.dtype, f"Hq={hq} Hkv={hkv}")
    d, out, ref, *_ = run_decode(st, orc, fused=True)
    compare(out, ref, st.dtype, f"Hq={hq} Hkv={hkv} fused")
    _gpu.assert_no_device_status()


def test_single_sequence_at_table_capacity(orc):
    st = make([8192], dtype=wl.BF16, seed=3, max_blocks_per_seq=512)
    for cfg in (None, config(num_ctas=1), config(min_blocks_per_cta=1)):
        d, out, ref, *_ = run_decode(st, orc, cfg)
        compare(out, ref, st.dtype, "L=8192")
    _gpu.assert_no_device_status()


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_context_one_returns_v_exactly(dtype, orc):
    st = make([1] * 9, dtype=dtype, seed=4)
    for fused in (False, True):
        d, out, ref, kp, vp = run_decode(st, orc, fused=fused)
        got = _gpu.to_bits(out)                      # [S, Hq, D]
        v = st.v_new                                 # the new token is the only one
        want = np.repeat(v, st.num_q_heads // st.num_kv_heads, axis=1)
        assert np.array_equal(got, want)
    _gpu.assert_no_device_status()


def test_constant_v_returns_constant(orc):
    st = make([3, 50, 700, 1500], dtype=wl.BF16, seed=5)
    rng = np.random.default_rng(9)
    vec = wl.float_to_bits(rng.standard_normal((2, 64)).astype(np.float32), st.dtype)
    st.v_pool[:] = vec[None, :, None, :]
    st.v_new[:] = vec[None, :, :]
    import _pins
    d, out, ref, *_ = run_decode(st, orc, config(min_blocks_per_cta=1))
    got = _gpu.to_f64(out)
    want = np.repeat(_pins.bits_to_f64(vec, st.dtype), 7, axis=0)[None]   # [1, Hq, D]
    ulp = np.abs(want) * 2.0 ** -7                      # one bf16 ulp (upper bound)
    assert np.all(np.abs(got - want) <= ulp)
    assert np.mean(got == want) > 0.99


def test_block_permutation_is_bit_identical(orc):
    st = make([33, 500, 1030, 9], seed=6, free_frac=0.5)
    ref, kp, vp = orc.step(st)
    a = DevStep(st, k_pool=kp, v_pool=vp).decode().clone()
    pi = np.random.default_rng(11).permutation(st.num_blocks)
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[pi] = kp
    vp2[pi] = vp
    st2 = wl.PagedStep(**{**st.__dict__})
    st2.block_tables = np.where(st.block_tables >= 0, pi[np.maximum(st.block_tables, 0)],
                                -1).astype(np.int32)
    b = DevStep(st2, k_pool=kp2, v_pool=vp2).decode()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    compare(b, ref, st.dtype)


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_nan_in_unused_slots_changes_nothing(dtype, orc):
    """Free blocks, block tails and the new tokens' slots hold NaN: the output
    is bit-identical to the run with finite garbage there."""
    lens = [1, 15, 16, 17, 250, 1000]
    clean = make(lens, dtype=dtype, seed=7)
    dirty = make(lens, dtype=dtype, seed=7, poison_unused=True)
    outs = []
    for st in (clean, dirty):
        d = DevStep(st)
        outs.append(d.fused().clone())
        d2 = DevStep(st)
        d2.append()
        outs.append(d2.decode().clone())
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[2]) and torch.equal(outs[1], outs[3])
    ref, *_ = orc.step(clean)
    compare(outs[2], ref, dtype)
    compare(outs[3], ref, dtype)
    _gpu.assert_no_device_status()


def test_zero_length_sequences_give_zero(orc):
    lens = np.array([0, 5, 0, 17, 40], np.int32)
    st = make(np.maximum(lens, 1), seed=8)
    st.context_lens = lens
    ref = orc.paged_attention(st.dtype, st.q, st.k_pool, st.v_pool, st.block_tables, lens, st.scale)
    d = DevStep(st)
    d.out.fill_(7.0)
    out = d.decode()
    torch.cuda.synchronize()
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    compare(out, ref, st.dtype)
    _gpu.assert_no_device_status()


def test_bad_block_id_is_flagged_not_read():
    st = make([40, 40], seed=9)
    st.block_tables[1, 1] = st.num_blocks + 100
    d = DevStep(st)
    d.decode()
    torch.cuda.synchronize()
    assert nb.ns_get_device_status(clear=True) & 0x1


def test_context_len_beyond_table_is_flagged():
    st = make([40, 40], seed=10)
    d = DevStep(st)
    d.context_lens = _gpu.dev_ints(np.array([40, 40 + 16 * st.max_blocks_per_seq], np.int32),
                                   np.int32)
    d.decode()
    torch.cuda.synchronize()
    assert nb.ns_get_device_status(clear=True) & 0x2


def test_fused_slot_mismatch_is_flagged():
    st = make([40, 41], seed=12)
    st.slot_mapping[1] = st.slot_mapping[0]
    d = DevStep(st)
    d.fused()
    torch.cuda.synchronize()
    assert nb.ns_get_device_status(clear=True) & 0x10


def test_host_side_validation():
    st = make([5, 6], seed=13)
    d = DevStep(st)
    with pytest.raises(nb.NsError) as e:
        nb.ns_paged_attn_decode(d.q, d.k_pool, d.v_pool, d.block_tables, d.context_lens,
                                st.scale, d.out, d.ws[:16])
    assert e.value.status == -1
    q96 = torch.zeros(2, 14, 96, dtype=torch.float16, device="cuda")
    kp96 = torch.zeros(4, 2, 16, 96, dtype=torch.float16, device="cuda")
    with pytest.raises(nb.NsError) as e:
        nb.ns_paged_attn_decode(q96, kp96, kp96, d.block_tables, d.context_lens, st.scale,
                                torch.empty_like(q96), d.ws)
    assert e.value.status == -2
    # head_dim 128 needs a larger workspace than the one sized for 64
    q128 = torch.zeros(2, 14, 128, dtype=torch.float16, device="cuda")
    kp128 = torch.zeros(4, 2, 16, 128, dtype=torch.float16, device="cuda")
    small = nb.ns_paged_attn_workspace_bytes(2, 14, 2, 64)
    assert nb.ns_paged_attn_workspace_bytes(2, 14, 2, 128) > small
    with pytest.raises(nb.NsError) as e:
        nb.ns_paged_attn_decode(q128, kp128, kp128, d.block_tables, d.context_lens, st.scale,
                                torch.empty_like(q128), d.ws[:small])
    assert e.value.status == -1
    # a misaligned (2-byte offset) q
    flat = torch.zeros(2 * 14 * 64 + 1, dtype=torch.float16, device="cuda")
    qmis = flat[1:].view(2, 14, 64)
    with pytest.raises(nb.NsError) as e:
        nb.ns_paged_attn_decode(qmis, d.k_pool, d.v_pool, d.block_tables, d.context_lens,
                                st.scale, d.out, d.ws)
    assert e.value.status == -1
    _gpu.assert_no_device_status()
