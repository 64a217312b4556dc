"""Helpers for the GPU parity tests: move a PagedStep to the device, round the
oracle's fp64 result to the output element type, and compare."""
from __future__ import annotations

import numpy as np
import torch

from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

# Tolerance on fp16 / bf16 attention outputs: max-abs error 2e-3 and relative
# L2 error 1e-3.  The final rounding of the output to its 16-bit type is not
# charged to the kernel:
#   * max-abs: |out - exact| <= 2e-3 + half an ulp of the output type at the
#     exact value (a value within the kernel's fp32 error of a rounding
#     midpoint may round either way: one bf16 ulp is 7.8e-3 in [1, 2));
#   * rel-L2: against the exact value rounded to the output type (rounding
#     exact values to bf16 alone gives a relative L2 near 1.6e-3).
MAX_ABS = 2e-3
REL_L2 = 1e-3


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the fp16 / bf16 numbers around |x| (normal range; the
    subnormal quantum below it)."""
    m, e = np.frexp(np.abs(np.asarray(x, dtype=np.float64)))
    p = 10 if dtype == wl.F16 else 7
    return np.maximum(np.ldexp(1.0, e - 1 - p), 2.0 ** -24 if dtype == wl.F16 else 2.0 ** -133)


def torch_dtype(dtype: str):
    return torch.float16 if dtype == wl.F16 else torch.bfloat16


def to_dev(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t.view(torch_dtype(dtype))


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_ints(a: np.ndarray, dtype, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=dtype)).to(device)


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp64 values to fp16 / bf16 with round-to-nearest-even (exact, one rounding)."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == wl.F16:
        return x.astype(np.float16).astype(np.float64)
    m, e = np.frexp(x)
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)      # 8 significant bits
    tiny = np.abs(x) < 2.0 ** -126                      # subnormal range: quantum 2^-133
    r[tiny] = np.ldexp(np.rint(np.ldexp(x[tiny], 133)), -133)
    return r


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def compare(got: torch.Tensor, ref64: np.ndarray, dtype: str, what: str = ""):
    """Assert the tolerance above.  Returns (kernel max-abs error beyond the
    output rounding, rel-L2 against the rounded oracle, raw max-abs vs fp64)."""
    g = to_f64(got).reshape(ref64.shape)
    r = round_to_dtype(ref64, dtype)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    raw = np.abs(g - ref64)
    excess = float(np.max(raw - 0.5 * ulp(ref64, dtype), initial=0.0))
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    assert excess <= MAX_ABS, f"{what}: max-abs {excess:.3g} beyond the output rounding > {MAX_ABS}"
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3g} > {REL_L2}"
    return excess, rel, float(raw.max(initial=0.0))


class DevStep:
    """A PagedStep on the device (pool BEFORE the step's append)."""

    def __init__(self, st: wl.PagedStep, device="cuda", k_pool=None, v_pool=None):
        self.st = st
        self.q = to_dev(st.q, st.dtype, device)
        self.k_pool = to_dev(st.k_pool if k_pool is None else k_pool, st.dtype, device)
        self.v_pool = to_dev(st.v_pool if v_pool is None else v_pool, st.dtype, device)
        self.k_new = to_dev(st.k_new, st.dtype, device)
        self.v_new = to_dev(st.v_new, st.dtype, device)
        self.slot_mapping = dev_ints(st.slot_mapping, np.int64, device)
        self.block_tables = dev_ints(st.block_tables, np.int32, device)
        self.context_lens = dev_ints(st.context_lens, np.int32, device)
        self.query_start_loc = dev_ints(st.query_start_loc, np.int32, device)
        self.out = torch.empty_like(self.q)
        self.ws = nb.alloc_workspace(st.num_tokens, st.num_q_heads, st.num_kv_heads,
                                     st.head_dim, device)

    def append(self):
        nb.ns_kv_append(self.k_new, self.v_new, self.slot_mapping, self.k_pool, self.v_pool)

    def decode(self, config=None):
        nb.ns_paged_attn_decode(self.q, self.k_pool, self.v_pool, self.block_tables,
                                self.context_lens, self.st.scale, self.out, self.ws, config=config)
        return self.out

    def fused(self):
        nb.ns_kv_append_paged_attn_decode(self.q, self.k_new, self.v_new, self.slot_mapping,
                                          self.k_pool, self.v_pool, self.block_tables,
                                          self.context_lens, self.st.scale, self.out, self.ws)
        return self.out

    def prefill(self):
        nb.ns_paged_attn_prefill(self.q, self.query_start_loc, self.k_pool, self.v_pool,
                                 self.block_tables, self.context_lens, self.st.scale, self.out,
                                 self.ws)
        return self.out


def assert_no_device_status():
    bits = nb.ns_get_device_status(clear=True)
    assert bits == 0, f"device status 0x{bits:x}"


def config(num_ctas=0, min_blocks_per_cta=0, whole_sequences=0):
    c = nb.DecodeConfig()
    c.num_ctas = num_ctas
    c.min_blocks_per_cta = min_blocks_per_cta
    c.whole_sequences = whole_sequences
    return c
