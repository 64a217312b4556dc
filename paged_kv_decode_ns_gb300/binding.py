"""Python binding of the C ABI in ``include/ns_paged.h`` (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it checks tensor shapes, takes device pointers and the
current CUDA stream from torch, calls the library and raises on a non-zero
status.  torch serves only as the allocator and stream provider.  There is
no CPU fallback: if ``_lib/libns_paged.so`` is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

NS_OK = 0
NS_F16 = 0
NS_BF16 = 1
NS_MAX_CTAS = 1024
NS_PREFILL_WALK = 1
NS_PREFILL_TENSOR_CORE = 2
NS_NOALLOC_MAX_PAIRS = 16384
DEV_BITS = {
    0x1: "NS_DEV_BAD_BLOCK_ID",
    0x2: "NS_DEV_BAD_CONTEXT_LEN",
    0x4: "NS_DEV_BAD_SLOT",
    0x8: "NS_DEV_WAIT_TIMEOUT",
    0x10: "NS_DEV_FUSED_SLOT",
    0x20: "NS_DEV_BAD_QUERY_SPAN",
    0x40: "NS_DEV_MERGE_QUEUE",
}


class NsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = lib().ns_status_string(status).decode()
        super().__init__(f"{what}: {msg} ({status})")


class DecodeConfig(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int), ("min_blocks_per_cta", ctypes.c_int),
                ("whole_sequences", ctypes.c_int), ("overlap_prologue", ctypes.c_int),
                ("wait_limit_ns", ctypes.c_int), ("merge_levels", ctypes.c_int), ("reserved", ctypes.c_int * 2)]


class PrefillConfig(ctypes.Structure):
    _fields_ = [("tensor_core_min_span", ctypes.c_int), ("phases", ctypes.c_int),
                ("reserved", ctypes.c_int * 6)]


class DecodePlan(ctypes.Structure):
    _fields_ = [("ctas_launched", ctypes.c_int32), ("ctas_active", ctypes.c_int32),
                ("total_blocks", ctypes.c_int64), ("split_pairs", ctypes.c_int32),
                ("max_pieces", ctypes.c_int32), ("whole_sequences", ctypes.c_int32),
                ("workers_active", ctypes.c_int32), ("merge_levels", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 7)]


_LIB = None
P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t

_SIGNATURES = {
    "ns_status_string": (ctypes.c_char_p, [I]),
    "ns_version": (I, []),
    "ns_kv_append": (I, [P, P, P, P, P, I, I, I, I, I64, I, P]),
    "ns_paged_attn_workspace_bytes": (SZ, [I, I, I, I]),
    "ns_paged_attn_workspace_init": (I, [P, SZ, P]),
    "ns_paged_attn_decode": (I, [P, P, P, P, P, I, I, I, I, I, F, P, P, I, I64, I, P, SZ]),
    "ns_paged_attn_decode_ex": (I, [P, P, P, P, P, I, I, I, I, I, F, P, P, I, I64, I, P, SZ,
                                    ctypes.POINTER(DecodeConfig)]),
    "ns_kv_append_paged_attn_decode": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, F, P, P, I,
                                           I64, I, P, SZ]),
    "ns_kv_append_paged_attn_decode_ex": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, F, P, P, I,
                                              I64, I, P, SZ, ctypes.POINTER(DecodeConfig)]),
    "ns_read_decode_plan": (I, [P, ctypes.POINTER(DecodePlan), P]),
    "ns_paged_attn_prefill": (I, [P, P, P, P, P, P, I, I, I, I, I, I, F, P, P, I, I64, I, P, SZ]),
    "ns_paged_attn_prefill_ex": (I, [P, P, P, P, P, P, I, I, I, I, I, I, F, P, P, I, I64, I, P, SZ,
                                     ctypes.POINTER(PrefillConfig)]),
    "ns_get_device_status": (I, [P, ctypes.POINTER(ctypes.c_uint32), I]),
    "ns_paged_attn_decode_noalloc": (I, [P, P, P, P, P, I, I, I, I, I, F, P, P, I, I64, I]),
    "ns_kv_append_q8_0": (I, [P, P, P, P, P, P, P, I, I, I, I, I64, I, P]),
    "ns_paged_attn_decode_q8_0": (I, [P, P, P, P, P, P, P, I, I, I, I, I, F, P, P, I, I64, I, P, SZ]),
    "ns_kv_append_paged_attn_decode_q8_0": (I, [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, P, P, I,
                                                I64, I, P, SZ]),
}


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded C library (raises if it was never built: there is no fallback)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(
                f"{_build.LIB} is missing: build it with __graft_entry__.build() "
                "(the paged-KV kernels have no CPU fallback)")
        handle = ctypes.CDLL(_build.LIB)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def _check(status: int, what: str):
    if status != NS_OK:
        raise NsError(status, what)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return NS_F16
    if t.dtype == torch.bfloat16:
        return NS_BF16
    raise TypeError(f"expected float16 or bfloat16, got {t.dtype}")


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if getattr(_capture, "on", False):
        return _STREAM_SLOT
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# While a call is prepared, the entry points record their marshalled arguments
# instead of calling the library, and the stream argument is a slot filled in
# at each run.
_capture = threading.local()
_STREAM_SLOT = object()


def _invoke(name: str, *args) -> int:
    if getattr(_capture, "on", False):
        _capture.record = (name, args)
        return NS_OK
    return getattr(lib(), name)(*args)


class PreparedCall:
    """One launching entry point with its arguments checked and marshalled once.

    Calling it runs the same C entry point again on the same buffers (with
    whatever they hold then) on ``stream`` (default: the current stream); only
    the stream is looked up per call.  The object references every tensor and
    config it was prepared with, so their memory stays allocated while it
    lives.  One object must not be called from two threads at once.
    """

    __slots__ = ("name", "_fn", "_args", "_slot", "_keep")

    def __init__(self, name: str, args: tuple, keep: list):
        self.name = name
        self._fn = getattr(lib(), name)
        self._args = list(args)
        slots = [i for i, a in enumerate(self._args) if a is _STREAM_SLOT]
        if len(slots) != 1:
            raise RuntimeError(f"{name}: expected one stream argument")
        self._slot = slots[0]
        self._keep = keep

    def __call__(self, stream=None):
        self._args[self._slot] = _stream(stream)
        _check(self._fn(*self._args), self.name)


def prepare(fn, *args, **kwargs) -> PreparedCall:
    """``fn`` (a launching entry point of this module: ns_kv_append,
    ns_paged_attn_decode, ns_kv_append_paged_attn_decode, ns_paged_attn_prefill
    or a q8_0 one) with these arguments, checked now and run by calling the
    returned object.  It is what a serving loop that calls the same step on the
    same buffers every iteration uses, so that a call costs the host one
    foreign call."""
    if kwargs.get("stream") is not None:
        raise ValueError("the stream is given to each run of a prepared call")
    _capture.on, _capture.record = True, None
    try:
        fn(*args, **kwargs)
    except ctypes.ArgumentError as e:  # an entry point that calls the library directly
        raise TypeError(f"{getattr(fn, '__name__', fn)} cannot be prepared") from e
    finally:
        _capture.on = False
    if _capture.record is None:
        raise TypeError(f"{getattr(fn, '__name__', fn)} cannot be prepared")
    name, marshalled = _capture.record
    _capture.record = None
    keep = [a for a in list(args) + list(kwargs.values()) if a is not None]
    return PreparedCall(name, marshalled, keep)


def ns_version() -> int:
    return lib().ns_version()


def ns_paged_attn_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                  head_dim: int = 64) -> int:
    return int(lib().ns_paged_attn_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim))


def alloc_workspace(num_rows: int, num_q_heads: int, num_kv_heads: int, head_dim: int = 64,
                    device=None) -> torch.Tensor:
    """A zero-filled workspace for up to ``num_rows`` query rows (sequences when decoding)."""
    n = ns_paged_attn_workspace_bytes(num_rows, num_q_heads, num_kv_heads, head_dim)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def ns_kv_append(k, v, slot_mapping, k_pool, v_pool, stream=None):
    """Write k/v [T, Hkv, D] into k_pool/v_pool [NB, Hkv, bs, D] at slot_mapping [T] (int64)."""
    T, hkv, d = k.shape
    nb, hkv2, bs, d2 = k_pool.shape
    if v.shape != k.shape or v_pool.shape != k_pool.shape or hkv2 != hkv or d2 != d:
        raise ValueError("shape mismatch")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    dt = _dtype_code(k)
    st = _invoke("ns_kv_append", _dev(k, "k"), _dev(v, "v", k.dtype),
                 _dev(slot_mapping, "slot_mapping", torch.int64),
                 _dev(k_pool, "k_pool", k.dtype), _dev(v_pool, "v_pool", k.dtype),
                 T, hkv, d, bs, nb, dt, _stream(stream))
    _check(st, "ns_kv_append")


def _attn_common(q, k_pool, v_pool, block_tables, context_lens, out, workspace):
    rows, hq, d = q.shape
    nb, hkv, bs, d2 = k_pool.shape
    if v_pool.shape != k_pool.shape or d2 != d:
        raise ValueError("pool shapes do not match q")
    if block_tables.dim() != 2:
        raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    dt = _dtype_code(q)
    ptrs = dict(q=_dev(q, "q"), k=_dev(k_pool, "k_pool", q.dtype), v=_dev(v_pool, "v_pool", q.dtype),
                bt=_dev(block_tables, "block_tables", torch.int32),
                cl=_dev(context_lens, "context_lens", torch.int32),
                out=_dev(out, "out", q.dtype), ws=_dev(workspace, "workspace", torch.uint8))
    return rows, hq, hkv, d, bs, nb, dt, ptrs


def ns_paged_attn_decode(q, k_pool, v_pool, block_tables, context_lens, scale, out, workspace,
                         config: DecodeConfig | None = None, stream=None):
    """out[s] = paged attention of q[s] over sequence s's blocks (one decode step)."""
    S, hq, hkv, d, bs, nb, dt, p = _attn_common(q, k_pool, v_pool, block_tables, context_lens,
                                                out, workspace)
    if context_lens.shape != (S,) or block_tables.shape[0] != S:
        raise ValueError("one context length and one table row per sequence")
    args = (p["q"], p["k"], p["v"], p["bt"], p["cl"], S, hq, hkv, d, bs, float(scale), p["out"],
            _stream(stream), block_tables.shape[1], nb, dt, p["ws"], workspace.numel())
    if config is None:
        _check(_invoke("ns_paged_attn_decode", *args), "ns_paged_attn_decode")
    else:
        _check(_invoke("ns_paged_attn_decode_ex", *args, ctypes.byref(config)), "ns_paged_attn_decode_ex")


def ns_paged_attn_decode_noalloc(q, k_pool, v_pool, block_tables, context_lens, scale, out,
                                 stream=None):
    """ns_paged_attn_decode for callers that cannot allocate device memory.

    Takes no workspace: the library's own scratch array holds the split
    partials and counters (at most NS_NOALLOC_MAX_PAIRS sequence x kv-head
    pairs).  The first call on a device must come before any stream capture;
    calls that overlap on the GPU race.
    """
    S, hq, d = q.shape
    nb_, hkv, bs, d2 = k_pool.shape
    if v_pool.shape != k_pool.shape or d2 != d or out.shape != q.shape:
        raise ValueError("shape mismatch")
    if context_lens.shape != (S,) or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("one context length and one table row per sequence")
    st = lib().ns_paged_attn_decode_noalloc(
        _dev(q, "q"), _dev(k_pool, "k_pool", q.dtype), _dev(v_pool, "v_pool", q.dtype),
        _dev(block_tables, "block_tables", torch.int32),
        _dev(context_lens, "context_lens", torch.int32), S, hq, hkv, d, bs, float(scale),
        _dev(out, "out", q.dtype), _stream(stream), block_tables.shape[1], nb_, _dtype_code(q))
    _check(st, "ns_paged_attn_decode_noalloc")


def ns_kv_append_paged_attn_decode(q, k_new, v_new, slot_mapping, k_pool, v_pool, block_tables,
                                   context_lens, scale, out, workspace, config: DecodeConfig | None = None,
                                   stream=None):
    """Append one new token per sequence and run the decode step, in one kernel."""
    S, hq, hkv, d, bs, nb, dt, p = _attn_common(q, k_pool, v_pool, block_tables, context_lens,
                                                out, workspace)
    if k_new.shape != (S, hkv, d) or v_new.shape != (S, hkv, d) or slot_mapping.shape != (S,):
        raise ValueError("k_new/v_new must be [num_seqs, Hkv, D], slot_mapping [num_seqs]")
    st = _invoke(
        "ns_kv_append_paged_attn_decode_ex",
        p["q"], _dev(k_new, "k_new", q.dtype), _dev(v_new, "v_new", q.dtype),
        _dev(slot_mapping, "slot_mapping", torch.int64), p["k"], p["v"], p["bt"], p["cl"], S, hq,
        hkv, d, bs, float(scale), p["out"], _stream(stream), block_tables.shape[1], nb, dt,
        p["ws"], workspace.numel(), ctypes.byref(config) if config is not None else None)
    _check(st, "ns_kv_append_paged_attn_decode")


def ns_paged_attn_prefill(q, query_start_loc, k_pool, v_pool, block_tables, context_lens, scale,
                          out, workspace, config: PrefillConfig | None = None, stream=None):
    """Chunked-prefill attention of the query spans ``query_start_loc`` over the paged pool."""
    T, hq, hkv, d, bs, nb, dt, p = _attn_common(q, k_pool, v_pool, block_tables, context_lens,
                                                out, workspace)
    S = context_lens.shape[0]
    if query_start_loc.shape != (S + 1,) or block_tables.shape[0] != S:
        raise ValueError("query_start_loc must be [num_seqs + 1]")
    args = (p["q"], _dev(query_start_loc, "query_start_loc", torch.int32), p["k"], p["v"], p["bt"],
            p["cl"], S, T, hq, hkv, d, bs, float(scale), p["out"], _stream(stream),
            block_tables.shape[1], nb, dt, p["ws"], workspace.numel())
    if config is None:
        _check(_invoke("ns_paged_attn_prefill", *args), "ns_paged_attn_prefill")
    else:
        _check(_invoke("ns_paged_attn_prefill_ex", *args, ctypes.byref(config)),
               "ns_paged_attn_prefill_ex")


def _q8_pools(k_codes, k_scales, v_codes, v_scales):
    nb, hkv, bs, d = k_codes.shape
    if v_codes.shape != k_codes.shape or k_scales.shape != (nb, hkv, bs, d // 32) \
            or v_scales.shape != k_scales.shape:
        raise ValueError("q8_0 pools: codes [NB, Hkv, bs, D] int8, scales [NB, Hkv, bs, D/32] fp16")
    return (nb, hkv, bs, d, _dev(k_codes, "k_codes", torch.int8), _dev(k_scales, "k_scales", torch.float16),
            _dev(v_codes, "v_codes", torch.int8), _dev(v_scales, "v_scales", torch.float16))


def ns_kv_append_q8_0(k, v, slot_mapping, k_codes, k_scales, v_codes, v_scales, stream=None):
    """Quantise k/v [T, Hkv, D] to q8_0 and write codes and scales at slot_mapping [T] (int64)."""
    T, hkv, d = k.shape
    nb, hkv2, bs, d2, kc, ks, vc, vs = _q8_pools(k_codes, k_scales, v_codes, v_scales)
    if v.shape != k.shape or hkv2 != hkv or d2 != d or slot_mapping.shape != (T,):
        raise ValueError("shape mismatch")
    st = _invoke("ns_kv_append_q8_0", _dev(k, "k"), _dev(v, "v", k.dtype),
                 _dev(slot_mapping, "slot_mapping", torch.int64), kc, ks, vc, vs, T, hkv, d,
                 bs, nb, _dtype_code(k), _stream(stream))
    _check(st, "ns_kv_append_q8_0")


def ns_paged_attn_decode_q8_0(q, k_codes, k_scales, v_codes, v_scales, block_tables, context_lens, scale,
                              out, workspace, stream=None):
    """Decode attention of q [S, Hq, D] over a q8_0 pool (block size 16)."""
    S, hq, d = q.shape
    nb, hkv, bs, d2, kc, ks, vc, vs = _q8_pools(k_codes, k_scales, v_codes, v_scales)
    if d2 != d or out.shape != q.shape or context_lens.shape != (S,) or block_tables.shape[0] != S:
        raise ValueError("shape mismatch")
    st = _invoke(
        "ns_paged_attn_decode_q8_0",
        _dev(q, "q"), kc, ks, vc, vs, _dev(block_tables, "block_tables", torch.int32),
        _dev(context_lens, "context_lens", torch.int32), S, hq, hkv, d, bs, float(scale),
        _dev(out, "out", q.dtype), _stream(stream), block_tables.shape[1], nb, _dtype_code(q),
        _dev(workspace, "workspace", torch.uint8), workspace.numel())
    _check(st, "ns_paged_attn_decode_q8_0")


def ns_kv_append_paged_attn_decode_q8_0(q, k_new, v_new, slot_mapping, k_codes, k_scales, v_codes, v_scales,
                                        block_tables, context_lens, scale, out, workspace, stream=None):
    """Quantise and append one new token per sequence, then decode over the q8_0 pool, in one kernel."""
    S, hq, d = q.shape
    nb, hkv, bs, d2, kc, ks, vc, vs = _q8_pools(k_codes, k_scales, v_codes, v_scales)
    if k_new.shape != (S, hkv, d) or v_new.shape != (S, hkv, d) or slot_mapping.shape != (S,):
        raise ValueError("k_new/v_new must be [num_seqs, Hkv, D], slot_mapping [num_seqs]")
    if d2 != d or out.shape != q.shape or context_lens.shape != (S,) or block_tables.shape[0] != S:
        raise ValueError("shape mismatch")
    st = _invoke("ns_kv_append_paged_attn_decode_q8_0", 
        _dev(q, "q"), _dev(k_new, "k_new", q.dtype), _dev(v_new, "v_new", q.dtype),
        _dev(slot_mapping, "slot_mapping", torch.int64), kc, ks, vc, vs,
        _dev(block_tables, "block_tables", torch.int32), _dev(context_lens, "context_lens", torch.int32), S, hq,
        hkv, d, bs, float(scale), _dev(out, "out", q.dtype), _stream(stream), block_tables.shape[1], nb,
        _dtype_code(q), _dev(workspace, "workspace", torch.uint8), workspace.numel())
    _check(st, "ns_kv_append_paged_attn_decode_q8_0")


def ns_read_decode_plan(workspace, stream=None) -> dict:
    plan = DecodePlan()
    _check(lib().ns_read_decode_plan(_dev(workspace, "workspace", torch.uint8), ctypes.byref(plan),
                                     _stream(stream)), "ns_read_decode_plan")
    return {f: getattr(plan, f) for f, _ in DecodePlan._fields_ if f != "reserved"}


def ns_get_device_status(clear: bool = True, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    _check(lib().ns_get_device_status(_stream(stream), ctypes.byref(bits), int(bool(clear))),
           "ns_get_device_status")
    return int(bits.value)


def raise_on_device_status(stream=None):
    """Raise NsError(NS_ERR_DEVICE) if a kernel raised a device status bit (and clear it)."""
    bits = ns_get_device_status(clear=True, stream=stream)
    if bits:
        names = [n for b, n in DEV_BITS.items() if bits & b]
        raise RuntimeError(f"device status 0x{bits:x}: {', '.join(names)}")
