"""fp64 CPU oracle for the paged-KV hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference arm may import this package.  The product path (the CUDA
library and its binding) never does, and this package imports nothing from
the product package: the two share no code.

The arithmetic lives in ``ns_oracle.c`` (plain C, double precision, written
from the definitions that file's header states).  This module compiles it
with the host compiler and wraps it with ctypes.  Every function pin (what
fixes the oracle to something other than itself) lives in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ns_oracle.c")
LIB_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIB_DIR, "libns_oracle.so")

_DTYPE_CODE = {"f16": 0, "bf16": 1}


def build(src: str = SRC, out: str = LIB, openmp: bool = True, extra_flags=()) -> str:
    """Compile the oracle into a shared library with gcc; return its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math"]
    if openmp:
        cmd.append("-fopenmp")
    cmd += list(extra_flags) + [src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _stale(lib: str, src: str) -> bool:
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(src)


class Oracle:
    """ctypes handle on one compiled copy of the oracle."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        lib.oracle_f16_to_double.restype = ctypes.c_double
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_kv_append.restype = ctypes.c_int
        lib.oracle_kv_append.argtypes = [P, P, P, P, P, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int64]
        lib.oracle_paged_attention.restype = ctypes.c_int
        lib.oracle_paged_attention.argtypes = [ctypes.c_int, P, P, P, P, P, ctypes.c_int, P,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                               ctypes.c_double, P, ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        self._lib = lib

    # -- element decoders ---------------------------------------------------
    def f16_to_double(self, bits: int) -> float:
        return self._lib.oracle_f16_to_double(int(bits))

    def bf16_to_double(self, bits: int) -> float:
        return self._lib.oracle_bf16_to_double(int(bits))

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())

    # -- the hot path ---------------------------------------------------------
    def kv_append(self, k_pool, v_pool, k_new, v_new, slot_mapping, block_size: int):
        """Return copies of (k_pool, v_pool) with the new tokens written to their slots."""
        kp = np.array(k_pool, dtype=np.uint16, copy=True, order="C")
        vp = np.array(v_pool, dtype=np.uint16, copy=True, order="C")
        k = np.ascontiguousarray(k_new, dtype=np.uint16)
        v = np.ascontiguousarray(v_new, dtype=np.uint16)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        num_blocks, hkv, bs, d = kp.shape
        assert bs == block_size
        rc = self._lib.oracle_kv_append(k.ctypes.data, v.ctypes.data, sm.ctypes.data,
                                        kp.ctypes.data, vp.ctypes.data, sm.shape[0],
                                        hkv, d, bs, num_blocks)
        if rc != 0:
            raise ValueError(f"oracle_kv_append failed ({rc})")
        return kp, vp

    def paged_attention(self, dtype: str, q, k_pool, v_pool, block_tables, context_lens,
                        scale: float, query_start_loc=None, num_threads: int = 1):
        """fp64 attention output [rows, Hq, D] for the query rows ``q``."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        kp = np.ascontiguousarray(k_pool, dtype=np.uint16)
        vp = np.ascontiguousarray(v_pool, dtype=np.uint16)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        num_blocks, hkv, bs, d = kp.shape
        rows, hq, dq = q.shape
        assert dq == d
        qsl_ptr = None
        if query_start_loc is not None:
            qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
            assert qsl.shape == (cl.shape[0] + 1,) and int(qsl[-1]) == rows
            qsl_ptr = qsl.ctypes.data
        else:
            assert rows == cl.shape[0]
        out = np.zeros((rows, hq, d), dtype=np.float64)
        rc = self._lib.oracle_paged_attention(_DTYPE_CODE[dtype], q.ctypes.data, qsl_ptr,
                                              kp.ctypes.data, vp.ctypes.data, bt.ctypes.data,
                                              bt.shape[1], cl.ctypes.data, cl.shape[0],
                                              hq, hkv, d, bs, num_blocks, float(scale),
                                              out.ctypes.data, int(num_threads))
        if rc != 0:
            raise ValueError(f"oracle_paged_attention failed ({rc})")
        return out

    # -- whole steps --------------------------------------------------------
    def step(self, st, num_threads: int = 1, with_append: bool = True):
        """Append ``st``'s new tokens, then attend every query row.

        Returns (out_fp64 [T, Hq, D], k_pool_after, v_pool_after).
        """
        if with_append:
            kp, vp = self.kv_append(st.k_pool, st.v_pool, st.k_new, st.v_new,
                                    st.slot_mapping, st.block_size)
        else:
            kp, vp = st.k_pool, st.v_pool
        qsl = None if st.is_decode else st.query_start_loc
        out = self.paged_attention(st.dtype, st.q, kp, vp, st.block_tables, st.context_lens,
                                   st.scale, query_start_loc=qsl, num_threads=num_threads)
        return out, kp, vp


_DEFAULT = None


def load(path: str | None = None) -> Oracle:
    """Load the oracle, compiling it first if the library is missing or stale."""
    global _DEFAULT
    if path is not None:
        return Oracle(path)
    if _DEFAULT is None:
        if _stale(LIB, SRC):
            build()
        _DEFAULT = Oracle(LIB)
    return _DEFAULT


def build_variant(src_text: str, flags=()) -> Oracle:
    """Compile an edited copy of the oracle source into a temp dir (used by the
    mutation tests, which plant a mistake in the oracle and check that a pin
    catches it)."""
    tmp = tempfile.mkdtemp(prefix="ns_oracle_variant_")
    src = os.path.join(tmp, "ns_oracle_variant.c")
    with open(src, "w") as f:
        f.write(src_text)
    out = os.path.join(tmp, "libns_oracle_variant.so")
    build(src=src, out=out, openmp=False, extra_flags=flags)
    return Oracle(out)
