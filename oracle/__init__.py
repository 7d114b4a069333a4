"""fp64 CPU oracle for the sliding-window ring / grouped global-verify attention path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``sliding_window_gqa_ring_gb300``) never imports it, and it never imports the
product library: the two share no code.  Inputs reach both sides from the
seeded generators in ``sliding_window_gqa_ring_gb300.synth``, which hold none of
the method's arithmetic.

The arithmetic lives in ``carat_oracle.c`` (plain C, fp64); this module only
compiles it with gcc, loads it with ctypes and converts numpy arrays.  Every
function cites the passage it follows in that file's header.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(library routine, closed forms, invariants, page-printed values) and the pins
are themselves checked to catch planted mistakes by
``tests/test_oracle_mutations.py``.
"""
from __future__ import annotations

import concurrent.futures
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "carat_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
LIBRARY = os.path.join(_BUILD_DIR, "libcarat_oracle.so")

_lock = threading.Lock()
_lib = None


def build(source: str = SOURCE, library: str = LIBRARY, extra_flags=()) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE double throughout)."""
    os.makedirs(os.path.dirname(library), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", *extra_flags, "-o", library, source, "-lm"]
    subprocess.run(cmd, check=True)
    return library


def _declare(lib):
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    vp = ctypes.c_void_p
    lib.oracle_ring_slot.restype = i64
    lib.oracle_ring_slot.argtypes = [i64, i64]
    lib.oracle_key_count.restype = i64
    lib.oracle_key_count.argtypes = [i64, i64]
    lib.oracle_window_first.restype = i64
    lib.oracle_window_first.argtypes = [i64, i64]
    lib.oracle_attention_row.restype = i32
    lib.oracle_attention_row.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, i32, i64, i64, dbl]
    lib.oracle_attention_request.restype = i32
    lib.oracle_attention_request.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i32, i32, i32,
                                             i64, dbl]
    lib.oracle_ring_expected.restype = i32
    lib.oracle_ring_expected.argtypes = [vp, vp, vp, i64, i64, i64, i64, i32, i32]
    lib.oracle_displaced_expected.restype = i32
    lib.oracle_displaced_expected.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i64, i32, i32]
    lib.oracle_attention_request_f64.restype = i32
    lib.oracle_attention_request_f64.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i32, i32,
                                                 i32, i64, dbl]
    lib.oracle_e4m3_decode.restype = dbl
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode.argtypes = [dbl]
    lib.oracle_quantize_bf16.restype = None
    lib.oracle_quantize_bf16.argtypes = [vp, vp, i64, ctypes.c_float]
    lib.oracle_ring_expected_bytes.restype = i32
    lib.oracle_ring_expected_bytes.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64]
    lib.oracle_displaced_expected_bytes.restype = i32
    lib.oracle_displaced_expected_bytes.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i64, i64]
    return lib


def load_library(path: str):
    """Load an oracle build (the default one, or a test's planted-mistake copy)."""
    return _declare(ctypes.CDLL(path))


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if (not os.path.exists(LIBRARY)
                    or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)):
                build()
            _lib = load_library(LIBRARY)
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 bit patterns must be uint16, got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc == -1:
        raise ValueError(f"{what}: a position the definition needs is not in the supplied history")
    if rc != 0:
        raise ValueError(f"{what}: bad argument (rc={rc})")


class Oracle:
    """The oracle's functions bound to one compiled library."""

    def __init__(self, library=None):
        self.lib = library if library is not None else lib()

    def ring_slot(self, position: int, window: int) -> int:
        return int(self.lib.oracle_ring_slot(position, window))

    def key_count(self, context_length: int, proposal_count: int) -> int:
        return int(self.lib.oracle_key_count(context_length, proposal_count))

    def window_first(self, position: int, window: int) -> int:
        return int(self.lib.oracle_window_first(position, window))

    def attention_row(self, q_row, k_hist, v_hist, hist_base, kv_head, position, window, scale):
        """One output row (double [head_dim]); window <= 0 means global."""
        q_row, k_hist, v_hist = _u16(q_row), _u16(k_hist), _u16(v_hist)
        hist_len, kv_heads, head_dim = k_hist.shape
        out = np.empty(head_dim, dtype=np.float64)
        rc = self.lib.oracle_attention_row(_ptr(out), _ptr(q_row), _ptr(k_hist), _ptr(v_hist),
                                           hist_base, hist_len, kv_heads, head_dim, kv_head,
                                           position, window, float(scale))
        _check(rc, "attention_row")
        return out

    def attention_request(self, q, k_hist, v_hist, hist_base, context_length, window, scale):
        """All rows of one request.

        q: uint16 [proposal_count][q_heads][head_dim]; k_hist, v_hist: uint16
        [hist_len][kv_heads][head_dim] holding positions hist_base...; returns
        float64 [proposal_count][q_heads][head_dim].
        """
        q, k_hist, v_hist = _u16(q), _u16(k_hist), _u16(v_hist)
        proposal_count, q_heads, head_dim = q.shape
        hist_len, kv_heads, head_dim_k = k_hist.shape
        if head_dim_k != head_dim or v_hist.shape != k_hist.shape:
            raise ValueError("shape mismatch")
        out = np.empty(q.shape, dtype=np.float64)
        rc = self.lib.oracle_attention_request(_ptr(out), _ptr(q), _ptr(k_hist), _ptr(v_hist),
                                               hist_base, hist_len, context_length,
                                               proposal_count, q_heads, kv_heads, head_dim,
                                               window, float(scale))
        _check(rc, "attention_request")
        return out

    def attention_batch(self, requests, threads=None):
        """attention_request over a list of argument tuples, in a thread pool.

        ctypes releases the GIL during the foreign call, so the requests run on
        separate cores.  Returns the list of outputs in input order.
        """
        threads = threads or os.cpu_count() or 1
        with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as pool:
            return list(pool.map(lambda a: self.attention_request(*a), requests))

    def ring_expected(self, hist, hist_base, key_count, window, ring=None, slot_valid=None):
        """Expected ring [window][kv_heads][head_dim] after positions [0, key_count)."""
        hist = _u16(hist)
        hist_len, kv_heads, head_dim = hist.shape
        if ring is None:
            ring = np.zeros((window, kv_heads, head_dim), dtype=np.uint16)
        if slot_valid is None:
            slot_valid = np.zeros(window, dtype=np.uint8)
        rc = self.lib.oracle_ring_expected(_ptr(ring), _ptr(slot_valid), _ptr(hist), hist_base,
                                           hist_len, key_count, window, kv_heads, head_dim)
        _check(rc, "ring_expected")
        return ring, slot_valid.astype(bool)

    def displaced_expected(self, k_hist, v_hist, hist_base, context_length, proposal_count,
                           window):
        """Expected displaced rows [proposal_count-1][2][kv_heads][head_dim] and validity."""
        k_hist, v_hist = _u16(k_hist), _u16(v_hist)
        hist_len, kv_heads, head_dim = k_hist.shape
        n = max(proposal_count - 1, 0)
        out = np.zeros((max(n, 1), 2, kv_heads, head_dim), dtype=np.uint16)
        valid = np.zeros(max(n, 1), dtype=np.uint8)
        rc = self.lib.oracle_displaced_expected(_ptr(out), _ptr(valid), _ptr(k_hist),
                                                _ptr(v_hist), hist_base, hist_len,
                                                context_length, proposal_count, window,
                                                kv_heads, head_dim)
        _check(rc, "displaced_expected")
        return out[:n], valid[:n].astype(bool)

    # ------------------------------------------------------------- FP8 KV cache
    def e4m3_decode(self, codes) -> np.ndarray:
        """float64 value of each e4m3 code (NaN for the NaN codes)."""
        codes = np.asarray(codes, dtype=np.uint8)
        flat = [self.lib.oracle_e4m3_decode(int(c)) for c in codes.ravel()]
        return np.asarray(flat, dtype=np.float64).reshape(codes.shape)

    def e4m3_encode(self, values) -> np.ndarray:
        """Nearest e4m3 code of each value (ties to even, saturating at 448)."""
        values = np.asarray(values, dtype=np.float64)
        flat = [self.lib.oracle_e4m3_encode(float(v)) for v in values.ravel()]
        return np.asarray(flat, dtype=np.uint8).reshape(values.shape)

    def quantize_bf16(self, bits, scale: float) -> np.ndarray:
        """FP8 cache codes of bf16 values for dequantisation scale `scale`."""
        bits = _u16(bits)
        out = np.empty(bits.shape, dtype=np.uint8)
        self.lib.oracle_quantize_bf16(_ptr(out), _ptr(bits), bits.size, float(scale))
        return out

    def dequantize(self, codes, scale: float) -> np.ndarray:
        """Values an FP8 cache holds: e4m3 value x scale (float64)."""
        table = self.e4m3_decode(np.arange(256, dtype=np.uint8)) * float(np.float32(scale))
        return table[np.asarray(codes, dtype=np.uint8)]

    def attention_request_f64(self, q, k_hist, v_hist, hist_base, context_length, window, scale):
        """attention_request with float64 K/V histories (e.g. a dequantised FP8 cache)."""
        q = _u16(q)
        k_hist = np.ascontiguousarray(k_hist, dtype=np.float64)
        v_hist = np.ascontiguousarray(v_hist, dtype=np.float64)
        proposal_count, q_heads, head_dim = q.shape
        hist_len, kv_heads, head_dim_k = k_hist.shape
        if head_dim_k != head_dim or v_hist.shape != k_hist.shape:
            raise ValueError("shape mismatch")
        out = np.empty(q.shape, dtype=np.float64)
        rc = self.lib.oracle_attention_request_f64(_ptr(out), _ptr(q), _ptr(k_hist),
                                                   _ptr(v_hist), hist_base, hist_len,
                                                   context_length, proposal_count, q_heads,
                                                   kv_heads, head_dim, window, float(scale))
        _check(rc, "attention_request_f64")
        return out

    def ring_expected_bytes(self, hist, hist_base, key_count, window):
        """Expected FP8 ring [window][...row bytes] after positions [0, key_count)."""
        hist = np.ascontiguousarray(hist, dtype=np.uint8)
        hist_len = hist.shape[0]
        row_bytes = int(np.prod(hist.shape[1:]))
        ring = np.zeros((window,) + hist.shape[1:], dtype=np.uint8)
        slot_valid = np.zeros(window, dtype=np.uint8)
        rc = self.lib.oracle_ring_expected_bytes(_ptr(ring), _ptr(slot_valid), _ptr(hist),
                                                 hist_base, hist_len, key_count, window,
                                                 row_bytes)
        _check(rc, "ring_expected_bytes")
        return ring, slot_valid.astype(bool)

    def displaced_expected_bytes(self, k_hist, v_hist, hist_base, context_length,
                                 proposal_count, window):
        """Expected FP8 displaced rows [proposal_count-1][2][...row] and validity."""
        k_hist = np.ascontiguousarray(k_hist, dtype=np.uint8)
        v_hist = np.ascontiguousarray(v_hist, dtype=np.uint8)
        hist_len = k_hist.shape[0]
        row_bytes = int(np.prod(k_hist.shape[1:]))
        n = max(proposal_count - 1, 0)
        out = np.zeros((max(n, 1), 2) + k_hist.shape[1:], dtype=np.uint8)
        valid = np.zeros(max(n, 1), dtype=np.uint8)
        rc = self.lib.oracle_displaced_expected_bytes(_ptr(out), _ptr(valid), _ptr(k_hist),
                                                      _ptr(v_hist), hist_base, hist_len,
                                                      context_length, proposal_count, window,
                                                      row_bytes)
        _check(rc, "displaced_expected_bytes")
        return out[:n], valid[:n].astype(bool)


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
