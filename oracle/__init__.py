"""fp64 CPU oracle for the gathered multi-LoRA delta (SGMV / BGMV shrink and expand).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import this package. The CUDA library never uses it, and it imports
nothing from the CUDA library or its binding.

The arithmetic lives in ``mlora_oracle.c`` (plain C, fp64, one rounding to the I/O type),
which follows Punica section 3.4 "The SGMV Operator" (shrink v = x·A, expand y += v·B),
the reference loop of "Multi-LoRA Serving, in depth" (slot per row, -1 = no adapter,
per-slot scale) and S-LoRA "Unified Paging" (a page is one H-vector; a rank-row of A^T or B
longer than a page spans consecutive entries of the page table).
This module only marshals numpy arrays into that code; it does no arithmetic of its own.

Every function here is pinned by ``tests/test_oracle_pins.py``; ``tests/test_oracle_mutants.py``
shows that planted mistakes in the C make those pins fail.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "mlora_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmlora_oracle.so")

DTYPE_BF16 = 0
DTYPE_FP16 = 1
POOL_STACKED = 0
POOL_PAGED = 1

# Status bits reported by the oracle (its own definitions, in mlora_oracle.c).
BAD_OFFSETS = 1
BAD_SLOT = 2
BAD_RANK = 4
BAD_PAGE = 8


def build(force: bool = False, src: str = SOURCE, out: str = _LIB_PATH) -> str:
    """Compile the oracle's C into a shared library (plain gcc, -O2, no fast-math and no FMA
    contraction, so every product and every sum is one IEEE fp64 operation)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    stale = (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src)
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
               "-Wall", "-Wextra", "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


class _PoolStruct(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("num_slots", ctypes.c_int32), ("num_layers", ctypes.c_int32), ("r_max", ctypes.c_int32),
        ("d_in", ctypes.c_int32), ("d_out", ctypes.c_int32),
        ("a_t", ctypes.c_void_p), ("b", ctypes.c_void_p), ("pages", ctypes.c_void_p),
        ("page_elems", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("a_page_table", ctypes.c_void_p), ("b_page_table", ctypes.c_void_p),
        ("rank", ctypes.c_void_p), ("scale", ctypes.c_void_p),
    ]


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


class Pool:
    """Host copy of an adapter pool, as the oracle reads it.

    Stacked: ``a_t`` [num_slots][num_layers][r_max][d_in] and ``b`` [...][r_max][d_out], both
    uint16 bit patterns of the I/O type. Paged: ``pages`` [num_pages][page_elems] and two page
    tables [num_slots][num_layers][r_max][ceil(d / page_elems)] (int32; d = d_in for A, d_out for
    B: a vector longer than a page spans several). ``rank`` int32 [num_slots], ``scale`` float32.
    """

    def __init__(self, *, dtype, num_slots, num_layers, r_max, d_in, d_out, rank, scale,
                 a_t=None, b=None, pages=None, a_page_table=None, b_page_table=None):
        self.dtype = int(dtype)
        self.kind = POOL_PAGED if pages is not None else POOL_STACKED
        self.num_slots, self.num_layers, self.r_max = int(num_slots), int(num_layers), int(r_max)
        self.d_in, self.d_out = int(d_in), int(d_out)
        self.rank = _c(rank, np.int32)
        self.scale = _c(scale, np.float32)
        self.a_t = _c(a_t, np.uint16)
        self.b = _c(b, np.uint16)
        self.pages = _c(pages, np.uint16)
        self.a_page_table = _c(a_page_table, np.int32)
        self.b_page_table = _c(b_page_table, np.int32)
        if self.kind == POOL_STACKED:
            assert self.a_t.size == num_slots * num_layers * r_max * d_in
            assert self.b.size == num_slots * num_layers * r_max * d_out
        else:
            assert self.pages.ndim == 2
            pe = self.pages.shape[1]
            # one entry per page of each vector: ceil(d / page_elems) pages per vector
            assert self.a_page_table.size == num_slots * num_layers * r_max * (-(-d_in // pe))
            assert self.b_page_table.size == num_slots * num_layers * r_max * (-(-d_out // pe))
        assert self.rank.size == num_slots and self.scale.size == num_slots
        self._s = _PoolStruct(
            self.kind, self.dtype, self.num_slots, self.num_layers, self.r_max, self.d_in, self.d_out,
            _ptr(self.a_t), _ptr(self.b), _ptr(self.pages),
            0 if self.pages is None else self.pages.shape[1],
            0 if self.pages is None else self.pages.shape[0],
            _ptr(self.a_page_table), _ptr(self.b_page_table), _ptr(self.rank), _ptr(self.scale))

    @property
    def ref(self):
        return ctypes.byref(self._s)


def _rows_arg(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(rows, dtype=np.int32)
    return r, int(r.size)


def _check(rc):
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (rc={rc})")


class OracleLib:
    """Marshalling around one build of mlora_oracle.c (the default one, or a test's mutant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P, I, I64, V = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        lib.orc_sgmv_shrink.argtypes = [P, I, V, I64, V, V, I, I, V, I, V, V]
        lib.orc_sgmv_expand.argtypes = [P, I, V, V, I64, V, V, I, I, V, I, V, V]
        lib.orc_bgmv_shrink.argtypes = [P, I, V, I64, V, I, V, I, V, V]
        lib.orc_bgmv_expand.argtypes = [P, I, V, V, I64, V, I, V, I, V, V]
        for f in (lib.orc_sgmv_shrink, lib.orc_sgmv_expand, lib.orc_bgmv_shrink, lib.orc_bgmv_expand):
            f.restype = ctypes.c_int
        lib.orc_round_array.argtypes = [V, V, ctypes.c_size_t, I]
        lib.orc_decode_array.argtypes = [V, V, ctypes.c_size_t, I]
        self.lib = lib

    # ---- phases ------------------------------------------------------------------------
    def sgmv_shrink(self, pool: Pool, layer, x, offsets, seg_slot, rows=None):
        """v (fp64 [M][r_max], NaN where not computed) and the status bits."""
        x = _c(x, np.uint16)
        off, ss = _c(offsets, np.int32), _c(seg_slot, np.int32)
        M = x.shape[0]
        v = np.full((M, pool.r_max), np.nan)
        st = ctypes.c_int32(0)
        rr, nr = _rows_arg(rows)
        _check(self.lib.orc_sgmv_shrink(pool.ref, int(layer), _ptr(x), x.shape[1], _ptr(off), _ptr(ss), ss.size, M,
                                        _ptr(rr), nr, _ptr(v), ctypes.byref(st)))
        return v, st.value

    def sgmv_expand(self, pool: Pool, layer, v, y, offsets, seg_slot, rows=None):
        """(y' as uint16 bits, fp64 y + delta before rounding (NaN where not computed), status)."""
        v = _c(v, np.float64)
        y_out = np.array(y, dtype=np.uint16, copy=True, order="C")
        off, ss = _c(offsets, np.int32), _c(seg_slot, np.int32)
        M = y_out.shape[0]
        y_exact = np.full((M, pool.d_out), np.nan)
        st = ctypes.c_int32(0)
        rr, nr = _rows_arg(rows)
        _check(self.lib.orc_sgmv_expand(pool.ref, int(layer), _ptr(v), _ptr(y_out), y_out.shape[1], _ptr(off),
                                        _ptr(ss), ss.size, M, _ptr(rr), nr, _ptr(y_exact), ctypes.byref(st)))
        return y_out, y_exact, st.value

    def bgmv_shrink(self, pool: Pool, layer, x, row_slot, rows=None):
        x = _c(x, np.uint16)
        rs = _c(row_slot, np.int32)
        M = x.shape[0]
        v = np.full((M, pool.r_max), np.nan)
        st = ctypes.c_int32(0)
        rr, nr = _rows_arg(rows)
        _check(self.lib.orc_bgmv_shrink(pool.ref, int(layer), _ptr(x), x.shape[1], _ptr(rs), M, _ptr(rr), nr,
                                        _ptr(v), ctypes.byref(st)))
        return v, st.value

    def bgmv_expand(self, pool: Pool, layer, v, y, row_slot, rows=None):
        v = _c(v, np.float64)
        y_out = np.array(y, dtype=np.uint16, copy=True, order="C")
        rs = _c(row_slot, np.int32)
        M = y_out.shape[0]
        y_exact = np.full((M, pool.d_out), np.nan)
        st = ctypes.c_int32(0)
        rr, nr = _rows_arg(rows)
        _check(self.lib.orc_bgmv_expand(pool.ref, int(layer), _ptr(v), _ptr(y_out), y_out.shape[1], _ptr(rs), M,
                                        _ptr(rr), nr, _ptr(y_exact), ctypes.byref(st)))
        return y_out, y_exact, st.value

    # ---- both phases ---------------------------------------------------------------------
    def sgmv(self, pool: Pool, layer, x, y, offsets, seg_slot, rows=None):
        """Shrink into an fp64 v, then expand. Returns (y', v, y_exact, status)."""
        v, st1 = self.sgmv_shrink(pool, layer, x, offsets, seg_slot, rows)
        y_out, y_exact, st2 = self.sgmv_expand(pool, layer, v, y, offsets, seg_slot, rows)
        return y_out, v, y_exact, st1 | st2

    def bgmv(self, pool: Pool, layer, x, y, row_slot, rows=None):
        v, st1 = self.bgmv_shrink(pool, layer, x, row_slot, rows)
        y_out, y_exact, st2 = self.bgmv_expand(pool, layer, v, y, row_slot, rows)
        return y_out, v, y_exact, st1 | st2

    # ---- conversions -----------------------------------------------------------------------
    def round_to(self, values, dtype) -> np.ndarray:
        """fp64 -> bf16/fp16 bit patterns, round to nearest even (the oracle's own rounding)."""
        a = np.ascontiguousarray(values, dtype=np.float64)
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.orc_round_array(_ptr(a), _ptr(out), a.size, int(dtype))
        return out

    def decode(self, bits, dtype) -> np.ndarray:
        """bf16/fp16 bit patterns -> exact fp64 values (the oracle's own decoding)."""
        a = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(a.shape, dtype=np.float64)
        self.lib.orc_decode_array(_ptr(a), _ptr(out), a.size, int(dtype))
        return out


_lock = threading.Lock()
_default = None


def default() -> OracleLib:
    """The oracle built from mlora_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
    return _default


def load(path: str) -> OracleLib:
    return OracleLib(path)


def sgmv_shrink(*a, **k):
    return default().sgmv_shrink(*a, **k)


def sgmv_expand(*a, **k):
    return default().sgmv_expand(*a, **k)


def bgmv_shrink(*a, **k):
    return default().bgmv_shrink(*a, **k)


def bgmv_expand(*a, **k):
    return default().bgmv_expand(*a, **k)


def sgmv(*a, **k):
    return default().sgmv(*a, **k)


def bgmv(*a, **k):
    return default().bgmv(*a, **k)


def round_to(*a, **k):
    return default().round_to(*a, **k)


def decode(*a, **k):
    return default().decode(*a, **k)
