"""Python binding of libmlora: gathered multi-LoRA shrink / expand on GB300 (sm_103a).

Argument marshalling only. Every function has the name of the C entry point it calls
(include/mlora.h) and passes device pointers, sizes and the current CUDA stream through
ctypes; all arithmetic runs in the library's CUDA kernels. PyTorch is used for device memory
and streams. There is no fallback: if libmlora.so is missing, or a tensor is not a CUDA
tensor, the call raises.

Pools are described once with :func:`make_pool` (any object with the attributes of
``workloads.Pool`` works) and reused for every call.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmlora.so")

MLORA_BF16, MLORA_FP16 = 0, 1
MLORA_POOL_STACKED, MLORA_POOL_PAGED = 0, 1
MLORA_MAX_GROUP = 8
MLORA_MAX_RANK = 128
STATUS_BAD_OFFSETS, STATUS_BAD_SLOT, STATUS_BAD_RANK, STATUS_BAD_PAGE, STATUS_TIMEOUT = 1, 2, 4, 8, 16
ERR_NULL, ERR_DTYPE, ERR_SHAPE, ERR_ALIGN, ERR_POOL, ERR_CUDA, ERR_TOO_LARGE = -1, -2, -3, -4, -5, -6, -7
NOALLOC_MAX_FLOATS = 1 << 20
LAUNCH_PROGRAMMATIC, LAUNCH_GROUP_ROWS, LAUNCH_NO_GROUPING = 1, 2, 4

_DT = {torch.bfloat16: MLORA_BF16, torch.float16: MLORA_FP16}


class MloraError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libmlora error {code}: {msg}")
        self.code = code


class mlora_pool(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("dtype", ctypes.c_int32), ("num_slots", ctypes.c_int32),
                ("num_layers", ctypes.c_int32), ("r_max", ctypes.c_int32), ("d_in", ctypes.c_int32),
                ("d_out", ctypes.c_int32), ("a_t", ctypes.c_void_p), ("b", ctypes.c_void_p),
                ("pages", ctypes.c_void_p), ("page_elems", ctypes.c_int64), ("num_pages", ctypes.c_int64),
                ("a_page_table", ctypes.c_void_p), ("b_page_table", ctypes.c_void_p), ("rank", ctypes.c_void_p),
                ("scale", ctypes.c_void_p)]


class mlora_problem(ctypes.Structure):
    _fields_ = [("y", ctypes.c_void_p), ("ldy", ctypes.c_int64), ("x", ctypes.c_void_p), ("ldx", ctypes.c_int64),
                ("pool", ctypes.POINTER(mlora_pool)), ("layer", ctypes.c_int32), ("v_scratch", ctypes.c_void_p)]


class mlora_group(ctypes.Structure):
    _fields_ = [("problems", ctypes.POINTER(mlora_problem)), ("num_problems", ctypes.c_int32),
                ("seg_offsets", ctypes.c_void_p), ("seg_slot", ctypes.c_void_p), ("num_segments", ctypes.c_int32),
                ("num_rows", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None

_P, _I32, _I64, _V = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
_PP = ctypes.POINTER(mlora_pool)
SIGNATURES = {
    "lora_sgmv_shrink": [_V, _V, _I64, _PP, _V, _V, _I32, _I32, _I32, _V, _V],
    "lora_sgmv_expand": [_V, _I64, _V, _PP, _V, _V, _I32, _I32, _I32, _V, _V],
    "lora_bgmv_shrink": [_V, _V, _I64, _PP, _V, _I32, _I32, _V, _V],
    "lora_bgmv_expand": [_V, _I64, _V, _PP, _V, _I32, _I32, _V, _V],
    "lora_sgmv": [_V, _I64, _V, _I64, _PP, _V, _V, _I32, _I32, _I32, _V, _V, _V],
    "lora_bgmv": [_V, _I64, _V, _I64, _PP, _V, _I32, _I32, _V, _V, _V],
    "lora_bgmv_ex": [_V, _I64, _V, _I64, _PP, _V, _I32, _I32, _V, ctypes.c_uint32, _V, _V],
    "lora_sgmv_noalloc": [_V, _I64, _V, _I64, _PP, _V, _V, _I32, _I32, _I32, _V, _V],
    "lora_sgmv_grouped": [ctypes.POINTER(mlora_problem), _I32, _V, _V, _I32, _I32, _V, _V],
    "lora_sgmv_grouped_ex": [ctypes.POINTER(mlora_problem), _I32, _V, _V, _I32, _I32, ctypes.c_uint32, _V, _V],
    "lora_sgmv_sequence": [ctypes.POINTER(mlora_group), _I32, ctypes.c_uint32, _V, _V],
}


def lib():
    """The loaded libmlora (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m adapter_gemv_gb300.build`")
                L = ctypes.CDLL(LIB_PATH)
                for name, args in SIGNATURES.items():
                    fn = getattr(L, name)
                    fn.argtypes = args
                    fn.restype = ctypes.c_int
                L.lora_error_string.argtypes = [ctypes.c_int]
                L.lora_error_string.restype = ctypes.c_char_p
                L.lora_abi_version.restype = ctypes.c_int
                L.lora_launch_count.restype = ctypes.c_int64
                L.lora_set_programmatic_launch.argtypes = [ctypes.c_int]
                L.lora_set_programmatic_launch.restype = ctypes.c_int
                L.lora_test_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
                L.lora_test_set_wait_limit_ns.restype = None
                _lib = L
    return _lib


def _check(rc: int):
    if rc != 0:
        raise MloraError(rc, lib().lora_error_string(rc).decode())


def _dev(t: Optional[torch.Tensor], what: str, dtype=None) -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor (libmlora has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _rows(t: torch.Tensor, what: str, dtype) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{what} must be a 2-D tensor with unit column stride")
    _dev(t, what, dtype)
    return t.stride(0)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class PoolHandle:
    """A pool descriptor plus references to the tensors it points at."""

    def __init__(self, p):
        self.src = p
        self.dtype = p.dtype
        paged = getattr(p, "pages", None) is not None
        s = mlora_pool()
        s.kind = MLORA_POOL_PAGED if paged else MLORA_POOL_STACKED
        s.dtype = _DT[p.dtype]
        s.num_slots, s.num_layers, s.r_max = int(p.num_slots), int(p.num_layers), int(p.r_max)
        s.d_in, s.d_out = int(p.d_in), int(p.d_out)
        if paged:
            s.pages = _dev(p.pages, "pages", p.dtype)
            s.page_elems, s.num_pages = int(p.pages.shape[1]), int(p.pages.shape[0])
            s.a_page_table = _dev(p.a_page_table, "a_page_table", torch.int32)
            s.b_page_table = _dev(p.b_page_table, "b_page_table", torch.int32)
            for t in (p.pages, p.a_page_table, p.b_page_table):
                assert t.is_contiguous()
        else:
            s.a_t = _dev(p.a_t, "a_t", p.dtype)
            s.b = _dev(p.b, "b", p.dtype)
            assert p.a_t.is_contiguous() and p.b.is_contiguous()
        s.rank = _dev(p.rank, "rank", torch.int32)
        s.scale = _dev(p.scale, "scale", torch.float32)
        self.struct = s
        self.ref = ctypes.pointer(s)


def make_pool(p) -> PoolHandle:
    return p if isinstance(p, PoolHandle) else PoolHandle(p)


def _i32(t: Optional[torch.Tensor], what: str) -> int:
    return _dev(t, what, torch.int32) if t is not None else 0


# ---------------------------------------------------------------------------------------------
# entry points (same names as the C ABI)


def lora_sgmv_shrink(v, x, pool, seg_offsets, seg_slot, layer, status=None, stream=None):
    h = make_pool(pool)
    _check(lib().lora_sgmv_shrink(_dev(v, "v", torch.float32), _dev(x, "x", h.dtype), _rows(x, "x", h.dtype), h.ref,
                                  _i32(seg_offsets, "seg_offsets"), _i32(seg_slot, "seg_slot"),
                                  int(seg_slot.numel()), int(x.shape[0]), int(layer), _i32(status, "status"),
                                  _stream(stream)))


def lora_sgmv_expand(y, v, pool, seg_offsets, seg_slot, layer, status=None, stream=None):
    h = make_pool(pool)
    _check(lib().lora_sgmv_expand(_dev(y, "y", h.dtype), _rows(y, "y", h.dtype), _dev(v, "v", torch.float32), h.ref,
                                  _i32(seg_offsets, "seg_offsets"), _i32(seg_slot, "seg_slot"),
                                  int(seg_slot.numel()), int(y.shape[0]), int(layer), _i32(status, "status"),
                                  _stream(stream)))


def lora_bgmv_shrink(v, x, pool, row_slot, layer, status=None, stream=None):
    h = make_pool(pool)
    _check(lib().lora_bgmv_shrink(_dev(v, "v", torch.float32), _dev(x, "x", h.dtype), _rows(x, "x", h.dtype), h.ref,
                                  _i32(row_slot, "row_slot"), int(x.shape[0]), int(layer), _i32(status, "status"),
                                  _stream(stream)))


def lora_bgmv_expand(y, v, pool, row_slot, layer, status=None, stream=None):
    h = make_pool(pool)
    _check(lib().lora_bgmv_expand(_dev(y, "y", h.dtype), _rows(y, "y", h.dtype), _dev(v, "v", torch.float32), h.ref,
                                  _i32(row_slot, "row_slot"), int(y.shape[0]), int(layer), _i32(status, "status"),
                                  _stream(stream)))


def lora_sgmv(y, x, pool, seg_offsets, seg_slot, layer, v_scratch, status=None, stream=None):
    h = make_pool(pool)
    _check(lib().lora_sgmv(_dev(y, "y", h.dtype), _rows(y, "y", h.dtype), _dev(x, "x", h.dtype),
                           _rows(x, "x", h.dtype), h.ref, _i32(seg_offsets, "seg_offsets"),
                           _i32(seg_slot, "seg_slot"), int(seg_slot.numel()), int(y.shape[0]), int(layer),
                           _dev(v_scratch, "v_scratch", torch.float32), _i32(status, "status"), _stream(stream)))


def lora_sgmv_noalloc(y, x, pool, seg_offsets, seg_slot, layer, status=None, stream=None):
    """lora_sgmv without a scratch argument, for callers that cannot allocate device memory; the
    library's built-in scratch holds num_rows * r_max <= NOALLOC_MAX_FLOATS fp32 values and is
    shared by all calls (order calls that could overlap on the GPU)."""
    h = make_pool(pool)
    _check(lib().lora_sgmv_noalloc(_dev(y, "y", h.dtype), _rows(y, "y", h.dtype), _dev(x, "x", h.dtype),
                                   _rows(x, "x", h.dtype), h.ref, _i32(seg_offsets, "seg_offsets"),
                                   _i32(seg_slot, "seg_slot"), int(seg_slot.numel()), int(y.shape[0]), int(layer),
                                   _i32(status, "status"), _stream(stream)))


def lora_bgmv(y, x, pool, row_slot, layer, v_scratch, status=None, stream=None):
    h = make_pool(pool)
    _check(lib().lora_bgmv(_dev(y, "y", h.dtype), _rows(y, "y", h.dtype), _dev(x, "x", h.dtype),
                           _rows(x, "x", h.dtype), h.ref, _i32(row_slot, "row_slot"), int(y.shape[0]), int(layer),
                           _dev(v_scratch, "v_scratch", torch.float32), _i32(status, "status"), _stream(stream)))


def lora_bgmv_ex(y, x, pool, row_slot, layer, v_scratch, flags: int = 0, status=None, stream=None):
    """lora_bgmv with launch flags (LAUNCH_GROUP_ROWS / LAUNCH_NO_GROUPING / LAUNCH_PROGRAMMATIC)."""
    h = make_pool(pool)
    _check(lib().lora_bgmv_ex(_dev(y, "y", h.dtype), _rows(y, "y", h.dtype), _dev(x, "x", h.dtype),
                              _rows(x, "x", h.dtype), h.ref, _i32(row_slot, "row_slot"), int(y.shape[0]), int(layer),
                              _dev(v_scratch, "v_scratch", torch.float32), int(flags), _i32(status, "status"),
                              _stream(stream)))


class Group:
    """A prepared lora_sgmv_grouped_ex call: the problem array is built once and reused."""

    def __init__(self, problems: Sequence[tuple], seg_offsets, seg_slot, num_rows: int, status=None,
                 programmatic: bool = False):
        """problems: (y, x, pool, layer, v_scratch) tuples sharing the rows' segments.
        programmatic: launch with programmatic dependent launch (LAUNCH_PROGRAMMATIC)."""
        if not 1 <= len(problems) <= MLORA_MAX_GROUP:
            raise ValueError(f"a group holds 1..{MLORA_MAX_GROUP} problems")
        self.handles = [make_pool(p[2]) for p in problems]
        self.arr = (mlora_problem * len(problems))()
        for q, ((y, x, _pool, layer, v), h) in enumerate(zip(problems, self.handles)):
            a = self.arr[q]
            a.y, a.ldy = _dev(y, "y", h.dtype), _rows(y, "y", h.dtype)
            a.x, a.ldx = _dev(x, "x", h.dtype), _rows(x, "x", h.dtype)
            a.pool = h.ref
            a.layer = int(layer)
            a.v_scratch = _dev(v, "v_scratch", torch.float32)
        self.keep = (problems, seg_offsets, seg_slot, status)
        self.n = len(problems)
        self.off, self.slot = _i32(seg_offsets, "seg_offsets"), _i32(seg_slot, "seg_slot")
        self.nseg, self.M = int(seg_slot.numel()), int(num_rows)
        self.status = _i32(status, "status")
        self.flags = LAUNCH_PROGRAMMATIC if programmatic else 0
        self.fn = lib().lora_sgmv_grouped_ex

    def __call__(self, stream=None):
        _check(self.fn(self.arr, self.n, self.off, self.slot, self.nseg, self.M, self.flags, self.status,
                       _stream(stream)))


def lora_sgmv_grouped(problems, seg_offsets, seg_slot, status=None, stream=None):
    num_rows = int(problems[0][0].shape[0])
    g = Group(problems, seg_offsets, seg_slot, num_rows, status)
    _check(lib().lora_sgmv_grouped(g.arr, g.n, g.off, g.slot, g.nseg, g.M, g.status, _stream(stream)))


def lora_sgmv_grouped_ex(problems, seg_offsets, seg_slot, flags: int = 0, status=None, stream=None):
    num_rows = int(problems[0][0].shape[0])
    g = Group(problems, seg_offsets, seg_slot, num_rows, status)
    _check(lib().lora_sgmv_grouped_ex(g.arr, g.n, g.off, g.slot, g.nseg, g.M, int(flags), g.status,
                                      _stream(stream)))


class CallSequence:
    """A prepared lora_sgmv_sequence call: the grouped calls of a whole step, issued by one call
    into the library (which launches them in order from native code)."""

    def __init__(self, groups: "Sequence[Group]", programmatic: bool = False, status=None):
        self.groups = list(groups)
        self.arr = (mlora_group * len(self.groups))()
        for a, g in zip(self.arr, self.groups):
            a.problems = ctypes.cast(g.arr, ctypes.POINTER(mlora_problem))
            a.num_problems = g.n
            a.seg_offsets, a.seg_slot = g.off, g.slot
            a.num_segments, a.num_rows = g.nseg, g.M
        self.flags = LAUNCH_PROGRAMMATIC if programmatic else 0
        self.status = _i32(status, "status")
        self.fn = lib().lora_sgmv_sequence

    def __call__(self, stream=None):
        _check(self.fn(self.arr, len(self.groups), self.flags, self.status, _stream(stream)))


def lora_sgmv_sequence(groups, programmatic: bool = False, status=None, stream=None):
    """groups: prepared Group objects (each a grouped call over its rows), issued in order."""
    CallSequence(groups, programmatic, status)(stream)


def launch_count() -> int:
    return int(lib().lora_launch_count())


def lora_set_programmatic_launch(enable: bool) -> bool:
    """Programmatic dependent launch for the calling thread's later calls (see include/mlora.h);
    returns this thread's previous setting."""
    return bool(lib().lora_set_programmatic_launch(1 if enable else 0))


def lora_test_set_wait_limit_ns(limit_ns: int) -> None:
    """Testing hook: time limit of the CUDA-core kernels' waits for this thread's later calls
    (0 = the default). Only the tests of the time-out path use it."""
    lib().lora_test_set_wait_limit_ns(int(limit_ns))


def abi_version() -> int:
    return int(lib().lora_abi_version())
