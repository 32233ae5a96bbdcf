"""The C-ABI library on the host: it loads, exports every declared symbol, and rejects
host-detectable bad arguments with the documented codes before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import adapter_gemv_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(m.LIB_PATH):
        from adapter_gemv_gb300 import build
        build.build()
    return m.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mlora.h")).read()
    return sorted(set(re.findall(r"MLORA_API\s+[\w\s\*]*?\b(lora_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("lora_sgmv_shrink", "lora_sgmv_expand", "lora_bgmv_shrink", "lora_bgmv_expand"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in mlora.h but not exported"
    assert L.lora_abi_version() == 1


def test_binding_names_match_the_abi():
    for name in declared_functions():
        if name not in ("lora_error_string", "lora_abi_version", "lora_launch_count"):
            assert callable(getattr(m, name)), f"binding lacks {name}"


def _pool(**kw):
    p = m.mlora_pool()
    p.kind, p.dtype, p.num_slots, p.num_layers, p.r_max, p.d_in, p.d_out = 0, 0, 4, 2, 16, 64, 64
    # fake but aligned device-looking addresses: validation only inspects them, nothing runs
    p.a_t, p.b, p.rank, p.scale = 0x10000, 0x20000, 0x30000, 0x40000
    for k, v in kw.items():
        setattr(p, k, v)
    return p


X, Y, V, OFF, SLOT = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000


def shrink(L, pool, x=X, ldx=64, v=V, off=OFF, slot=SLOT, nseg=2, rows=8, layer=0):
    return L.lora_sgmv_shrink(v, x, ldx, ctypes.byref(pool), off, slot, nseg, rows, layer, None, None)


def expand(L, pool, y=Y, ldy=64, v=V, off=OFF, slot=SLOT, nseg=2, rows=8, layer=0):
    return L.lora_sgmv_expand(y, ldy, v, ctypes.byref(pool), off, slot, nseg, rows, layer, None, None)


@pytest.mark.parametrize("case,code", [
    (dict(pool=None), m.ERR_NULL),
    (dict(x=0), m.ERR_NULL),
    (dict(v=0), m.ERR_NULL),
    (dict(off=0), m.ERR_NULL),
    (dict(slot=0), m.ERR_NULL),
    (dict(rows=-1), m.ERR_SHAPE),
    (dict(nseg=-1), m.ERR_SHAPE),
    (dict(layer=2), m.ERR_SHAPE),
    (dict(layer=-1), m.ERR_SHAPE),
    (dict(ldx=56), m.ERR_SHAPE),
    (dict(ldx=68), m.ERR_ALIGN),
    (dict(x=X + 8), m.ERR_ALIGN),
    (dict(v=V + 2), m.ERR_ALIGN),
    (dict(off=OFF + 2), m.ERR_ALIGN),
    (dict(pool_kw=dict(dtype=7)), m.ERR_DTYPE),
    (dict(pool_kw=dict(r_max=0)), m.ERR_SHAPE),
    (dict(pool_kw=dict(r_max=129)), m.ERR_SHAPE),
    (dict(pool_kw=dict(d_in=60)), m.ERR_ALIGN),
    (dict(pool_kw=dict(d_in=0)), m.ERR_SHAPE),
    (dict(pool_kw=dict(num_slots=0)), m.ERR_SHAPE),
    (dict(pool_kw=dict(a_t=0)), m.ERR_NULL),
    (dict(pool_kw=dict(a_t=0x10008)), m.ERR_ALIGN),
    (dict(pool_kw=dict(rank=0)), m.ERR_NULL),
    (dict(pool_kw=dict(kind=5)), m.ERR_POOL),
    (dict(pool_kw=dict(kind=1, pages=0x50000, page_elems=0, num_pages=10, a_page_table=0x60000,
                       b_page_table=0x70000)), m.ERR_POOL),  # empty pages (shorter pages than d are fine)
    (dict(pool_kw=dict(kind=1, pages=0x50000, page_elems=68, num_pages=10, a_page_table=0x60000,
                       b_page_table=0x70000)), m.ERR_ALIGN),
    (dict(pool_kw=dict(kind=1, pages=0, page_elems=64, num_pages=10, a_page_table=0x60000,
                       b_page_table=0x70000)), m.ERR_NULL),
])
def test_shrink_rejects_bad_arguments(L, case, code):
    case = dict(case)
    pool = None if case.pop("pool", 1) is None else _pool(**case.pop("pool_kw", {}))
    if pool is None:
        rc = L.lora_sgmv_shrink(V, X, 64, None, OFF, SLOT, 2, 8, 0, None, None)
    else:
        rc = shrink(L, pool, **case)
    assert rc == code
    assert L.lora_error_string(rc)


def test_expand_rejects_bad_arguments(L):
    assert expand(L, _pool(), y=0) == m.ERR_NULL
    assert expand(L, _pool(), ldy=60) == m.ERR_SHAPE
    assert expand(L, _pool(), y=Y + 4) == m.ERR_ALIGN
    assert expand(L, _pool(b=0)) == m.ERR_NULL
    # a pool without A is fine for the expand (it never reads A)
    assert expand(L, _pool(a_t=0), rows=0) == 0


def test_zero_rows_is_a_noop_without_launch(L):
    before = L.lora_launch_count()
    assert shrink(L, _pool(), rows=0, nseg=0) == 0
    assert expand(L, _pool(), rows=0, nseg=0) == 0
    assert L.lora_launch_count() == before


def test_grouped_limits(L):
    arr = (m.mlora_problem * 9)()
    assert L.lora_sgmv_grouped(arr, 9, OFF, SLOT, 1, 8, None, None) == m.ERR_SHAPE
    assert L.lora_sgmv_grouped(arr, 0, OFF, SLOT, 1, 8, None, None) == m.ERR_SHAPE
    assert L.lora_sgmv_grouped(None, 1, OFF, SLOT, 1, 8, None, None) == m.ERR_NULL
    p0, p1 = _pool(), _pool(dtype=1)
    arr = (m.mlora_problem * 2)()
    for q, p in enumerate((p0, p1)):
        arr[q].y, arr[q].ldy, arr[q].x, arr[q].ldx, arr[q].v_scratch = Y, 64, X, 64, V
        arr[q].pool = ctypes.pointer(p)
    assert L.lora_sgmv_grouped(arr, 2, OFF, SLOT, 1, 8, None, None) == m.ERR_DTYPE
    assert L.lora_sgmv_grouped_ex(arr, 2, OFF, SLOT, 1, 8, m.LAUNCH_PROGRAMMATIC, None, None) == m.ERR_DTYPE
    # unknown launch flags are refused before anything else is looked at
    assert L.lora_sgmv_grouped_ex(arr, 1, OFF, SLOT, 1, 8, 2, None, None) == m.ERR_SHAPE


def test_programmatic_launch_setting_is_per_thread(L):
    """lora_set_programmatic_launch changes the calling thread's setting only."""
    import threading
    assert L.lora_set_programmatic_launch(1) == 0
    seen = []
    t = threading.Thread(target=lambda: seen.append(L.lora_set_programmatic_launch(0)))
    t.start()
    t.join()
    assert seen == [0], "a new thread inherited another thread's setting"
    assert L.lora_set_programmatic_launch(0) == 1


def test_binding_refuses_cpu_tensors():
    import torch
    import workloads as W
    w = W.tiny_sgmv()
    with pytest.raises(ValueError, match="CUDA"):
        m.make_pool(w.ops[0].pool)
