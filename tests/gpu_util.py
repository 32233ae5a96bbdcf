"""Helpers shared by the GPU parity tests: moving workloads to the oracle, running the C ABI,
and the comparison rule.

Tolerance (fp32 accumulation, bf16/fp16 I/O): |gpu - oracle| <= 1e-2 * (1 + |oracle|) per
element of y and of v; routing (which rows change, which slot a row used) is bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import adapter_gemv_gb300 as m
import oracle
import workloads as W

TOL = 1e-2


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def odt(dtype) -> int:
    return oracle.DTYPE_BF16 if dtype == torch.bfloat16 else oracle.DTYPE_FP16


_pool_cache = {}


def oracle_pool(p: W.Pool) -> oracle.Pool:
    key = id(p)
    if key in _pool_cache and _pool_cache[key][0] is p:
        return _pool_cache[key][1]
    common = dict(dtype=odt(p.dtype), num_slots=p.num_slots, num_layers=p.num_layers, r_max=p.r_max, d_in=p.d_in,
                  d_out=p.d_out, rank=p.rank.cpu().numpy(), scale=p.scale.cpu().numpy())
    if p.paged:
        op = oracle.Pool(**common, pages=bits(p.pages), a_page_table=p.a_page_table.cpu().numpy(),
                         b_page_table=p.b_page_table.cpu().numpy())
    else:
        op = oracle.Pool(**common, a_t=bits(p.a_t), b=bits(p.b))
    _pool_cache[key] = (p, op)
    return op


def assert_close(got: np.ndarray, want: np.ndarray, what: str):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert got.shape == want.shape
    assert np.all(np.isfinite(want)), f"{what}: oracle produced non-finite values"
    err = np.abs(got - want)
    bad = ~(err <= TOL * (1.0 + np.abs(want)))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; first {idx.tolist()}: "
                             f"got {got[tuple(idx[0])]}, want {want[tuple(idx[0])]}")


def oracle_op(op: W.Op, batch: W.Batch, form: str, rows=None, y_in: np.ndarray = None):
    """Oracle y' (uint16), v (fp64) and status for one op, optionally on sampled rows."""
    pool = oracle_pool(op.pool)
    x, y = bits(op.x), bits(op.y) if y_in is None else y_in
    if form == "sgmv":
        y_o, v_o, _, st = oracle.sgmv(pool, op.layer, x, y, batch.seg_offsets.cpu().numpy(),
                                      batch.seg_slot.cpu().numpy(), rows=rows)
    else:
        y_o, v_o, _, st = oracle.bgmv(pool, op.layer, x, y, batch.row_slot.cpu().numpy(), rows=rows)
    return y_o, v_o, st


def check_op(op: W.Op, batch: W.Batch, form: str, y_gpu: torch.Tensor, v_gpu: torch.Tensor = None, rows=None,
             y_before: np.ndarray = None, what: str = ""):
    """Compare one op's GPU result with the oracle (all rows, or the sampled `rows`).
    Rows without an adapter must keep their exact input bits."""
    y_before = bits(op.y) if y_before is None else y_before
    y_o, v_o, st = oracle_op(op, batch, form, rows, y_before)
    assert st == 0, f"{what}: oracle reports status {st}"
    dt = odt(op.pool.dtype)
    got_bits = bits(y_gpu)
    sel = np.arange(batch.M) if rows is None else np.asarray(rows)
    slots = batch.row_slot.cpu().numpy()
    adapted = sel[slots[sel] >= 0]
    skipped = np.flatnonzero(slots < 0)
    assert np.array_equal(got_bits[skipped], y_before[skipped]), f"{what}: a slot -1 row changed"
    if adapted.size:
        assert_close(oracle.decode(got_bits[adapted], dt), oracle.decode(y_o[adapted], dt), f"{what} y")
        if v_gpu is not None:
            ranks = op.pool.rank.cpu().numpy()
            vg = v_gpu.double().cpu().numpy()
            for i in adapted:
                r = ranks[slots[i]]
                assert_close(vg[i, :r], v_o[i, :r], f"{what} v row {i}")


def new_v(M, r_max, device):
    return torch.full((M, r_max), float("nan"), dtype=torch.float32, device=device)


def run_op(op: W.Op, batch: W.Batch, form: str, mode: str, status=None):
    """Run one op through the C ABI on a copy of y. mode: 'two_phase' or 'fused'.
    Returns (y', v or None)."""
    dev = op.x.device
    pool = m.make_pool(op.pool)
    y = op.y.clone()
    v = new_v(batch.M, op.pool.r_max, dev)
    if form == "sgmv":
        if mode == "two_phase":
            m.lora_sgmv_shrink(v, op.x, pool, batch.seg_offsets, batch.seg_slot, op.layer, status)
            m.lora_sgmv_expand(y, v, pool, batch.seg_offsets, batch.seg_slot, op.layer, status)
            return y, v
        m.lora_sgmv(y, op.x, pool, batch.seg_offsets, batch.seg_slot, op.layer, v, status)
        return y, None
    if mode == "two_phase":
        m.lora_bgmv_shrink(v, op.x, pool, batch.row_slot, op.layer, status)
        m.lora_bgmv_expand(y, v, pool, batch.row_slot, op.layer, status)
        return y, v
    m.lora_bgmv(y, op.x, pool, batch.row_slot, op.layer, v, status)
    return y, None
