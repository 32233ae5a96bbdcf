"""GPU parity: libmlora (through the C ABI) against the fp64 oracle, element by element.

Covers the five workloads at their full sizes (sampled rows where the oracle would be slow),
in the launch configuration the bench times (grouped fused calls of a decode step), plus the
two-launch and fused forms of SGMV and BGMV. Tolerance: |gpu - oracle| <= 1e-2 (1 + |oracle|).
"""
import numpy as np
import pytest
import torch

import adapter_gemv_gb300 as m
import workloads as W
from adapter_gemv_gb300.plan import StepPlan
from gpu_util import bits, check_op, run_op

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not __import__("os").path.exists(m.LIB_PATH):
        from adapter_gemv_gb300 import build
        build.build()
    return torch.device("cuda:0")


def status_of(dev):
    return torch.zeros(1, dtype=torch.int32, device=dev)


@pytest.mark.parametrize("mode", ["two_phase", "fused"])
def test_tiny_sgmv_fp16(dev, mode):
    w = W.tiny_sgmv(device=dev)
    st = status_of(dev)
    y, v = run_op(w.ops[0], w.batch, "sgmv", mode, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    check_op(w.ops[0], w.batch, "sgmv", y, v, what=f"tiny sgmv {mode}")


@pytest.mark.parametrize("mode", ["two_phase", "fused"])
def test_bgmv_decode_q_proj(dev, mode):
    w = W.bgmv_decode_q(device=dev)
    st = status_of(dev)
    y, v = run_op(w.ops[0], w.batch, "bgmv", mode, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    check_op(w.ops[0], w.batch, "bgmv", y, v, what=f"bgmv q_proj {mode}")


@pytest.mark.parametrize("dist", ["distinct", "uniform", "skewed", "identical"])
def test_decode_step_7b_as_benched(dev, dist):
    """The whole decode step (7 projections x 32 layers, r = 16, bs 32) through the grouped
    fused calls the bench times; every op of layers 0, 17 and 31 checked on every row."""
    w = W.sgmv_decode_7b(device=dev, dist=dist)
    st = status_of(dev)
    before = {id(op): bits(op.y) for op in w.ops if op.layer in (0, 17, 31)}
    plan = StepPlan(w.ops, w.batch, st)
    assert plan.launches == 4 * 32
    plan()
    torch.cuda.synchronize()
    assert st.item() == 0
    for op in w.ops:
        if op.layer in (0, 17, 31):
            check_op(op, w.batch, "sgmv", op.y, y_before=before[id(op)], what=f"{dist} {op.name} L{op.layer}")


def ragged_rank16_step(dev, dtype, seed, page_elems=None):
    """Chained one-row problems whose pools have r_max 16: ranks 4/8/13/16 (padding rows hold NaN),
    d_in slices that end inside a pass of A (2056, 11008), a d_out that is not a multiple of the
    split (1000), a B much larger than A (up), two rows without adapter. page_elems: paged pools
    with pages of that many elements (0: one page per vector), else stacked pools."""
    g = W.generator(seed, dev)
    rng = np.random.default_rng(seed)
    projs = [W.Projection("q", 4096, 4096), W.Projection("k", 4096, 1024), W.Projection("up", 4096, 11008),
             W.Projection("o", 2056, 1000), W.Projection("down", 11008, 4096)]
    num_slots, M = 24, 20
    ranks = rng.choice(np.array([4, 8, 13, 16], np.int32), size=num_slots)
    ranks[:4] = [4, 8, 13, 16]
    if page_elems is None:
        pools = {p.name: W.stacked_pool(num_slots=num_slots, num_layers=2, r_max=16, d_in=p.d_in, d_out=p.d_out,
                                        dtype=dtype, gen=g, device=dev, ranks=ranks) for p in projs}
    else:
        pools = {p.name: W.paged_pool(num_slots=num_slots, num_layers=2, r_max=16, d_in=p.d_in, d_out=p.d_out,
                                      dtype=dtype, gen=g, device=dev, rng=rng, ranks=ranks,
                                      page_elems=page_elems or None) for p in projs}
    slots = np.r_[[-1, -1], rng.permutation(num_slots)[:M - 2]].astype(np.int32)
    slots.sort(kind="stable")
    batch = W.batch_from_slots(slots, sgmv=True).to(dev)
    x_qk = W.normal((M, 4096), 1.0, dtype, g, dev)
    x_o = W.normal((M, 2056), 1.0, dtype, g, dev)
    x_down = W.normal((M, 11008), 1.0, dtype, g, dev)
    ops = []
    for layer in (0, 1):
        for p in projs:
            x = x_qk if p.name in ("q", "k", "up") else x_o if p.name == "o" else x_down
            ops.append(W.Op(p.name, pools[p.name], layer, x, W.uniform((M, p.d_out), -1, 1, dtype, g, dev)))
    return batch, ops


@pytest.mark.parametrize("dtype,page_elems", [(torch.bfloat16, None), (torch.float16, None),
                                              (torch.bfloat16, 0), (torch.float16, 4096)])
def test_chained_rank16_step_ragged(dev, dtype, page_elems):
    """A step plan (programmatic dependent launch) over ragged rank <= 16 problems: every op on
    every row against the oracle; rows without adapter keep their bits."""
    batch, ops = ragged_rank16_step(dev, dtype, seed=11, page_elems=page_elems)
    st = status_of(dev)
    before = {id(op): bits(op.y) for op in ops}
    plan = StepPlan(ops, batch, st)
    plan()
    torch.cuda.synchronize()
    assert st.item() == 0
    for op in ops:
        check_op(op, batch, "sgmv", op.y, y_before=before[id(op)], what=f"ragged {op.name} L{op.layer}")


def test_chained_rank16_bgmv(dev):
    """BGMV calls issued back to back with programmatic dependent launch on (rows unsorted, two
    without adapter), ranks below r_max: the same results as the oracle."""
    batch, ops = ragged_rank16_step(dev, torch.bfloat16, seed=12)
    rs = batch.row_slot.cpu().numpy()[np.random.default_rng(3).permutation(batch.M)]
    bb = W.batch_from_slots(rs, sgmv=False).to(dev)
    st = status_of(dev)
    before = {id(op): bits(op.y) for op in ops}
    handles = {id(op.pool): m.make_pool(op.pool) for op in ops}
    v = torch.empty((bb.M, 16), dtype=torch.float32, device=dev)
    prev = m.lora_set_programmatic_launch(True)
    try:
        for op in ops:
            m.lora_bgmv(op.y, op.x, handles[id(op.pool)], bb.row_slot, op.layer, v, st)
    finally:
        m.lora_set_programmatic_launch(prev)
    torch.cuda.synchronize()
    assert st.item() == 0
    for op in ops:
        check_op(op, bb, "bgmv", op.y, y_before=before[id(op)], what=f"bgmv chained {op.name} L{op.layer}")


@pytest.mark.parametrize("mode", ["two_phase", "fused"])
def test_decode_7b_single_ops(dev, mode):
    w = W.sgmv_decode_7b(device=dev, dist="skewed", num_layers=2, layers=[1])
    for op in w.ops:
        y, v = run_op(op, w.batch, "sgmv", mode)
        torch.cuda.synchronize()
        check_op(op, w.batch, "sgmv", y, v, what=f"{op.name} {mode}")


def prefill_sample_rows(batch, per_segment=4, seed=0):
    rng = np.random.default_rng(seed)
    off = batch.seg_offsets.cpu().numpy()
    rows = []
    for t in range(len(off) - 1):
        lo, hi = off[t], off[t + 1]
        picks = {lo, hi - 1, min(hi - 1, lo + 127), min(hi - 1, lo + 128)}
        picks |= set(rng.integers(lo, hi, per_segment).tolist())
        rows.extend(sorted(picks))
    return np.array(rows)


@pytest.mark.parametrize("mode", ["two_phase", "fused"])
def test_prefill_13b_sampled(dev, mode):
    """8 prompts of U[128, 2048] rows, r = 64, all 7 Llama-2-13B projections; the oracle runs
    on sampled rows (segment ends, rows on both sides of a 128-row boundary, random rows)."""
    w = W.sgmv_prefill_13b(device=dev)
    rows = prefill_sample_rows(w.batch)
    st = status_of(dev)
    for op in w.ops:
        y, v = run_op(op, w.batch, "sgmv", mode, st)
        torch.cuda.synchronize()
        check_op(op, w.batch, "sgmv", y, v, rows=rows, what=f"prefill {op.name} {mode}")
    assert st.item() == 0


@pytest.mark.parametrize("mode", ["two_phase", "fused"])
def test_paged_hetero_rank_70b(dev, mode):
    """2000 adapters with ranks {8,16,32,64} in permuted pages (free pages hold NaN), 256 rows
    Zipf(1.2), BGMV, Llama-2-70B q_proj 8192 -> 8192: every row against the oracle."""
    w = W.paged_decode_70b(device=dev)
    st = status_of(dev)
    y, v = run_op(w.ops[0], w.batch, "bgmv", mode, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    check_op(w.ops[0], w.batch, "bgmv", y, v, what=f"paged 70b {mode}")


def test_mixed_prefill_decode_13b_sampled(dev):
    """The bench's mixed batch (Punica's batch layout: 3 prompts of 300-2000 rows, then 64 one-row
    decode segments on their own adapters; Llama-2-13B shapes, r = 64), all 7 projections through
    the fused call: the prompts on the tensor cores, the decode rows streamed on the CUDA cores
    (one cluster per row). The oracle checks every decode row and rows at both sides of every
    prompt's 128-row blocks."""
    w = W.mixed_prefill_decode_13b(device=dev)
    off = w.batch.seg_offsets.cpu().numpy()
    rows = np.unique(np.r_[prefill_sample_rows(W.Batch(int(off[3]), w.batch.row_slot[:off[3]],
                                                       w.batch.seg_offsets[:4], w.batch.seg_slot[:3])),
                           np.arange(off[3], w.batch.M)])
    st = status_of(dev)
    for op in w.ops:
        before = m.launch_count()
        y, _ = run_op(op, w.batch, "sgmv", "fused", st)
        torch.cuda.synchronize()
        assert m.launch_count() - before == 3, "the prompts did not run on the tensor cores"
        check_op(op, w.batch, "sgmv", y, rows=rows, what=f"mixed 13B {op.name}")
    assert st.item() == 0


def test_paged_70b_2048_rows_grouped_sampled(dev):
    """2048 rows over the 2000-adapter paged pool (the adapters used exceed L2): lora_bgmv groups
    the rows on the device and streams each row through one CTA; every 8th row of the grouped and
    of the ungrouped call against the oracle."""
    w = W.paged_decode_70b(device=dev, M=2048)
    op = w.ops[0]
    h = m.make_pool(op.pool)
    st = status_of(dev)
    y_g, y_p = op.y.clone(), op.y.clone()
    v = torch.empty((2048, op.pool.r_max), dtype=torch.float32, device=dev)
    m.lora_bgmv_ex(y_g, op.x, h, w.batch.row_slot, 0, v, m.LAUNCH_GROUP_ROWS, st)
    m.lora_bgmv_ex(y_p, op.x, h, w.batch.row_slot, 0, v, m.LAUNCH_NO_GROUPING, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    check_op(op, w.batch, "bgmv", y_g, rows=np.arange(0, 2048, 8), what="paged 70B 2048 rows grouped")
    check_op(op, w.batch, "bgmv", y_p, rows=np.arange(3, 2048, 8), what="paged 70B 2048 rows ungrouped")
