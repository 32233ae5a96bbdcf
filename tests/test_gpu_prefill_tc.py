"""Tensor-core prefill path against the oracle: long SGMV segments whose full 128-row blocks run
on tcgen05 kernels and whose tails run on the CUDA-core kernels. Segment lengths around the
128-row boundary, empty and -1 segments, K and N extents that are not multiples of the tile,
ranks below the padded rank (padding rows hold NaN), bf16 and fp16 pools, fp16 shrink results
beyond the fp16 range, every row compared."""
import numpy as np
import pytest
import torch

import adapter_gemv_gb300 as m
import workloads as W
from gpu_util import check_op, new_v

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    if not os.path.exists(m.LIB_PATH):
        from adapter_gemv_gb300 import build
        build.build()
    return torch.device("cuda:0")


CASES = [
    # r_max, ranks, d_in, d_out, segment lengths, segment slots
    (16, [16, 8, 1, 16], 264, 200, [128, 300, 0, 129, 5, 256], [0, 1, 2, -1, 3, 1]),
    (64, [64, 64, 33, 64], 5120, 640, [255, 130, 384], [2, 0, 1]),
    (40, [40, 17, 40], 512, 4104, [200, 128, 129], [1, 0, 2]),
    (128, [128, 96], 1032, 1104, [256, 131], [0, 1]),
    # segments around the 32-row threshold: partial tensor-core tiles next to CUDA-core segments
    (16, [16, 5, 16], 320, 328, [31, 32, 33, 64, 127, 200, 1], [0, 1, 2, 0, 1, 2, -1]),
    # many 128-row blocks: one CTA per block, no K split
    (16, [16, 16], 256, 136, [128 * 60 + 7, 128 * 41], [0, 1]),
    # few blocks: K split over a cluster of 4 (5120 / 128 K blocks do not divide evenly)
    (64, [64, 40], 5120, 264, [384, 131, 2], [0, 1, 1]),
]


def run_tc(dev, op, batch, mode, r_max):
    """One op through the tensor-core path (two launches or fused); checks that it ran there."""
    M = batch.M
    h = m.make_pool(op.pool)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    y = op.y.clone()
    v = new_v(M, r_max, dev)
    before = m.launch_count()
    if mode == "two_phase":
        m.lora_sgmv_shrink(v, op.x, h, batch.seg_offsets, batch.seg_slot, op.layer, st)
        m.lora_sgmv_expand(y, v, h, batch.seg_offsets, batch.seg_slot, op.layer, st)
        launches = 4  # tensor-core shrink + tails, tensor-core expand + tails
    else:
        m.lora_sgmv(y, op.x, h, batch.seg_offsets, batch.seg_slot, op.layer, v, st)
        launches = 3
    torch.cuda.synchronize()
    assert m.launch_count() - before == launches, "the tensor-core path did not run"
    assert st.item() == 0
    return y, v


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"r{c[0]}-{c[2]}x{c[3]}-M{sum(c[4])}")
@pytest.mark.parametrize("mode", ["two_phase", "fused"])
def test_prefill_tensor_core_path(dev, case, mode, dtype):
    r_max, ranks, d_in, d_out, lens, slots = case
    g = W.generator(7, dev)
    pool = W.stacked_pool(num_slots=len(ranks), num_layers=2, r_max=r_max, d_in=d_in, d_out=d_out,
                          dtype=dtype, gen=g, device=dev, ranks=ranks)
    batch = W.batch_from_segments(lens, slots).to(dev)
    M = batch.M
    x = W.normal((M, d_in), 1.0, dtype, g, dev)
    y0 = W.uniform((M, d_out), -1, 1, dtype, g, dev)
    op = W.Op("p", pool, 1, x, y0)
    y, v = run_tc(dev, op, batch, mode, r_max)
    check_op(op, batch, "sgmv", y, v if mode == "two_phase" else None, what=f"tc {mode}")


@pytest.mark.parametrize("mode", ["two_phase", "fused"])
def test_prefill_fp16_shrink_results_beyond_fp16_range(dev, mode):
    """fp16 pool whose shrink results v reach past 65504 (x std 4096, A std 8 / sqrt(d_in), so v
    has std 32768): the tensor-core expand stores each row of V scaled by a power of two and
    scales the row's sums back, so y still matches the oracle."""
    d_in, d_out, r = 1024, 512, 32
    g = W.generator(9, dev)
    pool = W.stacked_pool(num_slots=2, num_layers=1, r_max=r, d_in=d_in, d_out=d_out, dtype=torch.float16, gen=g,
                          device=dev, a_var=64.0 / d_in, b_var=1e-4)
    batch = W.batch_from_segments([256, 130], [0, 1]).to(dev)
    x = W.normal((batch.M, d_in), 4096.0 ** 2, torch.float16, g, dev)
    y0 = W.uniform((batch.M, d_out), -1, 1, torch.float16, g, dev)
    assert torch.isfinite(x).all()
    op = W.Op("big", pool, 0, x, y0)
    y, v = run_tc(dev, op, batch, mode, r)
    if mode == "two_phase":
        assert v.abs().max().item() > 65504.0, "the case does not reach past the fp16 range"
    assert torch.isfinite(y).all()
    check_op(op, batch, "sgmv", y, v if mode == "two_phase" else None, what=f"fp16 large v {mode}")


def test_prefill_bad_offsets_launch_tc_but_write_nothing(dev):
    g = W.generator(8, dev)
    pool = W.stacked_pool(num_slots=2, num_layers=1, r_max=16, d_in=128, d_out=128, dtype=torch.bfloat16, gen=g,
                          device=dev)
    M = 512
    x = W.normal((M, 128), 1.0, torch.bfloat16, g, dev)
    y = W.uniform((M, 128), -1, 1, torch.bfloat16, g, dev)
    y_ref = y.clone()
    off = torch.tensor([0, 256, 500], dtype=torch.int32, device=dev)  # ends at 500 != 512
    slot = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    m.lora_sgmv(y, x, m.make_pool(pool), off, slot, 0, new_v(M, 16, dev), st)
    torch.cuda.synchronize()
    assert st.item() == m.STATUS_BAD_OFFSETS
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


def mixed_batch(dev, dtype, seed, d_in, d_out, r_max=16):
    """Punica's batch layout: the prompts of new requests first (one segment and adapter each),
    then one-row decode segments (an adapter per request, some sharing a prompt's adapter, some
    without adapter)."""
    rng = np.random.default_rng(seed)
    g = W.generator(seed, dev)
    prompts = [300, 1200, 2000]
    num_slots = 40
    ranks = rng.integers(1, r_max + 1, num_slots).astype(np.int32)
    pool = W.stacked_pool(num_slots=num_slots, num_layers=1, r_max=r_max, d_in=d_in, d_out=d_out, dtype=dtype,
                          gen=g, device=dev, ranks=ranks)
    decode_slots = rng.integers(-1, num_slots, 64)
    decode_slots[:3] = [0, 1, 2]  # the prompts' adapters again, in decode rows
    lens = np.r_[prompts, np.ones(64, np.int64)]
    slots = np.r_[[0, 1, 2], decode_slots].astype(np.int32)
    batch = W.batch_from_segments(lens, slots).to(dev)
    x = W.normal((batch.M, d_in), 1.0, dtype, g, dev)
    y = W.uniform((batch.M, d_out), -1, 1, dtype, g, dev)
    return pool, batch, x, y


@pytest.mark.parametrize("form", ["two_phase", "fused", "grouped"])
def test_mixed_prefill_and_decode_batch(dev, form):
    """Three prompts of 300-2000 rows and 64 one-row decode segments in one SGMV batch: the
    prompts run on the tensor-core kernels, the decode rows on the CUDA-core kernel, and every
    row matches the oracle."""
    pool, batch, x, y0 = mixed_batch(dev, torch.bfloat16, 17, 1024, 1032)
    h = m.make_pool(pool)
    M = batch.M
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    before = m.launch_count()
    if form == "grouped":
        ys = [y0.clone(), y0.clone()]
        m.lora_sgmv_grouped([(ys[q], x, h, 0, new_v(M, 16, dev)) for q in range(2)], batch.seg_offsets,
                            batch.seg_slot, st)
        launches, outs, v = 2 * 2 + 1, ys, None
    else:
        op = W.Op("mixed", pool, 0, x, y0)
        y, v = run_tc(dev, op, batch, form, 16)
        launches, outs = 0, [y]
    torch.cuda.synchronize()
    if form == "grouped":
        assert m.launch_count() - before == launches, "the grouped call did not use the tensor-core kernels"
    assert st.item() == 0
    op = W.Op("mixed", pool, 0, x, y0)
    for y in outs:
        check_op(op, batch, "sgmv", y, v if form == "two_phase" else None, what=f"mixed batch {form}")


def test_mixed_batch_side_stream_and_graphs(dev):
    """The CUDA-core launch of a mixed batch runs on a second stream, beside the tensor-core
    kernels (forked from the caller's stream, joined back). A thread whose first such call is being
    captured in a CUDA graph keeps every launch on the caller's stream; a thread that has its second
    stream forks inside a capture too. Eager, captured-serial and captured-forked calls give the
    same bits, and the oracle's results."""
    import threading
    pool, batch, x, y0 = mixed_batch(dev, torch.bfloat16, 23, 1024, 1032)
    h = m.make_pool(pool)
    M = batch.M

    def call(y, v, st):
        m.lora_sgmv(y, x, h, batch.seg_offsets, batch.seg_slot, 0, v, st)

    def captured(out):
        y, v = y0.clone(), new_v(M, 16, dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            call(y, v, st)
        y.copy_(y0)
        g.replay()
        torch.cuda.synchronize()
        out.append((y.clone(), st.item()))

    fresh = []  # a new host thread: the first call is captured (no second stream yet)
    t = threading.Thread(target=captured, args=(fresh,))
    t.start()
    t.join()
    assert len(fresh) == 1, "the capture in a new thread failed"
    y_e, v_e = y0.clone(), new_v(M, 16, dev)  # eager, forked
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    call(y_e, v_e, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    forked = []
    captured(forked)  # this thread has its second stream now: the capture forks
    for y, status in fresh + forked:
        assert status == 0
        assert torch.equal(y, y_e), "a captured call differs from the eager call"
    check_op(W.Op("mixed", pool, 0, x, y0), batch, "sgmv", y_e, None, what="mixed batch, side stream")


# Paged pools on the tensor cores (S-LoRA "Unified Paging", MBGMM-style prefill over the pages):
# the A^T / B rows of a tile are gathered from their pages; pages as long as a vector, and pages
# shorter than a vector (one H-vector per page: 13B MLP rows of 13824 span three 5120-element
# pages), with ranks differing per adapter.
PAGED_CASES = [
    # r_max, ranks, d_in, d_out, segment lengths, segment slots, page_elems (None: max(d_in, d_out))
    (64, [64, 8, 33, 16], 5120, 640, [255, 130, 384, 3], [2, 0, 1, 3], None),
    (64, [64, 8, 33, 16], 5120, 13824, [200, 129, 300], [1, 3, 0], 5120),
    (32, [32, 1, 17], 13824, 5120, [128, 257, 5], [0, 2, 1], 5120),
    (16, [16, 5, 16], 1024, 328, [31, 33, 64, 127, 200, 1], [0, 1, 2, 0, 1, 2], 96),
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("case", PAGED_CASES, ids=lambda c: f"r{c[0]}-{c[2]}x{c[3]}-M{sum(c[4])}-pages{c[6]}")
@pytest.mark.parametrize("mode", ["two_phase", "fused"])
def test_prefill_tensor_core_path_paged(dev, case, mode, dtype):
    r_max, ranks, d_in, d_out, lens, slots, pe = case
    g = W.generator(13, dev)
    rng = np.random.default_rng(13)
    pool = W.paged_pool(num_slots=len(ranks), num_layers=2, r_max=r_max, d_in=d_in, d_out=d_out, dtype=dtype,
                        gen=g, device=dev, rng=rng, ranks=ranks, page_elems=pe)
    batch = W.batch_from_segments(lens, slots).to(dev)
    x = W.normal((batch.M, d_in), 1.0, dtype, g, dev)
    y0 = W.uniform((batch.M, d_out), -1, 1, dtype, g, dev)
    op = W.Op("p", pool, 1, x, y0)
    y, v = run_tc(dev, op, batch, mode, r_max)
    check_op(op, batch, "sgmv", y, v if mode == "two_phase" else None, what=f"paged tc {mode}")


def test_prefill_paged_13b_every_row(dev):
    """Llama-2-13B shapes on a paged pool: 4 prompts of U[128, 700] rows, each on its own adapter
    with ranks from {8, 16, 32, 64} (no padding to the largest), pages of one hidden-size vector
    (5120 elements: the MLP rows of 13824 span three pages), all 7 projections of one layer
    through the fused call; every row of every projection against the oracle."""
    rng = np.random.default_rng(41)
    g = W.generator(41, dev)
    lens = rng.integers(128, 701, 4)
    ranks = np.array([8, 16, 32, 64], np.int32)
    batch = W.batch_from_segments(lens, [3, 0, 2, 1]).to(dev)
    M = batch.M
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    x_h = W.normal((M, 5120), 1.0, torch.bfloat16, g, dev)
    for proj in W.LLAMA2_13B:
        pool = W.paged_pool(num_slots=4, num_layers=1, r_max=64, d_in=proj.d_in, d_out=proj.d_out,
                            dtype=torch.bfloat16, gen=g, device=dev, rng=rng, ranks=ranks, page_elems=5120)
        x = x_h if proj.d_in == 5120 else W.normal((M, proj.d_in), 1.0, torch.bfloat16, g, dev)
        op = W.Op(proj.name, pool, 0, x, W.uniform((M, proj.d_out), -1, 1, torch.bfloat16, g, dev))
        y = op.y.clone()
        before = m.launch_count()
        m.lora_sgmv(y, x, m.make_pool(pool), batch.seg_offsets, batch.seg_slot, 0, new_v(M, 64, dev), st)
        torch.cuda.synchronize()
        assert m.launch_count() - before == 3, f"{proj.name}: the tensor-core kernels did not run"
        assert st.item() == 0
        check_op(op, batch, "sgmv", y, what=f"paged 13B prefill {proj.name}")


def test_prefill_paged_bad_page_reported(dev):
    """A bad page id in a long segment's adapter: the tensor-core kernels report BAD_PAGE and leave
    that segment's rows untouched; the other segments are correct."""
    g = W.generator(14, dev)
    rng = np.random.default_rng(14)
    pool = W.paged_pool(num_slots=2, num_layers=1, r_max=16, d_in=256, d_out=264, dtype=torch.bfloat16, gen=g,
                        device=dev, rng=rng, ranks=[16, 8], page_elems=128)
    bt = pool.b_page_table.clone()
    bt[1, 0, 3, 1] = -7  # second page of row 3 of slot 1's B
    bad_pool = W.Pool(pool.dtype, 2, 1, 16, 256, 264, pool.rank, pool.scale, pages=pool.pages,
                      a_page_table=pool.a_page_table, b_page_table=bt)
    batch = W.batch_from_segments([300, 260], [0, 1]).to(dev)
    x = W.normal((batch.M, 256), 1.0, torch.bfloat16, g, dev)
    y0 = W.uniform((batch.M, 264), -1, 1, torch.bfloat16, g, dev)
    y = y0.clone()
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    m.lora_sgmv(y, x, m.make_pool(bad_pool), batch.seg_offsets, batch.seg_slot, 0, new_v(batch.M, 16, dev), st)
    torch.cuda.synchronize()
    assert st.item() == m.STATUS_BAD_PAGE
    assert torch.equal(y[300:].view(torch.int16), y0[300:].view(torch.int16))
    good = W.Batch(batch.M, batch.row_slot.masked_fill(batch.row_slot == 1, -1), None, None)
    check_op(W.Op("p", pool, 0, x, y0), good, "bgmv", y, what="segment with good pages")
