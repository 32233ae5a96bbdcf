"""The time-out path of the CUDA-core kernels, made to run out without any fault.

lora_test_set_wait_limit_ns shortens the limit of the kernels' waits (for their own bulk copies
and for their cluster peers' partial sums) to a few nanoseconds. A wait then gives up unless its
data has already landed: the kernel must set MLORA_STATUS_TIMEOUT, skip the work that needed the
data, drain the copies still in flight, and leave every element of y either untouched or equal
to the correct result. Nothing is made to fault or hang: the copies do land, just after the wait
stopped looking. Afterwards the default limit is restored and the same call gives the oracle's
result, so the context is still usable.
"""
import numpy as np
import pytest
import torch

import adapter_gemv_gb300 as m
import oracle
import workloads as W
from gpu_util import TOL, bits, odt, oracle_op

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


def untouched_or_correct(got_bits, before_bits, want_bits, dt):
    g = oracle.decode(got_bits, dt)
    w = oracle.decode(want_bits, dt)
    same = got_bits == before_bits
    close = np.abs(g - w) <= TOL * (1.0 + np.abs(w))
    return same | close


@pytest.mark.parametrize("form", ["sgmv", "bgmv"])
def test_short_wait_limit_reports_timeout_and_writes_nothing_wrong(dev, form):
    w = W.bgmv_decode_q(device=dev, M=16)  # one-row tiles in clusters of CTAs
    op, batch = w.ops[0], w.batch
    if form == "sgmv":
        batch = W.batch_from_segments(np.ones(16, np.int64), np.arange(16)).to(dev)
    h = m.make_pool(op.pool)
    want, _, st_o = oracle_op(op, batch, form)
    assert st_o == 0
    dt = odt(op.pool.dtype)
    before = bits(op.y)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    y = op.y.clone()
    v = torch.empty((16, op.pool.r_max), dtype=torch.float32, device=dev)
    m.lora_test_set_wait_limit_ns(2)
    try:
        for _ in range(3):
            if form == "sgmv":
                m.lora_sgmv(y, op.x, h, batch.seg_offsets, batch.seg_slot, 0, v, st)
            else:
                m.lora_bgmv(y, op.x, h, batch.row_slot, 0, v, st)
            torch.cuda.synchronize()
            ok = untouched_or_correct(bits(y), before, want, dt)
            assert ok.all(), f"{(~ok).sum()} elements neither untouched nor correct after a timed-out call"
            y.copy_(op.y)
    finally:
        m.lora_test_set_wait_limit_ns(0)
    assert st.item() & m.STATUS_TIMEOUT, "no wait gave up with a limit of 2 ns"
    assert st.item() & ~m.STATUS_TIMEOUT == 0
    # default limit again: the same call completes and matches the oracle
    st.zero_()
    y = op.y.clone()
    if form == "sgmv":
        m.lora_sgmv(y, op.x, h, batch.seg_offsets, batch.seg_slot, 0, v, st)
    else:
        m.lora_bgmv(y, op.x, h, batch.row_slot, 0, v, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    g, wv = oracle.decode(bits(y), dt), oracle.decode(want, dt)
    assert np.all(np.abs(g - wv) <= TOL * (1.0 + np.abs(wv)))


def test_status_bit_survives_a_clear_just_before_a_programmatic_call(dev):
    """The status word is an output: a kernel launched with programmatic dependent launch writes
    it only after waiting for the kernel before it, so a torch kernel that clears the word right
    before the call cannot wipe the bit out."""
    w = W.bgmv_decode_q(device=dev, M=8)
    op = w.ops[0]
    h = m.make_pool(op.pool)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    bad = torch.tensor([0, 1, 99, 2, 3, 4, 5, 6], dtype=torch.int32, device=dev)  # 99: no such slot
    v = torch.empty((8, op.pool.r_max), dtype=torch.float32, device=dev)
    prev = m.lora_set_programmatic_launch(True)
    try:
        for _ in range(20):
            st.fill_(0)  # a kernel writing the status word, launched just before the call
            y = op.y.clone()
            m.lora_bgmv(y, op.x, h, bad, 0, v, st)
            torch.cuda.synchronize()
            assert st.item() == m.STATUS_BAD_SLOT
    finally:
        m.lora_set_programmatic_launch(prev)


def test_short_wait_limit_streaming_bgmv(dev):
    """The same for grouped BGMV rows of a heterogeneous-rank paged pool, which a cluster of CTAs
    per row streams through shared-memory rings: producer and consumer warps give up on their
    waits, the cluster's partial-sum exchange gives up too, the producers wait for the copies they
    issued, and no element of y is wrong."""
    g = W.generator(21, dev)
    rng = np.random.default_rng(21)
    ranks = np.array([8, 32, 16, 32, 8, 24], np.int32)
    d_in, d_out = 8192, 4160  # a full-rank row is 786 KB: two CTAs per row
    pool = W.paged_pool(num_slots=6, num_layers=1, r_max=32, d_in=d_in, d_out=d_out, dtype=torch.bfloat16, gen=g,
                        device=dev, rng=rng, ranks=ranks, page_elems=1024)
    M = 40
    slots = rng.integers(-1, 6, M).astype(np.int32)
    batch = W.batch_from_slots(slots, sgmv=False).to(dev)
    x = W.normal((M, d_in), 1.0, torch.bfloat16, g, dev)
    y0 = W.uniform((M, d_out), -1, 1, torch.bfloat16, g, dev)
    op = W.Op("up", pool, 0, x, y0)
    want, _, st_o = oracle_op(op, batch, "bgmv")
    assert st_o == 0
    dt = odt(pool.dtype)
    before = bits(y0)
    h = m.make_pool(pool)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    v = torch.empty((M, 32), dtype=torch.float32, device=dev)
    m.lora_test_set_wait_limit_ns(2)
    try:
        for _ in range(3):
            y = y0.clone()
            m.lora_bgmv_ex(y, x, h, batch.row_slot, 0, v, m.LAUNCH_GROUP_ROWS, st)
            torch.cuda.synchronize()
            ok = untouched_or_correct(bits(y), before, want, dt)
            assert ok.all(), f"{(~ok).sum()} elements neither untouched nor correct after a timed-out call"
    finally:
        m.lora_test_set_wait_limit_ns(0)
    assert st.item() & m.STATUS_TIMEOUT, "no wait gave up with a limit of 2 ns"
    assert st.item() & ~m.STATUS_TIMEOUT == 0
    st.zero_()
    y = y0.clone()
    m.lora_bgmv_ex(y, x, h, batch.row_slot, 0, v, m.LAUNCH_GROUP_ROWS, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    gv, wv = oracle.decode(bits(y), dt), oracle.decode(want, dt)
    assert np.all(np.abs(gv - wv) <= TOL * (1.0 + np.abs(wv)))
