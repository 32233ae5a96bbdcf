"""lora_sgmv_noalloc against lora_sgmv.

lora_sgmv_noalloc exists for callers that cannot give the library a device buffer -- code that
may not allocate device memory, such as a plugin inside a host engine that owns all device
memory, or a latency-critical path where cudaMalloc's implicit synchronisation is not
acceptable. It uses a scratch array built into the library instead of v_scratch. These tests
call it through the C ABI twice in a row, on different batches, and check each result against
lora_sgmv on the same inputs, within the parity tolerance of the other GPU tests. The batches
have long segments, so the two-launch tensor-core path really uses the scratch.

The file is named so that pytest collects it last; it passes on its own in a fresh process and
after every other test.
"""
import numpy as np
import pytest
import torch

import adapter_gemv_gb300 as m
import workloads as W
from gpu_util import TOL, bits, check_op

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


def batch_case(dev, seed, lens, slots, r_max, d_in, d_out):
    g = W.generator(seed, dev)
    pool = W.stacked_pool(num_slots=max(slots) + 1, num_layers=1, r_max=r_max, d_in=d_in, d_out=d_out,
                          dtype=torch.bfloat16, gen=g, device=dev)
    batch = W.batch_from_segments(lens, slots).to(dev)
    x = W.normal((batch.M, d_in), 1.0, torch.bfloat16, g, dev)
    y = W.uniform((batch.M, d_out), -1, 1, torch.bfloat16, g, dev)
    return pool, batch, x, y


def run_both(dev, pool, batch, x, y):
    h = m.make_pool(pool)
    st_ref = torch.zeros(1, dtype=torch.int32, device=dev)
    st_na = torch.zeros(1, dtype=torch.int32, device=dev)
    y_ref = y.clone()
    v = torch.empty((batch.M, pool.r_max), dtype=torch.float32, device=dev)
    m.lora_sgmv(y_ref, x, h, batch.seg_offsets, batch.seg_slot, 0, v, st_ref)
    y_na = y.clone()
    m.lora_sgmv_noalloc(y_na, x, h, batch.seg_offsets, batch.seg_slot, 0, st_na)
    torch.cuda.synchronize()
    assert st_ref.item() == 0 and st_na.item() == 0
    return y_ref, y_na


def assert_within_tolerance(got, want):
    g, w = got.double().cpu().numpy(), want.double().cpu().numpy()
    assert np.all(np.isfinite(w))
    assert np.all(np.abs(g - w) <= TOL * (1.0 + np.abs(w)))


def test_noalloc_matches_lora_sgmv_on_two_calls_in_a_row(dev):
    # two different batches back to back: the second call must not depend on what the first
    # left in the shared scratch
    first = batch_case(dev, 31, [300, 129, 7, 200], [0, 1, 2, 1], 64, 1024, 768)
    second = batch_case(dev, 32, [128, 40, 513], [1, 0, 2], 16, 512, 1032)
    for pool, batch, x, y in (first, second):
        y_ref, y_na = run_both(dev, pool, batch, x, y)
        assert not np.array_equal(bits(y_na), bits(y)), "the call changed nothing"
        assert_within_tolerance(y_na, y_ref)
        # the same kernels with the same split run in both calls: the bits agree too
        assert np.array_equal(bits(y_na), bits(y_ref)), "lora_sgmv_noalloc and lora_sgmv differ in their bits"
        # and both agree with the fp64 oracle on every row
        check_op(W.Op("noalloc", pool, 0, x, y), batch, "sgmv", y_na, what="lora_sgmv_noalloc")


def test_noalloc_rejects_calls_beyond_its_scratch(dev):
    g = W.generator(33, dev)
    r_max = 64
    rows = m.NOALLOC_MAX_FLOATS // r_max + 1
    pool = W.stacked_pool(num_slots=1, num_layers=1, r_max=r_max, d_in=8, d_out=8, dtype=torch.bfloat16, gen=g,
                          device=dev)
    batch = W.batch_from_segments([rows], [0]).to(dev)
    x = torch.zeros((rows, 8), dtype=torch.bfloat16, device=dev)
    y = torch.zeros((rows, 8), dtype=torch.bfloat16, device=dev)
    before = m.launch_count()
    with pytest.raises(m.MloraError) as e:
        m.lora_sgmv_noalloc(y, x, pool, batch.seg_offsets, batch.seg_slot, 0)
    assert e.value.code == m.ERR_TOO_LARGE
    assert m.launch_count() == before
