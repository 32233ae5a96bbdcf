"""The CPU baseline legs of bench.py, on a small copy of the decode step (three layers of small
projections): the oracle gives the same bits when called from several threads at once as when
called serially (it has no shared state), and the all-cores sampler covers every layer with the
threads it reports."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import bench
import oracle
import workloads as W

SMALL = [W.Projection("q", 64, 64), W.Projection("o", 64, 64), W.Projection("gate", 64, 96),
         W.Projection("down", 96, 64)]


def small_step():
    return W.sgmv_decode_7b(device="cpu", num_layers=3, M=8, num_slots=8, projections=SMALL)


def test_oracle_threads_match_serial():
    w = small_step()
    off, ss = w.batch.seg_offsets.numpy(), w.batch.seg_slot.numpy()
    lib = oracle.default()
    inputs = [inp for layer in range(3) for inp in bench._oracle_layer_inputs(w, layer)]
    serial = [lib.sgmv(p, 0, x, y, off, ss) for p, x, y in inputs]
    with ThreadPoolExecutor(4) as ex:
        threaded = list(ex.map(lambda t: lib.sgmv(t[0], 0, t[1], t[2], off, ss), inputs))
    for (ys, vs, _, sts), (yt, vt, _, stt) in zip(serial, threaded):
        assert sts == 0 and stt == 0
        assert np.array_equal(ys, yt)
        assert np.array_equal(vs, vt, equal_nan=True)


def test_all_cores_sampler_covers_every_layer():
    w = small_step()
    per_step, layers, used = bench.oracle_sample_all_cores(w, budget_s=60.0, threads=2)
    assert per_step > 0
    assert layers == 3  # batches of 2 layers, then 1: the budget is not reached
    assert used == 2
