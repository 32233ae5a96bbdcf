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


def _bench(args, **env):
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    e = dict(os.environ, **env)
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], capture_output=True, text=True,
                       env=e, cwd=root, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return [json.loads(ln) for ln in lines]


def test_reference_arm_prints_one_line_on_rank0():
    (line,) = _bench(["--impl", "reference", "--steps", "1", "--warmup", "1"])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "rows/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    assert _bench(["--impl", "reference", "--steps", "1", "--warmup", "1"], RANK="1", LOCAL_RANK="1",
                  WORLD_SIZE="2") == []


def test_tensor_fraction_of_the_13b_prefill():
    # 12604 rows at rank 64 over the 7 Llama-2-13B projections: 2 * rows * r * (d_in + d_out) each
    import workloads.costmodel as C
    w = W.sgmv_prefill_13b(device="cpu", projections=W.LLAMA2_13B[:1])
    rows = w.batch.M
    q = W.LLAMA2_13B[0]
    flops = C.op_flops(d_in=q.d_in, d_out=q.d_out, row_ranks=[64] * rows)
    assert flops == 2 * rows * 64 * (5120 + 5120)
    t = bench.tensor_fraction(flops, 1e-3)
    assert abs(t["achieved_tflops"] - flops / 1e-3 / 1e12) < 0.1
    assert 0 < t["frac"] == round(t["achieved_tflops"] / t["peak_tflops"], 4)
