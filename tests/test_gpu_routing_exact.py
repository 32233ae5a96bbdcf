"""Bit-exact GPU routing pins: slot, layer and segment handling checked bit for bit against the
fp64 oracle, through every call form and kernel variant.

Pools and inputs are built so that every product and every partial sum the kernels form is
exactly representable in fp32 (and every V the tensor-core expand splits into hi + lo halves is
exact in the sum of the two halves):
  * A^T rows of (slot s, layer l) are the constant 2^-(4 + s + 3l), so v = d_in * x * A names the
    slot and the layer (the slot identification of the pages' reference loop, "Multi-LoRA
    Serving, in depth", with one adapter per row; S-LoRA "Unified Paging" for the paged pool);
  * B rows of (s, l) are 2^-(2 + (s + l) % 3) * (1 + n % 3), so a column shift changes the bits;
  * x row i is the constant +-2^-(i % 4) (a row mix-up changes the bits);
  * scale[s] = 2^-(s % 3); ranks differ per slot, rank-1 slots included (the rank-1 closed form
    delta = scale * rank * d_in * x * a * b).
Every fp32 sum is then the exact value, so the GPU's single rounding to the I/O type gives the
oracle's bits whatever the summation order, split or MMA schedule: routing is the only thing
that can make them differ. Rows without adapter hold a NaN payload in y that must survive.
"""
import zlib

import numpy as np
import pytest
import torch

import adapter_gemv_gb300 as m
import oracle
import workloads as W
from gpu_util import bits, odt

pytestmark = pytest.mark.gpu

NAN_BITS = {torch.bfloat16: 0x7FC3, torch.float16: 0x7E03}


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    if not os.path.exists(m.LIB_PATH):
        from adapter_gemv_gb300 import build
        build.build()
    return torch.device("cuda:0")


def a_value(s, layer):
    return 2.0 ** -(4 + s + 3 * layer)


def b_value(s, layer, n):
    return 2.0 ** -(2 + (s + layer) % 3) * (1 + n % 3)


def exact_pool(dev, dtype, *, num_slots, num_layers, r_max, d_in, d_out, ranks, paged, rng, page_pad=0,
               page_elems=None):
    ranks = np.asarray(ranks, np.int32)
    a_t = torch.empty((num_slots, num_layers, r_max, d_in), dtype=torch.float32)
    b = torch.empty((num_slots, num_layers, r_max, d_out), dtype=torch.float32)
    cols = torch.arange(d_out, dtype=torch.float32)
    for s in range(num_slots):
        for layer in range(num_layers):
            a_t[s, layer] = a_value(s, layer)
            b[s, layer] = (2.0 ** -(2 + (s + layer) % 3)) * (1 + cols % 3)
            a_t[s, layer, ranks[s]:] = float("nan")  # padding rows must never be read
            b[s, layer, ranks[s]:] = float("nan")
    a_t, b = a_t.to(dtype), b.to(dtype)  # exact: powers of two times 1, 2 or 3
    scale = (2.0 ** -(np.arange(num_slots) % 3)).astype(np.float32)
    rank_t = torch.from_numpy(ranks).to(dev)
    scale_t = torch.from_numpy(scale).to(dev)
    if not paged:
        return W.Pool(dtype, num_slots, num_layers, r_max, d_in, d_out, rank_t, scale_t,
                      a_t=a_t.to(dev), b=b.to(dev))
    # the same adapters in pages at permuted positions, free pages (NaN) interleaved; with
    # page_elems below d a vector is cut into ceil(d / page_elems) pages placed independently
    page_elems = max(d_in, d_out) + page_pad if page_elems is None else page_elems
    a_ppv, b_ppv = -(-d_in // page_elems), -(-d_out // page_elems)
    used = int(num_layers * ranks.sum() * (a_ppv + b_ppv))
    num_pages = used + used // 4 + 3
    phys = iter(rng.permutation(num_pages)[:used])
    pages = torch.full((num_pages, page_elems), float("nan"), dtype=dtype)
    a_tab = np.full((num_slots, num_layers, r_max, a_ppv), -1, np.int32)
    b_tab = np.full((num_slots, num_layers, r_max, b_ppv), -1, np.int32)
    for s in range(num_slots):
        for layer in range(num_layers):
            for j in range(ranks[s]):
                for tab, src, d, n in ((a_tab, a_t, d_in, a_ppv), (b_tab, b, d_out, b_ppv)):
                    for q in range(n):
                        pg = next(phys)
                        tab[s, layer, j, q] = pg
                        lo, hi = q * page_elems, min(d, (q + 1) * page_elems)
                        pages[pg, :hi - lo] = src[s, layer, j, lo:hi]
    return W.Pool(dtype, num_slots, num_layers, r_max, d_in, d_out, rank_t, scale_t, pages=pages.to(dev),
                  a_page_table=torch.from_numpy(a_tab).to(dev), b_page_table=torch.from_numpy(b_tab).to(dev))


def oracle_of(p: W.Pool) -> oracle.Pool:
    common = dict(dtype=odt(p.dtype), num_slots=p.num_slots, num_layers=p.num_layers, r_max=p.r_max, d_in=p.d_in,
                  d_out=p.d_out, rank=p.rank.cpu().numpy(), scale=p.scale.cpu().numpy())
    if p.paged:
        return oracle.Pool(**common, pages=bits(p.pages), a_page_table=p.a_page_table.cpu().numpy(),
                           b_page_table=p.b_page_table.cpu().numpy())
    return oracle.Pool(**common, a_t=bits(p.a_t), b=bits(p.b))


def exact_rows(dev, dtype, M, d_in, d_out, row_slot):
    i = torch.arange(M, dtype=torch.float32)
    xv = (2.0 ** -(i % 4)) * torch.where(i % 2 == 1, -1.0, 1.0)
    x = xv[:, None].expand(M, d_in).to(dtype).contiguous().to(dev)
    y = torch.zeros((M, d_out), dtype=dtype)
    skip = torch.from_numpy(np.asarray(row_slot) < 0)
    y.view(torch.int16)[skip] = NAN_BITS[dtype]  # rows without adapter: a NaN payload that must survive
    return x, y.to(dev)


def segments(rng, M, nseg, num_slots, allow_empty=True):
    cuts = np.sort(rng.integers(0 if allow_empty else 1, M + 1, nseg - 1)) if nseg > 1 else np.array([], int)
    off = np.r_[0, cuts, M].astype(np.int32)
    seg_slot = rng.integers(-1, num_slots, nseg).astype(np.int32)
    return off, seg_slot


def assert_bits_equal(got, want, what):
    got, want = np.asarray(got), np.asarray(want)
    bad = np.argwhere(got != want)
    assert bad.size == 0, (f"{what}: {len(bad)} elements differ from the oracle's bits; first at {bad[0].tolist()}: "
                           f"got {got[tuple(bad[0])]:#06x}, want {want[tuple(bad[0])]:#06x}")


def check_exact(pool, layer, x, y_before, y_gpu, form, meta, v_gpu=None, what=""):
    op = oracle_of(pool)
    if form == "sgmv":
        y_o, v_o, _, st = oracle.sgmv(op, layer, bits(x), bits(y_before), meta[0], meta[1])
        row_slot = np.repeat(meta[1], np.diff(meta[0]))
    else:
        y_o, v_o, _, st = oracle.bgmv(op, layer, bits(x), bits(y_before), meta)
        row_slot = np.asarray(meta)
    assert st == 0
    assert_bits_equal(bits(y_gpu), y_o, f"{what} y")
    if v_gpu is not None:
        vg = v_gpu.double().cpu().numpy()
        ranks = pool.rank.cpu().numpy()
        for i in np.flatnonzero(row_slot >= 0):
            r = ranks[row_slot[i]]
            assert np.array_equal(vg[i, :r], v_o[i, :r]), f"{what} v row {i}: {vg[i, :r]} vs {v_o[i, :r]}"


# dtype, paged, r_max, d_in, d_out, M, nseg, ranks: shapes that reach every decode-kernel variant
# (one-row tiles, 4-row tiles, the rank-aware A layouts of multi-pass one-row tiles, the generic
# multi-row path with A in several passes) on both pool kinds
DECODE_CASES = [
    (torch.bfloat16, False, 16, 4096, 4096, 32, 32, [16, 1, 7, 16, 3, 12]),   # one-row tiles
    (torch.bfloat16, True, 16, 4096, 11008, 32, 9, [16, 1, 7, 16, 3, 12]),    # 4-row tiles, paged
    (torch.float16, False, 16, 11008, 4096, 20, 20, [5, 16, 1, 9, 16, 2]),    # one-row, several CTAs
    (torch.float16, True, 32, 1024, 520, 24, 6, [32, 1, 17, 8, 32, 4]),       # 4-row tiles, fp16 paged
    (torch.bfloat16, False, 64, 6000, 1000, 200, 200, [1, 8, 16, 32, 33, 64]),  # rank-aware layouts
    (torch.bfloat16, True, 128, 7168, 520, 160, 160, [1, 9, 33, 64, 65, 128]),  # rank-aware, paged
    (torch.bfloat16, False, 128, 4104, 2056, 21, 4, [128, 1, 77, 128, 3, 64]),  # generic multi-row path
    # pages shorter than the vectors (S-LoRA: a page is one H-vector; MLP rows span several)
    (torch.bfloat16, True, 16, 4096, 11008, 32, 32, [16, 1, 7, 16, 3, 12], 4096),
    (torch.float16, True, 32, 11008, 4096, 24, 6, [32, 1, 17, 8, 32, 4], 4096),
    (torch.bfloat16, True, 64, 6000, 1000, 200, 200, [1, 8, 16, 32, 33, 64], 1000),
]


def ids(c):
    return (f"{'bf16' if c[0] == torch.bfloat16 else 'fp16'}-{'paged' if c[1] else 'stacked'}-r{c[2]}-"
            f"{c[3]}x{c[4]}-M{c[5]}-n{c[6]}" + (f"-pages{c[8]}" if len(c) > 8 else ""))


@pytest.mark.parametrize("case", DECODE_CASES, ids=ids)
def test_exact_routing_decode_kernels(dev, case):
    dtype, paged, r_max, d_in, d_out, M, nseg, ranks = case[:8]
    page_elems = case[8] if len(case) > 8 else None
    rng = np.random.default_rng(zlib.crc32(ids(case).encode()))
    num_layers = 2
    pool = exact_pool(dev, dtype, num_slots=len(ranks), num_layers=num_layers, r_max=r_max, d_in=d_in, d_out=d_out,
                      ranks=ranks, paged=paged, rng=rng, page_pad=8 * int(rng.integers(0, 3)), page_elems=page_elems)
    h = m.make_pool(pool)
    layer = 1
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    # SGMV over random segments (empty, repeated and -1 segments); segments of one row when nseg == M
    if nseg == M:
        off = np.arange(M + 1, dtype=np.int32)
        seg_slot = rng.integers(-1, len(ranks), M).astype(np.int32)
    else:
        off, seg_slot = segments(rng, M, nseg, len(ranks))
    row_slot = np.repeat(seg_slot, np.diff(off))
    x, y0 = exact_rows(dev, dtype, M, d_in, d_out, row_slot)
    offd, ssd = torch.from_numpy(off).to(dev), torch.from_numpy(seg_slot).to(dev)
    v = torch.full((M, r_max), float("nan"), device=dev)
    y2 = y0.clone()
    m.lora_sgmv_shrink(v, x, h, offd, ssd, layer, st)
    m.lora_sgmv_expand(y2, v, h, offd, ssd, layer, st)
    y1 = y0.clone()
    m.lora_sgmv(y1, x, h, offd, ssd, layer, torch.empty_like(v), st)
    yg = [y0.clone() for _ in range(2)]
    m.lora_sgmv_grouped([(yg[q], x, h, layer, torch.empty_like(v)) for q in range(2)], offd, ssd, st)
    # BGMV: the same rows in a shuffled order, -1 rows included
    perm = rng.permutation(M)
    rs_b = row_slot[perm].astype(np.int32)
    xb, yb0 = exact_rows(dev, dtype, M, d_in, d_out, rs_b)
    rsd = torch.from_numpy(rs_b).to(dev)
    vb = torch.full((M, r_max), float("nan"), device=dev)
    yb2 = yb0.clone()
    m.lora_bgmv_shrink(vb, xb, h, rsd, layer, st)
    m.lora_bgmv_expand(yb2, vb, h, rsd, layer, st)
    yb1 = yb0.clone()
    m.lora_bgmv(yb1, xb, h, rsd, layer, torch.empty_like(vb), st)
    torch.cuda.synchronize()
    assert st.item() == 0
    check_exact(pool, layer, x, y0, y2, "sgmv", (off, seg_slot), v, "sgmv two-launch")
    check_exact(pool, layer, x, y0, y1, "sgmv", (off, seg_slot), None, "sgmv fused")
    for q in range(2):
        check_exact(pool, layer, x, y0, yg[q], "sgmv", (off, seg_slot), None, f"grouped problem {q}")
    check_exact(pool, layer, xb, yb0, yb2, "bgmv", rs_b, vb, "bgmv two-launch")
    check_exact(pool, layer, xb, yb0, yb1, "bgmv", rs_b, None, "bgmv fused")


# long segments: the tensor-core kernels (full and partial 128-row blocks, K split over a cluster)
# next to short segments on the CUDA-core kernel; stacked pools (the tensor-core path's pools)
TC_CASES = [
    # dtype, r_max, d_in, d_out, segment lengths, slots, ranks
    (torch.bfloat16, 16, 256, 136, [128 * 60 + 7, 5, 128 * 41, 1, 33], [0, 2, 1, -1, 3], [16, 1, 9, 16]),
    (torch.bfloat16, 64, 5120, 640, [255, 3, 130, 0, 384], [2, 0, 0, 1, -1], [64, 1, 33]),
    (torch.float16, 32, 1024, 1104, [300, 31, 32, 129, 7], [1, 0, 2, 1, 2], [32, 1, 17]),
    (torch.float16, 128, 1032, 264, [256, 131, 2], [0, 1, 0], [128, 96]),
]


@pytest.mark.parametrize("pages", [None, "square", "short"])
@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: f"{'bf16' if c[0] == torch.bfloat16 else 'fp16'}-r{c[1]}-"
                         f"{c[2]}x{c[3]}-M{sum(c[4])}")
def test_exact_routing_tensor_core_path(dev, case, pages):
    """pages: stacked pool (None), paged with a page per vector, paged with pages of about a third
    of the longer vector (vectors span two to four pages; page boundaries fall inside atoms)."""
    dtype, r_max, d_in, d_out, lens, slots, ranks = case
    rng = np.random.default_rng(sum(lens))
    short = max(64, (max(d_in, d_out) // 3 + 7) // 8 * 8)
    pool = exact_pool(dev, dtype, num_slots=len(ranks), num_layers=2, r_max=r_max, d_in=d_in, d_out=d_out,
                      ranks=ranks, paged=pages is not None, rng=rng, page_elems=short if pages == "short" else None)
    h = m.make_pool(pool)
    off = np.r_[0, np.cumsum(lens)].astype(np.int32)
    seg_slot = np.asarray(slots, np.int32)
    M = int(off[-1])
    row_slot = np.repeat(seg_slot, lens)
    x, y0 = exact_rows(dev, dtype, M, d_in, d_out, row_slot)
    offd, ssd = torch.from_numpy(off).to(dev), torch.from_numpy(seg_slot).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    v = torch.full((M, r_max), float("nan"), device=dev)
    before = m.launch_count()
    y2 = y0.clone()
    m.lora_sgmv_shrink(v, x, h, offd, ssd, 1, st)
    m.lora_sgmv_expand(y2, v, h, offd, ssd, 1, st)
    y1 = y0.clone()
    m.lora_sgmv(y1, x, h, offd, ssd, 1, torch.empty_like(v), st)
    torch.cuda.synchronize()
    assert m.launch_count() - before == 4 + 3, "the tensor-core kernels did not run"
    assert st.item() == 0
    check_exact(pool, 1, x, y0, y2, "sgmv", (off, seg_slot), v, "tensor-core two-launch")
    check_exact(pool, 1, x, y0, y1, "sgmv", (off, seg_slot), None, "tensor-core fused")


def test_exact_rank1_closed_form(dev):
    """Rank 1 everywhere: every adapted element is y + scale * d_in * x_i * a * b, exactly."""
    dtype = torch.bfloat16
    rng = np.random.default_rng(5)
    d_in, d_out, M = 4096, 4096, 32
    pool = exact_pool(dev, dtype, num_slots=4, num_layers=1, r_max=16, d_in=d_in, d_out=d_out, ranks=[1, 1, 1, 1],
                      paged=False, rng=rng)
    rs = (np.arange(M) % 5 - 1).astype(np.int32)  # -1, 0, 1, 2, 3, -1, ...
    x, y0 = exact_rows(dev, dtype, M, d_in, d_out, rs)
    y = y0.clone()
    m.lora_bgmv(y, x, m.make_pool(pool), torch.from_numpy(rs).to(dev), 0,
                torch.empty((M, 16), dtype=torch.float32, device=dev))
    torch.cuda.synchronize()
    got = y.double().cpu().numpy()
    xs = x[:, 0].double().cpu().numpy()
    scale = pool.scale.cpu().numpy()
    for i in range(M):
        s = rs[i]
        if s < 0:
            assert np.array_equal(bits(y)[i], bits(y0)[i])
            continue
        want = scale[s] * d_in * xs[i] * a_value(s, 0) * np.array([b_value(s, 0, n) for n in range(d_out)])
        assert np.array_equal(got[i], want), f"row {i}: closed form differs"


# Chained one-row calls (programmatic dependent launch), bit for bit: projections whose d_in slice
# spans several passes of A and projections whose B is much larger than their A, on stacked pools
# and on paged pools with one page per vector or pages shorter than the vectors.
# dtype, paged, d_in, d_out, M, ranks, page_elems (None: one page per vector)
CHAINED_CASES = [
    (torch.bfloat16, False, 11008, 4096, 20, [16, 1, 7, 16, 3, 12], None),
    (torch.float16, True, 11008, 4096, 20, [5, 16, 1, 9, 16, 2], None),
    (torch.bfloat16, True, 11008, 4096, 24, [16, 4, 13, 16], 1536),
    (torch.bfloat16, False, 4096, 11008, 32, [16, 1, 7, 16, 3, 12], None),
    (torch.float16, True, 4096, 11008, 32, [16, 2, 9, 16, 8], 4096),
]


@pytest.mark.parametrize("case", CHAINED_CASES, ids=lambda c: f"{'bf16' if c[0] == torch.bfloat16 else 'fp16'}-"
                         f"{'paged' if c[1] else 'stacked'}-{c[2]}x{c[3]}-M{c[4]}" + (f"-pages{c[6]}" if c[6] else ""))
def test_exact_routing_chained_calls(dev, case):
    dtype, paged, d_in, d_out, M, ranks, page_elems = case
    rng = np.random.default_rng(zlib.crc32(repr(case[1:]).encode()))
    pool = exact_pool(dev, dtype, num_slots=len(ranks), num_layers=2, r_max=16, d_in=d_in, d_out=d_out, ranks=ranks,
                      paged=paged, rng=rng, page_elems=page_elems)
    h = m.make_pool(pool)
    layer = 1
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    off = np.arange(M + 1, dtype=np.int32)
    seg_slot = rng.integers(-1, len(ranks), M).astype(np.int32)
    x, y0 = exact_rows(dev, dtype, M, d_in, d_out, seg_slot)
    offd, ssd = torch.from_numpy(off).to(dev), torch.from_numpy(seg_slot).to(dev)
    v = torch.empty((M, 16), dtype=torch.float32, device=dev)
    ys = [y0.clone() for _ in range(3)]
    yg = [y0.clone() for _ in range(2)]
    perm = rng.permutation(M)
    rs_b = seg_slot[perm].astype(np.int32)
    xb, yb0 = exact_rows(dev, dtype, M, d_in, d_out, rs_b)
    yb = yb0.clone()
    prev = m.lora_set_programmatic_launch(True)
    try:
        for q in range(3):  # chained: every call after the first waits on the previous one
            m.lora_sgmv(ys[q], x, h, offd, ssd, layer, v, st)
        m.lora_sgmv_grouped([(yg[q], x, h, layer, torch.empty_like(v)) for q in range(2)], offd, ssd, st)
        m.lora_bgmv(yb, xb, h, torch.from_numpy(rs_b).to(dev), layer, v, st)
    finally:
        m.lora_set_programmatic_launch(prev)
    torch.cuda.synchronize()
    assert st.item() == 0
    for q in range(3):
        check_exact(pool, layer, x, y0, ys[q], "sgmv", (off, seg_slot), None, f"chained sgmv {q}")
    for q in range(2):
        check_exact(pool, layer, x, y0, yg[q], "sgmv", (off, seg_slot), None, f"chained grouped problem {q}")
    check_exact(pool, layer, xb, yb0, yb, "bgmv", rs_b, None, "chained bgmv")
