"""GPU edge cases against the oracle: random segment layouts (empty segments, repeated slots,
-1 segments), ragged sizes, ranks 1..128 (the maximum), stacked and paged pools, both dtypes,
guard regions around every output, the device status contract, determinism, and the
equivalences between the call forms."""
import numpy as np
import pytest
import torch

import adapter_gemv_gb300 as m
import oracle
import workloads as W
from gpu_util import assert_close, bits, check_op, new_v, odt, oracle_pool

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


def make_case(dev, seed, *, dtype, paged, r_max, d_in, d_out, M, num_slots=5, num_layers=2, max_seg=9,
              page_elems=None):
    rng = np.random.default_rng(seed)
    g = W.generator(seed, dev)
    ranks = rng.integers(1, r_max + 1, num_slots).astype(np.int32)
    ranks[0] = r_max
    ranks[-1] = 1
    if paged:
        pool = W.paged_pool(num_slots=num_slots, num_layers=num_layers, r_max=r_max, d_in=d_in, d_out=d_out,
                            dtype=dtype, gen=g, device=dev, rng=rng, ranks=ranks,
                            page_elems=page_elems or max(d_in, d_out) + 8 * int(rng.integers(0, 3)))
    else:
        pool = W.stacked_pool(num_slots=num_slots, num_layers=num_layers, r_max=r_max, d_in=d_in, d_out=d_out,
                              dtype=dtype, gen=g, device=dev, ranks=ranks)
    # segments: random lengths (some empty), random slots with -1 and repeats, summing to M
    nseg = int(rng.integers(1, max_seg + 1))
    cuts = np.sort(rng.integers(0, M + 1, nseg - 1)) if nseg > 1 else np.array([], int)
    off = np.r_[0, cuts, M].astype(np.int32)
    seg_slot = rng.integers(-1, num_slots, nseg).astype(np.int32)
    lens = np.diff(off)
    batch = W.Batch(M, torch.from_numpy(np.repeat(seg_slot, lens).astype(np.int32)), torch.from_numpy(off),
                    torch.from_numpy(seg_slot)).to(dev)
    x = W.normal((M, d_in), 1.0, dtype, g, dev)
    y = W.uniform((M, d_out), -1, 1, dtype, g, dev)
    layer = int(rng.integers(0, num_layers))
    return W.Op("fuzz", pool, layer, x, y), batch


class Guarded:
    """y and v inside larger buffers: guard rows before/after and guard columns past d_out."""

    def __init__(self, y: torch.Tensor, r_max: int, pad_cols=8):
        M, d = y.shape
        self.ybuf = torch.empty((M + 2, d + pad_cols), dtype=y.dtype, device=y.device)
        self.ybuf.view(torch.int16).fill_(0x5A5A)
        self.y = self.ybuf[1:M + 1, :d]
        self.y.copy_(y)
        self.vbuf = torch.full(((M + 2) * r_max,), 1234.5, dtype=torch.float32, device=y.device)
        self.v = self.vbuf[r_max:r_max + M * r_max].view(M, r_max)
        self.M, self.d, self.r = M, d, r_max

    def check(self, v_written: bool):
        yb = bits(self.ybuf)
        assert np.all(yb[0] == 0x5A5A) and np.all(yb[-1] == 0x5A5A), "y guard rows written"
        assert np.all(yb[:, self.d:] == 0x5A5A), "y guard columns written"
        vb = self.vbuf.cpu().numpy()
        assert np.all(vb[:self.r] == 1234.5) and np.all(vb[self.r + self.M * self.r:] == 1234.5), "v guards written"


SHAPES = [
    # dtype, paged, r_max, d_in, d_out, M
    (torch.bfloat16, False, 16, 264, 40, 33),
    (torch.float16, False, 8, 24, 520, 7),
    (torch.bfloat16, True, 64, 1032, 264, 130),
    (torch.float16, True, 1, 8, 8, 5),
    (torch.bfloat16, False, 128, 4104, 2056, 21),
    (torch.bfloat16, True, 128, 520, 4104, 12),
    (torch.float16, False, 32, 16384, 64, 3),
    (torch.bfloat16, False, 64, 96, 16384, 9),
    (torch.bfloat16, False, 16, 4096, 4096, 1),
    (torch.bfloat16, False, 16, 4096, 4096, 0),
]


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{'bf16' if s[0] == torch.bfloat16 else 'fp16'}-"
                         f"{'paged' if s[1] else 'stacked'}-r{s[2]}-{s[3]}x{s[4]}-M{s[5]}")
@pytest.mark.parametrize("form", ["sgmv", "bgmv"])
def test_fuzz_two_phase_and_fused(dev, shape, seed, form):
    dtype, paged, r_max, d_in, d_out, M = shape
    op, batch = make_case(dev, 100 + seed, dtype=dtype, paged=paged, r_max=r_max, d_in=d_in, d_out=d_out, M=M)
    pool = m.make_pool(op.pool)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    # two launches, with guard regions
    g2 = Guarded(op.y, r_max)
    if form == "sgmv":
        m.lora_sgmv_shrink(g2.v, op.x, pool, batch.seg_offsets, batch.seg_slot, op.layer, st)
        m.lora_sgmv_expand(g2.y, g2.v, pool, batch.seg_offsets, batch.seg_slot, op.layer, st)
    else:
        m.lora_bgmv_shrink(g2.v, op.x, pool, batch.row_slot, op.layer, st)
        m.lora_bgmv_expand(g2.y, g2.v, pool, batch.row_slot, op.layer, st)
    # fused, with guard regions
    g1 = Guarded(op.y, r_max)
    if form == "sgmv":
        m.lora_sgmv(g1.y, op.x, pool, batch.seg_offsets, batch.seg_slot, op.layer, g1.v, st)
    else:
        m.lora_bgmv(g1.y, op.x, pool, batch.row_slot, op.layer, g1.v, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    g2.check(True)
    g1.check(False)
    check_op(op, batch, form, g2.y, g2.v, what="two-phase")
    check_op(op, batch, form, g1.y, what="fused")



# S-LoRA "Unified Paging" with pages shorter than a vector: a rank-row of A^T (d_in) or B (d_out)
# spans ceil(d / page_elems) pages at unrelated places of the pool. Shapes of the MLP projections
# in hidden-size pages (gate/up: B rows of 11008 in 4096-element pages; down: A rows of 11008), and
# odd splits: a CTA's slice of d_in or d_out, its staged B rows and its passes of A cross pages.
SHORT_PAGES = [
    # dtype, r_max, d_in, d_out, M, page_elems
    (torch.bfloat16, 16, 4096, 11008, 32, 4096),
    (torch.bfloat16, 16, 11008, 4096, 20, 4096),
    (torch.float16, 64, 1032, 264, 130, 264),
    (torch.bfloat16, 128, 520, 4104, 12, 136),
    (torch.bfloat16, 64, 6000, 1000, 40, 1000),
    (torch.float16, 8, 24, 520, 7, 8),
]


@pytest.mark.parametrize("shape", SHORT_PAGES, ids=lambda s: f"{'bf16' if s[0] == torch.bfloat16 else 'fp16'}-"
                         f"r{s[1]}-{s[2]}x{s[3]}-M{s[4]}-pages{s[5]}")
@pytest.mark.parametrize("form", ["sgmv", "bgmv"])
def test_vectors_across_pages(dev, shape, form):
    dtype, r_max, d_in, d_out, M, pe = shape
    op, batch = make_case(dev, 300 + d_in, dtype=dtype, paged=True, r_max=r_max, d_in=d_in, d_out=d_out, M=M,
                          page_elems=pe)
    assert op.pool.a_page_table.shape[-1] == -(-d_in // pe) and op.pool.b_page_table.shape[-1] == -(-d_out // pe)
    pool = m.make_pool(op.pool)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    g2, g1 = Guarded(op.y, r_max), Guarded(op.y, r_max)
    if form == "sgmv":
        m.lora_sgmv_shrink(g2.v, op.x, pool, batch.seg_offsets, batch.seg_slot, op.layer, st)
        m.lora_sgmv_expand(g2.y, g2.v, pool, batch.seg_offsets, batch.seg_slot, op.layer, st)
        m.lora_sgmv(g1.y, op.x, pool, batch.seg_offsets, batch.seg_slot, op.layer, g1.v, st)
    else:
        m.lora_bgmv_shrink(g2.v, op.x, pool, batch.row_slot, op.layer, st)
        m.lora_bgmv_expand(g2.y, g2.v, pool, batch.row_slot, op.layer, st)
        m.lora_bgmv(g1.y, op.x, pool, batch.row_slot, op.layer, g1.v, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    g2.check(True)
    g1.check(False)
    check_op(op, batch, form, g2.y, g2.v, what="two-phase, short pages")
    check_op(op, batch, form, g1.y, what="fused, short pages")


def test_bad_page_in_a_later_piece_of_a_vector(dev):
    """A bad id in the second page of a vector is found like one in the first: BAD_PAGE, the
    row untouched, the other rows correct."""
    op, batch = make_case(dev, 9, dtype=torch.bfloat16, paged=True, r_max=8, d_in=64, d_out=48, M=8, num_slots=4,
                          page_elems=24)
    at = op.pool.a_page_table.clone()
    at[2, op.layer, 0, 1] = op.pool.pages.shape[0]  # second of the three pages of slot 2's first A vector
    p2 = W.Pool(op.pool.dtype, 4, op.pool.num_layers, 8, 64, 48, op.pool.rank, op.pool.scale, pages=op.pool.pages,
                a_page_table=at, b_page_table=op.pool.b_page_table)
    slots = torch.tensor([0, 1, 2, 3] * 2, dtype=torch.int32, device=dev)
    y = op.y.clone()
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    m.lora_bgmv(y, op.x, m.make_pool(p2), slots, op.layer, new_v(8, 8, dev), st)
    torch.cuda.synchronize()
    assert st.item() == m.STATUS_BAD_PAGE
    assert np.array_equal(bits(y)[2::4], bits(op.y)[2::4])
    good = W.Batch(8, slots.cpu().masked_fill(slots.cpu() == 2, -1), None, None)
    check_op(op, good.to(dev), "bgmv", y, what="rows of the other slots")


# One-row tiles whose d_in slice spans several passes of A hold as few rank rows per warp as
# their rank allows (1, 2, 4 or 8 of a warp's 8, 16 ways), and use the freed registers for more
# of d_in per pass, as long as whole passes stay inside the x slice in shared memory. The
# shapes are chosen, against the launcher's split rule, so that single calls produce such tiles:
#   r_max 64,  d_in 6000, M 200: 6 CTAs per row, slices of 1000, x slice 1024 wide; ranks <= 32
#     take one pass of 1024, ranks 33..64 two passes of 512;
#   r_max 128, d_in 7168, M 160: 7 CTAs per row, slices of 1024; ranks <= 32 one pass, ranks
#     33..64 two passes, ranks above 64 four passes of 256.
# The slots' ranks sit on both sides of every layout boundary; every seventh row has no adapter.
RANK_LAYOUT_CASES = [
    # r_max, d_in, d_out, M, ranks of the slots
    (64, 6000, 1000, 200, [1, 8, 9, 16, 17, 32, 33, 64]),
    (128, 7168, 520, 160, [1, 8, 9, 32, 33, 64, 65, 128]),
]


@pytest.mark.parametrize("paged", [False, True], ids=["stacked", "paged"])
@pytest.mark.parametrize("case", RANK_LAYOUT_CASES, ids=lambda c: f"r{c[0]}-{c[1]}x{c[2]}-M{c[3]}")
@pytest.mark.parametrize("form", ["sgmv", "bgmv"])
def test_rank_aware_a_layouts(dev, case, paged, form):
    r_max, d_in, d_out, M, slot_ranks = case
    rng = np.random.default_rng(7 + r_max)
    g = W.generator(7 + r_max, dev)
    ranks = np.asarray(slot_ranks, np.int32)
    kw = dict(num_slots=len(ranks), num_layers=1, r_max=r_max, d_in=d_in, d_out=d_out, dtype=torch.bfloat16,
              gen=g, device=dev, ranks=ranks)
    pool = W.paged_pool(rng=rng, **kw) if paged else W.stacked_pool(**kw)
    slots = (np.arange(M) % len(ranks)).astype(np.int32)
    slots[::7] = -1
    batch = W.batch_from_segments(np.ones(M, np.int64), slots).to(dev)  # one row per segment
    x = W.normal((M, d_in), 1.0, torch.bfloat16, g, dev)
    y = W.uniform((M, d_out), -1, 1, torch.bfloat16, g, dev)
    op = W.Op("rank_layouts", pool, 0, x, y)
    h = m.make_pool(pool)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    g2, g1 = Guarded(op.y, r_max), Guarded(op.y, r_max)
    if form == "sgmv":
        m.lora_sgmv_shrink(g2.v, x, h, batch.seg_offsets, batch.seg_slot, 0, st)
        m.lora_sgmv_expand(g2.y, g2.v, h, batch.seg_offsets, batch.seg_slot, 0, st)
        m.lora_sgmv(g1.y, x, h, batch.seg_offsets, batch.seg_slot, 0, g1.v, st)
    else:
        m.lora_bgmv_shrink(g2.v, x, h, batch.row_slot, 0, st)
        m.lora_bgmv_expand(g2.y, g2.v, h, batch.row_slot, 0, st)
        m.lora_bgmv(g1.y, x, h, batch.row_slot, 0, g1.v, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    g2.check(True)
    g1.check(False)
    check_op(op, batch, form, g2.y, g2.v, what="two-phase")
    check_op(op, batch, form, g1.y, what="fused")

def test_status_contract_matches_oracle(dev):
    """Bad offsets / slots / ranks / pages: same status bits as the oracle, affected rows
    untouched bit for bit, all other rows correct."""
    dt = torch.bfloat16
    op, batch = make_case(dev, 7, dtype=dt, paged=True, r_max=16, d_in=64, d_out=48, M=12, num_slots=4)
    pool = op.pool
    op_pool = oracle_pool(pool)

    def both(form, meta, rank=None, a_tab=None, b_tab=None):
        rk = pool.rank if rank is None else rank
        at = pool.a_page_table if a_tab is None else a_tab
        bt = pool.b_page_table if b_tab is None else b_tab
        p2 = W.Pool(dt, pool.num_slots, pool.num_layers, pool.r_max, pool.d_in, pool.d_out, rk, pool.scale,
                    pages=pool.pages, a_page_table=at, b_page_table=bt)
        h = m.make_pool(p2)
        y = op.y.clone()
        v = new_v(12, 16, dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        if form == "sgmv":
            off, ss = meta
            m.lora_sgmv(y, op.x, h, off.to(dev), ss.to(dev), op.layer, v, st)
        else:
            m.lora_bgmv(y, op.x, h, meta.to(dev), op.layer, v, st)
        torch.cuda.synchronize()
        opool = oracle.Pool(dtype=odt(dt), num_slots=p2.num_slots, num_layers=p2.num_layers, r_max=16, d_in=64,
                            d_out=48, rank=rk.cpu().numpy(), scale=pool.scale.cpu().numpy(),
                            pages=op_pool.pages, a_page_table=at.cpu().numpy(), b_page_table=bt.cpu().numpy())
        if form == "sgmv":
            yo, _, _, so = oracle.sgmv(opool, op.layer, bits(op.x), bits(op.y), meta[0].numpy(), meta[1].numpy())
        else:
            yo, _, _, so = oracle.bgmv(opool, op.layer, bits(op.x), bits(op.y), meta.numpy())
        return bits(y), yo, int(st.item()), so

    t = lambda a: torch.tensor(a, dtype=torch.int32)
    for off in ([1, 5, 12], [0, 7, 5, 12], [0, 6, 13]):
        g, o, sg, so = both("sgmv", (t(off), t([0] * (len(off) - 1))))
        assert sg == so == m.STATUS_BAD_OFFSETS and np.array_equal(g, bits(op.y))
    slots = t([0, 9, -1, 1, -3, 2, 3, 0, 1, 2, 3, -1])
    g, o, sg, so = both("bgmv", slots)
    assert sg == so == m.STATUS_BAD_SLOT
    for i in (1, 2, 4, 11):
        assert np.array_equal(g[i], bits(op.y)[i])
    ok_rows = [i for i in range(12) if i not in (1, 2, 4, 11)]
    assert_close(oracle.decode(g[ok_rows], odt(dt)), oracle.decode(o[ok_rows], odt(dt)), "status bgmv")
    rk = pool.rank.clone()
    rk[1] = 0
    rk[2] = 17
    g, o, sg, so = both("bgmv", t([0, 1, 2, 3] * 3), rank=rk)
    assert sg == so == m.STATUS_BAD_RANK
    assert np.array_equal(g[1::4], bits(op.y)[1::4]) and np.array_equal(g[2::4], bits(op.y)[2::4])
    at = pool.a_page_table.clone()
    at[3, op.layer, 0] = pool.pages.shape[0]
    g, o, sg, so = both("bgmv", t([0, 1, 2, 3] * 3), a_tab=at)
    assert sg == so == m.STATUS_BAD_PAGE and np.array_equal(g[3::4], bits(op.y)[3::4])
    assert_close(oracle.decode(g[0::4], odt(dt)), oracle.decode(o[0::4], odt(dt)), "bad page, other rows")


def test_minus_one_rows_keep_nan_payloads(dev):
    op, batch = make_case(dev, 11, dtype=torch.bfloat16, paged=False, r_max=8, d_in=64, d_out=64, M=6)
    y = op.y.clone()
    y[1].view(torch.int16).fill_(0x7F85)  # NaN with a payload
    y[3].view(torch.int16).fill_(-0x8000)  # -0.0
    slots = torch.tensor([0, -1, 1, -1, 2, 0], dtype=torch.int32, device=dev)
    yb = bits(y)
    h = m.make_pool(op.pool)
    m.lora_bgmv(y, op.x, h, slots, op.layer, new_v(6, 8, dev))
    torch.cuda.synchronize()
    assert np.array_equal(bits(y)[[1, 3]], yb[[1, 3]])


def test_deterministic_and_forms_agree(dev):
    """Same call twice: identical bits (fixed summation order, no atomics). BGMV on rows grouped
    like an SGMV batch, SGMV, and a grouped call all match the oracle; their split of d_in may
    differ (it follows the tile count), so they agree within tolerance, not bit for bit."""
    w = W.sgmv_decode_7b(device=dev, dist="uniform", num_layers=1)
    op = w.ops[0]
    h = m.make_pool(op.pool)
    outs = []
    for _ in range(2):
        y = op.y.clone()
        m.lora_sgmv(y, op.x, h, w.batch.seg_offsets, w.batch.seg_slot, 0, new_v(32, 16, dev))
        outs.append(y)
    yb = op.y.clone()
    m.lora_bgmv(yb, op.x, h, w.batch.row_slot, 0, new_v(32, 16, dev))
    yg = [op.y.clone() for _ in range(3)]
    m.lora_sgmv_grouped([(yg[q], op.x, h, 0, new_v(32, 16, dev)) for q in range(3)], w.batch.seg_offsets,
                        w.batch.seg_slot)
    torch.cuda.synchronize()
    assert np.array_equal(bits(outs[0]), bits(outs[1]))
    check_op(op, w.batch, "sgmv", outs[0], what="sgmv")
    check_op(op, w.batch, "bgmv", yb, what="bgmv of the grouped rows")
    for q in range(3):
        check_op(op, w.batch, "sgmv", yg[q], what=f"grouped problem {q}")
        assert np.array_equal(bits(yg[0]), bits(yg[q]))
    v1, v2 = new_v(32, 16, dev), new_v(32, 16, dev)
    m.lora_sgmv_shrink(v1, op.x, h, w.batch.seg_offsets, w.batch.seg_slot, 0)
    m.lora_sgmv_shrink(v2, op.x, h, w.batch.seg_offsets, w.batch.seg_slot, 0)
    torch.cuda.synchronize()
    assert torch.equal(v1, v2)


def test_host_errors_launch_nothing(dev):
    op, batch = make_case(dev, 3, dtype=torch.bfloat16, paged=False, r_max=8, d_in=64, d_out=64, M=4)
    before = m.launch_count()
    with pytest.raises(m.MloraError) as e:
        m.lora_sgmv(op.y, op.x, op.pool, batch.seg_offsets, batch.seg_slot, 5, new_v(4, 8, dev))
    assert e.value.code == m.ERR_SHAPE
    with pytest.raises(m.MloraError) as e:
        m.lora_sgmv(op.y[:, 1:], op.x, op.pool, batch.seg_offsets, batch.seg_slot, 0, new_v(4, 8, dev))
    assert e.value.code in (m.ERR_ALIGN, m.ERR_SHAPE)
    assert m.launch_count() == before


# Device-side grouping of BGMV rows (lora_bgmv_ex): the rows are walked in (rank descending, slot)
# order computed on the GPU; the caller's rows, x and y stay in place. On pools of r_max 32 and
# more the grouped rows are streamed one CTA per row.
@pytest.mark.parametrize("paged", [False, True], ids=["stacked", "paged"])
@pytest.mark.parametrize("M", [7, 200, 1500])
def test_bgmv_row_grouping_same_bits_and_oracle(dev, paged, M):
    rng = np.random.default_rng(M + paged)
    g = W.generator(M, dev)
    S = 60
    ranks = rng.choice(np.array([1, 8, 16, 32, 64], np.int32), S)
    kw = dict(num_slots=S, num_layers=1, r_max=64, d_in=1024, d_out=520, dtype=torch.bfloat16, gen=g, device=dev,
              ranks=ranks)
    pool = W.paged_pool(rng=rng, page_elems=512, **kw) if paged else W.stacked_pool(**kw)
    slots = rng.choice(S, M, p=W.zipf_probs(S, 1.2)).astype(np.int32)
    slots[::9] = -1
    batch = W.batch_from_slots(slots, sgmv=False).to(dev)
    x = W.normal((M, 1024), 1.0, torch.bfloat16, g, dev)
    y0 = W.uniform((M, 520), -1, 1, torch.bfloat16, g, dev)
    h = m.make_pool(pool)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = {}
    for name, flags in (("grouped", m.LAUNCH_GROUP_ROWS), ("grouped again", m.LAUNCH_GROUP_ROWS),
                        ("plain", m.LAUNCH_NO_GROUPING), ("default", 0)):
        y = y0.clone()
        before = m.launch_count()
        m.lora_bgmv_ex(y, x, h, batch.row_slot, 0, new_v(M, 64, dev), flags, st)
        torch.cuda.synchronize()
        launches = m.launch_count() - before
        assert launches == (2 if flags == m.LAUNCH_GROUP_ROWS or (flags == 0 and M >= 128) else 1), name
        outs[name] = y
    assert st.item() == 0
    # the grouped rows of this heterogeneous-rank pool are streamed one CTA per row (another order
    # of the sums than the plain launch's): each form against the oracle; a call is deterministic
    assert np.array_equal(bits(outs["grouped"]), bits(outs["grouped again"])), "grouped call not deterministic"
    assert np.array_equal(bits(outs["default"]), bits(outs["grouped" if M >= 128 else "plain"]))
    for name in ("grouped", "plain"):
        check_op(W.Op(name, pool, 0, x, y0), batch, "bgmv", outs[name], what=f"{name} BGMV")


def test_bgmv_row_grouping_status_contract(dev):
    """Invalid slots and ranks are still reported, and their rows left untouched, when the rows are
    grouped (invalid rows sort last)."""
    op, batch = make_case(dev, 5, dtype=torch.bfloat16, paged=False, r_max=16, d_in=64, d_out=48, M=12, num_slots=4)
    rk = op.pool.rank.clone()
    rk[1] = 0
    p2 = W.Pool(op.pool.dtype, 4, op.pool.num_layers, 16, 64, 48, rk, op.pool.scale, a_t=op.pool.a_t, b=op.pool.b)
    slots = torch.tensor([0, 9, -1, 1, -3, 2, 3, 0, 1, 2, 3, -1], dtype=torch.int32, device=dev)
    y = op.y.clone()
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    m.lora_bgmv_ex(y, op.x, m.make_pool(p2), slots, op.layer, new_v(12, 16, dev), m.LAUNCH_GROUP_ROWS, st)
    torch.cuda.synchronize()
    assert st.item() == m.STATUS_BAD_SLOT | m.STATUS_BAD_RANK
    for i in (1, 2, 3, 4, 8, 11):
        assert np.array_equal(bits(y)[i], bits(op.y)[i])
    good = slots.cpu().clone()
    good[[1, 2, 3, 4, 8, 11]] = -1
    check_op(op, W.Batch(12, good.to(dev), None, None), "bgmv", y, what="valid rows, grouped")


def test_streaming_status_contract(dev):
    """The streaming kernel (grouped BGMV rows on a pool of r_max >= 32, and the short segments of a
    fused SGMV call whose long segments take the tensor cores): the same status bits as the oracle
    for bad slots, ranks, page ids and offsets; affected rows untouched bit for bit; other rows
    correct."""
    dt = torch.bfloat16
    rng = np.random.default_rng(31)
    g = W.generator(31, dev)
    S, M = 6, 300
    ranks = np.array([32, 8, 17, 32, 1, 24], np.int32)
    pool = W.paged_pool(num_slots=S, num_layers=1, r_max=32, d_in=256, d_out=200, dtype=dt, gen=g, device=dev, rng=rng,
                        ranks=ranks, page_elems=128)
    x = W.normal((M, 256), 1.0, dt, g, dev)
    y0 = W.uniform((M, 200), -1, 1, dt, g, dev)
    op_pool = oracle_pool(pool)

    def both(form, meta, rank=None, a_tab=None):
        rk = pool.rank if rank is None else rank
        at = pool.a_page_table if a_tab is None else a_tab
        p2 = W.Pool(dt, S, 1, 32, 256, 200, rk, pool.scale, pages=pool.pages, a_page_table=at,
                    b_page_table=pool.b_page_table)
        h = m.make_pool(p2)
        y = y0.clone()
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        before = m.launch_count()
        if form == "sgmv":
            off, ss = meta
            m.lora_sgmv(y, x, h, off.to(dev), ss.to(dev), 0, new_v(M, 32, dev), st)
        else:
            m.lora_bgmv_ex(y, x, h, meta.to(dev), 0, new_v(M, 32, dev), m.LAUNCH_GROUP_ROWS, st)
        torch.cuda.synchronize()
        assert m.launch_count() - before == (3 if form == "sgmv" else 2)
        opool = oracle.Pool(dtype=odt(dt), num_slots=S, num_layers=1, r_max=32, d_in=256, d_out=200,
                            rank=rk.cpu().numpy(), scale=pool.scale.cpu().numpy(), pages=op_pool.pages,
                            a_page_table=at.cpu().numpy(), b_page_table=pool.b_page_table.cpu().numpy())
        if form == "sgmv":
            yo, _, _, so = oracle.sgmv(opool, 0, bits(x), bits(y0), meta[0].numpy(), meta[1].numpy())
        else:
            yo, _, _, so = oracle.bgmv(opool, 0, bits(x), bits(y0), meta.numpy())
        return bits(y), yo, int(st.item()), so

    t = lambda a: torch.tensor(a, dtype=torch.int32)
    # BGMV: slots with repeats (segments of several rows), -1 rows, slots past the pool
    slots = rng.integers(0, S, M).astype(np.int32)
    slots[::7] = -1
    slots[3::11] = 9
    slots[5::13] = -4
    gb, ob, sg, so = both("bgmv", t(slots))
    assert sg == so == m.STATUS_BAD_SLOT
    bad = (slots < 0) | (slots >= S)
    assert np.array_equal(gb[bad], bits(y0)[bad])
    assert_close(oracle.decode(gb[~bad], odt(dt)), oracle.decode(ob[~bad], odt(dt)), "streamed bgmv, valid rows")
    # a rank out of range, then a page id out of range
    rk = pool.rank.clone()
    rk[2] = 0
    s2 = np.tile(np.arange(S, dtype=np.int32), M // S)
    gb, ob, sg, so = both("bgmv", t(s2), rank=rk)
    assert sg == so == m.STATUS_BAD_RANK and np.array_equal(gb[s2 == 2], bits(y0)[s2 == 2])
    at = pool.a_page_table.clone()
    at[3, 0, 5, 1] = pool.pages.shape[0]
    gb, ob, sg, so = both("bgmv", t(s2), a_tab=at)
    assert sg == so == m.STATUS_BAD_PAGE and np.array_equal(gb[s2 == 3], bits(y0)[s2 == 3])
    ok = (s2 != 3)
    assert_close(oracle.decode(gb[ok], odt(dt)), oracle.decode(ob[ok], odt(dt)), "bad page, other rows")
    # SGMV: a long segment on the tensor cores, short ones streamed, one short segment on a bad slot
    off, ss = t([0, 260, 265, 266, 269, 300]), t([0, 1, 9, 3, 5])
    gs, os_, sg, so = both("sgmv", (off, ss))
    assert sg == so == m.STATUS_BAD_SLOT and np.array_equal(gs[265:266], bits(y0)[265:266])
    keep = np.r_[0:265, 266:300]
    assert_close(oracle.decode(gs[keep], odt(dt)), oracle.decode(os_[keep], odt(dt)), "streamed sgmv, valid rows")
    # malformed offsets: nothing written, the bit reported
    for bad_off in ([0, 260, 250, 269, 280, 300], [0, 260, 265, 266, 269, 299]):
        gs, os_, sg, so = both("sgmv", (t(bad_off), ss))
        assert sg == so == m.STATUS_BAD_OFFSETS and np.array_equal(gs, bits(y0))
