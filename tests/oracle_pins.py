"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each `pin_*` takes an oracle build (``oracle.OracleLib``) and raises AssertionError when the
build disagrees with an independent fact:
  * the IEEE-754 formats themselves (exhaustive decode against numpy / torch, ties, overflow,
    subnormals, round trip),
  * the Identical distribution, which is one dense GEMM (numpy BLAS),
  * the merged form W' = W + s·A·B ("Multi-LoRA Serving, in depth": with one adapter you
    can merge it; S-LoRA digest, section 2: merged weights),
  * a rank-r closed form with power-of-two operands (exact in every precision),
  * slot and layer identification by power-of-two weights (exact), on stacked and paged pools,
  * slot -1 rows left bit-for-bit untouched ("-1 means no adapter", the reference loop of
    "Multi-LoRA Serving, in depth"),
  * the status contract for metadata the pages do not define.
``tests/test_oracle_pins.py`` runs them on the real oracle; ``tests/test_oracle_mutants.py``
runs them on builds with planted mistakes and requires that some pin fails for each.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

BF16, FP16 = O.DTYPE_BF16, O.DTYPE_FP16


# ---------------------------------------------------------------------------------------------
# library conversions used as independent references


def lib_decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    bits = np.asarray(bits, np.uint16)
    if dtype == FP16:
        return bits.view(np.float16).astype(np.float64)
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def lib_round(values: np.ndarray, dtype: int) -> np.ndarray:
    """numpy's direct double->half conversion; torch's float->bfloat16 (values must be fp32-exact)."""
    values = np.asarray(values, np.float64)
    if dtype == FP16:
        with np.errstate(over="ignore"):
            return values.astype(np.float16).view(np.uint16)
    f32 = values.astype(np.float32)
    assert np.array_equal(f32.astype(np.float64), values, equal_nan=True)
    return torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def enc(values, dtype) -> np.ndarray:
    """Bit patterns of values that are exactly representable (checked)."""
    v = np.asarray(values, np.float64)
    b = lib_round(v, dtype)
    assert np.array_equal(lib_decode(b, dtype), v), "value not representable"
    return b


def _same_bits_or_both_nan(a, b, dtype):
    a, b = np.asarray(a, np.uint16), np.asarray(b, np.uint16)
    da, db = lib_decode(a, dtype), lib_decode(b, dtype)
    both_nan = np.isnan(da) & np.isnan(db)
    return np.all((a == b) | both_nan)


# ---------------------------------------------------------------------------------------------
# pool builders for the pins (host numpy, exact values)


def stacked(dtype, a_t_vals, b_vals, rank, scale):
    a_t_vals, b_vals = np.asarray(a_t_vals, np.float64), np.asarray(b_vals, np.float64)
    S, L, R, d_in = a_t_vals.shape
    d_out = b_vals.shape[-1]
    a_bits = np.where(np.isnan(a_t_vals), 0x7E01 if dtype == FP16 else 0x7FC1, 0).astype(np.uint16)
    b_bits = np.where(np.isnan(b_vals), 0x7E01 if dtype == FP16 else 0x7FC1, 0).astype(np.uint16)
    fin_a, fin_b = ~np.isnan(a_t_vals), ~np.isnan(b_vals)
    a_bits[fin_a] = lib_round(a_t_vals[fin_a], dtype)
    b_bits[fin_b] = lib_round(b_vals[fin_b], dtype)
    return O.Pool(dtype=dtype, num_slots=S, num_layers=L, r_max=R, d_in=d_in, d_out=d_out, rank=rank, scale=scale,
                  a_t=a_bits, b=b_bits)


def to_paged(pool: O.Pool, rng, page_elems=None, extra_free=7):
    """Same adapters as a stacked pool, moved to randomly placed pages; free pages and page
    tails hold NaN. A vector longer than page_elems is cut into ceil(d / page_elems) pages, each
    placed at its own random position (S-LoRA "Unified Paging": a page is one H-vector)."""
    S, L, R = pool.num_slots, pool.num_layers, pool.r_max
    page_elems = max(pool.d_in, pool.d_out) + 3 if page_elems is None else page_elems
    pa_n, pb_n = -(-pool.d_in // page_elems), -(-pool.d_out // page_elems)
    used = L * int(pool.rank.sum()) * (pa_n + pb_n)
    num_pages = used + extra_free
    phys = iter(rng.permutation(num_pages))
    nan = 0x7E01 if pool.dtype == FP16 else 0x7FC1
    pages = np.full((num_pages, page_elems), nan, np.uint16)
    a_tab = np.full((S, L, R, pa_n), -1, np.int32)
    b_tab = np.full((S, L, R, pb_n), -1, np.int32)
    a_t = pool.a_t.reshape(S, L, R, pool.d_in)
    b = pool.b.reshape(S, L, R, pool.d_out)
    for s in range(S):
        for layer in range(L):
            for j in range(int(pool.rank[s])):
                for tab, src, d, n in ((a_tab, a_t, pool.d_in, pa_n), (b_tab, b, pool.d_out, pb_n)):
                    for q in range(n):
                        pg = next(phys)
                        tab[s, layer, j, q] = pg
                        piece = src[s, layer, j, q * page_elems:(q + 1) * page_elems]
                        pages[pg, :piece.size] = piece
    return O.Pool(dtype=pool.dtype, num_slots=S, num_layers=L, r_max=R, d_in=pool.d_in, d_out=pool.d_out,
                  rank=pool.rank, scale=pool.scale, pages=pages, a_page_table=a_tab, b_page_table=b_tab)


def random_pool(rng, dtype, S, L, R, d_in, d_out, ranks=None, scales=None):
    ranks = np.full(S, R, np.int32) if ranks is None else np.asarray(ranks, np.int32)
    scales = rng.choice([0.25, 0.5, 1.0, 2.0, 4.0], S).astype(np.float32) if scales is None else scales
    # values already on the I/O grid (round through the library), padding rows NaN
    a = lib_decode(lib_round(rng.standard_normal((S, L, R, d_in)).astype(np.float32) / 8, dtype), dtype)
    b = lib_decode(lib_round(rng.standard_normal((S, L, R, d_out)).astype(np.float32) / 8, dtype), dtype)
    for s in range(S):
        a[s, :, ranks[s]:] = np.nan
        b[s, :, ranks[s]:] = np.nan
    return stacked(dtype, a, b, ranks, scales), a, b


def random_act(rng, dtype, M, d):
    return lib_round(rng.uniform(-1, 1, (M, d)).astype(np.float32), dtype)


def dense_A(a_t, s, layer, rank):
    """A_s (d_in x rank) from the stored A^T rows."""
    return a_t[s, layer, :rank].T


# ---------------------------------------------------------------------------------------------
# pins: number formats


def pin_decode_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dt in (BF16, FP16):
        got, ref = orc.decode(bits, dt), lib_decode(bits, dt)
        same = (got == ref) | (np.isnan(got) & np.isnan(ref))
        assert same.all(), f"decode differs for {np.count_nonzero(~same)} patterns (dtype {dt})"
        # signed zeros keep their sign
        assert np.signbit(orc.decode(np.array([0x8000], np.uint16), dt))[0]


def pin_round_trip_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dt in (BF16, FP16):
        vals = orc.decode(bits, dt)
        ok = ~np.isnan(vals)
        back = orc.round_to(vals[ok], dt)
        assert np.array_equal(back, bits[ok]), f"round(decode(b)) != b (dtype {dt})"


def pin_round_matches_library(orc, n=200_000, seed=11):
    rng = np.random.default_rng(seed)
    # fp16: arbitrary doubles over the whole range incl. subnormals and overflow (numpy rounds
    # double->half directly)
    mag = np.exp2(rng.uniform(-27, 17, n))
    v = mag * rng.choice([-1.0, 1.0], n)
    assert _same_bits_or_both_nan(orc.round_to(v, FP16), lib_round(v, FP16), FP16), "fp16 rounding differs"
    # bf16: random finite fp32 bit patterns (torch rounds float->bfloat16)
    raw = rng.integers(0, 2 ** 32, n, dtype=np.uint64).astype(np.uint32)
    f = raw.view(np.float32)
    f = f[np.isfinite(f)].astype(np.float64)
    assert _same_bits_or_both_nan(orc.round_to(f, BF16), lib_round(f, BF16), BF16), "bf16 rounding differs"


def pin_round_ties(orc):
    cases = [
        # (value, dtype, expected bits)
        (1 + 2 ** -8, BF16, 0x3F80),  # tie -> even (down)
        (1 + 3 * 2 ** -8, BF16, 0x3F82),  # tie -> even (up)
        (-(1 + 2 ** -8), BF16, 0xBF80),
        ((2 - 2 ** -8) * 2.0 ** 127, BF16, 0x7F80),  # tie above the largest finite -> +Inf
        ((2 - 2 ** -7) * 2.0 ** 127, BF16, 0x7F7F),  # largest finite stays
        (2.0 ** -134, BF16, 0x0000),  # half the smallest subnormal: tie -> 0
        (3 * 2.0 ** -134, BF16, 0x0002),  # 1.5 subnormal quanta: tie -> 2
        (1 + 2 ** -11, FP16, 0x3C00),
        (1 + 3 * 2 ** -11, FP16, 0x3C02),
        (65504.0, FP16, 0x7BFF),
        (65519.99, FP16, 0x7BFF),
        (65520.0, FP16, 0x7C00),  # tie between 65504 and 2^16 -> even -> Inf
        (-65520.0, FP16, 0xFC00),
        (2.0 ** -25, FP16, 0x0000),
        (3 * 2.0 ** -25, FP16, 0x0002),
        (2.0 ** -24, FP16, 0x0001),
        (2.0 ** -14 - 2.0 ** -25, FP16, 0x0400),  # rounds up into the smallest normal
        (-0.0, FP16, 0x8000),
        (-0.0, BF16, 0x8000),
    ]
    for v, dt, want in cases:
        got = int(orc.round_to([v], dt)[0])
        assert got == want, f"round({v!r}, {dt}) = {got:#06x}, want {want:#06x}"
    assert orc.round_to([np.inf], FP16)[0] == 0x7C00 and orc.round_to([-np.inf], BF16)[0] == 0xFF80
    assert np.isnan(orc.decode(orc.round_to([np.nan], BF16), BF16)[0])


# ---------------------------------------------------------------------------------------------
# pins: the operator


def pin_identical_is_dense_gemm(orc, seed=21):
    """One adapter for every row (Punica's Identical distribution): the result is the dense
    y + s·(X·A)·B, here computed by numpy's BLAS."""
    rng = np.random.default_rng(seed)
    for dt in (BF16, FP16):
        S, L, R, d_in, d_out, M = 3, 2, 5, 40, 24, 13
        pool, a, b = random_pool(rng, dt, S, L, R, d_in, d_out)
        s, layer = 2, 1
        x = random_act(rng, dt, M, d_in)
        y = random_act(rng, dt, M, d_out)
        X, Y = lib_decode(x, dt), lib_decode(y, dt)
        A, B = dense_A(a, s, layer, R), b[s, layer, :R]
        sc = float(pool.scale[s])
        V_ref = X @ A
        Y_ref = Y + sc * (V_ref @ B)
        for form in ("sgmv", "bgmv"):
            if form == "sgmv":
                y_out, v, y_ex, st = orc.sgmv(pool, layer, x, y, [0, M], [s])
            else:
                y_out, v, y_ex, st = orc.bgmv(pool, layer, x, y, np.full(M, s))
            assert st == 0
            scale_v = np.abs(X) @ np.abs(A)
            assert np.all(np.abs(v[:, :R] - V_ref) <= 1e-12 * (scale_v + 1e-300)), "v != X·A"
            scale_y = np.abs(Y) + sc * (scale_v @ np.abs(B))
            assert np.all(np.abs(y_ex - Y_ref) <= 1e-12 * scale_y), "y_exact != y + s·X·A·B"
            if dt == FP16:  # numpy rounds double->half directly: the output is RNE(y_exact)
                assert np.array_equal(y_out, lib_round(y_ex, dt)), "rounding of y"


def pin_merged_identity(orc, seed=22):
    """Unmerged result = merged W' = W + s·A·B, row by row with a slot per row."""
    rng = np.random.default_rng(seed)
    dt = BF16
    S, L, R, d_in, d_out, M = 4, 1, 8, 48, 64, 11
    ranks = np.array([8, 3, 5, 1], np.int32)
    pool, a, b = random_pool(rng, dt, S, L, R, d_in, d_out, ranks=ranks)
    x = random_act(rng, dt, M, d_in)
    y = random_act(rng, dt, M, d_out)
    X, Y = lib_decode(x, dt), lib_decode(y, dt)
    row_slot = rng.integers(-1, S, M).astype(np.int32)
    W = rng.standard_normal((d_in, d_out))
    y_out, v, y_ex, st = orc.bgmv(pool, 0, x, y, row_slot)
    assert st == 0
    for i in range(M):
        s = row_slot[i]
        if s < 0:
            continue
        r = ranks[s]
        Wm = W + float(pool.scale[s]) * (dense_A(a, s, 0, r) @ b[s, 0, :r])
        delta_merged = X[i] @ Wm - X[i] @ W
        tol = 1e-10 * (np.abs(X[i]) @ np.abs(Wm) + 1.0)
        assert np.all(np.abs((y_ex[i] - Y[i]) - delta_merged) <= tol), f"row {i}: unmerged != merged"


def pin_rank_closed_form(orc):
    """A = c·1, B = b·1, x = 1 with powers of two: delta = s·rank·d_in·c·b exactly, and the
    rounded output is the exact sum's bit pattern."""
    for dt in (BF16, FP16):
        S, L, R, d_in, d_out = 3, 2, 4, 64, 16
        ranks = np.array([1, 4, 2], np.int32)
        scales = np.array([2.0, 0.5, 0.25], np.float32)
        c, bb = 2.0 ** -4, 2.0 ** -3
        a = np.full((S, L, R, d_in), c)
        b = np.full((S, L, R, d_out), bb)
        for s in range(S):
            a[s, :, ranks[s]:] = np.nan
            b[s, :, ranks[s]:] = np.nan
        pool = stacked(dt, a, b, ranks, scales)
        M = 3
        x = enc(np.ones((M, d_in)), dt)
        y0 = 0.5
        y = enc(np.full((M, d_out), y0), dt)
        y_out, v, y_ex, st = orc.sgmv(pool, 1, x, y, [0, 1, 2, 3], [0, 1, 2])
        assert st == 0
        for s in range(S):
            delta = float(scales[s]) * ranks[s] * d_in * c * bb
            assert np.all(v[s, :ranks[s]] == d_in * c), "v closed form"
            assert np.all(y_ex[s] == y0 + delta), "delta closed form"
            assert np.all(y_out[s] == enc([y0 + delta], dt)[0]), "rounded closed form"
    # fp16 result in the subnormal range, exactly representable
    a = np.full((1, 1, 1, 8), 2.0 ** -12)
    b = np.full((1, 1, 1, 8), 2.0 ** -10)
    pool = stacked(FP16, a, b, [1], [1.0])
    y_out, _, y_ex, _ = orc.bgmv(pool, 0, enc(np.ones((1, 8)), FP16), enc(np.zeros((1, 8)), FP16), [0])
    assert np.all(y_ex == 8 * 2.0 ** -12 * 2.0 ** -10)  # = 2^-19, below the smallest normal 2^-14
    assert np.all(y_out == 0x0020)  # 2^-19 / 2^-24 = 32 subnormal quanta


def _ident_pool(dt, S, L, R, d_in, d_out, ranks):
    """A_s of layer l = 2^-(1 + s + 8l)·1, B = 1; rows past rank are NaN."""
    a = np.empty((S, L, R, d_in))
    b = np.ones((S, L, R, d_out))
    for s in range(S):
        for layer in range(L):
            a[s, layer] = 2.0 ** -(1 + s + 8 * layer)
        a[s, :, ranks[s]:] = np.nan
        b[s, :, ranks[s]:] = np.nan
    return stacked(dt, a, b, ranks, np.ones(S, np.float32))


def _check_identification(orc, pool, layer, ranks, x_onehot_rows, row_slot_expected, y_out, y_ex, v, y_in, dt):
    for i, s in enumerate(row_slot_expected):
        if s < 0:
            assert np.array_equal(y_out[i], y_in[i]), f"row {i} (slot -1) changed"
            assert np.all(np.isnan(v[i])), f"row {i} (slot -1) got a v"
            continue
        want = ranks[s] * 2.0 ** -(1 + s + 8 * layer)
        assert np.all(y_ex[i] == want), f"row {i}: delta {y_ex[i][0]} does not identify slot {s} layer {layer}"
        assert np.all(y_out[i] == enc([want], dt)[0])


def pin_slot_identification(orc, seed=23):
    """Power-of-two weights per (slot, layer) and one-hot x: each row's delta names the slot
    and layer it used. Random segments (empty ones, repeated slots, -1 segments), random BGMV
    slots with -1, on a stacked pool and on the same adapters in permuted pages."""
    rng = np.random.default_rng(seed)
    dt = BF16
    S, L, R, d_in, d_out = 6, 3, 4, 32, 24
    ranks = np.array([4, 1, 3, 2, 4, 1], np.int32)
    st_pool = _ident_pool(dt, S, L, R, d_in, d_out, ranks)
    pg_pool = to_paged(st_pool, rng)
    for trial in range(6):
        layer = trial % L
        nseg = int(rng.integers(1, 9))
        lens = rng.integers(0, 5, nseg)
        seg_slot = rng.integers(-1, S, nseg).astype(np.int32)
        M = int(lens.sum())
        off = np.r_[0, np.cumsum(lens)].astype(np.int32)
        expected = np.repeat(seg_slot, lens)
        x = enc(np.eye(d_in)[rng.integers(0, d_in, M)], dt) if M else np.zeros((0, d_in), np.uint16)
        y = enc(np.zeros((M, d_out)), dt)
        for pool in (st_pool, pg_pool):
            y_out, v, y_ex, st = orc.sgmv(pool, layer, x, y, off, seg_slot)
            assert st == 0
            _check_identification(orc, pool, layer, ranks, x, expected, y_out, y_ex, v, y, dt)
        row_slot = rng.integers(-1, S, M).astype(np.int32)
        for pool in (st_pool, pg_pool):
            y_out, v, y_ex, st = orc.bgmv(pool, layer, x, y, row_slot)
            assert st == 0
            _check_identification(orc, pool, layer, ranks, x, row_slot, y_out, y_ex, v, y, dt)


def pin_skip_rows_untouched(orc, seed=24):
    """Rows with slot -1 keep their exact bits (NaN payloads, -0.0) and get no v."""
    rng = np.random.default_rng(seed)
    for dt in (BF16, FP16):
        pool, _, _ = random_pool(rng, dt, 2, 1, 4, 16, 16)
        M = 6
        x = random_act(rng, dt, M, 16)
        y = random_act(rng, dt, M, 16)
        y[1, :] = 0x8000  # -0.0
        y[3, :5] = 0x7E55 if dt == FP16 else 0x7F85  # NaN payloads
        y[3, 5:] = 0xFE01 if dt == FP16 else 0xFFC3
        row_slot = np.array([0, -1, 1, -1, 0, -1], np.int32)
        y_out, v, _, st = orc.bgmv(pool, 0, x, y, row_slot)
        assert st == 0
        for i in (1, 3, 5):
            assert np.array_equal(y_out[i], y[i]) and np.all(np.isnan(v[i]))
        y_out2, v2, _, st = orc.sgmv(pool, 0, x, y, [0, 1, 2, 3, 4, 6], [0, -1, 1, -1, 0])
        assert st == 0 and np.array_equal(y_out2[1], y[1]) and np.array_equal(y_out2[3], y[3])


def pin_status_contract(orc, seed=25):
    """Metadata the pages leave undefined: status bits, affected rows untouched, others done."""
    rng = np.random.default_rng(seed)
    dt = BF16
    pool, _, _ = random_pool(rng, dt, 3, 1, 4, 16, 8, ranks=[4, 2, 4])
    M = 4
    x = random_act(rng, dt, M, 16)
    y = random_act(rng, dt, M, 8)
    for off in ([1, 2, 4], [0, 3, 2], [0, 2, 3]):  # s[0] != 0, decreasing, s[n] != M
        y_out, v, _, st = orc.sgmv(pool, 0, x, y, off, [0, 1])
        assert st == O.BAD_OFFSETS and np.array_equal(y_out, y) and np.all(np.isnan(v))
    y_out, v, _, st = orc.bgmv(pool, 0, x, y, [0, 3, -2, 1])
    assert st == O.BAD_SLOT
    assert np.array_equal(y_out[1], y[1]) and np.array_equal(y_out[2], y[2])
    assert not np.array_equal(y_out[0], y[0]) and not np.array_equal(y_out[3], y[3])
    bad_rank = O.Pool(dtype=dt, num_slots=3, num_layers=1, r_max=4, d_in=16, d_out=8, rank=[4, 0, 5],
                      scale=pool.scale, a_t=pool.a_t, b=pool.b)
    y_out, v, _, st = orc.bgmv(bad_rank, 0, x, y, [0, 1, 2, 0])
    assert st == O.BAD_RANK and np.array_equal(y_out[1:3], y[1:3]) and not np.array_equal(y_out[0], y[0])
    pg = to_paged(pool, rng)
    a_tab = pg.a_page_table.copy()
    a_tab[1, 0, 1] = pg.pages.shape[0]  # slot 1, j = 1 < rank 2: out of range
    b_tab = pg.b_page_table.copy()
    b_tab[2, 0, 0] = -1
    bad_pg = O.Pool(dtype=dt, num_slots=3, num_layers=1, r_max=4, d_in=16, d_out=8, rank=pool.rank,
                    scale=pool.scale, pages=pg.pages, a_page_table=a_tab, b_page_table=b_tab)
    v, st = orc.bgmv_shrink(bad_pg, 0, x, [0, 1, 2, 1])
    assert st == O.BAD_PAGE and np.all(np.isnan(v[1])) and np.all(np.isnan(v[3])) and not np.isnan(v[2, 0])
    y_out, _, st = orc.bgmv_expand(bad_pg, 0, np.ones((M, 4)), y, [0, 1, 2, 1])
    assert st == O.BAD_PAGE and np.array_equal(y_out[2], y[2]) and not np.array_equal(y_out[1], y[1])


def pin_sampled_rows(orc, seed=26):
    """Computing a sample of rows gives exactly those rows of the full computation."""
    rng = np.random.default_rng(seed)
    dt = BF16
    pool, _, _ = random_pool(rng, dt, 3, 2, 4, 24, 16)
    M = 9
    x, y = random_act(rng, dt, M, 24), random_act(rng, dt, M, 16)
    off, ss = [0, 2, 2, 7, 9], [1, 0, -1, 2]
    full = orc.sgmv(pool, 1, x, y, off, ss)
    rows = [8, 0, 4]
    part = orc.sgmv(pool, 1, x, y, off, ss, rows=rows)
    assert np.array_equal(part[0][rows], full[0][rows])
    assert np.array_equal(part[1][rows], full[1][rows], equal_nan=True)
    others = [i for i in range(M) if i not in rows]
    assert np.array_equal(part[0][others], y[others]) and np.all(np.isnan(part[1][others]))


def pin_sgmv_equals_bgmv_on_the_same_rows(orc, seed=27):
    """The two forms state one computation (Punica section 3.4: a segment is a run of rows with one
    adapter; "Multi-LoRA Serving, in depth": a slot per row): SGMV over random segments (empty,
    repeated slots, -1) and BGMV with each row's slot taken from its segment give the same bits,
    on stacked and paged pools, in both dtypes."""
    rng = np.random.default_rng(seed)
    for dt in (BF16, FP16):
        for paged in (False, True):
            S, L, R, d_in, d_out, M = 5, 2, 8, 40, 24, 23
            pool, _, _ = random_pool(rng, dt, S, L, R, d_in, d_out, ranks=rng.integers(1, R + 1, S))
            if paged:
                pool = to_paged(pool, rng)
            cuts = np.sort(rng.integers(0, M + 1, 6))
            off = np.r_[0, cuts, M].astype(np.int32)
            ss = rng.integers(-1, S, len(off) - 1).astype(np.int32)
            row_slot = np.repeat(ss, np.diff(off)).astype(np.int32)
            x, y = random_act(rng, dt, M, d_in), random_act(rng, dt, M, d_out)
            for layer in range(L):
                ys, vs, _, sts = orc.sgmv(pool, layer, x, y, off, ss)
                yb, vb, _, stb = orc.bgmv(pool, layer, x, y, row_slot)
                assert sts == 0 and stb == 0
                assert np.array_equal(ys, yb), f"y differs between the forms (dtype {dt}, paged {paged})"
                assert np.array_equal(vs, vb, equal_nan=True), "v differs between the forms"


def pin_vectors_across_pages_equal_stacked(orc, seed=28):
    """S-LoRA "Unified Paging" with pages shorter than a vector (a rank-row of A^T or B spans
    ceil(d / page_elems) pages, each at its own place in the pool): the same adapters give the
    same bits as the stacked pool, for SGMV over random segments and for BGMV, in both dtypes, with
    page sizes that divide d, that do not, and that exceed it."""
    rng = np.random.default_rng(seed)
    for dt in (BF16, FP16):
        S, L, R, d_in, d_out, M = 4, 2, 6, 40, 24, 17
        pool, _, _ = random_pool(rng, dt, S, L, R, d_in, d_out, ranks=rng.integers(1, R + 1, S))
        cuts = np.sort(rng.integers(0, M + 1, 5))
        off = np.r_[0, cuts, M].astype(np.int32)
        ss = rng.integers(-1, S, len(off) - 1).astype(np.int32)
        row_slot = rng.integers(-1, S, M).astype(np.int32)
        x, y = random_act(rng, dt, M, d_in), random_act(rng, dt, M, d_out)
        for pe in (8, 12, 24, 64):
            paged = to_paged(pool, rng, page_elems=pe)
            for layer in range(L):
                want = orc.sgmv(pool, layer, x, y, off, ss)
                got = orc.sgmv(paged, layer, x, y, off, ss)
                assert got[3] == 0 and np.array_equal(got[0], want[0]), f"SGMV y differs with {pe}-element pages"
                assert np.array_equal(got[1], want[1], equal_nan=True), f"SGMV v differs with {pe}-element pages"
                want = orc.bgmv(pool, layer, x, y, row_slot)
                got = orc.bgmv(paged, layer, x, y, row_slot)
                assert got[3] == 0 and np.array_equal(got[0], want[0]), f"BGMV y differs with {pe}-element pages"


ALL_PINS = [pin_decode_exhaustive, pin_round_trip_exhaustive, pin_round_matches_library, pin_round_ties,
            pin_identical_is_dense_gemm, pin_merged_identity, pin_rank_closed_form, pin_slot_identification,
            pin_skip_rows_untouched, pin_status_contract, pin_sampled_rows, pin_sgmv_equals_bgmv_on_the_same_rows,
            pin_vectors_across_pages_equal_stacked]
