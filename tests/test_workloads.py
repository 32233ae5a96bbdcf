"""The seeded input generators: shapes, distributions and pool structure (CPU only)."""
import numpy as np
import torch

import workloads as W


def test_tiny_sgmv_layout():
    w = W.tiny_sgmv()
    assert w.batch.seg_offsets.tolist() == [0, 3, 8, 9, 16] and w.batch.seg_slot.tolist() == [0, 1, 2, 3]
    op = w.ops[0]
    assert op.x.shape == (16, 256) and op.x.dtype == torch.float16
    assert op.pool.a_t.shape == (4, 1, 8, 256) and torch.all(op.pool.scale == 2.0)
    assert float(op.x.abs().max()) <= 1.0


def test_distributions():
    rng = np.random.default_rng(0)
    assert W.draw_slots("distinct", 32, 32, rng).tolist() == list(range(32))
    u = W.draw_slots("uniform", 32, 32, rng)
    vals, counts = np.unique(u, return_counts=True)
    assert len(vals) == 8 and set(counts) == {4}
    assert set(W.draw_slots("identical", 32, 32, rng)) == {0}
    sk = W.draw_slots("skewed", 100_000, 32, np.random.default_rng(1), zipf_alpha=1.5)
    freq = np.bincount(sk, minlength=32) / sk.size
    assert np.allclose(freq, W.zipf_probs(32, 1.5), atol=5e-3)


def test_group_rows_and_segments():
    rs = np.array([3, 1, 3, -1, 1, 0, 3], np.int32)
    perm, off, ss = W.group_rows(rs)
    grouped = rs[perm]
    assert grouped.tolist() == sorted(rs.tolist())
    assert off.tolist() == [0, 1, 2, 4, 7] and ss.tolist() == [-1, 0, 1, 3]
    # stable: equal slots keep their original order
    assert perm[4:].tolist() == [0, 2, 6]


def test_decode_7b_small():
    w = W.sgmv_decode_7b(dist="uniform", num_layers=2, projections=[W.Projection("q", 64, 64),
                                                                     W.Projection("down", 96, 64)])
    assert len(w.ops) == 4
    off = w.batch.seg_offsets.numpy()
    assert off[0] == 0 and off[-1] == 32 and np.all(np.diff(off) == 4)
    assert torch.equal(torch.repeat_interleave(w.batch.seg_slot, torch.diff(w.batch.seg_offsets)),
                       w.batch.row_slot)


def test_paged_pool_structure():
    rng = np.random.default_rng(5)
    g = W.generator(5, "cpu")
    ranks = np.array([8, 16, 8, 32], np.int32)
    p = W.paged_pool(num_slots=4, num_layers=2, r_max=32, d_in=64, d_out=48, dtype=torch.bfloat16, gen=g,
                     device="cpu", rng=rng, ranks=ranks)
    used = 2 * 2 * ranks.sum()
    ids = torch.cat([p.a_page_table[p.a_page_table >= 0], p.b_page_table[p.b_page_table >= 0]])
    assert ids.numel() == used and ids.unique().numel() == used
    assert p.pages.shape[0] >= used * 1.09
    free = torch.ones(p.pages.shape[0], dtype=torch.bool)
    free[ids.long()] = False
    assert torch.isnan(p.pages[free].float()).all()
    for s in range(4):
        assert (p.a_page_table[s, :, ranks[s]:] == -1).all() and (p.a_page_table[s, :, :ranks[s]] >= 0).all()
    a_rows = p.pages[p.a_page_table[p.a_page_table >= 0].long()]
    assert torch.isfinite(a_rows[:, :64].float()).all() and torch.isnan(a_rows[:, 64:].float()).all()


def test_stacked_padding_poisoned():
    g = W.generator(3, "cpu")
    p = W.stacked_pool(num_slots=3, num_layers=1, r_max=8, d_in=16, d_out=16, dtype=torch.bfloat16, gen=g,
                       device="cpu", ranks=[8, 2, 5])
    assert torch.isnan(p.a_t[1, :, 2:].float()).all() and torch.isfinite(p.a_t[1, :, :2].float()).all()
    assert torch.isnan(p.b[2, :, 5:].float()).all()
    assert torch.allclose(p.scale, torch.tensor([4.0, 16.0, 6.4]))


def test_seeded_determinism():
    a = W.bgmv_decode_q(M=4, d=64, r=4, num_slots=4)
    b = W.bgmv_decode_q(M=4, d=64, r=4, num_slots=4)
    assert torch.equal(a.ops[0].x, b.ops[0].x) and torch.equal(a.ops[0].pool.b, b.ops[0].pool.b)
