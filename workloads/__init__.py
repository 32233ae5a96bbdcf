"""Seeded synthetic inputs for the gathered multi-LoRA workloads.

This module only draws random numbers and lays them out; it holds none of the arithmetic of
the shrink/expand (that lives in the CUDA library and, independently, in the oracle). Both
the GPU tests and the oracle are fed from here, and so is the bench.

Shapes and distributions follow the pages' workloads:
  * Llama-2 projection shapes per layer: q, k, v, o, gate, up, down ("7 LoRA add-ons per
    layer", zh-TW Punica digest 5.3; Llama-2-7B hidden 4096 / MLP 11008, 13B 5120 / 13824,
    70B q_proj 8192).
  * adapter-assignment distributions Distinct / Uniform / Skewed / Identical (Punica
    section 5, "four request distributions"); Skewed is a finite power law p_i ~ i^-alpha.
  * a paged, heterogeneous-rank pool (S-LoRA "Unified Paging": one page per rank-row of
    A^T and of B; ranks differ between adapters, no padding).
Readings where the pages are silent (variance vs std of N(0, s), base y, alpha) are
stated once in the design notes and applied here: N(0, s) means variance s; base y ~ U(-1, 1);
alpha = 32 unless a workload fixes the scale.

Everything is a torch tensor on the requested device; generation is deterministic for a
given seed and device.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclasses.dataclass(frozen=True)
class Projection:
    name: str
    d_in: int
    d_out: int


def llama_projections(hidden: int, mlp: int) -> List[Projection]:
    """The seven adapted projections of one Llama decoder layer."""
    return [Projection("q", hidden, hidden), Projection("k", hidden, hidden), Projection("v", hidden, hidden),
            Projection("o", hidden, hidden), Projection("gate", hidden, mlp), Projection("up", hidden, mlp),
            Projection("down", mlp, hidden)]


LLAMA2_7B = llama_projections(4096, 11008)
LLAMA2_13B = llama_projections(5120, 13824)


@dataclasses.dataclass
class Pool:
    """An adapter pool for one projection shape (d_in -> d_out), all layers, all slots.

    stacked: a_t [num_slots][num_layers][r_max][d_in] (rows of A^T = columns of A) and
             b   [num_slots][num_layers][r_max][d_out] (rows of B).
    paged:   pages [num_pages][page_elems]; a_page_table / b_page_table
             [num_slots][num_layers][r_max][ceil(d / page_elems)] int32 page ids (-1 where
             j >= rank): a vector longer than a page spans several.
    rank int32 [num_slots], scale float32 [num_slots].
    """
    dtype: torch.dtype
    num_slots: int
    num_layers: int
    r_max: int
    d_in: int
    d_out: int
    rank: torch.Tensor
    scale: torch.Tensor
    a_t: Optional[torch.Tensor] = None
    b: Optional[torch.Tensor] = None
    pages: Optional[torch.Tensor] = None
    a_page_table: Optional[torch.Tensor] = None
    b_page_table: Optional[torch.Tensor] = None

    @property
    def paged(self) -> bool:
        return self.pages is not None

    def to(self, device) -> "Pool":
        f = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in dataclasses.asdict(self).items()}
        return Pool(**f)


@dataclasses.dataclass
class Batch:
    """Rows of one step: the slot per row plus, for SGMV, the segment form of the same rows."""
    M: int
    row_slot: torch.Tensor  # int32 [M], -1 = no adapter
    seg_offsets: Optional[torch.Tensor] = None  # int32 [n+1]
    seg_slot: Optional[torch.Tensor] = None  # int32 [n]

    def to(self, device) -> "Batch":
        mv = lambda t: None if t is None else t.to(device)
        return Batch(self.M, mv(self.row_slot), mv(self.seg_offsets), mv(self.seg_slot))


# --------------------------------------------------------------------------------------------
# random helpers


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, var: float, dtype, gen: torch.Generator, device) -> torch.Tensor:
    """N(0, var) drawn in fp32, rounded to `dtype` (round to nearest even by torch)."""
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    t.mul_(math.sqrt(var))
    return t.to(dtype)


def uniform(shape, lo: float, hi: float, dtype, gen: torch.Generator, device) -> torch.Tensor:
    t = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
    t.mul_(hi - lo).add_(lo)
    return t.to(dtype)


def fill_normal_(t: torch.Tensor, var: float, gen: torch.Generator, chunk: int = 1 << 26) -> torch.Tensor:
    """In-place N(0, var) fill of a big bf16/fp16 tensor, in chunks to bound the fp32 scratch."""
    flat = t.view(-1)
    for s in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - s)
        flat[s:s + n] = normal((n,), var, t.dtype, gen, t.device)
    return t


NAN_BITS = {torch.bfloat16: 0x7FC1, torch.float16: 0x7E01}  # quiet NaNs with a payload


def poison_(t: torch.Tensor) -> torch.Tensor:
    """Fill with a NaN payload: any read of these elements poisons the result visibly."""
    t.view(torch.int16).fill_(NAN_BITS[t.dtype])
    return t


# --------------------------------------------------------------------------------------------
# adapter-assignment distributions (Punica section 5)


def zipf_probs(n: int, alpha: float) -> np.ndarray:
    w = np.arange(1, n + 1, dtype=np.float64) ** (-alpha)
    return w / w.sum()


def draw_slots(dist: str, M: int, num_slots: int, rng: np.random.Generator, *, uniform_adapters: int = 8,
               zipf_alpha: float = 1.5) -> np.ndarray:
    """Slot per row for one step. Slot ids double as popularity ranks for the Zipf draw."""
    if dist == "distinct":
        if M > num_slots:
            raise ValueError("distinct needs a slot per row")
        return np.arange(M, dtype=np.int32)
    if dist == "uniform":
        k = uniform_adapters
        if M % k:
            raise ValueError("uniform needs M divisible by the adapter count")
        chosen = rng.choice(num_slots, size=k, replace=False)
        slots = np.repeat(chosen, M // k)
        rng.shuffle(slots)
        return slots.astype(np.int32)
    if dist == "skewed":
        return rng.choice(num_slots, size=M, p=zipf_probs(num_slots, zipf_alpha)).astype(np.int32)
    if dist == "identical":
        return np.zeros(M, dtype=np.int32)
    raise ValueError(dist)


def segments_of(sorted_slots: Sequence[int]):
    """Runs of equal slots in an already grouped slot vector -> (offsets [n+1], seg_slot [n])."""
    s = np.asarray(sorted_slots, dtype=np.int64)
    if s.size == 0:
        return np.zeros(1, np.int32), np.zeros(0, np.int32)
    starts = np.flatnonzero(np.r_[True, s[1:] != s[:-1]])
    offsets = np.r_[starts, s.size].astype(np.int32)
    return offsets, s[starts].astype(np.int32)


def group_rows(row_slot: np.ndarray):
    """Stable grouping of rows by slot (the batch-layout step: rows sharing an adapter become
    one contiguous segment). Returns (perm, offsets, seg_slot): row perm[q] goes to position q."""
    rs = np.asarray(row_slot)
    perm = np.argsort(rs, kind="stable").astype(np.int64)
    offsets, seg_slot = segments_of(rs[perm])
    return perm, offsets, seg_slot


def batch_from_slots(row_slot: np.ndarray, *, sgmv: bool) -> Batch:
    """A Batch whose rows are already grouped when `sgmv` is set (caller permuted the rows)."""
    rs = np.asarray(row_slot, dtype=np.int32)
    if sgmv:
        offsets, seg_slot = segments_of(rs)
        return Batch(int(rs.size), torch.from_numpy(rs.copy()), torch.from_numpy(offsets), torch.from_numpy(seg_slot))
    return Batch(int(rs.size), torch.from_numpy(rs.copy()))


def batch_from_segments(lengths: Sequence[int], slots: Sequence[int]) -> Batch:
    lengths = np.asarray(lengths, dtype=np.int64)
    offsets = np.r_[0, np.cumsum(lengths)].astype(np.int32)
    seg_slot = np.asarray(slots, dtype=np.int32)
    row_slot = np.repeat(seg_slot, lengths).astype(np.int32)
    return Batch(int(offsets[-1]), torch.from_numpy(row_slot), torch.from_numpy(offsets), torch.from_numpy(seg_slot))


# --------------------------------------------------------------------------------------------
# pools


def stacked_pool(*, num_slots, num_layers, r_max, d_in, d_out, dtype, gen, device, ranks=None, scales=None,
                 alpha: float = 32.0, a_var: Optional[float] = None, b_var: float = 0.02,
                 poison_padding: bool = True) -> Pool:
    """Stacked pool; A ~ N(0, 1/d_in) unless a_var is given, B ~ N(0, b_var); scale = alpha/rank.
    Rows j >= rank[s] of a slot are padding and hold NaNs when `poison_padding`."""
    ranks = np.full(num_slots, r_max, np.int32) if ranks is None else np.asarray(ranks, np.int32)
    if scales is None:
        scales = (alpha / ranks.astype(np.float64)).astype(np.float32)
    a_var = 1.0 / d_in if a_var is None else a_var
    a_t = torch.empty((num_slots, num_layers, r_max, d_in), dtype=dtype, device=device)
    b = torch.empty((num_slots, num_layers, r_max, d_out), dtype=dtype, device=device)
    fill_normal_(a_t, a_var, gen)
    fill_normal_(b, b_var, gen)
    if poison_padding:
        for s in range(num_slots):
            if ranks[s] < r_max:
                poison_(a_t[s, :, ranks[s]:])
                poison_(b[s, :, ranks[s]:])
    return Pool(dtype, num_slots, num_layers, r_max, d_in, d_out,
                torch.from_numpy(ranks).to(device), torch.from_numpy(np.asarray(scales, np.float32)).to(device),
                a_t=a_t, b=b)


def paged_pool(*, num_slots, num_layers, r_max, d_in, d_out, dtype, gen, device, rng: np.random.Generator,
               ranks, page_elems: Optional[int] = None, free_fraction: float = 0.10, alpha: float = 32.0,
               a_var: Optional[float] = None, b_var: float = 0.02) -> Pool:
    """S-LoRA-style paged pool: every rank-row of A^T and of B is stored in pages of `page_elems`
    elements at random physical positions; about `free_fraction` of the pages are free and hold
    NaNs, interleaved with the used ones. A vector longer than a page (page_elems < d) spans
    ceil(d / page_elems) pages, each placed on its own; page tables are
    [num_slots][num_layers][r_max][ceil(d / page_elems)] (-1 where j >= rank). Elements of a page
    past the vector's end are NaN."""
    ranks = np.asarray(ranks, np.int32)
    page_elems = max(d_in, d_out) if page_elems is None else page_elems
    a_ppv, b_ppv = -(-d_in // page_elems), -(-d_out // page_elems)
    used = int(num_layers * ranks.sum() * (a_ppv + b_ppv))
    num_pages = int(math.ceil(used * (1.0 + free_fraction)))
    phys = rng.permutation(num_pages)[:used].astype(np.int32)
    a_tab = np.full((num_slots, num_layers, r_max, a_ppv), -1, np.int32)
    b_tab = np.full((num_slots, num_layers, r_max, b_ppv), -1, np.int32)
    q = 0
    for s in range(num_slots):
        r = int(ranks[s])
        for layer in range(num_layers):
            a_tab[s, layer, :r] = phys[q:q + r * a_ppv].reshape(r, a_ppv)
            q += r * a_ppv
            b_tab[s, layer, :r] = phys[q:q + r * b_ppv].reshape(r, b_ppv)
            q += r * b_ppv
    pages = torch.empty((num_pages, page_elems), dtype=dtype, device=device)
    poison_(pages)
    a_var = 1.0 / d_in if a_var is None else a_var
    for tab, d, var in ((a_tab, d_in, a_var), (b_tab, d_out, b_var)):
        vecs = tab[tab[..., 0] >= 0]  # [vectors][ppv] page ids, in table order
        chunk = max(1, (1 << 26) // d)
        for s0 in range(0, vecs.shape[0], chunk):
            sel = vecs[s0:s0 + chunk]
            vals = normal((sel.shape[0], d), var, dtype, gen, device)
            for q in range(sel.shape[1]):  # piece q of every vector goes to its own page
                lo, hi = q * page_elems, min(d, (q + 1) * page_elems)
                pages[torch.from_numpy(sel[:, q].astype(np.int64)).to(device), :hi - lo] = vals[:, lo:hi]
    scales = (alpha / ranks.astype(np.float64)).astype(np.float32)
    return Pool(dtype, num_slots, num_layers, r_max, d_in, d_out,
                torch.from_numpy(ranks).to(device), torch.from_numpy(scales).to(device),
                pages=pages, a_page_table=torch.from_numpy(a_tab).to(device),
                b_page_table=torch.from_numpy(b_tab).to(device))


# --------------------------------------------------------------------------------------------
# the five workloads


@dataclasses.dataclass
class Op:
    """One adapted projection of one layer: y[M][d_out] += delta(x[M][d_in])."""
    name: str
    pool: Pool
    layer: int
    x: torch.Tensor
    y: torch.Tensor


@dataclasses.dataclass
class Workload:
    name: str
    dtype: torch.dtype
    batch: Batch
    ops: List[Op]
    form: str  # "sgmv" or "bgmv"
    pools: List[Pool]
    note: str = ""


def tiny_sgmv(device="cpu", seed=1) -> Workload:
    """fp16, d_in = d_out = 256, r = 8, 4 adapters, segments [3, 5, 1, 7] on slots 0..3,
    x ~ U(-1,1), A ~ N(0, 1/256), B ~ N(0, 0.02), y ~ U(-1,1), scale = 16/r."""
    g = generator(seed, device)
    dt = torch.float16
    pool = stacked_pool(num_slots=4, num_layers=1, r_max=8, d_in=256, d_out=256, dtype=dt, gen=g, device=device,
                        scales=np.full(4, 16.0 / 8, np.float32), a_var=1.0 / 256)
    batch = batch_from_segments([3, 5, 1, 7], [0, 1, 2, 3]).to(device)
    x = uniform((16, 256), -1, 1, dt, g, device)
    y = uniform((16, 256), -1, 1, dt, g, device)
    return Workload("tiny_sgmv_fp16_d256_r8", dt, batch, [Op("proj", pool, 0, x, y)], "sgmv", [pool])


def bgmv_decode_q(device="cpu", seed=2, M=32, d=4096, r=16, num_slots=32) -> Workload:
    """bf16 Llama-2-7B q_proj shape, 32 resident slots, row i -> slot i (Distinct),
    x ~ N(0,1), A ~ N(0, 1/4096), B ~ N(0, 0.02), alpha = 32, y ~ U(-1,1)."""
    g = generator(seed, device)
    dt = torch.bfloat16
    pool = stacked_pool(num_slots=num_slots, num_layers=1, r_max=r, d_in=d, d_out=d, dtype=dt, gen=g, device=device)
    batch = batch_from_slots(np.arange(M, dtype=np.int32) % num_slots, sgmv=False).to(device)
    x = normal((M, d), 1.0, dt, g, device)
    y = uniform((M, d), -1, 1, dt, g, device)
    return Workload(f"bgmv_decode_q_proj_d{d}_r{r}_bs{M}_distinct", dt, batch, [Op("q", pool, 0, x, y)], "bgmv", [pool])


def sgmv_decode_7b(device="cpu", seed=3, dist="distinct", M=32, num_layers=32, r=16, num_slots=32,
                   projections: Sequence[Projection] = LLAMA2_7B, layers: Optional[Sequence[int]] = None) -> Workload:
    """bf16 decode step: all seven Llama-2-7B projections of every layer, r = 16, 32 slots,
    one stacked pool per projection [32 slots][32 layers][16][d]. Slots per row from `dist`;
    rows grouped into segments (the batch layout), reused by every op of the step. Every layer
    has its own activations, as in a real step: q/k/v/gate/up of a layer read one x [M][4096]
    (the normalised hidden state), o reads its own [M][4096], down reads [M][11008]."""
    g = generator(seed, device)
    rng = np.random.default_rng(seed)
    dt = torch.bfloat16
    slots = draw_slots(dist, M, num_slots, rng)
    _, offsets, seg_slot = group_rows(slots)
    batch = Batch(M, torch.from_numpy(np.sort(slots, kind="stable").astype(np.int32)),
                  torch.from_numpy(offsets), torch.from_numpy(seg_slot)).to(device)
    pools = {p.name: stacked_pool(num_slots=num_slots, num_layers=num_layers, r_max=r, d_in=p.d_in, d_out=p.d_out,
                                  dtype=dt, gen=g, device=device) for p in projections}
    hidden = projections[0].d_in
    ops = []
    for layer in (range(num_layers) if layers is None else layers):
        x_shared = normal((M, hidden), 1.0, dt, g, device)
        x_o = normal((M, hidden), 1.0, dt, g, device)
        x_down = {p.name: normal((M, p.d_in), 1.0, dt, g, device) for p in projections if p.name == "down"}
        for p in projections:
            x = x_o if p.name == "o" else x_down[p.name] if p.name == "down" else x_shared
            y = uniform((M, p.d_out), -1, 1, dt, g, device)
            ops.append(Op(p.name, pools[p.name], layer, x, y))
    return Workload(f"sgmv_decode_llama2_7b_bs{M}_r{r}_{dist}", dt, batch, ops, "sgmv", list(pools.values()))


def sgmv_prefill_13b(device="cpu", seed=4, r=64, num_requests=8, min_len=128, max_len=2048,
                     projections: Sequence[Projection] = LLAMA2_13B, lengths: Optional[Sequence[int]] = None) -> Workload:
    """bf16 prefill: 8 prompts with lengths ~ U[128, 2048] (integers, inclusive), one segment
    and one adapter per prompt, r = 64, all seven Llama-2-13B projections of one layer,
    x ~ N(0,1), A ~ N(0, 1/d_in), B ~ N(0, 0.02), scale = 32/64."""
    g = generator(seed, device)
    rng = np.random.default_rng(seed)
    dt = torch.bfloat16
    if lengths is None:
        lengths = rng.integers(min_len, max_len + 1, num_requests)
    batch = batch_from_segments(lengths, np.arange(len(lengths))).to(device)
    M = batch.M
    pools = {p.name: stacked_pool(num_slots=len(lengths), num_layers=1, r_max=r, d_in=p.d_in, d_out=p.d_out,
                                  dtype=dt, gen=g, device=device) for p in projections}
    hidden = projections[0].d_in
    x_shared = normal((M, hidden), 1.0, dt, g, device)
    x_o = normal((M, hidden), 1.0, dt, g, device)
    ops = []
    for p in projections:
        x = x_o if p.name == "o" else normal((M, p.d_in), 1.0, dt, g, device) if p.name == "down" else x_shared
        y = uniform((M, p.d_out), -1, 1, dt, g, device)
        ops.append(Op(p.name, pools[p.name], 0, x, y))
    return Workload(f"sgmv_prefill_llama2_13b_r{r}_M{M}", dt, batch, ops, "sgmv", list(pools.values()))


def paged_decode_70b(device="cpu", seed=5, M=256, num_adapters=2000, d=8192, rank_choices=(8, 16, 32, 64),
                     zipf_alpha=1.2) -> Workload:
    """bf16 S-LoRA-style decode: 2000 adapters with ranks uniform over {8,16,32,64} in a paged
    pool of d-element pages at permuted physical positions (~10% free pages interleaved),
    Llama-2-70B q_proj 8192 -> 8192, one layer, 256 rows with adapters drawn Zipf(1.2) over
    the 2000, BGMV form (unsorted), scale = 32/rank."""
    g = generator(seed, device)
    rng = np.random.default_rng(seed)
    dt = torch.bfloat16
    ranks = rng.choice(np.asarray(rank_choices, np.int32), size=num_adapters)
    pool = paged_pool(num_slots=num_adapters, num_layers=1, r_max=max(rank_choices), d_in=d, d_out=d, dtype=dt,
                      gen=g, device=device, rng=rng, ranks=ranks)
    slots = rng.choice(num_adapters, size=M, p=zipf_probs(num_adapters, zipf_alpha)).astype(np.int32)
    batch = batch_from_slots(slots, sgmv=False).to(device)
    x = normal((M, d), 1.0, dt, g, device)
    y = uniform((M, d), -1, 1, dt, g, device)
    return Workload(f"paged_bgmv_llama2_70b_q_proj_bs{M}_{num_adapters}_adapters", dt, batch,
                    [Op("q", pool, 0, x, y)], "bgmv", [pool])


def mixed_prefill_decode_13b(device="cpu", seed=6, r=64, prompts=(300, 1200, 2000), decode_rows=64,
                             projections: Sequence[Projection] = LLAMA2_13B) -> Workload:
    """bf16 mixed batch in Punica's batch layout (section 3.4, "Batch Layout Construction"): the
    prompts of new requests first, one segment and adapter each, then `decode_rows` one-row decode
    segments, each request on its own adapter; Llama-2-13B shapes, all seven projections of one
    layer, r = 64, scale 32/64. The prompts are long segments (the tensor-core kernels), the decode
    rows short ones (the CUDA-core kernel), in one SGMV call per projection."""
    g = generator(seed, device)
    dt = torch.bfloat16
    n_adapters = len(prompts) + decode_rows
    lens = np.r_[np.asarray(prompts, np.int64), np.ones(decode_rows, np.int64)]
    batch = batch_from_segments(lens, np.arange(n_adapters)).to(device)
    M = batch.M
    pools = {p.name: stacked_pool(num_slots=n_adapters, num_layers=1, r_max=r, d_in=p.d_in, d_out=p.d_out,
                                  dtype=dt, gen=g, device=device) for p in projections}
    hidden = projections[0].d_in
    x_shared = normal((M, hidden), 1.0, dt, g, device)
    x_o = normal((M, hidden), 1.0, dt, g, device)
    ops = []
    for p in projections:
        x = x_o if p.name == "o" else normal((M, p.d_in), 1.0, dt, g, device) if p.name == "down" else x_shared
        ops.append(Op(p.name, pools[p.name], 0, x, uniform((M, p.d_out), -1, 1, dt, g, device)))
    return Workload(f"mixed_prefill_decode_llama2_13b_r{r}_M{M}", dt, batch, ops, "sgmv", list(pools.values()))
