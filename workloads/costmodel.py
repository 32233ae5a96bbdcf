"""Algorithmic bytes and flops of the gathered multi-LoRA delta -- measurement only.

These are the denominators of every roofline number the bench reports: what the method must
move and compute, not what a kernel happens to move.

Sources:
  * "Multi-LoRA Serving, in depth", section "Worked example": a LoRA pair costs
    r * (d_in + d_out) parameters; section "The decode cost model": a good kernel reads each
    adapter once per step, so the extra bytes of a step are (#distinct adapters) x adapter bytes.
  * S-LoRA digest, section 3 "Technical Approach": x·A·B costs 2·B·r·(h + d) flops.
  * Punica, section 3.4 "Roofline analysis grounding" (Figure 7): the intensity of SGMV is
    s_n·h_i·h_o·2 / ((s_n·(h_i + h_o) + n·h_i·h_o)·2); zh-TW Punica digest 6.2: Gather-BMM moves
    s_n·h_i·h_o·2 more elements than SGMV.
"""
from __future__ import annotations

from typing import Iterable, Sequence


def adapter_params(r: int, d_in: int, d_out: int) -> int:
    """Parameters of one LoRA pair A (d_in x r), B (r x d_out)."""
    return r * (d_in + d_out)


def model_adapter_params(r: int, projections: Iterable, num_layers: int) -> int:
    """Parameters of an adapter over the given projections of every layer."""
    return num_layers * sum(adapter_params(r, p.d_in, p.d_out) for p in projections)


def lora_flops(rows: int, r: int, d_in: int, d_out: int) -> int:
    """Shrink + expand flops for `rows` rows at rank r (multiply-add counted as 2)."""
    return 2 * rows * r * (d_in + d_out)


def sgmv_intensity(s_n: int, n: int, h_i: int, h_o: int) -> float:
    """Punica's SGMV roofline intensity (flop per byte) for one SGMV of h_i -> h_o over s_n
    inputs in n segments with 16-bit elements."""
    return (s_n * h_i * h_o * 2) / ((s_n * (h_i + h_o) + n * h_i * h_o) * 2)


def gather_bmm_extra_elements(s_n: int, h_i: int, h_o: int) -> int:
    """Elements Gather-BMM moves beyond SGMV (write then re-read of the gathered stack)."""
    return s_n * h_i * h_o * 2


def decode_extra_bytes(distinct_adapters: int, adapter_bytes: float) -> float:
    """Adapter bytes one decode step reads when each distinct adapter is read once."""
    return distinct_adapters * adapter_bytes


def op_bytes(*, d_in: int, d_out: int, row_ranks: Sequence[int], distinct_ranks: Sequence[int], elem: int = 2,
             v_roundtrip: bool) -> int:
    """Algorithmic bytes of one adapted projection.

    row_ranks      rank of the adapter of every row that has one (rows with slot -1 move nothing)
    distinct_ranks rank of every distinct adapter used (each is read once: d_in + d_out per rank-row)
    v_roundtrip    True for the two-launch form (fp32 v written by the shrink, read by the expand)

    x is read once per adapted row, y is read and written once per adapted row.
    """
    rows = len(row_ranks)
    b = elem * rows * d_in  # x
    b += elem * sum(distinct_ranks) * (d_in + d_out)  # A and B of each distinct adapter, once
    b += 2 * elem * rows * d_out  # y read + write
    if v_roundtrip:
        b += 2 * 4 * sum(row_ranks)  # v fp32 write + read
    return int(b)


def op_flops(*, d_in: int, d_out: int, row_ranks: Sequence[int]) -> int:
    return int(2 * sum(row_ranks) * (d_in + d_out))
