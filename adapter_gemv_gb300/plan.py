"""Step plans: the adapted projections of a decoder step issued as grouped calls.

Punica builds the batch's segment indices once and reuses them for all 7 projections of every
layer (section 3.4, "Batch Layout Construction"). A plan does the host side of that: it walks
the ops of a step in order, puts consecutive ops of the same layer that read the same x into one
``lora_sgmv_grouped`` call (q, k, v; gate, up), and prepares every call once, so replaying the
step is a loop of C calls (or a CUDA-graph replay of them).
"""
from __future__ import annotations

from typing import List, Sequence

import torch

from . import MLORA_MAX_GROUP, CallSequence, Group, make_pool


def group_ops(ops: Sequence) -> List[List]:
    """Consecutive ops of one layer that read the same x (same storage) and whose pools share a
    dtype, at most MLORA_MAX_GROUP at a time, in step order: the problems of one grouped call."""
    groups: List[List] = []
    for op in ops:
        g = groups[-1] if groups else None
        if (g and len(g) < MLORA_MAX_GROUP and g[0].layer == op.layer
                and g[0].x.data_ptr() == op.x.data_ptr() and g[0].pool.dtype == op.pool.dtype):
            g.append(op)
        else:
            groups.append([op])
    return groups


class StepPlan:
    def __init__(self, ops: Sequence, batch, status=None, programmatic: bool = True):
        """ops: objects with .pool .layer .x .y (as workloads.Op); batch: .M .seg_offsets .seg_slot.
        programmatic: launch every call but the first with programmatic dependent launch (a flag
        of that call alone). Safe because the kernel before each of those calls is this library's
        previous call, which writes none of the inputs a call reads before its wait (metadata,
        pool). The first call keeps an ordinary dependency on whatever ran before the step."""
        self.programmatic = programmatic
        self.handles = {}
        groups = group_ops(ops)
        dev = ops[0].x.device
        r_max = max(op.pool.r_max for op in ops)
        width = max(len(g) for g in groups)
        # one scratch per position in a group (problems of one launch never share scratch)
        self.scratch = [torch.empty((batch.M, r_max), dtype=torch.float32, device=dev) for _ in range(width)]
        self.calls = []
        for g in groups:
            probs = []
            for q, op in enumerate(g):
                h = self.handles.setdefault(id(op.pool), make_pool(op.pool))
                v = self.scratch[q].view(-1)[:batch.M * op.pool.r_max].view(batch.M, op.pool.r_max)  # row stride r_max
                probs.append((op.y, op.x, h, op.layer, v))
            self.calls.append(Group(probs, batch.seg_offsets, batch.seg_slot, batch.M, status,
                                    programmatic=programmatic and len(self.calls) > 0))
        self.groups = groups
        # the whole step as one call into the library (the same launches as the calls above)
        self.sequence = CallSequence(self.calls, programmatic, status)

    def __call__(self, stream=None):
        """Issue the step: one lora_sgmv_sequence call (every grouped call, launched natively)."""
        self.sequence(stream)

    def call_one_by_one(self, stream=None):
        """Issue the step as one lora_sgmv_grouped_ex call per group (the same launches)."""
        for c in self.calls:
            c(stream)

    @property
    def launches(self) -> int:
        return len(self.calls)
