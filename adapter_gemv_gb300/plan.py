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

from . import MLORA_MAX_GROUP, Group, lora_set_programmatic_launch, make_pool


class StepPlan:
    def __init__(self, ops: Sequence, batch, status=None, programmatic: bool = True, prefetch_next: bool = False):
        """ops: objects with .pool .layer .x .y (as workloads.Op); batch: .M .seg_offsets .seg_slot.
        programmatic: launch every call but the first with programmatic dependent launch. Safe
        because the kernel before each of those calls is this library's previous call, which
        writes none of the inputs a call reads before its wait (metadata, pool). The first call
        keeps an ordinary dependency on whatever ran before the step.
        prefetch_next: each call carries the next call's problems as an L2 prefetch hint. Off by
        default: on a decode step the hint's extra traffic is issued while each call's own adapter
        rows are in flight and slows the step down (about 3% on the Llama-2-7B bs32 step)."""
        self.programmatic = programmatic
        self.handles = {}
        groups: List[List] = []
        for op in ops:
            g = groups[-1] if groups else None
            if (g and len(g) < MLORA_MAX_GROUP and g[0].layer == op.layer
                    and g[0].x.data_ptr() == op.x.data_ptr() and g[0].pool.dtype == op.pool.dtype):
                g.append(op)
            else:
                groups.append([op])
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
            self.calls.append(Group(probs, batch.seg_offsets, batch.seg_slot, batch.M, status))
        if prefetch_next:
            for a, b in zip(self.calls, self.calls[1:]):
                a.set_next(b)  # each call prefetches the next call's adapter rows into L2
        self.groups = groups

    def __call__(self, stream=None):
        prev = lora_set_programmatic_launch(False)
        try:
            for q, c in enumerate(self.calls):
                if q == 1:
                    lora_set_programmatic_launch(self.programmatic)
                c(stream)
        finally:
            lora_set_programmatic_launch(prev)

    @property
    def launches(self) -> int:
        return len(self.calls)
