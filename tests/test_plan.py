"""The step plan's grouping rule (host logic, CPU): consecutive ops of one layer that read the same
x and whose pools share a dtype go into one grouped call, at most MLORA_MAX_GROUP of them; the
Llama decode step becomes q,k,v / o / gate,up / down per layer (Punica section 3.4, "Batch
Layout Construction": one batch layout reused by every projection of every layer)."""
from types import SimpleNamespace

import torch

import workloads as W
from adapter_gemv_gb300 import MLORA_MAX_GROUP
from adapter_gemv_gb300.plan import group_ops

SMALL = [W.Projection("q", 64, 64), W.Projection("k", 64, 64), W.Projection("v", 64, 64),
         W.Projection("o", 64, 64), W.Projection("gate", 64, 96), W.Projection("up", 64, 96),
         W.Projection("down", 96, 64)]


def test_decode_step_groups():
    w = W.sgmv_decode_7b(device="cpu", num_layers=3, M=8, num_slots=8, projections=SMALL)
    groups = group_ops(w.ops)
    names = [[op.name for op in g] for g in groups]
    assert names == [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]] * 3
    assert [g[0].layer for g in groups] == [l for l in range(3) for _ in range(4)]
    # every op exactly once, in step order
    assert [op for g in groups for op in g] == list(w.ops)


def _op(x, layer=0, dtype=torch.bfloat16):
    return SimpleNamespace(x=x, layer=layer, pool=SimpleNamespace(dtype=dtype))


def test_group_breaks():
    xa, xb = torch.zeros(4, 8), torch.zeros(4, 8)
    ops = [_op(xa), _op(xa), _op(xb), _op(xa), _op(xa, layer=1), _op(xa, layer=1, dtype=torch.float16)]
    sizes = [len(g) for g in group_ops(ops)]
    assert sizes == [2, 1, 1, 1, 1]  # another x, the same x again later, another layer, another dtype


def test_group_size_limit():
    x = torch.zeros(4, 8)
    ops = [_op(x) for _ in range(2 * MLORA_MAX_GROUP + 3)]
    assert [len(g) for g in group_ops(ops)] == [MLORA_MAX_GROUP, MLORA_MAX_GROUP, 3]


def test_views_of_one_storage_group():
    base = torch.zeros(4, 8)
    ops = [_op(base), _op(base.view(4, 8)), _op(base[1:])]
    # the first two start at the same address; a view at an offset reads other data
    assert [len(g) for g in group_ops(ops)] == [2, 1]
