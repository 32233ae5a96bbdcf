"""The byte/flop model against the pages' worked numbers (tests/golden/byte_model.json)."""
import json
import os

import pytest

from workloads import Projection, costmodel as C

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "byte_model.json")))


def llama3_8b_projections():
    g = GOLD["mls_worked_example"]["llama3_8b"]
    h, kv = g["hidden"], g["kv_heads"] * g["head_dim"]
    return {"q": Projection("q", h, h), "k": Projection("k", h, kv), "v": Projection("v", h, kv),
            "o": Projection("o", h, h), "gate": Projection("gate", h, g["mlp"]),
            "up": Projection("up", h, g["mlp"]), "down": Projection("down", g["mlp"], h)}


def test_mls_worked_example():
    g = GOLD["mls_worked_example"]
    P = llama3_8b_projections()
    L, r = g["llama3_8b"]["layers"], g["rank"]
    all7 = C.model_adapter_params(r, P.values(), L)
    assert round(all7 / 1e6, 1) == GOLD["mls_decode_cost_model"]["adapter_params_approx_M"]
    assert round(2 * all7 / 1e6, 1) == GOLD["mls_decode_cost_model"]["adapter_bytes"] / 1e6
    qv = C.model_adapter_params(r, [P["q"], P["v"]], L)
    assert qv == g["q_v_only_params"]
    assert round(2 * qv / 1e6) == g["q_v_only_bytes_approx_MB"]
    assert round(2 * C.model_adapter_params(64, P.values(), L) / 1e6) == g["rank64_all_projections_bytes_approx_MB"]
    assert round(16 * 2 * all7 / 1e9, 1) == g["sixteen_rank16_adapters_approx_GB"]
    assert round(16 * 2 * C.model_adapter_params(64, P.values(), L) / 1e9, 1) == g["sixteen_rank64_adapters_approx_GB"]


@pytest.mark.parametrize("row", GOLD["mls_decode_cost_model"]["rows"])
def test_mls_decode_cost_table(row):
    g = GOLD["mls_decode_cost_model"]
    distinct, gb, pct = row
    extra = C.decode_extra_bytes(distinct, g["adapter_bytes"])
    assert f"{extra / 1e9:5.2f}".strip() == f"{gb:.2f}"
    assert f"{100 * extra / g['base_bytes']:5.1f}".strip() == f"{pct:.1f}"


def test_slora_numbers():
    g = GOLD["slora_adapter_size"]
    p = Projection("attn", g["hidden"], g["hidden"])
    params = C.model_adapter_params(g["rank"], [p] * g["projections"], g["layers"])
    assert params == 16_777_216
    assert round(params / 1e6, 1) == g["params_approx_M"] and round(2 * params / 1e6, 1) == g["bytes_approx_MB"]
    u = GOLD["slora_unified_paging"]
    assert 4096 * 2 == u["page_bytes"]
    per_adapter = g["layers"] * g["projections"] * 2 * g["rank"]
    assert per_adapter == u["pages_per_adapter"] and 10 * per_adapter == u["pages_for_10_adapters"]
    f = GOLD["slora_flops"]
    assert C.lora_flops(32, 16, 4096, 4096) == f["adapter_flops_formula"]
    assert round(2 * 32 * 4096 * 4096 / 1e9, 2) == f["base_flops_approx_billion"]


def test_punica_intensity_regimes():
    # Distinct (n = s_n): intensity does not depend on the batch; Identical (n = 1): it grows
    d = [C.sgmv_intensity(s, s, 16, 4096) for s in (1, 2, 8, 64)]
    assert max(d) - min(d) < 1e-12
    i = [C.sgmv_intensity(s, 1, 16, 4096) for s in (1, 2, 8, 64)]
    assert all(b > a for a, b in zip(i, i[1:]))
    assert C.sgmv_intensity(64, 1, 16, 4096) == pytest.approx(64 * 16 * 4096 / (64 * 4112 + 16 * 4096))
    assert C.gather_bmm_extra_elements(64, 16, 4096) == 64 * 16 * 4096 * 2


def test_op_bytes_decode_q_proj():
    # 32 distinct rank-16 adapters on a 4096 -> 4096 projection, two launches
    b = C.op_bytes(d_in=4096, d_out=4096, row_ranks=[16] * 32, distinct_ranks=[16] * 32, v_roundtrip=True)
    assert b == 2 * 32 * 4096 + 2 * 32 * 16 * 8192 + 4 * 32 * 4096 + 8 * 32 * 16 == 9_179_136
    # one adapter shared by all rows: its weights count once
    b1 = C.op_bytes(d_in=4096, d_out=4096, row_ranks=[16] * 32, distinct_ranks=[16], v_roundtrip=False)
    assert b1 == 2 * 32 * 4096 + 2 * 16 * 8192 + 4 * 32 * 4096
