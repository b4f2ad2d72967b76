"""Pins for the memory arithmetic against the numbers the pages print
(tests/golden/utilisation.json, each entry citing its page and section)."""
import json
import math
import os

import pytest

from oracle import utilisation as U

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "utilisation.json")))
KB, MB, GB = 1024, 1024 ** 2, 1024 ** 3   # the worked example uses binary units


def test_contiguous_utilisation():
    for c in G["contiguous_utilisation"]["cases"]:
        assert U.u_contig(c["L"], c["L_max"]) == c["U"]
        assert round(100 * (1 - U.u_contig(c["L"], c["L_max"]))) == c["wasted_percent"]


def test_paged_waste_bounds():
    p = G["paged_waste"]
    B = p["B"]
    assert U.paged_worst_waste(B) == p["worst_case_tokens"]
    assert max(U.paged_waste_tokens(L, B) for L in range(1, 10 * B)) == p["worst_case_tokens"]
    assert U.paged_mean_waste(B) == p["mean_tokens"]
    assert 100 * U.paged_worst_waste(B) / p["L_for_ceiling"] < p["ceiling_below_percent"]
    # utilisation closed form: full blocks waste nothing, one extra token wastes B-1
    assert U.u_paged(4 * B, B) == 1.0
    assert U.u_paged(4 * B + 1, B) == (4 * B + 1) / (5 * B)


def test_per_token_bytes_opt13b():
    p = G["per_token_bytes"]
    # the page folds n_kv_heads x head_dim into the model width
    b = U.kv_bytes_per_token(p["n_layers"], 1, p["kv_width"], p["dtype_bytes"])
    assert b == p["kb_per_token"] * KB
    assert round(p["tokens"] * b / 1e9, 1) == pytest.approx(p["approx_gb"], abs=0.1)


def test_worked_example_concurrency():
    w = G["worked_example"]
    bpt = w["kb_per_token"] * KB
    free = w["free_gb"] * GB
    contig = U.contiguous_request_bytes(w["L_max"], bpt)
    assert contig == w["contiguous_mb_per_request"] * MB
    assert U.concurrency(free, contig) == w["contiguous_requests"]
    assert math.ceil(w["L"] / w["B"]) == w["paged_blocks_per_request"]
    assert U.paged_slots(w["L"], w["B"]) == w["paged_slots_per_request"]
    paged = U.paged_request_bytes(w["L"], w["B"], bpt)
    assert paged == w["paged_mb_per_request"] * MB
    assert U.concurrency(free, paged) == w["paged_requests"]
    assert round(w["paged_requests"] / w["contiguous_requests"]) == w["approx_ratio"]


def test_llama3_70b_slot_size():
    p = G["llama3_70b_slots"]
    b = U.kv_bytes_per_token(p["n_layers"], p["n_kv_heads"], p["head_dim"], p["dtype_bytes"])
    assert b == p["kib_per_slot"] * KB
    assert p["slots"] * b == p["mb_total"] * MB


def test_rdna4_swarm_budget():
    p = G["rdna4_swarm"]
    mb = p["mb_per_token"]          # this page uses decimal units
    r16 = p["reserve_16k"]
    per16 = U.contiguous_request_bytes(r16["tokens"], mb) / 1000
    assert per16 == pytest.approx(r16["gb_per_agent"])
    assert round(p["agents"] * per16, 1) == r16["gb_total"]
    assert U.concurrency(p["kv_budget_gb"], per16) == r16["admitted"]
    r8 = p["reserve_8k"]
    per8 = U.contiguous_request_bytes(r8["tokens"], mb) / 1000
    assert per8 == pytest.approx(r8["gb_per_agent"])
    assert round(p["agents"] * per8, 1) == r8["gb_total"]
    assert U.concurrency(p["kv_budget_gb"], per8) >= r8["admitted"]
    live = p["agents"] * r8["live_tokens_each"] * mb / 1000
    assert round(live, 1) == r8["live_gb"]
    waste = U.contiguous_waste_fraction(r8["live_tokens_each"], r8["tokens"])
    assert abs(100 * waste - r8["wasted_percent"]) < 0.6          # 62.5% printed as 63
    pg = p["paged_16"]
    mean_waste = U.paged_mean_waste(pg["B"]) / r8["live_tokens_each"]
    assert 100 * mean_waste < pg["wasted_below_percent"]
    assert round(p["kv_budget_gb"] * 1000 / mb / 1000) == pg["approx_aggregate_ktokens"]
