"""Stored cases (tests/golden/oracle_cases.json, written by make_golden.py from
the oracle alone) reproduced by the oracle on this machine, and by the C
planner where the case is a planning result.  A failure here means the oracle's
arithmetic (or the platform's) changed since the fixture was written."""
import json
import math
import os

import numpy as np
import pytest

from oracle import flexicache as fx
from oracle import tangram as tg

CASES = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "oracle_cases.json")))


def f32(bits):
    return np.array(bits, dtype=np.uint32).view(np.float32)


def test_every_case_cites_its_passage():
    for name, case in CASES.items():
        assert "paper-review page" in case["cite"], name


def test_retained_count():
    for c in CASES["retained_count"]["cases"]:
        assert tg.retained_count(f32(c["B_f32_bits"]), c["N"]) == c["n"]


def test_effective_budget():
    c = CASES["effective_budget"]
    got = tg.effective_budget(f32(c["Bhat_f32_bits"]), c["alpha"])
    assert np.array_equal(got.view(np.uint32), np.array(c["B_f32_bits"], np.uint32))


def test_top_indices():
    for c in CASES["top_indices"]["cases"]:
        assert tg.top_indices(f32(c["s_f32_bits"]), c["n"]).tolist() == c["idx"]


def test_split_map(lib):
    for c in CASES["split_map"]["cases"]:
        assert tg.split_map_row(c["Phi"], c["N_CTA"]) == c["S"]
        assert lib.tg_split_map([c["Phi"]], c["N_CTA"])[0].tolist() == c["S"]


@pytest.mark.parametrize("key", ["build_pages_cluster0", "build_pages_cluster1"])
def test_build_pages_and_work_list(lib, key):
    c = CASES[key]
    Bh = f32(c["Bhat_f32_bits"]).reshape(c["L"], c["H"])
    N = np.array(c["N"], np.int32)
    for impl in ("oracle", "c"):
        if impl == "oracle":
            pg = tg.build_pages(c["L"], c["batch"], c["H"], c["H_p"], c["P"], c["alpha"], Bh, N, c["cluster"])
        else:
            pg = lib.tg_build_pages(c["L"], c["batch"], c["H"], c["H_p"], c["P"], c["alpha"], Bh, N, c["cluster"])
        for k in ("order", "ntok", "pt_off", "pt_ids", "Phi"):
            assert np.asarray(pg[k]).tolist() == c[k], (impl, k)
        assert pg["n_pages"] == c["n_pages"] and pg["n_pages_monolithic"] == c["n_pages_monolithic"]
    S = tg.split_map(np.array(c["Phi"]), c["N_CTA"])
    assert S.tolist() == c["S"]
    for l in range(c["L"]):
        assert tg.work_list(S[l], np.array(c["ntok"][l]), c["order"][l], c["H_p"]) == c["work_list"][l]


def test_attention():
    c = CASES["attention"]
    q, K, V = np.array(c["q"]), np.array(c["K"]), np.array(c["V"])
    out, lse = tg.attention(q, K, V, c["scale"])
    np.testing.assert_allclose(out, c["out"], rtol=0, atol=1e-15)
    assert abs(lse - c["lse"]) <= 1e-15
    parts = [tg.attention_partial(q, K[a:b], V[a:b], c["scale"]) for a, b in ((0, 4), (4, 5), (5, 11))]
    mo, ml = tg.merge_partials(parts)
    np.testing.assert_allclose(mo, c["merged_out"], rtol=0, atol=1e-15)
    assert abs(ml - c["merged_lse"]) <= 1e-15


def test_quest():
    c = CASES["quest"]
    K = f32(c["K_f32_bits"])
    mn, mx = fx.page_minmax(K, c["P"])
    assert np.array_equal(mn.view(np.uint32), np.array(c["mn_f32_bits"], np.uint32))
    assert np.array_equal(mx.view(np.uint32), np.array(c["mx_f32_bits"], np.uint32))
    sc = fx.page_scores(f32(c["q_f32_bits"]), mn, mx)
    assert np.array_equal(sc.view(np.uint32), np.array(c["score_f32_bits"], np.uint32))
    assert fx.top_pages(sc, 3).tolist() == c["top3"]
