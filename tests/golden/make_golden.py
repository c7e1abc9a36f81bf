"""Write tests/golden/oracle_cases.json from the oracle alone.

The reference pages print formulas but no worked numbers, so the stored
expected values come from this script, which calls only oracle/ (and numpy
for seeded inputs, which are stored in the fixture too).  Regenerate with

    python tests/golden/make_golden.py

and review the diff: a changed value means the oracle's arithmetic changed.
"""
import json
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import flexicache as fx  # noqa: E402
from oracle import tangram as tg  # noqa: E402

TANGRAM = "Tangram: Unlocking Non-Uniform KV Cache Compression for Efficient Multi-turn LLM Serving (paper-review page)"
FLEXI = "FlexiCache: Leveraging Temporal Stability of Attention Heads for Efficient KV Cache Management (MLSys 2026) (paper-review page)"


def f32hex(x):
    return np.float32(x).view(np.uint32).item()


def main():
    r = np.random.default_rng(20261202)
    cases = {}
    # 3.1: n = ceil(B N) of the float32 budget
    rc = []
    for B in [0.3, 0.1, 1.0, 0.5, 1e-30, 0.7, 0.999999, 0.123456]:
        for N in [0, 1, 3, 1000, 4096, 32768, 100000]:
            Bf = np.float32(B)
            rc.append({"B_f32_bits": f32hex(Bf), "N": N, "n": tg.retained_count(Bf, N)})
    cases["retained_count"] = {"cite": f"{TANGRAM}, 3.1 Budget Reservation, Top(ceil(B N), s)", "cases": rc}
    # 3.1: effective budget with the safety coefficient
    Bhat = r.uniform(0.05, 0.9, size=6).astype(np.float32)
    cases["effective_budget"] = {"cite": f"{TANGRAM}, 3.1 Budget Reservation (safety coefficient alpha)",
                                 "alpha": 2.0, "Bhat_f32_bits": [f32hex(x) for x in Bhat],
                                 "B_f32_bits": [f32hex(x) for x in tg.effective_budget(Bhat, 2.0)]}
    # 3.1: Top with ties and signed zeros
    tk = []
    for s in ([0.0, -0.0, 1.0, 1.0, -1.0, 0.5, 0.5, 0.5], [2.0] * 6, list(r.standard_normal(20).astype(np.float32))):
        s = np.array(s, np.float32)
        for n in (0, 1, 3, len(s)):
            tk.append({"s_f32_bits": [f32hex(x) for x in s], "n": n, "idx": tg.top_indices(s, n).tolist()})
    cases["top_indices"] = {"cite": f"{TANGRAM}, 3.1 Budget Reservation (I = Top(n, s)); ties to the lower index",
                            "cases": tk}
    # 3.3: split map
    sm = []
    for Phi, n_cta in (([10, 30], 8), ([5, 5, 5], 7), ([0, 0], 4), ([1, 2, 3, 4], 10), ([7, 1, 7, 1], 148),
                       ([123456, 7, 99999], 152)):
        sm.append({"Phi": Phi, "N_CTA": n_cta, "S": tg.split_map_row(Phi, n_cta)})
    cases["split_map"] = {"cite": f"{TANGRAM}, 3.3 AOT Load Balancing (Algorithm 1, Workload Split Map)", "cases": sm}
    # 3.2 + 3.3: a small ragged build and its work list
    L, batch, H, H_p, P = 2, 3, 4, 2, 16
    Bh = r.uniform(0.05, 1.0, size=(L, H)).astype(np.float32)
    N = np.array([37, 0, 70], np.int32)
    for cluster in (False, True):
        pg = tg.build_pages(L, batch, H, H_p, P, 1.5, Bh, N, cluster)
        S = tg.split_map(pg["Phi"], 6)
        wl = [tg.work_list(S[l], pg["ntok"][l], pg["order"][l], H_p) for l in range(L)]
        cases[f"build_pages_cluster{int(cluster)}"] = {
            "cite": f"{TANGRAM}, 3.2 Ragged Paging (H_p-head groups, budget-aware clustering), 3.3 (split map)",
            "L": L, "batch": batch, "H": H, "H_p": H_p, "P": P, "alpha": 1.5, "cluster": cluster,
            "Bhat_f32_bits": [f32hex(x) for x in Bh.ravel()], "N": N.tolist(),
            "order": pg["order"].tolist(), "ntok": pg["ntok"].tolist(), "pt_off": pg["pt_off"].tolist(),
            "pt_ids": pg["pt_ids"].tolist(), "n_pages": pg["n_pages"], "n_pages_monolithic": pg["n_pages_monolithic"],
            "Phi": pg["Phi"].tolist(), "N_CTA": 6, "S": S.tolist(), "work_list": wl}
    # attention and the log-sum-exp merge (float64)
    q = r.standard_normal(8)
    K = r.standard_normal((11, 8))
    V = r.standard_normal((11, 8))
    out, lse = tg.attention(q, K, V, 1 / math.sqrt(8))
    parts = [tg.attention_partial(q, K[a:b], V[a:b], 1 / math.sqrt(8)) for a, b in ((0, 4), (4, 5), (5, 11))]
    mo, ml = tg.merge_partials(parts)
    cases["attention"] = {"cite": f"{TANGRAM}, 3.3 (split-KV partials merged by log-sum-exp); {FLEXI}, Sparse decode",
                          "q": q.tolist(), "K": K.tolist(), "V": V.tolist(), "scale": 1 / math.sqrt(8),
                          "out": out.tolist(), "lse": lse, "merged_out": mo.tolist(), "merged_lse": ml}
    # Quest: min/max, float32 score in the fixed order, top-K
    d, Pq, n_pages = 32, 4, 7
    Kq = r.standard_normal((n_pages * Pq - 2, d)).astype(np.float32)
    Kq = Kq.astype(np.float64).astype(np.float32)
    mn, mx = fx.page_minmax(Kq, Pq)
    qh = r.standard_normal((2, d)).astype(np.float32)
    sc = fx.page_scores(qh, mn, mx)
    cases["quest"] = {"cite": f"{FLEXI}, Core method / Sparse decode (min-max page bound, top-K pages)",
                      "P": Pq, "K_f32_bits": [[f32hex(x) for x in row] for row in Kq],
                      "q_f32_bits": [[f32hex(x) for x in row] for row in qh],
                      "mn_f32_bits": [[f32hex(x) for x in row] for row in mn],
                      "mx_f32_bits": [[f32hex(x) for x in row] for row in mx],
                      "score_f32_bits": [f32hex(x) for x in sc],
                      "top3": fx.top_pages(sc, 3).tolist()}
    with open(os.path.join(HERE, "oracle_cases.json"), "w") as f:
        json.dump(cases, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main()
