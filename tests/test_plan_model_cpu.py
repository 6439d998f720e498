"""Properties of the planner's stated rules (host logic, via the Python model):
the items of one (sequence, kv head) tile exactly the key band without overlap,
split pieces respect the chunk, and the capacity bound of the workspace holds; for
16- and 8-row decode tiles, and with decode units run by the prefill kernel."""
import numpy as np
import pytest

import rpa_inputs as ri
from plan_model import band, plan


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("dec_rows,dec_on_pf", [(16, False), (8, False), (16, True)])
def test_items_cover_the_bands(seed, dec_rows, dec_on_pf):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 40))
    G = int(rng.choice([1, 2, 4, 8]))
    ql = rng.integers(0, 40, size=S)
    ql[rng.random(S) < 0.5] = 1
    kl = ql + rng.integers(0, 3000, size=S)
    p = ri.build(seed=seed, q_lens=ql, kv_lens=kl, num_q_heads=2 * G, num_kv_heads=2, head_dim=64,
                 page_size=16, sliding_window=(int(rng.integers(1, 500)) if seed % 2 else None))
    slots = int(rng.integers(1, 300))
    pl = plan(p, slots, dec_rows=dec_rows, dec_on_pf=dec_on_pf, n_sms=152, dec_bps=3, pf_bps=1)
    assert pl["status"] == 0
    items = np.concatenate([pl["dec"], pl["pf"]])
    for s in range(S):
        for h in range(2):
            mine = items[(items[:, 0] == s) & (items[:, 1] == h)]
            if ql[s] == 0:
                assert len(mine) == 0
                continue
            toks = np.zeros(ql[s], int)
            for it in mine:
                toks[it[2]: it[2] + it[3]] += 1
                lo, hi = band(int(kl[s]), int(ql[s]), int(it[2]), int(it[2] + it[3]), True,
                              p.sliding_window or 0)
                assert lo <= it[4] < it[5] <= hi
            dec_like = ql[s] * G <= dec_rows
            if dec_like:
                spans = sorted((int(it[4]), int(it[5])) for it in mine)
                lo, hi = band(int(kl[s]), int(ql[s]), 0, int(ql[s]), True, p.sliding_window or 0)
                assert spans[0][0] == lo and spans[-1][1] == hi
                for a, b in zip(spans, spans[1:]):
                    assert a[1] == b[0]
                assert all(b - a <= pl["chunk"] for a, b in spans)
            else:
                assert (toks == 1).all()
    # capacity bound used by rpa_create: units <= S + waves*slots/Hkv + 1 (decode)
    n_dec_units = len(pl["dec"]) // 2
    assert n_dec_units <= S + -(-4 * slots // 2) + 1


def test_bad_lengths_give_no_items():
    p = ri.random_small(3, num_seqs=3)
    p.kv_lens[1] = 0
    assert plan(p, 10)["status"] == 5
