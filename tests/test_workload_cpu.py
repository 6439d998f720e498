"""The roofline's numerator: rpa_inputs.algorithmic_work against a direct count.

bench.py charges each kernel with algorithmic bytes (K/V of the keys some query may read, q and o,
the page-table and length words) and FLOPs (4 * Hq * D per allowed query-key pair).  Here both are
recounted key by key with an explicit mask, for random batches with and without causality and
windows, and the per-class split (decode / prefill) must add up to the totals."""
import numpy as np
import pytest

import rpa_inputs as ri


def direct_count(p, decode_rows):
    Hq, Hkv, D = p.num_q_heads, p.num_kv_heads, p.head_dim
    G = Hq // Hkv
    elt = 2 if p.kv_dtype == "bf16" else 1
    tot = dict(decode=[0, 0, 0], prefill=[0, 0, 0])  # bytes, pairs, tokens
    for s in range(p.num_seqs):
        ql = int(p.cu_q_lens[s + 1] - p.cu_q_lens[s])
        kl = int(p.kv_lens[s])
        if ql == 0:
            continue
        keys, pairs = set(), 0
        for i in range(ql):
            pos = kl - ql + i
            for j in range(kl):
                if p.is_causal and j > pos:
                    continue
                if p.sliding_window and pos - p.sliding_window >= j:
                    continue
                keys.add(j)
                pairs += 1
        c = tot["decode" if ql * G <= decode_rows else "prefill"]
        pages = (kl + p.page_size - 1) // p.page_size
        c[0] += len(keys) * 2 * Hkv * D * elt + 2 * ql * Hq * D * 2 + 4 * pages
        c[1] += pairs
        c[2] += ql
    return tot


@pytest.mark.parametrize("seed", range(8))
def test_algorithmic_work_matches_a_direct_count(seed):
    rng = np.random.default_rng([11, seed])
    causal = bool(seed % 2)
    window = None if seed % 4 < 2 else int(rng.integers(1, 60))
    kv_dtype = "fp8_e4m3" if seed >= 6 else "bf16"
    p = ri.random_small(300 + seed, num_seqs=int(rng.integers(1, 7)), max_q=int(rng.integers(1, 40)),
                        max_kv=200, num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
                        kv_dtype=kv_dtype, is_causal=causal, sliding_window=window,
                        k_scale=0.05 if kv_dtype != "bf16" else None, v_scale=0.05 if kv_dtype != "bf16" else None)
    for decode_rows in (8, 16):
        w = ri.algorithmic_work(p, decode_rows=decode_rows)
        d = direct_count(p, decode_rows)
        Hq, D = p.num_q_heads, p.head_dim
        for k in ("decode", "prefill"):
            assert w[k]["bytes"] == d[k][0], k
            assert w[k]["flops"] == 4 * Hq * D * d[k][1], k
            assert w[k]["q_tokens"] == d[k][2], k
        assert w["flops"] == w["decode"]["flops"] + w["prefill"]["flops"]
        assert w["bytes"] == w["decode"]["bytes"] + w["prefill"]["bytes"] + 4 * (2 * p.num_seqs + 1)
        assert w["q_tokens"] == int(p.cu_q_lens[p.num_seqs])
