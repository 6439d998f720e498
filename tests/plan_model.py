"""Python re-derivation of the device planner's work list (host logic, no GPU).

Written from the planner's stated rules, not from its code: decode-class
sequences (q_len * G <= decode rows) are cut into key pieces of `chunk` keys,
prefill-class sequences into query tiles of pf_tokens tokens; each unit's
key range is the band its rows can see; units are ordered decode first (by
cost descending), then prefill (sequences by their heaviest unit descending,
a sequence's units together, then cost descending; weights and costs in
16-key buckets), ties by unit index; each unit yields one item per kv head.
"""
import numpy as np


def band(kl, ql, i0, i1, causal, window):
    p_lo = kl - ql + i0
    p_hi = kl - ql + i1 - 1
    hi = min(kl, p_hi + 1) if causal else kl
    lo = max(0, p_lo - window + 1) if window else 0
    return lo, max(hi, lo)


# rates of the SM-split model (FLOP/ns per SM on prefill, B/ns per SM decode, HBM B/ns)
PF_SM_GFLOPS_TC, PF_SM_GFLOPS_MMA, DEC_SM_GBS, HBM_GBS = 6500, 800, 78, 6700


def split(prob, dec_keyheads, pf_keys, n_sms, dec_bps, pf_bps, concurrent, force_pf=0, force_dec=0):
    """(prefill CTAs, decode CTAs): minimise max(prefill time, decode time) over the
    prefill SM count, integer nanoseconds, first minimum wins."""
    latent = getattr(prob, "kv_layout", "split") == "latent"
    kv_elt = 2 if prob.kv_dtype in ("bf16", "f16") else 1
    tc = not latent and kv_elt == 2 and prob.head_dim in (64, 128)
    D, Hkv = prob.head_dim, prob.num_kv_heads
    pf_rows = 256 if tc else 16 if latent else 128
    rate = PF_SM_GFLOPS_MMA if latent else PF_SM_GFLOPS_TC
    dec_bytes = dec_keyheads * 2 * D * kv_elt
    pf_flops = pf_keys * Hkv * pf_rows * 4 * D
    pf_sms = dec_sms = n_sms
    if concurrent and dec_bytes > 0 and pf_flops > 0:
        best, best_x = None, 1
        for x in range(1, n_sms):
            tp = pf_flops // (x * rate)
            td = dec_bytes // min(HBM_GBS, (n_sms - x) * DEC_SM_GBS)
            c = max(tp, td)
            if best is None or c < best:
                best, best_x = c, x
        if force_pf > 0:
            best_x = min(force_pf, n_sms - 1)
        pf_sms, dec_sms = best_x, n_sms - best_x
    if force_dec > 0:
        dec_sms = min(force_dec, n_sms)
    return pf_sms * pf_bps, dec_sms * dec_bps


def plan(prob, dec_slots=None, dec_rows=16, pf_tokens=None, waves=4, min_chunk=512, align=64,
         max_sort=8192, n_sms=None, dec_bps=None, pf_bps=1, concurrent=False, dec_on_pf=False):
    """dec_on_pf: decode units become items of the prefill kernel (leading its list) and their
    key pieces are sized for the prefill kernel's CTAs."""
    Hkv = prob.num_kv_heads
    G = prob.num_q_heads // Hkv
    Tq = max(1, pf_tokens if pf_tokens is not None else 64 // G)
    S = prob.num_seqs
    cu = prob.cu_q_lens.astype(np.int64)
    kvl = prob.kv_lens.astype(np.int64)
    win = prob.sliding_window or 0
    causal = prob.is_causal
    cls, cnt = [], []
    total = 0
    pf_keys = 0
    for s in range(S):
        q0, q1, kl = cu[s], cu[s + 1], kvl[s]
        ql = q1 - q0
        if q0 < 0 or ql < 0 or kl < 0 or kl > prob.pages_per_seq * prob.page_size or ql > kl \
                or q1 > prob.num_q_tokens:
            return dict(status=5, dec=np.zeros((0, 8), np.int32), pf=np.zeros((0, 8), np.int32))
        if ql == 0:
            cls.append(0); cnt.append(0)
        elif ql * G <= dec_rows:
            lo, hi = band(kl, ql, 0, ql, causal, win)
            cls.append(1); cnt.append(hi - lo)
            total += (hi - lo) * Hkv
        else:
            cls.append(2); cnt.append(-(-ql // Tq))
            for k in range(cnt[-1]):
                lo, hi = band(kl, ql, k * Tq, min(ql, (k + 1) * Tq), causal, win)
                pf_keys += hi - lo
    if n_sms is not None:
        pf_ctas, dec_ctas = split(prob, total, pf_keys, n_sms, dec_bps, pf_bps, concurrent)
    else:
        pf_ctas, dec_ctas = None, dec_slots
    target = waves * max(1, pf_ctas if dec_on_pf else dec_ctas)
    chunk = max(-(-total // target), min_chunk)
    chunk = -(-chunk // align) * align
    chunk = min(chunk, 1 << 30)
    units = []  # (cls_bit, cost, desc[8])
    part = 0
    for s in range(S):
        if cls[s] != 1:
            continue
        ql = int(cu[s + 1] - cu[s])
        lo, hi = band(int(kvl[s]), ql, 0, ql, causal, win)
        pieces = -(-cnt[s] // chunk)
        base = part if pieces > 1 else -1
        if pieces > 1:
            part += pieces * Hkv
        for k in range(pieces):
            kb = lo + k * chunk
            ke = min(hi, kb + chunk)
            units.append((0, ke - kb, [s, 0, ql, kb, ke, base, k, pieces]))
    weight = {}
    for s in range(S):
        if cls[s] != 2:
            continue
        ql = int(cu[s + 1] - cu[s])
        for k in range(cnt[s]):
            t0 = k * Tq
            nt = min(Tq, ql - t0)
            lo, hi = band(int(kvl[s]), ql, t0, t0 + nt, causal, win)
            units.append((1, hi - lo, [s, t0, nt, lo, hi, -1, 0, 1]))
            weight[s] = max(weight.get(s, 0), hi - lo)
    n = len(units)
    order = list(range(n))
    if n <= max_sort and S < 65536:
        # decode: cost descending; prefill: sequences by heaviest unit descending, a sequence's
        # units together, then cost descending (weights and costs in 16-key buckets); ties by unit
        def key(u):
            c, cost, d = units[u]
            if c == 0:
                return (0, 0x7FFFFFFF - cost, 0, 0, u)
            return (1, 0xFFFF - min(weight[d[0]] >> 4, 0xFFFF), d[0], 0xFFFF - min(cost >> 4, 0xFFFF), u)
        order.sort(key=key)
    dec, pf = [], []
    for u in order:
        c, _, d = units[u]
        for h in range(Hkv):
            item = [d[0], h, d[1], d[2], d[3], d[4], d[5] + h * d[7] + d[6] if d[5] >= 0 else -1, d[6]]
            (dec if c == 0 and not dec_on_pf else pf).append(item)
    return dict(status=0, chunk=chunk, sorted=int(n <= max_sort and S < 65536), n_units=n, n_part=part,
                pf_ctas=pf_ctas, dec_ctas=dec_ctas,
                dec=np.array(dec, np.int32).reshape(-1, 8), pf=np.array(pf, np.int32).reshape(-1, 8))
