"""Pins for the fp64 oracle, independent of the oracle's own code.

Each pin is chosen so that a plausible slip in the oracle (a dropped scale, an
off-by-one in the query position, a swapped K/V head, a wrong window edge, a
mis-decoded fp8 code) fails at least one of them:

* format decoders (bf16, f16, e4m3fn, e5m2) against numpy / torch casts over
  their codes and the formats' fixed points; f16 / f32 queries and f16, e5m2
  and int8 K/V in the brute-force cases;
* brute-force dense attention in numpy (explicit mask matrix, softmax over a
  dense score matrix) on tiny unpaged inputs scattered into shuffled pages;
* closed forms: uniform V, a single allowed key, one-key sequences, zero-query
  means, two-key weights, zero-query means shrunk by a sink (n / (n + e^s));
* latent attention over a paged latent cache (the "from_qwen_ops.rs" page, "The
  latent-attention family at whole-tile widths"): a dense brute force, the
  split layout with zero-padded values, and zero-query means;
* attention sinks (the "from_qwen_ops.rs" page, flat_softmax_rows_at): the
  brute force takes the sink as one more always-allowed column with a zero
  value row; a very negative sink changes nothing;
* the softcap identity c*tanh(x/c) = 2c*sigmoid(2x/c) - c of the
  "from_qwen_ops.rs" page (``capped``) used as an independent formula;
* invariants: page placement, decode = last prefill row, poisoned tails,
  sequence order, GQA = MHA with repeated K/V, fp8 scales = pre-scaled bf16 K/V.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import rpa_inputs as ri
from rpa_inputs import Problem


# ------------------------------------------------------------------ helpers
def dense_problem(rng, q_lens, kv_lens, Hq, Hkv, D, ps, kv_dtype="bf16", q_dtype="bf16", **knobs):
    """Dense per-sequence K/V/Q drawn here, then scattered into shuffled pages.

    Returns (problem, dense) where dense[s] = (Q [ql,Hq,D], K [kl,Hkv,D], V [kl,Hkv,D])
    as float64 values of the stored bits (before k/v scales)."""
    S = len(q_lens)
    npages = [(k + ps - 1) // ps for k in kv_lens]
    N = sum(npages) + 2
    P = max(npages + [1])
    perm = rng.permutation(N)
    page_indices = np.zeros((S, P), np.int32)
    off = 0
    for s in range(S):
        page_indices[s, :npages[s]] = perm[off:off + npages[s]]
        page_indices[s, npages[s]:] = perm[-1]
        off += npages[s]
    T = int(sum(q_lens))
    qx = rng.standard_normal((T, Hq, D)).astype(np.float32)
    q = {"bf16": lambda: ri.f32_to_bf16_bits(qx), "f16": lambda: qx.astype(np.float16).view(np.uint16),
         "f32": lambda: qx}[q_dtype]()
    x = rng.standard_normal((N, ps, 2 * Hkv, D)).astype(np.float32)
    if kv_dtype == "bf16":
        kv = ri.f32_to_bf16_bits(x)
    elif kv_dtype == "f16":
        kv = x.astype(np.float16).view(np.uint16)
    elif kv_dtype == "fp8_e4m3":
        kv = ri.f32_to_e4m3_bits(np.clip(x / 0.05, -448, 448))
    elif kv_dtype == "fp8_e5m2":
        kv = ri.f32_to_e5m2_bits(np.clip(x / 0.05, -57344, 57344))
    else:
        kv = np.clip(np.rint(x / 0.04), -127, 127).astype(np.int8)
    dec = lambda b: ri.values_f64(b, kv_dtype)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    if knobs.get("sinks") is not None:
        knobs["sinks"] = np.asarray(knobs["sinks"], np.float32)
    prob = Problem(num_q_tokens=T, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                   total_num_pages=N, page_size=ps, max_num_seqs=S, pages_per_seq=P,
                   kv_dtype=kv_dtype, q_dtype=q_dtype, num_seqs=S, q=q, kv_pages=kv,
                   kv_lens=np.asarray(kv_lens, np.int32), page_indices=page_indices,
                   cu_q_lens=cu, sm_scale=knobs.pop("sm_scale", 1.0 / math.sqrt(D)), **knobs)
    qf = ri.values_f64(q, q_dtype)
    kvf = dec(kv).astype(np.float64)
    dense = []
    for s in range(S):
        kl = kv_lens[s]
        pg = page_indices[s, np.arange(kl) // ps]
        slot = np.arange(kl) % ps
        K = kvf[pg, slot][:, 0::2, :]
        V = kvf[pg, slot][:, 1::2, :]
        dense.append((qf[cu[s]:cu[s + 1]], K, V))
    return prob, dense


def brute(prob, dense, capped_form=False):
    """Dense softmax attention with an explicit mask matrix, fp64."""
    G = prob.num_q_heads // prob.num_kv_heads
    ks = prob.k_scale or 1.0
    vs = prob.v_scale or 1.0
    out = np.zeros((prob.num_q_tokens, prob.num_q_heads, prob.head_dim))
    for s, (Q, K, V) in enumerate(dense):
        ql, kl = Q.shape[0], K.shape[0]
        q0 = prob.cu_q_lens[s]
        pos = kl - ql + np.arange(ql)[:, None]
        col = np.arange(kl)[None, :]
        allowed = np.ones((ql, kl), bool)
        if prob.is_causal:
            allowed &= col <= pos
        if prob.sliding_window is not None:
            allowed &= ~(pos - prob.sliding_window >= col)
        for qh in range(prob.num_q_heads):
            h = qh // G
            x = prob.sm_scale * (Q[:, qh, :] @ (K[:, h, :] * ks).T)
            if prob.soft_cap is not None:
                c = prob.soft_cap
                if capped_form:
                    x = 2 * c / (1 + np.exp(-2 * x / c)) - c
                else:
                    x = c * np.tanh(x / c)
            x = np.where(allowed, x, -np.inf)
            Vh = V[:, h, :] * vs
            if prob.sinks is not None:
                # the sink as one more column of the score matrix, always allowed, whose value
                # row is zero
                x = np.concatenate([x, np.full((ql, 1), float(prob.sinks[qh]))], axis=1)
                allowed_s = np.concatenate([allowed, np.ones((ql, 1), bool)], axis=1)
                Vh = np.concatenate([Vh, np.zeros((1, Vh.shape[1]))], axis=0)
            else:
                allowed_s = allowed
            m = x.max(axis=1, keepdims=True)
            has = np.isfinite(m)
            w = np.where(allowed_s, np.exp(x - np.where(has, m, 0.0)), 0.0)
            den = w.sum(axis=1, keepdims=True)
            o = (w @ Vh) / np.where(den > 0, den, 1.0)
            # a row with no allowed key is zero (with a sink too: the sink carries no value)
            o[~allowed.any(axis=1)] = 0.0
            out[q0:q0 + ql, qh, :] = o
    return out


def dense_latent_problem(rng, q_lens, kv_lens, Hq, Hkv, D, Dv, ps, **knobs):
    """A latent-layout problem: one row of D elements per kv head and slot, drawn here and
    scattered into shuffled pages.  Returns (problem, dense) with dense[s] = (Q [ql,Hq,D],
    R [kl,Hkv,D]) as float64 values of the stored bits."""
    S = len(q_lens)
    npages = [(k + ps - 1) // ps for k in kv_lens]
    N = sum(npages) + 2
    P = max(npages + [1])
    perm = rng.permutation(N)
    page_indices = np.zeros((S, P), np.int32)
    off = 0
    for s in range(S):
        page_indices[s, :npages[s]] = perm[off:off + npages[s]]
        page_indices[s, npages[s]:] = perm[-1]
        off += npages[s]
    T = int(sum(q_lens))
    q = ri.f32_to_bf16_bits(rng.standard_normal((T, Hq, D)).astype(np.float32))
    kv = ri.f32_to_bf16_bits(rng.standard_normal((N, ps, Hkv, D)).astype(np.float32))
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    if knobs.get("sinks") is not None:
        knobs["sinks"] = np.asarray(knobs["sinks"], np.float32)
    prob = Problem(num_q_tokens=T, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                   total_num_pages=N, page_size=ps, max_num_seqs=S, pages_per_seq=P,
                   kv_dtype="bf16", kv_layout="latent", v_head_dim=Dv, num_seqs=S, q=q, kv_pages=kv,
                   kv_lens=np.asarray(kv_lens, np.int32), page_indices=page_indices,
                   cu_q_lens=cu, sm_scale=knobs.pop("sm_scale", 1.0 / math.sqrt(D)), **knobs)
    qf = ri.bf16_bits_to_f32(q).astype(np.float64)
    kvf = ri.bf16_bits_to_f32(kv).astype(np.float64)
    dense = []
    for s in range(S):
        kl = kv_lens[s]
        R = kvf[page_indices[s, np.arange(kl) // ps], np.arange(kl) % ps]
        dense.append((qf[cu[s]:cu[s + 1]], R))
    return prob, dense


def brute_latent(prob, dense):
    """Dense softmax attention over latent rows: K = the row, V = its first v_head_dim."""
    Dv = prob.v_head_dim
    split = [(Q, R, R[:, :, :Dv]) for Q, R in dense]
    out = np.zeros((prob.num_q_tokens, prob.num_q_heads, Dv))
    G = prob.num_q_heads // prob.num_kv_heads
    for s, (Q, K, V) in enumerate(split):
        ql, kl = Q.shape[0], K.shape[0]
        q0 = prob.cu_q_lens[s]
        pos = kl - ql + np.arange(ql)[:, None]
        col = np.arange(kl)[None, :]
        allowed = np.ones((ql, kl), bool)
        if prob.is_causal:
            allowed &= col <= pos
        if prob.sliding_window is not None:
            allowed &= ~(pos - prob.sliding_window >= col)
        for qh in range(prob.num_q_heads):
            h = qh // G
            x = prob.sm_scale * (Q[:, qh, :] @ K[:, h, :].T)
            if prob.soft_cap is not None:
                x = prob.soft_cap * np.tanh(x / prob.soft_cap)
            x = np.where(allowed, x, -np.inf)
            Vh = V[:, h, :]
            allowed_s = allowed
            if prob.sinks is not None:
                x = np.concatenate([x, np.full((ql, 1), float(prob.sinks[qh]))], axis=1)
                allowed_s = np.concatenate([allowed, np.ones((ql, 1), bool)], axis=1)
                Vh = np.concatenate([Vh, np.zeros((1, Dv))], axis=0)
            m = x.max(axis=1, keepdims=True)
            w = np.where(allowed_s, np.exp(x - m), 0.0)
            out[q0:q0 + ql, qh, :] = (w @ Vh) / w.sum(axis=1, keepdims=True)
    return out


def close(a, b, tol=1e-12):
    scale = max(1.0, float(np.abs(b).max()))
    err = float(np.abs(a - b).max()) / scale
    assert err <= tol, err


# ------------------------------------------------------------------ decoders
def test_bf16_decoder_matches_float32_view():
    for bits in list(range(0, 65536, 7)) + [0x3F80, 0xBF80, 0x7F7F, 0x0001, 0x8000]:
        ref = float(np.array([bits << 16], np.uint32).view(np.float32)[0])
        got = oracle.decode_bf16(bits)
        assert (math.isnan(ref) and math.isnan(got)) or ref == got, bits


def test_f16_decoder_all_codes():
    ref = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    for code in range(65536):
        got = oracle.decode_f16(code)
        r = float(ref[code])
        assert (math.isnan(r) and math.isnan(got)) or r == got, code
    # fixed points: 1, -2, max normal, min subnormal, min normal, infinities
    assert oracle.decode_f16(0x3C00) == 1.0 and oracle.decode_f16(0xC000) == -2.0
    assert oracle.decode_f16(0x7BFF) == 65504.0
    assert oracle.decode_f16(0x0001) == 2.0 ** -24 and oracle.decode_f16(0x0400) == 2.0 ** -14
    assert oracle.decode_f16(0x7C00) == math.inf and oracle.decode_f16(0xFC00) == -math.inf


def test_e5m2_decoder_all_codes():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e5m2).double()
    for code in range(256):
        got = oracle.decode_e5m2(code)
        r = float(ref[code])
        assert (math.isnan(r) and math.isnan(got)) or r == got, code
    # e5m2 is the upper byte of a binary16, and its fixed points: max 57344, min subnormal 2^-16
    for code in range(256):
        a, b = oracle.decode_e5m2(code), oracle.decode_f16(code << 8)
        assert (math.isnan(a) and math.isnan(b)) or a == b, code
    assert oracle.decode_e5m2(0x7B) == 57344.0 and oracle.decode_e5m2(0x01) == 2.0 ** -16
    assert oracle.decode_e5m2(0x3C) == 1.0 and oracle.decode_e5m2(0x7C) == math.inf


def test_e4m3_decoder_all_codes():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double()
    for code in range(256):
        got = oracle.decode_e4m3(code)
        r = float(ref[code])
        assert (math.isnan(r) and math.isnan(got)) or r == got, code
    # fixed points of the format: max normal, min subnormal, 1, -1, NaN
    assert oracle.decode_e4m3(0x7E) == 448.0
    assert oracle.decode_e4m3(0x01) == 2.0 ** -9
    assert oracle.decode_e4m3(0x08) == 2.0 ** -6
    assert oracle.decode_e4m3(0x38) == 1.0
    assert oracle.decode_e4m3(0xB8) == -1.0
    assert math.isnan(oracle.decode_e4m3(0x7F)) and math.isnan(oracle.decode_e4m3(0xFF))


# ------------------------------------------------------------------ brute force
CASES = [
    dict(q_lens=[1, 5, 16], kv_lens=[17, 40, 64], Hq=4, Hkv=2, D=64, ps=16),
    dict(q_lens=[3, 1, 7, 2], kv_lens=[3, 9, 30, 2], Hq=4, Hkv=4, D=16, ps=4),
    dict(q_lens=[6, 2], kv_lens=[20, 33], Hq=8, Hkv=2, D=16, ps=8, sliding_window=5),
    dict(q_lens=[4, 4], kv_lens=[11, 4], Hq=2, Hkv=1, D=16, ps=4, soft_cap=0.7, sm_scale=0.9),
    dict(q_lens=[5, 1], kv_lens=[9, 13], Hq=4, Hkv=2, D=16, ps=4, is_causal=False),
    dict(q_lens=[5, 3], kv_lens=[9, 13], Hq=4, Hkv=2, D=16, ps=4, is_causal=False,
         sliding_window=3),
    dict(q_lens=[3, 8], kv_lens=[40, 21], Hq=4, Hkv=2, D=32, ps=8, kv_dtype="fp8_e4m3",
         k_scale=0.05, v_scale=0.07, soft_cap=5.0, sliding_window=9, sm_scale=0.125),
    # attention sinks: plain, with soft cap and window, and sinks far above / below the logits
    dict(q_lens=[1, 5, 16], kv_lens=[17, 40, 64], Hq=4, Hkv=2, D=64, ps=16,
         sinks=[0.5, -1.0, 2.0, 0.0]),
    dict(q_lens=[6, 2], kv_lens=[20, 33], Hq=8, Hkv=2, D=16, ps=8, sliding_window=5, soft_cap=2.0,
         sinks=[3.0, -3.0, 0.1, 1.7, -0.4, 5.0, 0.0, 1.0]),
    dict(q_lens=[4, 4], kv_lens=[11, 4], Hq=2, Hkv=1, D=16, ps=4, is_causal=False, sinks=[40.0, -40.0]),
    # element types: f16 q and K/V; f32 q over bf16 K/V; e5m2 and int8 K/V with scales
    dict(q_lens=[1, 5, 16], kv_lens=[17, 40, 64], Hq=4, Hkv=2, D=64, ps=16, q_dtype="f16", kv_dtype="f16"),
    dict(q_lens=[6, 2], kv_lens=[20, 33], Hq=8, Hkv=2, D=16, ps=8, q_dtype="f32", sliding_window=5, soft_cap=2.0),
    dict(q_lens=[3, 8], kv_lens=[40, 21], Hq=4, Hkv=2, D=32, ps=8, kv_dtype="fp8_e5m2",
         k_scale=0.05, v_scale=0.07, soft_cap=5.0, sm_scale=0.125),
    dict(q_lens=[5, 3], kv_lens=[9, 30], Hq=4, Hkv=1, D=32, ps=4, q_dtype="f16", kv_dtype="int8",
         k_scale=0.04, v_scale=0.03, is_causal=False, sm_scale=0.2),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_oracle_equals_dense_brute_force(case):
    kw = dict(CASES[case])
    rng = np.random.default_rng(100 + case)
    prob, dense = dense_problem(rng, kw.pop("q_lens"), kw.pop("kv_lens"), kw.pop("Hq"),
                                kw.pop("Hkv"), kw.pop("D"), kw.pop("ps"), **kw)
    close(oracle.forward(prob), brute(prob, dense))


@pytest.mark.parametrize("seed", range(24))
def test_oracle_random_configs_equal_brute_force(seed):
    """Random small configurations (ragged lengths, GQA factor, page size, causal or not,
    window, soft cap, bf16 or fp8 with scales) against the dense brute force."""
    rng = np.random.default_rng([7, seed])
    S = int(rng.integers(1, 5))
    q_lens = [int(x) for x in rng.integers(1, 9, size=S)]
    kv_lens = [int(rng.integers(q, 49)) for q in q_lens]
    Hkv = int(rng.integers(1, 4))
    Hq = Hkv * int(rng.choice([1, 2, 4]))
    D = int(rng.choice([16, 32]))
    ps = int(rng.choice([4, 8, 16]))
    kw = dict(is_causal=bool(rng.integers(0, 2)), sm_scale=float(rng.uniform(0.05, 0.5)))
    if rng.integers(0, 2):
        kw["sliding_window"] = int(rng.integers(1, 40))
    if rng.integers(0, 2):
        kw["soft_cap"] = float(rng.uniform(0.5, 30.0))
    kvd = str(rng.choice(["bf16", "f16", "fp8_e4m3", "fp8_e5m2", "int8"]))
    kw["kv_dtype"] = kvd
    kw["q_dtype"] = str(rng.choice(["bf16", "f16", "f32"]))
    if kvd not in ("bf16", "f16"):
        kw.update(k_scale=float(rng.uniform(0.01, 0.1)), v_scale=float(rng.uniform(0.01, 0.1)))
    if rng.integers(0, 2):
        kw["sinks"] = (rng.standard_normal(Hq) * 2).astype(np.float32)
    prob, dense = dense_problem(rng, q_lens, kv_lens, Hq, Hkv, D, ps, **kw)
    close(oracle.forward(prob), brute(prob, dense))


def test_softcap_identity_from_capped_form():
    rng = np.random.default_rng(7)
    prob, dense = dense_problem(rng, [4, 9], [12, 30], 4, 2, 32, 8, soft_cap=1.5, sm_scale=1.0)
    close(oracle.forward(prob), brute(prob, dense, capped_form=True), 1e-12)
    # with a cap the logits never leave [-cap, cap]: scaling q by 1e3 must not blow up
    prob.q = ri.f32_to_bf16_bits(ri.bf16_bits_to_f32(prob.q) * 1000)
    o = oracle.forward(prob)
    assert np.isfinite(o).all()


def test_mask_value_additive_reading():
    """The page adds mask_value (-2.38e38) to masked logits; in f32 their exp is 0, so
    the additive mask equals dropping the key whenever a row keeps >= 1 key."""
    rng = np.random.default_rng(11)
    prob, dense = dense_problem(rng, [6], [10], 2, 1, 16, 4, sm_scale=0.3)
    Q, K, V = dense[0]
    pos = 10 - 6 + np.arange(6)[:, None]
    masked = np.arange(10)[None, :] > pos
    x = (prob.sm_scale * (Q[:, 0, :] @ K[:, 0, :].T)).astype(np.float32)
    x = x + np.where(masked, np.float32(ri.MASK_VALUE), np.float32(0))
    w = np.exp(x - x.max(axis=1, keepdims=True))
    o32 = (w @ V[:, 0, :]) / w.sum(axis=1, keepdims=True)
    assert (w[masked] == 0).all()
    close(oracle.forward(prob)[:, 0, :], o32, 1e-5)


# ------------------------------------------------------------------ closed forms
def test_uniform_v_gives_v():
    rng = np.random.default_rng(3)
    prob, _ = dense_problem(rng, [3, 7], [30, 17], 4, 2, 16, 4, soft_cap=3.0, sliding_window=6)
    vals = ri.f32_to_bf16_bits(rng.standard_normal((2, 16)).astype(np.float32))
    prob.kv_pages[:, :, 1, :] = vals[0]
    prob.kv_pages[:, :, 3, :] = vals[1]
    o = oracle.forward(prob)
    v = ri.bf16_bits_to_f32(vals).astype(np.float64)
    for qh in range(4):
        close(o[:, qh, :], np.broadcast_to(v[qh // 2], o[:, qh, :].shape), 1e-14)


def test_window_one_selects_own_position():
    """sliding_window = 1 keeps exactly key p = kv_len - q_len + i, so o = V[p]."""
    rng = np.random.default_rng(4)
    prob, dense = dense_problem(rng, [4, 1], [9, 6], 2, 1, 16, 4, sliding_window=1)
    o = oracle.forward(prob)
    for s, (Q, K, V) in enumerate(dense):
        ql, kl = Q.shape[0], K.shape[0]
        for i in range(ql):
            t = prob.cu_q_lens[s] + i
            for qh in range(2):
                close(o[t, qh], V[kl - ql + i, 0], 1e-14)


@pytest.mark.parametrize("causal,window", [(True, None), (True, 3), (True, 7), (False, None), (False, 4)])
def test_zero_query_averages_the_allowed_keys(causal, window):
    """q = 0 makes every logit 0, so o is the plain mean of V over the allowed keys: with the
    causal mask keys 0..p, with a window of w also j > p - w, without causality all keys (and
    j > p - w under a window).  Pins both mask edges and the 1 / sum normalisation."""
    rng = np.random.default_rng(12)
    prob, dense = dense_problem(rng, [5, 2], [12, 9], 2, 1, 16, 4, is_causal=causal,
                                sliding_window=window)
    prob.q = np.zeros_like(prob.q)
    o = oracle.forward(prob)
    for s, (Q, K, V) in enumerate(dense):
        ql, kl = Q.shape[0], K.shape[0]
        for i in range(ql):
            p = kl - ql + i
            lo = 0 if window is None else max(0, p - window + 1)
            hi = p if causal else kl - 1
            want = V[lo:hi + 1, 0].mean(axis=0)
            for qh in range(2):
                close(o[prob.cu_q_lens[s] + i, qh], want, 1e-13)


@pytest.mark.parametrize("sink", [0.0, math.log(3.0), -2.5])
def test_zero_query_mean_shrunk_by_a_sink(sink):
    """q = 0 makes every allowed logit 0, so each allowed key weighs 1 and the sink e^s: o is the
    mean of V over the n allowed keys times n / (n + e^s) (s = ln 3: n / (n + 3))."""
    rng = np.random.default_rng(14)
    Hq = 2
    prob, dense = dense_problem(rng, [5, 2], [12, 9], Hq, 1, 16, 4, sliding_window=4,
                                sinks=[sink, 0.0])
    prob.q = np.zeros_like(prob.q)
    o = oracle.forward(prob)
    for s, (Q, K, V) in enumerate(dense):
        ql, kl = Q.shape[0], K.shape[0]
        for i in range(ql):
            p = kl - ql + i
            lo = max(0, p - 4 + 1)
            n = p - lo + 1
            mean = V[lo:p + 1, 0].mean(axis=0)
            # the sink is stored as fp32: the closed form takes that value
            for qh, sv in ((0, float(np.float32(sink))), (1, 0.0)):
                close(o[prob.cu_q_lens[s] + i, qh], mean * n / (n + math.exp(sv)), 1e-13)


def test_very_negative_sink_changes_nothing():
    """A sink far below every logit has weight exp(-1e30) = 0 and does not move the maximum: the
    output equals the one without sinks, bit for bit."""
    prob = ri.random_small(28, num_seqs=4, max_q=9, max_kv=60, num_q_heads=4, num_kv_heads=2,
                           head_dim=32, page_size=8, soft_cap=10.0, sliding_window=20)
    o1 = oracle.forward(prob)
    prob.sinks = np.full(4, -1e30, np.float32)
    assert np.array_equal(o1, oracle.forward(prob))
    prob.sinks = np.zeros(4, np.float32)
    assert not np.array_equal(o1, oracle.forward(prob))


def test_two_keys_closed_form_weights():
    """Logits 0 and ln 3 (q = e_0, k_0 = 0, k_1 = 2 e_0, sm_scale = ln 3 / 2) weight V by 1/4 and
    3/4; with a soft cap c the second logit is c tanh(ln 3 / c)."""
    D = 16
    for cap in (None, 0.8):
        rng = np.random.default_rng(13)
        prob, dense = dense_problem(rng, [1], [2], 1, 1, D, 4, sm_scale=math.log(3.0) / 2,
                                    soft_cap=cap)
        q = np.zeros((1, 1, D), np.float32)
        q[0, 0, 0] = 1.0
        prob.q = ri.f32_to_bf16_bits(q)
        kvb = np.zeros(prob.kv_pages.shape, np.float32)
        vals = rng.standard_normal((2, D)).astype(np.float32)
        pg = prob.page_indices[0, 0]
        kvb[pg, 1, 0, 0] = 2.0           # K of key 1 (key 0 stays 0)
        kvb[pg, 0, 1, :] = vals[0]       # V of key 0
        kvb[pg, 1, 1, :] = vals[1]       # V of key 1
        prob.kv_pages = ri.f32_to_bf16_bits(kvb)
        v = ri.bf16_bits_to_f32(prob.kv_pages[pg, :2, 1, :]).astype(np.float64)
        x1 = prob.sm_scale * 2.0  # the oracle computes in fp64 from the configured scale
        if cap is not None:
            x1 = cap * math.tanh(x1 / cap)
        w1 = math.exp(x1) / (1.0 + math.exp(x1))
        want = (1 - w1) * v[0] + w1 * v[1]
        close(oracle.forward(prob)[0, 0], want, 1e-13)
        if cap is None:
            assert abs(w1 - 0.75) < 1e-6


def test_single_key_sequence():
    rng = np.random.default_rng(5)
    prob, dense = dense_problem(rng, [1, 1], [1, 1], 4, 2, 16, 4)
    o = oracle.forward(prob)
    for s, (Q, K, V) in enumerate(dense):
        for qh in range(4):
            close(o[s, qh], V[0, qh // 2], 1e-14)


# ------------------------------------------------------------------ latent attention
LATENT_CASES = [
    dict(q_lens=[1, 5, 9], kv_lens=[17, 40, 30], Hq=8, Hkv=1, D=48, Dv=32, ps=8),
    dict(q_lens=[3, 1], kv_lens=[20, 33], Hq=4, Hkv=2, D=40, Dv=24, ps=4, sliding_window=6, soft_cap=3.0,
         sinks=[0.5, -1.0, 2.0, 0.0]),
    dict(q_lens=[4, 2], kv_lens=[9, 13], Hq=16, Hkv=1, D=72, Dv=64, ps=16, is_causal=False, sm_scale=0.1),
]


@pytest.mark.parametrize("case", range(len(LATENT_CASES)))
def test_latent_oracle_equals_dense_brute_force(case):
    kw = dict(LATENT_CASES[case])
    rng = np.random.default_rng(300 + case)
    prob, dense = dense_latent_problem(rng, kw.pop("q_lens"), kw.pop("kv_lens"), kw.pop("Hq"), kw.pop("Hkv"),
                                       kw.pop("D"), kw.pop("Dv"), kw.pop("ps"), **kw)
    close(oracle.forward(prob), brute_latent(prob, dense))


def test_latent_equals_split_layout_with_padded_values():
    """The latent layout is the split layout whose K row is the latent row and whose V row is the
    latent row's first v_head_dim elements followed by zeros: the split output's first v_head_dim
    columns equal the latent output bit for bit, and its other columns are zero."""
    rng = np.random.default_rng(310)
    Dv = 24
    lat, _ = dense_latent_problem(rng, [3, 6], [15, 26], 6, 2, 40, Dv, 4, soft_cap=4.0, sliding_window=9)
    o_lat = oracle.forward(lat)
    kvl = lat.kv_pages  # [N, ps, Hkv, D]
    split_kv = np.zeros(kvl.shape[:2] + (2 * kvl.shape[2], kvl.shape[3]), kvl.dtype)
    split_kv[:, :, 0::2] = kvl
    split_kv[:, :, 1::2, :Dv] = kvl[:, :, :, :Dv]
    sp = Problem(**{**lat.__dict__, "kv_layout": "split", "v_head_dim": None, "kv_pages": split_kv})
    o_sp = oracle.forward(sp)
    assert np.array_equal(o_sp[:, :, :Dv], o_lat)
    assert (o_sp[:, :, Dv:] == 0).all()


def test_latent_zero_query_averages_the_value_part():
    """q = 0: every allowed key weighs 1, so o is the mean of the allowed rows' first v_head_dim."""
    rng = np.random.default_rng(311)
    prob, dense = dense_latent_problem(rng, [4], [11], 2, 1, 32, 16, 4)
    prob.q = np.zeros_like(prob.q)
    o = oracle.forward(prob)
    Q, R = dense[0]
    for i in range(4):
        p = 11 - 4 + i
        for qh in range(2):
            close(o[i, qh], R[:p + 1, 0, :16].mean(axis=0), 1e-13)


# ------------------------------------------------------------------ invariants
def test_page_placement_invariance_bit_identical():
    prob = ri.random_small(21, num_seqs=4, max_q=7, max_kv=60, page_size=8)
    o1 = oracle.forward(prob)
    rng = np.random.default_rng(0)
    perm = rng.permutation(prob.total_num_pages)  # new physical slot of each page
    kv2 = np.empty_like(prob.kv_pages)
    kv2[perm] = prob.kv_pages
    prob.kv_pages = kv2
    prob.page_indices = perm[prob.page_indices].astype(np.int32)
    o2 = oracle.forward(prob)
    assert np.array_equal(o1, o2)


def test_decode_equals_last_prefill_row():
    L = 37
    pf = ri.build(seed=9, q_lens=[L], kv_lens=[L], num_q_heads=4, num_kv_heads=2, head_dim=32,
                  page_size=8, sliding_window=20, soft_cap=2.0)
    o_pf = oracle.forward(pf)
    dec = ri.build(seed=9, q_lens=[1], kv_lens=[L], num_q_heads=4, num_kv_heads=2, head_dim=32,
                   page_size=8, sliding_window=20, soft_cap=2.0)
    dec.kv_pages = pf.kv_pages
    dec.page_indices = pf.page_indices
    dec.q = pf.q[L - 1:L].copy()
    o_dec = oracle.forward(dec)
    assert np.array_equal(o_dec[0], o_pf[L - 1])


def test_tail_and_unused_pages_do_not_matter():
    prob = ri.random_small(22, num_seqs=3, max_q=5, max_kv=45, page_size=16)
    o1 = oracle.forward(prob)
    kvf = prob.kv_pages.copy()
    ps = prob.page_size
    used = set()
    for s in range(prob.num_seqs):
        kl = int(prob.kv_lens[s])
        for j in range((kl + ps - 1) // ps):
            used.add(int(prob.page_indices[s, j]))
    nan_bits = np.uint16(0x7FC0)
    for pg in range(prob.total_num_pages):
        if pg not in used:
            kvf[pg] = nan_bits
    for s in range(prob.num_seqs):
        kl = int(prob.kv_lens[s])
        if kl % ps:
            kvf[prob.page_indices[s, kl // ps], kl % ps:] = nan_bits
    prob.kv_pages = kvf
    assert np.array_equal(o1, oracle.forward(prob))


def test_sequence_order_invariance():
    prob = ri.random_small(23, num_seqs=4, max_q=6, max_kv=40)
    o1 = oracle.forward(prob)
    order = [2, 0, 3, 1]
    ql = prob.q_lens
    cu = prob.cu_q_lens
    q2 = np.concatenate([prob.q[cu[s]:cu[s + 1]] for s in order])
    prob2 = ri.build(seed=23, q_lens=ql[order], kv_lens=prob.kv_lens[order], num_q_heads=4,
                     num_kv_heads=2, head_dim=64, page_size=16,
                     total_num_pages=prob.total_num_pages)
    prob2.q = q2
    prob2.kv_pages = prob.kv_pages
    prob2.page_indices = prob.page_indices[order]
    o2 = oracle.forward(prob2)
    o1r = np.concatenate([o1[cu[s]:cu[s + 1]] for s in order])
    assert np.array_equal(o1r, o2)


def test_gqa_equals_mha_with_repeated_kv():
    prob = ri.random_small(24, num_seqs=3, max_q=5, max_kv=30, num_q_heads=6, num_kv_heads=2,
                           head_dim=16, page_size=4, soft_cap=4.0)
    o1 = oracle.forward(prob)
    G = 3
    kv = prob.kv_pages  # [N, ps, 2*Hkv, D]
    k = kv[:, :, 0::2]
    v = kv[:, :, 1::2]
    k = np.repeat(k, G, axis=2)
    v = np.repeat(v, G, axis=2)
    kv2 = np.empty(kv.shape[:2] + (2 * 6, kv.shape[3]), kv.dtype)
    kv2[:, :, 0::2] = k
    kv2[:, :, 1::2] = v
    prob.kv_pages = kv2
    prob.num_kv_heads = 6
    assert np.array_equal(o1, oracle.forward(prob))


def test_uncovered_tokens_are_zero():
    prob = ri.build(seed=25, q_lens=[2, 3], kv_lens=[5, 9], num_q_heads=2, num_kv_heads=1,
                    head_dim=16, page_size=4, extra_tokens=3)
    o = oracle.forward(prob)
    assert (o[5:] == 0).all() and (np.abs(o[:5]).sum() > 0)


# ------------------------------------------------------------------ validation
def test_validation_codes():
    prob = ri.random_small(26, num_seqs=3)
    assert oracle.validate(prob) == 0
    bad = ri.random_small(26, num_seqs=3)
    bad.page_indices[0, 0] = bad.total_num_pages
    assert oracle.validate(bad) == 4
    bad = ri.random_small(26, num_seqs=3)
    bad.kv_lens[1] = bad.pages_per_seq * bad.page_size + 1
    assert oracle.validate(bad) == 5
    bad = ri.random_small(26, num_seqs=3)
    bad.kv_lens[2] = int(bad.cu_q_lens[3] - bad.cu_q_lens[2]) - 1
    assert oracle.validate(bad) == 5
    bad = ri.random_small(26, num_seqs=3)
    bad.cu_q_lens[2] = bad.cu_q_lens[1] - 1
    assert oracle.validate(bad) == 5
    with pytest.raises(oracle.OracleError):
        oracle.forward(bad)


def test_scale_folding_equals_prescaled_bf16():
    """fp8 K/V with k_scale / v_scale equals bf16 K/V holding the decoded values times the scales
    (up to bf16 rounding of those products): the scales multiply K and V, not Q, O or the logits
    in some other place."""
    ks, vs = 0.05, 0.07
    p8 = ri.random_small(26, num_seqs=3, max_q=6, max_kv=40, num_q_heads=4, num_kv_heads=2, head_dim=32,
                         page_size=8, kv_dtype="fp8_e4m3", k_scale=ks, v_scale=vs, soft_cap=8.0)
    o8 = oracle.forward(p8)
    dec = torch.from_numpy(p8.kv_pages).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    scaled = dec.copy()
    scaled[:, :, 0::2] *= ks
    scaled[:, :, 1::2] *= vs
    pb = ri.random_small(26, num_seqs=3, max_q=6, max_kv=40, num_q_heads=4, num_kv_heads=2, head_dim=32,
                         page_size=8, soft_cap=8.0)
    assert np.array_equal(pb.kv_lens, p8.kv_lens) and np.array_equal(pb.cu_q_lens, p8.cu_q_lens)
    pb.q = p8.q
    pb.page_indices = p8.page_indices
    pb.kv_pages = ri.f32_to_bf16_bits(scaled.astype(np.float32))
    ob = oracle.forward(pb)
    assert np.abs(o8 - ob).max() <= 1e-2 * max(1.0, np.abs(o8).max())
    # and dropping either scale is visible
    p8.k_scale = None
    assert np.abs(oracle.forward(p8) - o8).max() > 1e-2


def test_rows_equal_forward_bit_for_bit():
    """oracle.rows (used for the sampled rows of the full-size parity cases and the CPU
    baseline) computes exactly the rows oracle.forward does, on one thread or several."""
    prob = ri.random_small(27, num_seqs=4, max_q=12, max_kv=80, num_q_heads=6, num_kv_heads=2,
                           head_dim=32, page_size=8, soft_cap=10.0, sliding_window=20)
    full = oracle.forward(prob)
    T = int(prob.cu_q_lens[prob.num_seqs])
    rng = np.random.default_rng(5)
    rows = np.stack([rng.integers(0, T, 40), rng.integers(0, prob.num_q_heads, 40)], axis=1).astype(np.int64)
    for nthreads in (1, 0):
        got = oracle.rows(prob, rows, nthreads=nthreads)
        assert np.array_equal(got, full[rows[:, 0], rows[:, 1]])
