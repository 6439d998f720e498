"""Seeded synthetic inputs for ragged paged attention.

This module only *draws* inputs: sequence lengths, a shuffled page table,
queries and the paged K/V cache.  It holds none of the attention arithmetic,
so both the CUDA path and the CPU oracle can consume the same bytes.

Layouts follow the "ragged_paged.zig" page (kernel arguments of ``run``):

* ``q``            [num_q_tokens, num_q_heads, head_dim]   bf16 or f16 bits
                   (uint16), or float32
* ``kv_pages``     [total_num_pages, page_size, 2*num_kv_heads, head_dim]
                   bf16 or f16 bits (uint16), fp8 e4m3fn / e5m2 bytes (uint8)
                   or int8; combined head 2h is K of kv head h, 2h+1 is V of
                   kv head h.
                   Latent layout: [total_num_pages, page_size, num_kv_heads,
                   head_dim], K = the row, V = its first v_head_dim elements.
* ``kv_lens``      [max_num_seqs]                 int32
* ``page_indices`` [max_num_seqs, pages_per_seq]  int32
* ``cu_q_lens``    [max_num_seqs + 1]             int32

Recipe (fixed, so every run sees the same bytes):

1. ``default_rng([seed, 0])`` draws the lengths, then a permutation of the
   physical pages, then the page ids of unused page-table entries.
2. Logical pages of the sequences take the permutation in order (sequence 0's
   pages first), so physical placement is shuffled.
3. ``q`` and ``kv_pages`` are filled chunk by chunk (2**22 elements per chunk)
   from ``default_rng([seed, 1, chunk])`` and ``default_rng([seed, 2, chunk])``.
   Every element of ``kv_pages`` is drawn, tail slots and unused pages too.
4. Values are N(0, 1) in float32, rounded to bf16 (or f16) with
   round-to-nearest-even, or kept as float32 for f32 q.  fp8 K/V values are
   ``clip(N(0,1) / 0.05, -448, 448)`` rounded to e4m3fn, or
   ``clip(N(0,1) / 0.05, -57344, 57344)`` rounded to e5m2; int8 K/V values are
   ``clip(rint(N(0,1) / 0.04), -127, 127)`` (used with scales 0.05 / 0.04).
5. Attention sinks, when asked for, are one float32 logit per query head drawn
   as N(0, 2^2) from ``default_rng([seed, 3])``.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

MASK_VALUE = -2.38197633e38  # "ragged_paged.zig", Cfg.mask_value default
CHUNK = 1 << 22


@dataclass
class Problem:
    """One ragged paged attention call: configuration plus host arrays."""

    num_q_tokens: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    total_num_pages: int
    page_size: int
    max_num_seqs: int
    pages_per_seq: int
    kv_dtype: str  # "bf16", "f16", "fp8_e4m3", "fp8_e5m2" or "int8"
    sm_scale: float
    soft_cap: float | None = None
    k_scale: float | None = None
    v_scale: float | None = None
    is_causal: bool = True
    sliding_window: int | None = None
    mask_value: float = MASK_VALUE
    sinks: np.ndarray | None = field(default=None, repr=False)  # float32 [num_q_heads] sink logits
    q_dtype: str = "bf16"  # "bf16", "f16" or "f32" (o has the same type)
    kv_layout: str = "split"  # "split" ([N, ps, 2*Hkv, D], K/V interleaved) or "latent" ([N, ps, Hkv, D])
    v_head_dim: int | None = None  # latent layout: width of V and o (the first v_head_dim of each row)
    num_seqs: int = 0
    q: np.ndarray = field(default=None, repr=False)
    kv_pages: np.ndarray = field(default=None, repr=False)
    kv_lens: np.ndarray = field(default=None, repr=False)
    page_indices: np.ndarray = field(default=None, repr=False)
    cu_q_lens: np.ndarray = field(default=None, repr=False)
    name: str = "custom"

    def cfg_dict(self) -> dict:
        return dict(
            num_q_tokens=self.num_q_tokens, num_q_heads=self.num_q_heads,
            num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
            total_num_pages=self.total_num_pages, page_size=self.page_size,
            max_num_seqs=self.max_num_seqs, pages_per_seq=self.pages_per_seq,
            kv_dtype=self.kv_dtype, sm_scale=self.sm_scale,
            soft_cap=self.soft_cap, k_scale=self.k_scale, v_scale=self.v_scale,
            is_causal=self.is_causal, sliding_window=self.sliding_window,
            mask_value=self.mask_value, sinks=self.sinks, q_dtype=self.q_dtype,
            kv_layout=self.kv_layout, v_head_dim=self.v_head_dim)

    @property
    def out_dim(self) -> int:
        """Width of V and of the output rows."""
        return self.v_head_dim if self.v_head_dim else self.head_dim

    @property
    def q_lens(self) -> np.ndarray:
        cu = self.cu_q_lens[: self.num_seqs + 1].astype(np.int64)
        return np.diff(cu)

    @property
    def seq_kv_lens(self) -> np.ndarray:
        return self.kv_lens[: self.num_seqs].astype(np.int64)


# ---------------------------------------------------------------- encoders
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bits.

    Inputs are finite, so no NaN special case is needed."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).copy()
    u += ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return (u >> 16).astype(np.uint16)


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 (already within +-448) to fp8 e4m3fn bytes via torch."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_e5m2_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 (already within +-57344) to fp8 e5m2 bytes via torch."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e5m2).view(torch.uint8).numpy().copy()


# storage type of each element type of q and kv_pages
Q_STORAGE = {"bf16": np.uint16, "f16": np.uint16, "f32": np.float32}
KV_STORAGE = {"bf16": np.uint16, "f16": np.uint16, "fp8_e4m3": np.uint8, "fp8_e5m2": np.uint8, "int8": np.int8}
KV_ELT = {"bf16": 2, "f16": 2, "fp8_e4m3": 1, "fp8_e5m2": 1, "int8": 1}
# fill kinds (the names of the first two are the recipe's originals)
_KV_FILL = {"bf16": "bf16", "f16": "f16", "fp8_e4m3": "fp8", "fp8_e5m2": "e5m2", "int8": "int8"}


def values_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact values of stored q / o / K / V elements of type `dtype` (via numpy / torch casts)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(bits).astype(np.float64)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "f32":
        return bits.astype(np.float64)
    if dtype == "int8":
        return bits.astype(np.float64)
    import torch

    tt = torch.float8_e4m3fn if dtype == "fp8_e4m3" else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(bits)).view(tt).double().numpy()


# ---------------------------------------------------------------- fills
def _fill(out_flat: np.ndarray, seed: int, stream: int, kind: str,
          threads: int | None = None) -> None:
    n = out_flat.size
    nchunks = (n + CHUNK - 1) // CHUNK

    def work(c: int) -> None:
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        rng = np.random.default_rng([seed, stream, c])
        x = rng.standard_normal(hi - lo, dtype=np.float32)
        if kind == "bf16":
            out_flat[lo:hi] = f32_to_bf16_bits(x)
        elif kind == "f16":
            out_flat[lo:hi] = x.astype(np.float16).view(np.uint16)
        elif kind == "f32":
            out_flat[lo:hi] = x
        elif kind == "fp8":
            np.clip(x / np.float32(0.05), -448.0, 448.0, out=x)
            out_flat[lo:hi] = f32_to_e4m3_bits(x)
        elif kind == "e5m2":
            np.clip(x / np.float32(0.05), -57344.0, 57344.0, out=x)
            out_flat[lo:hi] = f32_to_e5m2_bits(x)
        else:  # int8
            out_flat[lo:hi] = np.clip(np.rint(x / np.float32(0.04)), -127, 127).astype(np.int8)

    threads = threads or min(32, os.cpu_count() or 1)
    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
        return
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, range(nchunks)))


def build(*, seed: int, q_lens, kv_lens, num_q_heads: int, num_kv_heads: int,
          head_dim: int, page_size: int, pages_per_seq: int | None = None,
          total_num_pages: int | None = None, kv_dtype: str = "bf16",
          sm_scale: float | None = None, soft_cap=None, k_scale=None,
          v_scale=None, is_causal: bool = True, sliding_window=None,
          max_num_seqs: int | None = None, extra_tokens: int = 0,
          extra_pages: int = 0, name: str = "custom", sinks=None, q_dtype: str = "bf16",
          kv_layout: str = "split", v_head_dim: int | None = None,
          rng_lengths: np.random.Generator | None = None) -> Problem:
    """Build a problem with the given lengths (already drawn by the caller).

    ``sinks``: None (no attention sinks), True (drawn, recipe step 5) or an
    array of num_q_heads logits."""
    q_lens = np.asarray(q_lens, dtype=np.int64)
    kv_lens_a = np.asarray(kv_lens, dtype=np.int64)
    S = len(q_lens)
    assert len(kv_lens_a) == S
    npages = (kv_lens_a + page_size - 1) // page_size
    if pages_per_seq is None:
        pages_per_seq = max(1, int(npages.max()) if S else 1)
    used = int(npages.sum())
    if total_num_pages is None:
        total_num_pages = max(1, used + extra_pages)
    assert total_num_pages >= used
    max_num_seqs = max_num_seqs or max(S, 1)
    T = int(q_lens.sum()) + extra_tokens

    rng = rng_lengths if rng_lengths is not None else np.random.default_rng([seed, 0])
    perm = rng.permutation(total_num_pages).astype(np.int32)
    page_indices = rng.integers(0, total_num_pages, size=(max_num_seqs, pages_per_seq),
                                dtype=np.int64).astype(np.int32)
    off = 0
    for s in range(S):
        n = int(npages[s])
        page_indices[s, :n] = perm[off: off + n]
        off += n

    cu = np.zeros(max_num_seqs + 1, dtype=np.int32)
    cu[1: S + 1] = np.cumsum(q_lens)
    cu[S + 1:] = cu[S]
    kvl = np.zeros(max_num_seqs, dtype=np.int32)
    kvl[:S] = kv_lens_a

    Hq, Hkv, D = num_q_heads, num_kv_heads, head_dim
    q = np.empty((T, Hq, D), dtype=Q_STORAGE[q_dtype])
    _fill(q.reshape(-1), seed, 1, q_dtype)
    rows_per_slot = Hkv if kv_layout == "latent" else 2 * Hkv
    kv = np.empty((total_num_pages, page_size, rows_per_slot, D), dtype=KV_STORAGE[kv_dtype])
    _fill(kv.reshape(-1), seed, 2, _KV_FILL[kv_dtype])

    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if sinks is True:
        sinks = (np.random.default_rng([seed, 3]).standard_normal(Hq) * 2.0).astype(np.float32)
    elif sinks is not None:
        sinks = np.ascontiguousarray(sinks, dtype=np.float32).reshape(Hq)
    return Problem(
        num_q_tokens=T, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
        total_num_pages=total_num_pages, page_size=page_size,
        max_num_seqs=max_num_seqs, pages_per_seq=pages_per_seq,
        kv_dtype=kv_dtype, sm_scale=float(sm_scale), soft_cap=soft_cap,
        k_scale=k_scale, v_scale=v_scale, is_causal=is_causal,
        sliding_window=sliding_window, sinks=sinks, q_dtype=q_dtype, kv_layout=kv_layout,
        v_head_dim=v_head_dim if kv_layout == "latent" else None, num_seqs=S, q=q, kv_pages=kv,
        kv_lens=kvl, page_indices=page_indices, cu_q_lens=cu, name=name)


# ---------------------------------------------------------------- the five workloads
WORKLOADS = ("tiny", "decode", "mixed", "fp8_window", "long_prefill", "decode_quarter",
             "fp8_window_quarter", "mla_decode", "long_prefill_d256", "decode_g16")


def workload(name: str) -> Problem:
    """The named workloads (each with a seed of its own)."""
    if name == "tiny":
        # 3 sequences, q_lens {1,5,16}, kv_lens {17,40,64}, 16 physical pages.
        return build(seed=0, q_lens=[1, 5, 16], kv_lens=[17, 40, 64], num_q_heads=4,
                     num_kv_heads=2, head_dim=64, page_size=16, pages_per_seq=4,
                     total_num_pages=16, sm_scale=1.0 / 8.0, name=name)
    if name == "decode":
        # Llama-3-8B-like decode: 256 x q_len 1, kv_len ~ U[512, 8192].
        rng = np.random.default_rng([1, 0])
        kl = rng.integers(512, 8192, size=256, endpoint=True)
        return build(seed=1, q_lens=np.ones(256, np.int64), kv_lens=kl, num_q_heads=32,
                     num_kv_heads=8, head_dim=128, page_size=16, pages_per_seq=512,
                     sm_scale=1.0 / math.sqrt(128), name=name, rng_lengths=rng)
    if name == "decode_quarter":
        # the decode workload's first 64 sequences (same lengths and seeds): a
        # smaller case for profiler captures (K/V ~1.1 GB, still far above L2)
        rng = np.random.default_rng([1, 0])
        kl = rng.integers(512, 8192, size=256, endpoint=True)[:64]
        return build(seed=1, q_lens=np.ones(64, np.int64), kv_lens=kl, num_q_heads=32,
                     num_kv_heads=8, head_dim=128, page_size=16, pages_per_seq=512,
                     sm_scale=1.0 / math.sqrt(128), name=name, rng_lengths=rng)
    if name == "mixed":
        # 8 chunked-prefill chunks of 512 tokens + 56 decodes (4152 tokens).
        rng = np.random.default_rng([2, 0])
        kl_pf = rng.integers(0, 16384, size=8, endpoint=True) + 512
        kl_dec = rng.integers(1024, 32768, size=56, endpoint=True)
        ql = np.concatenate([np.full(8, 512), np.ones(56, np.int64)])
        kl = np.concatenate([kl_pf, kl_dec])
        return build(seed=2, q_lens=ql, kv_lens=kl, num_q_heads=32, num_kv_heads=8,
                     head_dim=128, page_size=32, pages_per_seq=1024,
                     sm_scale=1.0 / math.sqrt(128), name=name, rng_lengths=rng)
    if name == "fp8_window":
        # Gemma-2-like knobs with fp8 e4m3 K/V.
        rng = np.random.default_rng([3, 0])
        ql = rng.integers(1, 64, size=128, endpoint=True)
        kl = rng.integers(256, 16384, size=128, endpoint=True)
        return build(seed=3, q_lens=ql, kv_lens=kl, num_q_heads=16, num_kv_heads=8,
                     head_dim=256, page_size=16, pages_per_seq=1024, kv_dtype="fp8_e4m3",
                     sm_scale=1.0 / 16.0, soft_cap=50.0, k_scale=0.05, v_scale=0.05,
                     sliding_window=4096, name=name, rng_lengths=rng)
    if name == "fp8_window_quarter":
        # the fp8_window workload's first 32 sequences (same lengths and seeds): a
        # smaller case for profiler captures (K/V ~1.2 GB, still far above L2)
        rng = np.random.default_rng([3, 0])
        ql = rng.integers(1, 64, size=128, endpoint=True)[:32]
        kl = rng.integers(256, 16384, size=128, endpoint=True)[:32]
        return build(seed=3, q_lens=ql, kv_lens=kl, num_q_heads=16, num_kv_heads=8,
                     head_dim=256, page_size=16, pages_per_seq=1024, kv_dtype="fp8_e4m3",
                     sm_scale=1.0 / 16.0, soft_cap=50.0, k_scale=0.05, v_scale=0.05,
                     sliding_window=4096, name=name, rng_lengths=rng)
    if name == "long_prefill":
        # 4 fresh prefills of 8192 tokens, 64 q heads / 8 kv heads.
        rng = np.random.default_rng([4, 0])
        return build(seed=4, q_lens=[8192] * 4, kv_lens=[8192] * 4, num_q_heads=64,
                     num_kv_heads=8, head_dim=128, page_size=64, pages_per_seq=128,
                     total_num_pages=512, sm_scale=1.0 / math.sqrt(128), name=name,
                     rng_lengths=rng)
    if name == "long_prefill_d256":
        # long fresh prefill at head_dim 256 (Gemma-2-9B-like heads): 4 x 8192 tokens, 16 q heads /
        # 8 kv heads, page 64, bf16, causal
        rng = np.random.default_rng([6, 0])
        return build(seed=6, q_lens=[8192] * 4, kv_lens=[8192] * 4, num_q_heads=16, num_kv_heads=8,
                     head_dim=256, page_size=64, pages_per_seq=128, total_num_pages=512,
                     sm_scale=1.0 / 16.0, name=name, rng_lengths=rng)
    if name == "mla_decode":
        # latent attention decode, DeepSeek-V2-Lite-like: 128 x q_len 1, kv_len ~ U[1024, 8192],
        # 16 q heads on one latent kv head, rows of 576 (512 latent + 64 rope), values of 512,
        # page 64, bf16, softmax scale 1/sqrt(192) (the q.k width before the latent absorption)
        rng = np.random.default_rng([5, 0])
        kl = rng.integers(1024, 8192, size=128, endpoint=True)
        return build(seed=5, q_lens=np.ones(128, np.int64), kv_lens=kl, num_q_heads=16,
                     num_kv_heads=1, head_dim=576, page_size=64, pages_per_seq=128,
                     kv_layout="latent", v_head_dim=512, sm_scale=1.0 / math.sqrt(192), name=name,
                     rng_lengths=rng)
    if name == "decode_g16":
        # grouped decode with 16 q heads per kv head (the 16-row decode tiles): 256 x q_len 1,
        # kv_len ~ U[512, 8192], Hq 32 / Hkv 2, D 128, page 16, bf16
        rng = np.random.default_rng([7, 0])
        kl = rng.integers(512, 8192, size=256, endpoint=True)
        return build(seed=7, q_lens=np.ones(256, np.int64), kv_lens=kl, num_q_heads=32,
                     num_kv_heads=2, head_dim=128, page_size=16, pages_per_seq=512,
                     sm_scale=1.0 / math.sqrt(128), name=name, rng_lengths=rng)
    raise KeyError(name)


def random_small(seed: int, *, num_seqs: int = 3, max_q: int = 9, max_kv: int = 50,
                 num_q_heads: int = 4, num_kv_heads: int = 2, head_dim: int = 64,
                 page_size: int = 16, kv_dtype: str = "bf16", decode_only: bool = False,
                 **knobs) -> Problem:
    """A small random ragged batch (q_len <= kv_len) for tests."""
    rng = np.random.default_rng([seed, 0])
    kl = rng.integers(1, max_kv, size=num_seqs, endpoint=True)
    if decode_only:
        ql = np.ones(num_seqs, np.int64)
    else:
        ql = np.minimum(rng.integers(1, max_q, size=num_seqs, endpoint=True), kl)
    return build(seed=seed, q_lens=ql, kv_lens=kl, num_q_heads=num_q_heads,
                 num_kv_heads=num_kv_heads, head_dim=head_dim, page_size=page_size,
                 kv_dtype=kv_dtype, rng_lengths=rng, extra_pages=3, **knobs)


def algorithmic_work(p: Problem, decode_rows: int = 16) -> dict:
    """Algorithmic bytes and FLOPs of one call (keys in the allowed band only).

    bytes = sum_s n_kv(s) * row_bytes + T_used*Hq*(D + Dv)*q_elt + 4*(pages used + 2S + 1)
    flops = sum_s sum_i 2*Hq*(D + Dv)*n_allowed(s, i)

    row_bytes = 2*Hkv*D*kv_elt (K and V rows), or Hkv*D*kv_elt for the latent layout (K and V
    share the row); Dv = v_head_dim (= D except for the latent layout).

    The same sums split by sequence class are returned as ``decode`` and
    ``prefill`` (a sequence is decode-class when q_len * G <= decode_rows),
    so that each attention kernel is charged with the work it does.
    """
    Hq, Hkv, D = p.num_q_heads, p.num_kv_heads, p.head_dim
    kv_elt = KV_ELT[p.kv_dtype]
    q_elt = 4 if p.q_dtype == "f32" else 2  # q and o
    Dv = p.out_dim
    # bytes of one key's cache rows: K and V rows of every kv head, or (latent) the one shared row
    row_bytes = (Hkv * D if p.kv_layout == "latent" else 2 * Hkv * D) * kv_elt
    G = Hq // Hkv
    sw = p.sliding_window
    part = {"decode": [0, 0, 0, 0], "prefill": [0, 0, 0, 0]}  # bytes, pairs, pages, tokens
    for s in range(p.num_seqs):
        ql = int(p.cu_q_lens[s + 1] - p.cu_q_lens[s])
        kl = int(p.kv_lens[s])
        if ql == 0:
            continue
        i = np.arange(ql, dtype=np.int64)
        pos = kl - ql + i
        hi = np.minimum(pos + 1, kl) if p.is_causal else np.full(ql, kl)
        lo = np.maximum(pos - sw + 1, 0) if sw else np.zeros(ql, np.int64)
        n_allowed = np.maximum(hi - lo, 0)
        c = part["decode" if ql * G <= decode_rows else "prefill"]
        c[0] += (int(hi.max()) - int(lo.min())) * row_bytes + ql * Hq * (D + Dv) * q_elt
        c[1] += int(n_allowed.sum())
        c[2] += (kl + p.page_size - 1) // p.page_size
        c[3] += ql
    out = {}
    fpp = 2 * Hq * (D + Dv)  # FLOPs of one (query, key) pair over all q heads: QK^T and PV
    for k, (b, pairs, pages, toks) in part.items():
        out[k] = dict(bytes=b + 4 * pages, flops=fpp * pairs, q_tokens=toks)
    t_used = int(p.cu_q_lens[p.num_seqs])
    byts = out["decode"]["bytes"] + out["prefill"]["bytes"] + 4 * (2 * p.num_seqs + 1)
    pairs = (out["decode"]["flops"] + out["prefill"]["flops"]) // fpp
    return dict(bytes=byts, flops=fpp * pairs, exps=Hq * pairs, q_tokens=t_used,
                decode=out["decode"], prefill=out["prefill"])
