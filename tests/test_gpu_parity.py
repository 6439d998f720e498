"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerance: |gpu - oracle| <= 2e-2 + 2e-2*|oracle| for bf16 K/V and
6e-2 + 6e-2*|oracle| for fp8 K/V, element by element.  Small cases compare
every row; the full-size workloads compare every row (decode, mixed,
fp8_window) or a seeded sample of over 8 k rows that holds every query tile's
first and last row (long_prefill, 2.1 M rows), plus whole-output properties.
"""
import numpy as np
import pytest

import oracle
import rpa_inputs as ri
from gpu_util import assert_close, o_to_f64, run, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def test_tiny_workload_all_rows():
    p = ri.workload("tiny")
    got, st = run(p)
    assert st == 0
    assert_close(got, oracle.forward(p), p.kv_dtype, "tiny")


SMALL = [
    # (seed, kwargs) -- several tiles, ragged tails, every knob and head_dim
    (30, dict(num_seqs=5, max_q=40, max_kv=300, num_q_heads=8, num_kv_heads=2, head_dim=128)),
    (31, dict(num_seqs=4, max_q=90, max_kv=400, num_q_heads=4, num_kv_heads=4, head_dim=64,
              page_size=8)),
    (32, dict(num_seqs=3, max_q=70, max_kv=500, num_q_heads=16, num_kv_heads=8, head_dim=256,
              page_size=16, soft_cap=50.0, sliding_window=100, sm_scale=1 / 16)),
    (33, dict(num_seqs=6, max_q=20, max_kv=700, num_q_heads=16, num_kv_heads=8, head_dim=256,
              kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05, soft_cap=50.0, sliding_window=300,
              sm_scale=1 / 16)),
    (34, dict(num_seqs=5, max_q=50, max_kv=300, num_q_heads=8, num_kv_heads=1, head_dim=128,
              is_causal=False)),
    (35, dict(num_seqs=5, max_q=50, max_kv=300, num_q_heads=8, num_kv_heads=2, head_dim=64,
              is_causal=False, sliding_window=40, soft_cap=5.0)),
    (36, dict(num_seqs=16, decode_only=True, max_kv=3000, num_q_heads=32, num_kv_heads=8,
              head_dim=128)),
    (37, dict(num_seqs=9, decode_only=True, max_kv=2500, num_q_heads=16, num_kv_heads=8,
              head_dim=128, kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.07)),
    (38, dict(num_seqs=4, max_q=30, max_kv=200, num_q_heads=64, num_kv_heads=1, head_dim=64,
              page_size=64)),
    (39, dict(num_seqs=7, max_q=12, max_kv=2000, num_q_heads=12, num_kv_heads=3, head_dim=128,
              page_size=32, kv_dtype="fp8_e4m3", k_scale=0.5, sliding_window=1)),
    # fp8 prefill on the tensor-memory kernel: page runs of 64 / 8 keys, G = 8, 1 and 3
    (40, dict(num_seqs=4, max_q=300, max_kv=900, num_q_heads=16, num_kv_heads=2, head_dim=128,
              page_size=64, kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05, is_causal=False)),
    (41, dict(num_seqs=3, max_q=200, max_kv=600, num_q_heads=4, num_kv_heads=4, head_dim=256,
              page_size=8, kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.2, sm_scale=1 / 16)),
    (42, dict(num_seqs=5, max_q=100, max_kv=400, num_q_heads=6, num_kv_heads=2, head_dim=128,
              page_size=16, kv_dtype="fp8_e4m3", k_scale=0.05, soft_cap=30.0, sliding_window=150)),
    # decode tiles of <= 8 rows (keys on the MMA's M side): G = 8 / 1 / 3 at the 8-row class
    # boundary, D 64 / 256 / 128, long keys split across CTAs; and 16-row tiles for G = 16
    (43, dict(num_seqs=12, decode_only=True, max_kv=5000, num_q_heads=16, num_kv_heads=2, head_dim=64,
              page_size=32)),
    (44, dict(num_seqs=10, max_q=12, max_kv=3000, num_q_heads=4, num_kv_heads=4, head_dim=256,
              page_size=8, sliding_window=700)),
    (45, dict(num_seqs=9, max_q=3, max_kv=4000, num_q_heads=9, num_kv_heads=3, head_dim=128,
              soft_cap=20.0, is_causal=False)),
    (46, dict(num_seqs=8, decode_only=True, max_kv=4000, num_q_heads=32, num_kv_heads=2, head_dim=128)),
    # fp8 tensor-memory prefill with 8 / 4 / 2 / 1 copies of each query row (items of <= 16, 32,
    # 64 and 128 rows): G = 2 at D 256 with soft cap and window, G = 4 at D 128
    (47, dict(num_seqs=14, max_q=64, max_kv=1500, num_q_heads=16, num_kv_heads=8, head_dim=256,
              page_size=16, kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05, soft_cap=50.0,
              sliding_window=400, sm_scale=1 / 16)),
    (48, dict(num_seqs=10, max_q=40, max_kv=1200, num_q_heads=16, num_kv_heads=4, head_dim=128,
              page_size=32, kv_dtype="fp8_e4m3", k_scale=0.08, v_scale=0.1)),
    # fp8 K/V at D 64 on the tensor-memory kernel (one 128-byte column block a row; decode rows too)
    (70, dict(num_seqs=8, max_q=40, max_kv=900, num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
              kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.07, soft_cap=20.0, sliding_window=300)),
    (71, dict(num_seqs=10, decode_only=True, max_kv=3000, num_q_heads=8, num_kv_heads=2, head_dim=64,
              page_size=32, kv_dtype="fp8_e4m3", k_scale=0.08, v_scale=0.05)),
    # fp8 K/V with G >= 16 on the tensor-memory kernel: query tiles of 8, 4 and 2 tokens; decode rows
    # (q_len 1, G 16) as split pieces merged by the combine kernel
    (72, dict(num_seqs=9, max_q=20, max_kv=3000, num_q_heads=32, num_kv_heads=2, head_dim=128, page_size=16,
              kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05)),
    (73, dict(num_seqs=7, max_q=10, max_kv=2000, num_q_heads=32, num_kv_heads=1, head_dim=256, page_size=32,
              kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.06, soft_cap=50.0, sliding_window=700,
              sm_scale=1 / 16)),
    (74, dict(num_seqs=6, max_q=6, max_kv=1500, num_q_heads=64, num_kv_heads=1, head_dim=128, page_size=16,
              kv_dtype="fp8_e4m3", k_scale=0.07, v_scale=0.05, is_causal=False)),
    (75, dict(num_seqs=8, decode_only=True, max_kv=6000, num_q_heads=32, num_kv_heads=2, head_dim=256,
              page_size=16, kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05, sm_scale=1 / 16)),
    # attention sinks on every kernel: 8-row decode tiles and the bf16 tensor-memory prefill; 16-row
    # decode tiles with split pieces (the combine kernel adds the sink once); the fp8 tensor-memory
    # kernel with split pieces, soft cap and window; its direct mode (bf16 D 256) and D 64 (fp8)
    (76, dict(num_seqs=10, max_q=200, max_kv=2500, num_q_heads=16, num_kv_heads=4, head_dim=128, sinks=True)),
    (77, dict(num_seqs=8, max_q=2, max_kv=5000, num_q_heads=32, num_kv_heads=2, head_dim=128, sinks=True)),
    (78, dict(num_seqs=12, max_q=40, max_kv=5000, num_q_heads=16, num_kv_heads=8, head_dim=256, page_size=16,
              kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05, soft_cap=50.0, sliding_window=1500,
              sm_scale=1 / 16, sinks=True)),
    (79, dict(num_seqs=5, max_q=70, max_kv=900, num_q_heads=8, num_kv_heads=2, head_dim=256, sinks=True)),
    (80, dict(num_seqs=8, max_q=30, max_kv=3000, num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
              kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.07, sinks=True)),
    # fp8 K/V at D 64 with G 32 (4-token query tiles) over page runs of 4 keys (16 copies a tile),
    # non-causal; and G 16 decode rows over long keys (split pieces, sinks)
    (82, dict(num_seqs=7, max_q=10, max_kv=2500, num_q_heads=32, num_kv_heads=1, head_dim=64, page_size=4,
              kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05, is_causal=False)),
    (83, dict(num_seqs=6, decode_only=True, max_kv=7000, num_q_heads=16, num_kv_heads=1, head_dim=64,
              page_size=64, kv_dtype="fp8_e4m3", k_scale=0.06, v_scale=0.05, sinks=True)),
    # int8 K/V at D 64 with G 64 (2-token query tiles, 8 copies of each row), page runs of 8 keys, window
    (84, dict(num_seqs=5, max_q=6, max_kv=1200, num_q_heads=64, num_kv_heads=1, head_dim=64, page_size=8,
              kv_dtype="int8", k_scale=0.04, v_scale=0.04, sliding_window=500)),
    (81, dict(num_seqs=16, decode_only=True, max_kv=8000, num_q_heads=32, num_kv_heads=8, head_dim=128,
              sinks=True)),
]


# Page sizes that are not powers of two (multiples of 4, or of 8 for the latent layout): the gather's
# page runs are the largest power of two dividing the page size (4, 8 or 16 slots), every run inside
# one page, on each kernel: 8-row decode tiles with the bf16 128-key-tile prefill, 16-row decode
# tiles, the 8-bit 64-key-tile kernel, its direct mode (bf16 D 256) and the latent kernel
ODD_PAGES = [
    (110, dict(num_seqs=8, max_q=150, max_kv=2500, num_q_heads=16, num_kv_heads=4, head_dim=128, page_size=48)),
    (111, dict(num_seqs=10, max_q=2, max_kv=3000, num_q_heads=32, num_kv_heads=2, head_dim=128, page_size=12)),
    (112, dict(num_seqs=8, max_q=60, max_kv=2500, num_q_heads=16, num_kv_heads=8, head_dim=256, page_size=24,
               kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05, soft_cap=50.0, sliding_window=900, sm_scale=1 / 16)),
    (113, dict(num_seqs=6, max_q=80, max_kv=1500, num_q_heads=8, num_kv_heads=4, head_dim=256, page_size=80,
               sm_scale=1 / 16)),
    (114, dict(num_seqs=8, max_q=3, max_kv=3000, num_q_heads=16, num_kv_heads=1, head_dim=576, page_size=40,
               kv_layout="latent", v_head_dim=512, sm_scale=1 / 24)),
    (115, dict(num_seqs=7, max_q=40, max_kv=2000, num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=20,
               kv_dtype="int8", k_scale=0.04, v_scale=0.04)),
]


@pytest.mark.parametrize("case", range(len(ODD_PAGES)))
def test_page_sizes_not_powers_of_two(case):
    seed, kw = ODD_PAGES[case]
    p = ri.random_small(seed, **kw)
    got, st = run(p)
    assert st == 0
    assert_close(got, oracle.forward(p), p.kv_dtype, f"page size {kw['page_size']}")


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_cases_all_rows(case):
    seed, kw = SMALL[case]
    p = ri.random_small(seed, **kw)
    got, st = run(p)
    assert st == 0
    assert_close(got, oracle.forward(p), p.kv_dtype, f"small case {case}")


# Element types (q / o, and K/V) on every kernel that serves them.  f16 K/V: f16 MMAs on the 8- and
# 16-row decode tiles, the tensor-memory prefill (D 64, 128) and the 64-key-tile kernel's direct
# mode (D 256).  e5m2 and int8 K/V: the 8-bit tensor-memory kernel (D 64, 128, 256; decode rows
# too, split pieces).  q of another type than the MMA operand type: rounded
# into the workspace first (f32 q; f16 q with bf16 K/V; bf16 q with f16 K/V); f16 q with 8-bit K/V
# read as it is.  o has q's type.
DTYPE_CASES = [
    (90, dict(num_seqs=10, max_q=150, max_kv=2500, num_q_heads=16, num_kv_heads=4, head_dim=128,
              q_dtype="f16", kv_dtype="f16")),
    (91, dict(num_seqs=8, max_q=60, max_kv=1500, num_q_heads=8, num_kv_heads=8, head_dim=64, page_size=32,
              q_dtype="f16", kv_dtype="f16", soft_cap=20.0, sliding_window=300)),
    (92, dict(num_seqs=9, max_q=3, max_kv=4000, num_q_heads=32, num_kv_heads=2, head_dim=128,
              q_dtype="bf16", kv_dtype="f16")),
    (93, dict(num_seqs=6, max_q=70, max_kv=900, num_q_heads=8, num_kv_heads=2, head_dim=256,
              q_dtype="f16", kv_dtype="f16", sm_scale=1 / 16)),
    (94, dict(num_seqs=10, max_q=120, max_kv=2000, num_q_heads=16, num_kv_heads=4, head_dim=128,
              q_dtype="f16", kv_dtype="bf16", sinks=True)),
    (95, dict(num_seqs=10, max_q=120, max_kv=2000, num_q_heads=16, num_kv_heads=4, head_dim=128,
              q_dtype="f32", kv_dtype="bf16", sliding_window=500)),
    (96, dict(num_seqs=12, max_q=40, max_kv=4000, num_q_heads=16, num_kv_heads=8, head_dim=256, page_size=16,
              kv_dtype="fp8_e5m2", k_scale=0.05, v_scale=0.05, soft_cap=50.0, sm_scale=1 / 16)),
    (97, dict(num_seqs=10, max_q=40, max_kv=3000, num_q_heads=16, num_kv_heads=4, head_dim=128, page_size=32,
              q_dtype="f16", kv_dtype="fp8_e5m2", k_scale=0.05, v_scale=0.06, sliding_window=700)),
    (98, dict(num_seqs=12, max_q=40, max_kv=4000, num_q_heads=16, num_kv_heads=8, head_dim=256, page_size=16,
              kv_dtype="int8", k_scale=0.04, v_scale=0.04, sm_scale=1 / 16, sinks=True)),
    (99, dict(num_seqs=10, max_q=40, max_kv=3000, num_q_heads=32, num_kv_heads=2, head_dim=128, page_size=16,
              q_dtype="f32", kv_dtype="int8", k_scale=0.04, v_scale=0.03)),
    (100, dict(num_seqs=8, max_q=30, max_kv=2500, num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
               kv_dtype="fp8_e5m2", k_scale=0.05, v_scale=0.05, soft_cap=20.0)),
    (101, dict(num_seqs=8, max_q=30, max_kv=2500, num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
               q_dtype="f16", kv_dtype="int8", k_scale=0.04, v_scale=0.04)),
    (102, dict(num_seqs=8, max_q=30, max_kv=2500, num_q_heads=16, num_kv_heads=8, head_dim=256, page_size=16,
               q_dtype="f16", kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05, sm_scale=1 / 16)),
]


# 2-byte K/V at D 256 on the 64-key-tile tensor-memory kernel (direct mode: K and V copied straight
# into the MMA tiles): decode rows as split pieces, G = 16 with page runs of 8 keys, f16 with sinks
# and no causal mask
D256_CASES = [
    (115, dict(num_seqs=10, decode_only=True, max_kv=6000, num_q_heads=16, num_kv_heads=8, head_dim=256,
               sm_scale=1 / 16)),
    (116, dict(num_seqs=8, max_q=20, max_kv=1500, num_q_heads=32, num_kv_heads=2, head_dim=256, page_size=8,
               soft_cap=50.0, sliding_window=500, sm_scale=1 / 16)),
    (117, dict(num_seqs=7, max_q=150, max_kv=1200, num_q_heads=8, num_kv_heads=2, head_dim=256, page_size=32,
               q_dtype="f16", kv_dtype="f16", is_causal=False, sinks=True, sm_scale=1 / 16)),
    # page runs of a whole 64-key tile: one copy per K (V) tile
    (118, dict(num_seqs=6, max_q=300, max_kv=1400, num_q_heads=16, num_kv_heads=8, head_dim=256, page_size=64,
               sm_scale=1 / 16)),
    (119, dict(num_seqs=9, max_q=90, max_kv=2000, num_q_heads=8, num_kv_heads=4, head_dim=256, page_size=128,
               kv_dtype="f16", q_dtype="f32", sliding_window=700, soft_cap=30.0, sm_scale=1 / 16)),
]


@pytest.mark.parametrize("case", range(len(D256_CASES)), ids=[f"seed{c[0]}" for c in D256_CASES])
def test_d256_tensor_memory_cases_all_rows(case):
    seed, kw = D256_CASES[case]
    p = ri.random_small(seed, **kw)
    got, st = run(p)
    assert st == 0
    assert_close(got, oracle.forward(p), p.kv_dtype, f"D 256 case {case}")


def test_d256_repeated_calls_identical_and_in_tolerance():
    """The 64-key-tile kernel's pipeline (three K/V buffers a tile apart, P ready and V ready on
    barriers of their own) under repetition: every call of the whole-tile page-run cases matches
    the oracle and the first call bit for bit (a barrier phase completed by the wrong tile's
    arrivals shows as a call that reads P or V before it is written)."""
    for seed, kw in D256_CASES[3:]:
        p = ri.random_small(seed, **kw)
        ref = oracle.forward(p)
        t = to_dev(p)
        first = None
        for _ in range(6):
            got, st = run(p, tensors=t)
            assert st == 0
            assert_close(got, ref, p.kv_dtype, f"D 256 seed {seed}")
            if first is None:
                first = got
            assert np.array_equal(got, first)


MANY_PIECES = [
    # decode kernel (8-row tiles): three long decodes split into ~78 pieces each
    ("decode-bf16", dict(q_lens=[1, 1, 1], kv_lens=[60000, 45000, 70000], num_q_heads=32, num_kv_heads=8,
                         head_dim=128, page_size=16, sm_scale=1 / 11.3)),
    # 64-key-tile kernel (8-bit K/V at D 256): one decode across every CTA (~76 pieces)
    ("tc8-fp8", dict(q_lens=[1], kv_lens=[70000], num_q_heads=16, num_kv_heads=8, head_dim=256, page_size=16,
                     kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05, sm_scale=1 / 16)),
    # latent kernel: ~60-80 pieces a sequence, with sinks (added once, by the merge)
    ("latent-sinks", dict(q_lens=[1, 1], kv_lens=[40000, 30000], num_q_heads=16, num_kv_heads=1, head_dim=576,
                          v_head_dim=512, kv_layout="latent", page_size=64, sinks=True, sm_scale=1 / 24)),
]


@pytest.mark.parametrize("case", range(len(MANY_PIECES)), ids=[c[0] for c in MANY_PIECES])
def test_many_split_pieces_all_rows(case):
    """Long decodes split into more than 32 pieces: the combine's streaming path (pieces beyond the
    eight held in registers, scale factors beyond the first 32 recomputed), all rows vs the oracle."""
    name, kw = MANY_PIECES[case]
    p = ri.build(seed=130 + case, name=name, **kw)
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention

    att = RaggedPagedAttention(**p.cfg_dict())
    o = att.forward(*to_dev(p), p.num_seqs)
    assert att.status() == 0
    info, items = att.plan()
    pieces = {}
    for it in items:
        key = (int(it[0]), int(it[1]))
        pieces[key] = pieces.get(key, 0) + 1
    assert max(pieces.values()) > 32, pieces
    got = o_to_f64(o)
    att.close()
    assert_close(got, oracle.forward(p), p.kv_dtype, f"many pieces {name}")


@pytest.mark.parametrize("case", range(len(DTYPE_CASES)), ids=[f"{c[1].get('q_dtype', 'bf16')}-"
                                                               f"{c[1]['kv_dtype']}-seed{c[0]}" for c in DTYPE_CASES])
def test_dtype_cases_all_rows(case):
    seed, kw = DTYPE_CASES[case]
    p = ri.random_small(seed, **kw)
    got, st = run(p)
    assert st == 0
    assert_close(got, oracle.forward(p), p.kv_dtype, f"dtype case {case}")


# Latent attention over a paged latent cache (rows of 576: a 512-wide latent, whose part is the
# value, and a 64-wide rope part): decode rows split into pieces (combine kernel), prefill tiles,
# G = 16, 8 and 128 (blocks of 16 q heads per item), two kv heads, f16 rows, f32 q, sinks, soft cap
# and window, page sizes 16 and 64.
LATENT = dict(kv_layout="latent", head_dim=576, v_head_dim=512, sm_scale=1 / 24)
MLA_CASES = [
    (110, dict(num_seqs=10, decode_only=True, max_kv=4000, num_q_heads=16, num_kv_heads=1, page_size=64, **LATENT)),
    (111, dict(num_seqs=6, max_q=40, max_kv=900, num_q_heads=16, num_kv_heads=1, page_size=16, **LATENT)),
    (112, dict(num_seqs=8, max_q=9, max_kv=2000, num_q_heads=8, num_kv_heads=1, page_size=32, soft_cap=30.0,
               sliding_window=700, sinks=True, **LATENT)),
    (113, dict(num_seqs=5, max_q=3, max_kv=1500, num_q_heads=128, num_kv_heads=1, page_size=64, **LATENT)),
    (114, dict(num_seqs=6, max_q=12, max_kv=1200, num_q_heads=32, num_kv_heads=2, page_size=16, kv_dtype="f16",
               q_dtype="f32", is_causal=False, **LATENT)),
    # pages of whole 64-slot runs (one copy per stage), 12 q heads a latent kv head (rows past the tile's 12)
    (120, dict(num_seqs=6, max_q=40, max_kv=900, num_q_heads=16, num_kv_heads=1, page_size=64, **LATENT)),
    (121, dict(num_seqs=8, max_q=9, max_kv=2000, num_q_heads=8, num_kv_heads=1, page_size=128, soft_cap=30.0,
               sliding_window=700, sinks=True, **LATENT)),
    (122, dict(num_seqs=6, max_q=12, max_kv=1200, num_q_heads=32, num_kv_heads=2, page_size=64, kv_dtype="f16",
               q_dtype="f32", is_causal=False, **LATENT)),
    (123, dict(num_seqs=7, max_q=5, max_kv=3000, num_q_heads=12, num_kv_heads=1, page_size=64, **LATENT)),
]


@pytest.mark.parametrize("case", range(len(MLA_CASES)), ids=[f"seed{c[0]}" for c in MLA_CASES])
def test_latent_cases_all_rows(case):
    seed, kw = MLA_CASES[case]
    p = ri.random_small(seed, **kw)
    got, st = run(p)
    assert st == 0
    assert got.shape == (p.num_q_tokens, p.num_q_heads, 512)
    assert_close(got, oracle.forward(p), p.kv_dtype, f"latent case {case}")


@pytest.mark.parametrize("page_size", [16, 64])
def test_latent_poisoned_tails_and_unused_pages(page_size):
    """Latent rows past kv_len hold NaN and unused pages +inf, with page runs of 16 slots and of a
    whole 64-key stage (the value rows outside the key range are zeroed before the PV)."""
    p = ri.random_small(124, num_seqs=6, max_q=20, max_kv=700, num_q_heads=16, num_kv_heads=1,
                        page_size=page_size, extra_tokens=0, **LATENT)
    ref = oracle.forward(p)
    used = set()
    ps = p.page_size
    for s in range(p.num_seqs):
        kl = int(p.kv_lens[s])
        used.update(int(x) for x in p.page_indices[s, : (kl + ps - 1) // ps])
        if kl % ps:
            p.kv_pages[p.page_indices[s, kl // ps], kl % ps:] = 0x7FC0
    for pg in range(p.total_num_pages):
        if pg not in used:
            p.kv_pages[pg] = 0x7F80
    got, st = run(p)
    assert st == 0
    assert_close(got, ref, p.kv_dtype, "latent poisoned")


def _sample_rows(p, n, seed, tile_tokens):
    """n random (token, q head) rows, plus, for every query tile of `tile_tokens` tokens of every
    sequence, its first and last token, each with the first and the last q head of a random kv
    group (the first and last MMA rows of the tile), and every sequence's first and last token."""
    rng = np.random.default_rng(seed)
    G = p.num_q_heads // p.num_kv_heads
    T = int(p.cu_q_lens[p.num_seqs])
    toks, heads = [rng.integers(0, T, size=n)], [rng.integers(0, p.num_q_heads, size=n)]
    for s in range(p.num_seqs):
        q0, q1 = int(p.cu_q_lens[s]), int(p.cu_q_lens[s + 1])
        if q1 == q0:
            continue
        first = np.arange(q0, q1, tile_tokens)
        last = np.minimum(first + tile_tokens, q1) - 1
        for t in (first, last):
            grp = rng.integers(0, p.num_kv_heads, size=t.size) * G
            toks += [t, t]
            heads += [grp, grp + G - 1]
    rows = np.unique(np.stack([np.concatenate(toks), np.concatenate(heads)], axis=1), axis=0)
    return rows.astype(np.int64)


SAMPLED = {"long_prefill": 8000, "long_prefill_d256": 4000, "mla_decode": 800}


@pytest.mark.parametrize("name", ["decode", "mixed", "fp8_window", "long_prefill", "long_prefill_d256",
                                  "mla_decode", "decode_g16"])
def test_full_workloads(name):
    """The full-size workloads in the launch configuration the benchmark times.  decode, mixed,
    fp8_window and decode_g16: every output row against the oracle.  long_prefill (2.1 M rows), long_prefill_d256
    (0.5 M rows) and mla_decode (2 k rows of 8 k keys): a seeded sample holding the first and last
    row of every 128-row query tile (every sequence's token for the decode batch) beside random
    rows."""
    p = ri.workload(name)
    got, st = run(p)
    assert st == 0
    assert np.isfinite(got).all()
    if name not in SAMPLED:
        ref = oracle.forward(p)
        assert_close(got, ref, p.kv_dtype, name)
    else:
        G = p.num_q_heads // p.num_kv_heads
        rows = _sample_rows(p, 2000 if name != "mla_decode" else 800, 1234, tile_tokens=max(1, 128 // G))
        assert len(rows) >= SAMPLED[name]
        ref = oracle.rows(p, rows)
        assert_close(got[rows[:, 0], rows[:, 1]], ref, p.kv_dtype, name)


@pytest.mark.parametrize("kw,dec_bps,pf_bps", [
    # 8-row decode tiles: three CTAs per SM at D 128; 16-row tiles: two; the tensor-memory and latent
    # kernels: one
    (dict(num_q_heads=32, num_kv_heads=8, head_dim=128), 3, 1),
    (dict(num_q_heads=32, num_kv_heads=2, head_dim=128), 2, 1),
    (dict(num_q_heads=16, num_kv_heads=1, kv_layout="latent", head_dim=576, v_head_dim=512, page_size=64,
          sm_scale=1 / 24), None, 1),
    # 8-bit K/V: the 64-key-tile kernel takes the decode rows too (one CTA per SM), D 64 and 256
    (dict(num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05), 1, 1),
    (dict(num_q_heads=16, num_kv_heads=8, head_dim=256, kv_dtype="int8", k_scale=0.04, v_scale=0.04), 1, 1),
])
def test_resident_ctas_per_sm_as_designed(kw, dec_bps, pf_bps):
    """The kernels' register and shared-memory budgets give the occupancy they were designed for
    (rpa_read_plan info[13], info[14]): a budget over by a few registers silently halves a decode
    kernel's CTAs per SM."""
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention

    p = ri.random_small(51, num_seqs=4, max_q=3, max_kv=300, **kw)
    att = RaggedPagedAttention(**p.cfg_dict())
    att.forward(*to_dev(p), p.num_seqs)
    info = att.plan(max_items=1)[0]
    assert info[0] == 0
    if dec_bps is not None:
        assert int(info[13]) == dec_bps
    assert int(info[14]) == pf_bps
    att.close()


def test_planner_matches_python_rederivation():
    """The device planner's items, chunk, CTA split and sort flag equal a plain Python restatement.
    The cases span the sort's ranges: a few keys, a few thousand, and decode batches whose
    whole-chunk pieces skip the sort."""
    from plan_model import plan
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention

    for name in ("tiny", "mixed", "fp8", "decode", "long_prefill", "mla_decode", "decode_g16", "many_units",
                 "many_seqs"):
        if name in ("tiny", "decode", "long_prefill", "mla_decode", "decode_g16"):
            p = ri.workload(name)
        elif name == "mixed":
            p = ri.random_small(40, num_seqs=60, max_q=300, max_kv=5000, num_q_heads=32, num_kv_heads=8,
                                head_dim=128, sliding_window=777)
        elif name == "many_units":  # more units than the planner keeps in shared memory (1024)
            p = ri.random_small(42, num_seqs=300, max_q=250, max_kv=3000, num_q_heads=8, num_kv_heads=1,
                                head_dim=64)
        elif name == "many_seqs":  # more sequences than the planner's shared-memory scratch holds (4096)
            p = ri.random_small(43, num_seqs=5000, decode_only=True, max_kv=100, num_q_heads=4,
                                num_kv_heads=1, head_dim=64)
        else:  # fp8 K/V on tensor memory: decode units become prefill-kernel items
            p = ri.random_small(41, num_seqs=50, max_q=60, max_kv=6000, num_q_heads=16, num_kv_heads=8,
                                head_dim=256, kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05,
                                sliding_window=2000)
        att = RaggedPagedAttention(**p.cfg_dict())
        att.forward(*to_dev(p), p.num_seqs)
        info, items = att.plan()
        # the 64-key-tile kernel (8-bit K/V here) aims at 2 decode items a CTA, the others at 4
        ref = plan(p, dec_rows=int(info[5]), pf_tokens=int(info[6]), n_sms=int(info[12]), dec_bps=int(info[13]),
                   pf_bps=int(info[14]), concurrent=bool(info[15] & 1), dec_on_pf=bool(info[15] & 2),
                   waves=2 if name == "fp8" else 4)
        assert info[0] == 0 and info[4] == ref["chunk"] and info[8] == ref["n_units"]
        assert info[10] == ref["dec_ctas"] and info[11] == ref["pf_ctas"]
        assert info[9] == ref["sorted"] and info[7] == ref["n_part"]
        if name == "many_units":
            assert info[8] > 1024

        assert np.array_equal(items[: info[1]], ref["dec"])
        assert np.array_equal(items[info[1]:], ref["pf"])
        att.close()


def test_page_placement_invariance_bit_identical():
    p = ri.random_small(41, num_seqs=6, max_q=40, max_kv=900, num_q_heads=8, num_kv_heads=2,
                        head_dim=128)
    a, _ = run(p)
    perm = np.random.default_rng(1).permutation(p.total_num_pages)
    kv2 = np.empty_like(p.kv_pages)
    kv2[perm] = p.kv_pages
    p.kv_pages = kv2
    p.page_indices = perm[p.page_indices].astype(np.int32)
    b, _ = run(p)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("kv_dtype,head_dim,page_size", [("bf16", 128, 16), ("fp8_e4m3", 128, 16),
                                                         ("fp8_e4m3", 256, 16), ("f16", 128, 16),
                                                         ("fp8_e5m2", 256, 16), ("int8", 128, 16),
                                                         ("bf16", 256, 16), ("f16", 256, 16), ("bf16", 256, 64),
                                                         ("f16", 256, 128)])
def test_poisoned_tails_and_unused_pages(kv_dtype, head_dim, page_size):
    extra = {} if kv_dtype in ("bf16", "f16") else dict(k_scale=0.05, v_scale=0.05)
    p = ri.random_small(42, num_seqs=5, max_q=130, max_kv=500, num_q_heads=8, num_kv_heads=2,
                        head_dim=head_dim, page_size=page_size, extra_tokens=0, kv_dtype=kv_dtype, **extra)
    ref = oracle.forward(p)
    used = set()
    ps = p.page_size
    # NaN in the tails and +inf in the unused pages: bf16 0x7FC0 / 0x7F80, f16 0x7E00 / 0x7C00,
    # e5m2 0x7F / 0x7C; e4m3fn has no inf (NaN 0x7F in both); int8 has neither (extremes)
    nan, inf = {"bf16": (0x7FC0, 0x7F80), "f16": (0x7E00, 0x7C00), "fp8_e4m3": (0x7F, 0x7F),
                "fp8_e5m2": (0x7F, 0x7C), "int8": (-128, 127)}[kv_dtype]
    for s in range(p.num_seqs):
        kl = int(p.kv_lens[s])
        used.update(int(x) for x in p.page_indices[s, : (kl + ps - 1) // ps])
        if kl % ps:
            p.kv_pages[p.page_indices[s, kl // ps], kl % ps:] = nan
    for pg in range(p.total_num_pages):
        if pg not in used:
            p.kv_pages[pg] = inf
    got, st = run(p)
    assert st == 0
    assert_close(got, ref, p.kv_dtype, "poisoned")


def test_uncovered_tokens_and_padding_rows():
    p = ri.build(seed=43, q_lens=[3, 0, 17, 1], kv_lens=[40, 9, 200, 1], num_q_heads=8,
                 num_kv_heads=2, head_dim=64, page_size=16, extra_tokens=5, max_num_seqs=7)
    import torch

    t = to_dev(p)
    out = torch.full_like(t[0], 3.0)
    got, st = run(p, tensors=t, out=out)
    assert st == 0
    assert (got[21:] == 0).all()
    assert_close(got, oracle.forward(p), p.kv_dtype, "padding")


@pytest.mark.parametrize("kv_dtype,head_dim,q_lens", [
    ("bf16", 128, [1, 37, 5, 300]),
    ("fp8_e4m3", 256, [1, 37, 5, 130]),
])
def test_full_page_tables(kv_dtype, head_dim, q_lens):
    """Sequences whose kv_len is the largest the page table holds (pages_per_seq * page_size):
    every page slot of their row is used, the last key sits in the last slot of the last page."""
    ps = 16
    kv = [1024, 1024, 700, 1024]  # pages_per_seq = 64 from the longest
    p = ri.build(seed=45, q_lens=q_lens, kv_lens=kv, num_q_heads=16, num_kv_heads=4, head_dim=head_dim,
                 page_size=ps, kv_dtype=kv_dtype, k_scale=0.05 if kv_dtype != "bf16" else None,
                 v_scale=0.05 if kv_dtype != "bf16" else None, soft_cap=30.0, sliding_window=600)
    assert p.pages_per_seq * p.page_size == 1024
    got, st = run(p)
    assert st == 0
    assert_close(got, oracle.forward(p), p.kv_dtype, "full page tables")


def test_zero_sequences_writes_zeros():
    p = ri.build(seed=44, q_lens=[4], kv_lens=[10], num_q_heads=4, num_kv_heads=2, head_dim=64,
                 page_size=16)
    p.num_seqs = 0
    import torch

    t = to_dev(p)
    out = torch.full_like(t[0], 7.0)
    got, st = run(p, tensors=t, out=out)
    assert st == 0 and (got == 0).all()


def test_bad_page_index_sets_status():
    p = ri.random_small(45, num_seqs=3, max_q=5, max_kv=60)
    p.page_indices[1, 0] = p.total_num_pages + 5
    got, st = run(p)
    assert st == 4
    assert np.isfinite(got).all()


@pytest.mark.parametrize("mut", ["kv_too_long", "q_gt_kv", "cu_decreasing", "cu_past_T"])
def test_bad_lengths_set_status_and_zero_output(mut):
    p = ri.random_small(46, num_seqs=3, max_q=5, max_kv=60)
    if mut == "kv_too_long":
        p.kv_lens[0] = p.pages_per_seq * p.page_size + 1
    elif mut == "q_gt_kv":
        p.kv_lens[2] = int(p.cu_q_lens[3] - p.cu_q_lens[2]) - 1
    elif mut == "cu_decreasing":
        p.cu_q_lens[2] = p.cu_q_lens[1] - 1
    else:
        p.cu_q_lens[3] = p.num_q_tokens + 1
    assert oracle.validate(p) == 5
    import torch

    t = to_dev(p)
    out = torch.full_like(t[0], 5.0)
    got, st = run(p, tensors=t, out=out)
    assert st == 5 and (got == 0).all()


def test_forward_host_equals_forward():
    p = ri.random_small(47, num_seqs=6, max_q=20, max_kv=700, num_q_heads=8, num_kv_heads=2,
                        head_dim=128)
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention

    att = RaggedPagedAttention(**p.cfg_dict())
    t = to_dev(p)
    dev_out = o_to_f64(att.forward(*t, p.num_seqs))
    host = [x.cpu().pin_memory() for x in t]
    out_h = torch.empty_like(host[0]).pin_memory()
    att.forward_host(host[0], t[1], host[2], host[3], host[4], p.num_seqs, out_h)
    torch.cuda.synchronize()
    assert att.status() == 0
    assert np.array_equal(dev_out, o_to_f64(out_h))
    att.close()


def test_repeat_calls_are_deterministic():
    p = ri.random_small(48, num_seqs=10, decode_only=True, max_kv=4000, num_q_heads=32,
                        num_kv_heads=8, head_dim=128)
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention

    att = RaggedPagedAttention(**p.cfg_dict())
    t = to_dev(p)
    a = o_to_f64(att.forward(*t, p.num_seqs))
    b = o_to_f64(att.forward(*t, p.num_seqs))
    assert np.array_equal(a, b)
    att.close()


def test_bounded_wait_reports_timeout_and_context_survives():
    """The decode kernel's copy warp is told to issue nothing (the handle's test option): every
    consumer wait must expire after its bound, set RPA_ERR_TIMEOUT and return."""
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention
    from ragged_paged_attention_02_gb300.binding import RPA_OPT_TEST_STALL_PRODUCER, RPA_OPT_WAIT_TIMEOUT_MS

    p = ri.random_small(49, num_seqs=4, decode_only=True, max_kv=300, num_q_heads=8,
                        num_kv_heads=2, head_dim=128)
    att = RaggedPagedAttention(**p.cfg_dict())
    att.set_option(RPA_OPT_TEST_STALL_PRODUCER, 1)
    att.set_option(RPA_OPT_WAIT_TIMEOUT_MS, 50)
    t = to_dev(p)
    att.forward(*t, p.num_seqs)
    assert att.status() == 6
    att.set_option(RPA_OPT_TEST_STALL_PRODUCER, 0)
    att.forward(*t, p.num_seqs)  # the same handle works again once the hook is off
    assert att.status() == 0
    att.close()
    got, st = run(p, tensors=t)  # and a fresh handle on the same context
    assert st == 0
    assert_close(got, oracle.forward(p), p.kv_dtype, "after timeout")


def test_serial_option_matches_concurrent_bit_for_bit():
    """RPA_OPT_SERIAL runs decode and prefill one after the other instead of at once with an SM
    split (the decode kernel behind the prefill kernel, waiting for the planner's published
    epoch); the work items are the same, so the outputs are identical."""
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention
    from ragged_paged_attention_02_gb300.binding import RPA_OPT_SERIAL

    p = ri.random_small(50, num_seqs=20, max_q=200, max_kv=3000, num_q_heads=16, num_kv_heads=4,
                        head_dim=128)
    att = RaggedPagedAttention(**p.cfg_dict())
    t = to_dev(p)
    a = o_to_f64(att.forward(*t, p.num_seqs))
    info_a = att.plan(max_items=1)[0]
    att.set_option(RPA_OPT_SERIAL, 1)
    b = o_to_f64(att.forward(*t, p.num_seqs))
    info_b = att.plan(max_items=1)[0]
    assert att.status() == 0
    assert (info_a[15] & 1) == 1 and (info_b[15] & 1) == 0
    assert np.array_equal(a, b)
    att.close()


def _two_batches(kind):
    """Two batches of one configuration (same token count, page table shape and page count) with
    different lengths: consecutive calls rewrite what the previous call's kernels read."""
    rng = np.random.default_rng([55, 0])
    if kind == "concurrent":
        S, qmax, kmax, kw = 24, 150, 4000, dict(num_q_heads=16, num_kv_heads=4, head_dim=128, page_size=16)
    else:
        S, qmax, kmax, kw = 12, 3, 3000, dict(num_q_heads=16, num_kv_heads=1, head_dim=576, page_size=64,
                                               kv_layout="latent", v_head_dim=512, sm_scale=1 / 24)
    qa = rng.integers(1, qmax, size=S, endpoint=True)
    qb = qa[::-1].copy()
    ka = np.maximum(rng.integers(1, kmax, size=S, endpoint=True), qa)
    kb = np.maximum(rng.integers(1, kmax, size=S, endpoint=True), qb)
    ps = kw["page_size"]
    used = max(int(((ka + ps - 1) // ps).sum()), int(((kb + ps - 1) // ps).sum()))
    common = dict(pages_per_seq=(kmax + ps - 1) // ps, total_num_pages=used + 3, **kw)
    return [ri.build(seed=56, q_lens=qa, kv_lens=ka, **common), ri.build(seed=57, q_lens=qb, kv_lens=kb, **common)]


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["concurrent", "latent"])
def test_plan_early_option_back_to_back_calls(kind):
    """RPA_OPT_PLAN_EARLY lets each call's planner read its inputs while the previous call's last
    kernel still runs.  Back-to-back calls on one stream, alternating between two batches, give
    the same outputs as the default mode and the oracle."""
    import torch
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention
    from ragged_paged_attention_02_gb300.binding import RPA_OPT_PLAN_EARLY

    ps = _two_batches(kind)
    cfg = ps[0].cfg_dict()
    assert ps[1].cfg_dict() == cfg
    ts = [to_dev(p) for p in ps]
    outs = {}
    for early in (0, 1):
        att = RaggedPagedAttention(**cfg)
        att.set_option(RPA_OPT_PLAN_EARLY, early)
        res = []
        for i in range(6):  # no synchronisation between the calls
            res.append(att.forward(*ts[i % 2], ps[i % 2].num_seqs))
        torch.cuda.synchronize()
        assert att.status() == 0
        outs[early] = [o_to_f64(r) for r in res]
        att.close()
    for i in range(6):
        assert np.array_equal(outs[0][i], outs[1][i]), f"call {i}"
    for i in range(2):
        assert_close(outs[1][i], oracle.forward(ps[i]), ps[i].kv_dtype, f"{kind} batch {i}")


def _three_batches(kind):
    """Three batches of one configuration (rolled query lengths, fresh key lengths)."""
    rng = np.random.default_rng([77, 0])
    if kind == "concurrent":
        S, qmax, kmax, kw = 32, 200, 6000, dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    elif kind == "fp8":
        S, qmax, kmax, kw = 24, 64, 6000, dict(num_q_heads=16, num_kv_heads=8, head_dim=256, page_size=16,
                                               kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05, soft_cap=50.0,
                                               sliding_window=2000)
    else:
        S, qmax, kmax, kw = 24, 2, 6000, dict(num_q_heads=16, num_kv_heads=1, head_dim=576, page_size=64,
                                              kv_layout="latent", v_head_dim=512, sm_scale=1 / 24)
    base_q = rng.integers(1, qmax, size=S, endpoint=True)
    qs = [np.roll(base_q, i) for i in range(3)]
    ks = [np.maximum(rng.integers(1, kmax, size=S, endpoint=True), q) for q in qs]
    ps = kw["page_size"]
    used = max(int(((k + ps - 1) // ps).sum()) for k in ks)
    common = dict(pages_per_seq=(kmax + ps - 1) // ps, total_num_pages=used + 3, **kw)
    return [ri.build(seed=80 + i, q_lens=qs[i], kv_lens=ks[i], **common) for i in range(3)]


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["concurrent", "fp8", "latent"])
def test_back_to_back_calls_bit_equal_to_synchronised_calls(kind):
    """Forty calls in a seeded random order over three batches, with no synchronisation between
    them (each call's planner, attention kernels and merge overlapping its neighbours as the launch
    order allows, RPA_OPT_PLAN_EARLY on): every output bit-equal to a synchronised call on the same
    batch.  A race between consecutive calls would show as a mismatch."""
    import torch
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention
    from ragged_paged_attention_02_gb300.binding import RPA_OPT_PLAN_EARLY

    ps = _three_batches(kind)
    ts = [to_dev(p) for p in ps]
    att = RaggedPagedAttention(**ps[0].cfg_dict())
    att.set_option(RPA_OPT_PLAN_EARLY, 1)
    ref = []
    for i, p in enumerate(ps):
        ref.append(o_to_f64(att.forward(*ts[i], p.num_seqs)))
        torch.cuda.synchronize()
    order = [int(x) for x in np.random.default_rng([78, 0]).integers(0, 3, size=40)]
    outs = [att.forward(*ts[i], ps[i].num_seqs) for i in order]
    torch.cuda.synchronize()
    assert att.status() == 0
    for n, (o, i) in enumerate(zip(outs, order)):
        assert np.array_equal(o_to_f64(o), ref[i]), f"call {n} (batch {i})"
    att.close()
    assert_close(ref[0], oracle.forward(ps[0]), ps[0].kv_dtype, kind)


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["concurrent", "fp8", "latent"])
def test_cuda_graph_replay_bit_equal_to_eager_calls(kind):
    """One call captured into a CUDA graph over static buffers, then replayed back to back with
    each of three batches copied in first (no synchronisation between the replays): every output
    bit-equal to an eager call on the same batch.  A captured call replays its parameters, so the
    concurrent decode / prefill split must not depend on a per-call value baked into the graph."""
    import torch
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention

    ps = _three_batches(kind)
    ts = [to_dev(p) for p in ps]
    att = RaggedPagedAttention(**ps[0].cfg_dict())
    ref = []
    for i, p in enumerate(ps):
        ref.append(o_to_f64(att.forward(*ts[i], p.num_seqs)))
        torch.cuda.synchronize()
    static = [t.clone() for t in ts[0]]
    out = torch.empty_like(att.forward(*static, ps[0].num_seqs))
    torch.cuda.synchronize()
    num_seqs = ps[0].num_seqs
    assert all(p.num_seqs == num_seqs for p in ps)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        att.forward(*static, num_seqs, out=out)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        att.forward(*static, num_seqs, out=out)
    order = [int(x) for x in np.random.default_rng([79, 0]).integers(0, 3, size=12)]
    outs = []
    for i in order:
        for s, t in zip(static, ts[i]):
            s.copy_(t)
        graph.replay()
        outs.append(out.clone())
    torch.cuda.synchronize()
    assert att.status() == 0
    for n, (o, i) in enumerate(zip(outs, order)):
        assert np.array_equal(o_to_f64(o), ref[i]), f"replay {n} (batch {i})"
    del graph
    att.close()


@pytest.mark.gpu
def test_two_handles_on_two_streams_at_once():
    """Two handles (one workspace each) called on two streams with no synchronisation between
    them, each call's kernels free to share the GPU with the other handle's: every output bit-equal
    to a synchronised call, and both statuses clean.  The concurrent decode / prefill split polls
    a flag in its own handle's workspace only."""
    import torch
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention

    ps = _two_batches("concurrent")
    ts = [to_dev(p) for p in ps]
    atts = [RaggedPagedAttention(**p.cfg_dict()) for p in ps]
    ref = []
    for att, t, p in zip(atts, ts, ps):
        ref.append(o_to_f64(att.forward(*t, p.num_seqs)))
        torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = [[], []]
    for _ in range(8):
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                outs[i].append(atts[i].forward(*ts[i], ps[i].num_seqs))
    torch.cuda.synchronize()
    for i in range(2):
        assert atts[i].status() == 0
        for n, o in enumerate(outs[i]):
            assert np.array_equal(o_to_f64(o), ref[i]), f"handle {i} call {n}"
        atts[i].close()
