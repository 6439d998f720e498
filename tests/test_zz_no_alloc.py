"""rpa_forward_noalloc: the forward call for callers that cannot allocate.

Serving engines that give all device memory to their own arena allocator, or
that may not call cudaMalloc/cudaFree (an implicit device synchronisation)
where attention runs, call this entry point instead of rpa_create +
rpa_forward.  Its workspace is a fixed 32 MiB array inside the library.  This
test calls it through the C ABI, twice in a row per case, and checks each
output against the fp64 oracle and against the handle-based rpa_forward, at
the tolerance of the other parity tests.  The cases reach every kernel branch
of the entry point: the bf16 tensor-memory prefill, the 64-key-tile kernel
(fp8, and bf16 at D 256), the latent kernel, 8- and 16-row decode tiles and
split-KV pieces.  An oversized configuration is refused.
"""
import ctypes

import numpy as np
import pytest

import rpa_inputs as ri

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _noalloc(prob, t, out):
    import ragged_paged_attention_02_gb300 as rpa

    cfg = prob.cfg_dict()
    if cfg.get("sinks") is not None:
        cfg["sinks"] = torch.from_numpy(cfg["sinks"]).cuda()  # kept alive in cfg until the call returns
    c = rpa.make_cfg(**cfg)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    q, kv, kvl, pi, cu = t
    return rpa.lib().rpa_forward_noalloc(ctypes.byref(c), q.data_ptr(), kv.data_ptr(), kvl.data_ptr(),
                                         pi.data_ptr(), cu.data_ptr(), int(prob.num_seqs),
                                         out.data_ptr(), stream)


CASES = {
    "tiny": None,
    # 8-row decode tiles, long keys split into pieces (combine kernel)
    "split_decode": (60, dict(num_seqs=12, decode_only=True, max_kv=6000, num_q_heads=32, num_kv_heads=8,
                              head_dim=128)),
    # fp8 K/V at D 256: the fp8 tensor-memory prefill (decode rows as its items too)
    "fp8_mixed": (61, dict(num_seqs=8, max_q=80, max_kv=900, num_q_heads=16, num_kv_heads=8, head_dim=256,
                           kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05, soft_cap=50.0,
                           sliding_window=300, sm_scale=1 / 16)),
    # bf16 at D 256: the 64-key-tile kernel in direct mode
    "bf16_d256": (62, dict(num_seqs=6, max_q=70, max_kv=800, num_q_heads=8, num_kv_heads=4, head_dim=256,
                           soft_cap=30.0, sm_scale=1 / 16)),
    # bf16 with G = 16: 16-row decode tiles beside the bf16 tensor-memory prefill
    "bf16_g16": (63, dict(num_seqs=10, max_q=30, max_kv=3000, num_q_heads=32, num_kv_heads=2, head_dim=128)),
    # attention sinks read through the cfg's device pointer
    "sinks": (64, dict(num_seqs=9, max_q=60, max_kv=4000, num_q_heads=16, num_kv_heads=4, head_dim=128,
                       sinks=True)),
    # latent attention: the latent kernel, split pieces of 512-wide partials
    "latent": (66, dict(num_seqs=8, max_q=4, max_kv=3000, num_q_heads=16, num_kv_heads=1, page_size=64,
                        kv_layout="latent", head_dim=576, v_head_dim=512, sm_scale=1 / 24)),
    # f32 q rounded into the fixed array before the kernels read it; e5m2 K/V; f32 o
    "f32_q_e5m2": (65, dict(num_seqs=8, max_q=40, max_kv=3000, num_q_heads=16, num_kv_heads=8, head_dim=256,
                            q_dtype="f32", kv_dtype="fp8_e5m2", k_scale=0.05, v_scale=0.05, sm_scale=1 / 16)),
    # int8 K/V at D 64: the 64-key-tile kernel with one column block a row, decode rows split into pieces
    "int8_d64": (67, dict(num_seqs=9, max_q=30, max_kv=4000, num_q_heads=8, num_kv_heads=2, head_dim=64,
                          page_size=16, kv_dtype="int8", k_scale=0.04, v_scale=0.04)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_oracle_and_rpa_forward_twice(name):
    import oracle
    from gpu_util import assert_close, o_to_f64, to_dev

    from ragged_paged_attention_02_gb300 import RaggedPagedAttention

    case = CASES[name]
    p = ri.workload("tiny") if case is None else ri.random_small(case[0], **case[1])
    want = oracle.forward(p)
    t = to_dev(p)
    att = RaggedPagedAttention(**p.cfg_dict())
    ref = o_to_f64(att.forward(*t, p.num_seqs))
    assert att.status() == 0
    att.close()
    for _ in range(2):
        out = t[0].new_full((p.num_q_tokens, p.num_q_heads, p.out_dim), 9.0)
        assert _noalloc(p, t, out) == 0
        torch.cuda.synchronize()
        got = o_to_f64(out)
        assert_close(got, want, p.kv_dtype, f"noalloc {name} vs oracle")
        assert_close(got, ref, p.kv_dtype, f"noalloc {name} vs rpa_forward")


def test_noalloc_rejects_oversized_workspace():
    import ragged_paged_attention_02_gb300 as rpa

    p = ri.workload("tiny")
    cfg = p.cfg_dict()
    cfg["max_num_seqs"] = 1 << 21  # work-item lists alone need far more than 32 MiB
    c = rpa.make_cfg(**cfg)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    r = rpa.lib().rpa_forward_noalloc(ctypes.byref(c), dummy.data_ptr(), dummy.data_ptr(),
                                      dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), 1,
                                      dummy.data_ptr(), None)
    assert r == rpa.RPA_ERR_NO_ALLOC_LIMIT
