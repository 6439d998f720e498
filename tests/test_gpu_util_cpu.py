"""The GPU tests' helpers, run on CPU tensors: every element type goes to a tensor of the right
dtype and shape and comes back with its exact values."""
import numpy as np
import pytest

import rpa_inputs as ri
from gpu_util import TOL, o_to_f64, to_dev

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("q_dtype,kv_dtype", [("bf16", "bf16"), ("f16", "f16"), ("f32", "fp8_e4m3"),
                                              ("bf16", "fp8_e5m2"), ("f16", "int8")])
def test_to_dev_and_back_on_the_cpu(q_dtype, kv_dtype):
    extra = {} if kv_dtype in ("bf16", "f16") else dict(k_scale=0.05, v_scale=0.05)
    p = ri.random_small(5, num_seqs=3, q_dtype=q_dtype, kv_dtype=kv_dtype, sinks=True, **extra)
    q, kv, kvl, pi, cu = to_dev(p, dev="cpu")
    want_q = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[q_dtype]
    assert q.dtype == want_q and tuple(q.shape) == p.q.shape
    assert kv.element_size() == ri.KV_ELT[kv_dtype] and tuple(kv.shape) == p.kv_pages.shape
    assert kvl.dtype == pi.dtype == cu.dtype == torch.int32
    assert np.array_equal(o_to_f64(q), ri.values_f64(p.q, q_dtype))
    assert kv_dtype in TOL
