"""Helpers for the GPU tests: move a Problem to cuda:0, run it through the C ABI,
compare with the oracle at the stated tolerance."""
import numpy as np

import rpa_inputs as ri

TOL = {"bf16": (2e-2, 2e-2), "fp8_e4m3": (6e-2, 6e-2)}  # (abs, rel)


def to_dev(prob, dev="cuda:0"):
    import torch

    q = torch.from_numpy(prob.q.view(np.int16)).view(torch.bfloat16).to(dev)
    if prob.kv_dtype == "bf16":
        kv = torch.from_numpy(prob.kv_pages.view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        kv = torch.from_numpy(prob.kv_pages).to(dev)
    kvl = torch.from_numpy(np.ascontiguousarray(prob.kv_lens, np.int32)).to(dev)
    pi = torch.from_numpy(np.ascontiguousarray(prob.page_indices, np.int32)).to(dev)
    cu = torch.from_numpy(np.ascontiguousarray(prob.cu_q_lens, np.int32)).to(dev)
    return q, kv, kvl, pi, cu


def o_to_f64(o):
    import torch

    return ri.bf16_bits_to_f32(o.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


def run(prob, att=None, tensors=None, out=None):
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention

    own = att is None
    if own:
        att = RaggedPagedAttention(**prob.cfg_dict())
    t = tensors or to_dev(prob)
    o = att.forward(*t, prob.num_seqs, out=out)
    st = att.status()
    res = o_to_f64(o)
    if own:
        att.close()
    return res, st


def assert_close(got, ref, kv_dtype, what=""):
    atol, rtol = TOL[kv_dtype]
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())
