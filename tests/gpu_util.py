"""Helpers for the GPU tests: move a Problem to cuda:0, run it through the C ABI,
compare with the oracle at the stated tolerance."""
import numpy as np

import rpa_inputs as ri

# (abs, rel) by K/V element type: the stated tolerance for bf16 K/V, and for fp8 K/V; f16 K/V
# take the 16-bit one, e5m2 and int8 the 8-bit one
TOL = {"bf16": (2e-2, 2e-2), "f16": (2e-2, 2e-2), "fp8_e4m3": (6e-2, 6e-2), "fp8_e5m2": (6e-2, 6e-2),
       "int8": (6e-2, 6e-2)}


def _torch_view(a, dtype):
    import torch

    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    if dtype == "f16":
        return torch.from_numpy(a.view(np.int16)).view(torch.float16)
    return torch.from_numpy(a)  # float32, uint8 (fp8 bytes) or int8


def to_dev(prob, dev="cuda:0"):
    import torch

    q = _torch_view(prob.q, getattr(prob, "q_dtype", "bf16")).to(dev)
    kv = _torch_view(prob.kv_pages, prob.kv_dtype).to(dev)
    kvl = torch.from_numpy(np.ascontiguousarray(prob.kv_lens, np.int32)).to(dev)
    pi = torch.from_numpy(np.ascontiguousarray(prob.page_indices, np.int32)).to(dev)
    cu = torch.from_numpy(np.ascontiguousarray(prob.cu_q_lens, np.int32)).to(dev)
    return q, kv, kvl, pi, cu


def o_to_f64(o):
    import torch

    if o.dtype == torch.float32:
        return o.cpu().numpy().astype(np.float64)
    bits = o.view(torch.int16).cpu().numpy().view(np.uint16)
    return ri.values_f64(bits, "f16" if o.dtype == torch.float16 else "bf16")


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
