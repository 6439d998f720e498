"""The product path and the oracle stay apart, and the product fails loudly without its library
or a GPU (there is no CPU or PyTorch fallback)."""
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "ragged_paged_attention_02_gb300")


def _sources(*patterns):
    out = []
    for pat in patterns:
        out += glob.glob(os.path.join(ROOT, pat), recursive=True)
    return sorted(out)


def test_product_sources_never_reach_the_oracle():
    files = _sources("ragged_paged_attention_02_gb300/**/*.py", "ragged_paged_attention_02_gb300/**/*.cu",
                     "ragged_paged_attention_02_gb300/**/*.cuh", "include/*.h")
    assert files
    for f in files:
        src = open(f).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
        assert not re.search(r"#\s*include\s*[<\"][^>\"]*oracle", src), f
        assert "librpa_oracle" not in src and "rpa_oracle" not in src, f


def test_oracle_includes_only_system_headers():
    src = open(os.path.join(ROOT, "oracle", "rpa_oracle.c")).read()
    for inc in re.findall(r"#\s*include\s*([<\"][^>\"]+[>\"])", src):
        assert inc.startswith("<"), inc  # nothing of the CUDA tree (rpa.h, rpa_internal.cuh, ...)
    py = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert not re.search(r"^\s*(import|from)\s+ragged_paged_attention_02_gb300\b", py, re.M)


def test_missing_library_raises(monkeypatch):
    from ragged_paged_attention_02_gb300 import _build, binding

    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(_build, "LIB", os.path.join(ROOT, "no_such_dir", "librpa.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.lib()


def test_no_gpu_means_an_error_not_a_fallback():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import __graft_entry__
    import rpa_inputs as ri
    from ragged_paged_attention_02_gb300 import RaggedPagedAttention
    from ragged_paged_attention_02_gb300.binding import RpaError

    __graft_entry__.build()
    p = ri.workload("tiny")
    with pytest.raises((RpaError, RuntimeError)):
        RaggedPagedAttention(**p.cfg_dict())


def test_kernels_use_no_trap_or_closed_copy_calls():
    """Failures are reported through the status word, never by trapping the GPU; the batched
    memcpy calls that faulted GPUs of this class are not used (nor named)."""
    files = _sources("ragged_paged_attention_02_gb300/**/*.cu", "ragged_paged_attention_02_gb300/**/*.cuh",
                     "include/*.h", "ragged_paged_attention_02_gb300/**/*.py", "bench.py", "__graft_entry__.py")
    closed = ["Memcpy" + "BatchAsync", "Memcpy3D" + "BatchAsync"]
    for f in files:
        src = open(f).read()
        assert "__trap" not in src and not re.search(r"\btrap\s*;", src), f
        assert not re.search(r"(?<![A-Za-z_])assert\s*\(", src) or f.endswith(".py"), f
        for name in closed:
            assert name not in src, (f, name)
