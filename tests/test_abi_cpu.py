"""C-ABI checks that need no GPU: the library loads, exports every entry point
declared in include/rpa.h, and rejects bad configurations on the host."""
import os
import re

import pytest

import ragged_paged_attention_02_gb300 as rpa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__

    __graft_entry__.build()
    return rpa.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "rpa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rpa_[a-z_]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert header_functions() == sorted(rpa.EXPORTS)


def test_library_exports_every_header_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), name
    assert L.rpa_version() == 200


def test_strerror_covers_codes(L):
    for code in range(8):
        assert L.rpa_strerror(code).decode() != "unknown status code"


BASE = dict(num_q_tokens=22, num_q_heads=4, num_kv_heads=2, head_dim=64, total_num_pages=16,
            page_size=16, max_num_seqs=3, pages_per_seq=4, sm_scale=0.125)


@pytest.mark.parametrize("change,code", [
    ({}, rpa.RPA_OK),
    (dict(num_q_heads=6, num_kv_heads=4), rpa.RPA_ERR_UNSUPPORTED),
    (dict(head_dim=96), rpa.RPA_ERR_UNSUPPORTED),
    (dict(num_q_heads=130, num_kv_heads=1), rpa.RPA_ERR_UNSUPPORTED),
    (dict(mask_value=-1.0), rpa.RPA_ERR_UNSUPPORTED),
    (dict(page_size=0), rpa.RPA_ERR_INVALID_ARG),
    (dict(total_num_pages=0), rpa.RPA_ERR_INVALID_ARG),
    (dict(num_q_tokens=-1), rpa.RPA_ERR_INVALID_ARG),
    (dict(sliding_window=0), rpa.RPA_ERR_INVALID_ARG),
    (dict(soft_cap=-3.0), rpa.RPA_ERR_INVALID_ARG),
    (dict(sm_scale=float("nan")), rpa.RPA_ERR_INVALID_ARG),
    (dict(kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05), rpa.RPA_OK),
    (dict(pages_per_seq=1 << 20, page_size=1 << 12), rpa.RPA_ERR_INVALID_ARG),
    (dict(page_size=6), rpa.RPA_ERR_UNSUPPORTED),  # page runs of the gather are >= 4 slots
    (dict(page_size=4, pages_per_seq=16), rpa.RPA_OK),
    (dict(head_dim=256, num_q_heads=16, num_kv_heads=8), rpa.RPA_OK),
    # element types: f16 / f32 q, f16 / e5m2 / int8 K/V
    (dict(q_dtype="f16", kv_dtype="f16"), rpa.RPA_OK),
    (dict(q_dtype="f32", kv_dtype="fp8_e5m2", k_scale=0.05, v_scale=0.05), rpa.RPA_OK),
    (dict(q_dtype="f16", kv_dtype="int8", k_scale=0.04, v_scale=0.04), rpa.RPA_OK),
    # latent layout: 576 / 512 rows only, 2-byte rows, pages of a multiple of 8, blocks of 16 heads
    (dict(kv_layout="latent", head_dim=576, v_head_dim=512, num_q_heads=16, num_kv_heads=1, page_size=64), rpa.RPA_OK),
    (dict(kv_layout="latent", head_dim=576, v_head_dim=512, num_q_heads=128, num_kv_heads=1, page_size=16), rpa.RPA_OK),
    (dict(kv_layout="latent", head_dim=576, v_head_dim=512, num_q_heads=24, num_kv_heads=1, page_size=16),
     rpa.RPA_ERR_UNSUPPORTED),
    (dict(kv_layout="latent", head_dim=576, v_head_dim=512, num_q_heads=16, num_kv_heads=1, page_size=4),
     rpa.RPA_ERR_UNSUPPORTED),
    (dict(kv_layout="latent", head_dim=512, v_head_dim=512, num_q_heads=16, num_kv_heads=1, page_size=16),
     rpa.RPA_ERR_UNSUPPORTED),
    (dict(kv_layout="latent", head_dim=576, v_head_dim=512, num_q_heads=16, num_kv_heads=1, page_size=16,
          kv_dtype="fp8_e4m3"), rpa.RPA_ERR_UNSUPPORTED),
    (dict(v_head_dim=32), rpa.RPA_ERR_UNSUPPORTED),  # the split layout's V is head_dim wide
])
def test_validate_cfg(L, change, code):
    cfg = dict(BASE)
    cfg.update(change)
    assert rpa.validate_cfg(**cfg) == code


def test_null_handle_and_create_out(L):
    import ctypes

    assert L.rpa_forward(None, None, None, None, None, None, 0, None, None) == rpa.RPA_ERR_INVALID_ARG
    assert L.rpa_get_status(None, None) == rpa.RPA_ERR_INVALID_ARG
    assert L.rpa_set_option(None, rpa.RPA_OPT_SERIAL, 1) == rpa.RPA_ERR_INVALID_ARG
    c = rpa.make_cfg(**BASE)
    assert L.rpa_create(ctypes.byref(c), None) == rpa.RPA_ERR_INVALID_ARG
    bad = rpa.make_cfg(**dict(BASE, head_dim=80))
    h = ctypes.c_void_p(1)
    assert L.rpa_create(ctypes.byref(bad), ctypes.byref(h)) == rpa.RPA_ERR_UNSUPPORTED
    assert not h.value
    L.rpa_destroy(None)


def test_cfg_init_defaults_keep_the_shape(L):
    """rpa_cfg_init keeps the shape fields and sets the page's defaults for the rest."""
    import ctypes
    import math

    from ragged_paged_attention_02_gb300.binding import RPA_DT_BF16, RpaCfg

    c = RpaCfg()
    c.num_q_tokens, c.num_q_heads, c.num_kv_heads, c.head_dim = 22, 4, 2, 64
    c.total_num_pages, c.page_size, c.max_num_seqs, c.pages_per_seq = 16, 16, 3, 4
    c.is_causal, c.soft_cap, c.reserved = 0, 9.0, 5
    L.rpa_cfg_init(ctypes.byref(c))
    assert (c.num_q_tokens, c.num_q_heads, c.num_kv_heads, c.head_dim) == (22, 4, 2, 64)
    assert (c.total_num_pages, c.page_size, c.max_num_seqs, c.pages_per_seq) == (16, 16, 3, 4)
    assert c.q_dtype == RPA_DT_BF16 and c.kv_dtype == RPA_DT_BF16
    assert math.isclose(c.sm_scale, 1 / 8, rel_tol=1e-7)
    assert math.isclose(c.mask_value, -2.38197633e38, rel_tol=1e-7)
    assert c.is_causal == 1 and c.reserved == 0
    assert (c.has_soft_cap, c.has_k_scale, c.has_v_scale, c.has_sliding_window) == (0, 0, 0, 0)
    assert L.rpa_validate_cfg(ctypes.byref(c)) == rpa.RPA_OK


def test_dtypes_the_library_refuses(L):
    """K/V in f32 / i32 / i16 (the page's other packings) and q in 8-bit types are refused."""
    import ctypes

    for kv, q in ((rpa.RPA_DT_F32, rpa.RPA_DT_BF16), (7, rpa.RPA_DT_BF16), (rpa.RPA_DT_BF16, rpa.RPA_DT_FP8_E4M3),
                  (rpa.RPA_DT_BF16, rpa.RPA_DT_INT8)):
        c = rpa.make_cfg(**BASE)
        c.kv_dtype, c.q_dtype = kv, q
        assert L.rpa_validate_cfg(ctypes.byref(c)) == rpa.RPA_ERR_UNSUPPORTED, (kv, q)


def test_sinks_need_an_aligned_pointer(L):
    import ctypes

    c = rpa.make_cfg(**BASE)
    c.has_sinks, c.sinks = 1, None
    assert L.rpa_validate_cfg(ctypes.byref(c)) == rpa.RPA_ERR_INVALID_ARG
    c.sinks = 4098  # not 4-byte aligned
    assert L.rpa_validate_cfg(ctypes.byref(c)) == rpa.RPA_ERR_INVALID_ARG
    c.sinks = 4096
    assert L.rpa_validate_cfg(ctypes.byref(c)) == rpa.RPA_OK
    c.reserved = 1
    assert L.rpa_validate_cfg(ctypes.byref(c)) == rpa.RPA_ERR_INVALID_ARG
