"""fp64 CPU oracle for ragged paged attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and shares no code with
it.

The arithmetic lives in ``rpa_oracle.c`` (plain C, fp64, one output row at a
time); this module compiles it with gcc and marshals numpy arrays.  Every
function of the C file follows the "ragged_paged.zig" page, sections
``flashAttention`` (mask, softcap, online softmax, PV) and ``run`` (sequence
walk, GQA head mapping, dequant); see the C file's header for the readings.

Attention sinks follow the "from_qwen_ops.rs" page (flat_softmax_rows_at,
``sinks``): one extra logit per query head that starts the row maximum and
joins the denominator with no value.  Latent attention (the same page, "The
latent-attention family at whole-tile widths") reads a paged latent cache of
one row per kv head: K is the row, V its first v_head_dim elements.

Parity pins (tests/test_oracle_pins.py): brute-force dense attention on tiny
unpaged inputs (fixed and random configurations, with and without sinks),
closed forms (uniform V, single allowed key, one-key sequences, zero-query
means over the allowed keys, two-key weights, zero-query means shrunk by a
sink), the softcap identity of the "from_qwen_ops.rs" page
(``capped``), format decoders checked code by code, and the invariants of page
placement, decode-vs-prefill, tail poisoning, sequence order, GQA repetition
and fp8 scale folding.  tests/test_oracle_mutations.py plants slips in a copy
of the C source and checks that the pins catch each.  No function is left
with its parity unpinned.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rpa_oracle.c")
_LIB = os.path.join(_HERE, "librpa_oracle.so")
_lock = threading.Lock()
_lib = None


class OracleCfg(ctypes.Structure):
    _fields_ = [
        ("num_q_tokens", ctypes.c_int64), ("num_q_heads", ctypes.c_int64),
        ("num_kv_heads", ctypes.c_int64), ("head_dim", ctypes.c_int64),
        ("total_num_pages", ctypes.c_int64), ("page_size", ctypes.c_int64),
        ("max_num_seqs", ctypes.c_int64), ("pages_per_seq", ctypes.c_int64),
        ("kv_dtype", ctypes.c_int32), ("is_causal", ctypes.c_int32),
        ("sm_scale", ctypes.c_double),
        ("has_soft_cap", ctypes.c_int32), ("has_k_scale", ctypes.c_int32),
        ("soft_cap", ctypes.c_double), ("k_scale", ctypes.c_double),
        ("has_v_scale", ctypes.c_int32), ("has_sliding_window", ctypes.c_int32),
        ("v_scale", ctypes.c_double), ("sliding_window", ctypes.c_int64),
        ("has_sinks", ctypes.c_int32), ("sinks", ctypes.c_void_p),
        ("q_dtype", ctypes.c_int32), ("latent", ctypes.c_int32), ("v_head_dim", ctypes.c_int64),
    ]

# the oracle's own type codes (rpa_oracle.c: OracleKv, OracleQ)
KV_CODES = {"bf16": 0, "fp8_e4m3": 1, "f16": 2, "fp8_e5m2": 3, "int8": 4}
Q_CODES = {"bf16": 0, "f16": 1, "f32": 2}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (host code only; no CUDA)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                                   "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        p = ctypes.c_void_p
        lib.rpa_oracle_forward.argtypes = [ctypes.POINTER(OracleCfg), p, p, p, p, p,
                                           ctypes.c_int32, p, ctypes.c_int]
        lib.rpa_oracle_forward.restype = ctypes.c_int
        lib.rpa_oracle_rows.argtypes = [ctypes.POINTER(OracleCfg), p, p, p, p, p, ctypes.c_int32,
                                        p, ctypes.c_int64, p, ctypes.c_int]
        lib.rpa_oracle_rows.restype = ctypes.c_int
        lib.rpa_oracle_validate.argtypes = [ctypes.POINTER(OracleCfg), p, p, p, ctypes.c_int32]
        lib.rpa_oracle_validate.restype = ctypes.c_int
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_e5m2_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e5m2_to_f64.restype = ctypes.c_double
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        _lib = lib
    return _lib


def make_cfg(cfg: dict) -> OracleCfg:
    c = OracleCfg()
    for k in ("num_q_tokens", "num_q_heads", "num_kv_heads", "head_dim", "total_num_pages",
              "page_size", "max_num_seqs", "pages_per_seq"):
        setattr(c, k, int(cfg[k]))
    c.kv_dtype = KV_CODES[cfg.get("kv_dtype", "bf16")]
    c.q_dtype = Q_CODES[cfg.get("q_dtype", "bf16")]
    c.latent = 1 if cfg.get("kv_layout", "split") == "latent" else 0
    c.v_head_dim = int(cfg.get("v_head_dim") or cfg["head_dim"])
    c.is_causal = 1 if cfg.get("is_causal", True) else 0
    c.sm_scale = float(cfg["sm_scale"])
    for name in ("soft_cap", "k_scale", "v_scale"):
        v = cfg.get(name)
        setattr(c, "has_" + name, 0 if v is None else 1)
        setattr(c, name, 0.0 if v is None else float(v))
    sw = cfg.get("sliding_window")
    c.has_sliding_window = 0 if sw is None else 1
    c.sliding_window = 0 if sw is None else int(sw)
    sinks = cfg.get("sinks")
    c.has_sinks = 0 if sinks is None else 1
    if sinks is not None:
        # the fp32 values the library reads, widened exactly; kept alive with the structure
        arr = np.ascontiguousarray(np.asarray(sinks, dtype=np.float32).astype(np.float64))
        assert arr.shape == (int(cfg["num_q_heads"]),)
        c._sinks_keep = arr
        c.sinks = arr.ctypes.data
    return c


def _arrays(prob):
    q = np.ascontiguousarray(prob.q)
    assert q.dtype == (np.float32 if getattr(prob, "q_dtype", "bf16") == "f32" else np.uint16)
    kv = np.ascontiguousarray(prob.kv_pages)
    kvl = np.ascontiguousarray(prob.kv_lens, dtype=np.int32)
    pi = np.ascontiguousarray(prob.page_indices, dtype=np.int32)
    cu = np.ascontiguousarray(prob.cu_q_lens, dtype=np.int32)
    return q, kv, kvl, pi, cu


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle rejected the inputs (code {code})")
        self.code = code


def forward(prob, nthreads: int = 0, return_threads: bool = False):
    """All rows of ``o`` as float64 [num_q_tokens, num_q_heads, v_head_dim]."""
    lib = _load()
    c = make_cfg(prob.cfg_dict())
    q, kv, kvl, pi, cu = _arrays(prob)
    out = np.zeros((prob.num_q_tokens, prob.num_q_heads, prob.out_dim), dtype=np.float64)
    r = lib.rpa_oracle_forward(ctypes.byref(c), _ptr(q), _ptr(kv), _ptr(kvl), _ptr(pi), _ptr(cu),
                               int(prob.num_seqs), _ptr(out), int(nthreads))
    if r < 0:
        raise OracleError(-r)
    return (out, r) if return_threads else out


def rows(prob, rows_th: np.ndarray, nthreads: int = 0, return_threads: bool = False):
    """Selected rows: ``rows_th`` int64 [n, 2] of (token, q head); returns [n, v_head_dim]."""
    lib = _load()
    c = make_cfg(prob.cfg_dict())
    q, kv, kvl, pi, cu = _arrays(prob)
    rr = np.ascontiguousarray(rows_th, dtype=np.int64).reshape(-1, 2)
    out = np.zeros((rr.shape[0], prob.out_dim), dtype=np.float64)
    r = lib.rpa_oracle_rows(ctypes.byref(c), _ptr(q), _ptr(kv), _ptr(kvl), _ptr(pi), _ptr(cu),
                            int(prob.num_seqs), _ptr(rr), int(rr.shape[0]), _ptr(out), int(nthreads))
    if r < 0:
        raise OracleError(-r)
    return (out, r) if return_threads else out


def validate(prob) -> int:
    """0 if the lengths and page table are valid, 5 for bad lengths, 4 for a bad page id."""
    lib = _load()
    c = make_cfg(prob.cfg_dict())
    _, _, kvl, pi, cu = _arrays(prob)
    return int(lib.rpa_oracle_validate(ctypes.byref(c), _ptr(kvl), _ptr(pi), _ptr(cu),
                                       int(prob.num_seqs)))


def decode_bf16(bits: int) -> float:
    return float(_load().oracle_bf16_to_f64(int(bits)))


def decode_e4m3(byte: int) -> float:
    return float(_load().oracle_e4m3_to_f64(int(byte)))


def decode_e5m2(byte: int) -> float:
    return float(_load().oracle_e5m2_to_f64(int(byte)))


def decode_f16(bits: int) -> float:
    return float(_load().oracle_f16_to_f64(int(bits)))
