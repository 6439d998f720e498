"""Thin ctypes binding over librpa.so (include/rpa.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch supplies device memory and the current stream.  If the
library has not been built, every entry point raises -- there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

MASK_VALUE = -2.38197633e38

RPA_OK = 0
RPA_ERR_INVALID_ARG = 1
RPA_ERR_UNSUPPORTED = 2
RPA_ERR_CUDA = 3
RPA_ERR_BAD_PAGE_INDEX = 4
RPA_ERR_BAD_LENGTHS = 5
RPA_ERR_TIMEOUT = 6
RPA_ERR_NO_ALLOC_LIMIT = 7
RPA_DT_BF16 = 0
RPA_DT_FP8_E4M3 = 1
RPA_DT_F16 = 2
RPA_DT_F32 = 3
RPA_DT_FP8_E5M2 = 4
RPA_DT_INT8 = 5
RPA_KV_SPLIT = 0
RPA_KV_LATENT = 1
KV_LAYOUTS = {"split": RPA_KV_SPLIT, "latent": RPA_KV_LATENT}
# dtype names of the configuration (q / o, and kv_pages)
Q_DTYPES = {"bf16": RPA_DT_BF16, "f16": RPA_DT_F16, "f32": RPA_DT_F32}
KV_DTYPES = {"bf16": RPA_DT_BF16, "f16": RPA_DT_F16, "fp8_e4m3": RPA_DT_FP8_E4M3, "fp8_e5m2": RPA_DT_FP8_E5M2,
             "int8": RPA_DT_INT8}

# every entry point declared in include/rpa.h
EXPORTS = ("rpa_cfg_init", "rpa_validate_cfg", "rpa_create", "rpa_forward", "rpa_forward_host",
           "rpa_get_status", "rpa_read_plan", "rpa_profile_begin", "rpa_profile_read", "rpa_set_option",
           "rpa_forward_noalloc", "rpa_destroy", "rpa_strerror", "rpa_version")

RPA_OPT_WAIT_TIMEOUT_MS = 1
RPA_OPT_SERIAL = 2
RPA_OPT_PREFILL_SMS = 3
RPA_OPT_DECODE_SMS = 4
RPA_OPT_PLAN_EARLY = 5
RPA_OPT_TEST_STALL_PRODUCER = 100


class RpaCfg(ctypes.Structure):
    _fields_ = [
        ("num_q_tokens", ctypes.c_int64), ("num_q_heads", ctypes.c_int64),
        ("num_kv_heads", ctypes.c_int64), ("head_dim", ctypes.c_int64),
        ("total_num_pages", ctypes.c_int64), ("page_size", ctypes.c_int64),
        ("max_num_seqs", ctypes.c_int64), ("pages_per_seq", ctypes.c_int64),
        ("sliding_window", ctypes.c_int64),
        ("q_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
        ("sm_scale", ctypes.c_float), ("mask_value", ctypes.c_float),
        ("soft_cap", ctypes.c_float), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
        ("has_soft_cap", ctypes.c_int32), ("has_k_scale", ctypes.c_int32),
        ("has_v_scale", ctypes.c_int32), ("is_causal", ctypes.c_int32),
        ("has_sliding_window", ctypes.c_int32), ("has_sinks", ctypes.c_int32),
        ("kv_layout", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("v_head_dim", ctypes.c_int64), ("sinks", ctypes.c_void_p),
    ]


class RpaError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = lib().rpa_strerror(code).decode() if _lib is not None else str(code)
        super().__init__(f"{where}: {msg} (code {code})")
        self.code = code


_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """Load librpa.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"librpa.so not built ({path}); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.rpa_cfg_init.argtypes = [ctypes.POINTER(RpaCfg)]
        L.rpa_cfg_init.restype = None
        L.rpa_validate_cfg.argtypes = [ctypes.POINTER(RpaCfg)]
        L.rpa_validate_cfg.restype = ctypes.c_int
        L.rpa_create.argtypes = [ctypes.POINTER(RpaCfg), ctypes.POINTER(vp)]
        L.rpa_create.restype = ctypes.c_int
        L.rpa_forward.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp]
        L.rpa_forward.restype = ctypes.c_int
        L.rpa_forward_host.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp]
        L.rpa_forward_host.restype = ctypes.c_int
        L.rpa_get_status.argtypes = [vp, vp]
        L.rpa_get_status.restype = ctypes.c_int
        L.rpa_read_plan.argtypes = [vp, vp, vp, i64, vp]
        L.rpa_read_plan.restype = ctypes.c_int
        L.rpa_profile_begin.argtypes = [vp, i32]
        L.rpa_profile_begin.restype = ctypes.c_int
        L.rpa_profile_read.argtypes = [vp, vp, i32, vp]
        L.rpa_profile_read.restype = ctypes.c_int
        L.rpa_set_option.argtypes = [vp, i32, i64]
        L.rpa_set_option.restype = ctypes.c_int
        L.rpa_forward_noalloc.argtypes = [ctypes.POINTER(RpaCfg), vp, vp, vp, vp, vp, i32, vp, vp]
        L.rpa_forward_noalloc.restype = ctypes.c_int
        L.rpa_destroy.argtypes = [vp]
        L.rpa_destroy.restype = None
        L.rpa_strerror.argtypes = [ctypes.c_int]
        L.rpa_strerror.restype = ctypes.c_char_p
        L.rpa_version.argtypes = []
        L.rpa_version.restype = ctypes.c_int
        _lib = L
    return _lib


def _sinks_pointer(sinks, host_ok):
    """Device address of a float32 [Hq] sink tensor (a torch CUDA tensor, or an int address).
    A host (numpy) array is taken only where nothing is dereferenced (host-side validation)."""
    if sinks is None:
        return None
    if isinstance(sinks, int):
        return sinks
    if isinstance(sinks, np.ndarray):
        if not host_ok:
            raise ValueError("sinks must be a CUDA float32 tensor (RaggedPagedAttention converts numpy arrays)")
        return sinks.ctypes.data
    import torch

    if not (sinks.is_cuda and sinks.dtype == torch.float32 and sinks.is_contiguous()):
        raise ValueError("sinks must be a contiguous CUDA float32 tensor [num_q_heads]")
    return sinks.data_ptr()


def make_cfg(*, num_q_tokens, num_q_heads, num_kv_heads, head_dim, total_num_pages, page_size,
             max_num_seqs, pages_per_seq, sm_scale, kv_dtype="bf16", soft_cap=None, k_scale=None,
             v_scale=None, is_causal=True, sliding_window=None, mask_value=MASK_VALUE, sinks=None,
             q_dtype="bf16", kv_layout="split", v_head_dim=None, _host_ok=False, **_ignored) -> RpaCfg:
    c = RpaCfg()
    c.num_q_tokens, c.num_q_heads, c.num_kv_heads = int(num_q_tokens), int(num_q_heads), int(num_kv_heads)
    c.head_dim, c.total_num_pages, c.page_size = int(head_dim), int(total_num_pages), int(page_size)
    c.max_num_seqs, c.pages_per_seq = int(max_num_seqs), int(pages_per_seq)
    lib().rpa_cfg_init(ctypes.byref(c))
    c.kv_dtype = KV_DTYPES[kv_dtype]
    c.q_dtype = Q_DTYPES[q_dtype]
    c.sm_scale = float(sm_scale)
    c.mask_value = float(mask_value)
    c.has_soft_cap, c.soft_cap = (0, 0.0) if soft_cap is None else (1, float(soft_cap))
    c.has_k_scale, c.k_scale = (0, 1.0) if k_scale is None else (1, float(k_scale))
    c.has_v_scale, c.v_scale = (0, 1.0) if v_scale is None else (1, float(v_scale))
    c.is_causal = 1 if is_causal else 0
    c.has_sliding_window, c.sliding_window = (0, 0) if sliding_window is None else (1, int(sliding_window))
    ptr = _sinks_pointer(sinks, _host_ok)
    c.has_sinks, c.sinks = (0, None) if ptr is None else (1, ptr)
    c.kv_layout = KV_LAYOUTS[kv_layout]
    c.v_head_dim = 0 if v_head_dim is None else int(v_head_dim)
    return c


def validate_cfg(**cfg) -> int:
    """Host-only configuration check (no CUDA call): returns the status code."""
    c = make_cfg(_host_ok=True, **cfg)
    return int(lib().rpa_validate_cfg(ctypes.byref(c)))


def _stream_ptr(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class RaggedPagedAttention:
    """One configuration (shapes and knobs); owns the library workspace.

    ``forward`` takes CUDA tensors:
      q            [num_q_tokens, Hq, D] bfloat16, float16 or float32 (q_dtype)
      kv_pages     [total_num_pages, page_size, 2*Hkv, D] bfloat16 / float16, or
                   one-byte elements for fp8 (e4m3, e5m2) and int8 K/V
                   ([total_num_pages, page_size, Hkv, D] for kv_layout="latent")
      kv_lens      [max_num_seqs] int32
      page_indices [max_num_seqs, pages_per_seq] int32
      cu_q_lens    [max_num_seqs + 1] int32
    and returns o [num_q_tokens, Hq, Dv] of q's dtype (Dv = D, or v_head_dim for
    kv_layout="latent").  ``sinks`` (optional) is a
    float32 [Hq] array or CUDA tensor of attention-sink logits.
    """

    def __init__(self, **cfg):
        self.cfg = dict(cfg)
        sinks = cfg.get("sinks")
        if isinstance(sinks, np.ndarray):
            import torch

            # the library reads the sinks on the device at every call: keep them there, alive
            cfg["sinks"] = torch.from_numpy(np.ascontiguousarray(sinks, np.float32)).cuda()
        self._sinks = cfg.get("sinks")
        self._c = make_cfg(**cfg)
        h = ctypes.c_void_p()
        r = lib().rpa_create(ctypes.byref(self._c), ctypes.byref(h))
        if r != RPA_OK:
            raise RpaError(r, "rpa_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().rpa_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, q, kv_pages, kv_lens, page_indices, cu_q_lens, out):
        import torch

        c = self._c
        T, Hq, D = c.num_q_tokens, c.num_q_heads, c.head_dim
        qt = {RPA_DT_BF16: torch.bfloat16, RPA_DT_F16: torch.float16, RPA_DT_F32: torch.float32}[c.q_dtype]
        if q.dtype != qt or tuple(q.shape) != (T, Hq, D) or not q.is_contiguous():
            raise ValueError(f"q must be a contiguous {qt} tensor [num_q_tokens, Hq, D]")
        Dv = self.out_dim
        if out.dtype != qt or tuple(out.shape) != (T, Hq, Dv) or not out.is_contiguous():
            raise ValueError(f"out must be a contiguous {qt} tensor [num_q_tokens, Hq, {Dv}]")
        rows = c.num_kv_heads if c.kv_layout == RPA_KV_LATENT else 2 * c.num_kv_heads
        want_kv = (c.total_num_pages, c.page_size, rows, D)
        if tuple(kv_pages.shape) != want_kv or not kv_pages.is_contiguous():
            raise ValueError(f"kv_pages must be contiguous {want_kv}")
        if c.kv_dtype == RPA_DT_BF16 and kv_pages.dtype != torch.bfloat16:
            raise ValueError("kv_pages must be bfloat16")
        if c.kv_dtype == RPA_DT_F16 and kv_pages.dtype != torch.float16:
            raise ValueError("kv_pages must be float16")
        if c.kv_dtype in (RPA_DT_FP8_E4M3, RPA_DT_FP8_E5M2, RPA_DT_INT8) and kv_pages.element_size() != 1:
            raise ValueError("kv_pages must hold one byte per element (fp8 / int8)")
        for name, t, shape in (("kv_lens", kv_lens, (c.max_num_seqs,)),
                               ("page_indices", page_indices, (c.max_num_seqs, c.pages_per_seq)),
                               ("cu_q_lens", cu_q_lens, (c.max_num_seqs + 1,))):
            if t.dtype != torch.int32 or tuple(t.shape) != shape or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous int32 tensor {shape}")

    @property
    def out_dim(self) -> int:
        """Width of o: head_dim, or v_head_dim for the latent layout."""
        return int(self._c.v_head_dim) if self._c.kv_layout == RPA_KV_LATENT else int(self._c.head_dim)

    def forward(self, q, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, out=None, stream=None):
        if out is None:
            out = q.new_empty((q.shape[0], q.shape[1], self.out_dim))
        self._check(q, kv_pages, kv_lens, page_indices, cu_q_lens, out)
        for t in (q, kv_pages, kv_lens, page_indices, cu_q_lens, out):
            if not t.is_cuda:
                raise ValueError("forward takes CUDA tensors; use forward_host for host buffers")
        r = lib().rpa_forward(self._h, q.data_ptr(), kv_pages.data_ptr(), kv_lens.data_ptr(),
                              page_indices.data_ptr(), cu_q_lens.data_ptr(), int(num_seqs),
                              out.data_ptr(), _stream_ptr(stream))
        if r != RPA_OK:
            raise RpaError(r, "rpa_forward")
        return out

    def forward_host(self, q, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, out, stream=None):
        """q, kv_lens, page_indices, cu_q_lens and out in (pinned) host memory; kv_pages on device."""
        self._check(q, kv_pages, kv_lens, page_indices, cu_q_lens, out)
        if not kv_pages.is_cuda or q.is_cuda or out.is_cuda:
            raise ValueError("forward_host takes host q/int arrays/out and a device kv_pages")
        r = lib().rpa_forward_host(self._h, q.data_ptr(), kv_pages.data_ptr(), kv_lens.data_ptr(),
                                   page_indices.data_ptr(), cu_q_lens.data_ptr(), int(num_seqs),
                                   out.data_ptr(), _stream_ptr(stream))
        if r != RPA_OK:
            raise RpaError(r, "rpa_forward_host")
        return out

    def status(self, stream=None) -> int:
        return int(lib().rpa_get_status(self._h, _stream_ptr(stream)))

    def set_option(self, option: int, value: int):
        r = lib().rpa_set_option(self._h, int(option), int(value))
        if r != RPA_OK:
            raise RpaError(r, "rpa_set_option")

    def profile_begin(self, max_calls: int):
        r = lib().rpa_profile_begin(self._h, int(max_calls))
        if r != RPA_OK:
            raise RpaError(r, "rpa_profile_begin")

    def profile_read(self, max_calls: int) -> np.ndarray:
        """[calls, 4] kernel durations (ms): planner, decode, prefill, combine."""
        ms = np.zeros((max(1, int(max_calls)), 4), np.float32)
        n = ctypes.c_int32(0)
        r = lib().rpa_profile_read(self._h, ms.ctypes.data, int(max_calls), ctypes.byref(n))
        if r != RPA_OK:
            raise RpaError(r, "rpa_profile_read")
        return ms[: n.value]

    def plan(self, max_items: int = 1 << 20, stream=None):
        """(info[16], items[n, 8]) of the last call; synchronises the stream."""
        info = np.zeros(16, np.int32)
        r = lib().rpa_read_plan(self._h, info.ctypes.data, None, 0, _stream_ptr(stream))
        if r != RPA_OK:
            raise RpaError(r, "rpa_read_plan")
        n = min(int(info[1]) + int(info[2]), max_items)
        items = np.zeros((max(n, 1), 8), np.int32)
        r = lib().rpa_read_plan(self._h, info.ctypes.data, items.ctypes.data, n, _stream_ptr(stream))
        if r != RPA_OK:
            raise RpaError(r, "rpa_read_plan")
        return info, items[:n]
