"""Ragged paged attention for GB300 (sm_103a).

The computation lives in ``librpa.so`` (CUDA kernels behind the C ABI of
``include/rpa.h``); this package is the Python binding used by the tests and
the benchmark.  Build the library with ``__graft_entry__.build()`` or
``python -m ragged_paged_attention_02_gb300._build``.
"""

from .binding import (  # noqa: F401
    EXPORTS,
    MASK_VALUE,
    RPA_DT_BF16,
    RPA_DT_F16,
    RPA_DT_F32,
    RPA_DT_FP8_E4M3,
    RPA_DT_FP8_E5M2,
    RPA_DT_INT8,
    RPA_ERR_BAD_LENGTHS,
    RPA_ERR_BAD_PAGE_INDEX,
    RPA_ERR_CUDA,
    RPA_ERR_INVALID_ARG,
    RPA_ERR_NO_ALLOC_LIMIT,
    RPA_ERR_TIMEOUT,
    RPA_ERR_UNSUPPORTED,
    RPA_KV_LATENT,
    RPA_KV_SPLIT,
    RPA_OK,
    RPA_OPT_DECODE_SMS,
    RPA_OPT_PLAN_EARLY,
    RPA_OPT_PREFILL_SMS,
    RPA_OPT_SERIAL,
    RPA_OPT_TEST_STALL_PRODUCER,
    RPA_OPT_WAIT_TIMEOUT_MS,
    RaggedPagedAttention,
    RpaError,
    lib,
    library_path,
    make_cfg,
    validate_cfg,
)
