"""The binding's argument checks on the CPU (no handle is created: the checks only read the
configuration), so that a wrong shape, dtype or layout is refused before any pointer crosses the
C ABI."""
import pytest

torch = pytest.importorskip("torch")

import ragged_paged_attention_02_gb300 as rpa  # noqa: E402
from ragged_paged_attention_02_gb300.binding import RaggedPagedAttention  # noqa: E402

CFG = dict(num_q_tokens=22, num_q_heads=4, num_kv_heads=2, head_dim=64, total_num_pages=16,
           page_size=16, max_num_seqs=3, pages_per_seq=4, sm_scale=0.125)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _att(**over):
    a = object.__new__(RaggedPagedAttention)  # argument checks only: no rpa_create
    a._c = rpa.make_cfg(**dict(CFG, **over))
    a._h = None
    return a


def _args(kv_dtype=torch.bfloat16):
    q = torch.zeros(22, 4, 64, dtype=torch.bfloat16)
    kv = torch.zeros(16, 16, 4, 64, dtype=kv_dtype)
    kvl = torch.zeros(3, dtype=torch.int32)
    pi = torch.zeros(3, 4, dtype=torch.int32)
    cu = torch.zeros(4, dtype=torch.int32)
    out = torch.empty_like(q)
    return [q, kv, kvl, pi, cu, out]


def test_well_formed_arguments_pass():
    _att()._check(*_args())
    _att(kv_dtype="fp8_e4m3", k_scale=0.1, v_scale=0.1)._check(*_args(torch.uint8))


@pytest.mark.parametrize("index,bad", [
    (0, torch.zeros(22, 4, 64, dtype=torch.float16)),          # q not bf16
    (0, torch.zeros(21, 4, 64, dtype=torch.bfloat16)),         # q rows
    (0, torch.zeros(22, 64, 4, dtype=torch.bfloat16).transpose(1, 2)),  # q not contiguous
    (1, torch.zeros(16, 16, 2, 64, dtype=torch.bfloat16)),     # K and V not interleaved (2*Hkv)
    (1, torch.zeros(16, 16, 4, 64, dtype=torch.uint8)),        # bytes for a bf16 cache
    (2, torch.zeros(3, dtype=torch.int64)),                    # kv_lens int64
    (3, torch.zeros(3, 5, dtype=torch.int32)),                 # page_indices columns
    (4, torch.zeros(3, dtype=torch.int32)),                    # cu_q_lens needs max_num_seqs + 1
    (5, torch.zeros(22, 4, 64, dtype=torch.float32)),          # out dtype
])
def test_malformed_arguments_are_refused(index, bad):
    args = _args()
    args[index] = bad
    with pytest.raises(ValueError):
        _att()._check(*args)


def test_fp8_cache_must_hold_bytes():
    with pytest.raises(ValueError):
        _att(kv_dtype="fp8_e4m3")._check(*_args(torch.bfloat16))


def test_forward_refuses_host_tensors():
    with pytest.raises(ValueError, match="CUDA tensors"):
        _att().forward(*_args()[:5], num_seqs=1, out=_args()[5])
