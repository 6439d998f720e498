"""Mutation check of the oracle's pins: plant a plausible slip in a copy of the oracle's C source
(a mask edge, the query position, a dropped scale, a K/V or GQA index, the soft cap, the softmax
denominator, the fp8 decoder), compile it, and check that the pins of test_oracle_pins.py catch
it.  The mistakes are planted in a temporary copy on the CPU; the oracle itself is untouched."""
import ctypes
import math
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "rpa_oracle.c")

# (name, text in rpa_oracle.c, replacement); each text occurs at least once and every
# occurrence is replaced
MUTATIONS = [
    ("window edge", "p - c->sliding_window >= j", "p - c->sliding_window > j"),
    ("causal edge", "c->is_causal && j > p", "c->is_causal && j >= p"),
    ("query position", "const int64_t p = kv_len - q_len + i;", "const int64_t p = kv_len - q_len + i - 1;"),
    ("dropped sm_scale", "double xj = c->sm_scale * dot;", "double xj = dot;"),
    ("K read from the V head", "kv_elem(c, kv, page, slot, h, 0, d) * ks", "kv_elem(c, kv, page, slot, h, 1, d) * ks"),
    ("split V head off by one", "+ 2 * h + is_v) * c->head_dim + d;", "+ 2 * h + 2 * is_v) * c->head_dim + d;"),
    ("GQA map strided", "const int64_t h = qh / G;", "const int64_t h = qh % c->num_kv_heads;"),
    ("dropped k_scale", "const double ks = c->has_k_scale ? c->k_scale : 1.0;", "const double ks = 1.0;"),
    ("dropped v_scale", "const double vs = c->has_v_scale ? c->v_scale : 1.0;", "const double vs = 1.0;"),
    ("soft cap ignored", "if (c->has_soft_cap) xj = c->soft_cap * tanh(xj / c->soft_cap);", ""),
    ("soft cap without the outer factor", "xj = c->soft_cap * tanh(xj / c->soft_cap);", "xj = tanh(xj / c->soft_cap);"),
    ("denominator counts keys", "denom += w;", "denom += 1.0;"),
    ("slot off by one", "int64_t slot = j % c->page_size;", "int64_t slot = (j + 1) % c->page_size;"),
    ("e4m3 subnormal scale", "v = ldexp((double)m / 8.0, 1 - 7); /* subnormal */", "v = ldexp((double)m / 8.0, -7);"),
    ("e4m3 exponent bias", "v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("f16 exponent bias", "else v = ldexp(1.0 + (double)m / 1024.0, e - 15);",
     "else v = ldexp(1.0 + (double)m / 1024.0, e - 14);"),
    ("e5m2 mantissa width", "else v = ldexp(1.0 + (double)m / 4.0, e - 15);",
     "else v = ldexp(1.0 + (double)m / 8.0, e - 15);"),
    ("int8 read unsigned", "case OKV_I8: return (double)((const int8_t*)kv)[idx];",
     "case OKV_I8: return (double)((const uint8_t*)kv)[idx];"),
    ("f32 q read as bf16", "case OQ_F32: return f32_to_f64((const float*)q + idx);",
     "case OQ_F32: return oracle_bf16_to_f64(((const uint16_t*)q)[idx]);"),
    ("latent V from the end of the row", "for (int64_t d = 0; d < Dv; ++d) out[d] += w * (kv_elem(c, kv, page, slot, h, 1, d) * vs);",
     "for (int64_t d = 0; d < Dv; ++d) out[d] += w * (kv_elem(c, kv, page, slot, h, 1, d + D - Dv) * vs);"),
    ("latent rows strided like the split layout", "idx = ((page * c->page_size + slot) * c->num_kv_heads + h) * c->head_dim + d;",
     "idx = ((page * c->page_size + slot) * c->num_kv_heads + 2 * h) * c->head_dim + d;"),
    ("sink left out of the denominator", "if (c->has_sinks) denom += exp(c->sinks[qh] - xmax);", ""),
    ("sink of the wrong head", "if (c->has_sinks) denom += exp(c->sinks[qh] - xmax);",
     "if (c->has_sinks) denom += exp(c->sinks[qh / G] - xmax);"),
    ("sink with the wrong sign", "if (c->has_sinks) denom += exp(c->sinks[qh] - xmax);",
     "if (c->has_sinks) denom += exp(-c->sinks[qh] - xmax);"),
]


def _pin_calls():
    """Every pin of test_oracle_pins.py as a zero-argument call."""
    calls = [pins.test_e4m3_decoder_all_codes, pins.test_bf16_decoder_matches_float32_view,
             pins.test_f16_decoder_all_codes, pins.test_e5m2_decoder_all_codes]
    calls += [lambda c=c: pins.test_oracle_equals_dense_brute_force(c) for c in range(len(pins.CASES))]
    calls += [lambda s=s: pins.test_oracle_random_configs_equal_brute_force(s) for s in range(24)]
    calls += [lambda a=a, w=w: pins.test_zero_query_averages_the_allowed_keys(a, w)
              for a, w in [(True, None), (True, 3), (True, 7), (False, None), (False, 4)]]
    calls += [lambda v=v: pins.test_zero_query_mean_shrunk_by_a_sink(v) for v in (0.0, math.log(3.0), -2.5)]
    calls += [pins.test_very_negative_sink_changes_nothing]
    calls += [lambda c=c: pins.test_latent_oracle_equals_dense_brute_force(c) for c in range(len(pins.LATENT_CASES))]
    calls += [pins.test_latent_equals_split_layout_with_padded_values,
              pins.test_latent_zero_query_averages_the_value_part]
    calls += [pins.test_two_keys_closed_form_weights, pins.test_window_one_selects_own_position,
              pins.test_uniform_v_gives_v, pins.test_single_key_sequence,
              pins.test_decode_equals_last_prefill_row, pins.test_gqa_equals_mha_with_repeated_kv,
              pins.test_scale_folding_equals_prescaled_bf16, pins.test_softcap_identity_from_capped_form]
    return calls


def _load_mutant(path):
    lib = ctypes.CDLL(path)
    ref = oracle._load()
    for name in ("rpa_oracle_forward", "rpa_oracle_rows", "rpa_oracle_validate", "oracle_bf16_to_f64",
                 "oracle_e4m3_to_f64", "oracle_e5m2_to_f64", "oracle_f16_to_f64"):
        f, g = getattr(lib, name), getattr(ref, name)
        f.argtypes, f.restype = g.argtypes, g.restype
    return lib


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation target not found: {name}"
    mutant = tmp_path / "rpa_oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    so = tmp_path / "librpa_oracle_mutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so),
                           str(mutant), "-lm"])
    lib = _load_mutant(str(so))
    saved = oracle._load()
    oracle._lib = lib
    caught = []
    try:
        for call in _pin_calls():
            try:
                call()
            except Exception as e:  # a failed pin (AssertionError) or a rejected input
                caught.append(type(e).__name__)
                break
    finally:
        oracle._lib = saved
    assert caught, f"no pin caught the planted mistake: {name}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    """Control: the same harness with the source unchanged catches nothing."""
    so = tmp_path / "librpa_oracle_copy.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so), SRC, "-lm"])
    lib = _load_mutant(str(so))
    saved = oracle._load()
    oracle._lib = lib
    try:
        for call in _pin_calls():
            call()
    finally:
        oracle._lib = saved
