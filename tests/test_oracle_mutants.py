"""The oracle's pins must catch plausible mistakes.  Each mutant below is the
oracle's source with one planted error (a dropped term, a wrong sign, bias or
index, a transposed mapping); the test asserts that at least one pin in
``test_oracle.py`` fails on it.  Everything runs on the CPU."""
import importlib.util
import inspect
import os
import types

import numpy as np
import pytest

import oracle.paged_attention as real

HERE = os.path.dirname(__file__)

MUTANTS = {
    "slot_off_by_one": ("slots = j % PAGE_SIZE", "slots = (j + 1) % PAGE_SIZE"),
    "page_index_rounding": ("[j // PAGE_SIZE]", "[(j + 1) // PAGE_SIZE]"),
    "causal_off_by_one": ("limits = L - qn + np.arange(qn)", "limits = L - qn + np.arange(qn) - 1"),
    "causal_reversed": ("limits = L - qn + np.arange(qn)", "limits = L - 1 - np.arange(qn)"),
    "gqa_interleaved": ("heads = np.arange(hk * G, (hk + 1) * G)", "heads = np.arange(hk, Hq, Hkv)"),
    "scale_dropped": ("s = scale * (q_rows @ keys.T)", "s = (q_rows @ keys.T)"),
    "e4m3_bias": ("np.ldexp(1.0, (e - 7)", "np.ldexp(1.0, (e - 8)"),
    "e4m3_subnormal": ("* np.ldexp(1.0, -6)", "* np.ldexp(1.0, -7)"),
    "e4m3_mantissa": ("(1.0 + m / 8.0)", "(1.0 + m / 16.0)"),
    "e4m3_sign": ("np.where(s == 1, -1.0, 1.0)", "np.where(s == 1, 1.0, 1.0)"),
    "fp8_scale_dropped": ("v = e4m3fn_to_float64(raw) * np.float64(np.float32(tensor_scale))",
                          "v = e4m3fn_to_float64(raw)"),
    "lse_max_dropped": ("lse = m[:, 0] + np.log", "lse = np.log"),
    "weights_unnormalised": ("w = np.exp(s - lse[:, None])", "w = np.exp(s - m)"),
    "values_are_keys": ("out = w @ values", "out = w @ keys"),
    "bf16_shift": ("<< np.uint32(16)", "<< np.uint32(15)"),
    "window_off_by_one": ("allowed &= j > lim - window", "allowed &= j >= lim - window"),
    "window_from_sequence_start": ("allowed &= j > lim - window", "allowed &= j < window"),
    "sink_value_row_nonzero": ("np.zeros((1, values.shape[1]))", "np.ones((1, values.shape[1]))"),
    "sink_scaled": ("np.asarray(sinks, dtype=np.float64)[:, None]", "scale * np.asarray(sinks, dtype=np.float64)[:, None]"),
    "token_scale_dropped": ("v = v * np.asarray(token_scales", "v = v + 0 * np.asarray(token_scales"),
    "token_scale_slot_reversed": ("[pages, kv_head, tok % PAGE_SIZE]", "[pages, kv_head, PAGE_SIZE - 1 - tok % PAGE_SIZE]"),
    "token_scale_head_ignored": ("[pages, kv_head, tok % PAGE_SIZE]", "[pages, 0, tok % PAGE_SIZE]"),
    "token_scale_page_shifted": ("[tok // PAGE_SIZE]", "[(tok + 1) // PAGE_SIZE]"),
    "value_scales_for_keys": ("ks = gather_token_scales(k_token_scales", "ks = gather_token_scales(v_token_scales"),
}


def _mutant_module(name, old, new):
    src = inspect.getsource(real)
    assert src.count(old) == 1, (name, old)
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def _pins_module(name="test_oracle.py"):
    spec = importlib.util.spec_from_file_location("_pins_for_mutants_" + name[:-3], os.path.join(HERE, name))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _pin_calls(pins):
    yield pins.test_bf16_golden_points, ()
    yield pins.test_e4m3_golden_points, ()
    yield pins.test_e4m3_decode_matches_torch_all_codes, ()
    yield pins.test_fp8_scale_is_fp32_rounded, ()
    for kv in ("bf16", "fp8"):
        for ql in ((1,), (2, 3, 4)):
            yield pins.test_oracle_matches_sdpa_on_contiguous_kv, (kv, ql)
    yield pins.test_length_one_returns_first_value_row, ()
    yield pins.test_zero_query_gives_mean_value_and_log_length, ()
    yield pins.test_two_keys_closed_form, ()
    yield pins.test_gqa_mapping_consecutive_heads_share_kv_head, ()
    yield pins.test_mtp_row_equals_prefix_attention, ()
    yield pins.test_fp8_scale_folding_and_linearity, ()
    for win in (1, 5, 17):
        yield pins.test_sliding_window_matches_sdpa_with_window_mask, (win, (2, 3, 4))
    yield pins.test_window_of_one_returns_own_value_and_wide_window_changes_nothing, ()
    yield pins.test_sink_closed_form_against_the_sinkless_result, ()


def _pertoken_pin_calls(pt):
    for ql in ((1,), (2, 3, 4)):
        yield pt.test_per_token_oracle_matches_sdpa, (ql, (0.5, 3.0))
    yield pt.test_equal_token_scales_reduce_to_the_per_tensor_scale, ()
    yield pt.test_one_value_scale_doubled_adds_its_weighted_row, ()
    yield pt.test_per_token_page_permutation_invariance_bit_exact, ()
    yield pt.test_key_scale_is_indexed_by_head_then_slot, ()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    old, new = MUTANTS[name]
    mutant = _mutant_module(name, old, new)
    pins = _pins_module()
    pt = _pins_module("test_oracle_pertoken.py")
    pins.oracle = pt.oracle = types.SimpleNamespace(**{k: getattr(mutant, k) for k in (
        "PAGE_SIZE", "attend", "bf16_bits_to_float64", "dequantize", "e4m3fn_to_float64",
        "gather_sequence", "gather_token_scales", "paged_decode_attention", "run_workload")})
    caught = []
    for fn, args in list(_pin_calls(pins)) + list(_pertoken_pin_calls(pt)):
        try:
            with np.errstate(all="ignore"):   # a planted mistake may produce inf / NaN
                fn(*args)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught.append(fn.__name__)
    assert caught, f"no pin detects mutant {name}"


def test_unmutated_oracle_passes_the_same_calls():
    pins = _pins_module()
    pt = _pins_module("test_oracle_pertoken.py")
    for fn, args in list(_pin_calls(pins)) + list(_pertoken_pin_calls(pt)):
        fn(*args)
