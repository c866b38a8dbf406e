"""The MLA oracle's pins must catch plausible mistakes: each mutant is
``oracle/mla.py`` with one planted error (a dropped rotary term, a shifted
value slice, a wrong causal limit, a dropped scale, ...), and at least one pin
of ``test_oracle_mla.py`` must fail on it.  CPU only."""
import importlib.util
import inspect
import os
import types

import numpy as np
import pytest

import oracle
import oracle.mla as real

HERE = os.path.dirname(__file__)

MUTANTS = {
    "rope_term_dropped": ("s = sc * (qr @ C[:p + 1].T)",
                          "s = sc * (qr[:, :kv_lora_rank] @ C[:p + 1, :kv_lora_rank].T)"),
    "value_slice_from_the_end": ("values = C[:, :kv_lora_rank]", "values = C[:, Dqk - kv_lora_rank:]"),
    "causal_off_by_one": ("p = L - qn + r  ", "p = L - qn + r - 1  "),
    "causal_reversed": ("p = L - qn + r  ", "p = L - 1 - r  "),
    "query_row_of_first_token": ("qr = bf16_bits_to_float64(q_bits[t0 + r])", "qr = bf16_bits_to_float64(q_bits[t0])"),
    "kv_scale_dropped": ("return e4m3fn_to_float64(raw) * np.float64(np.float32(kv_scale))",
                         "return e4m3fn_to_float64(raw)"),
    "slot_off_by_one": ("cache[pages, j % PAGE_SIZE, :]", "cache[pages, (j + 1) % PAGE_SIZE, :]"),
    "page_index_rounding": ("[j // PAGE_SIZE]", "[(j + 1) // PAGE_SIZE]"),
    "scale_dropped": ("s = sc * (qr", "s = (qr"),
    "lse_max_dropped": ("l = m[:, 0] + np.log", "l = np.log"),
    "weights_unnormalised": ("np.exp(s - l[:, None])", "np.exp(s - m)"),
}


def _mutant_module(name, old, new):
    src = inspect.getsource(real)
    assert src.count(old) == 1, (name, old)
    mod = types.ModuleType(f"oracle.mla_mutant_{name}")
    mod.__package__ = "oracle"
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def _pins():
    spec = importlib.util.spec_from_file_location("_mla_pins_for_mutants", os.path.join(HERE, "test_oracle_mla.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _pin_calls(pins):
    for kv in ("bf16", "fp8"):
        for ql in ((1,), (2, 3, 4)):
            yield pins.test_mla_oracle_matches_sdpa, (kv, ql)
    yield pins.test_mla_zero_query_gives_mean_latent_and_log_length, ()
    yield pins.test_mla_rotary_part_alone_selects_a_planted_key, ()
    yield pins.test_mla_constant_latent_returns_it_whatever_the_rotary_keys, ()
    yield pins.test_mla_verification_rows_equal_prefix_decodes, ()
    yield pins.test_mla_page_permutation_invariance_bit_exact, ("bf16",)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mla_pins_catch_mutant(name):
    mutant = _mutant_module(name, *MUTANTS[name])
    pins = _pins()
    pins.oracle = types.SimpleNamespace(mla_decode=mutant.mla_decode, bf16_bits_to_float64=oracle.bf16_bits_to_float64,
                                        paged_decode_attention=oracle.paged_decode_attention)
    caught = []
    for fn, args in _pin_calls(pins):
        try:
            with np.errstate(all="ignore"):   # a planted mistake may produce inf / NaN
                fn(*args)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught.append(fn.__name__)
    assert caught, f"no pin detects mutant {name}"


def test_unmutated_mla_oracle_passes_the_same_calls():
    pins = _pins()
    for fn, args in _pin_calls(pins):
        fn(*args)
