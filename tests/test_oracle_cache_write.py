"""Pins for the cache-write oracle: the e4m3fn encoder against torch's
converter, the OCP grid's midpoints (ties to even) and saturation points, and
the scatter against an independent slot arithmetic."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.paged_attention import e4m3fn_to_float64


def test_encoder_matches_torch_inside_the_finite_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 30, 20000), rng.normal(0, 0.01, 5000), rng.uniform(-448, 448, 5000)])
    x32 = x.astype(np.float32)
    ours = oracle.e4m3fn_encode(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_every_grid_value_and_midpoint():
    codes = np.arange(0x7F, dtype=np.uint8)
    vals = e4m3fn_to_float64(codes)
    assert np.array_equal(oracle.e4m3fn_encode(vals), codes)
    assert np.array_equal(oracle.e4m3fn_encode(-vals[1:]), codes[1:] | 0x80)
    mids = (vals[:-1] + vals[1:]) / 2
    got = oracle.e4m3fn_encode(mids)
    expect = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])   # ties to the even code
    assert np.array_equal(got, expect)
    ref = torch.from_numpy(mids.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)                                 # mids are exact in fp32


@pytest.mark.parametrize("x,code", [(448.0, 0x7E), (449.0, 0x7E), (464.0, 0x7E), (1e30, 0x7E), (math.inf, 0x7E),
                                    (-math.inf, 0xFE), (-500.0, 0xFE), (2.0 ** -10, 0x00), (3 * 2.0 ** -11, 0x01),
                                    (-0.0, 0x80), (0.0, 0x00), (1.0, 0x38)])
def test_saturation_and_special_points(x, code):
    assert oracle.e4m3fn_encode(np.array([x]))[0] == code


def test_quantize_multiplies_by_the_fp32_reciprocal():
    bits = torch.tensor([0.3, -7.5, 15.0, 0.0123]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.quantize_rows(bits, 0.05)
    r = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(0.05, dtype=torch.float32)
    y = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float() * r
    assert np.array_equal(got, y.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    # 100 / 0.05 = 2000 is beyond the e4m3fn range: saturates (torch's cast would give NaN)
    big = torch.tensor([100.0, -100.0]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert oracle.quantize_rows(big, 0.05).tolist() == [0x7E, 0xFE]


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_scatter_against_page_offset_arithmetic(kv_dtype):
    rng = np.random.default_rng(3)
    T, Hkv, D, NB = 37, 2, 16, 9
    key = rng.normal(size=(T, Hkv, D)).astype(np.float32)
    val = rng.normal(size=(T, Hkv, D)).astype(np.float32)
    kb = torch.from_numpy(key).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    vb = torch.from_numpy(val).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    slots = rng.permutation(NB * 16)[:T].astype(np.int32)
    slots[[3, 11]] = -1                                         # padding tokens
    dt = np.uint8 if kv_dtype == "fp8" else np.uint16
    kc = rng.integers(0, 2 ** (8 * np.dtype(dt).itemsize), size=(NB, 16, Hkv, D)).astype(dt)
    vc = rng.integers(0, 2 ** (8 * np.dtype(dt).itemsize), size=(NB, 16, Hkv, D)).astype(dt)
    k2, v2 = oracle.cache_write(kb, vb, slots, kc, vc, 0.05, 0.07, kv_dtype)
    flat_k, flat_v = kc.reshape(NB * 16, Hkv, D).copy(), vc.reshape(NB * 16, Hkv, D).copy()
    for t in range(T):
        if slots[t] < 0:
            continue
        if kv_dtype == "bf16":
            flat_k[slots[t]], flat_v[slots[t]] = kb[t], vb[t]
        else:
            rk = torch.tensor(1.0) / torch.tensor(0.05)
            rv = torch.tensor(1.0) / torch.tensor(0.07)
            kq = (torch.from_numpy(kb[t].view(np.int16)).view(torch.bfloat16).float() * rk).to(torch.float8_e4m3fn)
            vq = (torch.from_numpy(vb[t].view(np.int16)).view(torch.bfloat16).float() * rv).to(torch.float8_e4m3fn)
            flat_k[slots[t]], flat_v[slots[t]] = kq.view(torch.uint8).numpy(), vq.view(torch.uint8).numpy()
    assert np.array_equal(k2, flat_k.reshape(kc.shape)) and np.array_equal(v2, flat_v.reshape(vc.shape))


def test_out_of_range_slots_write_nothing():
    kc = np.zeros((2, 16, 1, 4), dtype=np.uint16)
    kb = np.full((2, 1, 4), 0x3F80, dtype=np.uint16)
    k2, v2 = oracle.cache_write(kb, kb, np.array([32, 5]), kc, kc)
    assert k2[0, 5].tolist() == [[0x3F80] * 4] and int(k2.sum()) == 4 * 0x3F80


# ------------------------------------------------- planted mistakes are caught
import importlib.util as _ilu
import inspect as _inspect
import os as _os
import types as _types

import importlib as _il

_real_cw = _il.import_module("oracle.cache_write")   # the module (the package re-exports a function of the same name)

_CW_MUTANTS = {
    "ties_away_from_zero": ("(d_lo == d_hi) & (lo % 2 == 0)", "(d_lo == d_hi) & False"),
    "no_saturation": ("np.minimum(a, _VALUES[-1])", "np.minimum(a, _VALUES[-2])"),
    "multiply_by_scale": ("y32 = x32 * r32", "y32 = x32 * np.float32(scale)"),
    "slot_offset_swapped": ("page, off = int(s) // PAGE_SIZE, int(s) % PAGE_SIZE",
                            "off, page = int(s) // PAGE_SIZE, int(s) % PAGE_SIZE"),
    "sign_dropped": ("code = np.where(np.signbit(x), code | 0x80, code)", "code = np.where(np.signbit(x), code, code)"),
    "padding_written": ("if s < 0 or s >= NB * PAGE_SIZE:", "if s >= NB * PAGE_SIZE:"),
}


@pytest.mark.parametrize("name", sorted(_CW_MUTANTS))
def test_cache_write_pins_catch_mutant(name):
    old, new = _CW_MUTANTS[name]
    src = _inspect.getsource(_real_cw)
    assert src.count(old) == 1
    src = src.replace("from .paged_attention import", "from oracle.paged_attention import").replace(old, new)
    mod = _types.ModuleType("cw_mutant")
    exec(compile(src, f"<mutant {name}>", "exec"), mod.__dict__)
    spec = _ilu.spec_from_file_location("_cw_pins", _os.path.abspath(__file__))
    pins = _ilu.module_from_spec(spec)
    spec.loader.exec_module(pins)
    pins.oracle = _types.SimpleNamespace(e4m3fn_encode=mod.e4m3fn_encode, quantize_rows=mod.quantize_rows,
                                         cache_write=mod.cache_write)
    calls = [(pins.test_encoder_matches_torch_inside_the_finite_range, ()), (pins.test_every_grid_value_and_midpoint, ()),
             (pins.test_quantize_multiplies_by_the_fp32_reciprocal, ()), (pins.test_out_of_range_slots_write_nothing, ())]
    calls += [(pins.test_saturation_and_special_points, args) for args in
              [(448.0, 0x7E), (1e30, 0x7E), (-500.0, 0xFE), (-0.0, 0x80)]]
    calls += [(pins.test_scatter_against_page_offset_arithmetic, (k,)) for k in ("bf16", "fp8")]
    caught = 0
    for fn, args in calls:
        try:
            fn(*args)
        except (AssertionError, IndexError, ValueError):
            caught += 1
    assert caught, f"no pin detects mutant {name}"
