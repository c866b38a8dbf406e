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


def _torch_quantize(x_bf16, scale):
    """torch's own fp32 division and e4m3fn cast (NaN for quotients past 448
    in torch, so callers keep inside the finite range)."""
    return (x_bf16.float() / torch.tensor(scale, dtype=torch.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_quantize_divides_by_the_scale():
    bits = torch.tensor([0.3, -7.5, 15.0, 0.0123]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.quantize_rows(bits, 0.05)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    assert np.array_equal(got, _torch_quantize(x, 0.05))
    # 100 / 0.05 = 2000 is beyond the e4m3fn range: saturates (torch's cast would give NaN)
    big = torch.tensor([100.0, -100.0]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert oracle.quantize_rows(big, 0.05).tolist() == [0x7E, 0xFE]


def test_quantize_is_a_division_not_a_reciprocal_product():
    # x = 0.000732421875 * 2^k (exact in bf16) over the fp32 scale 0.03: the
    # quotient lands exactly on a midpoint of the e4m3fn grid (0.0244140625 =
    # 2^-6 * (1 + 4.5/8) for k = 0) and rounds to the even code, while x times
    # the fp32 reciprocal of 0.03 lands one fp32 ulp above it and rounds up
    x = torch.tensor([0.000732421875 * 2.0 ** k for k in range(4)] + [-0.00146484375]).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    got = oracle.quantize_rows(bits, 0.03)
    expect = _torch_quantize(x, 0.03)
    assert np.array_equal(got, expect)
    recip = (x.float() * (torch.tensor(1.0) / torch.tensor(0.03))).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (expect != recip).all()                                  # the case tells the two forms apart


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
            flat_k[slots[t]] = _torch_quantize(torch.from_numpy(kb[t].view(np.int16)).view(torch.bfloat16), 0.05)
            flat_v[slots[t]] = _torch_quantize(torch.from_numpy(vb[t].view(np.int16)).view(torch.bfloat16), 0.07)
    assert np.array_equal(k2, flat_k.reshape(kc.shape)) and np.array_equal(v2, flat_v.reshape(vc.shape))


def test_out_of_range_slots_write_nothing():
    kc = np.zeros((2, 16, 1, 4), dtype=np.uint16)
    kb = np.full((2, 1, 4), 0x3F80, dtype=np.uint16)
    k2, v2 = oracle.cache_write(kb, kb, np.array([32, 5]), kc, kc)
    assert k2[0, 5].tolist() == [[0x3F80] * 4] and int(k2.sum()) == 4 * 0x3F80


# ------------------------------------------------- per-token quantisation

def _bf16_bits(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_per_token_quantize_matches_torch_ops():
    rng = np.random.default_rng(8)
    x = rng.normal(size=(50, 4, 64)) * np.exp(rng.uniform(-8, 8, size=(50, 4, 1)))
    bits = _bf16_bits(x)
    codes, scales = oracle.quantize_rows_per_token(bits)
    xt = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float()
    amax = xt.abs().amax(dim=-1)
    ref_scale = amax / 448.0
    ref_codes = (xt / ref_scale[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(scales, ref_scale.numpy())
    assert np.array_equal(codes, ref_codes)


def test_per_token_codes_divide_by_the_stored_scale():
    # a row with max |x| = 0.78515625 (bf16 0x3F49): x = 1.1980533599853516e-05
    # over its scale 0.78515625 / 448 (fp32) is 0.0068359375, a midpoint of the
    # e4m3fn grid (7 * 2^-10, between the subnormal codes 3 and 4) that rounds to
    # the even code; x times the fp32 reciprocal 448 / 0.78515625 lands one fp32
    # ulp below it and rounds down instead
    x = torch.tensor([[0.78515625, 1.1980533599853516e-05, -1.1980533599853516e-05, 0.5]]).to(torch.bfloat16)
    codes, scales = oracle.quantize_rows_per_token(_bf16_bits(x.float()))
    s = x.float().abs().amax(dim=-1) / 448.0
    expect = (x.float() / s[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, expect) and scales[0] == s.item()
    recip = (x.float() * (torch.tensor(448.0) / x.float().abs().amax(dim=-1))[..., None])
    recip = recip.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (expect[0, 1:3] != recip[0, 1:3]).all()                 # the case tells the two forms apart


def test_per_token_row_max_lands_on_the_top_code():
    bits = _bf16_bits([[0.25, -3.0, 1.5, 2.0], [1.0, 7.0, -7.0, 0.0]])
    codes, scales = oracle.quantize_rows_per_token(bits)
    assert codes[0, 1] == 0xFE and set(codes[1, 1:3].tolist()) == {0x7E, 0xFE}
    assert scales[0] == np.float32(3.0) / np.float32(448.0)
    deq = oracle.e4m3fn_to_float64(codes) * scales[:, None].astype(np.float64)
    assert abs(deq[0, 1] + 3.0) <= 3.0 * 2.0 ** -23 and abs(deq[1, 1] - 7.0) <= 7.0 * 2.0 ** -23


def test_per_token_zero_row_and_power_of_two_rows():
    zero = np.array([[0, 0x8000] * 4], dtype=np.uint16)          # +0 and -0
    codes, scales = oracle.quantize_rows_per_token(zero)
    assert scales[0] == 0.0 and not codes.any()
    rng = np.random.default_rng(9)
    x = rng.normal(size=(1, 32)).astype(np.float32)
    c1, s1 = oracle.quantize_rows_per_token(_bf16_bits(x))
    c2, s2 = oracle.quantize_rows_per_token(_bf16_bits(x * 2.0 ** 20))      # exact in bf16
    assert np.array_equal(c1, c2) and s2[0] == s1[0] * np.float32(2.0 ** 20)


def test_per_token_round_trip_error_bound():
    # e4m3fn keeps 3 mantissa bits: |deq - x| <= 2^-4 |x| on the normal range,
    # and <= 2^-10 * scale on the subnormal one (plus fp32 rounding of r)
    rng = np.random.default_rng(10)
    x = rng.normal(size=(200, 128)) * np.exp(rng.uniform(-5, 5, size=(200, 1)))
    bits = _bf16_bits(x)
    xv = oracle.bf16_bits_to_float64(bits)
    codes, scales = oracle.quantize_rows_per_token(bits)
    deq = oracle.e4m3fn_to_float64(codes) * scales[:, None].astype(np.float64)
    bound = np.maximum(2.0 ** -4 * np.abs(xv), 2.0 ** -10 * scales[:, None]) * (1 + 2.0 ** -20) + 1e-30
    assert (np.abs(deq - xv) <= bound).all()


def test_per_token_scatter_against_page_offset_arithmetic():
    rng = np.random.default_rng(12)
    T, Hkv, D, NB = 29, 3, 16, 7
    kb = _bf16_bits(rng.normal(size=(T, Hkv, D)))
    vb = _bf16_bits(rng.normal(size=(T, Hkv, D)) * 5)
    slots = rng.permutation(NB * 16)[:T].astype(np.int32)
    slots[[2, 9]] = -1
    slots[5] = NB * 16 + 3                                       # past the pool: skipped
    kc = rng.integers(0, 256, size=(NB, 16, Hkv, D)).astype(np.uint8)
    vc = rng.integers(0, 256, size=(NB, 16, Hkv, D)).astype(np.uint8)
    ks = rng.uniform(size=(NB, Hkv, 16)).astype(np.float32)
    vs = rng.uniform(size=(NB, Hkv, 16)).astype(np.float32)
    k2, v2, ks2, vs2 = oracle.cache_write_per_token(kb, vb, slots, kc, vc, ks, vs)
    fk, fv = kc.reshape(NB * 16, Hkv, D).copy(), vc.reshape(NB * 16, Hkv, D).copy()
    fks, fvs = ks.transpose(0, 2, 1).reshape(NB * 16, Hkv).copy(), vs.transpose(0, 2, 1).reshape(NB * 16, Hkv).copy()
    for t in range(T):
        if not 0 <= slots[t] < NB * 16:
            continue
        for h in range(Hkv):
            xk = torch.from_numpy(kb[t, h].view(np.int16)).view(torch.bfloat16).float()
            xv = torch.from_numpy(vb[t, h].view(np.int16)).view(torch.bfloat16).float()
            for x, fc, fs in ((xk, fk, fks), (xv, fv, fvs)):
                amax = x.abs().max()
                fc[slots[t], h] = (x / (amax / 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                fs[slots[t], h] = (amax / 448.0).item()
    assert np.array_equal(k2, fk.reshape(kc.shape)) and np.array_equal(v2, fv.reshape(vc.shape))
    assert np.array_equal(ks2, fks.reshape(NB, 16, Hkv).transpose(0, 2, 1))
    assert np.array_equal(vs2, fvs.reshape(NB, 16, Hkv).transpose(0, 2, 1))


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
    "multiply_by_scale": ("y32 = x32 / np.float32(scale)", "y32 = x32 * np.float32(scale)"),
    "multiply_by_reciprocal": ("y32 = x32 / np.float32(scale)", "y32 = x32 * (np.float32(1) / np.float32(scale))"),
    "slot_offset_swapped": ("page, off = int(s) // PAGE_SIZE, int(s) % PAGE_SIZE",
                            "off, page = int(s) // PAGE_SIZE, int(s) % PAGE_SIZE"),
    "sign_dropped": ("code = np.where(np.signbit(x), code | 0x80, code)", "code = np.where(np.signbit(x), code, code)"),
    "padding_written": ("if s < 0 or s >= NB * PAGE_SIZE:", "if s >= NB * PAGE_SIZE:"),
    "pt_padding_written": ("if not 0 <= s < NB * PAGE_SIZE:", "if not s < NB * PAGE_SIZE:"),
    "pt_slot_offset_swapped": ("page, off = divmod(int(s), PAGE_SIZE)", "off, page = divmod(int(s), PAGE_SIZE)"),
    "pt_signed_max": ("amax = np.abs(x32).max(axis=-1)", "amax = x32.max(axis=-1)"),
    "pt_scale_inverted": ("scale = (amax / np.float32(E4M3_MAX))", "scale = (np.float32(E4M3_MAX) / amax)"),
    "pt_scale_slot_head_swapped": ("ks_out[page, :, off], vs_out[page, :, off] = ksc, vsc",
                                   "ks_out[page, off % ks_out.shape[1], :ksc.shape[0]], vs_out[page, off % vs_out.shape[1], :vsc.shape[0]] = ksc, vsc"),
    "pt_multiply_by_reciprocal": ("x32 / np.where(nonzero, scale, np.float32(1))[..., None]",
                                  "x32 * (np.float32(E4M3_MAX) / np.where(nonzero, amax, np.float32(1)))[..., None]"),
    "pt_multiply_by_scale": ("x32 / np.where(nonzero, scale, np.float32(1))[..., None]",
                             "x32 * np.where(nonzero, scale, np.float32(1))[..., None]"),
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
                                         cache_write=mod.cache_write, quantize_rows_per_token=mod.quantize_rows_per_token,
                                         cache_write_per_token=mod.cache_write_per_token,
                                         e4m3fn_to_float64=oracle.e4m3fn_to_float64,
                                         bf16_bits_to_float64=oracle.bf16_bits_to_float64)
    calls = [(pins.test_encoder_matches_torch_inside_the_finite_range, ()), (pins.test_every_grid_value_and_midpoint, ()),
             (pins.test_quantize_divides_by_the_scale, ()), (pins.test_quantize_is_a_division_not_a_reciprocal_product, ()),
             (pins.test_out_of_range_slots_write_nothing, ())]
    calls += [(pins.test_saturation_and_special_points, args) for args in
              [(448.0, 0x7E), (1e30, 0x7E), (-500.0, 0xFE), (-0.0, 0x80)]]
    calls += [(pins.test_scatter_against_page_offset_arithmetic, (k,)) for k in ("bf16", "fp8")]
    calls += [(pins.test_per_token_quantize_matches_torch_ops, ()), (pins.test_per_token_row_max_lands_on_the_top_code, ()),
              (pins.test_per_token_codes_divide_by_the_stored_scale, ()),
              (pins.test_per_token_zero_row_and_power_of_two_rows, ()), (pins.test_per_token_round_trip_error_bound, ()),
              (pins.test_per_token_scatter_against_page_offset_arithmetic, ())]
    caught = 0
    for fn, args in calls:
        try:
            with np.errstate(all="ignore"):   # a planted mistake may produce inf / NaN
                fn(*args)
        except (AssertionError, IndexError, ValueError):
            caught += 1
    assert caught, f"no pin detects mutant {name}"
