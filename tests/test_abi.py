"""The C ABI without a GPU: the library builds and loads, exports every symbol
that include/paged_attn.h declares, and rejects invalid arguments on the host
with the documented status codes before touching the device."""
import ctypes
import os
import re

import pytest
import torch

from paged_kv_decode_06_gb300 import binding
from paged_kv_decode_06_gb300 import build as builder

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_attn.h")


@pytest.fixture(scope="module")
def lib():
    builder.build()
    return binding.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(paged_attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("paged_attn_decode", "paged_attn_decode_ex", "paged_attn_plan", "paged_attn_reserve",
              "paged_attn_device_status", "paged_attn_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) == set(binding.EXPORTED)


def test_error_strings_and_version(lib):
    for st in range(5):
        assert binding.paged_attn_error_string(st).startswith("PA_")
    assert "unknown" in binding.paged_attn_error_string(99)
    assert binding.paged_attn_version() >= 100


def _good_args(T=3, Hq=8, Hkv=2, D=128, NB=10, B=3, MB=4, kv=torch.bfloat16):
    q = torch.zeros(T, Hq, D, dtype=torch.bfloat16)
    k = torch.zeros(NB, 16, Hkv, D, dtype=kv)
    v = torch.zeros(NB, 16, Hkv, D, dtype=kv)
    bt = torch.zeros(B, MB, dtype=torch.int32)
    sl = torch.ones(B, dtype=torch.int32)
    out = torch.zeros_like(q)
    lse = torch.zeros(T, Hq, dtype=torch.float32)
    return dict(q=q, k=k, v=v, bt=bt, sl=sl, qsl=None, out=out, lse=lse, max_qlen=1)


def _call(lib, a, scale=0.1):
    descs = [binding.tensor_desc(a[n]) for n in ("q", "k", "v", "bt", "sl", "qsl", "out", "lse")]
    refs = [ctypes.byref(d) for d in descs]
    return lib.paged_attn_decode(*refs[:6], a["max_qlen"], scale, 1.0, 1.0, refs[6], refs[7], None)


@pytest.mark.parametrize("mutate,expect", [
    (lambda a: a.update(q=a["q"].float()), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(out=a["out"].float()), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(bt=a["bt"].long()), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(v=torch.zeros(10, 16, 2, 128, dtype=torch.uint8)), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(k=torch.zeros(10, 8, 2, 128, dtype=torch.bfloat16),
                        v=torch.zeros(10, 8, 2, 128, dtype=torch.bfloat16)), binding.PA_ERR_UNSUPPORTED),
    (lambda a: a.update(q=torch.zeros(3, 8, 96, dtype=torch.bfloat16), out=torch.zeros(3, 8, 96, dtype=torch.bfloat16),
                        k=torch.zeros(10, 16, 2, 96, dtype=torch.bfloat16),
                        v=torch.zeros(10, 16, 2, 96, dtype=torch.bfloat16)), binding.PA_ERR_UNSUPPORTED),
    (lambda a: a.update(q=torch.zeros(3, 6, 128, dtype=torch.bfloat16), out=torch.zeros(3, 6, 128, dtype=torch.bfloat16),
                        k=torch.zeros(10, 16, 4, 128, dtype=torch.bfloat16),
                        v=torch.zeros(10, 16, 4, 128, dtype=torch.bfloat16), lse=None), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(sl=torch.ones(2, dtype=torch.int32)), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(q=torch.zeros(4, 8, 128, dtype=torch.bfloat16), out=torch.zeros(4, 8, 128, dtype=torch.bfloat16),
                        lse=None), binding.PA_ERR_INVALID_ARG),           # T != B without query_start_loc
    (lambda a: a.update(max_qlen=2), binding.PA_ERR_INVALID_ARG),         # max_qlen > 1 without query_start_loc
    (lambda a: a.update(q=torch.zeros(3, 8, 256, dtype=torch.bfloat16)[:, :, :128]), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(lse=torch.zeros(3, 4, dtype=torch.float32)), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(bt=torch.zeros(4, 3, dtype=torch.int32).t()), binding.PA_ERR_INVALID_ARG),
])
def test_invalid_arguments_rejected_on_host(lib, mutate, expect):
    a = _good_args()
    mutate(a)
    st = _call(lib, a)
    assert st == expect, binding.paged_attn_last_error_message()
    assert binding.paged_attn_last_error_message() != ""


def _rows_args(max_qlen, kv):
    """G = 32 query heads on one KV head; three sequences of max_qlen tokens."""
    a = _good_args(T=3 * max_qlen, Hq=32, Hkv=1)
    a["k"] = torch.zeros(10, 16, 1, 128, dtype=kv)
    a["v"] = torch.zeros(10, 16, 1, 128, dtype=kv)
    a["qsl"] = torch.arange(0, 3 * max_qlen + 1, max_qlen, dtype=torch.int32)
    a["max_qlen"] = max_qlen
    return a


def test_more_than_128_rows_per_kv_head_is_unsupported(lib):
    assert _call(lib, _rows_args(5, torch.bfloat16)) == binding.PA_ERR_UNSUPPORTED   # 160 rows
    assert "128" in binding.paged_attn_last_error_message()


def test_fp8_cache_over_64_rows_is_unsupported(lib):
    assert _call(lib, _rows_args(3, torch.float8_e4m3fn)) == binding.PA_ERR_UNSUPPORTED   # 96 rows
    assert "64" in binding.paged_attn_last_error_message()


def test_bf16_cache_up_to_128_rows_passes_host_validation(lib):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # 96 and 128 rows pass every host check; without a GPU the call then fails
    # at device set-up.
    for ql in (3, 4):
        assert _call(lib, _rows_args(ql, torch.bfloat16)) == binding.PA_ERR_CUDA


def _plan_status(lib, use_tcgen05, kv=binding.PA_BF16, Hq=8, max_qlen=1, heads_per_cta=0):
    opts = binding.make_options(use_tcgen05=use_tcgen05, heads_per_cta=heads_per_cta)
    plan = binding.PaPlan()
    return lib.paged_attn_plan(4, Hq, 1, 128, kv, max_qlen, ctypes.byref(opts), ctypes.byref(plan))


def test_tcgen05_switch_checked_on_the_host(lib):
    for bad in (-1, 3):
        assert _plan_status(lib, bad) == binding.PA_ERR_INVALID_ARG
    # forced on for an fp8 cache, forced off above 64 rows, more than one head per CTA
    assert _plan_status(lib, 2, kv=binding.PA_FP8_E4M3) == binding.PA_ERR_UNSUPPORTED
    assert _plan_status(lib, 1, Hq=32, max_qlen=3) == binding.PA_ERR_UNSUPPORTED
    assert _plan_status(lib, 0, Hq=32, max_qlen=3, heads_per_cta=2) == binding.PA_ERR_UNSUPPORTED


def test_null_descriptor_pointer(lib):
    a = _good_args()
    descs = [binding.tensor_desc(a[n]) for n in ("q", "k", "v", "bt", "sl", "qsl", "out", "lse")]
    refs = [ctypes.byref(d) for d in descs]
    st = lib.paged_attn_decode(None, *refs[1:6], 1, 0.1, 1.0, 1.0, refs[6], refs[7], None)
    assert st == binding.PA_ERR_INVALID_ARG


def test_non_finite_scale_rejected(lib):
    assert _call(lib, _good_args(), scale=float("nan")) == binding.PA_ERR_INVALID_ARG


def test_valid_arguments_without_gpu_report_cuda_error(lib):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call(lib, _good_args()) == binding.PA_ERR_CUDA


def test_plan_rejects_bad_shapes_without_device(lib):
    with pytest.raises(binding.PagedAttnError) as e:
        binding.paged_attn_plan(4, 8, 3, 128)
    assert e.value.status == binding.PA_ERR_INVALID_ARG
    with pytest.raises(binding.PagedAttnError) as e:
        binding.paged_attn_plan(4, 8, 2, 80)
    assert e.value.status == binding.PA_ERR_UNSUPPORTED


def _cw_args(T=4, Hkv=2, D=64, NB=3, kv=torch.bfloat16):
    return dict(key=torch.zeros(T, Hkv, D, dtype=torch.bfloat16), value=torch.zeros(T, Hkv, D, dtype=torch.bfloat16),
                slots=torch.zeros(T, dtype=torch.int32), kc=torch.zeros(NB, 16, Hkv, D, dtype=kv),
                vc=torch.zeros(NB, 16, Hkv, D, dtype=kv))


def _cw_call(lib, a, ks=1.0, vs=1.0):
    d = [binding.tensor_desc(a[n]) for n in ("key", "value", "slots", "kc", "vc")]
    return lib.paged_attn_cache_write(*[ctypes.byref(x) for x in d], ks, vs, None)


@pytest.mark.parametrize("mutate,expect", [
    (lambda a: a.update(key=a["key"].float()), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(slots=a["slots"].long()), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(slots=torch.zeros(3, dtype=torch.int32)), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(kc=torch.zeros(3, 8, 2, 64, dtype=torch.bfloat16)), binding.PA_ERR_UNSUPPORTED),
    (lambda a: a.update(kc=torch.zeros(3, 16, 4, 64, dtype=torch.bfloat16)), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(vc=torch.zeros(3, 16, 2, 64, dtype=torch.uint8)), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(key=torch.zeros(4, 2, 60, dtype=torch.bfloat16), value=torch.zeros(4, 2, 60, dtype=torch.bfloat16),
                        kc=torch.zeros(3, 16, 2, 60, dtype=torch.bfloat16), vc=torch.zeros(3, 16, 2, 60, dtype=torch.bfloat16)),
     binding.PA_ERR_UNSUPPORTED),
])
def test_cache_write_invalid_arguments(lib, mutate, expect):
    a = _cw_args()
    mutate(a)
    assert _cw_call(lib, a) == expect, binding.paged_attn_last_error_message()


def test_cache_write_fp8_needs_nonzero_scales(lib):
    a = _cw_args(kv=torch.uint8)
    assert _cw_call(lib, a, 0.0, 1.0) == binding.PA_ERR_INVALID_ARG


# ------------------------------------------------ per-token fp8 scales (host checks)

def _tok_call(lib, a, ks, vs):
    opts = binding.make_options(k_token_scales=ks, v_token_scales=vs)
    descs = [binding.tensor_desc(a[n]) for n in ("q", "k", "v", "bt", "sl", "qsl", "out", "lse")]
    refs = [ctypes.byref(d) for d in descs]
    return lib.paged_attn_decode_ex(*refs[:6], a["max_qlen"], 0.1, 1.0, 1.0, refs[6], refs[7], ctypes.byref(opts),
                                    None)


def _fp8_args():
    return _good_args(kv=torch.uint8)


@pytest.mark.parametrize("mutate,expect", [
    (lambda a, s: a.update(k=torch.zeros(10, 16, 2, 128, dtype=torch.bfloat16),
                           v=torch.zeros(10, 16, 2, 128, dtype=torch.bfloat16)), binding.PA_ERR_INVALID_ARG),  # bf16 cache
    (lambda a, s: s.update(ks=s["ks"].double()), binding.PA_ERR_INVALID_ARG),
    (lambda a, s: s.update(vs=torch.zeros(10, 2, 8)), binding.PA_ERR_INVALID_ARG),                   # shape
    (lambda a, s: s.update(ks=torch.zeros(9, 2, 16)), binding.PA_ERR_INVALID_ARG),                   # pages
    (lambda a, s: s.update(ks=torch.zeros(10, 16, 2).transpose(1, 2)), binding.PA_ERR_INVALID_ARG),  # layout
    (lambda a, s: s.update(vs=None), binding.PA_ERR_INVALID_ARG),                                    # only one
    (lambda a, s: s.update(ks=torch.zeros(10, 2, 17)[:, :, :16], vs=torch.zeros(10, 2, 17)[:, :, :16]),
     binding.PA_ERR_INVALID_ARG),                                                                    # head stride 17
])
def test_token_scale_arguments_rejected_on_host(lib, mutate, expect):
    a = _fp8_args()
    s = dict(ks=torch.zeros(10, 2, 16), vs=torch.zeros(10, 2, 16))
    mutate(a, s)
    assert _tok_call(lib, a, s["ks"], s["vs"]) == expect, binding.paged_attn_last_error_message()
    assert binding.paged_attn_last_error_message() != ""


def test_token_scales_pass_host_validation(lib):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _tok_call(lib, _fp8_args(), torch.zeros(10, 2, 16), torch.zeros(10, 2, 16)) == binding.PA_ERR_CUDA


def _cwt_call(lib, a, ks, vs):
    d = [binding.tensor_desc(t) for t in (a["key"], a["value"], a["slots"], a["kc"], a["vc"], ks, vs)]
    return lib.paged_attn_cache_write_per_token(*[ctypes.byref(x) for x in d], None)


def test_per_token_cache_write_arguments(lib):
    a = _cw_args(kv=torch.uint8)
    ok = torch.zeros(3, 2, 16)
    assert _cwt_call(lib, _cw_args(), ok, ok) == binding.PA_ERR_INVALID_ARG          # bf16 cache
    assert _cwt_call(lib, a, torch.zeros(3, 2, 8), ok) == binding.PA_ERR_INVALID_ARG  # scale shape
    assert _cwt_call(lib, a, ok, ok.double()) == binding.PA_ERR_INVALID_ARG          # scale dtype
    d = [binding.tensor_desc(t) for t in (a["key"], a["value"], a["slots"], a["kc"], a["vc"], ok)]
    assert lib.paged_attn_cache_write_per_token(*[ctypes.byref(x) for x in d], None, None) == binding.PA_ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert _cwt_call(lib, a, ok, ok) == binding.PA_ERR_CUDA


# ------------------------------------------------------------------ MLA decode

def _mla_args(T=3, Hq=16, NB=10, B=3, MB=4, kv=torch.bfloat16, Dqk=576, Dv=512):
    return dict(q=torch.zeros(T, Hq, Dqk, dtype=torch.bfloat16), c=torch.zeros(NB, 16, Dqk, dtype=kv),
                bt=torch.zeros(B, MB, dtype=torch.int32), sl=torch.ones(B, dtype=torch.int32), qsl=None,
                out=torch.zeros(T, Hq, Dv, dtype=torch.bfloat16), lse=torch.zeros(T, Hq, dtype=torch.float32),
                max_qlen=1, opts=None)


def _mla_call(lib, a, scale=0.07):
    descs = [binding.tensor_desc(a[n]) for n in ("q", "c", "bt", "sl", "qsl", "out", "lse")]
    refs = [ctypes.byref(d) for d in descs]
    if a["opts"] is None:
        return lib.paged_attn_mla_decode(*refs[:5], a["max_qlen"], scale, 1.0, refs[5], refs[6], None)
    return lib.paged_attn_mla_decode_ex(*refs[:5], a["max_qlen"], scale, 1.0, refs[5], refs[6],
                                        ctypes.byref(a["opts"]), None)


@pytest.mark.parametrize("mutate,expect", [
    (lambda a: a.update(q=a["q"].float()), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(out=torch.zeros(3, 16, 576, dtype=torch.bfloat16)), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(c=torch.zeros(10, 16, 1, 576, dtype=torch.bfloat16)), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(q=torch.zeros(3, 16, 512, dtype=torch.bfloat16),
                        c=torch.zeros(10, 16, 512, dtype=torch.bfloat16)), binding.PA_ERR_UNSUPPORTED),
    (lambda a: a.update(c=torch.zeros(10, 8, 576, dtype=torch.bfloat16)), binding.PA_ERR_UNSUPPORTED),
    (lambda a: a.update(c=torch.zeros(10, 16, 576, dtype=torch.float32)), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(q=torch.zeros(3, 16, 1152, dtype=torch.bfloat16)[:, :, :576]), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(c=torch.zeros(10, 16, 580, dtype=torch.bfloat16)[:, :, :576]), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(max_qlen=2), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(q=torch.zeros(33 * 3, 16, 576, dtype=torch.bfloat16),
                        out=torch.zeros(33 * 3, 16, 512, dtype=torch.bfloat16), lse=None,
                        qsl=torch.arange(0, 100, 33, dtype=torch.int32), max_qlen=33), binding.PA_ERR_UNSUPPORTED),
    (lambda a: a.update(opts=binding.make_options(sliding_window=8)), binding.PA_ERR_UNSUPPORTED),
    (lambda a: a.update(opts=binding.make_options(heads_per_cta=2)), binding.PA_ERR_UNSUPPORTED),
    (lambda a: a.update(opts=binding.make_options(use_tcgen05=3)), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(opts=binding.make_options(test_starve_cta=1)), binding.PA_ERR_UNSUPPORTED),
    (lambda a: a.update(opts=binding.make_options(use_tcgen05=2, segment_cost_pages=(1 << 20) + 1)),
     binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(opts=binding.make_options(wait_limit_us=-1)), binding.PA_ERR_INVALID_ARG),
    (lambda a: a.update(lse=torch.zeros(3, 8, dtype=torch.float32)), binding.PA_ERR_INVALID_ARG),
])
def test_mla_invalid_arguments_rejected_on_host(lib, mutate, expect):
    a = _mla_args()
    mutate(a)
    assert _mla_call(lib, a) == expect, binding.paged_attn_last_error_message()
    assert binding.paged_attn_last_error_message() != ""


def test_mla_non_finite_scale_rejected(lib):
    assert _mla_call(lib, _mla_args(), scale=float("inf")) == binding.PA_ERR_INVALID_ARG


def test_mla_valid_arguments_without_gpu_report_cuda_error(lib):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _mla_call(lib, _mla_args()) == binding.PA_ERR_CUDA
    a = _mla_args(kv=torch.float8_e4m3fn, T=6)
    a.update(qsl=torch.tensor([0, 1, 3, 6], dtype=torch.int32), max_qlen=3)
    assert _mla_call(lib, a) == binding.PA_ERR_CUDA


def test_mla_plan_rejects_bad_shapes_without_device(lib):
    for args, status in (((0, 16), binding.PA_ERR_UNSUPPORTED), ((4, 0), binding.PA_ERR_INVALID_ARG),
                         ((4, 16, 7), binding.PA_ERR_INVALID_ARG), ((4, 16, binding.PA_BF16, 33), binding.PA_ERR_UNSUPPORTED)):
        with pytest.raises(binding.PagedAttnError) as e:
            binding.paged_attn_mla_plan(*args)
        assert e.value.status == status
    with pytest.raises(binding.PagedAttnError) as e:
        binding.paged_attn_mla_reserve(4, 16, binding.PA_BF16, 0)
    assert e.value.status == binding.PA_ERR_INVALID_ARG



def _opt_call(lib, opts):
    a = _good_args()
    descs = [binding.tensor_desc(a[n]) for n in ("q", "k", "v", "bt", "sl", "qsl", "out", "lse")]
    refs = [ctypes.byref(d) for d in descs]
    return lib.paged_attn_decode_ex(*refs[:6], a["max_qlen"], 0.1, 1.0, 1.0, refs[6], refs[7], ctypes.byref(opts),
                                    None)


def test_wait_limit_and_starve_options_checked_on_the_host(lib):
    for bad in (binding.make_options(wait_limit_us=-5), binding.make_options(test_starve_cta=-1)):
        assert _opt_call(lib, bad) == binding.PA_ERR_INVALID_ARG
        assert "negative" in binding.paged_attn_last_error_message()
    if not torch.cuda.is_available():
        # valid values pass every host check; the call then fails at device set-up
        assert _opt_call(lib, binding.make_options(wait_limit_us=1000, test_starve_cta=3)) == binding.PA_ERR_CUDA


def test_options_struct_matches_the_header():
    """The binding's pa_options_t mirrors the header's fields, in order."""
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                            "paged_attn.h")).read()
    body = hdr[hdr.index("typedef struct pa_options_t {"):hdr.index("} pa_options_t;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = re.findall(r"\b(\w+);", body)
    assert names == [n for n, _ in binding.PaOptions._fields_]


class _NullStream:
    cuda_stream = 0


def test_prepared_calls_reach_the_host_checks(lib):
    """A prepared call passes its stored arguments in the entry point's order:
    an argument error is reported by the library's host checks (no device
    work), for decode and for MLA decode."""
    a = _good_args()
    call = binding.prepare_decode(a["q"].float(), a["k"], a["v"], a["bt"], a["sl"], None, 1, 0.1, 1.0, 1.0,
                                  out=a["out"], lse=a["lse"])
    with pytest.raises(binding.PagedAttnError) as e:
        call(stream=_NullStream())
    assert e.value.status == binding.PA_ERR_INVALID_ARG
    assert "q" in binding.paged_attn_last_error_message()
    call = binding.prepare_decode(a["q"], a["k"], a["v"], a["bt"], a["sl"], None, 2, 0.1, 1.0, 1.0,
                                  out=a["out"], lse=a["lse"], options=binding.make_options())
    with pytest.raises(binding.PagedAttnError) as e:
        call(stream=_NullStream())
    assert e.value.status == binding.PA_ERR_INVALID_ARG   # max_query_len 2 without query_start_loc
    m = _mla_args()
    call = binding.prepare_mla_decode(m["q"].float(), m["c"], m["bt"], m["sl"], None, 1, 0.07, 1.0,
                                      out=m["out"], lse=m["lse"])
    with pytest.raises(binding.PagedAttnError) as e:
        call(stream=_NullStream())
    assert e.value.status == binding.PA_ERR_INVALID_ARG
