"""Every e4m3fn code through the fp8 decode kernels, checked one by one.

Each sequence holds one cached token, so out = v_scale * (its value row) and,
with a query head one-hot on feature d, lse = scale * k_scale * (key feature d).
Sequence i's cached row holds code (16 i + d + offset) mod 256 at feature d, so
16 sequences x 16 query heads probe all 256 codes as keys, and every value row
holds them all.  The NaN codes 0x7F / 0xFF are replaced by 0 in the probed row;
the page's other slots hold NaN codes, which must never be read.  Outputs and
logits are compared with the float64 oracle relative to their size (bf16
rounding of out, fp32 rounding of lse), so a wrong exponent, mantissa or sign of
any single code, down to the smallest subnormal, fails.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_06_gb300 import binding

pytestmark = pytest.mark.gpu

NAN_CODES = (0x7F, 0xFF)
SCALE, K_SCALE, V_SCALE = 0.125, 0.25, 3.0


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    binding.paged_attn_device_status(clear=True)
    yield


def _code_row(i, width, probe_shift=0):
    c = (16 * i + np.arange(width) + probe_shift) % 256
    c[np.isin(c, NAN_CODES)] = 0
    return c.astype(np.uint8)


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _compare(out, lse, ref_out, ref_lse):
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    assert np.all(np.abs(o - ref_out) <= 2.0 ** -8 * np.abs(ref_out))      # bf16 rounding of out
    assert np.all(np.abs(l - ref_lse) <= 1e-5 * np.abs(ref_lse) + 1e-12)   # fp32 rounding of lse


def test_grouped_query_kernel_every_code():
    B, Hq, D = 16, 16, 128
    k = np.full((B, 16, 1, D), 0x7F, np.uint8)
    v = np.full((B, 16, 1, D), 0xFF, np.uint8)
    for i in range(B):
        k[i, 0, 0] = _code_row(i, D)
        v[i, 0, 0] = _code_row(i, D, probe_shift=7)
    q = np.zeros((B, Hq, D), np.float32)
    for h in range(Hq):
        q[:, h, h] = 1.0                          # head h reads key feature h: code 16 i + h
    qt = torch.from_numpy(q).to(torch.bfloat16)
    bt = np.arange(B, dtype=np.int32).reshape(B, 1)
    sl = np.ones(B, np.int32)
    ref_out, ref_lse = oracle.paged_decode_attention(_bits(qt), k, v, bt, sl, None, SCALE, K_SCALE, V_SCALE, "fp8")
    out, lse = binding.paged_attn_decode(qt.cuda(), torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                                         torch.from_numpy(bt).cuda(), torch.from_numpy(sl).cuda(), None, 1, SCALE,
                                         K_SCALE, V_SCALE)
    _compare(out, lse, ref_out, ref_lse)


def test_mla_kernel_every_code():
    B, Hq, W = 16, 16, 576
    c = np.full((B, 16, W), 0x7F, np.uint8)
    q = np.zeros((B, Hq, W), np.float32)
    for i in range(B):
        c[i, 0] = _code_row(i, W)
        # even sequences probe features 0-15, odd ones 128-143 (the last Q K^T
        # k-step of a column quarter); together they read all 256 codes
        d0 = 128 * (i % 2)
        for h in range(Hq):
            q[i, h, d0 + h] = 1.0
    qt = torch.from_numpy(q).to(torch.bfloat16)
    bt = np.arange(B, dtype=np.int32).reshape(B, 1)
    sl = np.ones(B, np.int32)
    qsl = np.arange(B + 1, dtype=np.int32)
    ref_out, ref_lse = oracle.mla_decode(_bits(qt), c, bt, sl, qsl, SCALE, K_SCALE, "fp8")
    out, lse = binding.paged_attn_mla_decode(qt.cuda(), torch.from_numpy(c).cuda(), torch.from_numpy(bt).cuda(),
                                             torch.from_numpy(sl).cuda(), torch.from_numpy(qsl).cuda(), 1, SCALE,
                                             K_SCALE)
    _compare(out, lse, ref_out, ref_lse)


def test_probe_layout_covers_every_code():
    """Host-side check of the probe layout itself (runs with the GPU tests)."""
    gqa = {int(_code_row(i, 128)[h]) for i in range(16) for h in range(16)}
    mla = {int(_code_row(i, 576)[128 * (i % 2) + h]) for i in range(16) for h in range(16)}
    every = set(range(256)) - set(NAN_CODES)
    assert every <= gqa and every <= mla
