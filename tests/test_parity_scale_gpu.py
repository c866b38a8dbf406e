"""Softmax scales other than 1/sqrt(D) on every kernel: a negative scale, a
zero scale (uniform weights: out = mean of the visible value rows, lse = ln of
their count) and a large positive one.  The kernels fold a positive scale into
the exponent and scale first otherwise, so both branches are compared with the
float64 oracle run at the same scale.  Tolerances as elsewhere: out 1e-2 (bf16
caches) / 2e-2 (fp8), lse 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_06_gb300 import binding
from paged_kv_decode_06_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_OUT = {"bf16": 1e-2, "fp8": 2e-2}
TOL_LSE = 1e-3
SCALES = [-0.07, 0.0, 0.3]


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    binding.paged_attn_device_status(clear=True)
    yield


def _compare(kv, out, lse, ref):
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(l).all()
    assert np.abs(o - ref[0]).max() <= TOL_OUT[kv]
    assert np.abs(l - ref[1]).max() <= TOL_LSE


def _gqa(kv, scale, G, Hkv, qlens, options=None, per_token=False):
    fp8 = kv == "fp8"
    spec = wl.custom_spec(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=128, kv_dtype=kv,
                          seq_lens=(1, 17, 40, 130), query_len_choices=qlens,
                          k_scale=(1.0 if per_token else 0.05) if fp8 else 1.0,
                          v_scale=(1.0 if per_token else 0.05) if fp8 else 1.0,
                          fp8_source_scale=(1 / 128 if per_token else 0.05) if fp8 else 1.0,
                          token_scale_range=(0.25 / 128, 1 / 128) if per_token else None, seed=77)
    w = wl.make_workload(spec, device="cuda")
    q, k, v = wl.host_arrays(w)
    ks, vs = wl.host_token_scales(w)
    ref = oracle.paged_decode_attention(q, k, v, w.block_tables, w.seq_lens, w.query_start_loc, scale, spec.k_scale,
                                        spec.v_scale, kv, k_token_scales=ks, v_token_scales=vs)
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    qsl = torch.from_numpy(w.query_start_loc).cuda() if w.query_start_loc is not None else None
    if per_token:
        options = binding.make_options(k_token_scales=w.k_token_scales, v_token_scales=w.v_token_scales)
    out, lse = binding.paged_attn_decode(w.q, w.k_cache, w.v_cache, bt, sl, qsl,
                                         spec.max_query_len if qsl is not None else 1, scale, spec.k_scale,
                                         spec.v_scale, options=options)
    _compare(kv, out, lse, ref)


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_split_kernel_scales(kv, scale):
    _gqa(kv, scale, G=4, Hkv=2, qlens=(1, 3))


@pytest.mark.parametrize("scale", SCALES)
def test_per_token_fp8_scales(scale):
    _gqa("fp8", scale, G=4, Hkv=2, qlens=(1, 2), per_token=True)


@pytest.mark.parametrize("scale", SCALES)
def test_tcgen05_kernel_scales(scale):
    _gqa("bf16", scale, G=16, Hkv=2, qlens=(5, 8))


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_mla_kernel_scales(kv, scale):
    fp8 = kv == "fp8"
    spec = wl.custom_mla_spec(num_q_heads=16, kv_dtype=kv, seq_lens=(1, 17, 40, 130), query_len_choices=(1, 4),
                              kv_scale=0.05 if fp8 else 1.0, fp8_source_scale=0.05 if fp8 else 1.0, seed=78)
    w = wl.make_mla_workload(spec, device="cuda")
    qb, c = wl.host_mla_arrays(w)
    ref = oracle.mla_decode(qb, c, w.block_tables, w.seq_lens, w.query_start_loc, scale, spec.kv_scale, kv)
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    qsl = torch.from_numpy(w.query_start_loc).cuda()
    out, lse = binding.paged_attn_mla_decode(w.q, w.kv_cache, bt, sl, qsl, spec.max_query_len, scale, spec.kv_scale)
    _compare(kv, out, lse, ref)
