"""paged_attn_decode_static_scratch: decode for callers that cannot allocate.

Some callers own all device memory through a pool, or run where allocation is
not allowed, so the library must not cudaMalloc its split scratch on their
behalf.  This entry point takes the scratch from a fixed 16 MiB device array
inside the library.  The test calls it through the C ABI twice in a row (the
second call finds the first call's data in the shared array) and checks each
result against the float64 oracle and against paged_attn_decode on the same
inputs, with the parity tolerances (out 1e-2 bf16 / 2e-2 fp8, lse 1e-3).  With
the library's own workspace released first, it checks that the calls left that
workspace empty: an ordinary call under stream capture, which may not allocate,
still finds no workspace.  It also checks that a shape needing more than 16 MiB
is refused on the host.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_06_gb300 import binding
from paged_kv_decode_06_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_OUT = {"bf16": 1e-2, "fp8": 2e-2}
TOL_LSE = 1e-3


def _device_args(w):
    dev = w.q.device
    bt = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    qsl = torch.from_numpy(w.query_start_loc).to(dev) if w.query_start_loc is not None else None
    mq = w.spec.max_query_len if qsl is not None else 1
    return bt, sl, qsl, mq


def _call(lib, fn_name, w, bt, sl, qsl, mq):
    s = w.spec
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device=w.q.device)
    descs = [binding.tensor_desc(t) for t in (w.q, w.k_cache, w.v_cache, bt, sl, qsl, out, lse)]
    refs = [ctypes.byref(d) for d in descs]
    stream = torch.cuda.current_stream().cuda_stream
    st = getattr(lib, fn_name)(*refs[:6], mq, s.scale, s.k_scale, s.v_scale, refs[6], refs[7], stream)
    assert st == binding.PA_OK, lib.paged_attn_last_error_message().decode()
    return out, lse


def test_static_scratch_matches_paged_attn_decode_on_two_calls_in_a_row(cuda_lib):
    lib = cuda_lib
    specs = [
        wl.custom_spec(num_q_heads=32, num_kv_heads=8, head_dim=128, kv_dtype="bf16",
                       seq_lens=(512, 4000, 77, 1500, 2048, 16, 900, 3300), seed=41),
        wl.custom_spec(num_q_heads=16, num_kv_heads=2, head_dim=128, kv_dtype="fp8",
                       seq_lens=(300, 33, 1200, 5), query_len_choices=(2, 3, 4), k_scale=0.05, v_scale=0.05,
                       fp8_source_scale=0.05, seed=42),
    ]
    works = [wl.make_workload(s, device="cuda") for s in specs]
    args = [_device_args(w) for w in works]
    oracle_ref = [oracle.run_workload(w) for w in works]
    binding.paged_attn_device_status(clear=True)
    binding.paged_attn_release()          # the library's own workspace: none from here on
    # two calls in a row through the static-scratch entry point
    got = [_call(lib, "paged_attn_decode_static_scratch", w, *a) for w, a in zip(works, args)]
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    _assert_no_library_workspace(lib, works[0], *args[0])
    # the same inputs through the ordinary entry point
    ref = [_call(lib, "paged_attn_decode", w, *a) for w, a in zip(works, args)]
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    for w, (o, l), (ro, rl), (oo, ol) in zip(works, got, ref, oracle_ref):
        assert torch.isfinite(o.float()).all() and torch.isfinite(l).all()
        tol = TOL_OUT[w.spec.kv_dtype]
        err_o = np.abs(o.float().cpu().numpy() - oo).max()
        err_l = np.abs(l.cpu().numpy() - ol).max()
        assert err_o <= tol, f"static scratch vs oracle: max|out| error {err_o:.3e}"
        assert err_l <= TOL_LSE, f"static scratch vs oracle: max|lse| error {err_l:.3e}"
        err_o = (o.float() - ro.float()).abs().max().item()
        err_l = (l - rl).abs().max().item()
        assert err_o <= tol, err_o
        assert err_l <= TOL_LSE, err_l


def _assert_no_library_workspace(lib, w, bt, sl, qsl, mq):
    """paged_attn_decode never allocates during stream capture: with no
    library workspace it returns PA_ERR_WORKSPACE before enqueueing anything."""
    s = w.spec
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device=w.q.device)
    descs = [binding.tensor_desc(t) for t in (w.q, w.k_cache, w.v_cache, bt, sl, qsl, out, lse)]
    refs = [ctypes.byref(d) for d in descs]
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        st = lib.paged_attn_decode(*refs[:6], mq, s.scale, s.k_scale, s.v_scale, refs[6], refs[7],
                                   stream.cuda_stream)
    assert st == binding.PA_ERR_WORKSPACE, (st, lib.paged_attn_last_error_message().decode())


def test_static_scratch_refuses_shapes_beyond_16_mib(cuda_lib):
    lib = cuda_lib
    spec = wl.CONFIGS["mtp"]          # 64 q heads over 8 KV heads, D 128, runs of up to 4 tokens
    need = binding.paged_attn_workspace_size(spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                                             binding.PA_BF16, spec.max_query_len)
    assert need > 16 * 2 ** 20
    B, T = spec.num_seqs, spec.num_seqs * 2
    q = torch.zeros(T, spec.num_q_heads, spec.head_dim, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(4, 16, spec.num_kv_heads, spec.head_dim, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    bt = torch.zeros(B, 1, dtype=torch.int32, device="cuda")
    sl = torch.full((B,), 2, dtype=torch.int32, device="cuda")
    qsl = torch.arange(0, T + 1, 2, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(T, spec.num_q_heads, dtype=torch.float32, device="cuda")
    descs = [binding.tensor_desc(t) for t in (q, k, v, bt, sl, qsl, out, lse)]
    refs = [ctypes.byref(d) for d in descs]
    st = lib.paged_attn_decode_static_scratch(*refs[:6], spec.max_query_len, spec.scale, 1.0, 1.0, refs[6], refs[7],
                                              torch.cuda.current_stream().cuda_stream)
    assert st == binding.PA_ERR_WORKSPACE
    msg = lib.paged_attn_last_error_message().decode()
    assert "16 MiB" in msg and str(need) in msg, msg
    torch.cuda.synchronize()
