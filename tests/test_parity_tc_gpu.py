"""The tcgen05 / tensor-memory split kernel against the float64 oracle.

It runs on its own above 64 query rows per KV head (bf16 caches, up to 128
rows: long verification runs or wide query groups), and on any bf16 shape
when forced with ``use_tcgen05=2``.  Same tolerances as the mma.sync kernel:
out 1e-2, lse 1e-3 (max absolute error)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_06_gb300 import binding
from paged_kv_decode_06_gb300 import workloads as wl

from test_parity_gpu import _check_opts, _sample_seqs, _spec, check, check_every_row

pytestmark = pytest.mark.gpu

FORCE = dict(use_tcgen05=2)


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    binding.paged_attn_device_status(clear=True)
    yield


def _plan(w, **kw):
    s = w.spec
    return binding.paged_attn_plan(s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim, binding.PA_BF16,
                                   s.max_query_len, options=binding.make_options(**kw))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G,Hkv,qlens", [(16, 2, (5, 6, 7, 8)), (8, 2, (9, 12, 16)), (32, 1, (3, 4)),
                                         (16, 1, (1, 8)), (128, 1, (1,)), (13, 2, (9,))])
def test_long_runs_select_the_tcgen05_kernel(D, G, Hkv, qlens):
    w = wl.make_workload(_spec(D=D, G=G, Hkv=Hkv, qlens=qlens, seq_lens=(9, 16, 17, 40, 130, 300), seed=G + D),
                         device="cuda")
    plan = _plan(w)
    assert plan["variant"] == 1 and plan["threads_per_cta"] == 384
    check(w)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G,Hkv,qlens", [(4, 2, (1,)), (8, 2, (2, 3, 4)), (1, 8, (1, 3)), (16, 1, (4,))])
def test_forced_on_short_groups(D, G, Hkv, qlens):
    w = wl.make_workload(_spec(D=D, G=G, Hkv=Hkv, qlens=qlens, seed=100 + G), device="cuda")
    assert _plan(w, **FORCE)["variant"] == 1
    check(w, options=binding.make_options(**FORCE))


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 64, 152, 300])
def test_forced_split_counts_exercise_the_merge(num_ctas):
    w = wl.make_workload(_spec(G=16, Hkv=2, qlens=(1, 5, 8), seq_lens=(3, 50, 300, 17, 1000), seed=num_ctas),
                         device="cuda")
    ref = oracle.run_workload(w)
    check(w, ref=ref, options=binding.make_options(num_ctas=num_ctas, min_pages_per_cta=1))


def test_both_kernels_on_the_same_inputs():
    w = wl.make_workload(_spec(G=8, Hkv=2, qlens=(2, 4), seq_lens=(700, 33, 1500), seed=5), device="cuda")
    ref = oracle.run_workload(w)
    assert _plan(w, use_tcgen05=1)["variant"] == 0 and _plan(w)["variant"] == 0
    check(w, ref=ref, options=binding.make_options(use_tcgen05=1))
    check(w, ref=ref, options=binding.make_options(**FORCE))


def test_non_finite_tail_slots_and_unused_pages_do_not_leak():
    w = wl.make_workload(_spec(G=16, Hkv=2, qlens=(1, 8), seq_lens=(3, 17, 40, 8)), device="cuda")
    ref = oracle.run_workload(w)
    nan = torch.tensor(float("nan")).to(torch.bfloat16)
    used = set()
    for i, L in enumerate(w.seq_lens):
        n = (int(L) + 15) // 16
        used.update(int(x) for x in w.block_tables[i, :n])
        last = int(w.block_tables[i, n - 1])
        tail = int(L) - 16 * (n - 1)
        w.k_cache[last, tail:] = nan
        w.v_cache[last, tail:] = nan
    for p in range(w.num_pages):
        if p not in used:
            w.k_cache[p] = nan
            w.v_cache[p] = nan
    check(w, ref=ref)


@pytest.mark.parametrize("window", [1, 5, 16, 17, 100])
def test_sliding_window(window):
    w = wl.make_workload(_spec(G=16, Hkv=2, qlens=(1, 4, 8), seq_lens=(8, 16, 17, 64, 250, 700), seed=window),
                         device="cuda")
    ref = oracle.run_workload(w, sliding_window=window)
    _check_opts(w, window=window, ref=ref)
    _check_opts(w, window=window, ref=ref, options_kw=dict(num_ctas=7, min_pages_per_cta=1))


@pytest.mark.parametrize("window", [0, 33])
@pytest.mark.parametrize("num_ctas", [0, 3, 64])
def test_attention_sinks(window, num_ctas):
    w = wl.make_workload(_spec(G=16, Hkv=2, qlens=(1, 6), seq_lens=(6, 20, 200, 900), seed=num_ctas + 2),
                         device="cuda")
    rng = np.random.default_rng(num_ctas)
    sinks = rng.normal(0, 2, size=32).astype(np.float32)
    sinks[3] = 30.0                                   # a sink that dominates its rows
    ref = oracle.run_workload(w, sliding_window=window, sinks=sinks)
    kw = dict(num_ctas=num_ctas, min_pages_per_cta=1) if num_ctas else None
    _check_opts(w, window=window, sinks=sinks, options_kw=kw, ref=ref)


def test_pages_before_the_window_are_never_read():
    w = wl.make_workload(_spec(G=16, Hkv=2, qlens=(8,), seq_lens=(300, 520, 77), seed=9), device="cuda")
    window = 40
    ref = oracle.run_workload(w, sliding_window=window)
    bt = w.block_tables.copy()
    for i, L in enumerate(w.seq_lens):
        first_page = max(0, int(L) - 8 - window + 1) // 16
        bt[i, :first_page] = w.num_pages + 1000          # out of range: reported if ever read
    w.block_tables = bt
    _check_opts(w, window=window, ref=ref)


def test_deterministic():
    w = wl.make_workload(_spec(G=16, Hkv=2, qlens=(3, 8), seq_lens=(500, 33, 1200, 64), seed=11), device="cuda")
    ref = oracle.run_workload(w)
    o1, l1, _, _ = check(w, ref=ref)
    o2, l2 = binding.decode_workload(w)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_out_of_range_page_id_is_reported():
    w = wl.make_workload(_spec(G=16, Hkv=2, qlens=(8,), seq_lens=(40, 20)), device="cuda")
    w.block_tables = w.block_tables.copy()
    w.block_tables[0, 1] = w.num_pages + 5
    binding.decode_workload(w)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) & binding.STATUS_PAGE_RANGE


def test_full_size_long_verification_every_row():
    w = wl.make_workload(wl.CONFIGS["verify8"], device="cuda")
    assert _plan(w)["variant"] == 1
    eo, el = check_every_row(w)
    print(f"verify8: all {w.q.shape[0]} query tokens: max|out err| {eo:.3e}, max|lse err| {el:.3e}")
