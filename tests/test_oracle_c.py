"""The plain-C float64 oracle (used for the timed CPU baseline) against the
pinned NumPy oracle: same inputs, agreement to 1e-11 on every output element
(the two differ only in summation order), over both cache dtypes, per-token
scales, ragged MTP runs, sliding windows, sinks and both head sizes; and the
result does not depend on the OpenMP thread count.  CPU only."""
import numpy as np
import pytest

import oracle
from oracle import c_oracle
from paged_kv_decode_06_gb300 import workloads as wl


def _w(kv="bf16", D=64, G=4, Hkv=2, qlens=(1,), seq_lens=(1, 15, 16, 17, 33, 100), per_token=False, seed=5):
    fp8 = kv == "fp8"
    return wl.make_workload(wl.custom_spec(
        num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, kv_dtype=kv, seq_lens=seq_lens, query_len_choices=qlens,
        k_scale=(1.0 if per_token else 0.05) if fp8 else 1.0, v_scale=(1.0 if per_token else 0.07) if fp8 else 1.0,
        fp8_source_scale=(1 / 128 if per_token else 0.05) if fp8 else 1.0,
        token_scale_range=(0.25 / 128, 1 / 128) if per_token else None, seed=seed))


def _agree(w, **kw):
    a = oracle.run_workload(w, **kw)
    b = c_oracle.run_workload(w, **kw)
    assert np.abs(a[0] - b[0]).max() < 1e-11 and np.abs(a[1] - b[1]).max() < 1e-11


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("qlens", [(1,), (2, 3, 4)])
def test_c_oracle_matches_numpy_oracle(kv, D, qlens):
    _agree(_w(kv=kv, D=D, qlens=qlens, seed=D + len(qlens)))


def test_c_oracle_per_token_scales():
    _agree(_w(kv="fp8", per_token=True, qlens=(1, 2), seed=9))


@pytest.mark.parametrize("window", [1, 5, 17, 40])
def test_c_oracle_sliding_window_and_sinks(window):
    w = _w(G=8, qlens=(1, 3), seq_lens=(1, 20, 70, 130), seed=window)
    sinks = np.random.default_rng(window).normal(0, 2, size=16).astype(np.float32)
    _agree(w, sliding_window=window)
    _agree(w, sinks=sinks)
    _agree(w, sliding_window=window, sinks=sinks)


def test_c_oracle_sampled_sequences_and_thread_counts():
    w = _w(G=8, Hkv=2, seq_lens=(3, 90, 17, 250, 64), seed=4)
    a = c_oracle.run_workload(w, seqs=[1, 3], threads=1)
    b = c_oracle.run_workload(w, seqs=[1, 3], threads=max(2, c_oracle.max_threads()))
    assert np.array_equal(a[0], b[0], equal_nan=True) and np.array_equal(a[1], b[1], equal_nan=True)
    assert np.isnan(a[0][0]).all() and np.isfinite(a[0][1]).all()
    ref = oracle.run_workload(w, seqs=[1, 3])
    assert np.abs(a[0][[1, 3]] - ref[0][[1, 3]]).max() < 1e-11


# ------------------------------------------------------------------ MLA

@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("qlens", [(1,), (2, 3, 4)])
def test_c_mla_oracle_matches_numpy_oracle(kv, qlens):
    fp8 = kv == "fp8"
    w = wl.make_mla_workload(wl.custom_mla_spec(num_q_heads=4, kv_dtype=kv, seq_lens=(1, 16, 17, 60),
                                                query_len_choices=qlens, kv_scale=0.05 if fp8 else 1.0,
                                                fp8_source_scale=0.05 if fp8 else 1.0, seed=len(qlens) + 3))
    a = oracle.run_mla_workload(w)
    b = c_oracle.run_mla_workload(w)
    assert np.abs(a[0] - b[0]).max() < 1e-11 and np.abs(a[1] - b[1]).max() < 1e-11
    c = c_oracle.run_mla_workload(w, threads=1)
    assert np.array_equal(b[0], c[0]) and np.array_equal(b[1], c[1])
