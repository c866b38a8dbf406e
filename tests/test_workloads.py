"""The seeded input generator: reproducible, shaped like the decode regimes,
and a valid page pool (every used page id distinct and in range)."""
import numpy as np
import pytest
import torch

from paged_kv_decode_06_gb300 import workloads as wl


@pytest.mark.parametrize("name", wl.CONFIG_ORDER)
def test_metadata_is_valid(name):
    spec = wl.CONFIGS[name]
    sl, ql, qsl, bt, pool = wl.draw_metadata(spec, np.random.default_rng(spec.seed))
    B = spec.num_seqs
    assert sl.shape == (B,) and ql.shape == (B,) and bt.shape[0] == B
    assert (ql >= 1).all() and (sl >= ql).all()
    n = (sl + 15) // 16
    used = np.concatenate([bt[i, :n[i]] for i in range(B)])
    assert len(np.unique(used)) == len(used)
    assert used.min() >= 0 and used.max() < pool
    for i in range(B):
        assert (bt[i, n[i]:] == -1).all()
    if qsl is None:
        assert (ql == 1).all()
    else:
        assert qsl[0] == 0 and (np.diff(qsl) == ql).all()
    if spec.seq_len_kind in ("uniform", "loguniform"):
        lo, hi = spec.seq_len_args
        assert sl.min() >= lo and sl.max() <= hi
    if spec.pool_pages is None:
        assert pool == int(np.ceil(1.1 * n.sum()))


def test_tiny_config_matches_its_description():
    w = wl.make_workload(wl.CONFIGS["tiny"])
    assert list(w.seq_lens) == [1, 17, 64, 200]
    assert w.num_pages == 64 and w.q.shape == (4, 8, 128)
    assert w.k_cache.shape == (64, 16, 2, 128) and w.k_cache.dtype == torch.bfloat16


def test_reproducible_and_seed_sensitive():
    spec = wl.custom_spec(seq_lens=(5, 40, 17))
    a = wl.make_workload(spec)
    b = wl.make_workload(spec)
    c = wl.make_workload(spec, seed=spec.seed + 1)
    assert torch.equal(a.q, b.q) and torch.equal(a.k_cache, b.k_cache)
    assert np.array_equal(a.block_tables, b.block_tables)
    assert not torch.equal(a.k_cache, c.k_cache)


def test_fp8_codes_are_finite_and_spread():
    spec = wl.custom_spec(kv_dtype="fp8", seq_lens=(300,), fp8_source_scale=0.05,
                          k_scale=0.05, v_scale=0.05)
    w = wl.make_workload(spec)
    vals = w.k_cache.view(torch.float8_e4m3fn).to(torch.float32)
    assert torch.isfinite(vals).all()
    assert 15 < vals.std().item() < 25          # N(0,1)/0.05
    assert w.k_cache.dtype == torch.uint8


def test_kv_bytes_counts_every_cached_token_once():
    w = wl.make_workload(wl.CONFIGS["tiny"])
    assert w.kv_bytes() == 282 * 2 * 128 * 2 * 2


@pytest.mark.parametrize("name", sorted(wl.MLA_CONFIGS))
def test_mla_metadata_and_shapes(name):
    spec = wl.MLA_CONFIGS[name]
    sl, ql, qsl, bt, pool = wl.draw_metadata(spec, np.random.default_rng(spec.seed))
    n = (sl + 15) // 16
    used = np.concatenate([bt[i, :n[i]] for i in range(spec.num_seqs)])
    assert len(np.unique(used)) == len(used) and used.max() < pool
    assert (sl >= ql).all() and (ql <= spec.max_query_len).all()
    assert spec.head_dim == spec.kv_lora_rank + spec.rope_dim == 576
    assert abs(spec.scale - 192 ** -0.5) < 1e-15


def test_mla_workload_is_reproducible_and_laid_out():
    spec = wl.MLA_CONFIGS["mla_tiny"]
    a, b = wl.make_mla_workload(spec), wl.make_mla_workload(spec)
    assert torch.equal(a.q, b.q) and torch.equal(a.kv_cache, b.kv_cache)
    assert a.q.shape == (4, 16, 576) and a.kv_cache.shape == (64, 16, 576)
    assert a.kv_bytes() == int(a.seq_lens.sum()) * 576 * 2
    f = wl.make_mla_workload(wl.custom_mla_spec(kv_dtype="fp8", kv_scale=0.05, fp8_source_scale=0.05))
    assert f.kv_cache.dtype == torch.uint8 and f.kv_bytes() == int(f.seq_lens.sum()) * 576
    codes = f.kv_cache.flatten()
    assert not ((codes & 0x7F) == 0x7F).any()          # no NaN codes
