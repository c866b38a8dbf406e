"""Pins for the MLA decode oracle (``oracle/mla.py``): a library attention
routine on a contiguous latent cache gathered by a different route, closed
forms (a zero query, a key planted through the rotary part alone, a constant
latent), the causal rows of a verification run against single-token decodes
of their prefixes, page-permutation invariance, fp8 decoded by torch's own
e4m3fn conversion, and agreement with the grouped-query oracle run with one KV
head.  CPU only."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_06_gb300 import workloads as wl


def _spec(qlens=(1,), seq_lens=(3, 16, 17, 50, 97), kv_dtype="bf16", Hq=4, rank=512, rope=64, seed=31):
    return wl.custom_mla_spec(num_q_heads=Hq, kv_dtype=kv_dtype, seq_lens=seq_lens, query_len_choices=qlens,
                              kv_scale=0.05 if kv_dtype == "fp8" else 1.0,
                              fp8_source_scale=0.05 if kv_dtype == "fp8" else 1.0, seed=seed,
                              kv_lora_rank=rank, rope_dim=rope)


def _run(w, q_bits=None, cache=None, block_tables=None):
    qb, c = wl.host_mla_arrays(w)
    s = w.spec
    return oracle.mla_decode(qb if q_bits is None else q_bits, c if cache is None else cache,
                             w.block_tables if block_tables is None else block_tables, w.seq_lens,
                             w.query_start_loc, s.scale, s.kv_scale, s.kv_dtype, s.kv_lora_rank)


def _torch_reference(w):
    """Pages indexed with the whole block-table row and reshaped into one
    contiguous [L, Dqk] cache per sequence; fp8 decoded by torch's e4m3fn
    conversion; float64 SDPA with the latent part as the value and an explicit
    causal mask."""
    s = w.spec
    if s.kv_dtype == "fp8":
        c = w.kv_cache.view(torch.float8_e4m3fn).to(torch.float64) * float(np.float32(s.kv_scale))
    else:
        c = w.kv_cache.to(torch.float64)
    q = w.q.to(torch.float64)
    qsl = w.query_start_loc if w.query_start_loc is not None else np.arange(s.num_seqs + 1)
    T, Hq, _ = q.shape
    out = torch.empty((T, Hq, s.kv_lora_rank), dtype=torch.float64)
    lse = torch.empty((T, Hq), dtype=torch.float64)
    scale = float(np.float32(s.scale))
    for i in range(s.num_seqs):
        L = int(w.seq_lens[i])
        n = (L + 15) // 16
        pages = torch.from_numpy(w.block_tables[i, :n].astype(np.int64))
        C = c[pages].reshape(n * 16, s.head_dim)[:L]
        K = C.unsqueeze(0).expand(Hq, L, s.head_dim)
        V = C[:, :s.kv_lora_rank].unsqueeze(0).expand(Hq, L, s.kv_lora_rank)
        t0, t1 = int(qsl[i]), int(qsl[i + 1])
        qn = t1 - t0
        Q = q[t0:t1].permute(1, 0, 2)
        mask = torch.arange(L)[None, :] <= (L - qn + torch.arange(qn))[:, None]
        out[t0:t1] = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask,
                                                                      scale=scale).permute(1, 0, 2)
        logits = (scale * (Q @ K.transpose(1, 2))).masked_fill(~mask, float("-inf"))
        lse[t0:t1] = torch.logsumexp(logits, dim=-1).permute(1, 0)
    return out.numpy(), lse.numpy()


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("qlens", [(1,), (2, 3, 4), (4,)])
def test_mla_oracle_matches_sdpa(kv_dtype, qlens):
    w = wl.make_mla_workload(_spec(qlens=qlens, kv_dtype=kv_dtype))
    out, lse = _run(w)
    ref_out, ref_lse = _torch_reference(w)
    assert np.abs(out - ref_out).max() < 1e-12
    assert np.abs(lse - ref_lse).max() < 1e-12


def test_mla_zero_query_gives_mean_latent_and_log_length():
    w = wl.make_mla_workload(_spec(seq_lens=(1, 9, 40), rank=32, rope=16))
    qb, c = wl.host_mla_arrays(w)
    out, lse = _run(w, q_bits=np.zeros_like(qb))
    for i, L in enumerate(w.seq_lens):
        L = int(L)
        rows = []
        for j in range(L):
            rows.append(oracle.bf16_bits_to_float64(c[w.block_tables[i, j // 16], j % 16, :32]))
        mean = np.mean(rows, axis=0)
        assert np.abs(out[i] - mean[None, :]).max() < 1e-12
        assert np.abs(lse[i] - np.log(L)).max() < 1e-12


def test_mla_rotary_part_alone_selects_a_planted_key():
    # the query's latent part is zero, so only the rotary part of each key can
    # raise its logit: a key whose rotary part matches the query's wins.
    rank, rope = 32, 16
    w = wl.make_mla_workload(_spec(seq_lens=(37,), Hq=2, rank=rank, rope=rope))
    qb, c = wl.host_mla_arrays(w)
    qb = qb.copy()
    c = c.copy()
    one = np.uint16(0x3F80)          # bf16 1.0
    qb[:, :, :rank] = 0
    qb[:, :, rank:] = one
    c[:, :, rank:] = 0
    j = 23
    c[w.block_tables[0, j // 16], j % 16, rank:] = np.uint16(0x4120)   # bf16 10.0
    out, lse = _run(w, q_bits=qb, cache=c)
    planted = oracle.bf16_bits_to_float64(c[w.block_tables[0, j // 16], j % 16, :rank])
    logit = np.float64(np.float32(w.spec.scale)) * 10.0 * rope
    # every other key has logit 0: out = (e^logit * planted + sum of others) / (e^logit + 36)
    others = [oracle.bf16_bits_to_float64(c[w.block_tables[0, k // 16], k % 16, :rank]) for k in range(37) if k != j]
    expect = (np.exp(logit) * planted + np.sum(others, axis=0)) / (np.exp(logit) + 36.0)
    assert np.abs(out[0] - expect[None, :]).max() < 1e-12
    assert np.abs(lse[0] - np.log(np.exp(logit) + 36.0)).max() < 1e-12


def test_mla_constant_latent_returns_it_whatever_the_rotary_keys():
    rank, rope = 32, 16
    w = wl.make_mla_workload(_spec(qlens=(1, 2), seq_lens=(5, 33, 70), rank=rank, rope=rope))
    qb, c = wl.host_mla_arrays(w)
    c = c.copy()
    v = (np.arange(rank) % 7 - 3).astype(np.float32) * 0.25        # exact in bf16
    c[:, :, :rank] = (v.view(np.uint32) >> 16).astype(np.uint16)[None, None, :]
    out, _ = _run(w, cache=c)
    assert np.abs(out - v.astype(np.float64)[None, None, :]).max() < 1e-12


def test_mla_verification_rows_equal_prefix_decodes():
    w = wl.make_mla_workload(_spec(qlens=(4,), seq_lens=(6, 31, 64), rank=64, rope=16))
    out, lse = _run(w)
    qb, c = wl.host_mla_arrays(w)
    s = w.spec
    for i in range(s.num_seqs):
        L = int(w.seq_lens[i])
        for r in range(4):
            t = int(w.query_start_loc[i]) + r
            o1, l1 = oracle.mla_decode(qb[t:t + 1], c, w.block_tables[i:i + 1], np.array([L - 4 + r + 1]), None,
                                       s.scale, s.kv_scale, s.kv_dtype, s.kv_lora_rank)
            assert np.abs(o1[0] - out[t]).max() < 1e-12
            assert np.abs(l1[0] - lse[t]).max() < 1e-12


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_mla_page_permutation_invariance_bit_exact(kv_dtype):
    w = wl.make_mla_workload(_spec(qlens=(1, 3), seq_lens=(3, 16, 40), kv_dtype=kv_dtype, rank=64, rope=16))
    out, lse = _run(w)
    qb, c = wl.host_mla_arrays(w)
    perm = np.random.default_rng(9).permutation(w.num_pages)
    c2 = np.empty_like(c)
    c2[perm] = c
    bt2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out2, lse2 = _run(w, cache=c2, block_tables=bt2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_mla_agrees_with_the_grouped_query_oracle_on_one_kv_head(kv_dtype):
    # one KV head whose K and V are both the whole latent row: the grouped
    # oracle's output restricted to the latent columns is the MLA output
    w = wl.make_mla_workload(_spec(qlens=(1, 2), seq_lens=(2, 18, 45), kv_dtype=kv_dtype, rank=64, rope=16))
    out, lse = _run(w)
    qb, c = wl.host_mla_arrays(w)
    s = w.spec
    kc = c[:, :, None, :]
    g_out, g_lse = oracle.paged_decode_attention(qb, kc, kc, w.block_tables, w.seq_lens, w.query_start_loc, s.scale,
                                                 s.kv_scale, s.kv_scale, kv_dtype)
    assert np.abs(out - g_out[:, :, :s.kv_lora_rank]).max() < 1e-12
    assert np.abs(lse - g_lse).max() < 1e-12
