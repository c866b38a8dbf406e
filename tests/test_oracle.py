"""Pins for the float64 oracle, against things other than itself: the bf16 and
OCP e4m3 encodings, a library attention routine on independently gathered
contiguous KV, closed forms, invariants and brute force on tiny inputs."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_06_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_points(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append((int(parts[0], 16), float(parts[1])))
    return rows


# ---------------------------------------------------------------- encodings

def test_bf16_golden_points():
    for bits, value in _read_points("bf16_points.txt"):
        got = oracle.bf16_bits_to_float64(np.array([bits], dtype=np.uint16))[0]
        assert got == value and math.copysign(1, got) == math.copysign(1, value), (hex(bits), got)


def test_bf16_decode_matches_torch_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_bits_to_float64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_golden_points():
    for code, value in _read_points("e4m3fn_points.txt"):
        got = oracle.e4m3fn_to_float64(np.array([code], dtype=np.uint8))[0]
        if math.isnan(value):
            assert math.isnan(got), hex(code)
        else:
            assert got == value and math.copysign(1, got) == math.copysign(1, value), (hex(code), got)


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3fn_to_float64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_fp8_scale_is_fp32_rounded():
    # the kernel receives k_scale as float32; 0.05 is not a float32 number
    x = oracle.dequantize(np.array([0x38], dtype=np.uint8), "fp8", 0.05)[0]
    assert x == float(np.float32(0.05)) and x != 0.05


# ---------------------------------------------------------- brute force

def _torch_reference(w, window=0):
    """Attention recomputed from scratch with torch: pages reshaped into a
    contiguous cache (a different indexing route from the oracle's per-token
    gather), K/V heads repeated per group, and the library's float64
    scaled_dot_product_attention with an explicit boolean causal mask."""
    s = w.spec
    G = s.group_size
    if s.kv_dtype == "fp8":
        kc = w.k_cache.view(torch.float8_e4m3fn).to(torch.float64) * float(np.float32(s.k_scale))
        vc = w.v_cache.view(torch.float8_e4m3fn).to(torch.float64) * float(np.float32(s.v_scale))
    else:
        kc = w.k_cache.to(torch.float64)
        vc = w.v_cache.to(torch.float64)
    q = w.q.to(torch.float64)
    qsl = w.query_start_loc if w.query_start_loc is not None else np.arange(s.num_seqs + 1)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float64)
    scale = float(np.float32(s.scale))
    for i in range(s.num_seqs):
        L = int(w.seq_lens[i])
        n = (L + 15) // 16
        pages = torch.from_numpy(w.block_tables[i, :n].astype(np.int64))
        K = kc[pages].reshape(n * 16, s.num_kv_heads, s.head_dim)[:L]
        V = vc[pages].reshape(n * 16, s.num_kv_heads, s.head_dim)[:L]
        K = K.repeat_interleave(G, dim=1).permute(1, 0, 2)        # [Hq, L, D]
        V = V.repeat_interleave(G, dim=1).permute(1, 0, 2)
        t0, t1 = int(qsl[i]), int(qsl[i + 1])
        Q = q[t0:t1].permute(1, 0, 2)                              # [Hq, qn, D]
        qn = t1 - t0
        lim = (L - qn + torch.arange(qn))[:, None]
        mask = torch.arange(L)[None, :] <= lim
        if window > 0:
            mask &= torch.arange(L)[None, :] > lim - window
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
        out[t0:t1] = o.permute(1, 0, 2)
        logits = scale * (Q @ K.transpose(1, 2))
        logits = logits.masked_fill(~mask, float("-inf"))
        lse[t0:t1] = torch.logsumexp(logits, dim=-1).permute(1, 0)
    return out.numpy(), lse.numpy()


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("qlens", [(1,), (2, 3, 4)])
def test_oracle_matches_sdpa_on_contiguous_kv(kv_dtype, qlens):
    spec = wl.custom_spec(num_q_heads=8, num_kv_heads=2, head_dim=64,
                          kv_dtype=kv_dtype, seq_lens=(4, 16, 17, 50, 97),
                          query_len_choices=qlens, k_scale=0.05 if kv_dtype == "fp8" else 1.0,
                          v_scale=0.07 if kv_dtype == "fp8" else 1.0,
                          fp8_source_scale=0.05 if kv_dtype == "fp8" else 1.0, seed=11)
    w = wl.make_workload(spec)
    out, lse = oracle.run_workload(w)
    ref_out, ref_lse = _torch_reference(w)
    assert np.abs(out - ref_out).max() < 1e-12
    assert np.abs(lse - ref_lse).max() < 1e-12


def test_oracle_matches_sdpa_tiny_config():
    w = wl.make_workload(wl.CONFIGS["tiny"])
    out, lse = oracle.run_workload(w)
    ref_out, ref_lse = _torch_reference(w)
    assert np.abs(out - ref_out).max() < 1e-12
    assert np.abs(lse - ref_lse).max() < 1e-12


# ---------------------------------------------------------- invariants

def _small(kv_dtype="bf16", qlens=(1,), seq_lens=(3, 16, 40), seed=5, G=2, Hkv=2, D=32):
    spec = wl.custom_spec(num_q_heads=G * Hkv, num_kv_heads=Hkv,
                          head_dim=D, kv_dtype=kv_dtype, seq_lens=seq_lens,
                          query_len_choices=qlens, seed=seed,
                          k_scale=0.05 if kv_dtype == "fp8" else 1.0,
                          v_scale=0.05 if kv_dtype == "fp8" else 1.0,
                          fp8_source_scale=0.05 if kv_dtype == "fp8" else 1.0)
    return wl.make_workload(spec)


def _call(w, q=None, k=None, v=None, bt=None, seq_lens=None, scale=None, k_scale=None, v_scale=None):
    q0, k0, v0 = wl.host_arrays(w)
    s = w.spec
    return oracle.paged_decode_attention(
        q0 if q is None else q, k0 if k is None else k, v0 if v is None else v,
        w.block_tables if bt is None else bt, w.seq_lens if seq_lens is None else seq_lens,
        w.query_start_loc, s.scale if scale is None else scale,
        s.k_scale if k_scale is None else k_scale, s.v_scale if v_scale is None else v_scale,
        s.kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_page_permutation_invariance_bit_exact(kv_dtype):
    w = _small(kv_dtype, qlens=(1, 2))
    out, lse = _call(w)
    _, k, v = wl.host_arrays(w)
    rng = np.random.default_rng(3)
    perm = rng.permutation(w.num_pages)          # new location of old page p is perm[p]
    k2 = np.empty_like(k); v2 = np.empty_like(v)
    k2[perm] = k; v2[perm] = v
    bt2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out2, lse2 = _call(w, k=k2, v=v2, bt=bt2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_constant_v_returns_v():
    w = _small()
    q, k, v = wl.host_arrays(w)
    row = torch.randn(w.spec.head_dim, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    bits = row.view(torch.int16).numpy().view(np.uint16)
    v2 = np.broadcast_to(bits, v.shape).copy()
    out, _ = _call(w, v=v2)
    expect = oracle.bf16_bits_to_float64(bits)
    assert np.abs(out - expect[None, None, :]).max() <= 1e-14 * np.abs(expect).max()


def test_length_one_returns_first_value_row():
    w = _small(seq_lens=(1, 1, 1))
    q, k, v = wl.host_arrays(w)
    out, lse = _call(w)
    G = w.spec.group_size
    for i in range(3):
        page = w.block_tables[i, 0]
        for hq in range(w.spec.num_q_heads):
            hk = hq // G
            vrow = oracle.bf16_bits_to_float64(v[page, 0, hk])
            krow = oracle.bf16_bits_to_float64(k[page, 0, hk])
            qrow = oracle.bf16_bits_to_float64(q[i, hq])
            assert np.array_equal(out[i, hq], vrow)
            s0 = float(np.float32(w.spec.scale)) * float(qrow @ krow)
            assert abs(lse[i, hq] - s0) < 1e-12


def test_zero_query_gives_mean_value_and_log_length():
    w = _small(seq_lens=(5, 16, 37))
    q, k, v = wl.host_arrays(w)
    out, lse = _call(w, q=np.zeros_like(q))
    G = w.spec.group_size
    for i, L in enumerate(w.seq_lens):
        assert np.allclose(lse[i], math.log(L), atol=1e-13, rtol=0)
        for hq in range(w.spec.num_q_heads):
            V = oracle.dequantize(oracle.gather_sequence(v, w.block_tables[i], int(L), hq // G), "bf16", 1.0)
            assert np.abs(out[i, hq] - V.mean(axis=0)).max() < 1e-13


def test_equal_keys_give_uniform_average():
    w = _small(seq_lens=(7, 23, 33))
    q, k, v = wl.host_arrays(w)
    k2 = np.broadcast_to(k[0, 0, 0], k.shape).copy()
    out, _ = _call(w, k=k2)
    G = w.spec.group_size
    for i, L in enumerate(w.seq_lens):
        for hq in range(w.spec.num_q_heads):
            V = oracle.dequantize(oracle.gather_sequence(v, w.block_tables[i], int(L), hq // G), "bf16", 1.0)
            assert np.abs(out[i, hq] - V.mean(axis=0)).max() < 1e-13


def test_dominant_key_selects_its_value_row():
    # one key aligned with q at a huge dot product; every other key is zero
    w = _small(seq_lens=(40, 40, 40), G=1, Hkv=1, D=32)
    q, k, v = wl.host_arrays(w)
    one = np.uint16(0x3F80)          # bf16 1.0
    big = np.uint16(0x4480)          # bf16 1024.0
    q2 = np.zeros_like(q); q2[:, :, 0] = one
    k2 = np.zeros_like(k)
    target = 13
    for i in range(3):
        page = w.block_tables[i, target // 16]
        k2[page, target % 16, 0, 0] = big
    out, lse = _call(w, q=q2, k=k2, scale=1.0)
    for i in range(3):
        page = w.block_tables[i, target // 16]
        vrow = oracle.bf16_bits_to_float64(v[page, target % 16, 0])
        assert np.abs(out[i, 0] - vrow).max() < 1e-12
        assert abs(lse[i, 0] - 1024.0) < 1e-12


def test_two_keys_closed_form():
    # s0 = 0, s1 = 1 (scale 1): weights 1/(1+e) and e/(1+e); lse = ln(1+e)
    w = _small(seq_lens=(2,), G=1, Hkv=1, D=8)
    q, k, v = wl.host_arrays(w)
    q2 = np.zeros_like(q); q2[0, 0, 3] = 0x3F80
    k2 = np.zeros_like(k)
    page = w.block_tables[0, 0]
    k2[page, 1, 0, 3] = 0x3F80
    out, lse = _call(w, q=q2, k=k2, scale=1.0)
    v0 = oracle.bf16_bits_to_float64(v[page, 0, 0])
    v1 = oracle.bf16_bits_to_float64(v[page, 1, 0])
    e = math.e
    assert np.abs(out[0, 0] - (v0 + e * v1) / (1 + e)).max() < 1e-15
    assert abs(lse[0, 0] - math.log1p(e)) < 1e-15


def test_gqa_mapping_consecutive_heads_share_kv_head():
    G, Hkv = 4, 3
    w = _small(seq_lens=(9, 20, 31), G=G, Hkv=Hkv, D=16)
    q, k, v = wl.host_arrays(w)
    v2 = np.zeros_like(v)
    for hk in range(Hkv):
        v2[:, :, hk, :] = torch.tensor(float(hk + 1)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out, _ = _call(w, v=v2)
    for hq in range(G * Hkv):
        assert np.abs(out[:, hq, :] - (hq // G + 1)).max() < 1e-13


def test_mtp_row_equals_prefix_attention():
    w = _small(qlens=(2, 3, 4), seq_lens=(5, 18, 47), seed=21)
    out, lse = _call(w)
    qsl = w.query_start_loc
    q, k, v = wl.host_arrays(w)
    for i in range(w.spec.num_seqs):
        L = int(w.seq_lens[i]); t0, t1 = int(qsl[i]), int(qsl[i + 1]); qn = t1 - t0
        for r in range(qn):
            # single-token decode over the prefix that ends at this token's position
            o1, l1 = oracle.paged_decode_attention(
                q[t0 + r:t0 + r + 1], k, v, w.block_tables[i:i + 1],
                np.array([L - qn + r + 1]), None, w.spec.scale, 1.0, 1.0, "bf16")
            assert np.abs(out[t0 + r] - o1[0]).max() < 1e-13
            assert np.abs(lse[t0 + r] - l1[0]).max() < 1e-13


def test_fp8_scale_folding_and_linearity():
    w = _small("fp8", seq_lens=(6, 30, 45))
    s = w.spec
    out, lse = _call(w)
    # doubling k_scale is the same as doubling the softmax scale (exact in fp64)
    o_a, l_a = _call(w, k_scale=2 * s.k_scale)
    o_b, l_b = _call(w, scale=2 * s.scale)
    assert np.abs(o_a - o_b).max() < 1e-13 and np.abs(l_a - l_b).max() < 1e-12
    # v_scale scales the output linearly (power of two: exact)
    o_c, l_c = _call(w, v_scale=4 * s.v_scale)
    assert np.array_equal(o_c, 4 * out) and np.array_equal(l_c, lse)


def test_split_merge_identity():
    """Attention over a sequence equals the log-sum-exp merge of attention
    over any page-aligned chunking of its keys (single query token)."""
    w = _small(seq_lens=(100, 77, 16), seed=4)
    out, lse = _call(w)
    q, k, v = wl.host_arrays(w)
    for i in range(w.spec.num_seqs):
        L = int(w.seq_lens[i]); n = (L + 15) // 16
        for cuts in ([0, n], [0, 1, n], [0, 2, 3, n], list(range(n + 1))):
            parts = []
            for a, b in zip(cuts[:-1], cuts[1:]):
                b = min(b, n)
                if a >= b:
                    continue
                Lc = min(L, 16 * b) - 16 * a
                o, l = oracle.paged_decode_attention(
                    q[i:i + 1], k, v, w.block_tables[i:i + 1, a:b], np.array([Lc]), None,
                    w.spec.scale, 1.0, 1.0, "bf16")
                parts.append((o[0], l[0]))
            M = np.max([p[1] for p in parts], axis=0)
            wsum = sum(np.exp(p[1] - M) for p in parts)
            merged = sum(np.exp(p[1] - M)[:, None] * p[0] for p in parts) / wsum[:, None]
            assert np.abs(merged - out[i]).max() < 1e-12
            assert np.abs(M + np.log(wsum) - lse[i]).max() < 1e-12


def test_entries_past_the_last_page_and_tail_slots_are_never_read():
    w = _small(seq_lens=(3, 17, 40))
    q, k, v = wl.host_arrays(w)
    out, lse = _call(w)
    nan_bits = np.uint16(0x7FC0)
    k2 = k.copy(); v2 = v.copy()
    used = set()
    for i, L in enumerate(w.seq_lens):
        n = (int(L) + 15) // 16
        for j in range(n):
            used.add(int(w.block_tables[i, j]))
        last = w.block_tables[i, n - 1]
        tail = int(L) - 16 * (n - 1)
        k2[last, tail:] = nan_bits; v2[last, tail:] = nan_bits
    for p in range(w.num_pages):
        if p not in used:
            k2[p] = nan_bits; v2[p] = nan_bits
    bt2 = w.block_tables.copy()
    bt2[bt2 < 0] = 10 ** 6           # out of range: would fail if read
    out2, lse2 = _call(w, k=k2, v=v2, bt=bt2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


# ---------------------------------------------- sliding window and attention sinks

@pytest.mark.parametrize("window", [1, 5, 16, 17, 40])
@pytest.mark.parametrize("qlens", [(1,), (2, 3, 4)])
def test_sliding_window_matches_sdpa_with_window_mask(window, qlens):
    spec = wl.custom_spec(num_q_heads=8, num_kv_heads=2, head_dim=64, seq_lens=(4, 16, 17, 50, 97),
                          query_len_choices=qlens, seed=31)
    w = wl.make_workload(spec)
    out, lse = oracle.run_workload(w, sliding_window=window)
    ref_out, ref_lse = _torch_reference(w, window=window)
    assert np.abs(out - ref_out).max() < 1e-12
    assert np.abs(lse - ref_lse).max() < 1e-12


def test_window_of_one_returns_own_value_and_wide_window_changes_nothing():
    w = _small(seq_lens=(3, 18, 40), G=2, Hkv=2, D=32)
    q, k, v = wl.host_arrays(w)
    s = w.spec
    o1, l1 = oracle.paged_decode_attention(q, k, v, w.block_tables, w.seq_lens, None, s.scale, sliding_window=1)
    G = s.group_size
    for i, L in enumerate(w.seq_lens):
        page, slot = w.block_tables[i, (L - 1) // 16], (L - 1) % 16
        for hq in range(s.num_q_heads):
            vrow = oracle.bf16_bits_to_float64(v[page, slot, hq // G])
            krow = oracle.bf16_bits_to_float64(k[page, slot, hq // G])
            assert np.array_equal(o1[i, hq], vrow)
            assert abs(l1[i, hq] - float(np.float32(s.scale)) * float(oracle.bf16_bits_to_float64(q[i, hq]) @ krow)) < 1e-12
    o_full, l_full = _call(w)
    o_w, l_w = oracle.paged_decode_attention(q, k, v, w.block_tables, w.seq_lens, None, s.scale, sliding_window=40)
    assert np.array_equal(o_full, o_w) and np.array_equal(l_full, l_w)


def test_sink_closed_form_against_the_sinkless_result():
    """A sink logit s with a zero value row: out_s = out * Z / (Z + e^s) and
    lse_s = ln(Z + e^s), with Z = e^lse of the sinkless attention."""
    w = _small(qlens=(1, 2), seq_lens=(5, 30, 47), G=4, Hkv=2, D=32, seed=8)
    q, k, v = wl.host_arrays(w)
    s = w.spec
    sinks = np.array([-3.0, 0.0, 0.5, 2.0, 7.25, -1.5, 0.1, 3.0], dtype=np.float32)
    o, l = _call(w)
    os_, ls_ = oracle.paged_decode_attention(q, k, v, w.block_tables, w.seq_lens, w.query_start_loc, s.scale,
                                             sinks=sinks)
    sk = sinks.astype(np.float64)[None, :]
    assert np.abs(ls_ - np.logaddexp(l, sk)).max() < 1e-12
    assert np.abs(os_ - o / (1.0 + np.exp(sk - l))[:, :, None]).max() < 1e-12
