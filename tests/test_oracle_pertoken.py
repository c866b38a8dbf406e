"""Pins for the oracle's per-token fp8 scales (one fp32 scale per cached row
and KV head, stored [num_pages, num_kv_heads, 16]): a library attention routine
on a contiguous cache dequantised by a different indexing route, the reduction
to per-tensor scales, a closed form for one row's scale, and page-permutation
invariance.  CPU only."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_06_gb300 import workloads as wl


def _spec(qlens=(1,), seq_lens=(4, 16, 17, 50, 97), k_scale=1.0, v_scale=1.0, seed=21, G=4, Hkv=2, D=64):
    return wl.custom_spec(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, kv_dtype="fp8",
                          seq_lens=seq_lens, query_len_choices=qlens, k_scale=k_scale, v_scale=v_scale,
                          fp8_source_scale=1.0 / 128, token_scale_range=(0.5 / 128, 2.0 / 128), seed=seed)


def _torch_reference(w):
    """Pages reshaped into a contiguous cache; each page's [Hkv, 16] scale
    block transposed onto its [16, Hkv] rows; float64 SDPA with an explicit
    causal mask and repeated KV heads."""
    s = w.spec
    G = s.group_size
    ks = w.k_token_scales.to(torch.float64).permute(0, 2, 1)[..., None]      # [NB, 16, Hkv, 1]
    vs = w.v_token_scales.to(torch.float64).permute(0, 2, 1)[..., None]
    kc = w.k_cache.view(torch.float8_e4m3fn).to(torch.float64) * float(np.float32(s.k_scale)) * ks
    vc = w.v_cache.view(torch.float8_e4m3fn).to(torch.float64) * float(np.float32(s.v_scale)) * vs
    q = w.q.to(torch.float64)
    qsl = w.query_start_loc if w.query_start_loc is not None else np.arange(s.num_seqs + 1)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float64)
    scale = float(np.float32(s.scale))
    for i in range(s.num_seqs):
        L = int(w.seq_lens[i])
        n = (L + 15) // 16
        pages = torch.from_numpy(w.block_tables[i, :n].astype(np.int64))
        K = kc[pages].reshape(n * 16, s.num_kv_heads, s.head_dim)[:L].repeat_interleave(G, dim=1).permute(1, 0, 2)
        V = vc[pages].reshape(n * 16, s.num_kv_heads, s.head_dim)[:L].repeat_interleave(G, dim=1).permute(1, 0, 2)
        t0, t1 = int(qsl[i]), int(qsl[i + 1])
        Q = q[t0:t1].permute(1, 0, 2)
        qn = t1 - t0
        mask = torch.arange(L)[None, :] <= (L - qn + torch.arange(qn))[:, None]
        out[t0:t1] = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale).permute(1, 0, 2)
        logits = (scale * (Q @ K.transpose(1, 2))).masked_fill(~mask, float("-inf"))
        lse[t0:t1] = torch.logsumexp(logits, dim=-1).permute(1, 0)
    return out.numpy(), lse.numpy()


@pytest.mark.parametrize("qlens", [(1,), (2, 3, 4)])
@pytest.mark.parametrize("tensor_scales", [(1.0, 1.0), (0.5, 3.0)])
def test_per_token_oracle_matches_sdpa(qlens, tensor_scales):
    w = wl.make_workload(_spec(qlens=qlens, k_scale=tensor_scales[0], v_scale=tensor_scales[1]))
    out, lse = oracle.run_workload(w)
    ref_out, ref_lse = _torch_reference(w)
    assert np.abs(out - ref_out).max() < 1e-12
    assert np.abs(lse - ref_lse).max() < 1e-12


def test_equal_token_scales_reduce_to_the_per_tensor_scale():
    w = wl.make_workload(_spec(seq_lens=(3, 33, 64)))
    q, k, v = wl.host_arrays(w)
    c_k, c_v = np.float32(0.0123), np.float32(0.0456)
    ks = np.full((w.num_pages, w.spec.num_kv_heads, 16), c_k, dtype=np.float32)
    vs = np.full_like(ks, c_v)
    a = oracle.paged_decode_attention(q, k, v, w.block_tables, w.seq_lens, None, w.spec.scale, 1.0, 1.0, "fp8",
                                      k_token_scales=ks, v_token_scales=vs)
    b = oracle.paged_decode_attention(q, k, v, w.block_tables, w.seq_lens, None, w.spec.scale, float(c_k),
                                      float(c_v), "fp8")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_one_value_scale_doubled_adds_its_weighted_row():
    # doubling token j's value scale adds w_j * V_j, w_j = exp(s_j - lse)
    w = wl.make_workload(_spec(seq_lens=(37,), G=1, Hkv=1, D=32))
    q, k, v = wl.host_arrays(w)
    ks, vs = wl.host_token_scales(w)
    args = (q, k, v, w.block_tables, w.seq_lens, None, w.spec.scale, 1.0, 1.0, "fp8")
    out, lse = oracle.paged_decode_attention(*args, k_token_scales=ks, v_token_scales=vs)
    j = 21
    page, slot = w.block_tables[0, j // 16], j % 16
    vs2 = vs.copy()
    vs2[page, 0, slot] *= 2
    out2, lse2 = oracle.paged_decode_attention(*args, k_token_scales=ks, v_token_scales=vs2)
    vj = oracle.e4m3fn_to_float64(v[page, slot, 0]) * np.float64(vs[page, 0, slot])
    kj = oracle.e4m3fn_to_float64(k[page, slot, 0]) * np.float64(ks[page, 0, slot])
    qrow = oracle.bf16_bits_to_float64(q[0, 0])
    wj = np.exp(np.float64(np.float32(w.spec.scale)) * (qrow @ kj) - lse[0, 0])
    assert np.abs(out2[0, 0] - (out[0, 0] + wj * vj)).max() < 1e-12
    assert lse2[0, 0] == lse[0, 0]


def test_per_token_page_permutation_invariance_bit_exact():
    w = wl.make_workload(_spec(qlens=(1, 2), seq_lens=(3, 16, 40)))
    q, k, v = wl.host_arrays(w)
    ks, vs = wl.host_token_scales(w)
    args = (w.query_start_loc, w.spec.scale, 1.0, 1.0, "fp8")
    out, lse = oracle.paged_decode_attention(q, k, v, w.block_tables, w.seq_lens, *args,
                                             k_token_scales=ks, v_token_scales=vs)
    perm = np.random.default_rng(4).permutation(w.num_pages)
    k2, v2, ks2, vs2 = (np.empty_like(a) for a in (k, v, ks, vs))
    k2[perm], v2[perm], ks2[perm], vs2[perm] = k, v, ks, vs
    bt2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out2, lse2 = oracle.paged_decode_attention(q, k2, v2, bt2, w.seq_lens, *args, k_token_scales=ks2,
                                               v_token_scales=vs2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_key_scale_is_indexed_by_head_then_slot():
    # a scale planted at [page, head 1, slot 3] must act on head 1's slot-3 key only
    w = wl.make_workload(_spec(seq_lens=(16,), G=1, Hkv=2, D=16))
    q, k, v = wl.host_arrays(w)
    ks = np.ones((w.num_pages, 2, 16), dtype=np.float32)
    vs = np.ones_like(ks)
    page = w.block_tables[0, 0]
    vs[page, 1, 3] = 0.0                      # head 1's slot-3 value row vanishes
    out, _ = oracle.paged_decode_attention(q, k, v, w.block_tables, w.seq_lens, None, 1.0, 1.0, 1.0, "fp8",
                                           k_token_scales=ks, v_token_scales=vs)
    K = oracle.e4m3fn_to_float64(k[page, :, 1])             # [16, D]
    V = oracle.e4m3fn_to_float64(v[page, :, 1])
    V[3] = 0.0
    s = oracle.bf16_bits_to_float64(q[0, 1]) @ K.T
    p = np.exp(s - s.max()); p /= p.sum()
    assert np.abs(out[0, 1] - p @ V).max() < 1e-9 * max(1.0, np.abs(p @ V).max())
