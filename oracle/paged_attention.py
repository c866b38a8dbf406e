"""Float64 CPU oracle for decode attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library
never calls it, and it shares no code with the CUDA path.

What it computes (ATOM model-operations guide, "Multi-head attention" forward
flow and "Attention dispatch"; configuration guide, ``kv_cache_block_size`` and
``kv_cache_dtype``; high-interactivity blog, "Attention Decode: Split Memory
Work to Fill the Device"): for every query token of every sequence and every
query head, softmax(scale * q K^T) V over the sequence's cached keys and
values, which are found page by page through the sequence's block table.

Readings adopted where the pages are silent (each is listed in the design
notes):

* cache layout ``[num_pages, 16, num_kv_heads, head_dim]`` (flash layout), K and
  V in separate tensors;
* ``seq_lens[i]`` counts the sequence's own query tokens (their K/V were written
  to the cache before attention runs);
* query row ``r`` of a run of ``q_i`` tokens sits at absolute position
  ``p_r = L_i - q_i + r`` and attends keys ``0 .. p_r`` (causal inside the run);
* grouped-query mapping: query head ``hq`` reads KV head ``hq // (Hq // Hkv)``;
* fp8 is OCP e4m3fn; a cached value is ``code * k_scale`` (K) or
  ``code * v_scale`` (V) with one fp32 scale per tensor; bf16 caches carry no
  scale;
* per-token fp8 scales (the pages' ``reshape_and_cache_with_pertoken_quant``
  write): one fp32 scale per cached (token slot, KV head) row, stored
  ``[num_pages, num_kv_heads, 16]``; the row's value is
  ``code * tensor_scale * token_scale`` (the per-tensor scale still multiplies;
  callers of a purely per-token cache pass 1.0);
* ``lse`` is the natural-log log-sum-exp of the scaled logits;
* sliding window W (``sliding_window`` > 0; the pages' models with
  ``sliding_window != -1``): query row r sees keys ``p_r - W < j <= p_r``;
* attention sinks (per query head logit ``sink[hq]``, as in GPT-OSS): the sink
  joins the softmax normaliser with a zero value row, and ``lse`` includes it.

Every function works in float64 on values decoded bit-exactly from the bf16
and e4m3 encodings.
"""
from __future__ import annotations

import numpy as np

PAGE_SIZE = 16


def bf16_bits_to_float64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (uint16): a bf16 value is the upper half of an
    IEEE-754 binary32, so shifting the pattern 16 bits up gives that float32
    exactly; widening to float64 is exact."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):          # NaN patterns stay NaN
        return b.view(np.float32).astype(np.float64)


def e4m3fn_to_float64(codes: np.ndarray) -> np.ndarray:
    """Decode OCP FP8 E4M3 ("fn": finite, no infinities) codes from their bit
    fields: sign s (bit 7), exponent e (bits 6..3, bias 7), mantissa m
    (bits 2..0).

    * e == 0:            value = (-1)^s * (m / 8) * 2^(1 - 7)      (subnormal)
    * e in 1..15:        value = (-1)^s * (1 + m / 8) * 2^(e - 7)
    * e == 15, m == 7:   NaN  (the only non-finite code; max finite is 448)
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    sign = np.where(s == 1, -1.0, 1.0)
    sub = sign * (m / 8.0) * np.ldexp(1.0, -6)
    nor = sign * (1.0 + m / 8.0) * np.ldexp(1.0, (e - 7).astype(np.int64))
    out = np.where(e == 0, sub, nor)
    out = np.where((e == 15) & (m == 7), np.nan, out)
    return out.astype(np.float64)


def dequantize(raw: np.ndarray, kv_dtype: str, tensor_scale: float, token_scales=None) -> np.ndarray:
    """Cached element -> float64.  bf16: the value itself.  fp8: code value
    times the tensor's scale, the scale taken as the fp32 number the kernel
    receives, and times the row's own fp32 scale when ``token_scales`` (one
    per row of ``raw``) is given."""
    if kv_dtype == "bf16":
        return bf16_bits_to_float64(raw)
    if kv_dtype == "fp8":
        v = e4m3fn_to_float64(raw) * np.float64(np.float32(tensor_scale))
        if token_scales is not None:
            v = v * np.asarray(token_scales, dtype=np.float32).astype(np.float64)[:, None]
        return v
    raise ValueError(kv_dtype)


def gather_token_scales(scales: np.ndarray, block_table_row: np.ndarray, seq_len: int,
                        kv_head: int) -> np.ndarray:
    """Per-token scales ``[num_pages, num_kv_heads, 16]`` of one KV head for
    logical tokens 0..seq_len-1 (token j: page ``block_table_row[j // 16]``,
    slot ``j % 16``)."""
    tok = np.arange(seq_len)
    pages = np.asarray(block_table_row)[tok // PAGE_SIZE].astype(np.int64)
    return np.asarray(scales)[pages, kv_head, tok % PAGE_SIZE]


def gather_sequence(cache: np.ndarray, block_table_row: np.ndarray, seq_len: int,
                    kv_head: int) -> np.ndarray:
    """Raw rows of one KV head for logical tokens 0..seq_len-1: token j lives
    in physical page ``block_table_row[j // 16]`` at slot ``j % 16``.  Only
    the first ceil(seq_len / 16) block-table entries are read."""
    j = np.arange(seq_len)
    pages = np.asarray(block_table_row)[j // PAGE_SIZE].astype(np.int64)
    slots = j % PAGE_SIZE
    return cache[pages, slots, kv_head, :]


def attend(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float,
           key_limits: np.ndarray, window: int = 0, sinks=None):
    """Softmax attention of each query row over keys ``0 .. key_limits[r]``
    (and, with window W > 0, only keys ``> key_limits[r] - W``).

    q_rows [R, D], keys/values [L, D] float64; sinks: optional per-row logit
    (float64 [R]) with a zero value row.  Returns (out [R, D], lse [R]):
    lse = m + ln sum_j exp(s_j - m) with m = max_j s_j over the allowed keys and
    the sink, and out = sum_j exp(s_j - lse) V_j, where s_j = scale * <q, k_j>.
    """
    R = q_rows.shape[0]
    L = keys.shape[0]
    s = scale * (q_rows @ keys.T)                       # [R, L]
    j = np.arange(L)[None, :]
    lim = np.asarray(key_limits)[:, None]
    allowed = j <= lim
    if window > 0:
        allowed &= j > lim - window
    s = np.where(allowed, s, -np.inf)
    if sinks is not None:
        s = np.concatenate([s, np.asarray(sinks, dtype=np.float64)[:, None]], axis=1)
        values = np.concatenate([values, np.zeros((1, values.shape[1]))], axis=0)
    m = s.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
    w = np.exp(s - lse[:, None])                        # 0 where not allowed
    out = w @ values
    assert out.shape == (R, values.shape[1])
    return out, lse


def paged_decode_attention(q_bits: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                           block_tables: np.ndarray, seq_lens: np.ndarray,
                           query_start_loc, scale: float, k_scale: float = 1.0,
                           v_scale: float = 1.0, kv_dtype: str = "bf16",
                           seqs=None, sliding_window: int = 0, sinks=None,
                           k_token_scales=None, v_token_scales=None):
    """Decode attention for a batch.

    q_bits      uint16 bf16 patterns [T, Hq, D]
    k_cache     uint16 (bf16) or uint8 (e4m3) [NB, 16, Hkv, D]; v_cache likewise
    block_tables int [B, max_blocks]; seq_lens int [B]
    query_start_loc int [B+1] or None (one query token per sequence)
    seqs        optional iterable of sequence indices to evaluate (others are
                left as NaN), for sampled checks of large batches.
    sliding_window  W > 0: each query sees only its last W positions (0 = off)
    sinks       optional float [Hq] per-query-head sink logits (taken as fp32)
    k_token_scales, v_token_scales  optional float32 [NB, Hkv, 16] per-token
                scales of fp8 caches (both or neither)

    Returns (out float64 [T, Hq, D], lse float64 [T, Hq]).
    """
    T, Hq, D = q_bits.shape
    NB, P, Hkv, D2 = k_cache.shape
    assert P == PAGE_SIZE and D2 == D and v_cache.shape == k_cache.shape
    assert Hq % Hkv == 0
    G = Hq // Hkv
    B = len(seq_lens)
    if query_start_loc is None:
        qsl = np.arange(B + 1)
    else:
        qsl = np.asarray(query_start_loc, dtype=np.int64)
    sc = np.float64(np.float32(scale))
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    for i in (range(B) if seqs is None else seqs):
        L = int(seq_lens[i])
        t0, t1 = int(qsl[i]), int(qsl[i + 1])
        qn = t1 - t0
        assert 1 <= qn <= L
        limits = L - qn + np.arange(qn)          # last key index each query token sees
        for hk in range(Hkv):
            ks = vs = None
            if k_token_scales is not None:
                ks = gather_token_scales(k_token_scales, block_tables[i], L, hk)
                vs = gather_token_scales(v_token_scales, block_tables[i], L, hk)
            K = dequantize(gather_sequence(k_cache, block_tables[i], L, hk), kv_dtype, k_scale, ks)
            V = dequantize(gather_sequence(v_cache, block_tables[i], L, hk), kv_dtype, v_scale, vs)
            heads = np.arange(hk * G, (hk + 1) * G)
            qr = bf16_bits_to_float64(q_bits[t0:t1][:, heads, :])      # [qn, G, D]
            sk = None
            if sinks is not None:
                sk = np.tile(np.asarray(sinks, dtype=np.float32).astype(np.float64)[heads], qn)
            o, l = attend(qr.reshape(qn * G, D), K, V, sc, np.repeat(limits, G), sliding_window, sk)
            out[t0:t1, hk * G:(hk + 1) * G, :] = o.reshape(qn, G, D)
            lse[t0:t1, hk * G:(hk + 1) * G] = l.reshape(qn, G)
    return out, lse


def run_workload(w, seqs=None, sliding_window=0, sinks=None):
    """Oracle outputs for a ``paged_kv_decode_06_gb300.workloads.Workload``."""
    from paged_kv_decode_06_gb300.workloads import host_arrays, host_token_scales
    q_bits, k, v = host_arrays(w)
    s = w.spec
    ks, vs = host_token_scales(w)
    return paged_decode_attention(q_bits, k, v, w.block_tables, w.seq_lens,
                                  w.query_start_loc, s.scale, s.k_scale, s.v_scale,
                                  s.kv_dtype, seqs=seqs, sliding_window=sliding_window, sinks=sinks,
                                  k_token_scales=ks, v_token_scales=vs)
