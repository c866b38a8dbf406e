"""Float64 CPU oracle for multi-head latent attention (MLA) decode over a paged
latent cache.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): imported by
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``; never by the library, and it shares no code with the CUDA path.
Its parity pins live in ``tests/test_oracle_mla.py``.

What it computes (ATOM model-operations guide, "Multi-head latent attention
(attention_mla.py)": the ``MLAModules`` fields ``kv_lora_rank``,
``qk_rope_head_dim``, ``v_head_dim`` and the decode forward flow, step 2: the
query is projected into the latent space together with the K up-projection,
``fused_qk_rope_concat_and_cache_mla`` writes one row per token to the cache,
``mla_decode_fwd`` attends over it, and the V up-projection follows in step 3;
high-interactivity blog, "Attention Decode": split count and fp32 per-split
log-sum-exp for MLA decode, and "Multi-Token Prediction": the query-length-four
verification shape).

Readings adopted where the pages are silent (listed in the design notes):

* one cached row per token is the concatenation ``[c_kv | k_pe]``: the
  compressed latent (``kv_lora_rank`` values) followed by the rotary key part
  (``qk_rope_head_dim`` values), stored ``[num_pages, 16, kv_lora_rank +
  qk_rope_head_dim]``; there is no head axis (every query head reads the same
  row, multi-query style);
* the query arrives already absorbed: ``q[t, h] = [q_nope W_UK | q_pe]`` with
  the same width as a cached row, so the logit is the plain dot product of
  the two rows times ``scale``;
* the value is the latent part of the row, ``c_kv`` (the first
  ``kv_lora_rank`` values); the attention output is in the latent space (the
  V up-projection is a later step, outside this path);
* fp8 caches hold OCP e4m3fn codes with one fp32 scale for the whole cache:
  a cached element is ``code * kv_scale`` in the logit and in the value;
* ``seq_lens`` include the query tokens, query row ``r`` of a run of ``q_i``
  tokens attends keys ``0 .. L_i - q_i + r``; ``lse`` is the natural-log
  log-sum-exp of the scaled logits.
"""
from __future__ import annotations

import numpy as np

from .paged_attention import PAGE_SIZE, bf16_bits_to_float64, e4m3fn_to_float64


def gather_latent(cache: np.ndarray, block_table_row: np.ndarray, seq_len: int) -> np.ndarray:
    """Raw cached rows of logical tokens 0..seq_len-1 (token j: physical page
    ``block_table_row[j // 16]``, slot ``j % 16``); only the first
    ceil(seq_len / 16) block-table entries are read."""
    j = np.arange(seq_len)
    pages = np.asarray(block_table_row)[j // PAGE_SIZE].astype(np.int64)
    return cache[pages, j % PAGE_SIZE, :]


def decode_latent(raw: np.ndarray, kv_dtype: str, kv_scale: float) -> np.ndarray:
    """Cached elements -> float64: bf16 exactly; fp8 as the code's value times
    the cache's fp32 scale."""
    if kv_dtype == "bf16":
        return bf16_bits_to_float64(raw)
    if kv_dtype == "fp8":
        return e4m3fn_to_float64(raw) * np.float64(np.float32(kv_scale))
    raise ValueError(kv_dtype)


def mla_decode(q_bits: np.ndarray, kv_cache: np.ndarray, block_tables: np.ndarray, seq_lens: np.ndarray,
               query_start_loc, scale: float, kv_scale: float = 1.0, kv_dtype: str = "bf16",
               kv_lora_rank: int = 512, seqs=None):
    """MLA decode for a batch.

    q_bits      uint16 bf16 patterns [T, Hq, kv_lora_rank + rope]
    kv_cache    uint16 (bf16) or uint8 (e4m3) [NB, 16, kv_lora_rank + rope]
    block_tables int [B, max_blocks]; seq_lens int [B]
    query_start_loc int [B+1] or None (one query token per sequence)
    seqs        optional iterable of sequence indices to evaluate (others stay NaN)

    For query row (t, h) at position p of sequence i, with C_j the decoded
    cached row of token j:
        s_j = scale * <q[t, h], C_j>            for j = 0 .. p
        lse = m + ln sum_j exp(s_j - m),        m = max_j s_j
        out = sum_j exp(s_j - lse) * C_j[:kv_lora_rank]
    Returns (out float64 [T, Hq, kv_lora_rank], lse float64 [T, Hq]).
    """
    T, Hq, Dqk = q_bits.shape
    NB, P, Dc = kv_cache.shape
    assert P == PAGE_SIZE and Dc == Dqk and 0 < kv_lora_rank <= Dqk
    B = len(seq_lens)
    qsl = np.arange(B + 1) if query_start_loc is None else np.asarray(query_start_loc, dtype=np.int64)
    sc = np.float64(np.float32(scale))
    out = np.full((T, Hq, kv_lora_rank), np.nan)
    lse = np.full((T, Hq), np.nan)
    for i in (range(B) if seqs is None else seqs):
        L = int(seq_lens[i])
        t0, t1 = int(qsl[i]), int(qsl[i + 1])
        qn = t1 - t0
        assert 1 <= qn <= L
        C = decode_latent(gather_latent(kv_cache, block_tables[i], L), kv_dtype, kv_scale)   # [L, Dqk]
        values = C[:, :kv_lora_rank]
        for r in range(qn):
            p = L - qn + r                                   # last key this query token sees
            qr = bf16_bits_to_float64(q_bits[t0 + r])        # [Hq, Dqk]
            s = sc * (qr @ C[:p + 1].T)                      # [Hq, p + 1]
            m = s.max(axis=1, keepdims=True)
            l = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
            out[t0 + r] = np.exp(s - l[:, None]) @ values[:p + 1]
            lse[t0 + r] = l
    return out, lse


def run_mla_workload(w, seqs=None):
    """Oracle outputs for a ``paged_kv_decode_06_gb300.workloads.MlaWorkload``."""
    from paged_kv_decode_06_gb300.workloads import host_mla_arrays
    q_bits, c = host_mla_arrays(w)
    s = w.spec
    return mla_decode(q_bits, c, w.block_tables, w.seq_lens, w.query_start_loc, s.scale, s.kv_scale, s.kv_dtype,
                      s.kv_lora_rank, seqs=seqs)
