"""Seeded synthetic inputs for paged decode attention.

This module only draws random numbers and lays them out in the paged-cache
format; it holds none of the attention arithmetic.  Both the float64 oracle
(test infrastructure) and the CUDA path take their inputs from here.

Layout (ATOM model-operations guide, "Attention dispatch" / "KV cache
operations"; configuration guide, ``kv_cache_block_size``):

* ``q``            bf16  ``[T, Hq, D]``          T = number of query tokens
* ``k_cache``      bf16 or fp8-e4m3 codes ``[NB, 16, Hkv, D]``  (flash layout)
* ``v_cache``      same dtype and shape as ``k_cache``
* ``block_tables`` int32 ``[B, max_blocks]``     logical page -> physical page,
                   ``-1`` past a sequence's last page
* ``seq_lens``     int32 ``[B]``  context length, *including* the sequence's
                   query tokens (their K/V are already in the cache)
* ``query_start_loc`` int32 ``[B+1]`` cumulative query-token offsets, or
                   ``None`` when every sequence has exactly one query token.
* ``k_token_scales``, ``v_token_scales`` (per-token fp8 workloads only) fp32
                   ``[NB, Hkv, 16]``: one positive scale per cached row, drawn
                   log-uniformly; the codes of such a cache are drawn from
                   N(0,1) / fp8_source_scale clamped to the e4m3 range.

Every page of the pool is filled with random data (never NaN), including the
tail slots of a sequence's last page and the pages no sequence uses.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

PAGE_SIZE = 16


@dataclasses.dataclass
class WorkloadSpec:
    """Shape and distribution of one synthetic decode batch."""

    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str                      # "bf16" or "fp8"
    seq_len_kind: str                  # "fixed" | "uniform" | "loguniform"
    seq_len_args: tuple
    query_len_choices: tuple = (1,)    # each sequence draws its query length from these
    pool_pages: Optional[int] = None   # physical pool size; default ceil(1.1 * used)
    k_scale: float = 1.0
    v_scale: float = 1.0
    fp8_source_scale: float = 1.0      # fp8 codes = e4m3(N(0,1) / fp8_source_scale)
    seed: int = 0
    token_scale_range: Optional[tuple] = None   # fp8: per-token scales ~ log-U[lo, hi] (None = per-tensor only)

    @property
    def group_size(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_query_len(self) -> int:
        return max(self.query_len_choices)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


# The decode regimes: a tiny parity case, a Llama-3-8B-shaped batch, a single
# long-context user, an fp8-KV batch at batch 256, an MTP verification batch
# with ragged query runs, and a longer verification batch.
CONFIGS = {
    "tiny": WorkloadSpec(
        name="tiny", num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=128,
        kv_dtype="bf16", seq_len_kind="fixed", seq_len_args=(1, 17, 64, 200),
        pool_pages=64, seed=1000),
    "llama3_8b": WorkloadSpec(
        name="llama3_8b", num_seqs=64, num_q_heads=32, num_kv_heads=8, head_dim=128,
        kv_dtype="bf16", seq_len_kind="uniform", seq_len_args=(512, 4096), seed=1001),
    "batch1_32k": WorkloadSpec(
        name="batch1_32k", num_seqs=1, num_q_heads=64, num_kv_heads=8, head_dim=64,
        kv_dtype="bf16", seq_len_kind="fixed", seq_len_args=(32768,), seed=1002),
    "fp8": WorkloadSpec(
        name="fp8", num_seqs=256, num_q_heads=32, num_kv_heads=8, head_dim=128,
        kv_dtype="fp8", seq_len_kind="loguniform", seq_len_args=(128, 8192),
        k_scale=0.05, v_scale=0.05, fp8_source_scale=0.05, seed=1003),
    "mtp": WorkloadSpec(
        name="mtp", num_seqs=32, num_q_heads=64, num_kv_heads=8, head_dim=128,
        kv_dtype="bf16", seq_len_kind="uniform", seq_len_args=(1024, 16384),
        query_len_choices=(2, 3, 4), seed=1004),
    # fp8 cache quantised per token (one scale per cached row and KV head),
    # the batch-256 shape of the per-tensor fp8 workload: codes spread over
    # the e4m3 range, row scales log-uniform in [1/512, 1/128] (dequantised
    # values N(0,1) times 1/4 to 1).
    "fp8_pertoken": WorkloadSpec(
        name="fp8_pertoken", num_seqs=256, num_q_heads=32, num_kv_heads=8, head_dim=128,
        kv_dtype="fp8", seq_len_kind="loguniform", seq_len_args=(128, 8192),
        fp8_source_scale=1.0 / 128, token_scale_range=(0.25 / 128, 1.0 / 128), seed=1006),
    # Longer speculative verification: runs of 1 + up to 7 draft tokens over a
    # 16-query-head group (Llama-3-405B-shaped heads, 128 over 8), so a KV
    # head serves up to 128 query rows, a dense tile for the tensor cores.
    "verify8": WorkloadSpec(
        name="verify8", num_seqs=32, num_q_heads=128, num_kv_heads=8, head_dim=128,
        kv_dtype="bf16", seq_len_kind="uniform", seq_len_args=(1024, 16384),
        query_len_choices=(2, 3, 4, 5, 6, 7, 8), seed=1005),
}

CONFIG_ORDER = ["tiny", "llama3_8b", "batch1_32k", "fp8", "mtp", "verify8", "fp8_pertoken"]


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    seq_lens: np.ndarray            # int32 [B]
    query_lens: np.ndarray          # int32 [B]
    query_start_loc: Optional[np.ndarray]   # int32 [B+1] or None
    block_tables: np.ndarray        # int32 [B, max_blocks], -1 padded
    num_pages: int                  # NB, physical pool size
    q: torch.Tensor                 # bf16 [T, Hq, D]
    k_cache: torch.Tensor           # bf16 or uint8 (e4m3 codes) [NB, 16, Hkv, D]
    v_cache: torch.Tensor
    k_token_scales: Optional[torch.Tensor] = None   # fp32 [NB, Hkv, 16] (per-token fp8 only)
    v_token_scales: Optional[torch.Tensor] = None

    @property
    def num_tokens(self) -> int:
        return int(self.query_lens.sum())

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.spec.kv_dtype == "fp8" else 2

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes of one step: every cached token's K and V row
        of every KV head, read once (with per-token scales, also the two fp32
        scales of each row)."""
        s = self.spec
        per_row = s.head_dim * self.kv_elem_bytes + (4 if self.k_token_scales is not None else 0)
        return int(self.seq_lens.astype(np.int64).sum()) * s.num_kv_heads * 2 * per_row


def draw_metadata(spec: WorkloadSpec, rng: np.random.Generator):
    """Sequence lengths, query lengths and a randomly permuted page pool."""
    B = spec.num_seqs
    if spec.seq_len_kind == "fixed":
        seq_lens = np.array(spec.seq_len_args, dtype=np.int64)
        assert seq_lens.shape == (B,) or seq_lens.shape == (1,)
        seq_lens = np.broadcast_to(seq_lens, (B,)).copy()
    elif spec.seq_len_kind == "uniform":
        lo, hi = spec.seq_len_args
        seq_lens = rng.integers(lo, hi, size=B, endpoint=True)
    elif spec.seq_len_kind == "loguniform":
        lo, hi = spec.seq_len_args
        seq_lens = np.floor(np.exp(rng.uniform(np.log(lo), np.log(hi + 1), size=B))).astype(np.int64)
        seq_lens = np.clip(seq_lens, lo, hi)
    else:
        raise ValueError(spec.seq_len_kind)
    query_lens = rng.choice(np.array(spec.query_len_choices, dtype=np.int64), size=B)
    seq_lens = np.maximum(seq_lens, query_lens)
    pages_per_seq = (seq_lens + PAGE_SIZE - 1) // PAGE_SIZE
    used = int(pages_per_seq.sum())
    pool = spec.pool_pages if spec.pool_pages is not None else int(math.ceil(1.1 * used))
    assert pool >= used, (pool, used)
    perm = rng.permutation(pool)
    max_blocks = int(pages_per_seq.max())
    block_tables = np.full((B, max_blocks), -1, dtype=np.int64)
    cursor = 0
    for i in range(B):
        n = int(pages_per_seq[i])
        block_tables[i, :n] = perm[cursor:cursor + n]
        cursor += n
    if spec.query_len_choices == (1,):
        qsl = None
    else:
        qsl = np.zeros(B + 1, dtype=np.int64)
        qsl[1:] = np.cumsum(query_lens)
        qsl = qsl.astype(np.int32)
    return (seq_lens.astype(np.int32), query_lens.astype(np.int32), qsl,
            block_tables.astype(np.int32), pool)


def _fill_normal(t: torch.Tensor, gen: torch.Generator, divisor: float, fp8: bool) -> None:
    """Fill ``t`` (bf16 or uint8) chunk by chunk with N(0,1)/divisor, rounded
    to nearest-even bf16 or encoded as e4m3fn codes."""
    flat = t.view(-1)
    n = flat.numel()
    chunk = 1 << 26
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=gen, device=t.device, dtype=torch.float32)
        if divisor != 1.0:
            x = x / divisor
        if fp8:
            flat[s:e] = x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        else:
            flat[s:e] = x.to(torch.bfloat16)


def make_workload(spec: WorkloadSpec, device: str = "cpu", seed: Optional[int] = None,
                  content_seed: Optional[int] = None) -> Workload:
    """Build one seeded batch.  Metadata comes from numpy's PCG64 with
    ``seed``; tensor contents from torch's generator on ``device`` with
    ``content_seed`` (default: the same seed; CPU and CUDA draws differ, but
    each is reproducible).  Batches that differ only in ``content_seed`` share
    lengths, block tables and pool size."""
    seed = spec.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    seq_lens, query_lens, qsl, block_tables, pool = draw_metadata(spec, rng)
    T = int(query_lens.sum())
    gen = torch.Generator(device=device)
    gen.manual_seed(seed if content_seed is None else content_seed)
    fp8 = spec.kv_dtype == "fp8"
    q = torch.empty((T, spec.num_q_heads, spec.head_dim), dtype=torch.bfloat16, device=device)
    _fill_normal(q, gen, 1.0, False)
    kv_shape = (pool, PAGE_SIZE, spec.num_kv_heads, spec.head_dim)
    kv_torch_dtype = torch.uint8 if fp8 else torch.bfloat16
    k_cache = torch.empty(kv_shape, dtype=kv_torch_dtype, device=device)
    v_cache = torch.empty(kv_shape, dtype=kv_torch_dtype, device=device)
    div = spec.fp8_source_scale if fp8 else 1.0
    _fill_normal(k_cache, gen, div, fp8)
    _fill_normal(v_cache, gen, div, fp8)
    ks = vs = None
    if fp8 and spec.token_scale_range is not None:
        lo, hi = (math.log(x) for x in spec.token_scale_range)
        shape = (pool, spec.num_kv_heads, PAGE_SIZE)
        ks = torch.exp(torch.rand(shape, generator=gen, device=device) * (hi - lo) + lo)
        vs = torch.exp(torch.rand(shape, generator=gen, device=device) * (hi - lo) + lo)
    return Workload(spec=spec, seq_lens=seq_lens, query_lens=query_lens,
                    query_start_loc=qsl, block_tables=block_tables, num_pages=pool,
                    q=q, k_cache=k_cache, v_cache=v_cache, k_token_scales=ks, v_token_scales=vs)


def custom_spec(name="custom", num_seqs=None, num_q_heads=4, num_kv_heads=2, head_dim=64,
                kv_dtype="bf16", seq_lens=(5, 16, 33), query_len_choices=(1,),
                pool_pages=None, k_scale=1.0, v_scale=1.0, fp8_source_scale=1.0,
                seed=7, token_scale_range=None) -> WorkloadSpec:
    """A small spec with explicit sequence lengths (for edge cases)."""
    return WorkloadSpec(name=name, num_seqs=len(seq_lens) if num_seqs is None else num_seqs,
                        num_q_heads=num_q_heads,
                        num_kv_heads=num_kv_heads, head_dim=head_dim, kv_dtype=kv_dtype,
                        seq_len_kind="fixed", seq_len_args=tuple(seq_lens),
                        query_len_choices=tuple(query_len_choices), pool_pages=pool_pages,
                        k_scale=k_scale, v_scale=v_scale, fp8_source_scale=fp8_source_scale,
                        seed=seed, token_scale_range=token_scale_range)


def host_arrays(w: Workload):
    """Raw host copies for the CPU side: bf16 as uint16 bit patterns, fp8 as
    uint8 codes."""
    q_bits = w.q.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    if w.spec.kv_dtype == "fp8":
        k = w.k_cache.detach().cpu().contiguous().numpy()
        v = w.v_cache.detach().cpu().contiguous().numpy()
    else:
        k = w.k_cache.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        v = w.v_cache.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return q_bits, k, v


def host_token_scales(w: Workload):
    """Host float32 copies of the per-token scales, or (None, None)."""
    if w.k_token_scales is None:
        return None, None
    return (w.k_token_scales.detach().cpu().contiguous().numpy(),
            w.v_token_scales.detach().cpu().contiguous().numpy())


# ---------------------------------------------------------------------------
# Multi-head latent attention (MLA) decode inputs.
#
# Layout (ATOM model-operations guide, "Multi-head latent attention": the
# ``MLAModules`` fields and the decode flow, where the absorbed query and one
# concatenated latent row per token meet in the decode kernel):
#
# * ``q``         bf16 ``[T, Hq, kv_lora_rank + rope]``: per query head the
#                 absorbed no-position part followed by the rotary part
# * ``kv_cache``  bf16 or fp8-e4m3 codes ``[NB, 16, kv_lora_rank + rope]``:
#                 per token the compressed latent followed by the rotary key
# * ``block_tables``, ``seq_lens``, ``query_start_loc`` as above.
#
# Dimensions are DeepSeek-V3's public ones (kv_lora_rank 512, rope 64, 128
# heads of qk_nope 128 + rope 64): the softmax scale is 1/sqrt(128 + 64).

@dataclasses.dataclass
class MlaSpec:
    """Shape and distribution of one synthetic MLA decode batch."""

    name: str
    num_seqs: int
    num_q_heads: int
    kv_dtype: str                      # "bf16" or "fp8"
    seq_len_kind: str
    seq_len_args: tuple
    query_len_choices: tuple = (1,)
    pool_pages: Optional[int] = None
    kv_lora_rank: int = 512
    rope_dim: int = 64
    qk_nope_head_dim: int = 128
    kv_scale: float = 1.0
    fp8_source_scale: float = 1.0
    seed: int = 0

    @property
    def head_dim(self) -> int:
        """Width of a cached row and of a query row."""
        return self.kv_lora_rank + self.rope_dim

    @property
    def max_query_len(self) -> int:
        return max(self.query_len_choices)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.qk_nope_head_dim + self.rope_dim)


# DeepSeek-V3-shaped MLA decode on one GPU of an 8-way tensor-parallel group
# (128 heads / 8 = 16 per GPU): a bf16 single-token batch, and an fp8 batch
# verifying query runs of four tokens (the MTP verification shape).
MLA_CONFIGS = {
    "mla_tiny": MlaSpec(
        name="mla_tiny", num_seqs=4, num_q_heads=16, kv_dtype="bf16", seq_len_kind="fixed",
        seq_len_args=(1, 17, 64, 200), pool_pages=64, seed=1007),
    "mla_tp8": MlaSpec(
        name="mla_tp8", num_seqs=64, num_q_heads=16, kv_dtype="bf16", seq_len_kind="uniform",
        seq_len_args=(512, 4096), seed=1008),
    "mla_mtp_fp8": MlaSpec(
        name="mla_mtp_fp8", num_seqs=32, num_q_heads=16, kv_dtype="fp8", seq_len_kind="uniform",
        seq_len_args=(1024, 16384), query_len_choices=(4,), kv_scale=0.05, fp8_source_scale=0.05, seed=1009),
}


@dataclasses.dataclass
class MlaWorkload:
    spec: MlaSpec
    seq_lens: np.ndarray
    query_lens: np.ndarray
    query_start_loc: Optional[np.ndarray]
    block_tables: np.ndarray
    num_pages: int
    q: torch.Tensor                 # bf16 [T, Hq, Dqk]
    kv_cache: torch.Tensor          # bf16 or uint8 (e4m3 codes) [NB, 16, Dqk]

    @property
    def num_tokens(self) -> int:
        return int(self.query_lens.sum())

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.spec.kv_dtype == "fp8" else 2

    def kv_bytes(self) -> int:
        """Algorithmic cache bytes of one step: every cached token's latent row
        (latent and rotary parts) read once; the value is part of that row."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.spec.head_dim * self.kv_elem_bytes


def make_mla_workload(spec: MlaSpec, device: str = "cpu", seed: Optional[int] = None,
                      content_seed: Optional[int] = None) -> MlaWorkload:
    """One seeded MLA batch: metadata from numpy's PCG64 with ``seed``, tensor
    contents from torch's generator on ``device`` with ``content_seed``
    (default: ``seed``): q and cache rows N(0,1); fp8 codes
    e4m3(N(0,1) / fp8_source_scale).  Batches that differ only in
    ``content_seed`` share lengths, block tables and pool size."""
    seed = spec.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    seq_lens, query_lens, qsl, block_tables, pool = draw_metadata(spec, rng)
    T = int(query_lens.sum())
    gen = torch.Generator(device=device)
    gen.manual_seed(seed if content_seed is None else content_seed)
    fp8 = spec.kv_dtype == "fp8"
    q = torch.empty((T, spec.num_q_heads, spec.head_dim), dtype=torch.bfloat16, device=device)
    _fill_normal(q, gen, 1.0, False)
    cache = torch.empty((pool, PAGE_SIZE, spec.head_dim), dtype=torch.uint8 if fp8 else torch.bfloat16,
                        device=device)
    _fill_normal(cache, gen, spec.fp8_source_scale if fp8 else 1.0, fp8)
    return MlaWorkload(spec=spec, seq_lens=seq_lens, query_lens=query_lens, query_start_loc=qsl,
                       block_tables=block_tables, num_pages=pool, q=q, kv_cache=cache)


def custom_mla_spec(name="custom_mla", num_q_heads=16, kv_dtype="bf16", seq_lens=(5, 16, 33),
                    query_len_choices=(1,), pool_pages=None, kv_scale=1.0, fp8_source_scale=1.0, seed=11,
                    kv_lora_rank=512, rope_dim=64) -> MlaSpec:
    """A small MLA spec with explicit sequence lengths (for edge cases)."""
    return MlaSpec(name=name, num_seqs=len(seq_lens), num_q_heads=num_q_heads, kv_dtype=kv_dtype,
                   seq_len_kind="fixed", seq_len_args=tuple(seq_lens), query_len_choices=tuple(query_len_choices),
                   pool_pages=pool_pages, kv_lora_rank=kv_lora_rank, rope_dim=rope_dim, kv_scale=kv_scale,
                   fp8_source_scale=fp8_source_scale, seed=seed)


def host_mla_arrays(w: MlaWorkload):
    """Host copies for the CPU side: q as uint16 bf16 patterns, the cache as
    uint16 patterns (bf16) or uint8 codes (fp8)."""
    q_bits = w.q.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    if w.spec.kv_dtype == "fp8":
        c = w.kv_cache.detach().cpu().contiguous().numpy()
    else:
        c = w.kv_cache.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return q_bits, c
