"""Float64 CPU oracle for the paged KV-cache write (TEST INFRASTRUCTURE ONLY).

What it computes (ATOM model-operations guide, "KV cache operations": standard
and FP8 KV cache write; model-operations guide, token_layout/slots.py:
``slot_mapping`` gives the KV slot a token is written to): each new token t
with slot s = slot_mapping[t] >= 0 stores its key and value rows of every KV
head at physical page s // 16, slot s % 16 of the caches; tokens with a
negative slot (padding) write nothing.  bf16 caches take the bf16 rows
unchanged; fp8 caches take e4m3fn codes of ``float32(x) / float32(scale)``,
one IEEE fp32 division by the tensor's one fp32 scale: a cached value is
read back as code * scale, so the code is the value divided by the scale.

Per-token quantisation (the pages' ``reshape_and_cache_with_pertoken_quant``,
FP8 KV cache write of MHA layers): every written (token, KV head) row gets its
own scale.  Readings adopted: the row's scale is ``s = float32(amax) / 448``
with ``amax = max_d |x_d|`` (448 = the largest finite e4m3fn magnitude), one
IEEE fp32 division; the codes are ``e4m3fn(float32(x) / s)``, again one IEEE
fp32 division by the stored scale (a row is read back as code * s, the same
rule as the per-tensor write), so the largest element lands on +-448 up to one
rounding; an all-zero row stores scale 0 and the code 0x00 throughout (its
-0 elements too: x / 0 has no value to take a sign from).  Scales are stored
``[num_pages, num_kv_heads, 16]`` float32.

Readings adopted where the pages are silent: the e4m3fn encoding rounds to
nearest, ties to even, and saturates finite magnitudes above 448 (and
infinities) to +-448 (the "satfinite" convention); a slot at or past the end
of the pool is an error and writes nothing.
"""
from __future__ import annotations

import numpy as np

from .paged_attention import PAGE_SIZE, bf16_bits_to_float64, e4m3fn_to_float64

_CODES = np.arange(0x7F, dtype=np.uint8)              # non-negative finite codes 0x00..0x7E
_VALUES = e4m3fn_to_float64(_CODES)                    # increasing with the code


def e4m3fn_encode(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3fn code, ties to the even code, saturating to +-448.

    Works on float64 copies of the inputs: for |x| below 448, the two grid
    values around |x| are found by search and the nearer one is taken (the one
    with the even code on a tie); |x| >= 448 and infinities give 448.  The sign
    bit is copied.  NaN encodes as 0x7F (0xFF when the sign bit is set)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    finite_a = np.where(np.isnan(a), 0.0, np.minimum(a, _VALUES[-1]))
    hi = np.searchsorted(_VALUES, finite_a, side="left")          # first grid value >= |x|
    lo = np.maximum(hi - 1, 0)
    d_lo = finite_a - _VALUES[lo]
    d_hi = _VALUES[hi] - finite_a
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(_VALUES[hi] == finite_a, hi, np.where(pick_lo, lo, hi)).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    code = np.where(np.isnan(x), np.where(np.signbit(x), 0xFF, 0x7F), code).astype(np.uint8)
    return code


def quantize_rows(bits: np.ndarray, scale: float) -> np.ndarray:
    """bf16 rows -> e4m3fn codes of float32(x) / float32(scale) (IEEE fp32 division)."""
    x32 = bf16_bits_to_float64(bits).astype(np.float32)
    with np.errstate(over="ignore"):           # a quotient past the fp32 range saturates below
        y32 = x32 / np.float32(scale)
    return e4m3fn_encode(y32.astype(np.float64))


def cache_write(key_bits, value_bits, slot_mapping, k_cache, v_cache, k_scale=1.0, v_scale=1.0,
                kv_dtype="bf16"):
    """Return new (k_cache, v_cache) after writing tokens into their slots.

    key_bits/value_bits uint16 bf16 patterns [T, Hkv, D]; slot_mapping int [T];
    k_cache/v_cache uint16 (bf16) or uint8 (e4m3) [NB, 16, Hkv, D].
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    NB = k_out.shape[0]
    for t, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if s < 0 or s >= NB * PAGE_SIZE:
            continue
        page, off = int(s) // PAGE_SIZE, int(s) % PAGE_SIZE
        if kv_dtype == "bf16":
            k_out[page, off] = key_bits[t]
            v_out[page, off] = value_bits[t]
        else:
            k_out[page, off] = quantize_rows(key_bits[t], k_scale)
            v_out[page, off] = quantize_rows(value_bits[t], v_scale)
    return k_out, v_out


E4M3_MAX = 448.0


def quantize_rows_per_token(bits: np.ndarray):
    """bf16 rows [..., D] -> (e4m3fn codes [..., D], float32 scales [...]).

    amax = max_d |x_d|; scale = float32(amax) / float32(448);
    codes = e4m3fn(float32(x) / scale) (IEEE fp32 division), or zeros with
    scale 0 when amax == 0."""
    x32 = bf16_bits_to_float64(bits).astype(np.float32)
    amax = np.abs(x32).max(axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    nonzero = scale > 0
    y32 = np.where(nonzero[..., None], x32 / np.where(nonzero, scale, np.float32(1))[..., None], np.float32(0))
    return e4m3fn_encode(y32.astype(np.float32).astype(np.float64)), scale


def cache_write_per_token(key_bits, value_bits, slot_mapping, k_cache, v_cache, k_scales, v_scales):
    """Per-token fp8 write: new (k_cache, v_cache, k_scales, v_scales).

    key_bits/value_bits uint16 bf16 [T, Hkv, D]; caches uint8 [NB, 16, Hkv, D];
    scales float32 [NB, Hkv, 16].  Slots as in ``cache_write``."""
    k_out, v_out = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
    ks_out = np.array(k_scales, dtype=np.float32, copy=True)
    vs_out = np.array(v_scales, dtype=np.float32, copy=True)
    NB = k_out.shape[0]
    for t, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if not 0 <= s < NB * PAGE_SIZE:        # padding or past the pool
            continue
        page, off = divmod(int(s), PAGE_SIZE)
        kc, ksc = quantize_rows_per_token(key_bits[t])          # [Hkv, D], [Hkv]
        vc, vsc = quantize_rows_per_token(value_bits[t])
        k_out[page, off], v_out[page, off] = kc, vc
        ks_out[page, :, off], vs_out[page, :, off] = ksc, vsc
    return k_out, v_out, ks_out, vs_out
