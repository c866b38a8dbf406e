"""Float64 CPU oracle for paged decode attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the library.  It shares no
code with the CUDA path.  Its parity pins live in ``tests/test_oracle.py``.
"""
from .paged_attention import (PAGE_SIZE, attend, bf16_bits_to_float64, dequantize,
                              e4m3fn_to_float64, gather_sequence, gather_token_scales,
                              paged_decode_attention,
                              run_workload)

from .mla import decode_latent, gather_latent, mla_decode, run_mla_workload

from .cache_write import (cache_write, cache_write_per_token, e4m3fn_encode, quantize_rows,
                          quantize_rows_per_token)

__all__ = ["decode_latent", "gather_latent", "mla_decode", "run_mla_workload", "cache_write", "cache_write_per_token", "quantize_rows_per_token", "e4m3fn_encode", "quantize_rows", "PAGE_SIZE", "attend", "bf16_bits_to_float64", "dequantize", "e4m3fn_to_float64",
           "gather_sequence", "gather_token_scales", "paged_decode_attention", "run_workload"]
