"""ctypes front end of the plain-C float64 oracle (``oracle/pa_oracle.c``).

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): used by ``tests/`` and
by the CPU-baseline leg of ``bench.py``; the CUDA library never loads it.
``build()`` compiles the C file with gcc (OpenMP when the compiler has it) into
``oracle/libpa_oracle.so``; nothing here shares code with the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
LIB = os.path.join(HERE, "libpa_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle if its source is newer than the library."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp"
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", "-o", tmp, SRC, "-lm"]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:                      # no OpenMP runtime: a serial build
        r = subprocess.run(base, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"gcc failed for {SRC}:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(LIB)
        P = ctypes.c_void_p
        lib.pa_oracle_decode.restype = ctypes.c_int
        lib.pa_oracle_decode.argtypes = [P, P, P, ctypes.c_int, P, ctypes.c_int64, P, P, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                         ctypes.c_float, ctypes.c_float, P, P, ctypes.c_int, P, P, P, P,
                                         ctypes.c_int]
        lib.pa_oracle_mla_decode.restype = ctypes.c_int
        lib.pa_oracle_mla_decode.argtypes = [P, P, ctypes.c_int, P, ctypes.c_int64, P, P, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                             ctypes.c_float, P, P, P, ctypes.c_int]
        lib.pa_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return load().pa_oracle_max_threads()


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def paged_decode_attention(q_bits, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale,
                           k_scale=1.0, v_scale=1.0, kv_dtype="bf16", seqs=None, sliding_window=0, sinks=None,
                           k_token_scales=None, v_token_scales=None, threads=0):
    """Same arguments and results as ``oracle.paged_decode_attention`` (plus
    ``threads``: OpenMP threads, 0 = all); rows outside ``seqs`` are NaN."""
    lib = load()
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    fp8 = kv_dtype == "fp8"
    k = np.ascontiguousarray(k_cache, dtype=np.uint8 if fp8 else np.uint16)
    v = np.ascontiguousarray(v_cache, dtype=np.uint8 if fp8 else np.uint16)
    T, Hq, D = q.shape
    NB, _, Hkv, _ = k.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = len(sl)
    qsl = None if query_start_loc is None else np.ascontiguousarray(query_start_loc, dtype=np.int32)
    kt = None if k_token_scales is None else np.ascontiguousarray(k_token_scales, dtype=np.float32)
    vt = None if v_token_scales is None else np.ascontiguousarray(v_token_scales, dtype=np.float32)
    sk = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float32)
    mask = None
    if seqs is not None:
        mask = np.zeros(B, dtype=np.uint8)
        mask[list(seqs)] = 1
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    st = lib.pa_oracle_decode(_ptr(q), _ptr(k), _ptr(v), int(fp8), _ptr(bt), bt.shape[1], _ptr(sl), _ptr(qsl), B, T,
                              Hq, Hkv, D, NB, float(scale), float(k_scale), float(v_scale), _ptr(kt), _ptr(vt),
                              int(sliding_window), _ptr(sk), _ptr(out), _ptr(lse), _ptr(mask), int(threads))
    if st != 0:
        raise ValueError("C oracle rejected the inputs")
    return out, lse


def run_workload(w, seqs=None, sliding_window=0, sinks=None, threads=0):
    """C-oracle outputs for a ``paged_kv_decode_06_gb300.workloads.Workload``."""
    from paged_kv_decode_06_gb300.workloads import host_arrays, host_token_scales
    q_bits, k, v = host_arrays(w)
    s = w.spec
    ks, vs = host_token_scales(w)
    return paged_decode_attention(q_bits, k, v, w.block_tables, w.seq_lens, w.query_start_loc, s.scale, s.k_scale,
                                  s.v_scale, s.kv_dtype, seqs=seqs, sliding_window=sliding_window, sinks=sinks,
                                  k_token_scales=ks, v_token_scales=vs, threads=threads)


def mla_decode(q_bits, cache, block_tables, seq_lens, query_start_loc, scale, kv_scale=1.0, kv_dtype="bf16",
               kv_lora_rank=512, seqs=None, threads=0):
    """Same arguments and results as ``oracle.mla_decode`` (plus ``threads``);
    rows outside ``seqs`` are NaN."""
    lib = load()
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    fp8 = kv_dtype == "fp8"
    c = np.ascontiguousarray(cache, dtype=np.uint8 if fp8 else np.uint16)
    T, Hq, Dqk = q.shape
    NB = c.shape[0]
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = len(sl)
    qsl = None if query_start_loc is None else np.ascontiguousarray(query_start_loc, dtype=np.int32)
    mask = None
    if seqs is not None:
        mask = np.zeros(B, dtype=np.uint8)
        mask[list(seqs)] = 1
    out = np.full((T, Hq, kv_lora_rank), np.nan)
    lse = np.full((T, Hq), np.nan)
    st = lib.pa_oracle_mla_decode(_ptr(q), _ptr(c), int(fp8), _ptr(bt), bt.shape[1], _ptr(sl), _ptr(qsl), B, T, Hq,
                                  Dqk, int(kv_lora_rank), NB, float(scale), float(kv_scale), _ptr(out), _ptr(lse),
                                  _ptr(mask), int(threads))
    if st != 0:
        raise ValueError("C oracle rejected the inputs")
    return out, lse


def run_mla_workload(w, seqs=None, threads=0):
    """C-oracle outputs for a ``paged_kv_decode_06_gb300.workloads.MlaWorkload``."""
    from paged_kv_decode_06_gb300.workloads import host_mla_arrays
    q_bits, c = host_mla_arrays(w)
    s = w.spec
    return mla_decode(q_bits, c, w.block_tables, w.seq_lens, w.query_start_loc, s.scale, s.kv_scale, s.kv_dtype,
                      s.kv_lora_rank, seqs=seqs, threads=threads)
