"""Thin ctypes binding over the C ABI of ``include/paged_attn.h``.

Argument marshalling only: every step of the computation runs in the CUDA
library.  If the library has not been built, ``load()`` raises; there is no
fallback implementation.  Function names mirror the C entry points.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpagedattn.so")

PA_BF16, PA_FP8_E4M3, PA_F32, PA_I32 = 1, 2, 3, 4
PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = 0, 1, 2, 3, 4

STATUS_PAGE_RANGE, STATUS_SEQ_LEN, STATUS_QUERY_LEN, STATUS_TIMEOUT, STATUS_F16_RANGE = 1, 2, 4, 8, 16


class PaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class PaOptions(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int32), ("min_pages_per_cta", ctypes.c_int32),
                ("heads_per_cta", ctypes.c_int32), ("disable_pdl", ctypes.c_int32),
                ("page_pairing", ctypes.c_int32), ("sliding_window", ctypes.c_int32),
                ("sinks", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("split_start_event", ctypes.c_void_p), ("split_stop_event", ctypes.c_void_p),
                ("use_tcgen05", ctypes.c_int32),
                ("k_token_scales", ctypes.POINTER(PaTensor)), ("v_token_scales", ctypes.POINTER(PaTensor)),
                ("wait_limit_us", ctypes.c_int32), ("test_starve_cta", ctypes.c_int32),
                ("segment_cost_pages", ctypes.c_int32)]


class PaPlan(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int32), ("heads_per_cta", ctypes.c_int32), ("row_tiles", ctypes.c_int32),
                ("num_stages", ctypes.c_int32), ("threads_per_cta", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("min_pages_per_cta", ctypes.c_int32), ("merge_rows", ctypes.c_int32),
                ("page_pairing", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("variant", ctypes.c_int32),
                ("block_pages", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"status {status}: {message}")
        self.status = status


_P = ctypes.POINTER(PaTensor)
_SIGNATURES = {
    "paged_attn_decode": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                                         ctypes.c_float, _P, _P, ctypes.c_void_p]),
    "paged_attn_decode_ex": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                                            ctypes.c_float, _P, _P, ctypes.POINTER(PaOptions), ctypes.c_void_p]),
    "paged_attn_decode_static_scratch": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int32, ctypes.c_float,
                                                        ctypes.c_float, ctypes.c_float, _P, _P, ctypes.c_void_p]),
    "paged_attn_cache_write": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_float, ctypes.c_float, ctypes.c_void_p]),
    "paged_attn_cache_write_per_token": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_void_p]),
    "paged_attn_mla_decode": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int32, ctypes.c_float, ctypes.c_float, _P,
                                             _P, ctypes.c_void_p]),
    "paged_attn_mla_decode_ex": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                                                _P, _P, ctypes.POINTER(PaOptions), ctypes.c_void_p]),
    "paged_attn_mla_plan": (ctypes.c_int, [ctypes.c_int32] * 4 + [ctypes.POINTER(PaOptions), ctypes.POINTER(PaPlan)]),
    "paged_attn_mla_workspace_size": (ctypes.c_int, [ctypes.c_int32] * 4 + [ctypes.POINTER(ctypes.c_size_t)]),
    "paged_attn_mla_reserve": (ctypes.c_int, [ctypes.c_int32] * 4),
    "paged_attn_plan": (ctypes.c_int, [ctypes.c_int32] * 6 + [ctypes.POINTER(PaOptions), ctypes.POINTER(PaPlan)]),
    "paged_attn_workspace_size": (ctypes.c_int, [ctypes.c_int32] * 6 + [ctypes.POINTER(ctypes.c_size_t)]),
    "paged_attn_reserve": (ctypes.c_int, [ctypes.c_int32] * 6),
    "paged_attn_release": (ctypes.c_int, []),
    "paged_attn_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32]),
    "paged_attn_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "paged_attn_last_error_message": (ctypes.c_char_p, []),
    "paged_attn_version": (ctypes.c_int32, []),
}

EXPORTED = tuple(_SIGNATURES)
_lib = None


def load(path: Optional[str] = None):
    """Load the built library (``build.build()`` makes it).  Raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing (run paged_kv_decode_06_gb300.build.build())")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return PA_FP8_E4M3
    if t.dtype == torch.float32:
        return PA_F32
    if t.dtype == torch.int32:
        return PA_I32
    return 0          # not a pa_dtype: the library rejects it with PA_ERR_INVALID_ARG


_DESC_CACHE = {}
_DESC_CACHE_MAX = 1024


def tensor_desc(t: Optional[torch.Tensor]) -> PaTensor:
    """The pa_tensor_t of a tensor.  Descriptors hold only (pointer, dtype,
    shape, strides), so one built for a key serves every later tensor with the
    same key: they are cached (a per-call decode then costs a few dictionary
    lookups instead of ctypes field assignments).  Treat the result as
    read-only."""
    if t is None:
        return _new_desc(None)
    key = (t.data_ptr(), t.dtype, t.shape, t.stride())
    d = _DESC_CACHE.get(key)
    if d is None:
        d = _new_desc(t)
        if len(_DESC_CACHE) >= _DESC_CACHE_MAX:
            _DESC_CACHE.clear()
        _DESC_CACHE[key] = d
    return d


def _new_desc(t: Optional[torch.Tensor]) -> PaTensor:
    d = PaTensor()
    if t is None:
        d.data = None
        return d
    if t.dim() > 4:
        raise ValueError("at most 4 dimensions")
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _dtype_code(t)
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _check(lib, status: int):
    if status != PA_OK:
        raise PagedAttnError(status, lib.paged_attn_last_error_message().decode() or
                             lib.paged_attn_error_string(status).decode())


# The current stream's raw handle without building a torch.cuda.Stream object
# (about 0.2 us a call instead of 3); the public route where torch lacks it.
_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream) -> int:
    if stream is None:
        if _RAW_STREAM is not None:
            return int(_RAW_STREAM(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def make_options(num_ctas=0, min_pages_per_cta=0, heads_per_cta=0, disable_pdl=False, workspace=None,
                 workspace_bytes=0, split_start_event=None, split_stop_event=None, page_pairing=0,
                 sliding_window=0, sinks=None, use_tcgen05=0, k_token_scales=None,
                 v_token_scales=None, wait_limit_us=0, test_starve_cta=0,
                 segment_cost_pages=0) -> PaOptions:
    """Options for paged_attn_decode_ex.  sinks: CUDA float32 tensor [Hq] (kept
    alive by the caller) or None.  use_tcgen05: 0 planner's choice, 1 never,
    2 always (bf16 caches).  k_token_scales / v_token_scales: CUDA float32
    [NB, Hkv, 16] per-token scales of an fp8 cache (kept alive by the caller).
    wait_limit_us: pipeline wait limit (0 = 2 s).  test_starve_cta: testing aid,
    k > 0 makes split CTA k-1 receive no pages (its waits run out).
    segment_cost_pages: tensor-memory MLA work split, pages charged per unit a
    CTA starts (0 planner's value, < 0 equal page split)."""
    o = PaOptions()
    o.num_ctas = num_ctas
    o.min_pages_per_cta = min_pages_per_cta
    o.heads_per_cta = heads_per_cta
    o.disable_pdl = int(bool(disable_pdl))
    o.page_pairing = page_pairing
    o.sliding_window = sliding_window
    o.use_tcgen05 = use_tcgen05
    o.wait_limit_us = wait_limit_us
    o.test_starve_cta = test_starve_cta
    o.segment_cost_pages = segment_cost_pages
    if sinks is not None:
        if sinks.dtype != torch.float32 or not sinks.is_contiguous():
            raise TypeError("sinks must be a contiguous float32 tensor")
        o.sinks = sinks.data_ptr()
    else:
        o.sinks = None
    o.workspace = workspace
    o.workspace_bytes = workspace_bytes
    o.split_start_event = int(split_start_event.cuda_event) if split_start_event is not None else None
    o.split_stop_event = int(split_stop_event.cuda_event) if split_stop_event is not None else None
    if k_token_scales is not None or v_token_scales is not None:
        # the descriptors live as long as the options object
        o._tok_descs = (tensor_desc(k_token_scales), tensor_desc(v_token_scales))
        o.k_token_scales = ctypes.pointer(o._tok_descs[0])
        o.v_token_scales = ctypes.pointer(o._tok_descs[1])
    return o


def paged_attn_decode(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc=None, max_query_len=1,
                      scale=None, k_scale=1.0, v_scale=1.0, out=None, lse=None, stream=None, options=None,
                      want_lse=True):
    """Decode attention over a paged KV cache (see include/paged_attn.h).

    Tensors are CUDA tensors: q bf16 [T, Hq, D]; k_cache / v_cache bf16 or
    uint8 (e4m3fn codes) [NB, 16, Hkv, D]; block_tables int32 [B, max_blocks];
    seq_lens int32 [B]; query_start_loc int32 [B+1] or None.  Returns
    (out bf16 [T, Hq, D], lse f32 [T, Hq] or None)."""
    lib = load()
    if scale is None:
        scale = q.shape[-1] ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    args = [tensor_desc(t) for t in (q, k_cache, v_cache, block_tables, seq_lens, query_start_loc)]
    o_desc, l_desc = tensor_desc(out), tensor_desc(lse)
    refs = [ctypes.byref(a) for a in args]
    if options is None:
        st = lib.paged_attn_decode(*refs, int(max_query_len), float(scale), float(k_scale), float(v_scale),
                                   ctypes.byref(o_desc), ctypes.byref(l_desc), _stream_handle(stream))
    else:
        st = lib.paged_attn_decode_ex(*refs, int(max_query_len), float(scale), float(k_scale), float(v_scale),
                                      ctypes.byref(o_desc), ctypes.byref(l_desc), ctypes.byref(options),
                                      _stream_handle(stream))
    _check(lib, st)
    return out, lse


def paged_attn_decode_static_scratch(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc=None,
                                     max_query_len=1, scale=None, k_scale=1.0, v_scale=1.0, out=None, lse=None,
                                     stream=None, want_lse=True):
    """paged_attn_decode without any device allocation inside the library:
    the split scratch is the library's fixed 16 MiB static device array.
    Same arguments and results as ``paged_attn_decode``."""
    lib = load()
    if scale is None:
        scale = q.shape[-1] ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    args = [tensor_desc(t) for t in (q, k_cache, v_cache, block_tables, seq_lens, query_start_loc)]
    o_desc, l_desc = tensor_desc(out), tensor_desc(lse)
    st = lib.paged_attn_decode_static_scratch(*[ctypes.byref(a) for a in args], int(max_query_len), float(scale),
                                              float(k_scale), float(v_scale), ctypes.byref(o_desc),
                                              ctypes.byref(l_desc), _stream_handle(stream))
    _check(lib, st)
    return out, lse


def paged_attn_cache_write(key, value, slot_mapping, k_cache, v_cache, k_scale=1.0, v_scale=1.0, stream=None):
    """Write new tokens' K/V rows into their page slots (see include/paged_attn.h).
    key/value bf16 [T, Hkv, D]; slot_mapping int32 [T]; caches bf16 or uint8
    (e4m3fn codes) [NB, 16, Hkv, D], updated in place."""
    lib = load()
    d = [tensor_desc(t) for t in (key, value, slot_mapping, k_cache, v_cache)]
    _check(lib, lib.paged_attn_cache_write(*[ctypes.byref(x) for x in d], float(k_scale), float(v_scale),
                                           _stream_handle(stream)))


def paged_attn_cache_write_per_token(key, value, slot_mapping, k_cache, v_cache, k_token_scales, v_token_scales,
                                     stream=None):
    """Per-token fp8 cache write (see include/paged_attn.h): codes of each
    (token, head) row quantised with its own scale amax / 448, written into
    the uint8 caches [NB, 16, Hkv, D]; the scales go to the float32 tensors
    [NB, Hkv, 16].  All updated in place."""
    lib = load()
    d = [tensor_desc(t) for t in (key, value, slot_mapping, k_cache, v_cache, k_token_scales, v_token_scales)]
    _check(lib, lib.paged_attn_cache_write_per_token(*[ctypes.byref(x) for x in d], _stream_handle(stream)))


def paged_attn_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype=PA_BF16, max_query_len=1,
                    options=None) -> dict:
    lib = load()
    plan = PaPlan()
    st = lib.paged_attn_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype, max_query_len,
                             ctypes.byref(options) if options is not None else None, ctypes.byref(plan))
    _check(lib, st)
    return plan.as_dict()


def paged_attn_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype=PA_BF16, max_query_len=1):
    lib = load()
    n = ctypes.c_size_t(0)
    _check(lib, lib.paged_attn_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype,
                                              max_query_len, ctypes.byref(n)))
    return n.value


def paged_attn_reserve(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype=PA_BF16, max_query_len=1):
    lib = load()
    _check(lib, lib.paged_attn_reserve(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype, max_query_len))


def paged_attn_release():
    lib = load()
    _check(lib, lib.paged_attn_release())


def paged_attn_device_status(clear: bool = True) -> int:
    lib = load()
    flags = ctypes.c_uint32(0)
    _check(lib, lib.paged_attn_device_status(ctypes.byref(flags), int(clear)))
    return flags.value


def paged_attn_error_string(status: int) -> str:
    return load().paged_attn_error_string(status).decode()


def paged_attn_last_error_message() -> str:
    return load().paged_attn_last_error_message().decode()


def paged_attn_version() -> int:
    return load().paged_attn_version()


def kv_dtype_code(kv_dtype: str) -> int:
    return PA_FP8_E4M3 if kv_dtype == "fp8" else PA_BF16


def decode_workload(w, out=None, lse=None, stream=None, options=None, want_lse=True):
    """Run the kernel on a ``workloads.Workload`` whose tensors live on the GPU.
    Metadata (block tables, lengths) is copied to the device here."""
    dev = w.q.device
    bt = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    qsl = torch.from_numpy(w.query_start_loc).to(dev) if w.query_start_loc is not None else None
    s = w.spec
    if w.k_token_scales is not None:
        if options is None:
            options = make_options()
        if not options.k_token_scales:
            options._tok_descs = (tensor_desc(w.k_token_scales), tensor_desc(w.v_token_scales))
            options.k_token_scales = ctypes.pointer(options._tok_descs[0])
            options.v_token_scales = ctypes.pointer(options._tok_descs[1])
    return paged_attn_decode(w.q, w.k_cache, w.v_cache, bt, sl, qsl, s.max_query_len if qsl is not None else 1,
                             s.scale, s.k_scale, s.v_scale, out=out, lse=lse, stream=stream, options=options,
                             want_lse=want_lse)


def paged_attn_mla_decode(q, kv_cache, block_tables, seq_lens, query_start_loc=None, max_query_len=1, scale=None,
                          kv_scale=1.0, out=None, lse=None, stream=None, options=None, want_lse=True):
    """MLA decode over a paged latent cache (see include/paged_attn.h).

    q bf16 [T, Hq, 576]; kv_cache bf16 or uint8 (e4m3fn codes) [NB, 16, 576];
    block_tables int32 [B, max_blocks]; seq_lens int32 [B]; query_start_loc
    int32 [B+1] or None.  Returns (out bf16 [T, Hq, 512], lse f32 [T, Hq] or
    None)."""
    lib = load()
    if scale is None:
        scale = 192 ** -0.5
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    args = [tensor_desc(t) for t in (q, kv_cache, block_tables, seq_lens, query_start_loc)]
    o_desc, l_desc = tensor_desc(out), tensor_desc(lse)
    refs = [ctypes.byref(a) for a in args]
    if options is None:
        st = lib.paged_attn_mla_decode(*refs, int(max_query_len), float(scale), float(kv_scale), ctypes.byref(o_desc),
                                       ctypes.byref(l_desc), _stream_handle(stream))
    else:
        st = lib.paged_attn_mla_decode_ex(*refs, int(max_query_len), float(scale), float(kv_scale),
                                          ctypes.byref(o_desc), ctypes.byref(l_desc), ctypes.byref(options),
                                          _stream_handle(stream))
    _check(lib, st)
    return out, lse


class PreparedCall:
    """One decode (or MLA decode) call with its arguments marshalled once, for
    a serving loop that reuses the same tensors every step and refreshes
    their contents in place (new q rows, block tables, lengths), as CUDA-graph
    static buffers are used.  ``call(stream=None)`` enqueues the C entry point
    with the stored descriptors on ``stream`` (None: torch's current stream)
    and returns (out, lse).  The tensors are kept referenced by the object;
    their addresses, shapes and strides must not change while it is used."""

    def __init__(self, fn, tensors, scalars, out, lse, options):
        self._lib = load()
        self._fn = fn
        self._keep = (tensors, out, lse, options)
        self._descs = [_new_desc(t) for t in tensors] + [_new_desc(out), _new_desc(lse)]
        n_in = len(tensors)
        refs = [ctypes.byref(d) for d in self._descs]
        head = refs[:n_in] + list(scalars) + refs[n_in:]
        if options is not None:
            head.append(ctypes.byref(options))
        self._args = tuple(head)
        self.out, self.lse = out, lse

    def __call__(self, stream=None):
        st = self._fn(*self._args, _stream_handle(stream))
        if st != PA_OK:
            _check(self._lib, st)
        return self.out, self.lse


def prepare_decode(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc=None, max_query_len=1, scale=None,
                   k_scale=1.0, v_scale=1.0, out=None, lse=None, options=None, want_lse=True) -> PreparedCall:
    """``paged_attn_decode`` with its arguments marshalled once (see PreparedCall)."""
    lib = load()
    if scale is None:
        scale = q.shape[-1] ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    scalars = (ctypes.c_int32(int(max_query_len)), ctypes.c_float(float(scale)), ctypes.c_float(float(k_scale)),
               ctypes.c_float(float(v_scale)))
    fn = lib.paged_attn_decode if options is None else lib.paged_attn_decode_ex
    return PreparedCall(fn, (q, k_cache, v_cache, block_tables, seq_lens, query_start_loc), scalars, out, lse, options)


def prepare_mla_decode(q, kv_cache, block_tables, seq_lens, query_start_loc=None, max_query_len=1, scale=None,
                       kv_scale=1.0, out=None, lse=None, options=None, want_lse=True) -> PreparedCall:
    """``paged_attn_mla_decode`` with its arguments marshalled once (see PreparedCall)."""
    lib = load()
    if scale is None:
        scale = 192 ** -0.5
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    scalars = (ctypes.c_int32(int(max_query_len)), ctypes.c_float(float(scale)), ctypes.c_float(float(kv_scale)))
    fn = lib.paged_attn_mla_decode if options is None else lib.paged_attn_mla_decode_ex
    return PreparedCall(fn, (q, kv_cache, block_tables, seq_lens, query_start_loc), scalars, out, lse, options)


def paged_attn_mla_plan(num_seqs, num_q_heads, kv_dtype=PA_BF16, max_query_len=1, options=None) -> dict:
    lib = load()
    plan = PaPlan()
    _check(lib, lib.paged_attn_mla_plan(num_seqs, num_q_heads, kv_dtype, max_query_len,
                                        ctypes.byref(options) if options is not None else None, ctypes.byref(plan)))
    return plan.as_dict()


def paged_attn_mla_workspace_size(num_seqs, num_q_heads, kv_dtype=PA_BF16, max_query_len=1) -> int:
    lib = load()
    n = ctypes.c_size_t(0)
    _check(lib, lib.paged_attn_mla_workspace_size(num_seqs, num_q_heads, kv_dtype, max_query_len, ctypes.byref(n)))
    return int(n.value)


def paged_attn_mla_reserve(num_seqs, num_q_heads, kv_dtype=PA_BF16, max_query_len=1):
    lib = load()
    _check(lib, lib.paged_attn_mla_reserve(num_seqs, num_q_heads, kv_dtype, max_query_len))


def mla_decode_workload(w, out=None, lse=None, stream=None, options=None, want_lse=True):
    """Run the MLA kernel on a ``workloads.MlaWorkload`` whose tensors live on
    the GPU (metadata is copied to the device here)."""
    dev = w.q.device
    bt = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    qsl = torch.from_numpy(w.query_start_loc).to(dev) if w.query_start_loc is not None else None
    s = w.spec
    return paged_attn_mla_decode(w.q, w.kv_cache, bt, sl, qsl, s.max_query_len if qsl is not None else 1, s.scale,
                                 s.kv_scale, out=out, lse=lse, stream=stream, options=options, want_lse=want_lse)
