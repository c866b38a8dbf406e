"""CUDA path vs the float64 oracle, element by element, through the C ABI.

Tolerances (max absolute error): out 1e-2 for bf16 caches, 2e-2 for fp8
caches; lse 1e-3.  Small cases are compared in full.  The full-size workloads
are compared on every query row against the plain-C float64 oracle (pinned to
the NumPy oracle to 1e-11; all host cores), and on sampled sequences against
the NumPy oracle as well, in the launch configuration the benchmark times (the
library's default plan)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import c_oracle
from paged_kv_decode_06_gb300 import binding
from paged_kv_decode_06_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_OUT = {"bf16": 1e-2, "fp8": 2e-2}
TOL_LSE = 1e-3


def _rows_of(w, seqs):
    qsl = w.query_start_loc if w.query_start_loc is not None else np.arange(w.spec.num_seqs + 1)
    return np.concatenate([np.arange(qsl[i], qsl[i + 1]) for i in seqs])


def check(w, seqs=None, options=None, ref=None, expect_status=0):
    out, lse = binding.decode_workload(w, options=options)
    torch.cuda.synchronize()
    status = binding.paged_attn_device_status(clear=True)
    assert status == expect_status, f"device status {status:#x}"
    if ref is None:
        ref = oracle.run_workload(w, seqs=seqs)
    ref_out, ref_lse = ref
    rows = _rows_of(w, range(w.spec.num_seqs) if seqs is None else seqs)
    o = out.float().cpu().numpy()[rows]
    l = lse.cpu().numpy()[rows]
    assert np.isfinite(o).all() and np.isfinite(l).all()
    err_o = np.abs(o - ref_out[rows]).max()
    err_l = np.abs(l - ref_lse[rows]).max()
    tol = TOL_OUT[w.spec.kv_dtype]
    assert err_o <= tol, f"max|out - oracle| = {err_o:.3e} > {tol}"
    assert err_l <= TOL_LSE, f"max|lse - oracle| = {err_l:.3e} > {TOL_LSE}"
    return out, lse, err_o, err_l


def _spec(kv="bf16", D=128, G=4, Hkv=2, seq_lens=(1, 15, 16, 17, 31, 32, 33, 100), qlens=(1,), seed=3,
          pool=None):
    fp8 = kv == "fp8"
    return wl.custom_spec(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, kv_dtype=kv, seq_lens=seq_lens,
                          query_len_choices=qlens, pool_pages=pool, seed=seed,
                          k_scale=0.05 if fp8 else 1.0, v_scale=0.05 if fp8 else 1.0,
                          fp8_source_scale=0.05 if fp8 else 1.0)


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    binding.paged_attn_device_status(clear=True)
    yield


def test_tiny_config_full():
    w = wl.make_workload(wl.CONFIGS["tiny"], device="cuda")
    check(w)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("D", [64, 128])
def test_page_boundaries_and_ragged_tails(kv, D):
    check(wl.make_workload(_spec(kv=kv, D=D), device="cuda"))


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("G,Hkv,qlens", [(8, 2, (2, 3, 4)), (4, 4, (1, 2)), (16, 1, (4,)), (1, 8, (1, 3)),
                                         (8, 1, (1,)), (2, 8, (3,))])
def test_group_sizes_and_mtp_runs(kv, G, Hkv, qlens):
    seq_lens = (4, 5, 16, 17, 40, 64, 130)
    check(wl.make_workload(_spec(kv=kv, G=G, Hkv=Hkv, qlens=qlens, seq_lens=seq_lens, seed=G * 10 + Hkv),
                           device="cuda"))


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 64, 152, 300])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_forced_split_counts_exercise_the_merge(num_ctas, kv):
    w = wl.make_workload(_spec(kv=kv, G=8, Hkv=2, qlens=(1, 2, 4), seq_lens=(3, 50, 300, 17, 1000), seed=num_ctas),
                         device="cuda")
    ref = oracle.run_workload(w)
    check(w, ref=ref, options=binding.make_options(num_ctas=num_ctas, min_pages_per_cta=1))


@pytest.mark.parametrize("hc", [1, 2, 4])
def test_heads_per_cta_variants(hc):
    w = wl.make_workload(_spec(G=4, Hkv=4, seq_lens=(7, 70, 700), seed=hc), device="cuda")
    ref = oracle.run_workload(w)
    check(w, ref=ref, options=binding.make_options(heads_per_cta=hc))
    check(w, ref=ref, options=binding.make_options(heads_per_cta=hc, num_ctas=5, min_pages_per_cta=1))


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_non_finite_tail_slots_and_unused_pages_do_not_leak(kv):
    w = wl.make_workload(_spec(kv=kv, seq_lens=(3, 17, 40, 1)), device="cuda")
    ref = oracle.run_workload(w)
    nan = torch.tensor(float("nan"))
    nan_code = nan.to(torch.bfloat16) if kv == "bf16" else torch.tensor(0x7F, dtype=torch.uint8)
    used = set()
    for i, L in enumerate(w.seq_lens):
        n = (int(L) + 15) // 16
        used.update(int(x) for x in w.block_tables[i, :n])
        last = int(w.block_tables[i, n - 1])
        tail = int(L) - 16 * (n - 1)
        w.k_cache[last, tail:] = nan_code
        w.v_cache[last, tail:] = nan_code
    for p in range(w.num_pages):
        if p not in used:
            w.k_cache[p] = nan_code
            w.v_cache[p] = nan_code
    check(w, ref=ref)


def test_strided_caches_and_lse_optional():
    spec = _spec(seq_lens=(20, 90, 33))
    w = wl.make_workload(spec, device="cuda")
    ref = oracle.run_workload(w)
    # K and V as two halves of one [NB, 2, 16, Hkv, D] allocation
    kv = torch.stack([w.k_cache, w.v_cache], dim=1).contiguous()
    w.k_cache, w.v_cache = kv[:, 0], kv[:, 1]
    assert not w.k_cache.is_contiguous()
    check(w, ref=ref)
    out, lse = binding.decode_workload(w, want_lse=False)
    assert lse is None
    torch.cuda.synchronize()
    assert np.abs(out.float().cpu().numpy() - ref[0]).max() <= TOL_OUT["bf16"]


def test_caller_workspace_and_deterministic_results():
    w = wl.make_workload(_spec(seq_lens=(500, 33, 1200), G=8, Hkv=2), device="cuda")
    n = binding.paged_attn_workspace_size(w.spec.num_seqs, w.spec.num_q_heads, w.spec.num_kv_heads,
                                          w.spec.head_dim)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    opts = binding.make_options(workspace=ws.data_ptr(), workspace_bytes=n)
    o1, l1, _, _ = check(w, options=opts)
    o2, l2 = binding.decode_workload(w)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    small = binding.make_options(workspace=ws.data_ptr(), workspace_bytes=64)
    with pytest.raises(binding.PagedAttnError) as e:
        binding.decode_workload(w, options=small)
    assert e.value.status == binding.PA_ERR_WORKSPACE


def test_out_of_range_page_id_is_reported():
    w = wl.make_workload(_spec(seq_lens=(40, 20)), device="cuda")
    w.block_tables = w.block_tables.copy()
    w.block_tables[0, 1] = w.num_pages + 5
    binding.decode_workload(w)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) & binding.STATUS_PAGE_RANGE


def test_cuda_graph_capture_and_replay_with_new_metadata():
    spec = _spec(seq_lens=(100, 300, 17, 64), G=4, Hkv=2, pool=200)
    w = wl.make_workload(spec, device="cuda")
    s = w.spec
    binding.paged_attn_reserve(s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim)
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    binding.paged_attn_decode(w.q, w.k_cache, w.v_cache, bt, sl, None, 1, s.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        binding.paged_attn_decode(w.q, w.k_cache, w.v_cache, bt, sl, None, 1, s.scale, out=out, lse=lse,
                                  stream=stream)
    rng = np.random.default_rng(5)
    for trial in range(3):
        new_lens = rng.integers(1, 301, size=s.num_seqs).astype(np.int32)
        n = (new_lens + 15) // 16
        perm = rng.permutation(w.num_pages)
        new_bt = np.full_like(w.block_tables, -1)
        cur = 0
        for i in range(s.num_seqs):
            new_bt[i, :n[i]] = perm[cur:cur + n[i]]
            cur += n[i]
        bt.copy_(torch.from_numpy(new_bt))
        sl.copy_(torch.from_numpy(new_lens))
        w.q.normal_()
        g.replay()
        torch.cuda.synchronize()
        w.block_tables, w.seq_lens = new_bt, new_lens
        ref = oracle.run_workload(w)
        assert np.abs(out.float().cpu().numpy() - ref[0]).max() <= TOL_OUT["bf16"]
        assert np.abs(lse.cpu().numpy() - ref[1]).max() <= TOL_LSE
    assert binding.paged_attn_device_status(clear=True) == 0


# ------------------------------------------------ full-size workloads (every row)

def _sample_seqs(w, k, seed):
    rng = np.random.default_rng(seed)
    B = w.spec.num_seqs
    idx = set(rng.choice(B, size=min(k, B), replace=False).tolist())
    idx.add(int(np.argmax(w.seq_lens)))
    idx.add(int(np.argmin(w.seq_lens)))
    return sorted(idx)


def check_every_row(w, **kw):
    """Every query row against the C oracle, then sampled sequences against
    the NumPy oracle (each on its own GPU call)."""
    _, _, eo, el = check(w, ref=c_oracle.run_workload(w), **kw)
    seqs = _sample_seqs(w, 3, seed=w.spec.seed)
    check(w, seqs=seqs, **kw)
    return eo, el


@pytest.mark.parametrize("name", ["llama3_8b", "batch1_32k", "fp8", "mtp"])
def test_full_size_configs_every_row(name):
    w = wl.make_workload(wl.CONFIGS[name], device="cuda")
    eo, el = check_every_row(w)
    print(f"{name}: all {w.q.shape[0]} query tokens: max|out err| {eo:.3e}, max|lse err| {el:.3e}")


# ------------------------------------------------ sliding window and attention sinks

def _check_opts(w, window=0, sinks=None, options_kw=None, ref=None):
    kw = dict(options_kw or {})
    sk_t = None
    if sinks is not None:
        sk_t = torch.from_numpy(np.asarray(sinks, dtype=np.float32)).cuda()
    opts = binding.make_options(sliding_window=window, sinks=sk_t, **kw)
    if ref is None:
        ref = oracle.run_workload(w, sliding_window=window, sinks=sinks)
    return check(w, options=opts, ref=ref)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("window", [1, 5, 16, 17, 100, 1000])
def test_sliding_window(kv, window):
    w = wl.make_workload(_spec(kv=kv, G=4, Hkv=2, qlens=(1, 2, 4), seq_lens=(3, 16, 17, 64, 250, 700), seed=window),
                         device="cuda")
    ref = oracle.run_workload(w, sliding_window=window)
    _check_opts(w, window=window, ref=ref)
    _check_opts(w, window=window, ref=ref, options_kw=dict(num_ctas=7, min_pages_per_cta=1))


def test_pages_before_the_window_are_never_read():
    w = wl.make_workload(_spec(G=4, Hkv=2, seq_lens=(300, 520, 77), seed=9), device="cuda")
    window = 40
    ref = oracle.run_workload(w, sliding_window=window)
    bt = w.block_tables.copy()
    for i, L in enumerate(w.seq_lens):
        first_page = max(0, int(L) - 1 - window + 1) // 16
        bt[i, :first_page] = w.num_pages + 1000          # out of range: reported if ever read
    w.block_tables = bt
    _check_opts(w, window=window, ref=ref)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("window", [0, 33])
@pytest.mark.parametrize("num_ctas", [0, 3, 64])
def test_attention_sinks(kv, window, num_ctas):
    w = wl.make_workload(_spec(kv=kv, G=8, Hkv=2, qlens=(1, 3), seq_lens=(1, 20, 200, 900), seed=num_ctas + 2),
                         device="cuda")
    rng = np.random.default_rng(num_ctas)
    sinks = rng.normal(0, 2, size=16).astype(np.float32)
    sinks[3] = 30.0                                   # a sink that dominates its rows
    ref = oracle.run_workload(w, sliding_window=window, sinks=sinks)
    kw = dict(num_ctas=num_ctas, min_pages_per_cta=1) if num_ctas else None
    _check_opts(w, window=window, sinks=sinks, options_kw=kw, ref=ref)


def test_split_timing_events_direct_and_captured():
    """split_start_event / split_stop_event bracket the split kernel both in a
    direct call and inside a captured graph (where they become event nodes)."""
    w = wl.make_workload(_spec(seq_lens=(300, 900, 40), G=4, Hkv=2), device="cuda")
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(); b.record()                      # torch times only events it has recorded once
    torch.cuda.synchronize()
    opts = binding.make_options(split_start_event=a, split_stop_event=b)
    out, lse = binding.decode_workload(w, options=opts)
    b.synchronize()
    assert a.elapsed_time(b) > 0.0
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    s = w.spec
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    cap = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        binding.paged_attn_decode(w.q, w.k_cache, w.v_cache, bt, sl, None, 1, s.scale, out=out2, lse=lse2,
                                  options=opts, stream=cap)
    g.replay()
    b.synchronize()
    assert a.elapsed_time(b) > 0.0
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("kv,qlens", [("bf16", (1,)), ("fp8", (1, 2, 3, 4)), ("bf16", (2, 3, 4))])
def test_batch_of_512_sequences(kv, qlens):
    # the engine's max_num_seqs: the device-side page prefix spans two scan passes
    rng = np.random.default_rng(513)
    lens = tuple(int(x) for x in rng.integers(4, 400, size=512))
    w = wl.make_workload(_spec(kv=kv, G=4, Hkv=8, qlens=qlens, seq_lens=lens, seed=513), device="cuda")
    seqs = sorted(set(rng.choice(512, size=16, replace=False).tolist()) | {0, 255, 256, 511})
    check(w, seqs=seqs)


# A sequence with an empty context (seq_len 0) owns no page: its rows come out
# as zeros with lse = -inf and the call reports status bit 1, while the other
# sequences (cut across CTAs, so merged) still match the oracle; with a forced
# split count and with every sequence empty.
@pytest.mark.parametrize("num_ctas", [0, 3])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_empty_context_rows_are_zero_and_reported(kv, num_ctas):
    w = wl.make_workload(_spec(kv=kv, seq_lens=(40, 17, 300, 5)), device="cuda")
    ref = oracle.run_workload(w)
    w.seq_lens = w.seq_lens.copy()
    w.seq_lens[1] = 0
    opts = binding.make_options(num_ctas=num_ctas, min_pages_per_cta=1) if num_ctas else None
    out, lse = binding.decode_workload(w, options=opts)
    torch.cuda.synchronize()
    status = binding.paged_attn_device_status(clear=True)
    assert status & binding.STATUS_SEQ_LEN
    rows = _rows_of(w, [0, 2, 3])
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    assert np.abs(o[rows] - ref[0][rows]).max() <= TOL_OUT[kv]
    assert np.abs(l[rows] - ref[1][rows]).max() <= TOL_LSE
    empty = _rows_of(w, [1])
    assert (o[empty] == 0).all() and np.isneginf(l[empty]).all()
    w.seq_lens[:] = 0
    out, lse = binding.decode_workload(w, options=opts)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) & binding.STATUS_SEQ_LEN
    assert (out.float().cpu().numpy() == 0).all() and np.isneginf(lse.cpu().numpy()).all()


def test_calls_run_on_the_current_stream_and_reuse_tensor_maps():
    """With no stream argument the call is enqueued on torch's current stream
    (the binding reads its raw handle), inside a stream context as well; the
    same call repeated (tensor maps then come from the library's memo) and the
    same caches after a second workload's maps were encoded give the oracle's
    results."""
    assert binding._stream_handle(None) == torch.cuda.current_stream().cuda_stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert binding._stream_handle(None) == s.cuda_stream
    w = wl.make_workload(wl.CONFIGS["tiny"], device="cuda")
    w2 = wl.make_workload(wl.CONFIGS["tiny"], device="cuda", seed=wl.CONFIGS["tiny"].seed + 5)
    ref = oracle.run_workload(w)
    check(w, ref=ref)
    with torch.cuda.stream(s):
        out, lse = binding.decode_workload(w)
    s.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    o1, l1 = binding.decode_workload(w)
    torch.cuda.synchronize()
    assert torch.equal(out, o1) and torch.equal(lse, l1)
    check(w2)
    check(w, ref=ref)


def test_prepared_call_follows_buffers_refreshed_in_place():
    """A prepared call (arguments marshalled once) over static buffers gives
    the oracle's results for each batch copied into those buffers."""
    spec = wl.CONFIGS["tiny"]
    w1 = wl.make_workload(spec, device="cuda")
    w2 = wl.make_workload(spec, device="cuda", seed=spec.seed + 11, content_seed=spec.seed + 12)
    q = w1.q.clone()
    bt = torch.from_numpy(w1.block_tables).cuda()
    sl = torch.from_numpy(w1.seq_lens).cuda()
    call = binding.prepare_decode(q, w1.k_cache, w1.v_cache, bt, sl, None, 1, spec.scale, spec.k_scale,
                                  spec.v_scale)
    for w in (w1, w2, w1):
        q.copy_(w.q)
        bt.copy_(torch.from_numpy(w.block_tables))
        sl.copy_(torch.from_numpy(w.seq_lens))
        # the second batch's pages live in its own caches: same shapes, other tensors
        if w is w2:
            call2 = binding.prepare_decode(q, w2.k_cache, w2.v_cache, bt, sl, None, 1, spec.scale, spec.k_scale,
                                           spec.v_scale)
            out, lse = call2()
        else:
            out, lse = call()
        torch.cuda.synchronize()
        assert binding.paged_attn_device_status(clear=True) == 0
        ref_out, ref_lse = oracle.run_workload(w)
        assert np.abs(out.float().cpu().numpy() - ref_out).max() <= TOL_OUT["bf16"]
        assert np.abs(lse.cpu().numpy() - ref_lse).max() <= TOL_LSE
