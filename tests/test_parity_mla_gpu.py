"""MLA decode on the GPU vs the float64 MLA oracle, element by element, through
the C ABI (paged_attn_mla_decode).

Tolerances (max absolute error): out 1e-2 for bf16 caches, 2e-2 for fp8
caches; lse 1e-3.  Small cases are compared in full; the full-size MLA
workloads on every row against the plain-C oracle and on sampled sequences
against the NumPy oracle, in the launch configuration the benchmark times.
The main cases run on both split kernels: the mma.sync kernel (use_tcgen05 =
1) and the tensor-memory (tcgen05) kernel (use_tcgen05 = 2); the planner's
default picks one of them."""
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


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    binding.paged_attn_device_status(clear=True)
    yield


def _rows_of(w, seqs):
    qsl = w.query_start_loc if w.query_start_loc is not None else np.arange(w.spec.num_seqs + 1)
    return np.concatenate([np.arange(qsl[i], qsl[i + 1]) for i in seqs])


KERNELS = {"tc": 2, "mma": 1}


def _opts(kernel, **kw):
    return binding.make_options(use_tcgen05=KERNELS[kernel], **kw)


def check(w, seqs=None, options=None, ref=None, kernel=None):
    if kernel is not None:
        assert options is None
        options = _opts(kernel)
    out, lse = binding.mla_decode_workload(w, options=options)
    torch.cuda.synchronize()
    status = binding.paged_attn_device_status(clear=True)
    assert status == 0, f"device status {status:#x}"
    if ref is None:
        ref = oracle.run_mla_workload(w, seqs=seqs)
    rows = _rows_of(w, range(w.spec.num_seqs) if seqs is None else seqs)
    o = out.float().cpu().numpy()[rows]
    l = lse.cpu().numpy()[rows]
    assert np.isfinite(o).all() and np.isfinite(l).all()
    err_o = np.abs(o - ref[0][rows]).max()
    err_l = np.abs(l - ref[1][rows]).max()
    tol = TOL_OUT[w.spec.kv_dtype]
    assert err_o <= tol, f"max|out - oracle| = {err_o:.3e} > {tol}"
    assert err_l <= TOL_LSE, f"max|lse - oracle| = {err_l:.3e} > {TOL_LSE}"
    return out, lse, err_o, err_l


def _spec(kv="bf16", Hq=16, seq_lens=(1, 15, 16, 17, 31, 32, 33, 100), qlens=(1,), seed=5, pool=None):
    fp8 = kv == "fp8"
    return wl.custom_mla_spec(num_q_heads=Hq, kv_dtype=kv, seq_lens=seq_lens, query_len_choices=qlens,
                              pool_pages=pool, kv_scale=0.05 if fp8 else 1.0, fp8_source_scale=0.05 if fp8 else 1.0,
                              seed=seed)


@pytest.mark.parametrize("kernel", ["tc", "mma"])
def test_mla_tiny_config_full(kernel):
    check(wl.make_mla_workload(wl.MLA_CONFIGS["mla_tiny"], device="cuda"), kernel=kernel)


@pytest.mark.parametrize("kernel", ["tc", "mma"])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_mla_page_boundaries_and_ragged_tails(kv, kernel):
    check(wl.make_mla_workload(_spec(kv=kv), device="cuda"), kernel=kernel)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_mla_plan_variants(kv):
    code = binding.PA_FP8_E4M3 if kv == "fp8" else binding.PA_BF16
    # default: the tensor-memory kernel for fp8 caches or more than 16 rows a unit
    assert binding.paged_attn_mla_plan(32, 16, code, 1)["variant"] == (3 if kv == "fp8" else 2)
    assert binding.paged_attn_mla_plan(32, 16, code, 4)["variant"] == 3
    assert binding.paged_attn_mla_plan(32, 16, code, 4, options=_opts("mma"))["variant"] == 2
    assert binding.paged_attn_mla_plan(32, 16, code, 4, options=_opts("tc"))["variant"] == 3


# heads x query lengths: 1 row tile (two teams a CTA), 2 row tiles, several head chunks
@pytest.mark.parametrize("kernel", ["tc", "mma"])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("Hq,qlens", [(16, (1,)), (8, (1,)), (1, (1,)), (16, (4,)), (16, (2, 3, 4)), (32, (1,)),
                                      (128, (1,)), (16, (3,)), (4, (1, 5, 8)), (2, (16,))])
def test_mla_heads_and_verification_runs(kv, Hq, qlens, kernel):
    w = wl.make_mla_workload(_spec(kv=kv, Hq=Hq, qlens=qlens, seq_lens=(16, 17, 40, 64, 130), seed=Hq + len(qlens)),
                             device="cuda")
    check(w, kernel=kernel)


@pytest.mark.parametrize("kernel", ["tc", "mma"])
@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 64, 152, 300])
@pytest.mark.parametrize("kv,Hq,qlens", [("bf16", 16, (1,)), ("fp8", 16, (4,))])
def test_mla_forced_split_counts_exercise_the_merge(num_ctas, kv, Hq, qlens, kernel):
    w = wl.make_mla_workload(_spec(kv=kv, Hq=Hq, qlens=qlens, seq_lens=(3, 50, 300, 17, 1000), seed=num_ctas),
                             device="cuda")
    ref = oracle.run_mla_workload(w)
    check(w, ref=ref, options=_opts(kernel, num_ctas=num_ctas, min_pages_per_cta=1))


# The tensor-memory kernel's work split charges every unit a CTA starts
# segment_cost_pages pages: an equal page split (< 0), small and large charges,
# one so large that CTAs between units get no pages at all; with few and many
# CTAs, so that units span several CTAs and CTAs span several units.
@pytest.mark.parametrize("num_ctas", [5, 152])
@pytest.mark.parametrize("seg_cost", [-1, 3, 40, 100000])
@pytest.mark.parametrize("kv,Hq,qlens", [("bf16", 16, (1,)), ("fp8", 16, (4,))])
def test_mla_tc_segment_cost_split(seg_cost, num_ctas, kv, Hq, qlens):
    w = wl.make_mla_workload(_spec(kv=kv, Hq=Hq, qlens=qlens, seq_lens=(3, 50, 300, 17, 1000, 1, 64, 700),
                                   seed=abs(seg_cost) % 97 + num_ctas), device="cuda")
    ref = oracle.run_mla_workload(w)
    check(w, ref=ref, options=_opts("tc", num_ctas=num_ctas, min_pages_per_cta=1, segment_cost_pages=seg_cost))


@pytest.mark.parametrize("kernel", ["tc", "mma"])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_mla_non_finite_tail_slots_and_unused_pages_do_not_leak(kv, kernel):
    w = wl.make_mla_workload(_spec(kv=kv, seq_lens=(3, 17, 40, 1)), device="cuda")
    ref = oracle.run_mla_workload(w)
    nan_code = torch.tensor(float("nan")).to(torch.bfloat16) if kv == "bf16" else torch.tensor(0x7F, dtype=torch.uint8)
    used = set()
    for i, L in enumerate(w.seq_lens):
        n = (int(L) + 15) // 16
        used.update(int(x) for x in w.block_tables[i, :n])
        last = int(w.block_tables[i, n - 1])
        w.kv_cache[last, int(L) - 16 * (n - 1):] = nan_code
    for p in range(w.num_pages):
        if p not in used:
            w.kv_cache[p] = nan_code
    check(w, ref=ref, kernel=kernel)


def test_mla_strided_cache_and_lse_optional():
    w = wl.make_mla_workload(_spec(seq_lens=(20, 90, 33)), device="cuda")
    ref = oracle.run_mla_workload(w)
    # the latent cache as one half of a [NB, 16, 2, 576] allocation (page and slot strides grow)
    big = torch.zeros((w.num_pages, 16, 2, 576), dtype=w.kv_cache.dtype, device="cuda")
    big[:, :, 0] = w.kv_cache
    w.kv_cache = big[:, :, 0]
    assert not w.kv_cache.is_contiguous()
    check(w, ref=ref)
    out, lse = binding.mla_decode_workload(w, want_lse=False)
    torch.cuda.synchronize()
    assert lse is None and np.abs(out.float().cpu().numpy() - ref[0]).max() <= TOL_OUT["bf16"]


def test_mla_caller_workspace_and_deterministic_results():
    w = wl.make_mla_workload(_spec(qlens=(1, 2), seq_lens=(500, 33, 1200)), device="cuda")
    n = binding.paged_attn_mla_workspace_size(w.spec.num_seqs, w.spec.num_q_heads, binding.PA_BF16, 2)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    o1, l1, _, _ = check(w, options=binding.make_options(workspace=ws.data_ptr(), workspace_bytes=n))
    o2, l2 = binding.mla_decode_workload(w)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    with pytest.raises(binding.PagedAttnError) as e:
        binding.mla_decode_workload(w, options=binding.make_options(workspace=ws.data_ptr(), workspace_bytes=64))
    assert e.value.status == binding.PA_ERR_WORKSPACE


def test_mla_out_of_range_page_id_is_reported():
    w = wl.make_mla_workload(_spec(seq_lens=(40, 20)), device="cuda")
    w.block_tables = w.block_tables.copy()
    w.block_tables[0, 1] = w.num_pages + 5
    binding.mla_decode_workload(w)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) & binding.STATUS_PAGE_RANGE


def test_mla_cuda_graph_capture_and_replay_with_new_metadata():
    w = wl.make_mla_workload(_spec(seq_lens=(100, 300, 17, 64), pool=200), device="cuda")
    s = w.spec
    binding.paged_attn_mla_reserve(s.num_seqs, s.num_q_heads, binding.PA_BF16, 1)
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    out = torch.empty((w.q.shape[0], s.num_q_heads, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    binding.paged_attn_mla_decode(w.q, w.kv_cache, bt, sl, None, 1, s.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        binding.paged_attn_mla_decode(w.q, w.kv_cache, bt, sl, None, 1, s.scale, out=out, lse=lse, stream=stream)
    rng = np.random.default_rng(6)
    for _ in range(3):
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
        ref = oracle.run_mla_workload(w)
        assert np.abs(out.float().cpu().numpy() - ref[0]).max() <= TOL_OUT["bf16"]
        assert np.abs(lse.cpu().numpy() - ref[1]).max() <= TOL_LSE
    assert binding.paged_attn_device_status(clear=True) == 0


@pytest.mark.parametrize("kernel", ["tc", "mma"])
@pytest.mark.parametrize("name", ["mla_tp8", "mla_mtp_fp8"])
def test_mla_full_size_configs_every_row(name, kernel):
    """Every query row against the C oracle; sampled sequences against the
    NumPy oracle too."""
    w = wl.make_mla_workload(wl.MLA_CONFIGS[name], device="cuda")
    _, _, eo, el = check(w, ref=c_oracle.run_mla_workload(w), kernel=kernel)
    rng = np.random.default_rng(len(name))
    seqs = set(rng.choice(w.spec.num_seqs, size=3, replace=False).tolist())
    seqs.update({int(np.argmax(w.seq_lens)), int(np.argmin(w.seq_lens))})
    check(w, seqs=sorted(seqs), kernel=kernel)
    print(f"{name}: all {w.q.shape[0]} query tokens: max|out err| {eo:.3e}, max|lse err| {el:.3e}")


def test_mla_padded_query_output_and_lse_strides():
    w = wl.make_mla_workload(_spec(qlens=(1, 3), seq_lens=(40, 7, 130)), device="cuda")
    ref = oracle.run_mla_workload(w)
    T, Hq = w.q.shape[:2]
    qbig = torch.zeros((T, Hq + 2, 576), dtype=torch.bfloat16, device="cuda")   # token stride (Hq + 2) * 576
    qbig[:, :Hq] = w.q
    w.q = qbig[:, :Hq]
    obig = torch.full((T, Hq + 1, 520), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = obig[:, :Hq, :512]
    lbig = torch.full((Hq, T + 3), float("nan"), dtype=torch.float32, device="cuda")
    lse = lbig[:, :T].t()
    binding.mla_decode_workload(w, out=out, lse=lse)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    assert np.abs(out.float().cpu().numpy() - ref[0]).max() <= TOL_OUT["bf16"]
    assert np.abs(lse.cpu().numpy() - ref[1]).max() <= TOL_LSE
    assert torch.isnan(obig[:, Hq:]).all() and torch.isnan(obig[:, :, 512:]).all()   # nothing written outside


def test_mla_context_shorter_than_its_query_run_is_reported():
    w = wl.make_mla_workload(_spec(qlens=(3,), seq_lens=(40, 20)), device="cuda")
    w.seq_lens = w.seq_lens.copy()
    w.seq_lens[1] = 2          # fewer cached tokens than the run's 3 query tokens
    binding.mla_decode_workload(w)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) & binding.STATUS_SEQ_LEN


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_mla_single_token_contexts_and_long_runs(kv):
    # L = q (every row sees a prefix of its own run), and runs of 16 tokens
    w = wl.make_mla_workload(_spec(kv=kv, Hq=2, qlens=(16,), seq_lens=(16, 17, 31, 33)), device="cuda")
    check(w)
    w = wl.make_mla_workload(_spec(kv=kv, Hq=16, seq_lens=(1, 1, 2, 1)), device="cuda")
    check(w)


@pytest.mark.parametrize("kv,qlens", [("bf16", (1,)), ("fp8", (1, 2, 3, 4))])
def test_mla_batch_of_512_sequences(kv, qlens):
    # the engine's max_num_seqs: lengths 1..300, sampled rows checked against the oracle
    rng = np.random.default_rng(512)
    lens = tuple(int(x) for x in rng.integers(4, 301, size=512))
    w = wl.make_mla_workload(_spec(kv=kv, Hq=16, qlens=qlens, seq_lens=lens, seed=512), device="cuda")
    seqs = sorted(set(rng.choice(512, size=12, replace=False).tolist()) | {0, 511})
    check(w, seqs=seqs)


def test_mla_partial_outputs_beyond_f16_range_are_reported():
    # a bf16 latent value of 1e6 in a sequence cut across CTAs: the pieces meet in
    # f16, which cannot hold it, and the status word says so
    w = wl.make_mla_workload(_spec(seq_lens=(300, 40)), device="cuda")
    page = int(w.block_tables[0, 3])
    w.kv_cache[page, :, :512] = 1.0e6
    binding.mla_decode_workload(w, options=binding.make_options(num_ctas=8, min_pages_per_cta=1))
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) & binding.STATUS_F16_RANGE
