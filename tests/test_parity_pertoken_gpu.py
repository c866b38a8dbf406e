"""Per-token fp8 scales on the GPU, through the C ABI, against the oracle.

Decode with k/v_token_scales: element by element (out max abs error <= 2e-2,
lse <= 1e-3, the fp8 tolerances) over ragged lengths, group sizes, MTP runs,
forced split counts, heads-per-CTA variants, windows and sinks, non-finite
scales in slots nobody may read, and the full-size per-token workload on
sampled sequences.  The per-token cache write: codes and scales bit-exact
against the oracle's quantiser, then decode over the written cache."""
import numpy as np
import pytest
import torch

import oracle
from oracle import c_oracle
from paged_kv_decode_06_gb300 import binding
from paged_kv_decode_06_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_OUT = 2e-2
TOL_LSE = 1e-3


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    binding.paged_attn_device_status(clear=True)
    yield


def _spec(D=128, G=4, Hkv=2, seq_lens=(1, 15, 16, 17, 31, 32, 33, 100), qlens=(1,), seed=3, k_scale=1.0,
          v_scale=1.0, pool=None):
    return wl.custom_spec(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, kv_dtype="fp8", seq_lens=seq_lens,
                          query_len_choices=qlens, pool_pages=pool, seed=seed, k_scale=k_scale, v_scale=v_scale,
                          fp8_source_scale=1.0 / 128, token_scale_range=(0.25 / 128, 1.0 / 128))


def _rows(w, seqs):
    qsl = w.query_start_loc if w.query_start_loc is not None else np.arange(w.spec.num_seqs + 1)
    return np.concatenate([np.arange(qsl[i], qsl[i + 1]) for i in seqs])


def check(w, seqs=None, ref=None, window=0, sinks=None, **opt_kw):
    sk = torch.from_numpy(np.asarray(sinks, dtype=np.float32)).cuda() if sinks is not None else None
    opts = binding.make_options(sliding_window=window, sinks=sk, k_token_scales=w.k_token_scales,
                                v_token_scales=w.v_token_scales, **opt_kw)
    out, lse = binding.decode_workload(w, options=opts)
    torch.cuda.synchronize()
    st = binding.paged_attn_device_status(clear=True)
    assert st == 0, f"device status {st:#x}"
    if ref is None:
        ref = oracle.run_workload(w, seqs=seqs, sliding_window=window, sinks=sinks)
    rows = _rows(w, range(w.spec.num_seqs) if seqs is None else seqs)
    o = out.float().cpu().numpy()[rows]
    l = lse.cpu().numpy()[rows]
    assert np.isfinite(o).all() and np.isfinite(l).all()
    eo = np.abs(o - ref[0][rows]).max()
    el = np.abs(l - ref[1][rows]).max()
    assert eo <= TOL_OUT, f"max|out - oracle| = {eo:.3e} (max|oracle out| {np.abs(ref[0][rows]).max():.3f})"
    assert el <= TOL_LSE, f"max|lse - oracle| = {el:.3e}"
    return out, lse, eo, el


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("tensor_scales", [(1.0, 1.0), (2.0, 0.75)])
def test_page_boundaries_and_ragged_tails(D, tensor_scales):
    check(wl.make_workload(_spec(D=D, k_scale=tensor_scales[0], v_scale=tensor_scales[1]), device="cuda"))


@pytest.mark.parametrize("G,Hkv,qlens", [(8, 2, (2, 3, 4)), (4, 4, (1, 2)), (16, 1, (4,)), (1, 8, (1, 3)),
                                         (8, 1, (1,)), (2, 8, (3,))])
def test_group_sizes_and_mtp_runs(G, Hkv, qlens):
    check(wl.make_workload(_spec(G=G, Hkv=Hkv, qlens=qlens, seq_lens=(4, 5, 16, 17, 40, 64, 130), seed=G + Hkv),
                           device="cuda"))


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 64, 152, 300])
def test_forced_split_counts(num_ctas):
    w = wl.make_workload(_spec(G=8, Hkv=2, qlens=(1, 2, 4), seq_lens=(3, 50, 300, 17, 1000), seed=num_ctas),
                         device="cuda")
    check(w, num_ctas=num_ctas, min_pages_per_cta=1)


@pytest.mark.parametrize("hc", [1, 2, 4])
def test_heads_per_cta_variants(hc):
    w = wl.make_workload(_spec(G=4, Hkv=4, seq_lens=(7, 70, 700), seed=hc), device="cuda")
    ref = oracle.run_workload(w)
    check(w, ref=ref, heads_per_cta=hc)
    check(w, ref=ref, heads_per_cta=hc, num_ctas=5, min_pages_per_cta=1, page_pairing=2)


def test_non_finite_scales_in_unread_slots_do_not_leak():
    w = wl.make_workload(_spec(seq_lens=(3, 17, 40, 1)), device="cuda")
    ref = oracle.run_workload(w)
    used = set()
    for i, L in enumerate(w.seq_lens):
        n = (int(L) + 15) // 16
        used.update(int(x) for x in w.block_tables[i, :n])
        last = int(w.block_tables[i, n - 1])
        tail = int(L) - 16 * (n - 1)
        w.k_token_scales[last, :, tail:] = float("nan")
        w.v_token_scales[last, :, tail:] = float("inf")
        w.k_cache[last, tail:] = 0x7F
        w.v_cache[last, tail:] = 0x7F
    for p in range(w.num_pages):
        if p not in used:
            w.k_token_scales[p] = float("nan")
            w.v_token_scales[p] = float("nan")
    check(w, ref=ref)


@pytest.mark.parametrize("window", [5, 17, 100])
def test_with_sliding_window_and_sinks(window):
    w = wl.make_workload(_spec(G=8, Hkv=2, qlens=(1, 3), seq_lens=(1, 20, 200, 900), seed=window), device="cuda")
    sinks = np.random.default_rng(window).normal(0, 2, size=16).astype(np.float32)
    check(w, window=window)
    check(w, window=window, sinks=sinks, num_ctas=7, min_pages_per_cta=1)


def test_equal_token_scales_match_the_per_tensor_path():
    w = wl.make_workload(_spec(seq_lens=(33, 400, 90), G=4, Hkv=2, seed=17), device="cuda")
    c_k, c_v = 0.0123, 0.0061          # dequantised values about N(0, 1.6^2) and N(0, 0.8^2)
    w.k_token_scales.fill_(c_k)
    w.v_token_scales.fill_(c_v)
    out_t, lse_t, _, _ = check(w)
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    out_p, lse_p = binding.paged_attn_decode(w.q, w.k_cache, w.v_cache, bt, sl, None, 1, w.spec.scale, c_k, c_v)
    torch.cuda.synchronize()
    assert (out_t.float() - out_p.float()).abs().max().item() <= 2 ** -7
    assert (lse_t - lse_p).abs().max().item() <= 1e-5


def test_full_size_per_token_workload_every_row():
    """Every query row against the C oracle; sampled sequences against the
    NumPy oracle too."""
    w = wl.make_workload(wl.CONFIGS["fp8_pertoken"], device="cuda")
    _, _, eo, el = check(w, ref=c_oracle.run_workload(w))
    rng = np.random.default_rng(6)
    seqs = sorted(set(rng.choice(w.spec.num_seqs, size=3, replace=False).tolist()) |
                  {int(np.argmax(w.seq_lens)), int(np.argmin(w.seq_lens))})
    check(w, seqs=seqs)
    print(f"fp8_pertoken: all {w.q.shape[0]} query tokens: max|out err| {eo:.3e}, max|lse err| {el:.3e}")


# ------------------------------------------------ per-token cache write

def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# head dims whose rows fill a power-of-two lane group (64, 128, 256), leave lanes
# of the group idle (16 -> two lanes, 96 -> 12 of 16) or give a lane two chunks (512)
@pytest.mark.parametrize("T,Hkv,D,NB", [(1, 1, 64, 2), (37, 2, 128, 9), (1000, 8, 128, 80), (513, 8, 64, 40),
                                        (77, 3, 16, 6), (150, 3, 96, 12), (61, 2, 256, 5), (45, 3, 512, 4),
                                        (16384, 8, 128, 1088)])   # the benchmarked chunk: several trips
def test_per_token_cache_write_bit_exact(T, Hkv, D, NB):
    g = torch.Generator(device="cuda").manual_seed(T * 7 + D)
    mag = torch.exp(torch.randn(T, Hkv, 1, device="cuda", generator=g) * 3)
    key = (torch.randn(T, Hkv, D, device="cuda", generator=g) * mag).to(torch.bfloat16)
    val = (torch.randn(T, Hkv, D, device="cuda", generator=g) * mag).to(torch.bfloat16)
    if T > 2:
        key[1, 0] = 0.0                                   # an all-zero row: scale 0, codes 0
        val[2, -1, 3] = -val[2, -1].abs().max() * 2       # a row whose max is negative
    rng = np.random.default_rng(T)
    slots = rng.permutation(NB * 16)[:T].astype(np.int32)
    slots[rng.random(T) < 0.1] = -1
    kc = torch.randint(0, 256, (NB, 16, Hkv, D), dtype=torch.uint8, device="cuda", generator=g)
    vc = torch.randint(0, 256, (NB, 16, Hkv, D), dtype=torch.uint8, device="cuda", generator=g)
    ks = torch.rand(NB, Hkv, 16, device="cuda", generator=g)
    vs = torch.rand(NB, Hkv, 16, device="cuda", generator=g)
    host = [t.cpu().numpy() for t in (kc, vc, ks, vs)]
    binding.paged_attn_cache_write_per_token(key, val, torch.from_numpy(slots).cuda(), kc, vc, ks, vs)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    exp = oracle.cache_write_per_token(_bits(key), _bits(val), slots, *host)
    for got, e in zip((kc, vc, ks, vs), exp):
        assert np.array_equal(got.cpu().numpy(), e)


def test_per_token_cache_write_strided_scales_and_bad_slot():
    T, Hkv, D, NB = 20, 2, 64, 4
    key = torch.randn(T, Hkv, D, device="cuda").to(torch.bfloat16)
    val = torch.randn(T, Hkv, D, device="cuda").to(torch.bfloat16)
    slots = np.arange(T, dtype=np.int32) * 3 % (NB * 16)
    slots[4] = NB * 16 + 1                                       # past the pool: skipped, reported
    kc = torch.zeros(NB, 16, Hkv, D, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    big = torch.zeros(NB, 16, 2 * Hkv, device="cuda")            # scales as a strided view [NB, Hkv, 16]
    ks = big[:, :, :Hkv].permute(0, 2, 1)
    vs = big[:, :, Hkv:].permute(0, 2, 1)
    host = [t.cpu().numpy() for t in (kc, vc, ks, vs)]
    binding.paged_attn_cache_write_per_token(key, val, torch.from_numpy(slots).cuda(), kc, vc, ks, vs)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) & binding.STATUS_PAGE_RANGE
    exp = oracle.cache_write_per_token(_bits(key), _bits(val), slots, *host)
    for got, e in zip((kc, vc, ks, vs), exp):
        assert np.array_equal(got.cpu().numpy(), e)


def test_write_then_decode_per_token():
    spec = _spec(seq_lens=(40, 129, 7), G=4, Hkv=2, seed=31)
    w = wl.make_workload(spec, device="cuda")
    # overwrite every cached row through the per-token write from fresh bf16 rows
    T = int(sum(w.seq_lens))
    slots = np.concatenate([w.block_tables[i, np.arange(L) // 16] * 16 + np.arange(L) % 16
                            for i, L in enumerate(w.seq_lens)]).astype(np.int32)
    g = torch.Generator(device="cuda").manual_seed(5)
    key = torch.randn(T, 2, 128, device="cuda", generator=g).to(torch.bfloat16)
    val = (torch.randn(T, 2, 128, device="cuda", generator=g) * 3).to(torch.bfloat16)
    binding.paged_attn_cache_write_per_token(key, val, torch.from_numpy(slots).cuda(), w.k_cache, w.v_cache,
                                             w.k_token_scales, w.v_token_scales)
    torch.cuda.synchronize()
    check(w)
    # the result is also close to attention over the unquantised bf16 rows
    kh, vh = _bits(key).reshape(T, 2, 128), _bits(val).reshape(T, 2, 128)
    kb = torch.zeros(w.num_pages, 16, 2, 128, dtype=torch.bfloat16)
    vb = torch.zeros_like(kb)
    kb.view(-1, 2, 128)[torch.from_numpy(slots.astype(np.int64))] = torch.from_numpy(kh.view(np.int16)).view(torch.bfloat16)
    vb.view(-1, 2, 128)[torch.from_numpy(slots.astype(np.int64))] = torch.from_numpy(vh.view(np.int16)).view(torch.bfloat16)
    q_bits = _bits(w.q)
    ref_bf16 = oracle.paged_decode_attention(q_bits, kb.view(torch.int16).numpy().view(np.uint16),
                                             vb.view(torch.int16).numpy().view(np.uint16), w.block_tables,
                                             w.seq_lens, None, spec.scale)
    out, _ = binding.decode_workload(w, options=binding.make_options(k_token_scales=w.k_token_scales,
                                                                     v_token_scales=w.v_token_scales))
    torch.cuda.synchronize()
    assert np.abs(out.float().cpu().numpy() - ref_bf16[0]).max() < 0.25   # e4m3 keeps ~2 significant digits


@pytest.mark.parametrize("D", [96, 128])
def test_per_token_cache_write_padded_strides_and_second_chunk_maxima(D):
    """Key/value rows and caches as views with padded strides; the row maxima
    sit in a lane's later chunks (the reduction must cover every chunk a lane
    holds, not only its first)."""
    T, Hkv, NB = 200, 3, 16
    g = torch.Generator(device="cuda").manual_seed(D)
    bigk = torch.randn(T, Hkv + 1, D + 24, device="cuda", generator=g).to(torch.bfloat16)
    bigv = torch.randn(T, Hkv + 1, D + 24, device="cuda", generator=g).to(torch.bfloat16)
    key, val = bigk[:, 1:, 8:8 + D], bigv[:, 1:, 8:8 + D]
    key[:, :, D - 3] = 50.0                  # the last chunk holds each key row's max
    val[:, :, D // 2 + 1] = -70.0            # a middle chunk holds each value row's max (negative)
    kbig = torch.randint(0, 256, (NB, 16, Hkv, D + 32), dtype=torch.uint8, device="cuda", generator=g)
    vbig = torch.randint(0, 256, (NB, 16, Hkv, D + 32), dtype=torch.uint8, device="cuda", generator=g)
    kc, vc = kbig[..., 16:16 + D], vbig[..., 16:16 + D]
    ks = torch.rand(NB, Hkv, 16, device="cuda", generator=g)
    vs = torch.rand(NB, Hkv, 16, device="cuda", generator=g)
    slots = np.random.default_rng(D).permutation(NB * 16)[:T].astype(np.int32)
    kb0, vb0 = kbig.cpu().numpy(), vbig.cpu().numpy()
    host = [kb0[..., 16:16 + D], vb0[..., 16:16 + D], ks.cpu().numpy(), vs.cpu().numpy()]
    binding.paged_attn_cache_write_per_token(key, val, torch.from_numpy(slots).cuda(), kc, vc, ks, vs)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    ek, ev, eks, evs = oracle.cache_write_per_token(_bits(key), _bits(val), slots, *host)
    for got, before, e in ((kbig, kb0, ek), (vbig, vb0, ev)):
        expect = before.copy()
        expect[..., 16:16 + D] = e
        assert np.array_equal(got.cpu().numpy(), expect)
    assert np.array_equal(ks.cpu().numpy(), eks) and np.array_equal(vs.cpu().numpy(), evs)
    written = eks[slots // 16, :, slots % 16]
    assert np.allclose(written, np.float32(50.0) / np.float32(448.0))   # the planted maxima decided the scales
