"""paged_attn_cache_write vs the cache-write oracle: the whole caches must come
out bit-identical (bf16 rows copied, fp8 codes from the same fp32 division and
round-to-nearest-even with saturation); then decode over the written cache
matches the oracle within the decode tolerances."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_06_gb300 import binding
from paged_kv_decode_06_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _host_cache(c):
    c = c.detach().cpu().contiguous()
    return c.numpy() if c.dtype == torch.uint8 else c.view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    binding.paged_attn_device_status(clear=True)
    yield


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("T,Hkv,D,NB", [(1, 1, 64, 2), (37, 2, 128, 9), (1000, 8, 128, 80), (513, 8, 64, 40),
                                        (77, 3, 16, 6), (150, 3, 96, 12), (45, 3, 512, 4),
                                        (16384, 8, 128, 1088)])   # the benchmarked chunk: several trips
def test_cache_write_bit_exact(kv, T, Hkv, D, NB):
    g = torch.Generator(device="cuda").manual_seed(T + Hkv + D)
    scale = 4.0 if kv == "fp8" else 1.0
    key = (torch.randn(T, Hkv, D, device="cuda", generator=g) * scale).to(torch.bfloat16)
    val = (torch.randn(T, Hkv, D, device="cuda", generator=g) * scale).to(torch.bfloat16)
    rng = np.random.default_rng(T)
    slots = rng.permutation(NB * 16)[:T].astype(np.int32)
    slots[rng.random(T) < 0.1] = -1
    if kv == "fp8":
        kc = torch.randint(0, 256, (NB, 16, Hkv, D), dtype=torch.uint8, device="cuda", generator=g)
        vc = torch.randint(0, 256, (NB, 16, Hkv, D), dtype=torch.uint8, device="cuda", generator=g)
    else:
        kc = torch.randn(NB, 16, Hkv, D, device="cuda", generator=g).to(torch.bfloat16)
        vc = torch.randn(NB, 16, Hkv, D, device="cuda", generator=g).to(torch.bfloat16)
    k0, v0 = _host_cache(kc), _host_cache(vc)
    binding.paged_attn_cache_write(key, val, torch.from_numpy(slots).cuda(), kc, vc, 0.05, 0.07)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    ek, ev = oracle.cache_write(_bits(key), _bits(val), slots, k0, v0, 0.05, 0.07, kv)
    assert np.array_equal(_host_cache(kc), ek)
    assert np.array_equal(_host_cache(vc), ev)


def test_saturation_and_signed_zero_in_fp8():
    x = torch.tensor([[[1000.0, -1000.0, 22.4, -0.0, 0.0, 3e-5, 448 * 0.05, -0.01] * 2]], device="cuda").to(torch.bfloat16)
    kc = torch.zeros(1, 16, 1, 16, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    binding.paged_attn_cache_write(x, x, torch.tensor([3], dtype=torch.int32, device="cuda"), kc, vc, 0.05, 0.05)
    torch.cuda.synchronize()
    expect = oracle.quantize_rows(_bits(x)[0], 0.05)
    assert np.array_equal(kc[0, 3].cpu().numpy(), expect)
    assert kc[0, 3, 0, 0].item() == 0x7E and kc[0, 3, 0, 1].item() == 0xFE and kc[0, 3, 0, 3].item() == 0x80


def test_out_of_range_slot_is_reported_and_skipped():
    key = torch.ones(2, 1, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(2, 16, 1, 64, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    binding.paged_attn_cache_write(key, key, torch.tensor([32, 5], dtype=torch.int32, device="cuda"), kc, vc)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) & binding.STATUS_PAGE_RANGE
    assert kc.float().sum().item() == 64 and kc[0, 5].float().sum().item() == 64


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_write_then_decode_matches_oracle(kv):
    """A decode step as the engine runs it: the new token's K/V is written into
    its slot, then attention reads the cache (seq_lens include the new token)."""
    fp8 = kv == "fp8"
    spec = wl.custom_spec(num_q_heads=16, num_kv_heads=4, head_dim=128, kv_dtype=kv,
                          seq_lens=(1, 40, 129, 700), k_scale=0.05 if fp8 else 1.0, v_scale=0.05 if fp8 else 1.0,
                          fp8_source_scale=0.05 if fp8 else 1.0, seed=12)
    w = wl.make_workload(spec, device="cuda")
    s = w.spec
    B = s.num_seqs
    g = torch.Generator(device="cuda").manual_seed(5)
    new_k = torch.randn(B, s.num_kv_heads, s.head_dim, device="cuda", generator=g).to(torch.bfloat16)
    new_v = torch.randn(B, s.num_kv_heads, s.head_dim, device="cuda", generator=g).to(torch.bfloat16)
    pos = w.seq_lens.astype(np.int64) - 1                           # the new token's position
    slots = np.array([w.block_tables[i, pos[i] // 16] * 16 + pos[i] % 16 for i in range(B)], dtype=np.int32)
    k_before, v_before = _host_cache(w.k_cache), _host_cache(w.v_cache)
    binding.paged_attn_cache_write(new_k, new_v, torch.from_numpy(slots).cuda(), w.k_cache, w.v_cache,
                                   s.k_scale, s.v_scale)
    out, lse = binding.decode_workload(w)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    ek, ev = oracle.cache_write(_bits(new_k), _bits(new_v), slots, k_before, v_before, s.k_scale, s.v_scale, kv)
    assert np.array_equal(_host_cache(w.k_cache), ek) and np.array_equal(_host_cache(w.v_cache), ev)
    ref_out, ref_lse = oracle.paged_decode_attention(_bits(w.q), ek, ev, w.block_tables, w.seq_lens, None,
                                                     s.scale, s.k_scale, s.v_scale, kv)
    tol = 2e-2 if fp8 else 1e-2
    assert np.abs(out.float().cpu().numpy() - ref_out).max() <= tol
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= 1e-3


def _padded_rows(T, Hkv, D, g, scale):
    """bf16 [T, Hkv, D] as a view of wider rows: padded head and token strides,
    a 16-byte offset."""
    big = (torch.randn(T, Hkv + 1, D + 24, device="cuda", generator=g) * scale).to(torch.bfloat16)
    return big[:, 1:, 8:8 + D]


def _padded_cache(NB, Hkv, D, kv, g):
    """A cache [NB, 16, Hkv, D] as a view of rows 32 elements wider (16 before,
    16 after), filled with random bytes that must survive the write."""
    if kv == "fp8":
        big = torch.randint(0, 256, (NB, 16, Hkv, D + 32), dtype=torch.uint8, device="cuda", generator=g)
    else:
        big = torch.randn(NB, 16, Hkv, D + 32, device="cuda", generator=g).to(torch.bfloat16)
    return big, big[..., 16:16 + D]


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("D", [64, 96])
def test_padded_strides_then_all_padding_slots(kv, D):
    T, Hkv, NB = 300, 3, 24
    g = torch.Generator(device="cuda").manual_seed(D + (kv == "fp8"))
    key = _padded_rows(T, Hkv, D, g, 4.0)
    val = _padded_rows(T, Hkv, D, g, 4.0)
    kbig, kc = _padded_cache(NB, Hkv, D, kv, g)
    vbig, vc = _padded_cache(NB, Hkv, D, kv, g)
    rng = np.random.default_rng(D)
    slots = rng.permutation(NB * 16)[:T].astype(np.int32)
    slots[rng.random(T) < 0.2] = -1
    kb0, vb0 = _host_cache(kbig), _host_cache(vbig)
    binding.paged_attn_cache_write(key, val, torch.from_numpy(slots).cuda(), kc, vc, 0.05, 0.07)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    ek, ev = oracle.cache_write(_bits(key), _bits(val), slots, kb0[..., 16:16 + D], vb0[..., 16:16 + D], 0.05, 0.07,
                                kv)
    for got, before, e in ((kbig, kb0, ek), (vbig, vb0, ev)):
        expect = before.copy()
        expect[..., 16:16 + D] = e
        assert np.array_equal(_host_cache(got), expect)          # the padding columns are untouched
    # every slot padding: nothing is written
    kb1, vb1 = _host_cache(kbig), _host_cache(vbig)
    binding.paged_attn_cache_write(key, val, torch.full((T,), -1, dtype=torch.int32, device="cuda"), kc, vc,
                                   0.05, 0.07)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    assert np.array_equal(_host_cache(kbig), kb1) and np.array_equal(_host_cache(vbig), vb1)


def test_fp8_writes_divide_by_the_scale():
    """Inputs whose quotient by the scale sits exactly on a midpoint of the
    e4m3fn grid, where an fp32 division and a product with the fp32 reciprocal
    round to different codes; tiny rows whose scale is an fp32 subnormal; rows
    of +0 and -0."""
    D = 16
    # per-tensor, scale 0.03: x = 0.000732421875 * 2^k lands on midpoints
    row = [0.000732421875 * 2.0 ** k for k in range(4)] + [-0.00146484375, 1.0, -3.0, 0.25]
    x = torch.tensor([[row * 2]], device="cuda").to(torch.bfloat16)
    kc = torch.zeros(1, 16, 1, D, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    binding.paged_attn_cache_write(x, x, torch.tensor([7], dtype=torch.int32, device="cuda"), kc, vc, 0.03, 0.03)
    torch.cuda.synchronize()
    assert np.array_equal(kc[0, 7].cpu().numpy(), oracle.quantize_rows(_bits(x)[0], 0.03))
    # per-token: max |x| = 0.78515625 puts 1.1980533599853516e-05 / scale on a midpoint;
    # a row of max 1e-39 (subnormal in bf16 and fp32); a row of +0 / -0
    rows = torch.tensor([[0.78515625, 1.1980533599853516e-05, -1.1980533599853516e-05, 0.5] * 4,
                         [1e-39, -3e-40, 5e-41, 0.0] * 4,
                         [0.0, -0.0, 0.0, -0.0] * 4], device="cuda").to(torch.bfloat16)[:, None, :]
    kc = torch.full((1, 16, 1, D), 0x55, dtype=torch.uint8, device="cuda")
    vc = torch.full_like(kc, 0x55)
    ks = torch.full((1, 1, 16), 7.0, device="cuda")
    vs = torch.full_like(ks, 7.0)
    host = [_host_cache(kc), _host_cache(vc), ks.cpu().numpy(), vs.cpu().numpy()]
    slots = np.array([2, 9, 12], dtype=np.int32)
    binding.paged_attn_cache_write_per_token(rows, rows, torch.from_numpy(slots).cuda(), kc, vc, ks, vs)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    ek, ev, eks, evs = oracle.cache_write_per_token(_bits(rows), _bits(rows), slots, *host)
    assert np.array_equal(_host_cache(kc), ek) and np.array_equal(_host_cache(vc), ev)
    assert np.array_equal(ks.cpu().numpy(), eks) and np.array_equal(vs.cpu().numpy(), evs)
    assert eks[0, 0, 9] > 0 and not ek[0, 12].any()
