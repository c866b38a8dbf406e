"""The bounded pipeline waits give up: with a short wait limit and one split
CTA whose producer issues no copies, that CTA's consumer warps wait out the
limit, set the timeout status bit and return; the call ends, and the next
ordinary call on the same stream matches the oracle with a clean status word.
Nothing is left in flight: the starved producer never issues a copy."""
import time

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_06_gb300 import binding
from paged_kv_decode_06_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    binding.paged_attn_device_status(clear=True)
    yield
    binding.paged_attn_device_status(clear=True)


def _workload(kv):
    fp8 = kv == "fp8"
    spec = wl.custom_spec(num_q_heads=32, num_kv_heads=8, head_dim=128, kv_dtype=kv,
                          seq_lens=(700, 1000, 333, 901, 640, 1023, 480, 777), seed=31,
                          k_scale=0.05 if fp8 else 1.0, v_scale=0.05 if fp8 else 1.0,
                          fp8_source_scale=0.05 if fp8 else 1.0)
    return wl.make_workload(spec, device="cuda")


def _parity(w, out, lse, ref):
    tol = 2e-2 if w.spec.kv_dtype == "fp8" else 1e-2
    assert np.abs(out.float().cpu().numpy() - ref[0]).max() <= tol
    assert np.abs(lse.cpu().numpy() - ref[1]).max() <= 1e-3


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("starve", [1, 6])
def test_starved_cta_times_out_and_the_next_call_is_clean(kv, starve):
    w = _workload(kv)
    ref = oracle.run_workload(w)
    plan = binding.paged_attn_plan(w.spec.num_seqs, 32, 8, 128, binding.PA_FP8_E4M3 if kv == "fp8" else binding.PA_BF16)
    assert starve - 1 < plan["num_ctas"]
    # an ordinary call first: the workspace then holds this shape's unit
    # descriptors, which the starved call's merge reads for the starved CTA's units
    out, lse = binding.decode_workload(w)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    _parity(w, out, lse, ref)

    opts = binding.make_options(wait_limit_us=1000, test_starve_cta=starve)
    t0 = time.perf_counter()
    binding.decode_workload(w, options=opts)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    status = binding.paged_attn_device_status(clear=True)
    assert status & binding.STATUS_TIMEOUT, f"status {status:#x}"
    assert elapsed < 1.0, f"the starved call took {elapsed:.3f} s with a 1 ms wait limit"

    out, lse = binding.decode_workload(w)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    _parity(w, out, lse, ref)


def test_a_wait_limit_alone_changes_nothing():
    w = _workload("bf16")
    ref = oracle.run_workload(w)
    out, lse = binding.decode_workload(w, options=binding.make_options(wait_limit_us=50000))
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    _parity(w, out, lse, ref)


def test_starving_is_refused_for_the_tensor_memory_kernel():
    w = _workload("bf16")
    with pytest.raises(binding.PagedAttnError) as e:
        binding.decode_workload(w, options=binding.make_options(use_tcgen05=2, test_starve_cta=1))
    assert e.value.status == binding.PA_ERR_UNSUPPORTED
