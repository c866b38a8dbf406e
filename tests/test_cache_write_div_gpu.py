"""The fp8 cache write's quotient x / scale (pa_cache_write.cu, div_by2: the
correctly rounded reciprocal and Markstein's correction step, two values at a
time) against CUDA's
IEEE division __fdiv_rn, over every fp32 x, on the GPU: the quotients on
[2^-20, 1000] bit for bit and the e4m3 codes everywhere.  Scales: the usual
per-tensor ones, reciprocal edge cases (significands of all ones, the limits
2^-64 and 2^64 of the fast path and beyond), both signs, and the per-token
scales amax / 448 of 64 bf16 amax values spread over the range.  A small CUDA
program that includes the write's source is built with nvcc and run."""
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r'''
#include "pa_cache_write.cu"
#include <cstdio>

namespace {
__device__ __forceinline__ unsigned short code2(float a) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(a));
  return r;
}

__global__ void check(float s, unsigned long long* bad) {
  const pa::ScaleDiv d = pa::scale_div(s);
  const unsigned long long total = 1ull << 32;
  const unsigned long long stride = static_cast<unsigned long long>(gridDim.x) * blockDim.x;
  unsigned long long nb = 0;
  for (unsigned long long i = static_cast<unsigned long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const float x = __uint_as_float(static_cast<unsigned int>(i));
    float q, q2;
    if (d.fast) {
      pa::div_by2(d, x, -x, q, q2);
    } else {
      q = __fdiv_rn(x, s);
      q2 = -q;
    }
    const float qd = __fdiv_rn(x, s), qd2 = __fdiv_rn(-x, s);
    if (!(__float_as_uint(q2) == __float_as_uint(qd2) || (isnan(q2) && isnan(qd2))) &&
        (isnan(qd2) || (fabsf(qd2) >= 9.5367431640625e-07f && fabsf(qd2) <= 1000.f)))
      ++nb;
    if (code2(q2) != code2(qd2)) ++nb;
    const bool bits = __float_as_uint(q) == __float_as_uint(qd) || (isnan(q) && isnan(qd));
    const bool ranged = isnan(qd) || (fabsf(qd) >= 9.5367431640625e-07f && fabsf(qd) <= 1000.f);
    if ((!bits && ranged) || code2(q) != code2(qd)) ++nb;
  }
  if (nb) atomicAdd(bad, nb);
}
}  // namespace

int main(int argc, char** argv) {
  unsigned long long* bad;
  if (cudaMalloc(&bad, sizeof(unsigned long long)) != cudaSuccess) return 3;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  unsigned long long all = 0;
  for (int a = 1; a < argc; ++a) {
    unsigned int b = static_cast<unsigned int>(strtoul(argv[a], nullptr, 16));
    float s;
    memcpy(&s, &b, 4);
    cudaMemset(bad, 0, sizeof(unsigned long long));
    check<<<sms * 8, 256>>>(s, bad);
    if (cudaDeviceSynchronize() != cudaSuccess) return 4;
    unsigned long long n = 0;
    cudaMemcpy(&n, bad, sizeof(n), cudaMemcpyDeviceToHost);
    if (n) printf("scale 0x%08x: %llu mismatches\n", b, n);
    all += n;
  }
  printf("mismatches %llu\n", all);
  return all == 0 ? 0 : 2;
}
'''


def _scales():
    f = lambda v: int(np.float32(v).view(np.uint32))
    s = [f(0.05), f(1 / 448), f(1.0), f(3.0), f(0.1), f(448.0), f(-0.05), f(-1 / 3),
         0x3FFFFFFF, 0x3F7FFFFF, 0x3F800001, 0x00800001, 0x1F800000, 0x5F800000,   # all-ones significands, 2^-64, 2^64
         0x1F7FFFFF, 0x5F800001]                                                   # just outside the fast path
    rng = np.random.default_rng(2024)
    amax = rng.integers(1, 0x7F80, size=64).astype(np.uint32) << 16               # positive finite bf16 values
    s += [f(np.float32(a.view(np.float32)) / np.float32(448)) for a in amax]
    return [format(x, "08x") for x in s]


def test_scale_division_matches_ieee_division_on_every_fp32_value(tmp_path, cuda_lib):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    src = tmp_path / "div_check.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "div_check"
    csrc = os.path.join(ROOT, "paged_kv_decode_06_gb300", "csrc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "--expt-relaxed-constexpr",
                    "-I", csrc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True,
                   capture_output=True)
    r = subprocess.run([str(exe)] + _scales(), capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0" in r.stdout
