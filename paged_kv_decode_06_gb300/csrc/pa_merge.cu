// Log-sum-exp merge of split partials (high-interactivity blog, "Attention
// Decode: Split Memory Work to Fill the Device": per-split log-sum-exp values
// kept in fp32, merged afterwards).
//
// One warp per (unit, query row).  A unit (sequence i, head chunk c) whose page
// range [a, b) lies inside one split CTA was finished by that CTA and is
// skipped.  Otherwise the CTAs g_first..g_last that cut it each left, in slot
// 2g (the CTA's first unit) or 2g+1 (its last unit), the unnormalised output
// O_s, the running max m_s (log2 units) and the sum l_s.  With M = max_s m_s:
//   out = v_scale * sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s
//   lse = ln 2 * (M + log2 sum_s 2^(m_s - M) l_s)
#include "pa_device.cuh"
#include "pa_kernels.h"

namespace pa {

constexpr int kMergeWarps = 8;

template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) pa_merge_kernel(const MergeParams p) {
  grid_dependency_wait();   // results of the split kernel (programmatic dependent launch)
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int u = blockIdx.x;
  const int i = u / p.NC;
  const int c = u - i * p.NC;
  const int row = blockIdx.y * kMergeWarps + warp;
  if (row >= p.HC * p.R_max) return;
  const int hh = row / p.R_max;
  const int rho = row - hh * p.R_max;

  int t0, qn;
  if (p.qsl != nullptr) {
    t0 = p.qsl[i];
    qn = p.qsl[i + 1] - t0;
  } else {
    t0 = i;
    qn = 1;
  }
  if (qn < 1 || qn > p.max_qlen || t0 < 0 || t0 + qn > p.num_tokens) return;   // reported by the split kernel
  if (rho >= p.G * qn) return;
  const int t = t0 + rho / p.G;
  const int hq = (c * p.HC + hh) * p.G + rho % p.G;
  uint16_t* orow = p.out + static_cast<int64_t>(t) * p.out_stride_t + static_cast<int64_t>(hq) * p.out_stride_h;
  float* lse_ptr = p.lse ? p.lse + static_cast<int64_t>(t) * p.lse_stride_t + static_cast<int64_t>(hq) * p.lse_stride_h
                         : nullptr;

  const int pre_i = p.ws_prefix[i];
  const int n = p.ws_prefix[i + 1] - pre_i;
  if (n == 0) {
    // empty context (invalid input): no split CTA touched this unit
    for (int d = 2 * lane; d < D; d += 64) *reinterpret_cast<uint32_t*>(orow + d) = 0u;
    if (lane == 0) {
      if (lse_ptr) *lse_ptr = -INFINITY;
      atomicOr(p.err, kErrSeqLen);
    }
    return;
  }
  const int64_t X = p.ws_meta[0];
  const int64_t NG = p.ws_meta[1];
  const int64_t a = static_cast<int64_t>(p.NC) * pre_i + static_cast<int64_t>(c) * n;
  const int64_t b = a + n;
  // largest g with floor(g*X/NG) <= x
  const int gf = static_cast<int>(((a + 1) * NG - 1) / X);
  const int gl = static_cast<int>((b * NG - 1) / X);
  if (gf == gl) return;
  const bool first_is_tail = (static_cast<int64_t>(gf) * X / NG) < a;   // unit is gf's last unit
  const int nparts = gl - gf + 1;
  auto slot_of = [&](int s) -> int64_t {
    const int gg = gf + s;
    const int which = (s == 0 && first_is_tail) ? 1 : 0;
    return (static_cast<int64_t>(2 * gg + which) * p.HC + hh) * p.R_max + rho;
  };

  float M = -INFINITY;
  for (int s = lane; s < nparts; s += 32) M = fmaxf(M, p.ws_ml[slot_of(s)].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float Mb = (M == -INFINITY) ? 0.f : M;

  constexpr int LPD = D / 4;          // lanes per partial row (float4 each)
  constexpr int PL = 32 / LPD;        // partials processed side by side
  const int dq = lane % LPD;
  const int pl = lane / LPD;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lsum = 0.f;
#pragma unroll 4
  for (int s = pl; s < nparts; s += PL) {
    const int64_t sl = slot_of(s);
    const float2 ml = p.ws_ml[sl];
    const float4 o = *reinterpret_cast<const float4*>(p.ws_o + sl * D + 4 * dq);
    const float wgt = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - Mb);
    acc.x += wgt * o.x;
    acc.y += wgt * o.y;
    acc.z += wgt * o.z;
    acc.w += wgt * o.w;
    lsum += wgt * ml.y;
  }
#pragma unroll
  for (int o = LPD; o < 32; o <<= 1) {
    acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
    acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
    acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
    acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  }
  if (pl == 0) {
    const float inv = lsum > 0.f ? p.v_scale / lsum : 0.f;
    uint2 pk;
    pk.x = pack_bf16(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(orow + 4 * dq) = pk;
  }
  if (lane == 0 && lse_ptr) *lse_ptr = lsum > 0.f ? (M + fast_log2(lsum)) * 0.69314718055994530942f : -INFINITY;
}

cudaError_t launch_merge(int head_dim, const MergeParams& p, int grid_x, int grid_y, bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid_x), static_cast<unsigned>(grid_y), 1);
  cfg.blockDim = dim3(32 * kMergeWarps, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (head_dim == 128) return cudaLaunchKernelEx(&cfg, pa_merge_kernel<128>, p);
  if (head_dim == 64) return cudaLaunchKernelEx(&cfg, pa_merge_kernel<64>, p);
  return cudaErrorInvalidValue;
}

}  // namespace pa
