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
constexpr int kWideThreads = 256;

struct MergeRow {
  bool work;        // row exists and its unit was cut into >= 2 pieces
  uint16_t* orow;
  float* lse_ptr;
  int hh, rho;
  int gf, nparts;
  bool first_is_tail;
};

// Locates (unit u, row) and the CTAs whose ranges cut the unit.  Rows whose unit
// was finished inside one CTA, or that do not exist for this sequence, report
// work = false.  An empty context writes out = 0, lse = -inf here.
template <int D>
__device__ __forceinline__ MergeRow merge_row(const MergeParams& p, int u, int row, int lane) {
  MergeRow m;
  m.work = false;
  const int i = u / p.NC;
  const int c = u - i * p.NC;
  if (row >= p.HC * p.R_max) return m;
  m.hh = row / p.R_max;
  m.rho = row - m.hh * p.R_max;
  int t0, qn;
  if (p.qsl != nullptr) {
    t0 = p.qsl[i];
    qn = p.qsl[i + 1] - t0;
  } else {
    t0 = i;
    qn = 1;
  }
  if (qn < 1 || qn > p.max_qlen || t0 < 0 || t0 + qn > p.num_tokens) return m;   // reported by the split kernel
  if (m.rho >= p.G * qn) return m;
  const int t = t0 + m.rho / p.G;
  const int hq = (c * p.HC + m.hh) * p.G + m.rho % p.G;
  m.orow = p.out + static_cast<int64_t>(t) * p.out_stride_t + static_cast<int64_t>(hq) * p.out_stride_h;
  m.lse_ptr = p.lse ? p.lse + static_cast<int64_t>(t) * p.lse_stride_t + static_cast<int64_t>(hq) * p.lse_stride_h
                    : nullptr;
  const int pre_i = p.ws_prefix[i];
  const int n = p.ws_prefix[i + 1] - pre_i;
  if (n == 0) {
    // empty context (invalid input): no split CTA touched this unit
    if (lane >= 0) {
      for (int d = 2 * lane; d < D; d += 64) *reinterpret_cast<uint32_t*>(m.orow + d) = 0u;
      if (lane == 0) {
        if (m.lse_ptr) *m.lse_ptr = -INFINITY;
        atomicOr(p.err, kErrSeqLen);
      }
    }
    return m;
  }
  const int64_t X = p.ws_meta[0];
  const int64_t NG = p.ws_meta[1];
  const int64_t a = static_cast<int64_t>(p.NC) * pre_i + static_cast<int64_t>(c) * n;
  const int64_t b = a + n;
  // largest g with floor(g*X/NG) <= x
  m.gf = static_cast<int>(((a + 1) * NG - 1) / X);
  const int gl = static_cast<int>((b * NG - 1) / X);
  if (m.gf == gl) return m;
  m.first_is_tail = (static_cast<int64_t>(m.gf) * X / NG) < a;   // the unit is CTA gf's last unit
  m.nparts = gl - m.gf + 1;
  m.work = true;
  return m;
}

__device__ __forceinline__ int64_t slot_row(const MergeParams& p, const MergeRow& m, int s) {
  const int which = (s == 0 && m.first_is_tail) ? 1 : 0;
  return (static_cast<int64_t>(2 * (m.gf + s) + which) * p.HC + m.hh) * p.R_max + m.rho;
}

__device__ __forceinline__ void write_merged(const MergeParams& p, const MergeRow& m, int dq, float4 acc, float lsum,
                                             float M, bool write_lse) {
  const float inv = lsum > 0.f ? p.v_scale / lsum : 0.f;
  uint2 pk;
  pk.x = pack_bf16(acc.x * inv, acc.y * inv);
  pk.y = pack_bf16(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(m.orow + 4 * dq) = pk;
  if (write_lse && m.lse_ptr) *m.lse_ptr = lsum > 0.f ? (M + fast_log2(lsum)) * 0.69314718055994530942f : -INFINITY;
}

// One warp per (unit, row).
template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) pa_merge_kernel(const MergeParams p) {
  grid_dependency_wait();   // results of the split kernel (programmatic dependent launch)
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const MergeRow m = merge_row<D>(p, blockIdx.x, blockIdx.y * kMergeWarps + warp, lane);
  if (!m.work) return;

  float M = -INFINITY;
  for (int s = lane; s < m.nparts; s += 32) M = fmaxf(M, p.ws_ml[slot_row(p, m, s)].x);
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
  for (int s = pl; s < m.nparts; s += PL) {
    const int64_t sl = slot_row(p, m, s);
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
  if (pl == 0) write_merged(p, m, dq, acc, lsum, M, lane == 0);
}

// One 256-thread block per (unit, row): the partials of a unit cut into many
// pieces (a long context spread over every SM) are read by all threads at once.
template <int D>
__global__ void __launch_bounds__(kWideThreads) pa_merge_wide_kernel(const MergeParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  constexpr int LPD = D / 4;
  constexpr int PG = kWideThreads / LPD;
  __shared__ float s_max[kWideThreads / 32];
  __shared__ float4 s_acc[PG][LPD];
  __shared__ float s_l[PG];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const MergeRow m = merge_row<D>(p, blockIdx.x, blockIdx.y, tid < 32 ? lane : -1);
  if (!m.work) return;

  float M = -INFINITY;
  for (int s = tid; s < m.nparts; s += kWideThreads) M = fmaxf(M, p.ws_ml[slot_row(p, m, s)].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) s_max[tid >> 5] = M;
  __syncthreads();
  M = s_max[0];
#pragma unroll
  for (int w = 1; w < kWideThreads / 32; ++w) M = fmaxf(M, s_max[w]);
  const float Mb = (M == -INFINITY) ? 0.f : M;

  const int dq = tid % LPD;
  const int pg = tid / LPD;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lsum = 0.f;
#pragma unroll 4
  for (int s = pg; s < m.nparts; s += PG) {
    const int64_t sl = slot_row(p, m, s);
    const float2 ml = p.ws_ml[sl];
    const float4 o = *reinterpret_cast<const float4*>(p.ws_o + sl * D + 4 * dq);
    const float wgt = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - Mb);
    acc.x += wgt * o.x;
    acc.y += wgt * o.y;
    acc.z += wgt * o.z;
    acc.w += wgt * o.w;
    lsum += wgt * ml.y;
  }
  s_acc[pg][dq] = acc;
  if (dq == 0) s_l[pg] = lsum;
  __syncthreads();
  if (pg == 0) {
    float4 t = s_acc[0][dq];
    float l = s_l[0];
#pragma unroll
    for (int g = 1; g < PG; ++g) {
      const float4 o = s_acc[g][dq];
      t.x += o.x;
      t.y += o.y;
      t.z += o.z;
      t.w += o.w;
      l += s_l[g];
    }
    write_merged(p, m, dq, t, l, M, dq == 0);
  }
}

cudaError_t launch_merge(int head_dim, const MergeParams& p, int units, int rows, bool wide, bool pdl,
                         cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  if (wide) {
    cfg.gridDim = dim3(static_cast<unsigned>(units), static_cast<unsigned>(rows), 1);
    cfg.blockDim = dim3(kWideThreads, 1, 1);
  } else {
    cfg.gridDim = dim3(static_cast<unsigned>(units), static_cast<unsigned>((rows + kMergeWarps - 1) / kMergeWarps), 1);
    cfg.blockDim = dim3(32 * kMergeWarps, 1, 1);
  }
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (head_dim == 128)
    return wide ? cudaLaunchKernelEx(&cfg, pa_merge_wide_kernel<128>, p) : cudaLaunchKernelEx(&cfg, pa_merge_kernel<128>, p);
  if (head_dim == 64)
    return wide ? cudaLaunchKernelEx(&cfg, pa_merge_wide_kernel<64>, p) : cudaLaunchKernelEx(&cfg, pa_merge_kernel<64>, p);
  return cudaErrorInvalidValue;
}

}  // namespace pa
