// Log-sum-exp merge of split partials (high-interactivity blog, "Attention
// Decode: Split Memory Work to Fill the Device": per-split log-sum-exp values
// kept in fp32, merged afterwards).
//
// A unit (sequence i, head chunk c) whose page range lies inside one split CTA
// was finished by that CTA and is skipped.  Otherwise the CTAs g_first..g_last
// that cut it each left, in slot 2g (the CTA's first unit) or 2g+1 (its last
// unit), the unnormalised output O_s, the running max m_s (log2 units) and the
// sum l_s; the CTA holding the unit's first page also wrote the unit's
// descriptor (g_first, piece count, query tokens).  With M = max_s m_s:
//   out = v_scale * sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s
//   lse = ln 2 * (M + log2 sum_s 2^(m_s - M) l_s)
// accumulated online (running max), so each partial is loaded once.
#include <cuda_fp16.h>

#include "pa_device.cuh"
#include "pa_kernels.h"

namespace pa {

constexpr int kMergeWarps = 8;
constexpr int kWideThreads = 1024;

struct MergeRow {
  bool work;        // row exists and its unit was cut into >= 2 pieces
  uint16_t* orow;
  float* lse_ptr;
  int hh, rho, hq;
  int gf, nparts;
  bool first_is_tail;
};

// (unit u, row) -> output row and the pieces to merge, from the descriptor the
// split kernel wrote for the unit (one metadata load).  Rows of a unit that was
// finished inside one CTA, or that do not exist for the sequence, report
// work = false.  An empty context (no page ever touched) writes out = 0 and
// lse = -inf here.
template <int D>
__device__ __forceinline__ MergeRow merge_row(const MergeParams& p, int u, int row, int lane) {
  MergeRow m;
  m.work = false;
  if (row >= p.HC * p.R_max) return m;
  const int i = u / p.NC;
  const int c = u - i * p.NC;
  m.hh = row / p.R_max;
  m.rho = row - m.hh * p.R_max;
  const int4 d = p.ws_unit[u];
  const int L = p.seq_lens[i];
  if (L <= 0) {
    int t0 = i, qn = 1;
    if (p.qsl != nullptr) {
      t0 = p.qsl[i];
      qn = p.qsl[i + 1] - t0;
    }
    if (qn < 1 || qn > p.max_qlen || t0 < 0 || t0 + qn > p.num_tokens || m.rho >= p.G * qn || lane < 0) return m;
    uint16_t* orow = p.out + static_cast<int64_t>(t0 + m.rho / p.G) * p.out_stride_t +
                     static_cast<int64_t>((c * p.HC + m.hh) * p.G + m.rho % p.G) * p.out_stride_h;
    for (int dd = 2 * lane; dd < D; dd += 64) *reinterpret_cast<uint32_t*>(orow + dd) = 0u;
    if (lane == 0) {
      if (p.lse)
        p.lse[static_cast<int64_t>(t0 + m.rho / p.G) * p.lse_stride_t +
              static_cast<int64_t>((c * p.HC + m.hh) * p.G + m.rho % p.G) * p.lse_stride_h] = -INFINITY;
      atomicOr(p.err, kErrSeqLen);
    }
    return m;
  }
  m.gf = d.x;
  m.nparts = d.y & 0x3fffffff;
  m.first_is_tail = (d.y >> 30) & 1;
  const int t0 = d.z, qn = d.w;
  // A descriptor this call's split kernel did not write (its CTA gave up on a
  // timed-out wait) may hold anything: one that would index outside the
  // workspace or the outputs is skipped, so a failed call stays in bounds.
  if (m.gf < 0 || m.nparts > p.split_grid - m.gf || t0 < 0 || qn < 1 || qn > p.max_qlen || t0 > p.num_tokens - qn)
    return m;
  if (m.nparts <= 1 || m.rho >= p.G * qn) return m;
  const int t = t0 + m.rho / p.G;
  const int hq = (c * p.HC + m.hh) * p.G + m.rho % p.G;
  m.hq = hq;
  m.orow = p.out + static_cast<int64_t>(t) * p.out_stride_t + static_cast<int64_t>(hq) * p.out_stride_h;
  m.lse_ptr = p.lse ? p.lse + static_cast<int64_t>(t) * p.lse_stride_t + static_cast<int64_t>(hq) * p.lse_stride_h
                    : nullptr;
  m.work = true;
  return m;
}

__device__ __forceinline__ int64_t slot_row(const MergeParams& p, const MergeRow& m, int s) {
  const int which = (s == 0 && m.first_is_tail) ? 1 : 0;
  return (static_cast<int64_t>(2 * (m.gf + s) + which) * p.HC + m.hh) * p.R_max + m.rho;
}

// Online log-sum-exp accumulation of one partial (running max mx in log2 units).
__device__ __forceinline__ void lse_acc(float& mx, float& l, float4& acc, float m_s, float l_s, const float4& o) {
  if (m_s == -INFINITY) return;
  const float nm = fmaxf(mx, m_s);
  const float a = fast_exp2(mx - nm);     // 0 when mx = -inf
  const float b = fast_exp2(m_s - nm);
  acc.x = acc.x * a + o.x * b;
  acc.y = acc.y * a + o.y * b;
  acc.z = acc.z * a + o.z * b;
  acc.w = acc.w * a + o.w * b;
  l = l * a + l_s * b;
  mx = nm;
}

// Partials s = first, first + stride, ... of row m: loads of four partials are
// issued before any of them is combined.
template <int D>
__device__ __forceinline__ void gather_partials(const MergeParams& p, const MergeRow& m, int first, int stride, int dq,
                                                float& mx, float& l, float4& acc) {
  int s = first;
  for (; s + 3 * stride < m.nparts; s += 4 * stride) {
    float2 ml[4];
    float4 o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t sl = slot_row(p, m, s + u * stride);
      ml[u] = p.ws_ml[sl];
      o[u] = *reinterpret_cast<const float4*>(p.ws_o + sl * D + 4 * dq);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) lse_acc(mx, l, acc, ml[u].x, ml[u].y, o[u]);
  }
  for (; s < m.nparts; s += stride) {
    const int64_t sl = slot_row(p, m, s);
    const float2 ml = p.ws_ml[sl];
    const float4 o = *reinterpret_cast<const float4*>(p.ws_o + sl * D + 4 * dq);
    lse_acc(mx, l, acc, ml.x, ml.y, o);
  }
}

__device__ __forceinline__ void write_merged(const MergeParams& p, const MergeRow& m, int dq, float4 acc, float l,
                                             float mx, bool write_lse) {
  const float inv = l > 0.f ? p.v_scale / l : 0.f;
  uint2 pk;
  pk.x = pack_bf16(acc.x * inv, acc.y * inv);
  pk.y = pack_bf16(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(m.orow + 4 * dq) = pk;
  if (write_lse && m.lse_ptr) *m.lse_ptr = l > 0.f ? (mx + fast_log2(l)) * 0.69314718055994530942f : -INFINITY;
}

// One warp per (unit, row): units cut into a few pieces.
template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) pa_merge_kernel(const MergeParams p) {
  grid_dependency_wait();   // results of the split kernel (programmatic dependent launch)
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const MergeRow m = merge_row<D>(p, blockIdx.x, blockIdx.y * kMergeWarps + warp, lane);
  if (!m.work) return;
  constexpr int LPD = D / 4;          // lanes per partial row (float4 each)
  constexpr int PL = 32 / LPD;        // partials side by side
  const int dq = lane % LPD;
  const int pl = lane / LPD;
  float mx = -INFINITY, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  gather_partials<D>(p, m, pl, PL, dq, mx, l, acc);
#pragma unroll
  for (int o = LPD; o < 32; o <<= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, mx, o);
    const float lo = __shfl_xor_sync(0xffffffffu, l, o);
    float4 ao;
    ao.x = __shfl_xor_sync(0xffffffffu, acc.x, o);
    ao.y = __shfl_xor_sync(0xffffffffu, acc.y, o);
    ao.z = __shfl_xor_sync(0xffffffffu, acc.z, o);
    ao.w = __shfl_xor_sync(0xffffffffu, acc.w, o);
    lse_acc(mx, l, acc, mo, lo, ao);
  }
  if (pl == 0) write_merged(p, m, dq, acc, l, mx, lane == 0);
}

// One 1024-thread block per (unit, row): units cut into many pieces (a long
// context spread over every SM); each thread gathers a few partials in one
// round of loads, then a tree in shared memory combines the groups.
template <int D>
__global__ void __launch_bounds__(kWideThreads) pa_merge_wide_kernel(const MergeParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  constexpr int LPD = D / 4;
  constexpr int PG = kWideThreads / LPD;
  __shared__ float4 s_acc[PG][LPD];
  __shared__ float2 s_ml[PG][LPD];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int dq = tid % LPD;
  const int pg = tid / LPD;
  // A single unit (one sequence and head chunk over the whole grid, the
  // batch-1 case) starts at CTA 0's first page, so its piece s is CTA s's
  // slot 2s: those loads go out before the unit's descriptor returns (slots
  // past the piece count hold stale values and are dropped below).
  constexpr int kSpec = 256 / PG;   // up to 256 split CTAs
  const bool spec = gridDim.x == 1 && p.split_grid <= kSpec * PG;
  float2 sml[kSpec];
  float4 so[kSpec];
  if (spec) {
    const int hh = blockIdx.y / p.R_max, rho = blockIdx.y - hh * p.R_max;
#pragma unroll
    for (int u = 0; u < kSpec; ++u) {
      const int sp = pg + u * PG;
      if (sp < p.split_grid && blockIdx.y < p.HC * p.R_max) {
        const int64_t sl = (static_cast<int64_t>(2 * sp) * p.HC + hh) * p.R_max + rho;
        sml[u] = p.ws_ml[sl];
        so[u] = *reinterpret_cast<const float4*>(p.ws_o + sl * D + 4 * dq);
      }
    }
  }
  const MergeRow m = merge_row<D>(p, blockIdx.x, blockIdx.y, tid < 32 ? lane : -1);
  if (!m.work) return;
  float mx = -INFINITY, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (spec && m.gf == 0 && !m.first_is_tail) {
#pragma unroll
    for (int u = 0; u < kSpec; ++u)
      if (pg + u * PG < m.nparts) lse_acc(mx, l, acc, sml[u].x, sml[u].y, so[u]);
  } else {
    gather_partials<D>(p, m, pg, PG, dq, mx, l, acc);
  }
  s_acc[pg][dq] = acc;
  s_ml[pg][dq] = make_float2(mx, l);
  __syncthreads();
#pragma unroll
  for (int half = PG / 2; half >= 1; half >>= 1) {
    if (pg < half) {
      const float2 ml = s_ml[pg + half][dq];
      lse_acc(mx, l, acc, ml.x, ml.y, s_acc[pg + half][dq]);
      s_acc[pg][dq] = acc;
      s_ml[pg][dq] = make_float2(mx, l);
    }
    __syncthreads();
  }
  if (pg == 0) write_merged(p, m, dq, acc, l, mx, dq == 0);
}

// MLA: 512 value columns per row (the latent width); the split kernel leaves
// each piece's normalised output O_s / l_s in f16 (p.ws_o read as f16) with
// (m_s, l_s), so a piece weighs 2^(m_s - M) l_s.  One warp per (unit, row),
// lane l holding columns 4 l + 128 j (j < 4); two partials' loads are issued
// before either is combined.
__device__ __forceinline__ float4 f16x4_to_float4(uint2 v) {
  const __half2 a = *reinterpret_cast<const __half2*>(&v.x);
  const __half2 b = *reinterpret_cast<const __half2*>(&v.y);
  const float2 fa = __half22float2(a), fb = __half22float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}

// true if one of the four f16 values is infinite or NaN (exponent all ones)
__device__ __forceinline__ bool f16x4_overflow(uint2 v) {
  return ((v.x & 0x7C00u) == 0x7C00u) || ((v.x & 0x7C000000u) == 0x7C000000u) || ((v.y & 0x7C00u) == 0x7C00u) ||
         ((v.y & 0x7C000000u) == 0x7C000000u);
}

__device__ __forceinline__ void lse_acc4(float& mx, float& l, float4 (&acc)[4], float2 ml, const uint2 (&o)[4],
                                         bool& overflow) {
  if (ml.x == -INFINITY || !(ml.y > 0.f)) return;
#pragma unroll
  for (int j = 0; j < 4; ++j) overflow |= f16x4_overflow(o[j]);
  const float nm = fmaxf(mx, ml.x);
  const float a = fast_exp2(mx - nm);
  const float b = fast_exp2(ml.x - nm);
  const float bw = b * ml.y;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 v = f16x4_to_float4(o[j]);
    acc[j].x = acc[j].x * a + v.x * bw;
    acc[j].y = acc[j].y * a + v.y * bw;
    acc[j].z = acc[j].z * a + v.z * bw;
    acc[j].w = acc[j].w * a + v.w * bw;
  }
  l = l * a + bw;
  mx = nm;
}

__global__ void __launch_bounds__(32 * kMergeWarps) pa_merge_mla_kernel(const MergeParams p) {
  constexpr int D = 512;
  grid_dependency_wait();
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const MergeRow m = merge_row<D>(p, blockIdx.x, blockIdx.y * kMergeWarps + warp, lane);
  if (!m.work) return;
  const uint16_t* ws = reinterpret_cast<const uint16_t*>(p.ws_o);
  float mx = -INFINITY, l = 0.f;
  bool overflow = false;   // a piece's f16 output beyond the f16 range
  float4 acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  int s = 0;
  for (; s + 1 < m.nparts; s += 2) {
    const int64_t sa = slot_row(p, m, s), sb = slot_row(p, m, s + 1);
    const float2 ma = p.ws_ml[sa], mb = p.ws_ml[sb];
    uint2 oa[4], ob[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      oa[j] = *reinterpret_cast<const uint2*>(ws + sa * D + 4 * lane + 128 * j);
      ob[j] = *reinterpret_cast<const uint2*>(ws + sb * D + 4 * lane + 128 * j);
    }
    lse_acc4(mx, l, acc, ma, oa, overflow);
    lse_acc4(mx, l, acc, mb, ob, overflow);
  }
  if (s < m.nparts) {
    const int64_t sa = slot_row(p, m, s);
    const float2 ma = p.ws_ml[sa];
    uint2 oa[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) oa[j] = *reinterpret_cast<const uint2*>(ws + sa * D + 4 * lane + 128 * j);
    lse_acc4(mx, l, acc, ma, oa, overflow);
  }
  if (overflow) atomicOr(p.err, kErrF16Range);
#pragma unroll
  for (int j = 0; j < 4; ++j) write_merged(p, m, lane + 32 * j, acc[j], l, mx, lane == 0 && j == 0);
}

cudaError_t launch_merge_mla(const MergeParams& p, int units, int rows, bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units), static_cast<unsigned>((rows + kMergeWarps - 1) / kMergeWarps), 1);
  cfg.blockDim = dim3(32 * kMergeWarps, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, pa_merge_mla_kernel, p);
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
