// KV-cache write (ATOM model-operations guide, "KV cache operations": standard
// and FP8 KV cache writes; token_layout/slots.py: slot_mapping): every new token
// with slot s >= 0 stores its key and value rows of all KV heads at page s / 16,
// slot s % 16 of the paged caches.  bf16 caches take the rows as they are; fp8
// caches take e4m3fn codes of x / scale (a cached value reads back as code *
// scale): the IEEE fp32 quotient (round to nearest even; see div_by2), then
// e4m3 round to nearest even, saturating to +-448.
//
// One thread moves 8 consecutive features (16 bytes of bf16 input) of one
// (token, head) row; a grid of one wave of resident blocks strides over all
// tokens x heads x 8-feature chunks.  A token's rows of all heads are one contiguous run in the cache, so
// the stores of a warp are contiguous.
#include "pa_device.cuh"
#include "pa_kernels.h"
#include "pa_pack.cuh"

namespace pa {

__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Division by a scale that stays fixed over many values: the IEEE
// round-to-nearest quotient x / s formed from the correctly rounded reciprocal
// r = 1/s by Markstein's correction step (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990; also Muller et al., "Handbook of Floating-Point
// Arithmetic", division with a fused multiply-add): q0 = x r rounded, the
// remainder x - q0 s exact by one FMA, and q0 + (x - q0 s) r rounded once.
// Kept from q0: a zero quotient (its sign: the correction's sum of zeros
// would be +0) and |q0| >= 1024 or NaN (the e4m3 code saturates at 448 either
// way, and an infinite q0 would make the remainder NaN).  Outside
// 2^-64 <= |s| <= 2^64 the plain IEEE division is used.  Checked equal to
// __fdiv_rn (quotients on [2^-20, 1000] and e4m3 codes everywhere) over every
// fp32 x, for every scale amax / 448 of a positive finite bf16 amax and 10000
// random scales (and, for a set of scales, by tests/test_cache_write_div_gpu.py).
struct ScaleDiv {
  float s, r;
  bool fast;
};

__device__ __forceinline__ ScaleDiv scale_div(float s) {
  ScaleDiv d;
  d.s = s;
  d.r = __frcp_rn(s);
  d.fast = fabsf(s) >= 5.421010862427522e-20f && fabsf(s) <= 1.8446744073709552e+19f;   // 2^-64 .. 2^64
  return d;
}

// (a, b) / s on the fast path, two at a time (packed f32x2 arithmetic, each
// half rounded as its scalar form would be).
__device__ __forceinline__ void div_by2(const ScaleDiv& d, float a, float b, float& qa, float& qb) {
  const uint64_t x = f2_pack(a, b);
  const uint64_t r2 = f2_pack(d.r, d.r), ns2 = f2_pack(-d.s, -d.s);
  const uint64_t q0 = fmul2(x, r2);
  const uint64_t q1 = ffma2(ffma2(q0, ns2, x), r2, q0);
  float a0, b0, a1, b1;
  f2_unpack(q0, a0, b0);
  f2_unpack(q1, a1, b1);
  qa = (a0 == 0.f || !(fabsf(a0) < 1024.f)) ? a0 : a1;
  qb = (b0 == 0.f || !(fabsf(b0) < 1024.f)) ? b0 : b1;
}

// Four e4m3fn code pairs of eight bf16 values (one 16-byte chunk) divided by
// the scale: every quotient the IEEE round-to-nearest fp32 division.
__device__ __forceinline__ uint2 e4m3x8_div(const uint4 v, const ScaleDiv& d) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t q[4];
  if (d.fast) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float lo, hi;
      div_by2(d, bf16_lo(w[e]), bf16_hi(w[e]), lo, hi);
      q[e] = e4m3x2_from_f32(lo, hi);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      q[e] = e4m3x2_from_f32(__fdiv_rn(bf16_lo(w[e]), d.s), __fdiv_rn(bf16_hi(w[e]), d.s));
  }
  return make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
}

// Integer quotient of an index by a per-call divisor: 32-bit when the index
// range fits (every practical call), 64-bit otherwise (a uniform branch).
__device__ __forceinline__ int64_t cw_div(int64_t a, int64_t b, bool narrow) {
  return narrow ? static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b)) : a / b;
}

// Per-tensor scales (or a bf16 copy).  A trip takes U chunk indices a grid
// apart; every row load is issued before any slot is looked at (a padding
// token's row is read and dropped), so a trip waits for one memory latency,
// not a slot lookup followed by the row loads.
template <bool FP8, int U>
__global__ void __launch_bounds__(256) pa_cache_write_kernel(const CacheWriteParams p) {
  const int cph = p.head_dim / 8;
  const int64_t cpt = static_cast<int64_t>(p.num_kv_heads) * cph;   // chunks per token
  const int64_t total = static_cast<int64_t>(p.num_tokens) * cpt;
  const bool narrow = total <= 0xFFFFFFFFll;
  const int64_t num_slots = static_cast<int64_t>(p.num_pages) * kPage;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const ScaleDiv dk = scale_div(p.k_scale), dv = scale_div(p.v_scale);
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < total; i0 += U * stride) {
    int64_t t[U];
    int h[U], d0[U], slot[U];
    uint4 x[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t idx = i0 + u * stride;
      const bool in = idx < total;
      t[u] = in ? cw_div(idx, cpt, narrow) : 0;
      const int rem = static_cast<int>(idx - t[u] * cpt);
      h[u] = in ? rem / cph : 0;
      d0[u] = in ? (rem - h[u] * cph) * 8 : 0;
      slot[u] = in ? p.slot_mapping[t[u]] : -1;
      x[u][0] = x[u][1] = make_uint4(0u, 0u, 0u, 0u);
      if (in) {
        x[u][0] = *reinterpret_cast<const uint4*>(p.key + t[u] * p.k_stride_t + h[u] * p.k_stride_h + d0[u]);
        x[u][1] = *reinterpret_cast<const uint4*>(p.value + t[u] * p.v_stride_t + h[u] * p.v_stride_h + d0[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (slot[u] < 0) continue;                   // padding token (or past the end)
      if (slot[u] >= num_slots) {
        if (d0[u] == 0 && h[u] == 0) atomicOr(p.err, kErrPageRange);
        continue;
      }
      const int64_t page = slot[u] / kPage;
      const int64_t off = slot[u] - page * kPage;
#pragma unroll
      for (int tensor = 0; tensor < 2; ++tensor) {
        const int64_t dst_elem = page * (tensor ? p.vc_stride_page : p.kc_stride_page) +
                                 off * (tensor ? p.vc_stride_slot : p.kc_stride_slot) +
                                 static_cast<int64_t>(h[u]) * (tensor ? p.vc_stride_head : p.kc_stride_head) + d0[u];
        if constexpr (FP8) {
          *reinterpret_cast<uint2*>((tensor ? p.v_cache : p.k_cache) + dst_elem) =
              e4m3x8_div(x[u][tensor], tensor ? dv : dk);
        } else {
          *reinterpret_cast<uint4*>((tensor ? p.v_cache : p.k_cache) + dst_elem * 2) = x[u][tensor];
        }
      }
    }
  }
}

// Largest of two pairs of 16-bit unsigned integers, half by half.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Per-token fp8 write (the pages' reshape_and_cache_with_pertoken_quant).  A
// (token, head) row of D / 8 16-byte chunks belongs to a group of G lanes of
// one warp, each lane taking CPL chunks c0, c0 + G, ... (G = the power of two
// with CPL * G covering the row, at most 32; chunks past the row's end idle), so the
// row's max |x| is an xor-shuffle reduction inside the group.  For finite bf16
// values the bit patterns with the sign cleared order like |x|, so the maxima
// are 16-bit integer maxima (exact), K's and V's carried in one 32-bit word.
// scale = amax / 448 and the codes e4m3fn(x / scale) are IEEE fp32 divisions
// (round to nearest even, saturating); a zero row stores scale 0 and zero
// codes.  The trip test is on the warp's first row, so every lane of a
// warp runs the same trips and the shuffles see full warps.  A trip takes U rows
// per group, a grid apart, and issues all their loads (K and V) together with
// the slot lookups.
template <int CPL, int U>
__global__ void __launch_bounds__(256) pa_cache_write_tok_kernel(const CacheWriteParams p, int G) {
  const int lane = threadIdx.x & 31;
  const int c0 = lane & (G - 1);
  const int rpw = 32 / G;                                   // rows per warp per index group
  const int64_t rows = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads;
  const bool narrow = rows <= 0xFFFFFFFFll;
  const int64_t num_slots = static_cast<int64_t>(p.num_pages) * kPage;
  const int64_t wpass = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32) * rpw;   // rows per grid pass
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32) * rpw;
  for (int64_t rb = w0; rb < rows; rb += U * wpass) {
    int64_t t[U];
    int h[U], slot[U];
    uint4 x[U][CPL][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t r = rb + u * wpass + lane / G;
      const bool in = r < rows;
      t[u] = in ? cw_div(r, p.num_kv_heads, narrow) : 0;
      h[u] = in ? static_cast<int>(r - t[u] * p.num_kv_heads) : 0;
      slot[u] = in ? p.slot_mapping[t[u]] : -1;
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        const int d0 = (c0 + k * G) * 8;
        x[u][k][0] = x[u][k][1] = make_uint4(0u, 0u, 0u, 0u);
        if (in && d0 < p.head_dim) {
          x[u][k][0] = *reinterpret_cast<const uint4*>(p.key + t[u] * p.k_stride_t + h[u] * p.k_stride_h + d0);
          x[u][k][1] = *reinterpret_cast<const uint4*>(p.value + t[u] * p.v_stride_t + h[u] * p.v_stride_h + d0);
        }
      }
    }
    uint32_t m[U];   // |x| maxima as bf16 bits: K's in the low half, V's in the high half
#pragma unroll
    for (int u = 0; u < U; ++u) {
      uint32_t mk = 0u, mv = 0u;
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        const uint4 a = x[u][k][0], b = x[u][k][1];
        mk = max_u16x2(mk, max_u16x2(max_u16x2(a.x & 0x7FFF7FFFu, a.y & 0x7FFF7FFFu),
                                     max_u16x2(a.z & 0x7FFF7FFFu, a.w & 0x7FFF7FFFu)));
        mv = max_u16x2(mv, max_u16x2(max_u16x2(b.x & 0x7FFF7FFFu, b.y & 0x7FFF7FFFu),
                                     max_u16x2(b.z & 0x7FFF7FFFu, b.w & 0x7FFF7FFFu)));
      }
      m[u] = max_u16x2(__byte_perm(mk, mv, 0x5410), __byte_perm(mk, mv, 0x7632));
    }
    for (int o = 1; o < G; o <<= 1)
#pragma unroll
      for (int u = 0; u < U; ++u) m[u] = max_u16x2(m[u], __shfl_xor_sync(0xffffffffu, m[u], o));
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (slot[u] < 0) continue;
      if (slot[u] >= num_slots) {
        if (c0 == 0 && h[u] == 0) atomicOr(p.err, kErrPageRange);
        continue;
      }
      const int64_t page = slot[u] / kPage;
      const int64_t off = slot[u] - page * kPage;
      // every lane of the group forms the row's two scales (the same IEEE
      // quotients), so no broadcast is needed; an all-zero row's scale is 0
      const float sc[2] = {__fdiv_rn(__uint_as_float(m[u] << 16), 448.f),
                           __fdiv_rn(__uint_as_float(m[u] & 0xFFFF0000u), 448.f)};
      const ScaleDiv ds[2] = {scale_div(sc[0]), scale_div(sc[1])};
#pragma unroll
      for (int tensor = 0; tensor < 2; ++tensor) {
        uint8_t* row = (tensor ? p.v_cache : p.k_cache) + page * (tensor ? p.vc_stride_page : p.kc_stride_page) +
                       off * (tensor ? p.vc_stride_slot : p.kc_stride_slot) +
                       static_cast<int64_t>(h[u]) * (tensor ? p.vc_stride_head : p.kc_stride_head);
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
          const int d0 = (c0 + k * G) * 8;
          if (d0 >= p.head_dim) continue;
          // an all-zero row (its elements +0 or -0) stores the code 0x00 throughout
          *reinterpret_cast<uint2*>(row + d0) =
              sc[tensor] > 0.f ? e4m3x8_div(x[u][k][tensor], ds[tensor]) : make_uint2(0u, 0u);
        }
      }
      // the row's two scales: lane c0 = 0 stores K's and c0 = 1 V's (one lane
      // both when G = 1)
      for (int j = c0; j < 2; j += G) {
        float* dst = j ? p.v_tok : p.k_tok;
        dst[page * (j ? p.vs_stride_page : p.ks_stride_page) +
            static_cast<int64_t>(h[u]) * (j ? p.vs_stride_head : p.ks_stride_head) +
            off * (j ? p.vs_stride_slot : p.ks_stride_slot)] = sc[j];
      }
    }
  }
}

namespace {

int g_occ[3] = {1, 1, 1};   // resident 256-thread blocks per SM of each write kernel

template <typename K>
int resident_blocks(K kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, 0) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();
    n = 1;
  }
  return n;
}

int grid_for(int64_t need, int num_sms, int occ) {
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(need, int64_t(num_sms) * occ)));
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Chosen by timing the 16384-token chunk (8 KV heads, D128) over chunks per
// lane x index groups per trip: more rows in flight per thread cost occupancy
// and gained nothing; four chunks per lane share one row's reduction, divisions
// and address arithmetic.
constexpr int kU = 1;          // per-tensor write: index groups per trip
constexpr int kCpl = 4;        // per-token write: chunks of a row per lane (kCpl * 32 * 8 >= 512 features)
constexpr int kUTok = 1;       // per-token write: rows per lane group per trip

}  // namespace

void init_cache_write_occupancy() {
  g_occ[0] = resident_blocks(pa_cache_write_kernel<false, kU>);
  g_occ[1] = resident_blocks(pa_cache_write_kernel<true, kU>);
  g_occ[2] = resident_blocks(pa_cache_write_tok_kernel<kCpl, kUTok>);
}

// Grid: the blocks that fit on the device at once (one wave), fewer when the
// call has less work than one trip of each thread.
cudaError_t launch_cache_write(bool fp8, const CacheWriteParams& p, int num_sms, cudaStream_t stream) {
  const int cph = p.head_dim / 8;
  if (p.k_tok != nullptr) {
    int G = 1;
    while (kCpl * G < cph && G < 32) G <<= 1;
    const int64_t rows = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads;
    pa_cache_write_tok_kernel<kCpl, kUTok>
        <<<grid_for(ceil_div(rows, int64_t(8) * (32 / G) * kUTok), num_sms, g_occ[2]), 256, 0, stream>>>(p, G);
    return cudaGetLastError();
  }
  const int64_t need = ceil_div(static_cast<int64_t>(p.num_tokens) * p.num_kv_heads * cph, int64_t(256) * kU);
  if (fp8)
    pa_cache_write_kernel<true, kU><<<grid_for(need, num_sms, g_occ[1]), 256, 0, stream>>>(p);
  else
    pa_cache_write_kernel<false, kU><<<grid_for(need, num_sms, g_occ[0]), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
