// KV-cache write (ATOM model-operations guide, "KV cache operations": standard
// and FP8 KV cache writes; token_layout/slots.py: slot_mapping): every new token
// with slot s >= 0 stores its key and value rows of all KV heads at page s / 16,
// slot s % 16 of the paged caches.  bf16 caches take the rows as they are; fp8
// caches take e4m3fn codes of x * (1 / scale) (the reciprocal rounded once to
// fp32 on the host; round to nearest even, saturating to +-448).
//
// One thread moves 8 consecutive features (16 bytes of bf16 input) of one
// (token, head) row; the grid strides over all tokens x heads x 8-feature
// chunks.  A token's rows of all heads are one contiguous run in the cache, so
// the stores of a warp are contiguous.
#include "pa_device.cuh"
#include "pa_kernels.h"

namespace pa {

__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <bool FP8>
__global__ void __launch_bounds__(256) pa_cache_write_kernel(const CacheWriteParams p) {
  const int chunks_per_head = p.head_dim / 8;
  const int64_t chunks_per_token = static_cast<int64_t>(p.num_kv_heads) * chunks_per_head;
  const int64_t total = static_cast<int64_t>(p.num_tokens) * chunks_per_token;
  const int64_t num_slots = static_cast<int64_t>(p.num_pages) * kPage;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = idx / chunks_per_token;
    const int64_t rem = idx - t * chunks_per_token;
    const int h = static_cast<int>(rem / chunks_per_head);
    const int d0 = static_cast<int>(rem - static_cast<int64_t>(h) * chunks_per_head) * 8;
    const int64_t slot = p.slot_mapping[t];
    if (slot < 0) continue;                       // padding token
    if (slot >= num_slots) {
      if (d0 == 0 && h == 0) atomicOr(p.err, kErrPageRange);
      continue;
    }
    const int64_t page = slot / kPage;
    const int64_t off = slot - page * kPage;
#pragma unroll
    for (int tensor = 0; tensor < 2; ++tensor) {
      const uint16_t* src = (tensor ? p.value : p.key) + t * (tensor ? p.v_stride_t : p.k_stride_t) +
                            static_cast<int64_t>(h) * (tensor ? p.v_stride_h : p.k_stride_h) + d0;
      const int64_t dst_elem = page * (tensor ? p.vc_stride_page : p.kc_stride_page) +
                               off * (tensor ? p.vc_stride_slot : p.kc_stride_slot) +
                               static_cast<int64_t>(h) * (tensor ? p.vc_stride_head : p.kc_stride_head) + d0;
      const uint4 x = *reinterpret_cast<const uint4*>(src);
      if constexpr (FP8) {
        const float r = tensor ? p.v_rscale : p.k_rscale;
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t q[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          q[e] = e4m3x2_from_f32(bf16_lo(w[e]) * r, bf16_hi(w[e]) * r);
        uint2 out;
        out.x = q[0] | (q[1] << 16);
        out.y = q[2] | (q[3] << 16);
        uint8_t* dst = (tensor ? p.v_cache : p.k_cache) + dst_elem;
        *reinterpret_cast<uint2*>(dst) = out;
      } else {
        uint8_t* dst = (tensor ? p.v_cache : p.k_cache) + dst_elem * 2;
        *reinterpret_cast<uint4*>(dst) = x;
      }
    }
  }
}

// Per-token fp8 write (the pages' reshape_and_cache_with_pertoken_quant): the
// D / 8 threads of one (token, head) row sit on consecutive lanes of a warp
// (a row starts at a multiple of D / 8 in the flattened index, and D / 8
// divides 32), so the row's max |x| is an xor-shuffle reduction inside that
// lane group.  scale = amax / 448 and r = 448 / amax are IEEE fp32 divisions;
// codes = e4m3fn(x * r), round to nearest even, saturating; a zero row stores
// scale 0 and zero codes.  Every lane of a warp runs the same number of loop
// trips (the trip test is on the block's first index), so the shuffles see
// full warps.  A trip takes two index groups a grid apart and issues all four
// row loads (K and V of each) before the reductions.
__global__ void __launch_bounds__(256) pa_cache_write_tok_kernel(const CacheWriteParams p) {
  constexpr int U = 2;              // index groups per trip, all loads issued before any reduction
  const int cph = p.head_dim / 8;   // chunks per head (8 or 16)
  const int64_t chunks_per_token = static_cast<int64_t>(p.num_kv_heads) * cph;
  const int64_t total = static_cast<int64_t>(p.num_tokens) * chunks_per_token;
  const int64_t num_slots = static_cast<int64_t>(p.num_pages) * kPage;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x; i0 < total; i0 += U * stride) {
    int64_t t[U], page[U], off[U];
    int h[U], d0[U];
    bool live[U];
    uint4 xs[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t idx = i0 + u * stride + threadIdx.x;
      const bool in = idx < total;
      t[u] = in ? idx / chunks_per_token : 0;
      const int64_t rem = idx - t[u] * chunks_per_token;
      h[u] = in ? static_cast<int>(rem / cph) : 0;
      d0[u] = in ? static_cast<int>(rem - static_cast<int64_t>(h[u]) * cph) * 8 : 0;
      const int64_t slot = in ? p.slot_mapping[t[u]] : -1;
      if (in && slot >= num_slots && d0[u] == 0 && h[u] == 0) atomicOr(p.err, kErrPageRange);
      live[u] = in && slot >= 0 && slot < num_slots;
      page[u] = live[u] ? slot / kPage : 0;
      off[u] = live[u] ? slot - page[u] * kPage : 0;
      xs[u][0] = xs[u][1] = make_uint4(0u, 0u, 0u, 0u);
      if (live[u]) {
        xs[u][0] = *reinterpret_cast<const uint4*>(p.key + t[u] * p.k_stride_t +
                                                   static_cast<int64_t>(h[u]) * p.k_stride_h + d0[u]);
        xs[u][1] = *reinterpret_cast<const uint4*>(p.value + t[u] * p.v_stride_t +
                                                   static_cast<int64_t>(h[u]) * p.v_stride_h + d0[u]);
      }
    }
    float amax[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int tensor = 0; tensor < 2; ++tensor) {
        const uint4 x = xs[u][tensor];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
        amax[u][tensor] = a;
      }
    for (int o = 1; o < cph; o <<= 1)
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int tensor = 0; tensor < 2; ++tensor)
          amax[u][tensor] = fmaxf(amax[u][tensor], __shfl_xor_sync(0xffffffffu, amax[u][tensor], o));
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!live[u]) continue;
#pragma unroll
      for (int tensor = 0; tensor < 2; ++tensor) {
        const uint4 x = xs[u][tensor];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        const float a = amax[u][tensor];
        const float r = a > 0.f ? __fdiv_rn(448.f, a) : 0.f;
        uint32_t q[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) q[e] = e4m3x2_from_f32(bf16_lo(w[e]) * r, bf16_hi(w[e]) * r);
        const int64_t dst_elem = page[u] * (tensor ? p.vc_stride_page : p.kc_stride_page) +
                                 off[u] * (tensor ? p.vc_stride_slot : p.kc_stride_slot) +
                                 static_cast<int64_t>(h[u]) * (tensor ? p.vc_stride_head : p.kc_stride_head) + d0[u];
        *reinterpret_cast<uint2*>((tensor ? p.v_cache : p.k_cache) + dst_elem) =
            make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
        if (d0[u] == 0) {
          float* sc = tensor ? p.v_tok : p.k_tok;
          sc[page[u] * (tensor ? p.vs_stride_page : p.ks_stride_page) +
             static_cast<int64_t>(h[u]) * (tensor ? p.vs_stride_head : p.ks_stride_head) +
             off[u] * (tensor ? p.vs_stride_slot : p.ks_stride_slot)] = __fdiv_rn(a, 448.f);
        }
      }
    }
  }
}

cudaError_t launch_cache_write(bool fp8, const CacheWriteParams& p, int grid, cudaStream_t stream) {
  if (p.k_tok != nullptr) {
    pa_cache_write_tok_kernel<<<grid, 256, 0, stream>>>(p);
  } else if (fp8) {
    pa_cache_write_kernel<true><<<grid, 256, 0, stream>>>(p);
  } else {
    pa_cache_write_kernel<false><<<grid, 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace pa
