// Split-KV paged decode kernel (sm_103a).
//
// Work decomposition (high-interactivity blog, "Attention Decode: Split Memory
// Work to Fill the Device": split the KV walk so the device is full, keep the
// per-split log-sum-exp in fp32 and merge afterwards):
//   * a work unit is (sequence i, chunk c of HC consecutive KV heads); it has
//     n_i = ceil(L_i / 16) pages.  Units are laid end to end in (i, c, page)
//     order, X pages in total;
//   * CTA g of the NG CTAs in use takes the contiguous page range
//     [g*X/NG, (g+1)*X/NG), so every CTA moves the same number of bytes
//     whatever the ragged sequence lengths.  A unit that lies wholly inside one
//     CTA's range is finished there (out and lse written); the pieces of a unit
//     cut by a range boundary leave fp32 partials (unnormalised O, running max,
//     running sum) in the workspace for the merge kernel.  A CTA has at most two
//     such pieces: its first and its last unit.
//
// CTA layout: warp 0 is the producer, warps 1..HC*MT are consumers.
//   * producer: for every page of its range, reads the block-table entry (32 at
//     a time, one per lane, the next 32 prefetched) and issues TMA tile loads of
//     that page's K and V rows for the HC heads into a ring of `nstage`
//     shared-memory stages: one box per tensor and 128-byte column block, box =
//     (128 or 64 bytes of the row) x 16 slots x HC heads with the matching
//     swizzle, so a page of all HC heads costs 2-4 TMA instructions; at the
//     first page of a unit it also bulk-copies the unit's query rows into one of
//     two query slots.
//   * consumer (kv head hh of the chunk, 16-row tile w): query rows
//     rho = 16w .. 16w+15 of that head, where rho = r*G + gg is query token r of
//     the run and query head gg of the group.  Per page it computes
//     S = Q K^T with mma.sync m16n8k16 (bf16, or f16 for fp8 caches: e4m3 -> f16
//     is exact), applies the causal / tail mask, runs the online softmax in the
//     exp2 domain with quad shuffles, and accumulates O += P V.
// All waits are bounded (they report a timeout in the status word and stop).
#pragma once

#include <climits>

#include "pa_device.cuh"
#include "pa_kernels.h"
#include "pa_pack.cuh"

namespace pa {

constexpr int kSplitMaxThreads = 32 * 9;   // producer + up to 8 consumer warps

struct Cursor {
  int i;   // sequence
  int c;   // head chunk
  int j;   // page within the sequence
  int n;   // pages of sequence i
};

__device__ __forceinline__ int pages_of(const int32_t* pre, int i) { return pre[i + 1] - pre[i]; }

// Position x (0 <= x < X) of the flattened (sequence, head chunk, page) order.
__device__ __forceinline__ Cursor locate(const int32_t* pre, int B, int NC, int64_t x) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(NC) * pre[mid] <= x) lo = mid; else hi = mid - 1;
  }
  Cursor cu;
  cu.i = lo;
  cu.n = pages_of(pre, lo);
  const int64_t off = x - static_cast<int64_t>(NC) * pre[lo];
  cu.c = static_cast<int>(off / cu.n);
  cu.j = static_cast<int>(off % cu.n);
  return cu;
}

__device__ __forceinline__ void advance(Cursor& cu, const int32_t* pre, int B, int NC) {
  if (++cu.j < cu.n) return;
  cu.j = 0;
  if (++cu.c < NC) return;
  cu.c = 0;
  do {
    ++cu.i;
  } while (cu.i < B && pages_of(pre, cu.i) == 0);
  cu.n = (cu.i < B) ? pages_of(pre, cu.i) : 1;
}

struct SeqInfo {
  int L;    // cached tokens (including the query tokens)
  int t0;   // first query token
  int qn;   // query tokens (0 if the metadata is invalid)
  int js;   // first page any query row can see (sliding window), else 0
};

// First page a sequence's query rows can see: with a sliding window of W keys
// the earliest visible key is L - qn - W + 1 (query row 0); pages before it are
// never fetched.
__device__ __forceinline__ int first_visible_page(int L, int qn, int window) {
  if (window <= 0 || qn < 1) return 0;
  const int first_key = L - qn - window + 1;
  return first_key > 0 ? first_key / kPage : 0;
}

// Sequence metadata from the shared-memory copies made in the prologue.
__device__ __forceinline__ SeqInfo seq_info(const SplitParams& p, const int32_t* s_len, const int32_t* s_qsl, int i,
                                            bool report, int window) {
  SeqInfo s;
  s.L = s_len[i];
  s.t0 = s_qsl[i];
  s.qn = s_qsl[i + 1] - s.t0;
  if (s.qn < 1 || s.qn > p.max_qlen || s.t0 < 0 || s.t0 + s.qn > p.num_tokens) {
    if (report) atomicOr(p.err, kErrQueryLen);
    s.qn = 0;
  } else if (s.qn > s.L && report) {
    atomicOr(p.err, kErrSeqLen);
  }
  s.js = first_visible_page(s.L, s.qn, window);
  return s;
}

template <int D, bool FP8>
struct Geo {
  static constexpr int ESZ = FP8 ? 1 : 2;            // bytes per cached element
  static constexpr int ROWB = D * ESZ;               // bytes of one cached row
  static constexpr int RB = ROWB >= 128 ? 128 : 64;  // bytes per box row (swizzle span)
  static constexpr int NBOX = ROWB / RB;             // boxes per row
  static constexpr int CPB = RB / 16;                // 16-byte chunks per box row
  static constexpr int BOX_BYTES = 16 * RB;          // one 16-row box
  static constexpr int KS = D / 16;                  // k-steps of Q K^T
  static constexpr int NT = D / 8;                   // n-tiles of P V
};

// Byte offset of 16-byte chunk `chunk` of row `row` of one head's tiles.  A
// stage holds, per tensor, NBOX column blocks of HC heads x 16 rows; the column
// blocks are `block_stride` = HC * BOX_BYTES apart, heads BOX_BYTES apart.
template <int D, bool FP8>
__device__ __forceinline__ uint32_t tile_off(int row, int chunk, uint32_t block_stride) {
  using GG = Geo<D, FP8>;
  return (chunk / GG::CPB) * block_stride + swz<GG::RB>(row, chunk % GG::CPB);
}

// Output feature index of element e (0/1) of accumulator tile J for lane tig.
template <int D, bool FP8>
__device__ __forceinline__ int d_of(int J, int e, int tig) {
  if constexpr (FP8) {
    return 16 * (J >> 1) + 4 * tig + 2 * e + (J & 1);
  } else {
    return 8 * J + 2 * tig + e;
  }
}

// Prologue shared by the split kernels (all threads of the CTA call it):
// sequence lengths and query starts copied to shared memory, pages of work per
// sequence (pages before a sliding window excluded) and their exclusive prefix.
__device__ __forceinline__ void page_prefix(const SplitParams& p, int window, int32_t* s_pre, int32_t* s_len,
                                            int32_t* s_qsl, int* s_scan, int* s_total) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nwarps = blockDim.x >> 5;
  const int B = p.num_seqs;
  int carry = 0;
  for (int b0 = 0; b0 < B; b0 += blockDim.x) {
    const int i = b0 + tid;
    int v = 0;
    if (i < B) {
      const int L = p.seq_lens[i];
      s_len[i] = L;
      s_qsl[i] = p.qsl != nullptr ? p.qsl[i] : i;
      v = L > 0 ? (L + kPage - 1) / kPage : 0;
      if (v > p.max_blocks) {       // context longer than its block-table row: never read past the row
        atomicOr(p.err, kErrSeqLen);
        v = p.max_blocks;
      }
      const int qn = p.qsl != nullptr ? p.qsl[i + 1] - p.qsl[i] : 1;
      v -= min(v, first_visible_page(L, qn, window));   // pages before the sliding window are skipped
    }
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_scan[warp] = x;
    __syncthreads();
    if (warp == 0) {
      const int wv = lane < nwarps ? s_scan[lane] : 0;
      int xs = wv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, xs, o);
        if (lane >= o) xs += y;
      }
      if (lane < nwarps) s_scan[lane] = xs - wv;
      if (lane == 31) *s_total = xs;
    }
    __syncthreads();
    if (i < B) s_pre[i] = carry + s_scan[warp] + x - v;
    carry += *s_total;
    __syncthreads();
  }
  if (tid == 0) {
    s_pre[B] = carry;
    s_qsl[B] = p.qsl != nullptr ? p.qsl[B] : B;
  }
}

// Block-table entries for the producer warp: 32 at a time (one per lane),
// the batch the traversal reaches next loaded ahead of use.  All lanes call
// lookup() with the same cursor; it returns the physical page of cu.
struct BlockTableCache {
  int bt_i = -1, bt_j0 = 0, bt_val = 0;   // entries [bt_j0, bt_j0 + 32) of sequence bt_i
  int nx_i = -1, nx_j0 = 0, nx_val = 0;   // the batch after it

  __device__ __forceinline__ int lookup(const SplitParams& p, const Cursor& cu, const int32_t* s_pre,
                                        const int32_t* s_len, const int32_t* s_qsl, int B, int NC, int window,
                                        int lane) {
    if (cu.i != bt_i || cu.j < bt_j0 || cu.j >= bt_j0 + 32) {
      if (cu.i == nx_i && cu.j == nx_j0) {
        bt_val = nx_val;
      } else {
        const int jj = cu.j + lane;
        const int js = first_visible_page(s_len[cu.i], s_qsl[cu.i + 1] - s_qsl[cu.i], window);
        bt_val = (jj < cu.n) ? p.block_tables[static_cast<int64_t>(cu.i) * p.bt_stride + js + jj] : 0;
      }
      bt_i = cu.i;
      bt_j0 = cu.j;
      int ni = -1, nj = 0;
      if (bt_j0 + 32 < cu.n) {
        ni = cu.i;
        nj = bt_j0 + 32;
      } else if (cu.c + 1 < NC) {
        ni = cu.i;
      } else {
        ni = cu.i + 1;
        while (ni < B && pages_of(s_pre, ni) == 0) ++ni;
        if (ni >= B) ni = -1;
      }
      nx_i = ni;
      nx_j0 = nj;
      if (ni >= 0) {
        const int jj = nj + lane;
        const int js = first_visible_page(s_len[ni], s_qsl[ni + 1] - s_qsl[ni], window);
        nx_val = (jj < pages_of(s_pre, ni)) ? p.block_tables[static_cast<int64_t>(ni) * p.bt_stride + js + jj] : 0;
      }
    }
    return __shfl_sync(0xffffffffu, bt_val, cu.j - bt_j0);
  }
};

// Per-warp online-softmax state for 16 query rows of one KV head.
template <int D, bool FP8>
struct ConsumerState {
  using GG = Geo<D, FP8>;
  float O[GG::NT][4];       // unnormalised output, mma C fragments
  uint32_t Qf[GG::KS][4];   // query rows, mma A fragments
  float m0, m1, l0, l1;     // running max (log2 units) and this lane's share of the sum, rows g and g+8

  __device__ __forceinline__ void reset() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int J = 0; J < GG::NT; ++J) O[J][0] = O[J][1] = O[J][2] = O[J][3] = 0.f;
  }

  // Query rows (bf16 in shared memory) into A fragments.  For fp8 caches the
  // rows become f16 with the feature order of the fp8 K fragments: inside a
  // k-step, k = 2*tig + {0,1} holds d = 16*ks + 4*tig + {0,1} and
  // k = 2*tig + 8 + {0,1} holds d + 2.  Returns false if a value overflowed f16.
  __device__ __forceinline__ bool load_query(const uint8_t* q0p, const uint8_t* q1p, bool ok0, bool ok1, int tig) {
    bool fine = true;
#pragma unroll
    for (int ks = 0; ks < GG::KS; ++ks) {
      if constexpr (FP8) {
        const uint2 a = ok0 ? *reinterpret_cast<const uint2*>(q0p + (16 * ks + 4 * tig) * 2) : make_uint2(0u, 0u);
        const uint2 b = ok1 ? *reinterpret_cast<const uint2*>(q1p + (16 * ks + 4 * tig) * 2) : make_uint2(0u, 0u);
        Qf[ks][0] = pack_f16(bf16_lo(a.x), bf16_hi(a.x));
        Qf[ks][1] = pack_f16(bf16_lo(b.x), bf16_hi(b.x));
        Qf[ks][2] = pack_f16(bf16_lo(a.y), bf16_hi(a.y));
        Qf[ks][3] = pack_f16(bf16_lo(b.y), bf16_hi(b.y));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t v = Qf[ks][e];
          fine &= ((v & 0x7C00u) != 0x7C00u) && ((v & 0x7C000000u) != 0x7C000000u);
        }
      } else {
        Qf[ks][0] = ok0 ? *reinterpret_cast<const uint32_t*>(q0p + (16 * ks + 2 * tig) * 2) : 0u;
        Qf[ks][1] = ok1 ? *reinterpret_cast<const uint32_t*>(q1p + (16 * ks + 2 * tig) * 2) : 0u;
        Qf[ks][2] = ok0 ? *reinterpret_cast<const uint32_t*>(q0p + (16 * ks + 8 + 2 * tig) * 2) : 0u;
        Qf[ks][3] = ok1 ? *reinterpret_cast<const uint32_t*>(q1p + (16 * ks + 8 + 2 * tig) * 2) : 0u;
      }
    }
    return fine;
  }

  // Two adjacent output features of row (half ? g+8 : g): values and the first
  // feature index.  J is even; jj selects which pair.
  __device__ __forceinline__ void pair_at(int J, int jj, int half, int tig, float& a, float& b, int& d) const {
    if constexpr (FP8) {
      // (even tile, odd tile) at element jj are adjacent features
      a = O[J][2 * half + jj];
      b = O[J + 1][2 * half + jj];
      d = d_of<D, FP8>(J, jj, tig);
    } else {
      a = O[J + jj][2 * half];
      b = O[J + jj][2 * half + 1];
      d = d_of<D, FP8>(J + jj, 0, tig);
    }
  }
};

// P V for NP pages; MASK zeroes value rows at or past the sequence end.
template <int D, bool FP8, int NP, bool MASK>
__device__ __forceinline__ void pv_pages(ConsumerState<D, FP8>& cs, const uint32_t (&vb)[NP],
                                         const uint32_t (&Pa)[NP][4], uint32_t block_stride,
                                         const uint32_t (&mb0)[NP], const uint32_t (&mb1)[NP], int lane) {
  const int mi = lane >> 3, rr = lane & 7;
  if constexpr (FP8) {
#pragma unroll
    for (int c = 0; c < D / 16; c += 2) {
#pragma unroll
      for (int pg = 0; pg < NP; ++pg) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(vb[pg] + tile_off<D, FP8>(rr + 8 * (mi & 1), c + (mi >> 1), block_stride), r0, r1, r2, r3);
        const uint32_t u0 = prmt(r0, 0u, 0x3120u), u1 = prmt(r1, 0u, 0x3120u);
        const uint32_t u2 = prmt(r2, 0u, 0x3120u), u3 = prmt(r3, 0u, 0x3120u);
        uint32_t b[8] = {e4m3x2_to_f16x2(u0), e4m3x2_to_f16x2(u1), e4m3x2_to_f16x2(u0 >> 16),
                         e4m3x2_to_f16x2(u1 >> 16), e4m3x2_to_f16x2(u2), e4m3x2_to_f16x2(u3),
                         e4m3x2_to_f16x2(u2 >> 16), e4m3x2_to_f16x2(u3 >> 16)};
        if constexpr (MASK) {
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            b[e] &= mb0[pg];
            b[e + 1] &= mb1[pg];
          }
        }
        mma_f16(cs.O[2 * c], Pa[pg], b[0], b[1]);
        mma_f16(cs.O[2 * c + 1], Pa[pg], b[2], b[3]);
        mma_f16(cs.O[2 * c + 2], Pa[pg], b[4], b[5]);
        mma_f16(cs.O[2 * c + 3], Pa[pg], b[6], b[7]);
      }
    }
  } else {
#pragma unroll
    for (int J = 0; J < Geo<D, FP8>::NT; J += 2) {
#pragma unroll
      for (int pg = 0; pg < NP; ++pg) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(vb[pg] + tile_off<D, FP8>(rr + 8 * (mi & 1), J + (mi >> 1), block_stride), r0, r1, r2, r3);
        if constexpr (MASK) {
          r0 &= mb0[pg];
          r1 &= mb1[pg];
          r2 &= mb0[pg];
          r3 &= mb1[pg];
        }
        mma_bf16(cs.O[J], Pa[pg], r0, r1);
        mma_bf16(cs.O[J + 1], Pa[pg], r2, r3);
      }
    }
  }
}

// One block of NP consecutive pages of a segment for one warp: S = Q K^T,
// causal / tail mask by token index, online softmax (exp2 domain), O += P V.
// hb[pg] is the shared-memory address of this warp's head in the page's stage;
// V follows K at +kv_bytes.  tb = first token of the block; min_lim = L - qn.
// TOKS: per-token scales; ts[pg] is the shared-memory address of this warp's
// head's 16 K scales in page pg's stage, its 16 V scales tok_bytes further.
template <int D, bool FP8, int NP, bool TOKS = false>
__device__ __forceinline__ void consume_pages(ConsumerState<D, FP8>& cs, const uint32_t (&hb)[NP], uint32_t kv_bytes,
                                              uint32_t block_stride, int tb, int L, int min_lim, int lim0, int lim1,
                                              int window, float scale_log2, int lane, const uint32_t (&ts)[NP],
                                              uint32_t tok_bytes) {
  using GG = Geo<D, FP8>;
  const int tig = lane & 3, mi = lane >> 3, rr = lane & 7;
  float S[2 * NP][4];
#pragma unroll
  for (int n = 0; n < 2 * NP; ++n) S[n][0] = S[n][1] = S[n][2] = S[n][3] = 0.f;
  if constexpr (FP8) {
#pragma unroll
    for (int ks = 0; ks < GG::KS; ks += 2) {
#pragma unroll
      for (int pg = 0; pg < NP; ++pg) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(hb[pg] + tile_off<D, FP8>(rr + 8 * (mi & 1), ks + (mi >> 1), block_stride), r0, r1, r2, r3);
        mma_f16(S[2 * pg], cs.Qf[ks], e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r0 >> 16));
        mma_f16(S[2 * pg + 1], cs.Qf[ks], e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r1 >> 16));
        mma_f16(S[2 * pg], cs.Qf[ks + 1], e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r2 >> 16));
        mma_f16(S[2 * pg + 1], cs.Qf[ks + 1], e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r3 >> 16));
      }
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < GG::KS; ++ks) {
#pragma unroll
      for (int pg = 0; pg < NP; ++pg) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(hb[pg] + tile_off<D, FP8>(rr + 8 * (mi >> 1), 2 * ks + (mi & 1), block_stride), r0, r1, r2, r3);
        mma_bf16(S[2 * pg], cs.Qf[ks], r0, r1);
        mma_bf16(S[2 * pg + 1], cs.Qf[ks], r2, r3);
      }
    }
  }
  float x[2 * NP][4];
  // fp8 caches (whose consumers are issue-bound): with a positive scale and no
  // per-key scales the maximum is taken over the raw scores and the scale is
  // folded into the exponent's FMA, and the softmax arithmetic runs on packed
  // f32x2 pairs.  bf16 caches keep scalar arithmetic (there the packed form
  // costs registers and measured slower).
  constexpr bool kPacked = FP8;
  const bool fold = kPacked && !TOKS && scale_log2 > 0.f;
  if constexpr (TOKS) {
    // key token 8n + 2*tig + e of the block: the logit takes that key's scale
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
#pragma unroll
      for (int h8 = 0; h8 < 2; ++h8) {
        const float2 ks = lds_f2(ts[pg] + 32u * h8 + 8u * tig);
        const uint64_t c2 = f2_pack(scale_log2 * ks.x, scale_log2 * ks.y);
        const int n = 2 * pg + h8;
        f2_unpack(fmul2(f2_pack(S[n][0], S[n][1]), c2), x[n][0], x[n][1]);
        f2_unpack(fmul2(f2_pack(S[n][2], S[n][3]), c2), x[n][2], x[n][3]);
      }
    }
  } else if (fold) {
#pragma unroll
    for (int n = 0; n < 2 * NP; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[n][e] = S[n][e];
  } else {
#pragma unroll
    for (int n = 0; n < 2 * NP; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[n][e] = S[n][e] * scale_log2;
  }
  const float csc = fold ? scale_log2 : 1.f;   // scale still to apply in the exponent
  // keys allowed for a row: lim - W < token <= lim (causal run end; sliding
  // window start when W > 0, whose largest start is L - W for the last row)
  if (tb + kPage * NP - 1 > min_lim || (window > 0 && tb < L - window)) {
    const int lo0 = window > 0 ? lim0 - window + 1 : INT_MIN;
    const int lo1 = window > 0 ? lim1 - window + 1 : INT_MIN;
#pragma unroll
    for (int n = 0; n < 2 * NP; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = tb + 8 * n + 2 * tig + e;
        if (tok > lim0 || tok < lo0) x[n][e] = -INFINITY;
        if (tok > lim1 || tok < lo1) x[n][2 + e] = -INFINITY;
      }
  }
  float mx0 = fmaxf(x[0][0], x[0][1]);
  float mx1 = fmaxf(x[0][2], x[0][3]);
#pragma unroll
  for (int n = 1; n < 2 * NP; ++n) {
    if constexpr (kPacked) {
      mx0 = fmax3(mx0, x[n][0], x[n][1]);
      mx1 = fmax3(mx1, x[n][2], x[n][3]);
    } else {
      mx0 = fmaxf(mx0, fmaxf(x[n][0], x[n][1]));
      mx1 = fmaxf(mx1, fmaxf(x[n][2], x[n][3]));
    }
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  mx0 *= csc;
  mx1 *= csc;
  const float mn0 = fmaxf(cs.m0, mx0);
  const float mn1 = fmaxf(cs.m1, mx1);
  const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
  const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
  const float a0 = fast_exp2(cs.m0 - base0);
  const float a1 = fast_exp2(cs.m1 - base1);
  cs.m0 = mn0;
  cs.m1 = mn1;
  if constexpr (!kPacked) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int n = 0; n < 2 * NP; ++n) {
      x[n][0] = fast_exp2(x[n][0] - base0);
      x[n][1] = fast_exp2(x[n][1] - base0);
      x[n][2] = fast_exp2(x[n][2] - base1);
      x[n][3] = fast_exp2(x[n][3] - base1);
      s0 += x[n][0] + x[n][1];
      s1 += x[n][2] + x[n][3];
    }
    cs.l0 = cs.l0 * a0 + s0;
    cs.l1 = cs.l1 * a1 + s1;
    if (__any_sync(0xffffffffu, (a0 != 1.f) || (a1 != 1.f))) {
#pragma unroll
      for (int J = 0; J < GG::NT; ++J) {
        cs.O[J][0] *= a0;
        cs.O[J][1] *= a0;
        cs.O[J][2] *= a1;
        cs.O[J][3] *= a1;
      }
    }
  } else {
  // exponent arguments, exponentials' row sums and the O rescale as packed
  // pairs (the mma accumulator quads hold row g's two columns, then row g+8's)
  const uint64_t csc2 = f2_pack(csc, csc);
  const uint64_t nb0 = f2_pack(-base0, -base0), nb1 = f2_pack(-base1, -base1);
  uint64_t s0p = f2_pack(0.f, 0.f), s1p = s0p;
#pragma unroll
  for (int n = 0; n < 2 * NP; ++n) {
    f2_unpack(ffma2(f2_pack(x[n][0], x[n][1]), csc2, nb0), x[n][0], x[n][1]);
    f2_unpack(ffma2(f2_pack(x[n][2], x[n][3]), csc2, nb1), x[n][2], x[n][3]);
#pragma unroll
    for (int e = 0; e < 4; ++e) x[n][e] = fast_exp2(x[n][e]);
    s0p = fadd2(s0p, f2_pack(x[n][0], x[n][1]));
    s1p = fadd2(s1p, f2_pack(x[n][2], x[n][3]));
  }
  {
    float u0, u1, v0, v1;
    f2_unpack(s0p, u0, u1);
    f2_unpack(s1p, v0, v1);
    cs.l0 = cs.l0 * a0 + (u0 + u1);
    cs.l1 = cs.l1 * a1 + (v0 + v1);
  }
  if (__any_sync(0xffffffffu, (a0 != 1.f) || (a1 != 1.f))) {
    const uint64_t a00 = f2_pack(a0, a0), a11 = f2_pack(a1, a1);
#pragma unroll
    for (int J = 0; J < GG::NT; ++J) {
      f2_unpack(fmul2(f2_pack(cs.O[J][0], cs.O[J][1]), a00), cs.O[J][0], cs.O[J][1]);
      f2_unpack(fmul2(f2_pack(cs.O[J][2], cs.O[J][3]), a11), cs.O[J][2], cs.O[J][3]);
    }
  }
  }
  if constexpr (TOKS) {
    // P V with per-token value scales: each weight takes its value row's scale
    // (the sum l above keeps the unscaled weights).  Slots past the sequence
    // end take 0, so a non-finite scale there cannot reach O.
    const bool tail = L - tb < kPage * NP;
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const int vt = L - tb - kPage * pg;   // value rows of this page inside the sequence
#pragma unroll
      for (int h8 = 0; h8 < 2; ++h8) {
        const float2 vs = lds_f2(ts[pg] + tok_bytes + 32u * h8 + 8u * tig);
        const int t0 = 8 * h8 + 2 * tig;
        float c0 = vs.x, c1 = vs.y;
        if (tail) {
          c0 = t0 < vt ? c0 : 0.f;
          c1 = t0 + 1 < vt ? c1 : 0.f;
        }
        const uint64_t c2 = f2_pack(c0, c1);
        const int n = 2 * pg + h8;
        f2_unpack(fmul2(f2_pack(x[n][0], x[n][1]), c2), x[n][0], x[n][1]);
        f2_unpack(fmul2(f2_pack(x[n][2], x[n][3]), c2), x[n][2], x[n][3]);
      }
    }
  }
  uint32_t Pa[NP][4];
#pragma unroll
  for (int pg = 0; pg < NP; ++pg) {
    if constexpr (FP8) {
      Pa[pg][0] = pack_f16(x[2 * pg][0], x[2 * pg][1]);
      Pa[pg][1] = pack_f16(x[2 * pg][2], x[2 * pg][3]);
      Pa[pg][2] = pack_f16(x[2 * pg + 1][0], x[2 * pg + 1][1]);
      Pa[pg][3] = pack_f16(x[2 * pg + 1][2], x[2 * pg + 1][3]);
    } else {
      Pa[pg][0] = pack_bf16(x[2 * pg][0], x[2 * pg][1]);
      Pa[pg][1] = pack_bf16(x[2 * pg][2], x[2 * pg][3]);
      Pa[pg][2] = pack_bf16(x[2 * pg + 1][0], x[2 * pg + 1][1]);
      Pa[pg][3] = pack_bf16(x[2 * pg + 1][2], x[2 * pg + 1][3]);
    }
  }
  uint32_t vb[NP];
#pragma unroll
  for (int pg = 0; pg < NP; ++pg) vb[pg] = hb[pg] + kv_bytes;
  // Value rows at or past the end of the sequence are zeroed so that stale
  // (even non-finite) tail slots cannot leak through P == 0.
  if (L - tb < kPage * NP) {
    uint32_t mb0[NP], mb1[NP];
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const int vt = L - tb - kPage * pg;
      mb0[pg] = (2 * tig < vt ? 0x0000ffffu : 0u) | (2 * tig + 1 < vt ? 0xffff0000u : 0u);
      mb1[pg] = (2 * tig + 8 < vt ? 0x0000ffffu : 0u) | (2 * tig + 9 < vt ? 0xffff0000u : 0u);
    }
    pv_pages<D, FP8, NP, true>(cs, vb, Pa, block_stride, mb0, mb1, lane);
  } else {
    const uint32_t none[NP] = {};
    pv_pages<D, FP8, NP, false>(cs, vb, Pa, block_stride, none, none, lane);
  }
}

// WINDOW: the sliding-window variant (a separate instantiation, so the
// windowless kernels carry none of its code).  TOKS: fp8 caches with per-token
// scales, staged by the producer behind each page's K and V tiles.
template <int D, bool FP8, bool WINDOW, bool TOKS = false>
__global__ void __launch_bounds__(kSplitMaxThreads, 1)
    pa_split_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                    const SplitParams p) {
  using GG = Geo<D, FP8>;
  const int window = WINDOW ? p.window : 0;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_scan[kSplitMaxThreads / 32 + 1];
  __shared__ int s_total;

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  int32_t* const s_pre = reinterpret_cast<int32_t*>(gbase + p.off_prefix);
  int32_t* const s_len = s_pre + (p.num_seqs + 1);
  int32_t* const s_qsl = s_len + p.num_seqs;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int B = p.num_seqs;
  if (tid == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  // Inputs may come from the previous kernel in the stream (programmatic
  // dependent launch): nothing global is read before this point.
  // The pipeline barriers live in shared memory only, so they are set up
  // while the previous kernel may still be running.
  const uint32_t bar0 = base + p.off_bar;
  const int nstage = p.nstage;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (nstage + s); };
  auto qfull_bar = [&](int s) { return bar0 + 8u * (2 * nstage + s); };
  auto qempty_bar = [&](int s) { return bar0 + 8u * (2 * nstage + 2 + s); };
  const int ncw = p.HC * p.MT;   // consumer warps
  if (tid == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), ncw);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(qfull_bar(s), 1);
      mbar_init(qempty_bar(s), ncw);
    }
    fence_mbar_init();
  }

  grid_dependency_wait();

  // ---- prologue: metadata to shared memory, pages per sequence, prefix -----
  page_prefix(p, window, s_pre, s_len, s_qsl, s_scan, &s_total);
  __syncthreads();   // the prefix totals and the mbarrier initialisation above

  const int64_t X = static_cast<int64_t>(p.NC) * s_pre[B];
  int64_t ng64 = (X + p.min_pages - 1) / p.min_pages;
  if (ng64 < 1) ng64 = 1;
  const int NG = static_cast<int>(ng64 < gridDim.x ? ng64 : gridDim.x);
  grid_launch_dependents();

  const int g = blockIdx.x;
  if (g >= NG || X == 0) return;
  const int64_t start = static_cast<int64_t>(g) * X / NG;
  const int64_t end = static_cast<int64_t>(g + 1) * X / NG;
  const int64_t count = end - start;
  if (count <= 0) return;

  const int HC = p.HC, G = p.G, NC = p.NC;
  const uint32_t qrow_bytes = static_cast<uint32_t>(HC * G * D * 2);   // one query token, HC heads

  if (warp == 0) {
    // ============================ producer =================================
    if (g == p.starve_cta) return;   // testing aid: this CTA's pages never arrive
    Cursor cu = locate(s_pre, B, NC, start);
    int qseg = 0;
    BlockTableCache btc;
    const uint32_t block_stride = static_cast<uint32_t>(HC * GG::BOX_BYTES);
    int stage = 0;
    uint32_t round = 0;    // k / nstage
    for (int64_t k = 0; k < count; ++k) {
      if (round > 0) {
        if (!mbar_wait(empty_bar(stage), (round - 1) & 1u, p.wait_ns)) {
          if (lane == 0) atomicOr(p.err, kErrTimeout);
          break;
        }
      }
      if (k == 0 || cu.j == 0) {
        const int qs = qseg & 1;
        if (qseg >= 2) {
          if (!mbar_wait(qempty_bar(qs), static_cast<uint32_t>((qseg >> 1) - 1) & 1u, p.wait_ns)) {
            if (lane == 0) atomicOr(p.err, kErrTimeout);
            break;
          }
        }
        const SeqInfo si = seq_info(p, s_len, s_qsl, cu.i, false, window);
        if (lane == 0) mbar_arrive_expect_tx(qfull_bar(qs), static_cast<uint32_t>(si.qn) * qrow_bytes);
        __syncwarp();
        const uint32_t qdst = base + p.off_q + static_cast<uint32_t>(qs) * p.q_slot_bytes;
        for (int r = lane; r < si.qn; r += 32) {
          const uint16_t* src = p.q + static_cast<int64_t>(si.t0 + r) * p.q_stride_t +
                                static_cast<int64_t>(cu.c) * HC * G * D;
          bulk_load(qdst + static_cast<uint32_t>(r) * qrow_bytes, src, qrow_bytes, qfull_bar(qs));
        }
        ++qseg;
      }
      const int phys = btc.lookup(p, cu, s_pre, s_len, s_qsl, B, NC, window, lane);
      const bool bad_page = phys < 0 || phys >= p.num_pages;
      if (bad_page && lane == 0) atomicOr(p.err, kErrPageRange);
      // An out-of-range page id reads as zeros (TMA fills outside the tensor).
      if constexpr (TOKS) {
        if (lane == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * p.kv_bytes + 2 * p.tok_bytes);
        __syncwarp();
        if (lane >= 30) {
          // the page's [HC][16] K (lane 30) or V (lane 31) scales; an
          // out-of-range page id reads page 0's (its rows are undefined anyway)
          const float* src = (lane == 30 ? p.k_tok : p.v_tok) +
                             static_cast<int64_t>(bad_page ? 0 : phys) * p.tok_stride_page + cu.c * HC * kPage;
          const uint32_t dst = base + p.off_stage + static_cast<uint32_t>(stage) * p.stage_bytes + 2 * p.kv_bytes +
                               static_cast<uint32_t>(lane - 30) * p.tok_bytes;
          bulk_load(dst, src, p.tok_bytes, full_bar(stage));
        }
      } else {
        if (lane == 0) mbar_arrive_expect_tx(full_bar(stage), p.stage_bytes);
        __syncwarp();
      }
      if (lane < 2 * GG::NBOX) {
        const int tensor = lane / GG::NBOX;
        const int bx = lane - tensor * GG::NBOX;
        const uint32_t dst = base + p.off_stage + static_cast<uint32_t>(stage) * p.stage_bytes +
                             static_cast<uint32_t>(tensor) * p.kv_bytes + static_cast<uint32_t>(bx) * block_stride;
        // box: RB bytes of the row x 16 slots x HC heads, starting at head c*HC of page phys
        tma_load_4d(dst, tensor ? &tmap_v : &tmap_k, bx * (GG::RB / GG::ESZ), 0, cu.c * HC, phys, full_bar(stage));
      }
      advance(cu, s_pre, B, NC);
      if (++stage == nstage) {
        stage = 0;
        ++round;
      }
    }
    return;
  }

  // ============================== consumers ================================
  const int cw = warp - 1;
  if (cw >= ncw) return;
  const int hh = cw / p.MT;         // KV head within the chunk
  const int w = cw - hh * p.MT;     // 16-row tile
  const int gq = lane >> 2;         // fragment row group
  const int tig = lane & 3;         // thread in group
  const int rho0 = 16 * w + gq;
  const int rho1 = rho0 + 8;
  const uint32_t block_stride = static_cast<uint32_t>(HC * GG::BOX_BYTES);
  const uint32_t head_base = base + p.off_stage + static_cast<uint32_t>(hh * GG::BOX_BYTES);
  // per-token scales of this warp's head in stage 0 (TOKS only)
  const uint32_t tok_base = base + p.off_stage + 2 * p.kv_bytes + static_cast<uint32_t>(hh * kPage * 4);

  Cursor cu = locate(s_pre, B, NC, start);
  int qseg = 0;
  int64_t seg_k0 = 0;
  int seg_j0 = 0;
  SeqInfo si = {0, 0, 0};
  bool active = false, ok0 = false, ok1 = false;
  int lim0 = 0, lim1 = 0;
  ConsumerState<D, FP8> cs;
  cs.reset();
#pragma unroll
  for (int ks = 0; ks < GG::KS; ++ks) cs.Qf[ks][0] = cs.Qf[ks][1] = cs.Qf[ks][2] = cs.Qf[ks][3] = 0u;

  int stage = 0;
  uint32_t round = 0;              // k / nstage for the page at `stage`
  int64_t k = 0;
  while (k < count) {
    if (!mbar_wait(full_bar(stage), round & 1u, p.wait_ns)) {
      if (lane == 0) atomicOr(p.err, kErrTimeout);
      break;
    }
    if (k == 0 || cu.j == 0) {
      // ---- new segment: query rows into registers, state reset ----
      si = seq_info(p, s_len, s_qsl, cu.i, lane == 0 && hh == 0 && w == 0, window);
      seg_k0 = k;
      seg_j0 = cu.j;
      const int qs = qseg & 1;
      if (!mbar_wait(qfull_bar(qs), static_cast<uint32_t>(qseg >> 1) & 1u, p.wait_ns)) {
        if (lane == 0) atomicOr(p.err, kErrTimeout);
        break;
      }
      if (seg_j0 == 0 && cw == 0 && lane == 0) {
        // This CTA holds the unit's first page: describe the unit for the merge.
        const int64_t a = static_cast<int64_t>(NC) * s_pre[cu.i] + static_cast<int64_t>(cu.c) * cu.n;
        const int last_cta = static_cast<int>(((a + cu.n) * NG - 1) / X);
        const int pieces = last_cta - g + 1;
        p.ws_unit[static_cast<int64_t>(cu.i) * NC + cu.c] =
            make_int4(g, pieces | (k != 0 ? (1 << 30) : 0), si.t0, si.qn);
      }
      const int R = G * si.qn;
      active = 16 * w < R;
      ok0 = rho0 < R;
      ok1 = rho1 < R;
      lim0 = si.L - si.qn + (ok0 ? rho0 / G : 0);
      lim1 = si.L - si.qn + (ok1 ? rho1 / G : 0);
      const uint8_t* qslot = gbase + p.off_q + qs * p.q_slot_bytes;
      const uint8_t* q0p = qslot + static_cast<size_t>(((rho0 / G) * HC + hh) * G + rho0 % G) * (D * 2);
      const uint8_t* q1p = qslot + static_cast<size_t>(((rho1 / G) * HC + hh) * G + rho1 % G) * (D * 2);
      if (!cs.load_query(q0p, q1p, ok0, ok1, tig)) atomicOr(p.err, kErrF16Range);
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty_bar(qs));
      ++qseg;
      cs.reset();
      if (p.sinks != nullptr && seg_j0 == 0) {
        // The sink is a virtual first key with logit sinks[hq] and a zero value
        // row: the piece holding the unit's first page starts from it, so every
        // row counts it exactly once (the merge needs no special case).
        const int hq_base = (cu.c * HC + hh) * G;
        if (ok0) {
          cs.m0 = p.sinks[hq_base + rho0 % G] * 1.4426950408889634f;
          cs.l0 = tig == 0 ? 1.f : 0.f;
        }
        if (ok1) {
          cs.m1 = p.sinks[hq_base + rho1 % G] * 1.4426950408889634f;
          cs.l1 = tig == 0 ? 1.f : 0.f;
        }
      }
    }
    // Two consecutive pages of the same segment are processed together when
    // the ring is deep enough (32-token blocks: more independent MMA chains,
    // one softmax reduction per 32 tokens).
    int stage2 = stage + 1;
    uint32_t round2 = round;
    if (stage2 == nstage) {
      stage2 = 0;
      ++round2;
    }
    const bool pair = p.pair_pages && (k + 1 < count) && (cu.j + 1 < cu.n);
    if (pair && !mbar_wait(full_bar(stage2), round2 & 1u, p.wait_ns)) {
      if (lane == 0) atomicOr(p.err, kErrTimeout);
      break;
    }
    const int tb = kPage * (si.js + cu.j);
    if (active) {
      if (pair) {
        const uint32_t hb[2] = {head_base + static_cast<uint32_t>(stage) * p.stage_bytes,
                                head_base + static_cast<uint32_t>(stage2) * p.stage_bytes};
        const uint32_t ts[2] = {tok_base + static_cast<uint32_t>(stage) * p.stage_bytes,
                                tok_base + static_cast<uint32_t>(stage2) * p.stage_bytes};
        consume_pages<D, FP8, 2, TOKS>(cs, hb, p.kv_bytes, block_stride, tb, si.L, si.L - si.qn, lim0, lim1, window,
                                       p.scale_log2, lane, ts, p.tok_bytes);
      } else {
        const uint32_t hb[1] = {head_base + static_cast<uint32_t>(stage) * p.stage_bytes};
        const uint32_t ts[1] = {tok_base + static_cast<uint32_t>(stage) * p.stage_bytes};
        consume_pages<D, FP8, 1, TOKS>(cs, hb, p.kv_bytes, block_stride, tb, si.L, si.L - si.qn, lim0, lim1, window,
                                       p.scale_log2, lane, ts, p.tok_bytes);
      }
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(empty_bar(stage));
      if (pair) mbar_arrive(empty_bar(stage2));
    }
    const int np = pair ? 2 : 1;
    const int j_last = cu.j + np - 1;
    const bool seg_last = (k + np == count) || (j_last == cu.n - 1);
    if (seg_last && active) {
      const bool complete = (seg_j0 == 0) && (j_last == cu.n - 1);
      float lt0 = cs.l0 + __shfl_xor_sync(0xffffffffu, cs.l0, 1);
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
      float lt1 = cs.l1 + __shfl_xor_sync(0xffffffffu, cs.l1, 1);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
      if (complete) {
        const int hq_base = (cu.c * HC + hh) * G;
        const float inv0 = lt0 > 0.f ? p.v_scale / lt0 : 0.f;
        const float inv1 = lt1 > 0.f ? p.v_scale / lt1 : 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const bool ok = half ? ok1 : ok0;
          if (!ok) continue;
          const int rho = half ? rho1 : rho0;
          const float inv = half ? inv1 : inv0;
          const int t = si.t0 + rho / G;
          const int hq = hq_base + rho % G;
          uint16_t* orow = p.out + static_cast<int64_t>(t) * p.out_stride_t + static_cast<int64_t>(hq) * p.out_stride_h;
#pragma unroll
          for (int J = 0; J < GG::NT; J += 2) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              float va, vb2;
              int d;
              cs.pair_at(J, jj, half, tig, va, vb2, d);
              *reinterpret_cast<uint32_t*>(orow + d) = pack_bf16(va * inv, vb2 * inv);
            }
          }
          if (p.lse != nullptr && tig == 0) {
            const float lt = half ? lt1 : lt0;
            const float mm = half ? cs.m1 : cs.m0;
            p.lse[static_cast<int64_t>(t) * p.lse_stride_t + static_cast<int64_t>(hq) * p.lse_stride_h] =
                lt > 0.f ? (mm + fast_log2(lt)) * 0.69314718055994530942f : -INFINITY;
          }
        }
      } else {
        const int which = (seg_k0 == 0) ? 0 : 1;
        const int64_t rowbase = (static_cast<int64_t>(2 * g + which) * HC + hh) * p.R_max;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const bool ok = half ? ok1 : ok0;
          if (!ok) continue;
          const int rho = half ? rho1 : rho0;
          float* orow = p.ws_o + (rowbase + rho) * D;
#pragma unroll
          for (int J = 0; J < GG::NT; J += 2) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              float va, vb2;
              int d;
              cs.pair_at(J, jj, half, tig, va, vb2, d);
              *reinterpret_cast<float2*>(orow + d) = make_float2(va, vb2);
            }
          }
          if (tig == 0) p.ws_ml[rowbase + rho] = make_float2(half ? cs.m1 : cs.m0, half ? lt1 : lt0);
        }
      }
    }
    for (int t = 0; t < np; ++t) {
      advance(cu, s_pre, B, NC);
      if (++stage == nstage) {
        stage = 0;
        ++round;
      }
    }
    k += np;
  }
}

}  // namespace pa
