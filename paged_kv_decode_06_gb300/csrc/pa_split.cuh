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

#include "pa_device.cuh"
#include "pa_kernels.h"

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
};

// Sequence metadata from the shared-memory copies made in the prologue.
__device__ __forceinline__ SeqInfo seq_info(const SplitParams& p, const int32_t* s_len, const int32_t* s_qsl, int i,
                                            bool report) {
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

template <int D, bool FP8>
__global__ void __launch_bounds__(kSplitMaxThreads, 1)
    pa_split_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                    const SplitParams p) {
  using GG = Geo<D, FP8>;
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
  const int nwarps = blockDim.x >> 5;
  const int B = p.num_seqs;
  if (tid == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  // Inputs may come from the previous kernel in the stream (programmatic
  // dependent launch): nothing global is read before this point.
  grid_dependency_wait();

  // ---- prologue: metadata to shared memory, pages per sequence, prefix -----
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
      if (lane == 31) s_total = xs;
    }
    __syncthreads();
    if (i < B) s_pre[i] = carry + s_scan[warp] + x - v;
    carry += s_total;
    __syncthreads();
  }
  if (tid == 0) {
    s_pre[B] = carry;
    s_qsl[B] = p.qsl != nullptr ? p.qsl[B] : B;
  }

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
  __syncthreads();

  const int64_t X = static_cast<int64_t>(p.NC) * s_pre[B];
  int64_t ng64 = (X + p.min_pages - 1) / p.min_pages;
  if (ng64 < 1) ng64 = 1;
  const int NG = static_cast<int>(ng64 < gridDim.x ? ng64 : gridDim.x);
  if (blockIdx.x == 0) {
    if (tid == 0) {
      p.ws_meta[0] = X;
      p.ws_meta[1] = NG;
    }
    for (int i = tid; i <= B; i += blockDim.x) p.ws_prefix[i] = s_pre[i];
  }
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
    Cursor cu = locate(s_pre, B, NC, start);
    int qseg = 0;
    int bt_i = -1, bt_j0 = 0, bt_val = 0;   // block-table entries [bt_j0, bt_j0 + 32) of sequence bt_i
    int nx_i = -1, nx_j0 = 0, nx_val = 0;   // the batch after it, loaded ahead of use
    const uint32_t block_stride = static_cast<uint32_t>(HC * GG::BOX_BYTES);
    for (int64_t k = 0; k < count; ++k) {
      const int stage = static_cast<int>(k % nstage);
      if (k >= nstage) {
        if (!mbar_wait(empty_bar(stage), static_cast<uint32_t>((k / nstage) - 1) & 1u)) {
          if (lane == 0) atomicOr(p.err, kErrTimeout);
          break;
        }
      }
      if (k == 0 || cu.j == 0) {
        const int qs = qseg & 1;
        if (qseg >= 2) {
          if (!mbar_wait(qempty_bar(qs), static_cast<uint32_t>((qseg >> 1) - 1) & 1u)) {
            if (lane == 0) atomicOr(p.err, kErrTimeout);
            break;
          }
        }
        const SeqInfo si = seq_info(p, s_len, s_qsl, cu.i, false);
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
      if (cu.i != bt_i || cu.j < bt_j0 || cu.j >= bt_j0 + 32) {
        if (cu.i == nx_i && cu.j == nx_j0) {
          bt_val = nx_val;
        } else {
          const int jj = cu.j + lane;
          bt_val = (jj < cu.n) ? p.block_tables[static_cast<int64_t>(cu.i) * p.bt_stride + jj] : 0;
        }
        bt_i = cu.i;
        bt_j0 = cu.j;
        // prefetch the batch the traversal reaches next
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
          nx_val = (jj < pages_of(s_pre, ni)) ? p.block_tables[static_cast<int64_t>(ni) * p.bt_stride + jj] : 0;
        }
      }
      const int phys = __shfl_sync(0xffffffffu, bt_val, cu.j - bt_j0);
      if ((phys < 0 || phys >= p.num_pages) && lane == 0) atomicOr(p.err, kErrPageRange);
      // An out-of-range page id reads as zeros (TMA fills outside the tensor).
      if (lane == 0) mbar_arrive_expect_tx(full_bar(stage), p.stage_bytes);
      __syncwarp();
      if (lane < 2 * GG::NBOX) {
        const int tensor = lane / GG::NBOX;
        const int bx = lane - tensor * GG::NBOX;
        const uint32_t dst = base + p.off_stage + static_cast<uint32_t>(stage) * p.stage_bytes +
                             static_cast<uint32_t>(tensor) * p.kv_bytes + static_cast<uint32_t>(bx) * block_stride;
        // box: RB bytes of the row x 16 slots x HC heads, starting at head c*HC of page phys
        tma_load_4d(dst, tensor ? &tmap_v : &tmap_k, bx * (GG::RB / GG::ESZ), 0, cu.c * HC, phys, full_bar(stage));
      }
      advance(cu, s_pre, B, NC);
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
  const int mi = lane >> 3;         // ldmatrix matrix index
  const int rr = lane & 7;          // ldmatrix row
  const int rho0 = 16 * w + gq;
  const int rho1 = rho0 + 8;
  const uint32_t block_stride = static_cast<uint32_t>(HC * GG::BOX_BYTES);

  Cursor cu = locate(s_pre, B, NC, start);
  int qseg = 0;
  int64_t seg_k0 = 0;
  int seg_j0 = 0;
  SeqInfo si = {0, 0, 0};
  bool active = false, ok0 = false, ok1 = false;
  int lim0 = 0, lim1 = 0;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float O[GG::NT][4];
  uint32_t Qf[GG::KS][4];
#pragma unroll
  for (int J = 0; J < GG::NT; ++J) O[J][0] = O[J][1] = O[J][2] = O[J][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < GG::KS; ++ks) Qf[ks][0] = Qf[ks][1] = Qf[ks][2] = Qf[ks][3] = 0u;

  for (int64_t k = 0; k < count; ++k) {
    const int stage = static_cast<int>(k % nstage);
    if (!mbar_wait(full_bar(stage), static_cast<uint32_t>(k / nstage) & 1u)) {
      if (lane == 0) atomicOr(p.err, kErrTimeout);
      break;
    }
    if (k == 0 || cu.j == 0) {
      // ---- new segment: query rows into registers, state reset ----
      si = seq_info(p, s_len, s_qsl, cu.i, lane == 0 && hh == 0 && w == 0);
      seg_k0 = k;
      seg_j0 = cu.j;
      const int qs = qseg & 1;
      if (!mbar_wait(qfull_bar(qs), static_cast<uint32_t>(qseg >> 1) & 1u)) {
        if (lane == 0) atomicOr(p.err, kErrTimeout);
        break;
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
      bool f16_overflow = false;
#pragma unroll
      for (int ks = 0; ks < GG::KS; ++ks) {
        if constexpr (FP8) {
          // d-order inside a k-step matches the fp8 K fragments: k = 2*tig + {0,1}
          // holds d = 16*ks + 4*tig + {0,1}; k = 2*tig + 8 + {0,1} holds d + 2.
          uint2 a = ok0 ? *reinterpret_cast<const uint2*>(q0p + (16 * ks + 4 * tig) * 2) : make_uint2(0u, 0u);
          uint2 b = ok1 ? *reinterpret_cast<const uint2*>(q1p + (16 * ks + 4 * tig) * 2) : make_uint2(0u, 0u);
          Qf[ks][0] = pack_f16(bf16_lo(a.x), bf16_hi(a.x));
          Qf[ks][1] = pack_f16(bf16_lo(b.x), bf16_hi(b.x));
          Qf[ks][2] = pack_f16(bf16_lo(a.y), bf16_hi(a.y));
          Qf[ks][3] = pack_f16(bf16_lo(b.y), bf16_hi(b.y));
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t v = Qf[ks][e];
            f16_overflow |= ((v & 0x7C00u) == 0x7C00u) || ((v & 0x7C000000u) == 0x7C000000u);
          }
        } else {
          Qf[ks][0] = ok0 ? *reinterpret_cast<const uint32_t*>(q0p + (16 * ks + 2 * tig) * 2) : 0u;
          Qf[ks][1] = ok1 ? *reinterpret_cast<const uint32_t*>(q1p + (16 * ks + 2 * tig) * 2) : 0u;
          Qf[ks][2] = ok0 ? *reinterpret_cast<const uint32_t*>(q0p + (16 * ks + 8 + 2 * tig) * 2) : 0u;
          Qf[ks][3] = ok1 ? *reinterpret_cast<const uint32_t*>(q1p + (16 * ks + 8 + 2 * tig) * 2) : 0u;
        }
      }
      if (FP8 && f16_overflow) atomicOr(p.err, kErrF16Range);
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty_bar(qs));
      ++qseg;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
#pragma unroll
      for (int J = 0; J < GG::NT; ++J) O[J][0] = O[J][1] = O[J][2] = O[J][3] = 0.f;
    }

    if (active) {
      const uint32_t kb = base + p.off_stage + static_cast<uint32_t>(stage) * p.stage_bytes +
                          static_cast<uint32_t>(hh * GG::BOX_BYTES);
      const uint32_t vb = kb + p.kv_bytes;
      // ---- S = Q K^T for the 16 tokens of this page ----
      float S[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if constexpr (FP8) {
#pragma unroll
        for (int ks = 0; ks < GG::KS; ks += 2) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(kb + tile_off<D, FP8>(rr + 8 * (mi & 1), ks + (mi >> 1), block_stride), r0, r1, r2, r3);
          mma_f16(S[0], Qf[ks], e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r0 >> 16));
          mma_f16(S[1], Qf[ks], e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r1 >> 16));
          mma_f16(S[0], Qf[ks + 1], e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r2 >> 16));
          mma_f16(S[1], Qf[ks + 1], e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r3 >> 16));
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < GG::KS; ++ks) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(kb + tile_off<D, FP8>(rr + 8 * (mi >> 1), 2 * ks + (mi & 1), block_stride), r0, r1, r2, r3);
          mma_bf16(S[0], Qf[ks], r0, r1);
          mma_bf16(S[1], Qf[ks], r2, r3);
        }
      }
      // ---- mask, online softmax (exp2 domain) ----
      const int tb = kPage * cu.j;
      float x[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[nt][e] = S[nt][e] * p.scale_log2;
      if (tb + kPage - 1 > si.L - si.qn) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int tok = tb + 8 * nt + 2 * tig + e;
            if (tok > lim0) x[nt][e] = -INFINITY;
            if (tok > lim1) x[nt][2 + e] = -INFINITY;
          }
      }
      float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
      float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0);
      const float mn1 = fmaxf(m1, mx1);
      const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float a0 = fast_exp2(m0 - base0);
      const float a1 = fast_exp2(m1 - base1);
      m0 = mn0;
      m1 = mn1;
      float pr[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        pr[nt][0] = fast_exp2(x[nt][0] - base0);
        pr[nt][1] = fast_exp2(x[nt][1] - base0);
        pr[nt][2] = fast_exp2(x[nt][2] - base1);
        pr[nt][3] = fast_exp2(x[nt][3] - base1);
      }
      l0 = l0 * a0 + ((pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
      l1 = l1 * a1 + ((pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]));
      if (__any_sync(0xffffffffu, (a0 != 1.f) || (a1 != 1.f))) {
#pragma unroll
        for (int J = 0; J < GG::NT; ++J) {
          O[J][0] *= a0;
          O[J][1] *= a0;
          O[J][2] *= a1;
          O[J][3] *= a1;
        }
      }
      uint32_t Pa[4];
      if constexpr (FP8) {
        Pa[0] = pack_f16(pr[0][0], pr[0][1]);
        Pa[1] = pack_f16(pr[0][2], pr[0][3]);
        Pa[2] = pack_f16(pr[1][0], pr[1][1]);
        Pa[3] = pack_f16(pr[1][2], pr[1][3]);
      } else {
        Pa[0] = pack_bf16(pr[0][0], pr[0][1]);
        Pa[1] = pack_bf16(pr[0][2], pr[0][3]);
        Pa[2] = pack_bf16(pr[1][0], pr[1][1]);
        Pa[3] = pack_bf16(pr[1][2], pr[1][3]);
      }
      // ---- O += P V; value rows past the sequence end are zeroed so that
      //      stale (even non-finite) tail slots cannot leak through P == 0 ----
      const int vt = si.L - tb;
      uint32_t mb0 = 0xffffffffu, mb1 = 0xffffffffu;
      if (vt < kPage) {
        mb0 = (2 * tig < vt ? 0x0000ffffu : 0u) | (2 * tig + 1 < vt ? 0xffff0000u : 0u);
        mb1 = (2 * tig + 8 < vt ? 0x0000ffffu : 0u) | (2 * tig + 9 < vt ? 0xffff0000u : 0u);
      }
      if constexpr (FP8) {
#pragma unroll
        for (int c = 0; c < D / 16; c += 2) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(vb + tile_off<D, FP8>(rr + 8 * (mi & 1), c + (mi >> 1), block_stride), r0, r1, r2, r3);
          const uint32_t u0 = prmt(r0, 0u, 0x3120u), u1 = prmt(r1, 0u, 0x3120u);
          const uint32_t u2 = prmt(r2, 0u, 0x3120u), u3 = prmt(r3, 0u, 0x3120u);
          mma_f16(O[2 * c], Pa, e4m3x2_to_f16x2(u0) & mb0, e4m3x2_to_f16x2(u1) & mb1);
          mma_f16(O[2 * c + 1], Pa, e4m3x2_to_f16x2(u0 >> 16) & mb0, e4m3x2_to_f16x2(u1 >> 16) & mb1);
          mma_f16(O[2 * c + 2], Pa, e4m3x2_to_f16x2(u2) & mb0, e4m3x2_to_f16x2(u3) & mb1);
          mma_f16(O[2 * c + 3], Pa, e4m3x2_to_f16x2(u2 >> 16) & mb0, e4m3x2_to_f16x2(u3 >> 16) & mb1);
        }
      } else {
#pragma unroll
        for (int J = 0; J < GG::NT; J += 2) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(vb + tile_off<D, FP8>(rr + 8 * (mi & 1), J + (mi >> 1), block_stride), r0, r1, r2, r3);
          mma_bf16(O[J], Pa, r0 & mb0, r1 & mb1);
          mma_bf16(O[J + 1], Pa, r2 & mb0, r3 & mb1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(stage));

    const bool seg_last = (k == count - 1) || (cu.j == cu.n - 1);
    if (seg_last && active) {
      float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
      float lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
      const bool complete = (seg_j0 == 0) && (cu.j == cu.n - 1);
      if (complete) {
        const float inv0 = lt0 > 0.f ? p.v_scale / lt0 : 0.f;
        const float inv1 = lt1 > 0.f ? p.v_scale / lt1 : 0.f;
        const int hq_base = (cu.c * HC + hh) * G;
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
              if constexpr (FP8) {
                // (even tile, odd tile) at element e are adjacent features
                const int e = jj;
                const float va = O[J][2 * half + e] * inv;
                const float vb2 = O[J + 1][2 * half + e] * inv;
                *reinterpret_cast<uint32_t*>(orow + d_of<D, FP8>(J, e, tig)) = pack_bf16(va, vb2);
              } else {
                const int Jt = J + jj;
                const float va = O[Jt][2 * half] * inv;
                const float vb2 = O[Jt][2 * half + 1] * inv;
                *reinterpret_cast<uint32_t*>(orow + d_of<D, FP8>(Jt, 0, tig)) = pack_bf16(va, vb2);
              }
            }
          }
          if (p.lse != nullptr && tig == 0) {
            const float lt = half ? lt1 : lt0;
            const float mm = half ? m1 : m0;
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
              if constexpr (FP8) {
                const int e = jj;
                *reinterpret_cast<float2*>(orow + d_of<D, FP8>(J, e, tig)) =
                    make_float2(O[J][2 * half + e], O[J + 1][2 * half + e]);
              } else {
                const int Jt = J + jj;
                *reinterpret_cast<float2*>(orow + d_of<D, FP8>(Jt, 0, tig)) =
                    make_float2(O[Jt][2 * half], O[Jt][2 * half + 1]);
              }
            }
          }
          if (tig == 0) p.ws_ml[rowbase + rho] = make_float2(half ? m1 : m0, half ? lt1 : lt0);
        }
      }
    }
    advance(cu, s_pre, B, NC);
  }
}

}  // namespace pa
