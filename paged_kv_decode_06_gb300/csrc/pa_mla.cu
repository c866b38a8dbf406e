// Multi-head latent attention (MLA) decode over a paged latent cache (sm_103a).
//
// What it computes (ATOM model-operations guide, "Multi-head latent attention
// (attention_mla.py)", decode flow step 2: mla_decode_fwd over the rows that
// fused_qk_rope_concat_and_cache_mla wrote): every cached token is one row
// C_j = [c_kv (512) | k_pe (64)] that all query heads share; a query row is as
// wide (the absorbed no-position part, then the rotary part), so
//   s_j = scale * <q, C_j>,   out = sum_j softmax(s)_j C_j[0:512],   lse = ln sum_j e^{s_j}.
//
// Work decomposition: that of the grouped-query split kernel (units
// (sequence, chunk of query heads) laid end to end in page order, every
// worker a contiguous page range, cut units leaving partials for the LSE
// merge: the normalised output in f16 with the fp32 running max and sum), with
// "worker" = team: a CTA holds one or two independent teams, each one producer
// warp and 4 * RT consumer warps (RT = 16-row tiles of a chunk, at most 2),
// with its own ring, query slot and barriers.
//
// The value part of a row is 512 wide, too wide for one warp's accumulator
// (16 rows x 512 fp32 = 256 registers a lane), so the four consumer warps of a
// row tile split the columns: warp quarter cq owns value columns
// [128 cq, 128 cq + 128) and Q K^T features [144 cq, 144 cq + 144).  Per step
// (one page, or two consecutive pages of a segment) each warp computes its
// partial 16-row score tile with mma.sync, the four partials meet in shared
// memory behind an mbarrier (four arrivals, bounded wait), every warp sums them
// in the same order (so all four hold identical scores, maxima and sums), runs
// the online softmax and accumulates P V for its own columns.
//
// Ring stage = one page: the whole [16, 576] row block in one TMA box
// (64 features x 16 slots x 9 column blocks), which lands as 9 blocks of 16
// swizzled rows (128-byte rows for bf16, 64-byte rows for fp8).  The value
// operand is the first 8 column blocks of the same stage: a cached row is read
// from HBM once.  fp8 codes are converted to f16 in registers (exact), with the
// query in f16; kv_scale is folded into the logit scale and the output.
// Every wait is bounded (kErrTimeout).
#include "pa_pack.cuh"
#include "pa_split.cuh"

namespace pa {

constexpr int kMlaDqk = 576;
constexpr int kMlaDv = 512;
constexpr int kMlaBoxes = kMlaDqk / 64;   // 64-feature column blocks of a row
constexpr int kMlaKs = 9;                 // 16-feature k-steps of Q K^T per column quarter

template <bool FP8>
struct MlaGeo {
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int RB = 64 * ESZ;               // bytes of a 64-feature box row (swizzle span)
  static constexpr int CPB = RB / 16;               // 16-byte chunks per box row
  static constexpr int BOX = 16 * RB;               // one column block of a page
  static constexpr uint32_t STAGE = kMlaBoxes * BOX;
};

template <int RT>
struct MlaTeams {
  static constexpr int NTEAM = RT == 1 ? 2 : 1;
  static constexpr int WARPS = 1 + 4 * RT;          // per team
  static constexpr int THREADS = NTEAM * 32 * WARPS;
};

// Byte offset of 16-byte chunk `chunk` (counted along the whole row) of row
// `row` inside a stage.
template <bool FP8>
__device__ __forceinline__ uint32_t mla_off(int row, int chunk) {
  using GG = MlaGeo<FP8>;
  return static_cast<uint32_t>(chunk / GG::CPB) * GG::BOX + swz<GG::RB>(row, chunk % GG::CPB);
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void sts_f4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

__device__ __forceinline__ void lds_u64x2(uint32_t addr, uint64_t& a, uint64_t& b) {
  asm volatile("ld.shared.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr) : "memory");
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// Online-softmax state of one consumer warp: 16 query rows, value columns
// [128 cq, 128 cq + 128).
template <bool FP8>
struct MlaWarp {
  float O[16][4];        // mma C fragments of 16 n-tiles
  uint32_t Qf[kMlaKs][4];  // A fragments of this quarter's 144 query features
  float m0, m1, l0, l1;  // running max (log2 units) and this lane's share of the sum, rows g and g + 8

  __device__ __forceinline__ void reset() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int J = 0; J < 16; ++J) O[J][0] = O[J][1] = O[J][2] = O[J][3] = 0.f;
  }

  // Query rows (bf16 in shared memory, row stride 576 elements) into A
  // fragments for k-steps 9 cq .. 9 cq + 8.  fp8: f16 values in the feature
  // order of the fp8 key fragments (k = 2 tig + {0,1} holds d = 16 ks + 4 tig
  // + {0,1}, k = 2 tig + 8 + {0,1} holds d + 2).  Returns false if a value
  // overflowed f16.
  __device__ __forceinline__ bool load_query(const uint8_t* q0p, const uint8_t* q1p, bool ok0, bool ok1, int cq,
                                             int tig) {
    bool fine = true;
#pragma unroll
    for (int kk = 0; kk < kMlaKs; ++kk) {
      const int ks = kMlaKs * cq + kk;
      if constexpr (FP8) {
        const uint2 a = ok0 ? *reinterpret_cast<const uint2*>(q0p + (16 * ks + 4 * tig) * 2) : make_uint2(0u, 0u);
        const uint2 b = ok1 ? *reinterpret_cast<const uint2*>(q1p + (16 * ks + 4 * tig) * 2) : make_uint2(0u, 0u);
        Qf[kk][0] = pack_f16(bf16_lo(a.x), bf16_hi(a.x));
        Qf[kk][1] = pack_f16(bf16_lo(b.x), bf16_hi(b.x));
        Qf[kk][2] = pack_f16(bf16_lo(a.y), bf16_hi(a.y));
        Qf[kk][3] = pack_f16(bf16_lo(b.y), bf16_hi(b.y));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t v = Qf[kk][e];
          fine &= ((v & 0x7C00u) != 0x7C00u) && ((v & 0x7C000000u) != 0x7C000000u);
        }
      } else {
        Qf[kk][0] = ok0 ? *reinterpret_cast<const uint32_t*>(q0p + (16 * ks + 2 * tig) * 2) : 0u;
        Qf[kk][1] = ok1 ? *reinterpret_cast<const uint32_t*>(q1p + (16 * ks + 2 * tig) * 2) : 0u;
        Qf[kk][2] = ok0 ? *reinterpret_cast<const uint32_t*>(q0p + (16 * ks + 8 + 2 * tig) * 2) : 0u;
        Qf[kk][3] = ok1 ? *reinterpret_cast<const uint32_t*>(q1p + (16 * ks + 8 + 2 * tig) * 2) : 0u;
      }
    }
    return fine;
  }

  // Two adjacent value columns (relative to the quarter) of row (half ? g+8 : g).
  __device__ __forceinline__ void pair_at(int J, int jj, int half, int tig, float& a, float& b, int& d) const {
    if constexpr (FP8) {
      a = O[J][2 * half + jj];
      b = O[J + 1][2 * half + jj];
      d = 16 * (J >> 1) + 4 * tig + 2 * jj;
    } else {
      a = O[J + jj][2 * half];
      b = O[J + jj][2 * half + 1];
      d = 8 * (J + jj) + 2 * tig;
    }
  }
};

// NP consecutive pages of a segment for one consumer warp.  st[pg]: page
// pg's stage; xbuf: this step's exchange buffer of the row tile (4 quarters x
// NP KB) and xbar / xpar its mbarrier (4 arrivals) and phase parity; tb: first
// token of the first page; lim0 / lim1: last key rows g / g+8 may see.
// Returns false if the exchange wait timed out.
template <bool FP8, int NP>
__device__ __forceinline__ bool mla_pages(MlaWarp<FP8>& ws, const uint32_t (&st)[NP], uint32_t xbuf, uint32_t xbar,
                                          uint32_t xpar, int cq, int tb, int L, int min_lim, int lim0, int lim1,
                                          float scale_log2, int lane, uint64_t wait_ns) {
  const int tig = lane & 3, mi = lane >> 3, rr = lane & 7;
  // ---- partial scores over this quarter's 144 features ----
  float S[2 * NP][4];
#pragma unroll
  for (int n = 0; n < 2 * NP; ++n) S[n][0] = S[n][1] = S[n][2] = S[n][3] = 0.f;
  if constexpr (FP8) {
#pragma unroll
    for (int kk = 0; kk < kMlaKs - 1; kk += 2) {
      const int ks = kMlaKs * cq + kk;
#pragma unroll
      for (int pg = 0; pg < NP; ++pg) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(st[pg] + mla_off<FP8>(rr + 8 * (mi & 1), ks + (mi >> 1)), r0, r1, r2, r3);
        mma_f16(S[2 * pg], ws.Qf[kk], e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r0 >> 16));
        mma_f16(S[2 * pg + 1], ws.Qf[kk], e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r1 >> 16));
        mma_f16(S[2 * pg], ws.Qf[kk + 1], e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r2 >> 16));
        mma_f16(S[2 * pg + 1], ws.Qf[kk + 1], e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r3 >> 16));
      }
    }
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      uint32_t r0, r1;   // the quarter's ninth k-step: keys 0-7 and 8-15 of one 16-feature chunk
      ldsm_x2(st[pg] + mla_off<FP8>(rr + 8 * (mi & 1), kMlaKs * cq + kMlaKs - 1), r0, r1);
      mma_f16(S[2 * pg], ws.Qf[kMlaKs - 1], e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r0 >> 16));
      mma_f16(S[2 * pg + 1], ws.Qf[kMlaKs - 1], e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r1 >> 16));
    }
  } else {
#pragma unroll
    for (int kk = 0; kk < kMlaKs; ++kk) {
      const int ks = kMlaKs * cq + kk;
#pragma unroll
      for (int pg = 0; pg < NP; ++pg) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(st[pg] + mla_off<FP8>(rr + 8 * (mi >> 1), 2 * ks + (mi & 1)), r0, r1, r2, r3);
        mma_bf16(S[2 * pg], ws.Qf[kk], r0, r1);
        mma_bf16(S[2 * pg + 1], ws.Qf[kk], r2, r3);
      }
    }
  }
  // ---- the four quarters' partials meet in shared memory ----
  const uint32_t mine = xbuf + static_cast<uint32_t>(cq) * (1024u * NP) + 16u * lane;
#pragma unroll
  for (int n = 0; n < 2 * NP; ++n) sts_f4(mine + 512u * n, S[n][0], S[n][1], S[n][2], S[n][3]);
  __syncwarp();
  if (lane == 0) mbar_arrive(xbar);
  if (!mbar_wait(xbar, xpar, wait_ns)) return false;
  // sums of the four partials as packed pairs (row g's two columns, row g+8's)
  uint64_t X[2 * NP][2];
#pragma unroll
  for (int n = 0; n < 2 * NP; ++n) lds_u64x2(xbuf + 512u * n + 16u * lane, X[n][0], X[n][1]);
#pragma unroll
  for (int q = 1; q < 4; ++q) {   // same order in every quarter: identical sums
#pragma unroll
    for (int n = 0; n < 2 * NP; ++n) {
      uint64_t a, b;
      lds_u64x2(xbuf + q * (1024u * NP) + 512u * n + 16u * lane, a, b);
      X[n][0] = fadd2(X[n][0], a);
      X[n][1] = fadd2(X[n][1], b);
    }
  }
  float x[2 * NP][4];
#pragma unroll
  for (int n = 0; n < 2 * NP; ++n) {
    f2_unpack(X[n][0], x[n][0], x[n][1]);
    f2_unpack(X[n][1], x[n][2], x[n][3]);
  }
  // With a positive scale the maximum is taken over the raw scores and the
  // scale is folded into the exponent's FMA; otherwise the scores are scaled first.
  const bool fold = scale_log2 > 0.f;
  if (!fold) {
#pragma unroll
    for (int n = 0; n < 2 * NP; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[n][e] *= scale_log2;
  }
  const float cs = fold ? scale_log2 : 1.f;
  // ---- causal run / context tail mask ----
  if (tb + kPage * NP - 1 > min_lim) {
#pragma unroll
    for (int n = 0; n < 2 * NP; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = tb + 8 * n + 2 * tig + e;
        if (tok > lim0) x[n][e] = -INFINITY;
        if (tok > lim1) x[n][2 + e] = -INFINITY;
      }
  }
  // ---- online softmax (exp2 domain) ----
  float mx0 = fmaxf(x[0][0], x[0][1]);
  float mx1 = fmaxf(x[0][2], x[0][3]);
#pragma unroll
  for (int n = 1; n < 2 * NP; ++n) {
    mx0 = fmax3(mx0, x[n][0], x[n][1]);
    mx1 = fmax3(mx1, x[n][2], x[n][3]);
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  mx0 *= cs;
  mx1 *= cs;
  const float mn0 = fmaxf(ws.m0, mx0);
  const float mn1 = fmaxf(ws.m1, mx1);
  const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
  const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
  const float a0 = fast_exp2(ws.m0 - base0);
  const float a1 = fast_exp2(ws.m1 - base1);
  ws.m0 = mn0;
  ws.m1 = mn1;
  const uint64_t cs2 = f2_pack(cs, cs);
  const uint64_t nb0 = f2_pack(-base0, -base0), nb1 = f2_pack(-base1, -base1);
  uint64_t s0 = f2_pack(0.f, 0.f), s1 = s0;
#pragma unroll
  for (int n = 0; n < 2 * NP; ++n) {
    f2_unpack(ffma2(f2_pack(x[n][0], x[n][1]), cs2, nb0), x[n][0], x[n][1]);
    f2_unpack(ffma2(f2_pack(x[n][2], x[n][3]), cs2, nb1), x[n][2], x[n][3]);
#pragma unroll
    for (int e = 0; e < 4; ++e) x[n][e] = fast_exp2(x[n][e]);
    s0 = fadd2(s0, f2_pack(x[n][0], x[n][1]));
    s1 = fadd2(s1, f2_pack(x[n][2], x[n][3]));
  }
  float s0a, s0b, s1a, s1b;
  f2_unpack(s0, s0a, s0b);
  f2_unpack(s1, s1a, s1b);
  ws.l0 = ws.l0 * a0 + (s0a + s0b);
  ws.l1 = ws.l1 * a1 + (s1a + s1b);
  if (__any_sync(0xffffffffu, (a0 != 1.f) || (a1 != 1.f))) {
#pragma unroll
    for (int J = 0; J < 16; ++J) {
      ws.O[J][0] *= a0;
      ws.O[J][1] *= a0;
      ws.O[J][2] *= a1;
      ws.O[J][3] *= a1;
    }
  }
  // ---- P V over this quarter's 128 value columns; rows at or past the
  // sequence end are zeroed (stale, even non-finite, tail slots) ----
#pragma unroll
  for (int pg = 0; pg < NP; ++pg) {
    uint32_t Pa[4];
    if constexpr (FP8) {
      Pa[0] = pack_f16(x[2 * pg][0], x[2 * pg][1]);
      Pa[1] = pack_f16(x[2 * pg][2], x[2 * pg][3]);
      Pa[2] = pack_f16(x[2 * pg + 1][0], x[2 * pg + 1][1]);
      Pa[3] = pack_f16(x[2 * pg + 1][2], x[2 * pg + 1][3]);
    } else {
      Pa[0] = pack_bf16(x[2 * pg][0], x[2 * pg][1]);
      Pa[1] = pack_bf16(x[2 * pg][2], x[2 * pg][3]);
      Pa[2] = pack_bf16(x[2 * pg + 1][0], x[2 * pg + 1][1]);
      Pa[3] = pack_bf16(x[2 * pg + 1][2], x[2 * pg + 1][3]);
    }
    const int vt = L - tb - kPage * pg;
    const bool tail = vt < kPage;
    const uint32_t mb0 = (2 * tig < vt ? 0x0000ffffu : 0u) | (2 * tig + 1 < vt ? 0xffff0000u : 0u);
    const uint32_t mb1 = (2 * tig + 8 < vt ? 0x0000ffffu : 0u) | (2 * tig + 9 < vt ? 0xffff0000u : 0u);
    if constexpr (FP8) {
#pragma unroll
      for (int c = 0; c < 8; c += 2) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(st[pg] + mla_off<FP8>(rr + 8 * (mi & 1), 8 * cq + c + (mi >> 1)), r0, r1, r2, r3);
        const uint32_t u0 = prmt(r0, 0u, 0x3120u), u1 = prmt(r1, 0u, 0x3120u);
        const uint32_t u2 = prmt(r2, 0u, 0x3120u), u3 = prmt(r3, 0u, 0x3120u);
        uint32_t b[8] = {e4m3x2_to_f16x2(u0), e4m3x2_to_f16x2(u1), e4m3x2_to_f16x2(u0 >> 16),
                         e4m3x2_to_f16x2(u1 >> 16), e4m3x2_to_f16x2(u2), e4m3x2_to_f16x2(u3),
                         e4m3x2_to_f16x2(u2 >> 16), e4m3x2_to_f16x2(u3 >> 16)};
        if (tail) {
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            b[e] &= mb0;
            b[e + 1] &= mb1;
          }
        }
        mma_f16(ws.O[2 * c], Pa, b[0], b[1]);
        mma_f16(ws.O[2 * c + 1], Pa, b[2], b[3]);
        mma_f16(ws.O[2 * c + 2], Pa, b[4], b[5]);
        mma_f16(ws.O[2 * c + 3], Pa, b[6], b[7]);
      }
    } else {
#pragma unroll
      for (int J = 0; J < 16; J += 2) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(st[pg] + mla_off<FP8>(rr + 8 * (mi & 1), 16 * cq + J + (mi >> 1)), r0, r1, r2, r3);
        if (tail) {
          r0 &= mb0;
          r1 &= mb1;
          r2 &= mb0;
          r3 &= mb1;
        }
        mma_bf16(ws.O[J], Pa, r0, r1);
        mma_bf16(ws.O[J + 1], Pa, r2, r3);
      }
    }
  }
  return true;
}

// Team layout in shared memory, from the team's base (team t at
// base + t * team_bytes): ring stages at off_stage, q_slots query slots at off_q,
// exchange buffers at off_xchg (2 steps x RT row tiles x 4 quarters x 2 KB),
// barriers at off_bar (full[nstage], empty[nstage], qfull[2], qempty[2],
// xfull[2][RT]: the exchange of step parity b of row tile rt).  The
// sequence metadata (page prefix, lengths, query starts) is shared by the CTA
// at off_prefix.
template <bool FP8, int RT>
__global__ void __launch_bounds__(MlaTeams<RT>::THREADS, 1)
    pa_mla_kernel(const __grid_constant__ CUtensorMap tmap, const SplitParams p) {
  using GG = MlaGeo<FP8>;
  using TT = MlaTeams<RT>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_scan[33];
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
  const int team = warp / TT::WARPS;
  const int wt = warp - team * TT::WARPS;          // warp within the team: 0 producer, 1.. consumers
  const int B = p.num_seqs;
  const uint32_t tbase = base + static_cast<uint32_t>(team) * p.team_bytes;
  const uint8_t* const tgbase = gbase + static_cast<size_t>(team) * p.team_bytes;
  const int nstage = p.nstage;
  const uint32_t bar0 = tbase + p.off_bar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (nstage + s); };
  auto qfull_bar = [&](int s) { return bar0 + 8u * (2 * nstage + s); };
  auto qempty_bar = [&](int s) { return bar0 + 8u * (2 * nstage + 2 + s); };
  auto xfull_bar = [&](int b, int r) { return bar0 + 8u * (2 * nstage + 4 + b * RT + r); };
  constexpr int ncw = 4 * RT;
  if (tid == 0) prefetch_tensormap(&tmap);
  if (wt == 0 && lane == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), ncw);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(qfull_bar(s), 1);
      mbar_init(qempty_bar(s), ncw);
      for (int r = 0; r < RT; ++r) mbar_init(xfull_bar(s, r), 4);
    }
    fence_mbar_init();
  }
  // Inputs may come from the previous kernel in the stream (programmatic
  // dependent launch): nothing global is read before this point.
  grid_dependency_wait();
  page_prefix(p, 0, s_pre, s_len, s_qsl, s_scan, &s_total);
  __syncthreads();   // prefix totals and the barrier initialisation above

  const int NC = p.NC, G = p.G;
  const int64_t X = static_cast<int64_t>(NC) * s_pre[B];
  int64_t ng64 = (X + p.min_pages - 1) / p.min_pages;
  if (ng64 < 1) ng64 = 1;
  const int64_t nworkers = static_cast<int64_t>(gridDim.x) * TT::NTEAM;
  const int NG = static_cast<int>(ng64 < nworkers ? ng64 : nworkers);
  grid_launch_dependents();

  // worker g: team-major, so that with fewer ranges than teams every SM gets one
  const int g = team * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
  if (g >= NG || X == 0) return;
  const int64_t start = static_cast<int64_t>(g) * X / NG;
  const int64_t end = static_cast<int64_t>(g + 1) * X / NG;
  const int count = static_cast<int>(end - start);   // pages of this worker (X / NG < 2^31)
  if (count <= 0) return;
  const uint32_t qrow_bytes = static_cast<uint32_t>(G * kMlaDqk * 2);   // one query token of a head chunk

  if (wt == 0) {
    // ============================ producer =================================
    Cursor cu = locate(s_pre, B, NC, start);
    int qseg = 0;
    BlockTableCache btc;
    int stage = 0;
    uint32_t round = 0;
    for (int k = 0; k < count; ++k) {
      if (round > 0) {
        if (!mbar_wait(empty_bar(stage), (round - 1) & 1u, p.wait_ns)) {
          if (lane == 0) atomicOr(p.err, kErrTimeout);
          break;
        }
      }
      if (k == 0 || cu.j == 0) {
        const int qs = qseg % p.q_slots;
        if (qseg >= p.q_slots) {
          if (!mbar_wait(qempty_bar(qs), static_cast<uint32_t>(qseg / p.q_slots - 1) & 1u, p.wait_ns)) {
            if (lane == 0) atomicOr(p.err, kErrTimeout);
            break;
          }
        }
        const SeqInfo si = seq_info(p, s_len, s_qsl, cu.i, false, 0);
        if (lane == 0) mbar_arrive_expect_tx(qfull_bar(qs), static_cast<uint32_t>(si.qn) * qrow_bytes);
        __syncwarp();
        const uint32_t qdst = tbase + p.off_q + static_cast<uint32_t>(qs) * p.q_slot_bytes;
        for (int r = lane; r < si.qn; r += 32) {
          const uint16_t* src = p.q + static_cast<int64_t>(si.t0 + r) * p.q_stride_t +
                                static_cast<int64_t>(cu.c) * G * kMlaDqk;
          bulk_load(qdst + static_cast<uint32_t>(r) * qrow_bytes, src, qrow_bytes, qfull_bar(qs));
        }
        ++qseg;
      }
      const int phys = btc.lookup(p, cu, s_pre, s_len, s_qsl, B, NC, 0, lane);
      if (lane == 0) {
        if (phys < 0 || phys >= p.num_pages) atomicOr(p.err, kErrPageRange);
        // the page's 16 rows, all 576 features: an out-of-range page id reads zeros
        mbar_arrive_expect_tx(full_bar(stage), GG::STAGE);
        tma_load_4d(tbase + p.off_stage + static_cast<uint32_t>(stage) * GG::STAGE, &tmap, 0, 0, 0, phys,
                    full_bar(stage));
      }
      __syncwarp();
      advance(cu, s_pre, B, NC);
      if (++stage == nstage) {
        stage = 0;
        ++round;
      }
    }
    return;
  }

  // ============================== consumers ================================
  // g, NG and X are needed only at segment boundaries: recomputed there from
  // shared memory and launch constants instead of staying live in registers.
  auto worker = [&]() { return team * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x); };
  auto total_pages = [&]() { return static_cast<int64_t>(p.NC) * s_pre[p.num_seqs]; };
  auto workers = [&](int64_t x) {
    int64_t n = (x + p.min_pages - 1) / p.min_pages;
    if (n < 1) n = 1;
    const int64_t nw = static_cast<int64_t>(gridDim.x) * TT::NTEAM;
    return static_cast<int>(n < nw ? n : nw);
  };
  const int cw = wt - 1;
  const int rt = cw >> 2;            // 16-row tile
  const int cq = cw & 3;             // column quarter
  const int gq = lane >> 2;
  const int tig = lane & 3;
  const int rho0 = 16 * rt + gq;
  const int rho1 = rho0 + 8;
  const uint32_t xbase = tbase + p.off_xchg + static_cast<uint32_t>(rt) * 8192u;

  Cursor cu = locate(s_pre, B, NC, start);
  int qseg = 0;
  bool seg_first_page = false;      // the segment starts at this worker's first page
  int seg_j0 = 0;
  SeqInfo si = {0, 0, 0, 0};
  bool active = false, ok0 = false, ok1 = false;
  int lim0 = 0, lim1 = 0;
  uint32_t step = 0;                 // exchange-buffer parity
  MlaWarp<FP8> ws;
  ws.reset();

  int stage = 0;
  uint32_t round = 0;
  int k = 0;
  while (k < count) {
    if (!mbar_wait(full_bar(stage), round & 1u, p.wait_ns)) {
      if (lane == 0) atomicOr(p.err, kErrTimeout);
      break;
    }
    if (k == 0 || cu.j == 0) {
      // ---- new segment: query rows into registers, state reset ----
      si = seq_info(p, s_len, s_qsl, cu.i, lane == 0 && cw == 0, 0);
      seg_first_page = k == 0;
      seg_j0 = cu.j;
      const int qs = qseg % p.q_slots;
      if (!mbar_wait(qfull_bar(qs), static_cast<uint32_t>(qseg / p.q_slots) & 1u, p.wait_ns)) {
        if (lane == 0) atomicOr(p.err, kErrTimeout);
        break;
      }
      if (seg_j0 == 0 && cw == 0 && lane == 0) {
        // This worker holds the unit's first page: describe the unit for the merge.
        const int64_t xt = total_pages();
        const int gw = worker();
        const int64_t a = static_cast<int64_t>(p.NC) * s_pre[cu.i] + static_cast<int64_t>(cu.c) * cu.n;
        const int last = static_cast<int>(((a + cu.n) * workers(xt) - 1) / xt);
        p.ws_unit[static_cast<int64_t>(cu.i) * p.NC + cu.c] =
            make_int4(gw, (last - gw + 1) | (k != 0 ? (1 << 30) : 0), si.t0, si.qn);
      }
      const int R = G * si.qn;
      active = 16 * rt < R;
      ok0 = rho0 < R;
      ok1 = rho1 < R;
      lim0 = si.L - si.qn + (ok0 ? rho0 / G : 0);
      lim1 = si.L - si.qn + (ok1 ? rho1 / G : 0);
      const uint8_t* qslot = tgbase + p.off_q + qs * p.q_slot_bytes;
      if (!ws.load_query(qslot + static_cast<size_t>(rho0) * (kMlaDqk * 2),
                         qslot + static_cast<size_t>(rho1) * (kMlaDqk * 2), ok0, ok1, cq, tig))
        atomicOr(p.err, kErrF16Range);
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty_bar(qs));
      ++qseg;
      ws.reset();
    }
    // Two consecutive pages of the segment are taken together when the ring
    // is deep enough (one exchange and one softmax reduction per 32 keys).
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
    const int tb = kPage * cu.j;
    if (active) {
      // exchange buffer b = step parity is used for the (step >> 1)-th time
      const int b = static_cast<int>(step & 1u);
      const uint32_t xb = xbase + static_cast<uint32_t>(b * RT) * 8192u;
      const uint32_t s0 = tbase + p.off_stage + static_cast<uint32_t>(stage) * GG::STAGE;
      bool ok;
      if (pair) {
        const uint32_t sts[2] = {s0, tbase + p.off_stage + static_cast<uint32_t>(stage2) * GG::STAGE};
        ok = mla_pages<FP8, 2>(ws, sts, xb, xfull_bar(b, rt), (step >> 1) & 1u, cq, tb, si.L, si.L - si.qn, lim0,
                               lim1, p.scale_log2, lane, p.wait_ns);
      } else {
        const uint32_t sts[1] = {s0};
        ok = mla_pages<FP8, 1>(ws, sts, xb, xfull_bar(b, rt), (step >> 1) & 1u, cq, tb, si.L, si.L - si.qn, lim0,
                               lim1, p.scale_log2, lane, p.wait_ns);
      }
      if (!ok) {
        if (lane == 0) atomicOr(p.err, kErrTimeout);
        break;
      }
      ++step;
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
      float lt0 = ws.l0 + __shfl_xor_sync(0xffffffffu, ws.l0, 1);
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
      float lt1 = ws.l1 + __shfl_xor_sync(0xffffffffu, ws.l1, 1);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
      if (complete) {
        const float inv0 = lt0 > 0.f ? p.v_scale / lt0 : 0.f;
        const float inv1 = lt1 > 0.f ? p.v_scale / lt1 : 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const bool ok = half ? ok1 : ok0;
          if (!ok) continue;
          const int rho = half ? rho1 : rho0;
          const float inv = half ? inv1 : inv0;
          const int t = si.t0 + rho / G;
          const int hq = cu.c * G + rho % G;
          uint16_t* orow = p.out + static_cast<int64_t>(t) * p.out_stride_t + static_cast<int64_t>(hq) * p.out_stride_h +
                           128 * cq;
#pragma unroll
          for (int J = 0; J < 16; J += 2) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              float va, vb;
              int d;
              ws.pair_at(J, jj, half, tig, va, vb, d);
              *reinterpret_cast<uint32_t*>(orow + d) = pack_bf16(va * inv, vb * inv);
            }
          }
          if (p.lse != nullptr && cq == 0 && tig == 0) {
            const float lt = half ? lt1 : lt0;
            const float mm = half ? ws.m1 : ws.m0;
            p.lse[static_cast<int64_t>(t) * p.lse_stride_t + static_cast<int64_t>(hq) * p.lse_stride_h] =
                lt > 0.f ? (mm + fast_log2(lt)) * 0.69314718055994530942f : -INFINITY;
          }
        }
      } else {
        const int which = seg_first_page ? 0 : 1;
        const int64_t rowbase = static_cast<int64_t>(2 * worker() + which) * p.R_max;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const bool ok = half ? ok1 : ok0;
          if (!ok) continue;
          const int rho = half ? rho1 : rho0;
          // the piece's normalised output O / l in f16 (a weighted average of
          // cached rows, 2^-11 relative error); the merge weighs it back with
          // l and reports a value beyond the f16 range (|v| > 65504, possible
          // only in a bf16 cache) as kErrF16Range.
          const float lt = half ? lt1 : lt0;
          const float inv = lt > 0.f ? 1.f / lt : 0.f;
          uint16_t* orow = reinterpret_cast<uint16_t*>(p.ws_o) + (rowbase + rho) * kMlaDv + 128 * cq;
#pragma unroll
          for (int J = 0; J < 16; J += 2) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              float va, vb;
              int d;
              ws.pair_at(J, jj, half, tig, va, vb, d);
              *reinterpret_cast<uint32_t*>(orow + d) = pack_f16(va * inv, vb * inv);
            }
          }
          if (cq == 0 && tig == 0) p.ws_ml[rowbase + rho] = make_float2(half ? ws.m1 : ws.m0, half ? lt1 : lt0);
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

template <bool FP8, int RT>
static cudaError_t launch_one(const CUtensorMap& tm, const SplitParams& p, int grid, int smem, bool pdl,
                              cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(MlaTeams<RT>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, pa_mla_kernel<FP8, RT>, tm, p);
}

int mla_threads(int rt) { return rt == 1 ? MlaTeams<1>::THREADS : MlaTeams<2>::THREADS; }
int mla_teams(int rt) { return rt == 1 ? MlaTeams<1>::NTEAM : MlaTeams<2>::NTEAM; }

cudaError_t launch_mla(bool fp8, int rt, const CUtensorMap& tm, const SplitParams& p, int grid, int smem, bool pdl,
                       cudaStream_t stream) {
  if (rt == 1) return fp8 ? launch_one<true, 1>(tm, p, grid, smem, pdl, stream)
                          : launch_one<false, 1>(tm, p, grid, smem, pdl, stream);
  if (rt == 2) return fp8 ? launch_one<true, 2>(tm, p, grid, smem, pdl, stream)
                          : launch_one<false, 2>(tm, p, grid, smem, pdl, stream);
  return cudaErrorInvalidValue;
}

cudaError_t set_mla_smem_limits(int smem) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(pa_mla_kernel<false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(pa_mla_kernel<false, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(pa_mla_kernel<true, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(pa_mla_kernel<true, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace pa
