// Split-KV paged decode on the 5th-generation tensor cores (tcgen05 + TMEM),
// for long verification runs: up to 128 query rows per KV head (G query heads
// x up to 128/G tokens of a ragged MTP run), bf16 caches.
//
// Work decomposition, workspace and merge are those of the mma.sync split
// kernel with one KV head per CTA: units (sequence, KV head) laid end to end
// in (sequence, head, page) order, each CTA a contiguous page range, cut units
// leaving fp32 partials for the same merge kernel.  What changes is the math:
// with 65-128 rows per KV head, Q K^T and P V are dense 128 x 16n and
// 128 x D products, which the tensor cores run from shared memory into tensor
// memory while the CUDA cores do only the softmax.
//
// A block is up to block_pages (4) pages of one segment (a segment is the
// part of one unit inside this CTA's range); the shared-memory ring holds one
// block per stage: [K d0..63 | K d64..127 | V d0..63 | V d64..127], each
// part block_pages x 16 rows x 128 bytes, 128-byte swizzled as TMA writes it.
//
// Roles (384 threads):
//   warps 0-1 producers: block-table lookups and TMA loads of each page's K
//             and V rows into the block's stage, the block's 2 KB boxes dealt
//             one per lane over both warps (a warp's TMA issue is serial, about
//             90 ns per 2 KB box, so one warp alone could not keep HBM busy);
//   warp 3    Q K^T issuer (one lane) and owner of the TMEM allocation:
//               S[b%2]  = Q[s%2] K_b^T     (TS-MMA, Q read from TMEM, N = 16 * pages)
//   warp 2    P V issuer (one lane):
//               O      += P[b%2] V_b   (TS-MMA, P read from TMEM, N = D)
//             Two issuers, because one lane issues a tcgen05.mma every ~60
//             cycles at best and a single issuer interleaving both streams
//             (S of block b+1 between P V of blocks b-1 and b) set the pace;
//   warps 4-11 softmax, two groups of four: group g takes the blocks b with
//             b % 2 == g, so two blocks' softmax work overlaps; in a group,
//             thread = query row = TMEM lane and owns all of a block's keys,
//             with the group's own running max, sum and O accumulator.  Per
//             block: load S, mask (causal run, context tail, sliding window),
//             update the running max, rescale O in TMEM only when the max grew
//             by more than 2^8 (lazy rescale), write P over the block's S in
//             bf16 and keep two row sums: of the weights (for the lse and the
//             merge) and of the weights as rounded into P, which normalises O
//             (O divided by it is a weighted mean of V rows, so P's rounding
//             perturbs the weights without leaving their sum: a row dominated
//             by one key keeps that key's V row).  At a segment's end the two
//             threads of a row exchange (max, sum, rounded sum), each combines
//             half of the two O accumulators and writes out / lse or the
//             partials (O rescaled by sum / rounded sum, so the merge's
//             O / sum is the same weighted mean).  They also store each
//             segment's Q rows into one of two TMEM slots.
// TMEM columns: O_0 [0,128) O_1 [128,256) S/P of group 0 [256,320) and of
//               group 1 [320,384) (S fp32, 16 columns per page; bf16 P over it,
//               8 columns per page) Q0 [384,448) Q1 [448,512).
// Shared memory holds only the ring (6 stages of 4 pages at D = 128) and
// metadata: Q lives in TMEM, as the A operand of a TS-MMA.
// Every wait is bounded (kErrTimeout); the CTA drains its MMAs before it frees
// tensor memory.
//
// Parity waits: mbarrier.try_wait.parity cannot tell "the wanted phase has
// completed" from "the barrier is still one phase behind it" (the phase before
// has the same parity), so each wait below is made only when the waiter knows
// the barrier's previous phase is complete.  The per-group "P V done" barrier
// is the delicate one: Q K^T of block b is issued only after P V(b-2) is done,
// so a softmax group that has seen S(b) knows P V(b-2) is complete before it
// waits for P V(b) (segment end) or P V(b-2) (rescale); letting Q K^T run
// further ahead (three S/P buffers) breaks this and lets the segment-end wait
// pass while P V(b-2) is still accumulating.
#pragma once

#include "pa_pack.cuh"
#include "pa_split.cuh"

namespace pa {

// Maximum of v[0..N) by a tree of three-input maxima (about N/2 instructions
// instead of N - 1); v is overwritten.
template <int N>
struct Max3Tree {
  static __device__ __forceinline__ float run(float* v) {
    constexpr int M = (N + 2) / 3;
#pragma unroll
    for (int i = 0; i < M; ++i) {
      const int a = 3 * i;
      if (a + 2 < N) v[i] = fmax3(v[a], v[a + 1], v[a + 2]);
      else if (a + 1 < N) v[i] = fmaxf(v[a], v[a + 1]);
      else v[i] = v[a];
    }
    return Max3Tree<M>::run(v);
  }
};
template <>
struct Max3Tree<1> {
  static __device__ __forceinline__ float run(float* v) { return v[0]; }
};

constexpr int kTcProducers = 2;
constexpr int kTcPvWarp = 2;
constexpr int kTcMmaWarp = 3;
constexpr int kTcSoftmaxWarp0 = 4;   // warps 4..11; a multiple of 4, so warp % 4 is the TMEM lane quarter
constexpr int kTcSoftmaxWarps = 8;
constexpr int kTcThreads = 32 * (kTcSoftmaxWarp0 + kTcSoftmaxWarps);
constexpr int kTcMaxBlockPages = 4;
constexpr uint32_t kTcCols = 512;
constexpr uint32_t kTmemO = 0;     // + 128 * group: fp32 O of softmax group g, D columns
constexpr uint32_t kTmemSP = 256;  // + 64 * group: fp32 S of the group's block, 16 columns per page;
constexpr uint32_t kTmemPhi = 0;   //   P overwrites it: bf16 P at + 8 * page
constexpr uint32_t kTmemQ = 384;   // + 64 * (segment % 2): bf16 Q, D / 2 columns
constexpr uint32_t kTcBox = 2048;  // one page of one 64-column half: 16 rows x 128 bytes
constexpr uint32_t kTcHalf = kTcMaxBlockPages * kTcBox;   // one 64-column half of a stage's K or V

// One block of the traversal.
struct TcBlock {
  int i, c;        // sequence, KV head
  int j0;          // first page (index among the sequence's visible pages)
  int n;           // visible pages of the sequence
  int np;          // pages in the block
  int64_t k0;      // position of the first page in the CTA's range
  bool first;      // first block of a segment
  bool last;       // last block of a segment
};

// Walks a CTA's page range block by block.  Producer, MMA issuer and softmax
// warps each run one and see the same sequence of blocks.
struct BlockWalker {
  Cursor cu;
  int64_t k, count;
  int npb;

  __device__ __forceinline__ BlockWalker(const int32_t* pre, int B, int NC, int64_t start, int64_t cnt, int block_pages)
      : cu(locate(pre, B, NC, start)), k(0), count(cnt), npb(block_pages) {}

  __device__ __forceinline__ bool more() const { return k < count; }

  __device__ __forceinline__ TcBlock next(const int32_t* pre, int B, int NC) {
    TcBlock t;
    t.i = cu.i;
    t.c = cu.c;
    t.j0 = cu.j;
    t.n = cu.n;
    t.k0 = k;
    t.first = (k == 0) || (cu.j == 0);
    int np = min(npb, cu.n - cu.j);
    if (count - k < np) np = static_cast<int>(count - k);
    t.np = np;
    t.last = (cu.j + np == cu.n) || (k + np == count);
    for (int q = 0; q < np; ++q) advance(cu, pre, B, NC);
    k += np;
    return t;
  }
};

// Warp-uniform bounded wait: true only if every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, limit_ns));
}

template <int D>
struct TcGeo {
  static constexpr int NH = D / 64;                    // 64-column halves
  static constexpr int KSTEPS = D / 16;
};

// Shared-memory descriptors.  A descriptor's address field is the byte
// address >> 4, so a descriptor for base + off is the base descriptor + off/16
// (no carry: shared addresses are below 2^18).  The kernel builds one base
// descriptor per operand and block and adds compile-time offsets, which keeps
// the MMA issue loop free of per-instruction descriptor arithmetic.
//   K  (K-major, 16 * np rows): k-step s at (s / 4) * kTcHalf + (s % 4) * 32
//   V  (MN-major, d contiguous): page pg at pg * kTcBox; 8-row groups 1 KB
//      apart (SBO), the two 64-column halves kTcHalf apart (LBO)
__device__ __forceinline__ constexpr uint32_t k_step(int s) { return ((s >> 2) * kTcHalf + (s & 3) * 32u) >> 4; }

template <int D, bool WINDOW>
__global__ void __launch_bounds__(kTcThreads, 1)
    pa_split_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                       const SplitParams p) {
  using TG = TcGeo<D>;
  const int window = WINDOW ? p.window : 0;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_scan[kTcThreads / 32 + 1];
  __shared__ int s_total;
  __shared__ uint32_t s_tmem;

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
  grid_dependency_wait();
  page_prefix(p, window, s_pre, s_len, s_qsl, s_scan, &s_total);

  const uint32_t bar0 = base + p.off_bar;
  const int nstage = p.nstage;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (nstage + s); };
  const uint32_t xb = bar0 + 8u * (2 * nstage);
  // per softmax group g (blocks b with b % 2 == g): S ready, P ready, P V done
  auto sfull_bar = [&](int g) { return xb + 8u * g; };
  auto pfull_bar = [&](int g) { return xb + 8u * (4 + g); };
  auto odone_bar = [&](int g) { return xb + 8u * (6 + g); };
  auto qfull_bar = [&](int x) { return xb + 8u * (8 + x); };
  const uint32_t ofree_bar = xb + 8u * 10;   // both O accumulators read by a segment's epilogue
  const uint32_t drain_bar = xb + 8u * 12;
  // a segment's (max, sum) exchange between the two groups' warps of one
  // TMEM lane quarter
  auto xstat_bar = [&](int q) { return xb + 8u * (18 + q); };
  const uint32_t drain2_bar = xb + 8u * 17;
  if (tid == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(full_bar(s), kTcProducers);   // each producer warp arrives once per block
      mbar_init(empty_bar(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(sfull_bar(x), 1);
      mbar_init(pfull_bar(x), kTcSoftmaxWarps / 2);
      mbar_init(odone_bar(x), 1);
      mbar_init(qfull_bar(x), kTcSoftmaxWarps);
    }
    mbar_init(ofree_bar, kTcSoftmaxWarps);
    for (int q = 0; q < 4; ++q) mbar_init(xstat_bar(q), 2);
    mbar_init(drain_bar, 1);
    mbar_init(drain2_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int NC = p.NC;   // == Hkv (one KV head per unit)
  const int64_t X = static_cast<int64_t>(NC) * s_pre[B];
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

  if (warp == kTcMmaWarp) tmem_alloc(smem_addr(&s_tmem), kTcCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = warp_uniform(s_tmem);

  const int G = p.G;
  constexpr uint32_t half_stride = kTcHalf;
  const uint32_t stage0 = base + p.off_stage;

  if (warp < kTcProducers) {
    // ============================ producers ================================
    BlockWalker wk(s_pre, B, NC, start, count, kTcMaxBlockPages);
    BlockTableCache btc;
    int stage = 0;
    uint32_t round = 0;
    while (wk.more()) {
      const TcBlock t = wk.next(s_pre, B, NC);
      if (round > 0 && !warp_wait(empty_bar(stage), (round - 1) & 1u, p.wait_ns)) {
        if (lane == 0) atomicOr(p.err, kErrTimeout);
        break;
      }
      // The block's 2 * NH boxes per page are dealt round-robin over the three
      // producer warps, one box per lane (box x = 3 * lane + warp), so each
      // warp issues its share with one TMA instruction; each warp announces
      // its bytes with its own arrival, before its copies.
      constexpr int BPP = 2 * TG::NH;                // boxes per page: K and V, each NH halves
      const int nbox = t.np * BPP;
      const int mine = nbox > warp ? (nbox - warp + kTcProducers - 1) / kTcProducers : 0;
      if (lane == 0) mbar_arrive_expect_tx(full_bar(stage), static_cast<uint32_t>(mine) * kTcBox);
      __syncwarp();
      int phys[kTcMaxBlockPages];
#pragma unroll
      for (int pg = 0; pg < kTcMaxBlockPages; ++pg) {
        phys[pg] = 0;
        if (pg < t.np) {
          Cursor pc;
          pc.i = t.i;
          pc.c = t.c;
          pc.j = t.j0 + pg;
          pc.n = t.n;
          phys[pg] = btc.lookup(p, pc, s_pre, s_len, s_qsl, B, NC, window, lane);
          if ((phys[pg] < 0 || phys[pg] >= p.num_pages) && lane == 0 && warp == 0) atomicOr(p.err, kErrPageRange);
        }
      }
      const int x = kTcProducers * lane + warp;
      if (x < nbox) {
        const int pg = x / BPP;
        const int kind = x - pg * BPP;
        const int tensor = kind / TG::NH;
        const int h = kind - tensor * TG::NH;
        int ph = phys[0];
#pragma unroll
        for (int q = 1; q < kTcMaxBlockPages; ++q) ph = pg == q ? phys[q] : ph;
        const uint32_t sb = stage0 + static_cast<uint32_t>(stage) * p.stage_bytes;
        const uint32_t dst = sb + static_cast<uint32_t>(tensor * TG::NH + h) * half_stride + static_cast<uint32_t>(pg) * kTcBox;
        // An out-of-range page id reads as zeros (TMA fills outside the tensor).
        tma_load_4d(dst, tensor ? &tmap_v : &tmap_k, h * 64, 0, t.c, ph, full_bar(stage));
      }
      if (++stage == nstage) {
        stage = 0;
        ++round;
      }
    }
  } else if (warp == kTcMmaWarp) {
    // ============================ Q K^T issuer =============================
    const uint32_t idesc_s_base = umma_idesc_bf16(128, 16, false) & ~(0x3Fu << 17);
    BlockWalker wk(s_pre, B, NC, start, count, kTcMaxBlockPages);
    int stage = 0;
    uint32_t round = 0;
    int b = 0, seg = -1;
    bool ok = true;
    while (wk.more()) {
      const TcBlock t = wk.next(s_pre, B, NC);
      if (t.first) ++seg;
      // S(b) goes where P(b-2), the same group's previous block, was: its P V
      // must be done (the group read S(b-2) before it wrote P(b-2)).
      if (!warp_wait(full_bar(stage), round & 1u, p.wait_ns) ||
          (b >= 2 && !warp_wait(odone_bar(b & 1), static_cast<uint32_t>((b >> 1) - 1) & 1u, p.wait_ns)) ||
          (t.first && !warp_wait(qfull_bar(seg & 1), static_cast<uint32_t>(seg >> 1) & 1u, p.wait_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tQ = warp_uniform(tbase + kTmemQ + 64u * static_cast<uint32_t>(seg & 1));
      const uint32_t sb = warp_uniform(stage0 + static_cast<uint32_t>(stage) * p.stage_bytes);
      const uint64_t kd = umma_sdesc_sw128(sb, 16u, 1024u);
      const uint32_t idesc_s = warp_uniform(idesc_s_base | (static_cast<uint32_t>(2 * t.np) << 17));   // N = 16 * np
      const uint32_t tS = warp_uniform(tbase + kTmemSP + 64u * static_cast<uint32_t>(b & 1));
      if (lane == 0) {
#pragma unroll
        for (int s = 0; s < TG::KSTEPS; ++s) umma_ts(tS, tQ + 8u * s, kd + k_step(s), idesc_s, s > 0);
        umma_commit(sfull_bar(b & 1));
      }
      __syncwarp();
      ++b;
      if (++stage == nstage) {
        stage = 0;
        ++round;
      }
    }
    if (!ok && lane == 0) atomicOr(p.err, kErrTimeout);
    // Every MMA this warp issued must be complete before tensor memory is freed.
    if (lane == 0) umma_commit(drain_bar);
    __syncwarp();
    if (!warp_wait(drain_bar, 0u, p.wait_ns) && lane == 0) atomicOr(p.err, kErrTimeout);
  } else if (warp == kTcPvWarp) {
    // ============================ P V issuer ===============================
    // Runs beside the Q K^T issuer, so the two MMA streams do not wait on
    // each other's barriers; the ordering they need comes through the
    // softmax: P V of block b waits for P(b), which the softmax writes only
    // after it has read S(b).
    const uint32_t idesc_o = umma_idesc_bf16(128, D, true);
    BlockWalker wk(s_pre, B, NC, start, count, kTcMaxBlockPages);
    int stage = 0;
    uint32_t round = 0;
    int b = 0, seg = -1, b0 = 0;
    bool ok = true;
    while (wk.more()) {
      const TcBlock t = wk.next(s_pre, B, NC);
      if (t.first) {
        ++seg;
        b0 = b;
      }
      // a group's first block of the segment overwrites its O
      const bool ofirst = b - b0 < 2;
      // full(stage) has completed before P(b) exists; waiting on it here makes
      // the stage's TMA data visible to this warp directly.
      if (!warp_wait(pfull_bar(b & 1), static_cast<uint32_t>(b >> 1) & 1u, p.wait_ns) ||
          !warp_wait(full_bar(stage), round & 1u, p.wait_ns) ||
          // the previous segment's epilogue must have read both O accumulators
          (ofirst && seg >= 1 && !warp_wait(ofree_bar, static_cast<uint32_t>(seg - 1) & 1u, p.wait_ns))) {
        ok = false;
        break;
      }
      int vt = kPage;
      if (t.j0 + t.np == t.n) {
        const SeqInfo si = seq_info(p, s_len, s_qsl, t.i, false, window);
        vt = si.L - kPage * (si.js + t.n - 1);
      }
      const uint32_t sb = warp_uniform(stage0 + static_cast<uint32_t>(stage) * p.stage_bytes);
      if (vt < kPage) {
        // Rows past the context in the unit's last page: zero them so that
        // whatever the pool holds there cannot reach O through 0 * NaN.
        uint8_t* const vg = gbase + (sb - base) + TG::NH * half_stride + (t.np - 1) * kTcBox;
        const int nbytes = (kPage - vt) * 128;
        for (int h = 0; h < TG::NH; ++h)
          for (int o = lane * 16; o < nbytes; o += 32 * 16)
            *reinterpret_cast<uint4*>(vg + h * half_stride + vt * 128 + o) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc_fence_after();
      const uint64_t vd0 = umma_sdesc_sw128(sb + TG::NH * half_stride, half_stride, 1024u);
      const uint32_t tO = warp_uniform(tbase + kTmemO + 128u * static_cast<uint32_t>(b & 1));
      const uint32_t tP = warp_uniform(tbase + kTmemSP + 64u * static_cast<uint32_t>(b & 1) + kTmemPhi);
      if (lane == 0) {
#pragma unroll
        for (int pg = 0; pg < kTcMaxBlockPages; ++pg) {
          if (pg < t.np) {
            const uint64_t vd = vd0 + static_cast<uint64_t>((pg * kTcBox) >> 4);
            umma_ts(tO, tP + 8u * pg, vd, idesc_o, !(ofirst && pg == 0));
          }
        }
        umma_commit(odone_bar(b & 1));
        umma_commit(empty_bar(stage));
      }
      __syncwarp();
      ++b;
      if (++stage == nstage) {
        stage = 0;
        ++round;
      }
    }
    if (!ok && lane == 0) atomicOr(p.err, kErrTimeout);
    if (lane == 0) umma_commit(drain2_bar);
    __syncwarp();
    if (!warp_wait(drain2_bar, 0u, p.wait_ns) && lane == 0) atomicOr(p.err, kErrTimeout);
  } else {
    // ============================ softmax ==================================
    // Two groups of four warps; group gi = (warp - 4) / 4 takes the blocks b
    // with b % 2 == gi, so two blocks' softmax work overlaps.  Warp q4 = warp % 4
    // of a group owns rows 32 * q4 .. +31 (thread = query row = TMEM lane) and
    // all of a block's keys, with its own running max and sum and its own O
    // accumulator in tensor memory.  At a segment's end the two threads of a
    // row exchange (max, sum) through shared memory and a bounded mbarrier
    // round and each combines half of O's columns.
    const int gi = (warp - kTcSoftmaxWarp0) >> 2;
    const int q4 = warp & 3;               // TMEM lane quarter this warp may access
    const int rho = 32 * q4 + lane;        // query row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    float4* const xstat = reinterpret_cast<float4*>(gbase + p.off_xchg);   // [segment % 2][group][128] (max, sum, rounded sum)
    constexpr int HD = D / 2;              // O columns each group's thread writes out
    constexpr int NP4 = kTcMaxBlockPages;
    BlockWalker wk(s_pre, B, NC, start, count, kTcMaxBlockPages);
    int b = 0, seg = -1, b0 = 0;
    SeqInfo si = {0, 0, 0, 0};
    bool row_ok = false;
    int lim = 0, seg_j0 = 0;
    int64_t seg_k0 = 0;
    float m = -INFINITY, l = 0.f;          // this group's running max (log2 units) and sum of the row
    float lr = 0.f;                        // the sum of the weights as rounded into P (O's normaliser)
    bool ok = true;

    // This thread's half (by group) of row rho of the segment starting at
    // block t, into TMEM Q slot `slot` (rows past G * qn are zero); q_full
    // counts the 8 warps.
    auto stage_q = [&](const TcBlock& t, int slot) {
      const SeqInfo s2 = seq_info(p, s_len, s_qsl, t.i, false, window);
      const bool have = rho < G * s2.qn;
      const uint4* src = nullptr;
      if (have)
        src = reinterpret_cast<const uint4*>(p.q + static_cast<int64_t>(s2.t0 + rho / G) * p.q_stride_t +
                                             static_cast<int64_t>(t.c * G + rho % G) * D);
      const uint32_t tq = tbase + lane_off + kTmemQ + 64u * static_cast<uint32_t>(slot) + (D / 4) * gi;
#pragma unroll
      for (int k = 0; k < D / 64; ++k) {      // 16 columns (32 features) at a time
        uint32_t w[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 v = have ? src[(D / 16) * gi + 4 * k + u] : make_uint4(0u, 0u, 0u, 0u);
          w[4 * u] = v.x;
          w[4 * u + 1] = v.y;
          w[4 * u + 2] = v.z;
          w[4 * u + 3] = v.w;
        }
        tmem_st16(tq + 16u * k, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(qfull_bar(slot));
    };

    while (wk.more()) {
      const TcBlock t = wk.next(s_pre, B, NC);
      if (t.first) {
        ++seg;
        b0 = b;
        if (seg == 0) stage_q(t, 0);
        si = seq_info(p, s_len, s_qsl, t.i, rho == 0 && gi == 0, window);
        row_ok = rho < G * si.qn;
        lim = si.L - si.qn + (row_ok ? rho / G : 0);
        seg_j0 = t.j0;
        seg_k0 = t.k0;
        m = -INFINITY;
        l = 0.f;
        lr = 0.f;
        if (seg_j0 == 0 && rho == 0 && gi == 0) {
          // This CTA holds the unit's first page: describe the unit for the merge.
          const int64_t a = static_cast<int64_t>(NC) * s_pre[t.i] + static_cast<int64_t>(t.c) * t.n;
          const int last_cta = static_cast<int>(((a + t.n) * NG - 1) / X);
          const int pieces = last_cta - g + 1;
          p.ws_unit[static_cast<int64_t>(t.i) * NC + t.c] =
              make_int4(g, pieces | (t.k0 != 0 ? (1 << 30) : 0), si.t0, si.qn);
        }
        if (p.sinks != nullptr && seg_j0 == 0 && row_ok && gi == (b & 1)) {
          // The sink is a virtual first key (logit sinks[hq], zero value row),
          // counted once, by the group taking the segment's first block in the
          // piece holding the unit's first page.
          m = p.sinks[t.c * G + rho % G] * 1.4426950408889634f;
          l = 1.f;
          lr = 1.f;                          // the sink's weight, exact (it is not in P)
        }
      }
      if ((b & 1) == gi) {
        // ---- the block's S row ----------------------------------------------
        if (!warp_wait(sfull_bar(gi), static_cast<uint32_t>(b >> 1) & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tSP = tbase + lane_off + kTmemSP + 64u * static_cast<uint32_t>(gi);
        float sv[NP4][16];
        {
          // every page's columns are read; pages past the block's end hold
          // stale scores that the mask below discards
          uint32_t r[NP4][16];
#pragma unroll
          for (int k = 0; k < NP4; ++k) tmem_ld16(tSP + 16u * k, r[k]);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < NP4; ++k)
#pragma unroll
            for (int e = 0; e < 16; ++e) sv[k][e] = __uint_as_float(r[k][e]);
        }
        // ---- mask, block max -------------------------------------------------
        // An interior block (all pages present, every token visible to every
        // row of the run, no window edge inside) needs no per-element mask:
        // its max is taken over the raw scores and the scale is folded into
        // the exponent's FFMA.  Rows past G * qn hold zero queries there and
        // produce values nobody reads.
        const int tb = kPage * (si.js + t.j0);
        const float c = p.scale_log2;
        bool interior = t.np == NP4 && c > 0.f && tb + NP4 * kPage <= si.L - si.qn + 1;
        if (WINDOW && window > 0) interior = interior && tb > si.L - 1 - window;
        float mb;
        if (interior) {
          float mx[16 * NP4];
#pragma unroll
          for (int k = 0; k < NP4; ++k)
#pragma unroll
            for (int e = 0; e < 16; ++e) mx[16 * k + e] = sv[k][e];
          mb = Max3Tree<16 * NP4>::run(mx) * c;
        } else {
          float mx[16 * NP4];
#pragma unroll
          for (int k = 0; k < NP4; ++k)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int tok = tb + 16 * k + e;
              bool vis = row_ok && k < t.np && tok <= lim;
              if (WINDOW && window > 0) vis = vis && tok > lim - window;
              const float x = vis ? sv[k][e] * c : -INFINITY;
              sv[k][e] = x;
              mx[16 * k + e] = x;
            }
          mb = Max3Tree<16 * NP4>::run(mx);
        }
        const float m_new = fmaxf(m, mb);
        const bool grow = m_new > m + 8.f;   // also true when m = -inf and m_new is finite
        if (b - b0 < 2) {
          // the group's first block of the segment: O has no history yet
          if (grow) {
            const float a = fast_exp2(m - m_new);   // only a sink carries weight here
            l *= a;
            lr *= a;
            m = m_new;
          }
        } else if (__any_sync(0xffffffffu, grow)) {
          // O must hold P V of the group's previous block before it is rescaled.
          if (!warp_wait(odone_bar(gi), static_cast<uint32_t>((b >> 1) - 1) & 1u, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = grow ? fast_exp2(m - m_new) : 1.f;
          const uint32_t tO = tbase + lane_off + kTmemO + 128u * static_cast<uint32_t>(gi);
#pragma unroll
          for (int ch = 0; ch < D / 16; ++ch) {
            uint32_t r[16];
            tmem_ld16(tO + 16u * ch, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st16(tO + 16u * ch, r);
          }
          tmem_wait_st();
          if (grow) {
            l *= alpha;
            lr *= alpha;
            m = m_new;
          }
        }
        // ---- P (bf16) over the block's S -----------------------------------------
        // This thread has read its whole S row above; P V of the group's
        // previous block read P from these columns before Q K^T of this block
        // was issued into them.
        {
          // exp2 of -inf is +0, so masked scores need no select once the
          // subtracted max is finite (it is -inf only while no key was visible).
          const float mneg = m == -INFINITY ? 0.f : -m;
          const float mult = interior ? c : 1.f;   // masked scores are already scaled
          const uint32_t tP = tSP + kTmemPhi;
          // pairs of scores through packed fp32 arithmetic: exponent argument
          // (one FMA for two) and two running sums, of the weights and of the
          // weights as rounded into P (O divided by the second stays a
          // weighted mean of V rows; the first gives the lse)
          const uint64_t mult2 = f2_pack(mult, mult), mneg2 = f2_pack(mneg, mneg);
          uint64_t lsum2 = f2_pack(0.f, 0.f), rsum2 = f2_pack(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < NP4; ++k) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              float x0, x1;
              f2_unpack(ffma2(f2_pack(sv[k][2 * e], sv[k][2 * e + 1]), mult2, mneg2), x0, x1);
              const float a0 = fast_exp2(x0);
              const float a1 = fast_exp2(x1);
              w[e] = pack_bf16(a0, a1);
              lsum2 = fadd2(lsum2, f2_pack(a0, a1));
              rsum2 = fadd2(rsum2, f2_pack(bf16_lo(w[e]), bf16_hi(w[e])));
            }
            tmem_st8(tP + 8u * k, w);
          }
          {
            float s0, s1;
            f2_unpack(lsum2, s0, s1);
            l += s0 + s1;
            f2_unpack(rsum2, s0, s1);
            lr += s0 + s1;
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pfull_bar(gi));
      }

      if (t.last) {
        // The next segment's Q goes into the other slot now, so its S can be
        // computed while this segment's output is written.
        if (wk.more()) {
          BlockWalker peek = wk;
          const TcBlock nt = peek.next(s_pre, B, NC);
          stage_q(nt, (seg + 1) & 1);
        }
        // the other group's (max, sum) of the row
        xstat[(seg & 1) * 256 + gi * 128 + rho] = make_float4(m, l, lr, 0.f);
        __syncwarp();
        if (lane == 0) mbar_arrive(xstat_bar(q4));
        if (!warp_wait(xstat_bar(q4), static_cast<uint32_t>(seg) & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        const float4 other = xstat[(seg & 1) * 256 + (gi ^ 1) * 128 + rho];
        // group 0's and group 1's statistics
        const float m0 = gi == 0 ? m : other.x, l0 = gi == 0 ? l : other.y, r0 = gi == 0 ? lr : other.z;
        const float m1 = gi == 0 ? other.x : m, l1 = gi == 0 ? other.y : l, r1 = gi == 0 ? other.z : lr;
        const float mt = fmaxf(m0, m1);
        const float a0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - mt);
        const float a1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - mt);
        const float lt = l0 * a0 + l1 * a1;    // the row's sum (lse, merge weights)
        const float lrt = r0 * a0 + r1 * a1;   // O's normaliser
        // Each group's last block of the segment: b and b - 1 (this block is
        // the segment's last); a group with no block in it has no O to read.
        const int bl0 = (b & 1) == 0 ? b : b - 1;
        const int bl1 = (b & 1) == 1 ? b : b - 1;
        const bool has0 = bl0 >= b0, has1 = bl1 >= b0;
        if ((has0 && !warp_wait(odone_bar(0), static_cast<uint32_t>(bl0 >> 1) & 1u, p.wait_ns)) ||
            (has1 && !warp_wait(odone_bar(1), static_cast<uint32_t>(bl1 >> 1) & 1u, p.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool complete = (seg_j0 == 0) && (t.j0 + t.np == t.n);
        const uint32_t tO0 = tbase + lane_off + kTmemO + HD * gi;   // this thread's half of the columns
        const uint32_t tO1 = tO0 + 128u;
        const int tok = si.t0 + rho / G;
        const int hq = t.c * G + rho % G;
        const float inv = lrt > 0.f ? p.v_scale / lrt : 0.f;
        // a piece's O goes to the merge scaled so that O / lt is O's weighted mean
        const float pscale = lrt > 0.f ? lt / lrt : 0.f;
        uint16_t* orow =
            p.out + static_cast<int64_t>(tok) * p.out_stride_t + static_cast<int64_t>(hq) * p.out_stride_h + HD * gi;
        const int which = (seg_k0 == 0) ? 0 : 1;
        const int64_t prow = static_cast<int64_t>(2 * g + which) * p.R_max + rho;
        float* wrow = p.ws_o + prow * D + HD * gi;
#pragma unroll
        for (int ch = 0; ch < HD / 16; ++ch) {
          float o[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = 0.f;
#pragma unroll
          for (int gg = 0; gg < 2; ++gg) {
            if (gg == 0 ? has0 : has1) {
              uint32_t r[16];
              tmem_ld16((gg == 0 ? tO0 : tO1) + 16u * ch, r);
              tmem_wait_ld();
              const float a = gg == 0 ? a0 : a1;
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = fmaf(__uint_as_float(r[e]), a, o[e]);
            }
          }
          if (row_ok) {
            if (complete) {
#pragma unroll
              for (int e = 0; e < 16; e += 4) {
                uint2 v;
                v.x = pack_bf16(o[e] * inv, o[e + 1] * inv);
                v.y = pack_bf16(o[e + 2] * inv, o[e + 3] * inv);
                *reinterpret_cast<uint2*>(orow + 16 * ch + e) = v;
              }
            } else {
#pragma unroll
              for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4*>(wrow + 16 * ch + e) =
                    make_float4(o[e] * pscale, o[e + 1] * pscale, o[e + 2] * pscale, o[e + 3] * pscale);
            }
          }
        }
        if (row_ok && gi == 0) {
          if (complete) {
            if (p.lse != nullptr)
              p.lse[static_cast<int64_t>(tok) * p.lse_stride_t + static_cast<int64_t>(hq) * p.lse_stride_h] =
                  lt > 0.f ? (mt + fast_log2(lt)) * 0.69314718055994530942f : -INFINITY;
          } else {
            p.ws_ml[prow] = make_float2(mt, lt);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ofree_bar);
      }
      ++b;
    }
    if (!ok && lane == 0) atomicOr(p.err, kErrTimeout);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kTcMmaWarp) tmem_dealloc(tbase, kTcCols);
}

}  // namespace pa
