// Multi-head latent attention (MLA) decode on the 5th-generation tensor cores
// (tcgen05 + tensor memory), sm_103a.
//
// What it computes is that of the mma.sync MLA kernel (ATOM model-operations
// guide, "Multi-head latent attention (attention_mla.py)", decode flow step 2:
// mla_decode_fwd over the rows fused_qk_rope_concat_and_cache_mla wrote): every
// cached token is one row C_j = [c_kv (512) | k_pe (64)] shared by all query
// heads, and a query row is as wide, so
//   s_j = scale * <q, C_j>,   out = sum_j softmax(s)_j C_j[0:512],   lse = ln sum_j e^{s_j}.
// Work split, unit descriptors and partials (normalised outputs in f16 with
// the fp32 running max and sum) are those of the mma.sync MLA kernel with one
// worker per CTA, so the same LSE merge kernel finishes cut units.
//
// Why this shape of kernel: a unit has at most 32 query rows (heads x query
// tokens), each with a 512-wide fp32 output.  As [rows x 512] the output alone
// would fill all 512 tensor-memory columns, so the P V product is taken
// transposed, O^T[512 x rows] += V^T[512 x keys] P^T[keys x rows]: four
// 128-lane blocks of R_pad (16 or 32) columns.  Q K^T stays row-major with the
// query rows on the tensor-memory lanes (the padded rows past R are never read),
// so the softmax is a thread per row that owns all of a block's keys.
//
// A block is up to 4 pages (64 keys) of one segment.  Per block:
//   S[128 x 16np]     = Q[128 x 576] K^T        36 TS-MMAs (Q in tensor memory)
//   O^T[vb][128 x R]  += V^T[vb] P^T            4 SS-MMAs a page (bf16 caches: twice,
//                                                P carried as bf16 hi + lo terms)
// Tensor memory (512 columns): O^T [0, 4 R_pad), S [128, 192), Q [192, 480).
//
// Roles (352 threads):
//   warp 0      producer: block-table lookups, one TMA box per page (the whole
//               16 x 576 row block) into a ring of raw page slots;
//   warp 1      Q K^T issuer, owner of the tensor-memory allocation;
//   warp 2      P V issuer;
//   warps 3, 8-10 converters: each raw page into the MMA layout of the block's
//               buffer ([column block][page][16 rows x 128 B], 128-byte
//               swizzle): bf16 rows are copied, fp8 codes become f16 (exact);
//               value rows past the sequence end are zeroed;
//   warps 4-7   softmax, thread = query row = tensor-memory lane: S row, mask,
//               block max, exponentials into the P buffer (shared memory, the
//               B operand of P V), lazy O rescale, segment epilogue.
// Every wait is bounded (kErrTimeout); the MMAs are drained before the tensor
// memory is freed.  Each parity wait is made only when its waiter has already
// seen the barrier's previous phase complete (directly, or through the chain of
// completions noted at the wait), so no wait can pass a phase early.
#include "pa_pack.cuh"
#include "pa_split_tc.cuh"   // BlockWalker, TcBlock, Max3Tree

namespace pa {

namespace {

constexpr int kMtcDqk = 576;
constexpr int kMtcDv = 512;
constexpr int kMtcCb = kMtcDqk / 64;             // 64-feature column blocks of a row
constexpr int kMtcBlockPages = 4;
constexpr uint32_t kMtcTile = 2048;               // MMA layout: one page of one column block, 16 x 128 B
constexpr uint32_t kMtcCbStride = kMtcBlockPages * kMtcTile;
constexpr uint32_t kMtcBuf = kMtcCb * kMtcCbStride;   // one block's rows in the MMA layout (72 KB)
constexpr int kMtcThreads = 352;
constexpr int kMtcProducer = 0, kMtcQkWarp = 1, kMtcPvWarp = 2, kMtcSoftmax0 = 4;
constexpr int kMtcConverters = 4;                 // warps 3, 8, 9, 10
constexpr uint32_t kMtcCols = 512;
constexpr uint32_t kMtcTmemO = 0, kMtcTmemS = 128, kMtcTmemQ = 192;
constexpr int kMtcQsteps = kMtcDqk / 16;          // k-steps of Q K^T

__device__ __forceinline__ int converter_index(int warp) { return warp == 3 ? 0 : warp - 7; }

// Instruction descriptor of kind::f16 (fp32 accumulator): A and B both bf16 or
// both f16; `a_mn` / `b_mn` select the MN-major (transposed) operand layout.
__device__ __forceinline__ uint32_t mtc_idesc(int M, int N, bool bf16, bool a_mn, bool b_mn) {
  uint32_t d = 1u << 4;                           // D: F32
  if (bf16) d |= (1u << 7) | (1u << 10);          // A, B: BF16 (0: F16)
  d |= (a_mn ? 1u : 0u) << 15;
  d |= (b_mn ? 1u : 0u) << 16;
  d |= static_cast<uint32_t>(N >> 3) << 17;
  d |= static_cast<uint32_t>(M >> 4) << 24;
  return d;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// Named-barrier-free bounded wait of all lanes of a warp.
__device__ __forceinline__ bool mtc_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, limit_ns));
}

// bf16x2 -> f16x2 with a flag for values beyond the f16 range.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x, bool& fine) {
  const uint32_t r = pack_f16(bf16_lo(x), bf16_hi(x));
  fine &= ((r & 0x7C00u) != 0x7C00u) && ((r & 0x7C000000u) != 0x7C000000u);
  return r;
}

}  // namespace

// Shared-memory layout (bytes from the 1024-aligned base), host and device:
//   off_buf   2 x kMtcBuf          the two block buffers in the MMA layout
//   off_q     P buffers            2 (block parity) x NPT (hi / lo) x R_pad x 128 B
//   off_stage raw page slots       nstage x (16 x 576 x esz), as the TMA box lands
//   off_bar   barriers
//   off_xchg  softmax exchange     alpha [2][128] f32, flags [2][4] u32, row stats [128] float2
//   off_prefix sequence metadata
template <bool FP8, int RP>
__global__ void __launch_bounds__(kMtcThreads, 1)
    pa_mla_tc_kernel(const __grid_constant__ CUtensorMap tmap, const SplitParams p) {
  constexpr int ESZ = FP8 ? 1 : 2;
  constexpr uint32_t kRawPage = kPage * kMtcDqk * ESZ;   // one TMA box: [9 blocks][16 rows][64 x esz B]
  constexpr uint32_t kRawBlock = 16u * 64u * ESZ;
  constexpr int NPT = FP8 ? 1 : 2;                       // P terms
  constexpr uint32_t kPbuf = static_cast<uint32_t>(RP) * 128u;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_scan[kMtcThreads / 32 + 1];
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
  const int nstage = p.nstage;
  const uint32_t bar0 = base + p.off_bar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (nstage + s); };
  const uint32_t xb = bar0 + 8u * (2 * nstage);
  auto cfull_bar = [&](int x) { return xb + 8u * x; };          // block buffer x converted (4 converter warps)
  auto bfree_bar = [&](int x) { return xb + 8u * (2 + x); };    // block buffer x read by both MMAs (commit)
  auto pfull_bar = [&](int x) { return xb + 8u * (4 + x); };    // P buffer x written (4 softmax warps)
  auto pfree_bar = [&](int x) { return xb + 8u * (6 + x); };    // P V of the block in P buffer x done (commit)
  const uint32_t sfull_bar = xb + 8u * 8;                       // S of a block in tensor memory (commit)
  const uint32_t sfree_bar = xb + 8u * 9;                       // S read, block statistics published (4 warps)
  const uint32_t qfull_bar = xb + 8u * 10;                      // a segment's Q in tensor memory (4 warps)
  const uint32_t ebar = xb + 8u * 11;                           // a segment's row statistics published (4 warps)
  const uint32_t ofree_bar = xb + 8u * 12;                      // O read by a segment's epilogue (4 warps)
  const uint32_t drain_bar = xb + 8u * 13;
  const uint32_t drain2_bar = xb + 8u * 14;
  float* const x_alpha = reinterpret_cast<float*>(gbase + p.off_xchg);              // [2][128]
  uint32_t* const x_flag = reinterpret_cast<uint32_t*>(gbase + p.off_xchg + 1024);  // [2][4]
  float2* const x_stat = reinterpret_cast<float2*>(gbase + p.off_xchg + 1280);      // [128] (m, l)

  if (tid == 0) {
    prefetch_tensormap(&tmap);
    for (int s = 0; s < nstage; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kMtcConverters);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(cfull_bar(x), kMtcConverters);
      mbar_init(bfree_bar(x), 1);
      mbar_init(pfull_bar(x), 4);
      mbar_init(pfree_bar(x), 1);
    }
    mbar_init(sfull_bar, 1);
    mbar_init(sfree_bar, 4);
    mbar_init(qfull_bar, 4);
    mbar_init(ebar, 4);
    mbar_init(ofree_bar, 4);
    mbar_init(drain_bar, 1);
    mbar_init(drain2_bar, 1);
    fence_mbar_init();
  }
  // Inputs may come from the previous kernel in the stream (programmatic
  // dependent launch): nothing global is read before this point.
  grid_dependency_wait();
  page_prefix(p, 0, s_pre, s_len, s_qsl, s_scan, &s_total);
  __syncthreads();

  const int NC = p.NC, G = p.G;
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

  if (warp == kMtcQkWarp) tmem_alloc(smem_addr(&s_tmem), kMtcCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = warp_uniform(s_tmem);
  const uint32_t buf0 = base + p.off_buf;
  const uint32_t pbuf0 = base + p.off_q;
  const uint32_t ring0 = base + p.off_stage;

  if (warp == kMtcProducer) {
    // ============================ producer =================================
    Cursor cu = locate(s_pre, B, NC, start);
    BlockTableCache btc;
    int stage = 0;
    uint32_t round = 0;
    for (int64_t k = 0; k < count; ++k) {
      if (round > 0 && !mtc_wait(empty_bar(stage), (round - 1) & 1u, p.wait_ns)) {
        if (lane == 0) atomicOr(p.err, kErrTimeout);
        break;
      }
      const int phys = btc.lookup(p, cu, s_pre, s_len, s_qsl, B, NC, 0, lane);
      if (lane == 0) {
        if (phys < 0 || phys >= p.num_pages) atomicOr(p.err, kErrPageRange);
        // the page's 16 rows, all 576 features; an out-of-range page id reads zeros
        mbar_arrive_expect_tx(full_bar(stage), kRawPage);
        tma_load_4d(ring0 + static_cast<uint32_t>(stage) * kRawPage, &tmap, 0, 0, 0, phys, full_bar(stage));
      }
      __syncwarp();
      advance(cu, s_pre, B, NC);
      if (++stage == nstage) {
        stage = 0;
        ++round;
      }
    }
  } else if (warp == 3 || warp >= kMtcSoftmax0 + 4) {
    // ============================ converters ===============================
    const int ct = converter_index(warp) * 32 + lane;   // 0..127
    BlockWalker wk(s_pre, B, NC, start, count, kMtcBlockPages);
    int b = 0;
    bool ok = true;
    while (wk.more() && ok) {
      const TcBlock t = wk.next(s_pre, B, NC);
      // buffer b % 2 was last read by the MMAs of block b - 2 (this warp saw
      // the completion of block b - 4's, the previous phase, at block b - 2)
      if (b >= 2 && !mtc_wait(bfree_bar(b & 1), static_cast<uint32_t>((b >> 1) - 1) & 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      const uint32_t dst0 = buf0 + static_cast<uint32_t>(b & 1) * kMtcBuf;
      const int L = s_len[t.i];
      for (int pg = 0; pg < t.np; ++pg) {
        const int64_t kk = t.k0 + pg;
        const int stage = static_cast<int>(kk % nstage);
        const uint32_t rnd = static_cast<uint32_t>(kk / nstage);
        if (!mtc_wait(full_bar(stage), rnd & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        const uint32_t src = ring0 + static_cast<uint32_t>(stage) * kRawPage;
        const int vt = L - kPage * (t.j0 + pg);   // rows of this page inside the sequence
        const uint32_t dst = dst0 + static_cast<uint32_t>(pg) * kMtcTile;
        if constexpr (FP8) {
          // 16 codes (a 64-byte-swizzled chunk) -> 16 f16 values (two chunks of
          // the 128-byte-swizzled MMA row)
          for (int x = ct; x < kMtcCb * 16 * 4; x += 128) {
            const int cb = x >> 6, r = (x >> 2) & 15, c = x & 3;
            uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
            if (r < vt) {
              const uint4 v = lds128(src + cb * kRawBlock + swz<64>(r, c));
              o0.x = e4m3x2_to_f16x2(v.x);
              o0.y = e4m3x2_to_f16x2(v.x >> 16);
              o0.z = e4m3x2_to_f16x2(v.y);
              o0.w = e4m3x2_to_f16x2(v.y >> 16);
              o1.x = e4m3x2_to_f16x2(v.z);
              o1.y = e4m3x2_to_f16x2(v.z >> 16);
              o1.z = e4m3x2_to_f16x2(v.w);
              o1.w = e4m3x2_to_f16x2(v.w >> 16);
            }
            const uint32_t d = dst + static_cast<uint32_t>(cb) * kMtcCbStride;
            sts128(d + swz<128>(r, 2 * c), o0);
            sts128(d + swz<128>(r, 2 * c + 1), o1);
          }
        } else {
          // a raw column block is already one 128-byte-swizzled 16 x 128 B tile
          for (int x = ct; x < kMtcCb * 16 * 8; x += 128) {
            const int cb = x >> 7, r = (x >> 3) & 15, c = x & 7;
            const uint32_t off = swz<128>(r, c);
            const uint4 v = r < vt ? lds128(src + cb * kRawBlock + off) : make_uint4(0u, 0u, 0u, 0u);
            sts128(dst + static_cast<uint32_t>(cb) * kMtcCbStride + off, v);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(stage));
      }
      if (!ok) break;
      fence_proxy_async_smem();   // the tensor cores read what these generic stores wrote
      __syncwarp();
      if (lane == 0) mbar_arrive(cfull_bar(b & 1));
      ++b;
    }
    if (!ok && lane == 0) atomicOr(p.err, kErrTimeout);
  } else if (warp == kMtcQkWarp) {
    // ============================ Q K^T issuer =============================
    const uint32_t idesc0 = mtc_idesc(128, 16, !FP8, false, false) & ~(0x3Fu << 17);
    const uint32_t tS = tbase + kMtcTmemS;
    const uint32_t tQ = tbase + kMtcTmemQ;
    BlockWalker wk(s_pre, B, NC, start, count, kMtcBlockPages);
    int b = 0, seg = -1;
    bool ok = true;
    while (wk.more()) {
      const TcBlock t = wk.next(s_pre, B, NC);
      if (t.first) ++seg;
      // converted rows of the block; the single S buffer read by the softmax
      // (phase b - 1, after phase b - 2 seen at the previous block); at a
      // segment's first block its Q (every segment's phase seen in order)
      if (!mtc_wait(cfull_bar(b & 1), static_cast<uint32_t>(b >> 1) & 1u, p.wait_ns) ||
          (b >= 1 && !mtc_wait(sfree_bar, static_cast<uint32_t>(b - 1) & 1u, p.wait_ns)) ||
          (t.first && !mtc_wait(qfull_bar, static_cast<uint32_t>(seg) & 1u, p.wait_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t kb = warp_uniform(buf0 + static_cast<uint32_t>(b & 1) * kMtcBuf);
      const uint64_t kd = umma_sdesc_sw128(kb, 16u, 1024u);
      const uint32_t idesc = warp_uniform(idesc0 | (static_cast<uint32_t>(2 * t.np) << 17));   // N = 16 np
      if (lane == 0) {
#pragma unroll 4
        for (int s = 0; s < kMtcQsteps; ++s) {
          const uint32_t koff = static_cast<uint32_t>(s >> 2) * kMtcCbStride + static_cast<uint32_t>(s & 3) * 32u;
          umma_ts(tS, tQ + 8u * s, kd + (koff >> 4), idesc, s > 0);
        }
        umma_commit(sfull_bar);
      }
      __syncwarp();
      ++b;
    }
    if (!ok && lane == 0) atomicOr(p.err, kErrTimeout);
    if (lane == 0) umma_commit(drain_bar);
    __syncwarp();
    if (!mtc_wait(drain_bar, 0u, p.wait_ns) && lane == 0) atomicOr(p.err, kErrTimeout);
  } else if (warp == kMtcPvWarp) {
    // ============================ P V issuer ===============================
    const uint32_t idesc = mtc_idesc(128, RP, !FP8, true, false);
    BlockWalker wk(s_pre, B, NC, start, count, kMtcBlockPages);
    int b = 0, seg = -1;
    bool ok = true;
    while (wk.more()) {
      const TcBlock t = wk.next(s_pre, B, NC);
      if (t.first) ++seg;
      // P of the block (every phase seen in order); its converted rows, waited
      // here too so the stores are visible to this warp's MMAs; at a
      // segment's first block, the previous segment's epilogue done with O
      if (!mtc_wait(pfull_bar(b & 1), static_cast<uint32_t>(b >> 1) & 1u, p.wait_ns) ||
          !mtc_wait(cfull_bar(b & 1), static_cast<uint32_t>(b >> 1) & 1u, p.wait_ns) ||
          (t.first && seg >= 1 && !mtc_wait(ofree_bar, static_cast<uint32_t>(seg - 1) & 1u, p.wait_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t vb0 = warp_uniform(buf0 + static_cast<uint32_t>(b & 1) * kMtcBuf);
      const uint32_t pb = warp_uniform(pbuf0 + static_cast<uint32_t>(b & 1) * NPT * kPbuf);
      if (lane == 0) {
        for (int pg = 0; pg < t.np; ++pg) {
#pragma unroll
          for (int vb = 0; vb < kMtcDv / 128; ++vb) {
            // V^T block vb: value columns 128 vb .. +127 (column blocks 2 vb, 2 vb + 1,
            // kMtcCbStride apart) over the page's 16 keys (two 8-key groups, 1024 B apart)
            const uint64_t ad = umma_sdesc_sw128(vb0 + static_cast<uint32_t>(2 * vb) * kMtcCbStride +
                                                     static_cast<uint32_t>(pg) * kMtcTile,
                                                 kMtcCbStride, 1024u);
            const uint32_t tO = tbase + kMtcTmemO + static_cast<uint32_t>(vb * RP);
#pragma unroll
            for (int h = 0; h < NPT; ++h) {
              const uint64_t bd = umma_sdesc_sw128(pb + static_cast<uint32_t>(h) * kPbuf + 32u * pg, 16u, 1024u);
              umma_ss(tO, ad, bd, idesc, !(t.first && pg == 0 && h == 0));
            }
          }
        }
        umma_commit(pfree_bar(b & 1));
        umma_commit(bfree_bar(b & 1));
      }
      __syncwarp();
      ++b;
    }
    if (!ok && lane == 0) atomicOr(p.err, kErrTimeout);
    if (lane == 0) umma_commit(drain2_bar);
    __syncwarp();
    if (!mtc_wait(drain2_bar, 0u, p.wait_ns) && lane == 0) atomicOr(p.err, kErrTimeout);
  } else {
    // ============================ softmax ==================================
    const int q4 = warp & 3;                 // tensor-memory lane quarter of this warp
    const int rho = 32 * q4 + lane;          // query row = lane of S and Q
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const uint32_t tS = tbase + lane_off + kMtcTmemS;
    const uint32_t tQ = tbase + lane_off + kMtcTmemQ;
    const uint32_t tO = tbase + lane_off + kMtcTmemO;
    const float c = p.scale_log2;
    BlockWalker wk(s_pre, B, NC, start, count, kMtcBlockPages);
    int b = 0, seg = -1;
    SeqInfo si = {0, 0, 0, 0};
    bool row_ok = false, fine = true;
    int lim = 0, seg_j0 = 0, seg_c = 0;
    int64_t seg_k0 = 0;
    float m = -INFINITY, l = 0.f;
    bool ok = true;

    // Row rho of the segment starting at block t into tensor memory (the A
    // operand of Q K^T; fp8 caches: f16 with a range check), zeros past R.
    auto stage_q = [&](const TcBlock& t) {
      const SeqInfo s2 = seq_info(p, s_len, s_qsl, t.i, false, 0);
      const bool have = rho < G * s2.qn;
      const uint4* src = nullptr;
      if (have)
        src = reinterpret_cast<const uint4*>(p.q + static_cast<int64_t>(s2.t0 + rho / G) * p.q_stride_t +
                                             static_cast<int64_t>(t.c * G + rho % G) * kMtcDqk);
#pragma unroll 1
      for (int k = 0; k < kMtcDqk / 32; ++k) {   // 16 columns (32 features) at a time
        uint32_t w[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 v = have ? src[4 * k + u] : make_uint4(0u, 0u, 0u, 0u);
          w[4 * u] = v.x;
          w[4 * u + 1] = v.y;
          w[4 * u + 2] = v.z;
          w[4 * u + 3] = v.w;
        }
        if constexpr (FP8) {
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = bf16x2_to_f16x2(w[e], fine);
        }
        tmem_st16(tQ + 16u * k, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(qfull_bar);
    };

    while (wk.more()) {
      const TcBlock t = wk.next(s_pre, B, NC);
      if (t.first) {
        ++seg;
        if (seg == 0) stage_q(t);
        si = seq_info(p, s_len, s_qsl, t.i, rho == 0, 0);
        row_ok = rho < G * si.qn;
        lim = si.L - si.qn + (row_ok ? rho / G : 0);
        seg_j0 = t.j0;
        seg_k0 = t.k0;
        seg_c = t.c;
        m = -INFINITY;
        l = 0.f;
        if (seg_j0 == 0 && rho == 0) {
          // This CTA holds the unit's first page: describe the unit for the merge.
          const int64_t a = static_cast<int64_t>(NC) * s_pre[t.i] + static_cast<int64_t>(t.c) * t.n;
          const int last_cta = static_cast<int>(((a + t.n) * NG - 1) / X);
          p.ws_unit[static_cast<int64_t>(t.i) * NC + t.c] =
              make_int4(g, (last_cta - g + 1) | (t.k0 != 0 ? (1 << 30) : 0), si.t0, si.qn);
        }
      }
      // ---- S row of the block (every phase of S seen in order) ----------------
      if (!mtc_wait(sfull_bar, static_cast<uint32_t>(b) & 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[4][16];
      {
        uint32_t r[4][16];
#pragma unroll
        for (int k = 0; k < 4; ++k) tmem_ld16(tS + 16u * k, r[k]);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int e = 0; e < 16; ++e) sv[k][e] = __uint_as_float(r[k][e]);
      }
      // ---- mask and block max (interior blocks: no per-key mask, the scale
      // folded into the exponent) -------------------------------------------------
      const int tb = kPage * t.j0;
      const bool interior = t.np == kMtcBlockPages && c > 0.f && tb + kMtcBlockPages * kPage <= si.L - si.qn + 1;
      float mb;
      {
        float mx[64];
        if (interior) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int e = 0; e < 16; ++e) mx[16 * k + e] = sv[k][e];
          mb = Max3Tree<64>::run(mx) * c;
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int tok = tb + 16 * k + e;
              const bool vis = row_ok && k < t.np && tok <= lim;
              const float x = vis ? sv[k][e] * c : -INFINITY;
              sv[k][e] = x;
              mx[16 * k + e] = x;
            }
          mb = Max3Tree<64>::run(mx);
        }
      }
      if (!row_ok) mb = -INFINITY;
      const float m_new = fmaxf(m, mb);
      const bool grow = m_new > m + 8.f;     // also true when m = -inf and m_new is finite
      float alpha = 1.f;
      if (grow) {
        alpha = fast_exp2(m - m_new);        // 0 when m = -inf
        l *= alpha;
        m = m_new;
      }
      // publish: this row's O factor and whether this warp needs an O rescale
      // (a segment's first block has no O history: its P V overwrites O)
      x_alpha[(b & 1) * 128 + rho] = alpha;
      const bool need = __any_sync(0xffffffffu, grow && !t.first && row_ok);
      if (lane == 0) x_flag[(b & 1) * 4 + q4] = need ? 1u : 0u;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfree_bar);
      if (!mtc_wait(sfree_bar, static_cast<uint32_t>(b) & 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      const bool any = (x_flag[(b & 1) * 4 + 0] | x_flag[(b & 1) * 4 + 1] | x_flag[(b & 1) * 4 + 2] |
                        x_flag[(b & 1) * 4 + 3]) != 0u;
      if (any) {
        // ---- lazy O rescale: O must hold P V of block b - 1 first (this warp
        // saw block b - 3's completion, the previous phase, at block b - 1) ----
        if (!mtc_wait(pfree_bar((b - 1) & 1), static_cast<uint32_t>((b - 1) >> 1) & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* al = x_alpha + (b & 1) * 128;
#pragma unroll 1
        for (int vb = 0; vb < kMtcDv / 128; ++vb) {
#pragma unroll
          for (int h = 0; h < RP / 16; ++h) {
            uint32_t r[16];
            const uint32_t ta = tO + static_cast<uint32_t>(vb * RP + 16 * h);
            tmem_ld16(ta, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * al[16 * h + e]);
            tmem_st16(ta, r);
          }
        }
        tmem_wait_st();
      }
      // ---- P buffer b % 2: free once P V of block b - 2 is done (its
      // previous phase, block b - 4, seen at block b - 2) --------------------------
      if (b >= 2 && !mtc_wait(pfree_bar(b & 1), static_cast<uint32_t>((b >> 1) - 1) & 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      {
        const float mneg = m == -INFINITY ? 0.f : -m;
        const float mult = interior ? c : 1.f;   // masked scores are already scaled
        const uint64_t mult2 = f2_pack(mult, mult), mneg2 = f2_pack(mneg, mneg);
        uint64_t lsum2 = f2_pack(0.f, 0.f);
        const uint32_t prow = pbuf0 + static_cast<uint32_t>(b & 1) * NPT * kPbuf +
                              static_cast<uint32_t>(rho >> 3) * 1024u + static_cast<uint32_t>(rho & 7) * 128u;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {       // 8 keys (one 16-byte chunk of the P row) at a time
          uint32_t w[4], wl[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = ch >> 1, i0 = 8 * (ch & 1) + 2 * e;
            float x0, x1;
            f2_unpack(ffma2(f2_pack(sv[k][i0], sv[k][i0 + 1]), mult2, mneg2), x0, x1);
            float a0 = fast_exp2(x0), a1 = fast_exp2(x1);
            if (!row_ok) a0 = a1 = 0.f;
            lsum2 = fadd2(lsum2, f2_pack(a0, a1));
            if constexpr (FP8) {
              w[e] = pack_f16(a0, a1);
            } else {
              w[e] = pack_bf16(a0, a1);
              float r0, r1;   // exact residues a - bf16(a), rounded once below
              f2_unpack(ffma2(f2_pack(bf16_lo(w[e]), bf16_hi(w[e])), f2_pack(-1.f, -1.f), f2_pack(a0, a1)), r0, r1);
              wl[e] = pack_bf16(r0, r1);
            }
          }
          if (rho < RP) {
            const uint32_t off = static_cast<uint32_t>((ch ^ (rho & 7)) << 4);
            sts128(prow + off, make_uint4(w[0], w[1], w[2], w[3]));
            if constexpr (!FP8) sts128(prow + kPbuf + off, make_uint4(wl[0], wl[1], wl[2], wl[3]));
          }
        }
        float s0, s1;
        f2_unpack(lsum2, s0, s1);
        l += s0 + s1;
      }
      fence_proxy_async_smem();   // the P V MMA reads what these stores wrote
      __syncwarp();
      if (lane == 0) mbar_arrive(pfull_bar(b & 1));

      if (t.last) {
        // Every Q K^T of this segment is complete (S of its last block was read
        // above): the next segment's Q goes in now.
        if (wk.more()) {
          BlockWalker peek = wk;
          const TcBlock nt = peek.next(s_pre, B, NC);
          stage_q(nt);
        }
        // O complete once P V of this block is done (previous phase, block
        // b - 2, seen above)
        if (!mtc_wait(pfree_bar(b & 1), static_cast<uint32_t>(b >> 1) & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        x_stat[rho] = make_float2(m, l);
        __syncwarp();
        if (lane == 0) mbar_arrive(ebar);
        if (!mtc_wait(ebar, static_cast<uint32_t>(seg) & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool complete = (seg_j0 == 0) && (t.j0 + t.np == t.n);
        const int R = G * si.qn;
        const int which = (seg_k0 == 0) ? 0 : 1;
        const int64_t rowbase = static_cast<int64_t>(2 * g + which) * p.R_max;
#pragma unroll 1
        for (int vb = 0; vb < kMtcDv / 128; ++vb) {
          const int col = 128 * vb + rho;   // this thread's value column (its lane of O^T)
#pragma unroll
          for (int h = 0; h < RP / 16; ++h) {
            uint32_t r[16];
            tmem_ld16(tO + static_cast<uint32_t>(vb * RP + 16 * h), r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int rr = 16 * h + e;
              if (rr >= R) continue;
              const float2 st = x_stat[rr];
              const float o = __uint_as_float(r[e]);
              if (complete) {
                const float inv = st.y > 0.f ? p.v_scale / st.y : 0.f;
                const int tok = si.t0 + rr / G;
                const int hq = seg_c * G + rr % G;
                p.out[static_cast<int64_t>(tok) * p.out_stride_t + static_cast<int64_t>(hq) * p.out_stride_h + col] =
                    static_cast<uint16_t>(pack_bf16(o * inv, 0.f) & 0xFFFFu);
              } else {
                const float inv = st.y > 0.f ? 1.f / st.y : 0.f;
                reinterpret_cast<uint16_t*>(p.ws_o)[(rowbase + rr) * kMtcDv + col] =
                    static_cast<uint16_t>(pack_f16(o * inv, 0.f) & 0xFFFFu);
              }
            }
          }
        }
        if (row_ok) {
          const int tok = si.t0 + rho / G;
          const int hq = seg_c * G + rho % G;
          if (complete) {
            if (p.lse != nullptr)
              p.lse[static_cast<int64_t>(tok) * p.lse_stride_t + static_cast<int64_t>(hq) * p.lse_stride_h] =
                  l > 0.f ? (m + fast_log2(l)) * 0.69314718055994530942f : -INFINITY;
          } else {
            p.ws_ml[rowbase + rho] = make_float2(m, l);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ofree_bar);
      }
      ++b;
    }
    if (!fine) atomicOr(p.err, kErrF16Range);
    if (!ok && lane == 0) atomicOr(p.err, kErrTimeout);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMtcQkWarp) tmem_dealloc(tbase, kMtcCols);
}

template <bool FP8, int RP>
static cudaError_t launch_mla_tc_one(const CUtensorMap& tm, const SplitParams& p, int grid, int smem, bool pdl,
                                     cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kMtcThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, pa_mla_tc_kernel<FP8, RP>, tm, p);
}

int mla_tc_threads() { return kMtcThreads; }

cudaError_t launch_mla_tc(bool fp8, int rpad, const CUtensorMap& tm, const SplitParams& p, int grid, int smem,
                          bool pdl, cudaStream_t stream) {
  if (rpad == 16) return fp8 ? launch_mla_tc_one<true, 16>(tm, p, grid, smem, pdl, stream)
                             : launch_mla_tc_one<false, 16>(tm, p, grid, smem, pdl, stream);
  if (rpad == 32) return fp8 ? launch_mla_tc_one<true, 32>(tm, p, grid, smem, pdl, stream)
                             : launch_mla_tc_one<false, 32>(tm, p, grid, smem, pdl, stream);
  return cudaErrorInvalidValue;
}

cudaError_t set_mla_tc_smem_limits(int smem) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(pa_mla_tc_kernel<false, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(pa_mla_tc_kernel<false, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(pa_mla_tc_kernel<true, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
      cudaSuccess)
    return e;
  return cudaFuncSetAttribute(pa_mla_tc_kernel<true, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace pa
