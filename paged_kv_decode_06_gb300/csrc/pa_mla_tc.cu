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
// A block is up to 3 pages (48 keys) of one segment.  Per block:
//   S[128 x 16np]     = Q[128 x 576] K^T        36 TS-MMAs (Q in tensor memory)
//   O^T[vb][128 x R]  += V^T[vb] P^T            4 SS-MMAs a page (P in f16 for fp8
//                                                caches, bf16 for bf16 caches, as the
//                                                mma.sync MLA kernel carries it)
// Tensor memory (512 columns): O^T [0, 4 R_pad), S [4 R_pad, +64) (two S
// buffers [64, 192) for R_pad = 16), Q [192, 480).
//
// A block's rows sit in one of three block buffers in the MMA layout
// ([column block][page][16 rows x 128 B], 128-byte swizzle), so the rows of the
// next two blocks arrive while a block is computed.
// Roles (352 threads):
//   bf16 caches: warps 0, 3, 8-10 producers: block-table lookups and one TMA
//               box (16 rows x 64 features) per page and column block, straight
//               into the block's buffer, the boxes dealt one a lane over the five
//               warps;
//   fp8 caches: warp 0 producer: one TMA box per page (the whole 16 x 576 row
//               block) into a ring of raw page slots; warps 3, 8-10 converters:
//               each raw page into the block's buffer, codes to f16 (exact),
//               rows past the sequence end zeroed;
//   warp 1      Q K^T issuer, owner of the tensor-memory allocation;
//   warp 2      P V issuer (bf16 caches: zeroes the value rows past the
//               sequence end first);
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
constexpr int kMtcBlockPages = 3;
constexpr int kMtcNbuf = 3;                       // block buffers
constexpr uint32_t kMtcTile = 2048;               // MMA layout: one page of one column block, 16 x 128 B
constexpr uint32_t kMtcCbStride = kMtcBlockPages * kMtcTile;
constexpr uint32_t kMtcBuf = kMtcCb * kMtcCbStride;   // one block's rows in the MMA layout (54 KB)
constexpr int kMtcThreads = 352;
constexpr int kMtcProducer = 0, kMtcQkWarp = 1, kMtcPvWarp = 2, kMtcSoftmax0 = 4;
constexpr int kMtcTmemUsers = 6;                   // warps 1, 2, 4..7 (named barrier 1 at set-up)
constexpr int kMtcConverters = 4;                 // fp8: warps 3, 8, 9, 10
constexpr int kMtcBoxProducers = 5;               // bf16: warps 0, 3, 8, 9, 10
constexpr uint32_t kMtcCols = 512;
constexpr uint32_t kMtcTmemO = 0, kMtcTmemQ = 176;   // S: see mtc_tmem_s
constexpr int kMtcQsteps = kMtcDqk / 16;          // k-steps of Q K^T
// Q staging ring: a slot holds one 96-feature slice (192 B) of every row, rows
// 208 B apart (odd multiple of 16 B: the 16-byte reads of 8 lanes hit
// distinct banks)
constexpr int kMtcQslices = 6;
constexpr uint32_t kMtcQsliceBytes = kMtcDqk * 2 / kMtcQslices;
constexpr uint32_t kMtcQrow = kMtcQsliceBytes + 16;
static_assert(kMtcQsliceBytes % 64 == 0, "a slice is whole groups of 16 tensor-memory columns");

__device__ __forceinline__ int converter_index(int warp) { return warp == 3 ? 0 : warp - 7; }
__device__ __forceinline__ int box_producer_index(int warp) { return warp == 0 ? 0 : (warp == 3 ? 1 : warp - 6); }

// Tensor memory (512 columns): O^T at 0 (4 x R_pad columns), Q at 176 (288
// columns), two S buffers of 48 columns (Q K^T of the next block runs while
// the softmax reads this one): at 64 and 128 for 16-row units, at 128 and
// 464 for 32-row units.  Tensor-memory column of S buffer x.
template <int RP>
__device__ __forceinline__ constexpr uint32_t mtc_tmem_s(int x) {
  return RP == 16 ? 64u + 64u * static_cast<uint32_t>(x) : (x == 0 ? 128u : 464u);
}

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

// 16 bytes global -> shared without a register round trip (L2 only); this
// thread's copies complete in commit-group order.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}
// An arrival on `bar` once every earlier copy of this thread has landed (the
// barrier's expected count includes it).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Has the phase with the given parity completed?  Never suspends the thread.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// f16x2 -> its two floats (exact).
__device__ __forceinline__ void f16x2_unpack(uint32_t x, float& lo, float& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(x));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// mbarrier.try_wait with a suspend-time hint: a thread whose phase is not
// complete may sleep up to hint_ns (it resumes when the phase completes), so
// waiting warps leave the issue slots of their SM sub-partition to the warps
// that work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait of all lanes of a warp (kErrTimeout after limit_ns).
__device__ __forceinline__ bool mtc_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  bool done = mbar_try_wait_sleep(bar, parity, 4096u);
  if (!done) {
    const uint64_t t0 = global_timer_ns();
    while (!(done = mbar_try_wait_sleep(bar, parity, 4096u)))
      if (global_timer_ns() - t0 > limit_ns) break;
  }
  return __all_sync(0xffffffffu, done);
}

// Work split.  The flattened positions (sequence, head chunk, page) are cut
// into contiguous ranges, one a CTA, of equal cost: a position costs one
// page, and every unit (sequence, head chunk) but the first adds W just
// before its first page, since a CTA pays for every unit it opens (a Q
// staging, an epilogue, a pipeline refill).  Cost prefix of x: the positions
// before x plus W for each unit after the first that starts at or before x.
// Inside a unit the prefix grows by one a page, so (with at most one CTA a
// page of cost) the CTAs holding a unit's pages are consecutive and none of
// them is empty.  Units of sequences without pages count too, which keeps
// the prefix a plain non-decreasing function of the position.
__device__ __forceinline__ int64_t split_cost(const int32_t* pre, int B, int NC, int64_t W, int64_t x, int64_t X) {
  if (x >= X) return X + W * (static_cast<int64_t>(NC) * B - 1);
  const Cursor cu = locate(pre, B, NC, x);
  return x + W * (static_cast<int64_t>(NC) * cu.i + cu.c);
}

// First position x in [0, X] whose cost prefix reaches gi / NG of the total:
// the first sequence whose last position reaches it (a binary search over
// the sequences), then the head chunk and page by arithmetic (inside a
// sequence of n pages the prefix runs over chunks of n pages, W apart).
__device__ int64_t split_point(const int32_t* pre, int B, int NC, int64_t W, int64_t X, int NG, int gi) {
  const int64_t total = X + W * (static_cast<int64_t>(NC) * B - 1);
  const int64_t tau = (static_cast<int64_t>(gi) * total + NG - 1) / NG;   // cost prefix >= tau
  int lo = 0, hi = B;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int64_t last = static_cast<int64_t>(NC) * pre[mid + 1] - 1 + W * (static_cast<int64_t>(NC) * mid + NC - 1);
    if (last >= tau) hi = mid; else lo = mid + 1;
  }
  if (lo == B) return X;
  const int64_t n = pre[lo + 1] - pre[lo];
  const int64_t s0 = static_cast<int64_t>(NC) * pre[lo];
  if (n == 0) return s0;
  const int64_t d = tau - (s0 + W * NC * lo);
  if (d <= 0) return s0;
  const int64_t c = d / (n + W), r = d - c * (n + W);
  return r < n ? s0 + c * n + r : s0 + (c + 1) * n;
}

// bf16x2 -> f16x2 with a flag for values beyond the f16 range.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x, bool& fine) {
  const uint32_t r = pack_f16(bf16_lo(x), bf16_hi(x));
  fine &= ((r & 0x7C00u) != 0x7C00u) && ((r & 0x7C000000u) != 0x7C000000u);
  return r;
}

}  // namespace

// Shared-memory layout (bytes from the 1024-aligned base), host and device:
//   off_buf   3 x kMtcBuf          the block buffers in the MMA layout
//   off_q     P buffers            2 (block parity) x R_pad x 128 B
//   off_stage raw page slots       fp8: nstage x 16 x 576 bytes, as the TMA box lands
//   off_qring Q staging ring       q_slots x R_pad rows x 208 B (a 192-byte slice of each row)
//   off_bar   barriers
//   off_xchg  softmax exchange     alpha [4][32] f32, flags [4][4] u32, row factors [32] f32,
//                                  row outputs [32] pointers
//   off_prefix sequence metadata
template <bool FP8, int RP>
__global__ void __launch_bounds__(kMtcThreads, 1)
    pa_mla_tc_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_box,
                     const SplitParams p) {
  constexpr int ESZ = FP8 ? 1 : 2;
  constexpr uint32_t kRawPage = kPage * kMtcDqk * ESZ;   // one TMA box: [9 blocks][16 rows][64 x esz B]
  constexpr uint32_t kRawBlock = 16u * 64u * ESZ;
  constexpr int NPT = 1;                                 // P terms
  constexpr uint32_t kPbuf = static_cast<uint32_t>(RP) * 128u;
  constexpr int NSB = 2;                                 // S buffers
  constexpr uint32_t kS = 16u * kMtcBlockPages;          // columns of an S buffer
  static_assert(kMtcTmemO + 4u * RP <= mtc_tmem_s<RP>(0) && mtc_tmem_s<RP>(0) + kS <= kMtcTmemQ &&
                    (RP == 32 || mtc_tmem_s<RP>(1) + kS <= kMtcTmemQ) &&
                    kMtcTmemQ + kMtcDqk / 2 <= kMtcCols && (RP == 16 || (kMtcTmemQ + kMtcDqk / 2 <= mtc_tmem_s<RP>(1) &&
                                                                          mtc_tmem_s<RP>(1) + kS <= kMtcCols)),
                "tensor-memory regions overlap");
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_scan[kMtcThreads / 32 + 1];
  __shared__ int s_total;
  __shared__ uint32_t s_tmem;
  __shared__ int64_t s_split[2];

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
  // block buffer x (blocks b with b % 3 == x, phase b / 3): filled (fp8: 4
  // converter warps; bf16: 5 producer warps and their bytes); read by both
  // MMAs (commit)
  auto cfull_bar = [&](int x) { return xb + 8u * x; };
  auto bfree_bar = [&](int x) { return xb + 8u * (3 + x); };
  // P buffer x (blocks b with b % 2 == x): written (4 softmax warps); P V of
  // the block done (commit)
  auto pfull_bar = [&](int x) { return xb + 8u * (6 + x); };
  auto pfree_bar = [&](int x) { return xb + 8u * (8 + x); };
  // per S buffer x (blocks b with b % NSB == x, phase b / NSB): S in tensor
  // memory (commit); S read and the block's statistics published (4 warps)
  auto sfull_bar = [&](int x) { return xb + 8u * (10 + x); };
  auto sfree_bar = [&](int x) { return xb + 8u * (12 + x); };
  const uint32_t qfull_bar = xb + 8u * 14;                      // a segment's Q in tensor memory (its stager)
  const uint32_t ebar = xb + 8u * 15;                           // a segment's row statistics published (4 warps)
  const uint32_t ofree_bar = xb + 8u * 16;                      // O read by a segment's epilogue (4 warps)
  const uint32_t drain_bar = xb + 8u * 17;
  const uint32_t drain2_bar = xb + 8u * 18;
  auto qbar = [&](int x) { return xb + 8u * (19 + x); };       // Q ring slot x landed (32 lanes)
  const uint32_t qst0 = base + p.off_qring;
  const uint32_t qslot = static_cast<uint32_t>(RP) * kMtcQrow;
  // the softmax exchange, by block b % 4: a buffer is rewritten four blocks
  // later, after every softmax warp has passed block b + 2 (two S buffers) or
  // b + 1 (one), and so finished block b
  float* const x_alpha = reinterpret_cast<float*>(gbase + p.off_xchg);              // [4][32]
  uint32_t* const x_flag = reinterpret_cast<uint32_t*>(gbase + p.off_xchg + 2048);  // [4][4]
  float* const x_fac = reinterpret_cast<float*>(gbase + p.off_xchg + 2304);         // [32] output factor of a row
  uint16_t** const x_dst = reinterpret_cast<uint16_t**>(gbase + p.off_xchg + 2432);  // [32] output row of a row

  if (tid == 0) {
    prefetch_tensormap(FP8 ? &tmap : &tmap_box);
    for (int s = 0; s < nstage; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kMtcConverters);
    }
    for (int x = 0; x < kMtcNbuf; ++x) {
      mbar_init(cfull_bar(x), FP8 ? kMtcConverters : kMtcBoxProducers);
      mbar_init(bfree_bar(x), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(pfull_bar(x), 4);
      mbar_init(pfree_bar(x), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(sfull_bar(x), 1);
      mbar_init(sfree_bar(x), 4);
    }
    mbar_init(qfull_bar, 1);
    for (int x = 0; x < p.q_slots; ++x) mbar_init(qbar(x), 32);
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
  const int64_t W = p.seg_cost;
  const int64_t Ctot = split_cost(s_pre, B, NC, W, X, X);
  if (tid < 2) s_split[tid] = split_point(s_pre, B, NC, W, X, NG, g + tid);
  __syncthreads();
  const int64_t start = s_split[0];
  const int64_t end = s_split[1];
  const int64_t count = end - start;
  if (count <= 0) return;

  if (warp == kMtcSoftmax0) {
    // the Q rows of this CTA's first segments start towards L2 while tensor
    // memory is set up (a later staging then waits on L2, not on HBM)
    int64_t x = start;
    for (int sg = 0; sg < 4 && x < end; ++sg) {
      const Cursor cs = locate(s_pre, B, NC, x);
      const SeqInfo s0 = seq_info(p, s_len, s_qsl, cs.i, false, 0);
      if (lane < G * s0.qn) {
        const uint16_t* const src = p.q + static_cast<int64_t>(s0.t0 + lane / G) * p.q_stride_t +
                                    static_cast<int64_t>(cs.c * G + lane % G) * kMtcDqk;
#pragma unroll
        for (int k = 0; k < kMtcDqk * 2 / 128; ++k) prefetch_l2(src + 64 * k);
      }
      x += cs.n - cs.j;
    }
  }
  // fp8: only the tensor-memory users (Q K^T and P V issuers, softmax warps)
  // wait for the allocation, so the page producer and the converters start
  // at once (measured faster); bf16: the whole CTA waits (measured faster:
  // an earlier flood of box loads delays the first Q).
  const bool tmem_user = !FP8 || warp == kMtcQkWarp || warp == kMtcPvWarp ||
                         (warp >= kMtcSoftmax0 && warp < kMtcSoftmax0 + 4);
  uint32_t tbase = 0;
  if (tmem_user) {
    if (warp == kMtcQkWarp) tmem_alloc(smem_addr(&s_tmem), kMtcCols);
    tc_fence_before();
    if constexpr (FP8) {
      asm volatile("bar.sync 1, %0;" ::"n"(kMtcTmemUsers * 32) : "memory");
    } else {
      __syncthreads();
    }
    tc_fence_after();
    tbase = warp_uniform(s_tmem);
  }
  const uint32_t buf0 = base + p.off_buf;
  const uint32_t pbuf0 = base + p.off_q;
  const uint32_t ring0 = base + p.off_stage;   // raw page slots

  if (!FP8 && (warp == 0 || warp == 3 || warp >= kMtcSoftmax0 + 4)) {
    // ==================== bf16: box producers ==============================
    // Box x of a block (page x / 9, column block x % 9) goes to producer warp
    // x % 5, lane x / 5; each warp announces its own bytes on the block's full
    // barrier, then its lanes issue their boxes.
    const int pw = box_producer_index(warp);
    BlockWalker wk(s_pre, B, NC, start, count, kMtcBlockPages);
    BlockTableCache btc;
    int b = 0;
    bool ok = true;
    while (wk.more()) {
      const TcBlock t = wk.next(s_pre, B, NC);
      const int x = b % kMtcNbuf;
      // buffer x was last read by the MMAs of block b - 3 (its previous phase,
      // block b - 6, seen at block b - 3)
      if (b >= kMtcNbuf && !mtc_wait(bfree_bar(x), static_cast<uint32_t>(b / kMtcNbuf - 1) & 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      int phys[kMtcBlockPages];
#pragma unroll
      for (int pg = 0; pg < kMtcBlockPages; ++pg) {
        phys[pg] = 0;
        if (pg < t.np) {
          Cursor pc;
          pc.i = t.i;
          pc.c = t.c;
          pc.j = t.j0 + pg;
          pc.n = t.n;
          phys[pg] = btc.lookup(p, pc, s_pre, s_len, s_qsl, B, NC, 0, lane);
          if ((phys[pg] < 0 || phys[pg] >= p.num_pages) && lane == 0 && pw == 0) atomicOr(p.err, kErrPageRange);
        }
      }
      const int nbox = t.np * kMtcCb;
      const int mine = nbox > pw ? (nbox - pw + kMtcBoxProducers - 1) / kMtcBoxProducers : 0;
      if (lane == 0) mbar_arrive_expect_tx(cfull_bar(x), static_cast<uint32_t>(mine) * kMtcTile);
      __syncwarp();
      const int bx = kMtcBoxProducers * lane + pw;
      if (bx < nbox) {
        const int pg = bx / kMtcCb, cb = bx - pg * kMtcCb;
        int ph = phys[0];
#pragma unroll
        for (int q = 1; q < kMtcBlockPages; ++q) ph = pg == q ? phys[q] : ph;
        // an out-of-range page id reads zeros (TMA fills outside the tensor)
        tma_load_4d(buf0 + static_cast<uint32_t>(x) * kMtcBuf + static_cast<uint32_t>(cb) * kMtcCbStride +
                        static_cast<uint32_t>(pg) * kMtcTile,
                    &tmap_box, 0, 0, cb, ph, cfull_bar(x));
      }
      ++b;
    }
    if (!ok && lane == 0) atomicOr(p.err, kErrTimeout);
  } else if (FP8 && warp == kMtcProducer) {
    // ==================== fp8: page producer ===============================
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
  } else if (FP8 && (warp == 3 || warp >= kMtcSoftmax0 + 4)) {
    // ==================== fp8: converters ==================================
    // A page is split into 16-byte source chunks dealt over the 128 converter
    // threads.
    constexpr int kChunks = kMtcCb * 16 * 4;   // 16-byte source chunks of an fp8 page
    constexpr int kPer = (kChunks + 127) / 128;
    const int ct = converter_index(warp) * 32 + lane;   // 0..127
    BlockWalker wk(s_pre, B, NC, start, count, kMtcBlockPages);
    int b = 0, stage = 0;
    uint32_t round = 0;
    bool ok = true;
    while (wk.more() && ok) {
      const TcBlock t = wk.next(s_pre, B, NC);
      const int xbuf = b % kMtcNbuf;
      // buffer xbuf was last read by the MMAs of block b - 3 (this warp saw
      // the completion of block b - 6's, the previous phase, at block b - 3)
      if (b >= kMtcNbuf && !mtc_wait(bfree_bar(xbuf), static_cast<uint32_t>(b / kMtcNbuf - 1) & 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      uint8_t* const dst0 = gbase + p.off_buf + static_cast<uint32_t>(xbuf) * kMtcBuf;
      const int L = s_len[t.i];
#pragma unroll 1
      for (int pg = 0; pg < t.np; ++pg) {
        if (!mtc_wait(full_bar(stage), round & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        const uint8_t* const src = gbase + p.off_stage + static_cast<uint32_t>(stage) * kRawPage;
        uint8_t* const dst = dst0 + static_cast<uint32_t>(pg) * kMtcTile;
        const int vt = L - kPage * (t.j0 + pg);   // rows of this page inside the sequence
        uint4 v[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {   // all loads first, then all stores
          const int x = ct + 128 * i;
          const int cb = x >> 6, r = (x >> 2) & 15, c = x & 3;
          v[i] = make_uint4(0u, 0u, 0u, 0u);
          if (x < kChunks && r < vt) v[i] = *reinterpret_cast<const uint4*>(src + cb * kRawBlock + swz<64>(r, c));
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int x = ct + 128 * i;
          if (x < kChunks) {
            // 16 codes (a 64-byte-swizzled chunk) -> 16 f16 values (two chunks of
            // the 128-byte-swizzled MMA row); exact
            const int cb = x >> 6, r = (x >> 2) & 15, c = x & 3;
            uint8_t* const d = dst + cb * kMtcCbStride;
            const uint4 w = v[i];
            *reinterpret_cast<uint4*>(d + swz<128>(r, 2 * c)) =
                make_uint4(e4m3x2_to_f16x2(w.x), e4m3x2_to_f16x2(w.x >> 16), e4m3x2_to_f16x2(w.y),
                           e4m3x2_to_f16x2(w.y >> 16));
            *reinterpret_cast<uint4*>(d + swz<128>(r, 2 * c + 1)) =
                make_uint4(e4m3x2_to_f16x2(w.z), e4m3x2_to_f16x2(w.z >> 16), e4m3x2_to_f16x2(w.w),
                           e4m3x2_to_f16x2(w.w >> 16));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(stage));
        if (++stage == nstage) {
          stage = 0;
          ++round;
        }
      }
      if (!ok) break;
      fence_proxy_async_smem();   // the tensor cores read what these generic stores wrote
      __syncwarp();
      if (lane == 0) mbar_arrive(cfull_bar(xbuf));
      ++b;
    }
    if (!ok && lane == 0) atomicOr(p.err, kErrTimeout);
  } else if (warp == kMtcQkWarp) {
    // ============================ Q K^T issuer =============================
    const uint32_t idesc0 = mtc_idesc(128, 16, !FP8, false, false) & ~(0x3Fu << 17);
    const uint32_t tQ = tbase + kMtcTmemQ;
    BlockWalker wk(s_pre, B, NC, start, count, kMtcBlockPages);
    int b = 0, seg = -1;
    bool ok = true;
    while (wk.more()) {
      const TcBlock t = wk.next(s_pre, B, NC);
      if (t.first) ++seg;
      // converted rows of the block; its S buffer read by the softmax at block
      // b - NSB (that buffer's previous phase seen at block b - 2 NSB); at a
      // segment's first block its Q (every segment's phase seen in order)
      if (!mtc_wait(cfull_bar(b % kMtcNbuf), static_cast<uint32_t>(b / kMtcNbuf) & 1u, p.wait_ns) ||
          (b >= NSB && !mtc_wait(sfree_bar(b % NSB), static_cast<uint32_t>(b / NSB - 1) & 1u, p.wait_ns)) ||
          (t.first && !mtc_wait(qfull_bar, static_cast<uint32_t>(seg) & 1u, p.wait_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t kb = warp_uniform(buf0 + static_cast<uint32_t>(b % kMtcNbuf) * kMtcBuf);
      const uint64_t kd = umma_sdesc_sw128(kb, 16u, 1024u);
      const uint32_t idesc = warp_uniform(idesc0 | (static_cast<uint32_t>(2 * t.np) << 17));   // N = 16 np
      const uint32_t tS = warp_uniform(tbase + mtc_tmem_s<RP>(b % NSB));
      if (lane == 0) {
        // k-step s: features 16 s .. +15 = 32-byte slice (s % 4) of column block s / 4
#pragma unroll
        for (int s = 0; s < kMtcQsteps; ++s)
          umma_ts(tS, tQ + 8u * s, kd + ((static_cast<uint32_t>(s >> 2) * kMtcCbStride + (s & 3) * 32u) >> 4), idesc,
                  s > 0);
        umma_commit(sfull_bar(b % NSB));
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
          !mtc_wait(cfull_bar(b % kMtcNbuf), static_cast<uint32_t>(b / kMtcNbuf) & 1u, p.wait_ns) ||
          (t.first && seg >= 1 && !mtc_wait(ofree_bar, static_cast<uint32_t>(seg - 1) & 1u, p.wait_ns))) {
        ok = false;
        break;
      }
      const uint32_t vb0 = warp_uniform(buf0 + static_cast<uint32_t>(b % kMtcNbuf) * kMtcBuf);
      if constexpr (!FP8) {
        // Value rows past the context in the unit's last page: zero them so
        // that whatever the pool holds there cannot reach O through 0 * NaN
        // (Q K^T of this block, which also reads them, is complete: P exists).
        if (t.j0 + t.np == t.n) {
          const int vt = s_len[t.i] - kPage * (t.n - 1);
          if (vt < kPage) {
            uint8_t* const vg = gbase + (vb0 - base) + static_cast<uint32_t>(t.np - 1) * kMtcTile;
            const int nbytes = (kPage - vt) * 128;
            for (int cb = 0; cb < kMtcDv / 64; ++cb)
              for (int o = lane * 16; o < nbytes; o += 32 * 16)
                *reinterpret_cast<uint4*>(vg + cb * kMtcCbStride + vt * 128 + o) = make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
      }
      tc_fence_after();
      const uint32_t pb = warp_uniform(pbuf0 + static_cast<uint32_t>(b & 1) * NPT * kPbuf);
      // V^T block vb of page pg: value columns 128 vb .. +127 (column blocks
      // 2 vb, 2 vb + 1, kMtcCbStride apart) over the page's 16 keys (two 8-key
      // groups, 1024 B apart); P^T: the page's 32-byte slice of the P rows
      const uint64_t ad0 = umma_sdesc_sw128(vb0, kMtcCbStride, 1024u);
      const uint64_t bd0 = umma_sdesc_sw128(pb, 16u, 1024u);
      const uint32_t tO = tbase + kMtcTmemO;
      const bool first = t.first;
      const int np = t.np;
      if (lane == 0) {
#pragma unroll
        for (int pg = 0; pg < kMtcBlockPages; ++pg) {
          if (pg < np) {
#pragma unroll
            for (int vb = 0; vb < kMtcDv / 128; ++vb)
              umma_ss(tO + static_cast<uint32_t>(vb * RP),
                      ad0 + ((static_cast<uint32_t>(2 * vb) * kMtcCbStride + static_cast<uint32_t>(pg) * kMtcTile) >> 4),
                      bd0 + static_cast<uint32_t>(2 * pg), idesc, !(first && pg == 0));
          }
        }
        umma_commit(pfree_bar(b & 1));
        umma_commit(bfree_bar(b % kMtcNbuf));
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
    // Segment s keeps its Q rows, and so its S rows, in tensor-memory lane
    // quarter s % 2.  The softmax warp of that quarter owns the rows; the warp
    // of the other quarter meanwhile stages the next segment's Q into its own
    // lanes (rows the running Q K^T products compute but nothing reads).  Q
    // goes through a ring of shared-memory slots, one 96-feature slice of
    // every row a slot, filled by asynchronous copies a block ahead of their
    // use, so the staging rarely waits on a load.  Every warp owns 32 value columns of O^T (its
    // lanes) for the rescale and the epilogue.
    const int q4 = warp & 3;                 // tensor-memory lane quarter of this warp
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const uint32_t tQ = tbase + lane_off + kMtcTmemQ;
    const uint32_t tO = tbase + lane_off + kMtcTmemO;
    const float c = p.scale_log2;
    const int QR = p.q_slots;                // slots of the Q ring
    BlockWalker wk(s_pre, B, NC, start, count, kMtcBlockPages);
    int b = 0, seg = -1;
    SeqInfo si = {0, 0, 0, 0};
    bool act = false, row_ok = false, wact = false, fine = true;
    int lim = 0, seg_j0 = 0, seg_c = 0;
    int64_t seg_k0 = 0;
    float m = -INFINITY, l = 0.f, lr = 0.f;   // row max, row sum, row sum of the rounded weights
    bool ok = true;

    // Staging of segment qj's Q by this warp: slices issued and written.
    int qj = -1, q_iss = kMtcQslices, q_done = kMtcQslices;
    const uint16_t* q_src = nullptr;         // this lane's Q row (null past the rows)
    auto q_begin = [&](int i, int cc, int j) {
      const SeqInfo s2 = seq_info(p, s_len, s_qsl, i, false, 0);
      const int R2 = G * s2.qn;
      qj = j;
      q_iss = 0;
      q_done = 0;
      q_src = lane < R2 ? p.q + static_cast<int64_t>(s2.t0 + lane / G) * p.q_stride_t +
                              static_cast<int64_t>(cc * G + lane % G) * kMtcDqk
                        : nullptr;
    };
    // slice q_iss of this lane's row into its ring slot: 12 copies of 16 bytes
    // and an arrival on the slot's barrier once they land (every lane arrives);
    // slices of all stagings are numbered in order, and so are a slot's phases
    auto q_issue = [&]() {
      const int gs = kMtcQslices * qj + q_iss;
      const int x = gs % QR;
      const uint32_t dst = qst0 + static_cast<uint32_t>(x) * qslot + static_cast<uint32_t>(lane) * kMtcQrow;
      if (q_src != nullptr) {
        const uint16_t* const src = q_src + kMtcQsliceBytes / 2 * q_iss;
#pragma unroll
        for (int u = 0; u < static_cast<int>(kMtcQsliceBytes / 16); ++u) cp_async16(dst + 16u * u, src + 8 * u);
      }
      cp_async_arrive(qbar(x));
      ++q_iss;
    };
    // has slice q_done landed in every lane (no waiting)?
    auto q_ready = [&]() -> bool {
      const int gs = kMtcQslices * qj + q_done;
      return __all_sync(0xffffffffu, mbar_test(qbar(gs % QR), static_cast<uint32_t>(gs / QR) & 1u));
    };
    // slice q_done, landed, into this warp's lanes of tensor memory (each lane
    // reads back the row it copied; fp8 caches: f16 with a range check); the
    // last one announces the Q
    auto q_write = [&]() -> bool {
      const int gs = kMtcQslices * qj + q_done;
      const int x = gs % QR;
      if (!mtc_wait(qbar(x), static_cast<uint32_t>(gs / QR) & 1u, p.wait_ns)) return false;
      // lanes past the rows read row 0 and keep zeros, so the warp stays
      // converged for the tensor-memory stores
      const bool have = q_src != nullptr;
      const uint32_t row = qst0 + static_cast<uint32_t>(x) * qslot + (have ? static_cast<uint32_t>(lane) * kMtcQrow : 0u);
#pragma unroll
      for (int gq = 0; gq < kMtcQsliceBytes / 64; ++gq) {   // 16 tensor-memory columns at a time
        uint32_t w[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 v = lds128(row + 64u * gq + 16u * u);
          w[4 * u] = have ? v.x : 0u;
          w[4 * u + 1] = have ? v.y : 0u;
          w[4 * u + 2] = have ? v.z : 0u;
          w[4 * u + 3] = have ? v.w : 0u;
        }
        if constexpr (FP8) {
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = bf16x2_to_f16x2(w[e], fine);
        }
        __syncwarp();
        tmem_st16(tQ + static_cast<uint32_t>(16 * (kMtcQsliceBytes / 64 * q_done + gq)), w);
      }
      if (++q_done == kMtcQslices) {
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(qfull_bar);
      }
      return true;
    };
    // the rest of the staging, waiting on each slice
    auto q_finish = [&]() -> bool {
      while (q_done < kMtcQslices) {
        while (q_iss < kMtcQslices && q_iss - q_done < QR) q_issue();
        if (!q_write()) return false;
      }
      return true;
    };

    while (wk.more()) {
      const TcBlock t = wk.next(s_pre, B, NC);
      if (t.first) {
        ++seg;
        act = q4 == (seg & 1);
        if (seg == 0) {
          // the first segment's Q, into quarter 0; with a slot for every slice
          // the four warps issue the copies together, then warp 4 writes them
          q_begin(t.i, t.c, 0);
          if (QR >= kMtcQslices) {
            for (int k = q4; k < kMtcQslices; k += 4) {
              q_iss = k;
              q_issue();
            }
            q_iss = kMtcQslices;
          }
          if (q4 != 0) {
            q_done = kMtcQslices;
          } else if (!q_finish()) {
            ok = false;
            break;
          }
        }
        if (q4 == ((seg + 1) & 1) && t.k0 + (t.n - t.j0) < count) {
          // This warp stages the next segment's Q during this one, once this
          // segment's own staging is complete: the two share the ring (its
          // slots and their barriers).  This segment's phase of the Q barrier
          // is the last one before the phase this warp completes itself.
          if (!mtc_wait(qfull_bar, static_cast<uint32_t>(seg) & 1u, p.wait_ns)) {
            ok = false;
            break;
          }
          const Cursor nc = locate(s_pre, B, NC, start + t.k0 + (t.n - t.j0));
          q_begin(nc.i, nc.c, seg + 1);
        }
        si = seq_info(p, s_len, s_qsl, t.i, q4 == 0 && lane == 0, 0);
        row_ok = act && lane < G * si.qn;
        wact = __any_sync(0xffffffffu, row_ok);
        lim = si.L - si.qn + (row_ok ? lane / G : 0);
        seg_j0 = t.j0;
        seg_k0 = t.k0;
        seg_c = t.c;
        m = -INFINITY;
        l = 0.f;
        lr = 0.f;
        if (seg_j0 == 0 && q4 == 0 && lane == 0) {
          // This CTA holds the unit's first page: describe the unit for the merge.
          // the CTA holding the unit's last page, by the split's cost prefix
          const int64_t a = static_cast<int64_t>(NC) * s_pre[t.i] + static_cast<int64_t>(t.c) * t.n;
          const int64_t own = split_cost(s_pre, B, NC, W, a + t.n - 1, X) * NG / Ctot;
          const int last_cta = static_cast<int>(own < NG - 1 ? own : NG - 1);
          p.ws_unit[static_cast<int64_t>(t.i) * NC + t.c] =
              make_int4(g, (last_cta - g + 1) | (t.k0 != 0 ? (1 << 30) : 0), si.t0, si.qn);
        }
      }
      // the staging of the next segment's Q advances at every block
      const bool staging = qj == seg + 1 && q_done < kMtcQslices;
      if (staging)
        while (q_iss < kMtcQslices && q_iss - q_done < QR) q_issue();
      // ---- S row of the block (every phase of its S buffer seen in order) ------
      const int sx = b % NSB;
      const uint32_t tS = tbase + lane_off + mtc_tmem_s<RP>(sx);
      // A warp with no query row in this segment skips the S row, the maximum
      // and the exponentials; it keeps every barrier step.
      float sv[kMtcBlockPages][16];
      if (wact) {
        if (!mtc_wait(sfull_bar(sx), static_cast<uint32_t>(b / NSB) & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t r[kMtcBlockPages][16];
#pragma unroll
        for (int k = 0; k < kMtcBlockPages; ++k) tmem_ld16(tS + 16u * k, r[k]);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < kMtcBlockPages; ++k)
#pragma unroll
          for (int e = 0; e < 16; ++e) sv[k][e] = __uint_as_float(r[k][e]);
      }
      // ---- mask and block max (interior blocks: no per-key mask, the scale
      // folded into the exponent) -------------------------------------------------
      const int tb = kPage * t.j0;
      const bool interior = t.np == kMtcBlockPages && c > 0.f && tb + kMtcBlockPages * kPage <= si.L - si.qn + 1;
      float mb = -INFINITY;
      if (wact) {
        float mx[16 * kMtcBlockPages];
        if (interior) {
#pragma unroll
          for (int k = 0; k < kMtcBlockPages; ++k)
#pragma unroll
            for (int e = 0; e < 16; ++e) mx[16 * k + e] = sv[k][e];
          mb = Max3Tree<16 * kMtcBlockPages>::run(mx) * c;
        } else {
#pragma unroll
          for (int k = 0; k < kMtcBlockPages; ++k)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int tok = tb + 16 * k + e;
              const bool vis = row_ok && k < t.np && tok <= lim;
              const float x = vis ? sv[k][e] * c : -INFINITY;
              sv[k][e] = x;
              mx[16 * k + e] = x;
            }
          mb = Max3Tree<16 * kMtcBlockPages>::run(mx);
        }
      }
      if (!row_ok) mb = -INFINITY;
      const float m_new = fmaxf(m, mb);
      const bool grow = m_new > m + 8.f;     // also true when m = -inf and m_new is finite
      float alpha = 1.f;
      if (grow) {
        alpha = fast_exp2(m - m_new);        // 0 when m = -inf
        l *= alpha;
        lr *= alpha;
        m = m_new;
      }
      // publish: the rows' O factors and whether this warp needs an O rescale
      // (a segment's first block has no O history: its P V overwrites O)
      const int xq = b & 3;
      if (act) x_alpha[xq * 32 + lane] = alpha;
      const bool need = __any_sync(0xffffffffu, grow && !t.first && row_ok);
      if (lane == 0) x_flag[xq * 4 + q4] = need ? 1u : 0u;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfree_bar(sx));
      if (!mtc_wait(sfree_bar(sx), static_cast<uint32_t>(b / NSB) & 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      const uint4 fl = *reinterpret_cast<const uint4*>(x_flag + xq * 4);
      const bool any = (fl.x | fl.y | fl.z | fl.w) != 0u;
      if (any) {
        // ---- lazy O rescale: O must hold P V of block b - 1 first (this warp
        // saw block b - 3's completion, the previous phase, at block b - 1) ----
        if (!mtc_wait(pfree_bar((b - 1) & 1), static_cast<uint32_t>((b - 1) >> 1) & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* al = x_alpha + xq * 32;
#pragma unroll 1
        for (int vh = 0; vh < kMtcDv / 128 * (RP / 16); ++vh) {   // 16 columns of O^T at a time
          uint32_t r[16];
          const uint32_t ta = tO + static_cast<uint32_t>(16 * vh);
          const float* const a16 = al + 16 * (vh % (RP / 16));
          tmem_ld16(ta, r);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * a16[e]);
          tmem_st16(ta, r);
        }
        tmem_wait_st();
      }
      // ---- P buffer b % 2: free once P V of block b - 2 is done (its
      // previous phase, block b - 4, seen at block b - 2) --------------------------
      if (b >= 2 && !mtc_wait(pfree_bar(b & 1), static_cast<uint32_t>((b >> 1) - 1) & 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      if (wact) {
        // a row past the unit's rows gets zero weights through its exponent
        // argument: its scores are finite (zero query rows; masked ones -inf)
        const float mneg = row_ok ? (m == -INFINITY ? 0.f : -m) : -INFINITY;
        const float mult = interior ? c : 1.f;   // masked scores are already scaled
        const uint64_t mult2 = f2_pack(mult, mult), mneg2 = f2_pack(mneg, mneg);
        uint64_t lsum2 = f2_pack(0.f, 0.f), rsum2 = f2_pack(0.f, 0.f);
        const uint32_t prow = pbuf0 + static_cast<uint32_t>(b & 1) * NPT * kPbuf +
                              static_cast<uint32_t>(lane >> 3) * 1024u + static_cast<uint32_t>(lane & 7) * 128u;
#pragma unroll
        for (int ch = 0; ch < 2 * kMtcBlockPages; ++ch) {   // 8 keys (one 16-byte chunk of the P row) at a time
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = ch >> 1, i0 = 8 * (ch & 1) + 2 * e;
            float x0, x1;
            f2_unpack(ffma2(f2_pack(sv[k][i0], sv[k][i0 + 1]), mult2, mneg2), x0, x1);
            float a0 = fast_exp2(x0), a1 = fast_exp2(x1);
            lsum2 = fadd2(lsum2, f2_pack(a0, a1));
            w[e] = FP8 ? pack_f16(a0, a1) : pack_bf16(a0, a1);
            // bf16 P: a second row sum adds the weights as the P V product sees
            // them (rounded), so O divided by it stays a weighted mean of V rows
            // (a bf16 weight is off by up to 2^-9 of itself, and a row dominated
            // by one key would otherwise keep up to 2^-9 of that key's |v|).
            // f16 P (fp8 caches) is off by at most 2^-11 of each weight, so O
            // over the exact sum is within 2^-11 of the largest |v| of the mean:
            // for e4m3 values (|code| <= 448) a quarter of a bf16 unit of them.
            if constexpr (!FP8) rsum2 = fadd2(rsum2, f2_pack(bf16_lo(w[e]), bf16_hi(w[e])));
          }
          if (lane < RP) {
            const uint32_t off = static_cast<uint32_t>((ch ^ (lane & 7)) << 4);
            sts128(prow + off, make_uint4(w[0], w[1], w[2], w[3]));
          }
        }
        float s0, s1;
        f2_unpack(lsum2, s0, s1);
        l += s0 + s1;
        if constexpr (FP8) {
          lr = l;
        } else {
          f2_unpack(rsum2, s0, s1);
          lr += s0 + s1;
        }
      }
      if (wact) fence_proxy_async_smem();   // the P V MMA reads what these stores wrote
      __syncwarp();
      if (lane == 0) mbar_arrive(pfull_bar(b & 1));
      if (staging) {
        // the slices that have landed (in order), then more copies
        while (q_done < q_iss && q_ready())
          if (!q_write()) {
            ok = false;
            break;
          }
        if (!ok) break;
        while (q_iss < kMtcQslices && q_iss - q_done < QR) q_issue();
      }

      if (t.last) {
        // the next segment's Q complete before this one's epilogue
        if (qj == seg + 1 && !q_finish()) {
          ok = false;
          break;
        }
        // O complete once P V of this block is done (previous phase, block
        // b - 2, seen above)
        if (!mtc_wait(pfree_bar(b & 1), static_cast<uint32_t>(b >> 1) & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        const bool complete = (seg_j0 == 0) && (t.j0 + t.np == t.n);
        const int R = G * si.qn;
        const int which = (seg_k0 == 0) ? 0 : 1;
        const int64_t rowbase = static_cast<int64_t>(2 * g + which) * p.R_max;
        if (act && lane < RP) {
          // this row's output factor and destination, once per row: the store
          // loop below is then a multiply and a store per element
          float f = 0.f;
          uint16_t* dst = nullptr;
          if (row_ok) {
            if (complete) {
              f = lr > 0.f ? p.v_scale / lr : 0.f;
              dst = p.out + static_cast<int64_t>(si.t0 + lane / G) * p.out_stride_t +
                    static_cast<int64_t>(seg_c * G + lane % G) * p.out_stride_h;
            } else {
              f = lr > 0.f ? 1.f / lr : 0.f;
              dst = reinterpret_cast<uint16_t*>(p.ws_o) + (rowbase + lane) * kMtcDv;
            }
          }
          x_fac[lane] = f;
          x_dst[lane] = dst;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(ebar);
        if (!mtc_wait(ebar, static_cast<uint32_t>(seg) & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int vb = 0; vb < kMtcDv / 128; ++vb) {
          const int col = 128 * vb + 32 * q4 + lane;   // this thread's value column (its lane of O^T)
#pragma unroll
          for (int h = 0; h < RP / 16; ++h) {
            uint32_t r[16];
            tmem_ld16(tO + static_cast<uint32_t>(vb * RP + 16 * h), r);
            // the rows' factors and destinations are read before any store (a
            // store may not be moved above a later read it could alias)
            float f[16];
            uint16_t* d[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              f[e] = x_fac[16 * h + e];
              d[e] = x_dst[16 * h + e];
            }
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              if (16 * h + e >= R) continue;
              const float o = __uint_as_float(r[e]) * f[e];
              d[e][col] = static_cast<uint16_t>((complete ? pack_bf16(o, 0.f) : pack_f16(o, 0.f)) & 0xFFFFu);
            }
          }
        }
        if (row_ok) {
          const int tok = si.t0 + lane / G;
          const int hq = seg_c * G + lane % G;
          if (complete) {
            if (p.lse != nullptr)
              p.lse[static_cast<int64_t>(tok) * p.lse_stride_t + static_cast<int64_t>(hq) * p.lse_stride_h] =
                  l > 0.f ? (m + fast_log2(l)) * 0.69314718055994530942f : -INFINITY;
          } else {
            p.ws_ml[rowbase + lane] = make_float2(m, l);
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
static cudaError_t launch_mla_tc_one(const CUtensorMap& tm, const CUtensorMap& tb, const SplitParams& p, int grid,
                                     int smem, bool pdl, cudaStream_t stream) {
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
  return cudaLaunchKernelEx(&cfg, pa_mla_tc_kernel<FP8, RP>, tm, tb, p);
}

int mla_tc_threads() { return kMtcThreads; }

cudaError_t launch_mla_tc(bool fp8, int rpad, const CUtensorMap& tm, const CUtensorMap& tb, const SplitParams& p,
                          int grid, int smem, bool pdl, cudaStream_t stream) {
  if (rpad == 16) return fp8 ? launch_mla_tc_one<true, 16>(tm, tb, p, grid, smem, pdl, stream)
                             : launch_mla_tc_one<false, 16>(tm, tb, p, grid, smem, pdl, stream);
  if (rpad == 32) return fp8 ? launch_mla_tc_one<true, 32>(tm, tb, p, grid, smem, pdl, stream)
                             : launch_mla_tc_one<false, 32>(tm, tb, p, grid, smem, pdl, stream);
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
