// Host side of the C ABI declared in include/paged_attn.h: argument
// validation, the launch planner (tile variant, heads per CTA, pipeline depth,
// grid), the split workspace, TMA descriptor encoding and the two launches.
// The host never reads device memory and never synchronises the stream on the
// decode path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <initializer_list>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "paged_attn.h"
#include "pa_kernels.h"

namespace {

// Device status word (one per device context); kernels get its address.
__device__ uint32_t g_status_word;

constexpr int kPageSize = 16;
constexpr int kMaxDevices = 64;
constexpr int kMaxSeqs = 8192;
constexpr int kMaxConsumerWarps = 8;
constexpr int kMaxStages = 32;
constexpr int kMaxSegCost = 1 << 20;           // segment_cost_pages bound (keeps the split's cost prefix in range)
constexpr int kMlaTcSegCostBf16 = 12, kMlaTcSegCostFp8 = 36;
constexpr int kDefaultMinPages = 4;
constexpr int kMaxRowsMma = 64;      // query rows per KV head of the mma.sync kernel
constexpr int kMaxRowsTc = 128;      // ... and of the tensor-memory kernel (bf16 caches)
constexpr int kTcBlockPages = 4;
constexpr int kTcThreads = 384;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;   // pipeline wait limit without wait_limit_us

// Wait limit and starved CTA of a call (pa_options_t.wait_limit_us, test_starve_cta).
uint64_t wait_limit_ns(const pa_options_t* opts) {
  return (opts && opts->wait_limit_us > 0) ? static_cast<uint64_t>(opts->wait_limit_us) * 1000ull : kDefaultWaitNs;
}
int starved_cta(const pa_options_t* opts) { return (opts && opts->test_starve_cta > 0) ? opts->test_starve_cta - 1 : -1; }

thread_local std::string t_last_error;

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int smem_optin = 0;
  uint32_t* status = nullptr;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};

DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Per-device set-up: attributes, kernel shared-memory limits, status word
// address.  Caller holds g_mu.
int device_state(DeviceState** out, int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    if ((e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(MultiProcessorCount)");
    if ((e = cudaDeviceGetAttribute(&s.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(MaxSharedMemoryPerBlockOptin)");
    s.smem_optin -= 1024;   // room for the kernels' static shared memory
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major * 10 + minor != 103)
      return fail(PA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major,
                  minor);
    if ((e = pa::set_split_smem_limits_bf16(s.smem_optin)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(split bf16)");
    if ((e = pa::set_split_smem_limits_fp8(s.smem_optin)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(split fp8)");
    if ((e = pa::set_split_smem_limits_fp8_tok(s.smem_optin)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(split fp8, per-token scales)");
    if ((e = pa::set_split_smem_limits_tc(s.smem_optin)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(split tcgen05)");
    if ((e = pa::set_mla_smem_limits(s.smem_optin)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(MLA)");
    if ((e = pa::set_mla_tc_smem_limits(s.smem_optin)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(MLA, tcgen05)");
    pa::init_cache_write_occupancy();
    void* ptr = nullptr;
    if ((e = cudaGetSymbolAddress(&ptr, g_status_word)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    s.status = static_cast<uint32_t*>(ptr);
    // the no-allocation entry point's scratch array: its address (and module)
    // now, before a caller's pool may take the device's free memory
    if (pa::static_scratch_setup() != PA_OK) return PA_ERR_CUDA;
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
        return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    s.ready = true;
  }
  *out = &s;
  if (dev_out) *dev_out = dev;
  return PA_OK;
}

// ----------------------------------------------------------------- planning
struct Plan {
  int B, Hq, Hkv, D, esz, max_qlen;
  int G, R_max, MT, HC, NC, nstage, threads, grid, min_pages, pair;
  bool tc;            // tensor-memory (tcgen05) kernel
  bool tok;           // per-token fp8 scales staged behind each page's K and V tiles
  uint32_t tok_bytes; // tok: one tensor's scales of one page (HC * 16 * 4)
  int block_pages;    // tc: pages per ring stage
  uint32_t stage_bytes, kv_bytes, q_slot_bytes;
  uint32_t off_stage, off_q, off_bar, off_prefix, off_xchg, smem;
  size_t ws_unit, ws_ml, ws_o, ws_bytes;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int check_shape_args(int B, int Hq, int Hkv, int D, int kv_dtype, int max_qlen) {
  if (B < 1 || B > kMaxSeqs) return fail(PA_ERR_UNSUPPORTED, "num_seqs %d outside [1, %d]", B, kMaxSeqs);
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads %d must be a positive multiple of num_kv_heads %d", Hq, Hkv);
  if (D != 64 && D != 128) return fail(PA_ERR_UNSUPPORTED, "head_dim %d not in {64, 128}", D);
  if (kv_dtype != PA_BF16 && kv_dtype != PA_FP8_E4M3)
    return fail(PA_ERR_INVALID_ARG, "kv dtype %d is neither PA_BF16 nor PA_FP8_E4M3", kv_dtype);
  if (max_qlen < 1) return fail(PA_ERR_INVALID_ARG, "max_query_len %d < 1", max_qlen);
  const int G = Hq / Hkv;
  const int64_t rows = static_cast<int64_t>(G) * max_qlen;
  const int limit = kv_dtype == PA_BF16 ? kMaxRowsTc : kMaxRowsMma;
  if (rows > limit)
    return fail(PA_ERR_UNSUPPORTED, "group size %d x max_query_len %d exceeds %d query rows per KV head (%s cache)", G,
                max_qlen, limit, kv_dtype == PA_BF16 ? "bf16" : "fp8");
  return PA_OK;
}

// Kernel-choice options that the host can check before touching the device.
int check_variant_option(const pa_options_t* opts, int kv_dtype, int64_t rows) {
  const int use_tc = opts ? opts->use_tcgen05 : 0;
  if (use_tc < 0 || use_tc > 2) return fail(PA_ERR_INVALID_ARG, "use_tcgen05 %d not in {0, 1, 2}", use_tc);
  if (use_tc == 2 && kv_dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "the tcgen05 kernel needs a bf16 cache");
  if (rows > kMaxRowsMma && use_tc == 1)
    return fail(PA_ERR_UNSUPPORTED, "%lld query rows per KV head need the tcgen05 kernel", (long long)rows);
  if (opts && opts->heads_per_cta > 1 && (use_tc == 2 || rows > kMaxRowsMma))
    return fail(PA_ERR_UNSUPPORTED, "the tcgen05 kernel takes one KV head per CTA");
  return PA_OK;
}

bool has_token_scales(const pa_options_t* opts) {
  return opts && ((opts->k_token_scales && opts->k_token_scales->data) ||
                  (opts->v_token_scales && opts->v_token_scales->data));
}

// mma.sync kernel: heads per CTA, ring depth and shared-memory layout.
int plan_mma(Plan& p, int B, int Hkv, int D, int max_qlen, const pa_options_t* opts, int smem_optin) {
  const uint32_t bar_bytes = 8u * (2 * kMaxStages + 4);
  const uint32_t prefix_bytes = static_cast<uint32_t>(align_up(4u * (3 * B + 2), 16));   // prefix, lengths, starts
  const int forced_hc = opts ? opts->heads_per_cta : 0;
  if (forced_hc < 0 || (forced_hc > 0 && Hkv % forced_hc != 0))
    return fail(PA_ERR_INVALID_ARG, "heads_per_cta %d must divide num_kv_heads %d", forced_hc, Hkv);
  // Ring depth wanted, in order of preference.  bf16 pages are light on math,
  // so a deep ring (>= 5 stages, which lets consumers take page pairs) beats
  // more heads per CTA; fp8 needs the most consumer warps per CTA (its e4m3
  // conversions double the math per byte), so it takes the widest CTA with a
  // 3-stage ring.
  const int kWantBf16[3] = {5, 3, 2};
  const int kWantFp8[3] = {3, 2, 2};
  const int* want = p.esz == 1 ? kWantFp8 : kWantBf16;
  bool found = false;
  for (int pass = 0; pass < 3 && !found; ++pass) {
    const int want_stages = want[pass];
    for (int hc = (forced_hc > 0 ? forced_hc : std::min(Hkv, kMaxConsumerWarps)); hc >= 1; --hc) {
      if (Hkv % hc != 0 || hc * p.MT > kMaxConsumerWarps) {
        if (forced_hc > 0) break;
        continue;
      }
      const uint32_t kv = static_cast<uint32_t>(hc) * kPageSize * D * p.esz;
      // per-token scales ride behind K and V; stages stay 1024-byte aligned (swizzle span)
      const uint32_t stage =
          2 * kv + (p.tok ? static_cast<uint32_t>(align_up(2u * hc * kPageSize * 4u, 1024)) : 0u);
      const uint32_t qslot = static_cast<uint32_t>(align_up(static_cast<size_t>(max_qlen) * hc * p.G * D * 2, 128));
      const int64_t fixed = 1024 + 2 * qslot + bar_bytes + prefix_bytes;
      const int64_t room = smem_optin - fixed;
      const int nst = room > 0 ? static_cast<int>(std::min<int64_t>(kMaxStages, room / stage)) : 0;
      if (nst >= want_stages) {
        p.HC = hc;
        p.tok_bytes = p.tok ? static_cast<uint32_t>(hc) * kPageSize * 4u : 0u;
        p.kv_bytes = kv;
        p.stage_bytes = stage;
        p.q_slot_bytes = qslot;
        p.nstage = nst;
        found = true;
        break;
      }
      if (forced_hc > 0) break;
    }
  }
  if (!found) return fail(PA_ERR_UNSUPPORTED, "no launch configuration fits %d bytes of shared memory", smem_optin);
  p.NC = Hkv / p.HC;
  p.threads = 32 * (1 + p.HC * p.MT);
  // Two pages per consumer step when the ring is deep enough that holding two
  // stages still leaves most of it in flight.
  const int pairing = opts ? opts->page_pairing : 0;
  p.pair = pairing == 2 ? 1 : (pairing == 1 ? 0 : (p.nstage >= 5 ? 1 : 0));
  p.off_stage = 0;
  p.off_q = p.off_stage + p.nstage * p.stage_bytes;
  p.off_bar = p.off_q + 2 * p.q_slot_bytes;
  p.off_prefix = p.off_bar + bar_bytes;
  p.smem = 1024 + p.off_prefix + prefix_bytes;
  return PA_OK;
}

int make_plan(int B, int Hq, int Hkv, int D, int kv_dtype, int max_qlen, const pa_options_t* opts, int num_sms,
              int smem_optin, Plan* pl) {
  int st = check_shape_args(B, Hq, Hkv, D, kv_dtype, max_qlen);
  if (st != PA_OK) return st;
  Plan p = {};
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.max_qlen = max_qlen;
  p.esz = (kv_dtype == PA_FP8_E4M3) ? 1 : 2;
  p.G = Hq / Hkv;
  p.R_max = p.G * max_qlen;
  p.MT = (p.R_max + 15) / 16;
  p.min_pages = (opts && opts->min_pages_per_cta > 0) ? opts->min_pages_per_cta : kDefaultMinPages;
  p.grid = (opts && opts->num_ctas > 0) ? opts->num_ctas : num_sms;
  if ((st = check_variant_option(opts, kv_dtype, p.R_max)) != PA_OK) return st;
  p.tc = (opts && opts->use_tcgen05 == 2) || p.R_max > kMaxRowsMma;
  p.tok = has_token_scales(opts);
  if (p.tok && kv_dtype != PA_FP8_E4M3) return fail(PA_ERR_INVALID_ARG, "per-token scales need an fp8 cache");
  if (p.tc) {
    // One KV head per CTA; shared memory: ring stages of kTcBlockPages pages
    // (K and V), barriers, exchange buffers, sequence metadata (Q is in TMEM).
    p.HC = 1;
    p.NC = Hkv;
    p.MT = 8;
    p.threads = kTcThreads;
    p.pair = 0;
    p.block_pages = kTcBlockPages;
    p.kv_bytes = static_cast<uint32_t>(kPageSize * D * 2);
    p.stage_bytes = static_cast<uint32_t>(2 * p.block_pages) * p.kv_bytes;
    p.q_slot_bytes = 0;
    const uint32_t tc_bar_bytes = static_cast<uint32_t>(align_up(8u * (2 * kMaxStages + 40), 1024));
    const uint32_t tc_xchg_bytes = 8192;   // softmax warps' (max, sum, rounded sum) of a row, [2][2][128] float4
    const uint32_t tc_prefix_bytes = static_cast<uint32_t>(align_up(4u * (3 * B + 2), 16));
    const int64_t room = smem_optin - (1024 + static_cast<int64_t>(tc_bar_bytes) + tc_xchg_bytes + tc_prefix_bytes);
    p.nstage = room > 0 ? static_cast<int>(std::min<int64_t>(kMaxStages, room / p.stage_bytes)) : 0;
    if (p.nstage < 2)
      return fail(PA_ERR_UNSUPPORTED, "no tcgen05 launch configuration fits %d bytes of shared memory", smem_optin);
    p.off_stage = 0;
    p.off_q = p.nstage * p.stage_bytes;
    p.off_bar = p.off_q;
    p.off_xchg = p.off_bar + tc_bar_bytes;
    p.off_prefix = p.off_xchg + tc_xchg_bytes;
    p.smem = 1024 + p.off_prefix + tc_prefix_bytes;
  }
  if (!p.tc) {
    const int st2 = plan_mma(p, B, Hkv, D, max_qlen, opts, smem_optin);
    if (st2 != PA_OK) return st2;
  }
  const size_t rows = static_cast<size_t>(2) * p.grid * p.HC * p.R_max;
  p.ws_unit = 0;
  p.ws_ml = align_up(p.ws_unit + static_cast<size_t>(16) * B * p.NC, 256);
  p.ws_o = align_up(p.ws_ml + rows * 8, 256);
  p.ws_bytes = align_up(p.ws_o + rows * D * 4, 256);
  *pl = p;
  return PA_OK;
}

// ---------------------------------------------------------------- validation
bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

int check_tensor(const pa_tensor_t* t, const char* name, int ndim, bool allow_null) {
  if (t == nullptr) return fail(PA_ERR_INVALID_ARG, "%s: descriptor pointer is NULL", name);
  if (t->data == nullptr) {
    if (allow_null) return PA_OK;
    return fail(PA_ERR_INVALID_ARG, "%s: data pointer is NULL", name);
  }
  if (t->ndim != ndim) return fail(PA_ERR_INVALID_ARG, "%s: ndim %d, expected %d", name, t->ndim, ndim);
  for (int d = 0; d < ndim; ++d) {
    if (t->shape[d] < 0) return fail(PA_ERR_INVALID_ARG, "%s: negative shape[%d]", name, d);
    if (t->stride[d] < 0) return fail(PA_ERR_INVALID_ARG, "%s: negative stride[%d]", name, d);
  }
  return PA_OK;
}

// cuTensorMapEncodeTiled through a small memo: a map depends only on its
// arguments (address, geometry, layout), and a decode loop passes the same
// ones every step, so repeated encodes are copies of the stored map.  Caller
// holds g_mu.
struct MapKey {
  const void* ptr;
  uint64_t dims[4];
  uint64_t strides[3];
  uint32_t box[4];
  int32_t dtype, rank, swizzle;
};
struct MapMemo {
  bool used;
  MapKey key;
  CUtensorMap map;
};
constexpr int kMapMemo = 16;
MapMemo g_map_memo[kMapMemo];
int g_map_next = 0;

CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* ptr, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
  MapKey k;
  std::memset(&k, 0, sizeof(k));
  k.ptr = ptr;
  for (int d = 0; d < rank && d < 4; ++d) {
    k.dims[d] = dims[d];
    k.box[d] = box[d];
    if (d + 1 < rank) k.strides[d] = strides[d];
  }
  k.dtype = static_cast<int32_t>(dtype);
  k.rank = rank;
  k.swizzle = static_cast<int32_t>(swizzle);
  for (int i = 0; i < kMapMemo; ++i)
    if (g_map_memo[i].used && std::memcmp(&g_map_memo[i].key, &k, sizeof(k)) == 0) {
      *map = g_map_memo[i].map;
      return CUDA_SUCCESS;
    }
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), ptr, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS && rank <= 4) {
    MapMemo& m = g_map_memo[g_map_next];
    g_map_next = (g_map_next + 1) % kMapMemo;
    m.used = true;
    m.key = k;
    m.map = *map;
  }
  return r;
}

// TMA map over a cache [NB, 16, Hkv, D] with dimensions ordered (d, slot, head,
// page): one box is RB bytes of the row x 16 slots x HC heads, which lands in
// shared memory head-major, 16 swizzled rows per head.
int encode_cache_map(CUtensorMap* map, const pa_tensor_t* t, int esz, int D, int Hkv, int HC, int64_t NB) {
  const int rowb = D * esz;
  const int rb = rowb >= 128 ? 128 : 64;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(kPageSize), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(NB)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(t->stride[1]) * esz, static_cast<cuuint64_t>(t->stride[2]) * esz,
                           static_cast<cuuint64_t>(t->stride[0]) * esz};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(rb / esz), static_cast<cuuint32_t>(kPageSize),
                       static_cast<cuuint32_t>(HC), 1u};
  const CUresult r = encode_tiled(map, esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                                  t->data, dims, strides, box,
                                  rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d) for a KV cache", r);
  return PA_OK;
}

// Grow the library-owned workspace of a device to at least `bytes` (a free and
// a fresh allocation; the old contents need not survive).  Caller holds g_mu.
int grow_workspace(DeviceState* ds, size_t bytes) {
  if (ds->ws_bytes >= bytes) return PA_OK;
  cudaError_t e;
  if (ds->ws) {
    if ((e = cudaFree(ds->ws)) != cudaSuccess) return cuda_fail(e, "cudaFree(workspace)");
    ds->ws = nullptr;
    ds->ws_bytes = 0;
  }
  if ((e = cudaMalloc(&ds->ws, bytes)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
  ds->ws_bytes = bytes;
  return PA_OK;
}

// The split workspace of a call: the caller's (checked for size and
// alignment), or the library-owned one of the device, grown outside stream
// capture (during capture an undersized workspace is an error: the caller
// reserves it first with `reserve_fn`).  Caller holds g_mu.
int acquire_workspace(DeviceState* ds, const pa_options_t* opts, size_t bytes, cudaStream_t stream,
                      const char* reserve_fn, void** ws) {
  if (opts && opts->workspace) {
    if (opts->workspace_bytes < bytes)
      return fail(PA_ERR_WORKSPACE, "caller workspace %zu bytes < %zu needed", opts->workspace_bytes, bytes);
    if (!aligned(opts->workspace, 256)) return fail(PA_ERR_INVALID_ARG, "caller workspace must be 256-byte aligned");
    *ws = opts->workspace;
    return PA_OK;
  }
  if (ds->ws_bytes < bytes) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
      return fail(PA_ERR_WORKSPACE, "workspace must grow to %zu bytes, which is not allowed during stream capture; "
                  "call %s first", bytes, reserve_fn);
    const int st = grow_workspace(ds, bytes);
    if (st != PA_OK) return st;
  }
  *ws = ds->ws;
  return PA_OK;
}

int decode_impl(const pa_tensor_t* q, const pa_tensor_t* kc, const pa_tensor_t* vc, const pa_tensor_t* bt,
                const pa_tensor_t* sl, const pa_tensor_t* qsl, int32_t max_qlen, float scale, float k_scale,
                float v_scale, const pa_tensor_t* out, const pa_tensor_t* lse, const pa_options_t* opts,
                cudaStream_t stream) {
  int st;
  if ((st = check_tensor(q, "q", 3, false)) || (st = check_tensor(kc, "k_cache", 4, false)) ||
      (st = check_tensor(vc, "v_cache", 4, false)) || (st = check_tensor(bt, "block_tables", 2, false)) ||
      (st = check_tensor(sl, "seq_lens", 1, false)) || (st = check_tensor(qsl, "query_start_loc", 1, true)) ||
      (st = check_tensor(out, "out", 3, false)) || (st = check_tensor(lse, "lse", 2, true)))
    return st;
  if (q->dtype != PA_BF16) return fail(PA_ERR_INVALID_ARG, "q must be bf16");
  if (out->dtype != PA_BF16) return fail(PA_ERR_INVALID_ARG, "out must be bf16");
  if (kc->dtype != PA_BF16 && kc->dtype != PA_FP8_E4M3)
    return fail(PA_ERR_INVALID_ARG, "k_cache must be bf16 or fp8 e4m3");
  if (vc->dtype != kc->dtype) return fail(PA_ERR_INVALID_ARG, "v_cache dtype differs from k_cache");
  if (bt->dtype != PA_I32 || sl->dtype != PA_I32) return fail(PA_ERR_INVALID_ARG, "block_tables and seq_lens must be int32");
  if (qsl->data && qsl->dtype != PA_I32) return fail(PA_ERR_INVALID_ARG, "query_start_loc must be int32");
  if (lse->data && lse->dtype != PA_F32) return fail(PA_ERR_INVALID_ARG, "lse must be float32");
  const int64_t T = q->shape[0], Hq = q->shape[1], D = q->shape[2];
  const int64_t NB = kc->shape[0], P = kc->shape[1], Hkv = kc->shape[2];
  const int64_t B = bt->shape[0], MB = bt->shape[1];
  if (P != kPageSize) return fail(PA_ERR_UNSUPPORTED, "page size %lld, only 16 is supported", (long long)P);
  if (kc->shape[3] != D) return fail(PA_ERR_INVALID_ARG, "k_cache head_dim %lld != q head_dim %lld", (long long)kc->shape[3], (long long)D);
  for (int d = 0; d < 4; ++d)
    if (vc->shape[d] != kc->shape[d]) return fail(PA_ERR_INVALID_ARG, "v_cache shape differs from k_cache");
  if (Hq > (1 << 20) || Hkv > (1 << 20) || T > (int64_t(1) << 30) || NB > (int64_t(1) << 31) - 1 || MB > (1 << 28))
    return fail(PA_ERR_UNSUPPORTED, "tensor extents too large");
  if (sl->shape[0] != B) return fail(PA_ERR_INVALID_ARG, "seq_lens has %lld entries, block_tables %lld rows", (long long)sl->shape[0], (long long)B);
  if (B * MB > (int64_t(1) << 31)) return fail(PA_ERR_UNSUPPORTED, "block table too large");
  if (out->shape[0] != T || out->shape[1] != Hq || out->shape[2] != D) return fail(PA_ERR_INVALID_ARG, "out shape differs from q");
  if (lse->data && (lse->shape[0] != T || lse->shape[1] != Hq)) return fail(PA_ERR_INVALID_ARG, "lse shape must be [T, Hq]");
  if (B == 0 || T == 0) return PA_OK;   // nothing to do
  if (qsl->data) {
    if (qsl->shape[0] != B + 1) return fail(PA_ERR_INVALID_ARG, "query_start_loc must have B+1 entries");
    if (qsl->stride[0] != 1) return fail(PA_ERR_INVALID_ARG, "query_start_loc must be contiguous");
    if (T < B || T > B * static_cast<int64_t>(max_qlen))
      return fail(PA_ERR_INVALID_ARG, "T = %lld query tokens is outside [B, B * max_query_len]", (long long)T);
  } else {
    if (T != B) return fail(PA_ERR_INVALID_ARG, "without query_start_loc, q needs one token per sequence (T == B)");
    if (max_qlen != 1) return fail(PA_ERR_INVALID_ARG, "max_query_len must be 1 without query_start_loc");
  }
  if (sl->stride[0] != 1) return fail(PA_ERR_INVALID_ARG, "seq_lens must be contiguous");
  if (bt->stride[1] != 1) return fail(PA_ERR_INVALID_ARG, "block_tables rows must be contiguous");
  if (q->stride[2] != 1 || q->stride[1] != D) return fail(PA_ERR_INVALID_ARG, "q must have contiguous heads (stride[1] == D, stride[2] == 1)");
  if ((q->stride[0] * 2) % 16 != 0 || !aligned(q->data, 16)) return fail(PA_ERR_INVALID_ARG, "q rows must be 16-byte aligned");
  if (out->stride[2] != 1 || (out->stride[1] % 4) != 0 || (out->stride[0] % 4) != 0 || !aligned(out->data, 8))
    return fail(PA_ERR_INVALID_ARG, "out must have a contiguous last dim, strides multiple of 4 elements, 8-byte alignment");
  const int esz = kc->dtype == PA_FP8_E4M3 ? 1 : 2;
  for (const pa_tensor_t* c : {kc, vc}) {
    if (c->stride[3] != 1) return fail(PA_ERR_INVALID_ARG, "KV cache last dim must be contiguous");
    for (int d = 0; d < 3; ++d)
      if ((c->stride[d] * esz) % 16 != 0) return fail(PA_ERR_INVALID_ARG, "KV cache strides must be multiples of 16 bytes");
    if (!aligned(c->data, 16)) return fail(PA_ERR_INVALID_ARG, "KV cache data must be 16-byte aligned");
  }
  if (!std::isfinite(scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return fail(PA_ERR_INVALID_ARG, "scale, k_scale and v_scale must be finite");
  if (opts && opts->sinks && !aligned(opts->sinks, 4)) return fail(PA_ERR_INVALID_ARG, "sinks must be 4-byte aligned");
  if (opts && (opts->wait_limit_us < 0 || opts->test_starve_cta < 0))
    return fail(PA_ERR_INVALID_ARG, "wait_limit_us and test_starve_cta must not be negative");
  const bool tok = has_token_scales(opts);
  if (tok) {
    if (kc->dtype != PA_FP8_E4M3) return fail(PA_ERR_INVALID_ARG, "per-token scales need an fp8 cache");
    const pa_tensor_t* ts[2] = {opts->k_token_scales, opts->v_token_scales};
    const char* nm[2] = {"k_token_scales", "v_token_scales"};
    for (int x = 0; x < 2; ++x) {
      if (ts[x] == nullptr || ts[x]->data == nullptr)
        return fail(PA_ERR_INVALID_ARG, "k_token_scales and v_token_scales must be given together");
      if ((st = check_tensor(ts[x], nm[x], 3, false)) != PA_OK) return st;
      if (ts[x]->dtype != PA_F32) return fail(PA_ERR_INVALID_ARG, "%s must be float32", nm[x]);
      if (ts[x]->shape[0] != NB || ts[x]->shape[1] != Hkv || ts[x]->shape[2] != kPageSize)
        return fail(PA_ERR_INVALID_ARG, "%s must have shape [NB, Hkv, 16] = [%lld, %lld, 16]", nm[x], (long long)NB,
                    (long long)Hkv);
      if (ts[x]->stride[2] != 1 || ts[x]->stride[1] != kPageSize || ts[x]->stride[0] % 4 != 0 ||
          !aligned(ts[x]->data, 16))
        return fail(PA_ERR_INVALID_ARG, "%s: each page's [Hkv, 16] block must be contiguous and 16-byte aligned",
                    nm[x]);
    }
    if (ts[0]->stride[0] != ts[1]->stride[0])
      return fail(PA_ERR_INVALID_ARG, "k_token_scales and v_token_scales need the same page stride");
  }
  if ((st = check_shape_args(static_cast<int>(std::min<int64_t>(B, kMaxSeqs + 1)), static_cast<int>(Hq),
                             static_cast<int>(Hkv), static_cast<int>(D), kc->dtype, max_qlen)) != PA_OK)
    return st;
  if ((st = check_variant_option(opts, kc->dtype, (Hq / Hkv) * static_cast<int64_t>(max_qlen))) != PA_OK) return st;

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds, nullptr)) != PA_OK) return st;
  Plan pl{};
  if ((st = make_plan(static_cast<int>(B), static_cast<int>(Hq), static_cast<int>(Hkv), static_cast<int>(D),
                      kc->dtype, max_qlen, opts, ds->num_sms, ds->smem_optin, &pl)) != PA_OK)
    return st;

  void* ws = nullptr;
  if ((st = acquire_workspace(ds, opts, pl.ws_bytes, stream, "paged_attn_reserve", &ws)) != PA_OK) return st;

  CUtensorMap tk, tv;
  if ((st = encode_cache_map(&tk, kc, esz, static_cast<int>(D), static_cast<int>(Hkv), pl.HC, NB)) != PA_OK) return st;
  if ((st = encode_cache_map(&tv, vc, esz, static_cast<int>(D), static_cast<int>(Hkv), pl.HC, NB)) != PA_OK) return st;

  const float kLog2e = 1.4426950408889634f;
  pa::SplitParams sp = {};
  sp.q = static_cast<const uint16_t*>(q->data);
  sp.q_stride_t = q->stride[0];
  sp.out = static_cast<uint16_t*>(out->data);
  sp.out_stride_t = out->stride[0];
  sp.out_stride_h = out->stride[1];
  sp.lse = static_cast<float*>(lse->data);
  sp.lse_stride_t = lse->data ? lse->stride[0] : 0;
  sp.lse_stride_h = lse->data ? lse->stride[1] : 0;
  sp.block_tables = static_cast<const int32_t*>(bt->data);
  sp.bt_stride = bt->stride[0];
  sp.seq_lens = static_cast<const int32_t*>(sl->data);
  sp.qsl = static_cast<const int32_t*>(qsl->data);
  sp.num_seqs = static_cast<int32_t>(B);
  sp.num_tokens = static_cast<int32_t>(T);
  sp.Hq = static_cast<int32_t>(Hq);
  sp.Hkv = static_cast<int32_t>(Hkv);
  sp.G = pl.G;
  sp.max_qlen = max_qlen;
  sp.num_pages = static_cast<int32_t>(NB);
  sp.max_blocks = static_cast<int32_t>(MB);
  sp.HC = pl.HC;
  sp.NC = pl.NC;
  sp.MT = pl.MT;
  sp.R_max = pl.R_max;
  sp.nstage = pl.nstage;
  sp.min_pages = pl.min_pages;
  sp.pair_pages = pl.pair;
  sp.window = (opts && opts->sliding_window > 0) ? opts->sliding_window : 0;
  sp.sinks = opts ? static_cast<const float*>(opts->sinks) : nullptr;
  sp.scale_log2 = scale * (esz == 1 ? k_scale : 1.0f) * kLog2e;
  sp.v_scale = esz == 1 ? v_scale : 1.0f;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  sp.ws_unit = reinterpret_cast<int4*>(wsb + pl.ws_unit);
  sp.ws_ml = reinterpret_cast<float2*>(wsb + pl.ws_ml);
  sp.ws_o = reinterpret_cast<float*>(wsb + pl.ws_o);
  sp.err = ds->status;
  sp.off_prefix = pl.off_prefix;
  sp.off_bar = pl.off_bar;
  sp.off_q = pl.off_q;
  sp.q_slot_bytes = pl.q_slot_bytes;
  sp.off_stage = pl.off_stage;
  sp.stage_bytes = pl.stage_bytes;
  sp.kv_bytes = pl.kv_bytes;
  sp.block_pages = pl.block_pages;
  sp.off_xchg = pl.off_xchg;
  if (pl.tok) {
    sp.k_tok = static_cast<const float*>(opts->k_token_scales->data);
    sp.v_tok = static_cast<const float*>(opts->v_token_scales->data);
    sp.tok_stride_page = opts->k_token_scales->stride[0];
    sp.tok_bytes = pl.tok_bytes;
  }
  sp.wait_ns = wait_limit_ns(opts);
  sp.starve_cta = starved_cta(opts);
  if (sp.starve_cta >= 0 && pl.tc)
    return fail(PA_ERR_UNSUPPORTED, "test_starve_cta applies to the mma.sync split kernel only");

  pa::MergeParams mp = {};
  mp.out = sp.out;
  mp.out_stride_t = sp.out_stride_t;
  mp.out_stride_h = sp.out_stride_h;
  mp.lse = sp.lse;
  mp.lse_stride_t = sp.lse_stride_t;
  mp.lse_stride_h = sp.lse_stride_h;
  mp.seq_lens = sp.seq_lens;
  mp.qsl = sp.qsl;
  mp.num_seqs = sp.num_seqs;
  mp.num_tokens = sp.num_tokens;
  mp.G = pl.G;
  mp.HC = pl.HC;
  mp.NC = pl.NC;
  mp.R_max = pl.R_max;
  mp.max_qlen = max_qlen;
  mp.split_grid = pl.grid;
  mp.v_scale = sp.v_scale;
  mp.ws_unit = sp.ws_unit;
  mp.ws_ml = sp.ws_ml;
  mp.ws_o = sp.ws_o;
  mp.err = sp.err;

  cudaEvent_t ev0 = opts ? static_cast<cudaEvent_t>(opts->split_start_event) : nullptr;
  cudaEvent_t ev1 = opts ? static_cast<cudaEvent_t>(opts->split_stop_event) : nullptr;
  cudaError_t e;
  // Both kernels use programmatic dependent launch: each waits for its
  // predecessor in the stream before touching global memory, but its launch
  // overlaps the predecessor's tail.
  const bool pdl = !(opts && opts->disable_pdl);
  // Under stream capture the records become external event nodes (so a replay
  // records them); outside capture they are ordinary records.
  unsigned int rec_flags = cudaEventRecordDefault;
  if (ev0 || ev1) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if ((e = cudaStreamIsCapturing(stream, &cs)) != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cs == cudaStreamCaptureStatusActive) rec_flags = cudaEventRecordExternal;
  }
  if (ev0 && (e = cudaEventRecordWithFlags(ev0, stream, rec_flags)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord(start)");
  if (pl.tc)
    e = pa::launch_split_tc(static_cast<int>(D), tk, tv, sp, pl.grid, static_cast<int>(pl.smem), pdl && !ev0, stream);
  else if (pl.tok)
    e = pa::launch_split_fp8_tok(static_cast<int>(D), tk, tv, sp, pl.grid, pl.threads, static_cast<int>(pl.smem),
                                 pdl && !ev0, stream);
  else if (esz == 1)
    e = pa::launch_split_fp8(static_cast<int>(D), tk, tv, sp, pl.grid, pl.threads, static_cast<int>(pl.smem),
                             pdl && !ev0, stream);
  else
    e = pa::launch_split_bf16(static_cast<int>(D), tk, tv, sp, pl.grid, pl.threads, static_cast<int>(pl.smem),
                              pdl && !ev0, stream);
  if (e != cudaSuccess) return cuda_fail(e, "split kernel launch");
  if (ev1 && (e = cudaEventRecordWithFlags(ev1, stream, rec_flags)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord(stop)");
  // Many pieces per unit on average (few long contexts over many CTAs): the
  // wide merge reads a row's partials with a whole block.
  const bool wide = pl.grid >= 4 * static_cast<int>(B) * pl.NC;
  e = pa::launch_merge(static_cast<int>(D), mp, static_cast<int>(B) * pl.NC, pl.HC * pl.R_max, wide, pdl && !ev1, stream);
  if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
  return PA_OK;
}

// ------------------------------------------------------------------- MLA
// Latent rows of 512 (c_kv) + 64 (k_pe) features; the value is the latent part.
constexpr int kMlaDqk = 576;
constexpr int kMlaDv = 512;
constexpr int kMlaMaxRows = 32;   // query rows of one head chunk (2 tiles of 16)

struct MlaPlan {
  int B, Hq, max_qlen, esz;
  int Gc, NC, R_max, RT, nteam, threads, grid, min_pages, nstage, q_slots, pair;
  bool tc;     // tensor-memory kernel
  int rpad;    // tc: rows of a unit padded to 16 or 32 (the P V product's N)
  uint32_t stage_bytes, q_slot_bytes, off_stage, off_q, off_xchg, off_bar, team_bytes, off_prefix, smem, off_buf;
  uint32_t off_qring;   // tc: the Q staging ring
  int seg_cost;         // tc: pages the work split charges per unit a CTA starts
  size_t ws_unit, ws_ml, ws_o, ws_bytes;
};

int check_mla_options(const pa_options_t* opts) {
  if (opts == nullptr) return PA_OK;
  if (opts->use_tcgen05 < 0 || opts->use_tcgen05 > 2)
    return fail(PA_ERR_INVALID_ARG, "use_tcgen05 %d not in {0, 1, 2}", opts->use_tcgen05);
  if (opts->page_pairing < 0 || opts->page_pairing > 2)
    return fail(PA_ERR_INVALID_ARG, "page_pairing %d not in {0, 1, 2}", opts->page_pairing);
  if (opts->wait_limit_us < 0) return fail(PA_ERR_INVALID_ARG, "wait_limit_us %d is negative", opts->wait_limit_us);
  if (opts->segment_cost_pages > kMaxSegCost)
    return fail(PA_ERR_INVALID_ARG, "segment_cost_pages %d > %d", opts->segment_cost_pages, kMaxSegCost);
  if (opts->heads_per_cta != 0 || opts->sliding_window > 0 || opts->sinks != nullptr || has_token_scales(opts) ||
      opts->test_starve_cta != 0)
    return fail(PA_ERR_UNSUPPORTED, "MLA decode takes none of heads_per_cta, sliding_window, sinks, token scales, "
                "test_starve_cta");
  return PA_OK;
}

// Shape checks that need no device.
int check_mla_shape(int B, int Hq, int kv_dtype, int max_qlen, const pa_options_t* opts) {
  if (B < 1 || B > kMaxSeqs) return fail(PA_ERR_UNSUPPORTED, "num_seqs %d outside [1, %d]", B, kMaxSeqs);
  if (Hq < 1) return fail(PA_ERR_INVALID_ARG, "num_q_heads %d < 1", Hq);
  if (kv_dtype != PA_BF16 && kv_dtype != PA_FP8_E4M3)
    return fail(PA_ERR_INVALID_ARG, "kv dtype %d is neither PA_BF16 nor PA_FP8_E4M3", kv_dtype);
  if (max_qlen < 1) return fail(PA_ERR_INVALID_ARG, "max_query_len %d < 1", max_qlen);
  if (max_qlen > kMlaMaxRows)
    return fail(PA_ERR_UNSUPPORTED, "max_query_len %d > %d for MLA decode", max_qlen, kMlaMaxRows);
  return check_mla_options(opts);
}

int make_mla_plan(int B, int Hq, int kv_dtype, int max_qlen, const pa_options_t* opts, int num_sms, int smem_optin,
                  MlaPlan* out) {
  const int st = check_mla_shape(B, Hq, kv_dtype, max_qlen, opts);
  if (st != PA_OK) return st;
  MlaPlan p = {};
  p.B = B; p.Hq = Hq; p.max_qlen = max_qlen;
  p.esz = kv_dtype == PA_FP8_E4M3 ? 1 : 2;
  // heads per chunk: the largest divisor of Hq whose rows fit two 16-row tiles
  p.Gc = 1;
  for (int d = 1; d <= Hq; ++d)
    if (Hq % d == 0 && d * max_qlen <= kMlaMaxRows) p.Gc = d;
  p.NC = Hq / p.Gc;
  p.R_max = p.Gc * max_qlen;
  p.RT = (p.R_max + 15) / 16;
  p.min_pages = (opts && opts->min_pages_per_cta > 0) ? opts->min_pages_per_cta : kDefaultMinPages;
  p.grid = (opts && opts->num_ctas > 0) ? opts->num_ctas : num_sms;
  // The tensor-memory kernel when the caller asks for it (use_tcgen05 = 2) or,
  // by default, where it measured faster: fp8 caches (the converter warps
  // feed the tensor cores f16 rows once a page, where the mma.sync kernel
  // converts per fragment) and units of more than 16 rows (one M = 128 Q K^T
  // covers 32 rows as cheaply as 16).  A unit's rows (at most 32) always fit.
  const int tcsel = opts ? opts->use_tcgen05 : 0;
  p.tc = tcsel == 2 || (tcsel == 0 && (p.esz == 1 || p.R_max > 16));
  if (p.tc) {
    // one worker a CTA; shared memory: the three block buffers (3 pages of
    // rows in the MMA layout), the P buffers, a ring of raw page slots, the Q
    // staging ring, barriers, the softmax exchange, sequence metadata
    p.rpad = p.R_max <= 16 ? 16 : 32;
    // a unit a CTA starts costs about a Q staging, an epilogue and a pipeline
    // refill: measured, near 4 blocks of 3 pages (bf16) and 12 (fp8)
    const int sc = opts ? opts->segment_cost_pages : 0;
    p.seg_cost = sc < 0 ? 0 : (sc > 0 ? sc : (p.esz == 1 ? kMlaTcSegCostFp8 : kMlaTcSegCostBf16));
    p.nteam = 1;
    p.threads = pa::mla_tc_threads();
    p.pair = 0;
    // three block buffers of 3 pages in the MMA layout; fp8 caches add a ring
    // of raw page slots for the converters (bf16 boxes land in the buffers)
    const uint32_t buf_bytes = 3u * 9u * 3u * 2048u;
    const uint32_t p_bytes = 2u * static_cast<uint32_t>(p.rpad) * 128u;
    p.stage_bytes = static_cast<uint32_t>(kPageSize * kMlaDqk * p.esz);
    const uint32_t xchg = 3328;   // alpha [4][32] f32, flags [4][4], row factors [32] f32, row outputs [32] pointers
    const uint32_t prefix_bytes = static_cast<uint32_t>(align_up(4u * (3 * B + 2), 16));
    const uint32_t qslot = static_cast<uint32_t>(p.rpad) * 208u;   // one 192-byte slice of every Q row
    p.off_buf = 0;
    p.off_q = buf_bytes;
    p.off_stage = p.off_q + p_bytes;
    // A Q ring of 6 slots (a whole Q in flight) if it fits beside an fp8 raw
    // ring of at least 4 page slots, else 2 slots; then the deepest raw ring
    // whose barriers (2 a slot + 19 + 1 a Q slot) still fit
    uint32_t bars = 0;
    bool placed = false;
    for (const int qr : {6, 2}) {
      const int min_stages = p.esz == 1 ? (qr == 6 ? 4 : 2) : 0;
      for (p.nstage = p.esz == 1 ? kMaxStages : 0; p.nstage >= min_stages; --p.nstage) {
        bars = static_cast<uint32_t>(align_up(8u * (2 * p.nstage + 19 + qr), 128));
        if (1024 + static_cast<int64_t>(p.off_stage) + static_cast<int64_t>(p.nstage) * p.stage_bytes +
                static_cast<int64_t>(qr) * qslot + bars + xchg + prefix_bytes <=
            smem_optin) {
          placed = true;
          break;
        }
      }
      if (placed) {
        p.q_slots = qr;
        break;
      }
    }
    if (!placed)
      return fail(PA_ERR_UNSUPPORTED, "no tcgen05 MLA launch configuration fits %d bytes of shared memory", smem_optin);
    p.off_qring = p.off_stage + static_cast<uint32_t>(p.nstage) * p.stage_bytes;
    p.off_bar = p.off_qring + static_cast<uint32_t>(p.q_slots) * qslot;
    p.off_xchg = p.off_bar + bars;
    p.off_prefix = p.off_xchg + xchg;
    p.team_bytes = 0;
    p.q_slot_bytes = 0;
    p.smem = 1024 + p.off_prefix + prefix_bytes;
    const size_t rows = static_cast<size_t>(2) * p.grid * p.R_max;
    p.ws_unit = 0;
    p.ws_ml = align_up(p.ws_unit + static_cast<size_t>(16) * B * p.NC, 256);
    p.ws_o = align_up(p.ws_ml + rows * 8, 256);
    p.ws_bytes = align_up(p.ws_o + rows * kMlaDv * 2, 256);   // f16 normalised partial outputs
    *out = p;
    return PA_OK;
  }
  p.nteam = pa::mla_teams(p.RT);
  p.threads = pa::mla_threads(p.RT);
  p.stage_bytes = static_cast<uint32_t>(kPageSize * kMlaDqk * p.esz);
  p.q_slot_bytes = static_cast<uint32_t>(align_up(static_cast<size_t>(max_qlen) * p.Gc * kMlaDqk * 2, 1024));
  // One query slot a team: the next segment's rows are fetched once the
  // consumers hold the current ones in registers, and the room goes to the ring.
  p.q_slots = 1;
  const uint32_t xchg = 16384u * static_cast<uint32_t>(p.RT);   // 2 steps x 4 quarters x 2 KB a row tile
  const uint32_t bars = static_cast<uint32_t>(align_up(8u * (2 * kMaxStages + 4 + 2 * p.RT), 128));
  const uint32_t prefix_bytes = static_cast<uint32_t>(align_up(4u * (3 * B + 2), 16));
  const int64_t room = (static_cast<int64_t>(smem_optin) - 1024 - prefix_bytes) / p.nteam / 1024 * 1024;
  const int64_t fixed = static_cast<int64_t>(p.q_slots) * p.q_slot_bytes + xchg + bars;
  p.nstage = room > fixed ? static_cast<int>(std::min<int64_t>(kMaxStages, (room - fixed) / p.stage_bytes)) : 0;
  if (p.nstage < 2) return fail(PA_ERR_UNSUPPORTED, "no MLA launch configuration fits %d bytes of shared memory", smem_optin);
  p.off_stage = 0;
  p.off_q = p.off_stage + p.nstage * p.stage_bytes;
  p.off_xchg = p.off_q + static_cast<uint32_t>(p.q_slots) * p.q_slot_bytes;
  // Page pairs (a consumer step holds two stages) when the ring keeps two more in flight.
  const int pairing = opts ? opts->page_pairing : 0;
  p.pair = pairing == 2 ? 1 : (pairing == 1 ? 0 : (p.nstage >= 4 ? 1 : 0));
  p.off_bar = p.off_xchg + xchg;
  p.team_bytes = static_cast<uint32_t>(align_up(p.off_bar + bars, 1024));
  p.off_prefix = p.team_bytes * static_cast<uint32_t>(p.nteam);
  p.smem = 1024 + p.off_prefix + prefix_bytes;
  const size_t rows = static_cast<size_t>(2) * p.grid * p.nteam * p.R_max;
  p.ws_unit = 0;
  p.ws_ml = align_up(p.ws_unit + static_cast<size_t>(16) * B * p.NC, 256);
  p.ws_o = align_up(p.ws_ml + rows * 8, 256);
  p.ws_bytes = align_up(p.ws_o + rows * kMlaDv * 2, 256);   // f16 normalised partial outputs
  *out = p;
  return PA_OK;
}

// TMA map over a latent cache [NB, 16, 576] with dimensions (feature within a
// 64-feature block, slot, block, page): one box = a whole page, landing as 9
// column blocks of 16 swizzled rows (box_blocks = 9), or one column block of
// one page (box_blocks = 1).
int encode_mla_map(CUtensorMap* map, const pa_tensor_t* t, int esz, int64_t NB, int box_blocks) {
  cuuint64_t dims[4] = {64u, static_cast<cuuint64_t>(kPageSize), static_cast<cuuint64_t>(kMlaDqk / 64),
                        static_cast<cuuint64_t>(NB)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(t->stride[1]) * esz, static_cast<cuuint64_t>(64 * esz),
                           static_cast<cuuint64_t>(t->stride[0]) * esz};
  cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(kPageSize), static_cast<cuuint32_t>(box_blocks), 1u};
  const CUresult r = encode_tiled(map, esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                                  t->data, dims, strides, box,
                                  esz == 2 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d) for the latent cache", r);
  return PA_OK;
}

int mla_decode_impl(const pa_tensor_t* q, const pa_tensor_t* kc, const pa_tensor_t* bt, const pa_tensor_t* sl,
                    const pa_tensor_t* qsl, int32_t max_qlen, float scale, float kv_scale, const pa_tensor_t* out,
                    const pa_tensor_t* lse, const pa_options_t* opts, cudaStream_t stream) {
  int st;
  if ((st = check_tensor(q, "q", 3, false)) || (st = check_tensor(kc, "kv_cache", 3, false)) ||
      (st = check_tensor(bt, "block_tables", 2, false)) || (st = check_tensor(sl, "seq_lens", 1, false)) ||
      (st = check_tensor(qsl, "query_start_loc", 1, true)) || (st = check_tensor(out, "out", 3, false)) ||
      (st = check_tensor(lse, "lse", 2, true)))
    return st;
  if (q->dtype != PA_BF16 || out->dtype != PA_BF16) return fail(PA_ERR_INVALID_ARG, "q and out must be bf16");
  if (kc->dtype != PA_BF16 && kc->dtype != PA_FP8_E4M3)
    return fail(PA_ERR_INVALID_ARG, "kv_cache must be bf16 or fp8 e4m3");
  if (bt->dtype != PA_I32 || sl->dtype != PA_I32) return fail(PA_ERR_INVALID_ARG, "block_tables and seq_lens must be int32");
  if (qsl->data && qsl->dtype != PA_I32) return fail(PA_ERR_INVALID_ARG, "query_start_loc must be int32");
  if (lse->data && lse->dtype != PA_F32) return fail(PA_ERR_INVALID_ARG, "lse must be float32");
  const int64_t T = q->shape[0], Hq = q->shape[1], Dqk = q->shape[2];
  const int64_t NB = kc->shape[0], P = kc->shape[1];
  const int64_t B = bt->shape[0], MB = bt->shape[1];
  if (P != kPageSize) return fail(PA_ERR_UNSUPPORTED, "page size %lld, only 16 is supported", (long long)P);
  if (Dqk != kMlaDqk || kc->shape[2] != kMlaDqk)
    return fail(PA_ERR_UNSUPPORTED, "MLA rows of %lld (q) and %lld (cache) features; only 512 + 64 = 576 is supported",
                (long long)Dqk, (long long)kc->shape[2]);
  if (out->shape[0] != T || out->shape[1] != Hq || out->shape[2] != kMlaDv)
    return fail(PA_ERR_INVALID_ARG, "out must be [T, Hq, 512]");
  if (Hq > (1 << 20) || T > (int64_t(1) << 30) || NB > (int64_t(1) << 31) - 1 || MB > (1 << 28))
    return fail(PA_ERR_UNSUPPORTED, "tensor extents too large");
  if (sl->shape[0] != B) return fail(PA_ERR_INVALID_ARG, "seq_lens has %lld entries, block_tables %lld rows", (long long)sl->shape[0], (long long)B);
  if (B * MB > (int64_t(1) << 31)) return fail(PA_ERR_UNSUPPORTED, "block table too large");
  if (lse->data && (lse->shape[0] != T || lse->shape[1] != Hq)) return fail(PA_ERR_INVALID_ARG, "lse shape must be [T, Hq]");
  if (B == 0 || T == 0) return PA_OK;
  if (qsl->data) {
    if (qsl->shape[0] != B + 1) return fail(PA_ERR_INVALID_ARG, "query_start_loc must have B+1 entries");
    if (qsl->stride[0] != 1) return fail(PA_ERR_INVALID_ARG, "query_start_loc must be contiguous");
    if (T < B || T > B * static_cast<int64_t>(max_qlen))
      return fail(PA_ERR_INVALID_ARG, "T = %lld query tokens is outside [B, B * max_query_len]", (long long)T);
  } else {
    if (T != B) return fail(PA_ERR_INVALID_ARG, "without query_start_loc, q needs one token per sequence (T == B)");
    if (max_qlen != 1) return fail(PA_ERR_INVALID_ARG, "max_query_len must be 1 without query_start_loc");
  }
  if (sl->stride[0] != 1) return fail(PA_ERR_INVALID_ARG, "seq_lens must be contiguous");
  if (bt->stride[1] != 1) return fail(PA_ERR_INVALID_ARG, "block_tables rows must be contiguous");
  if (q->stride[2] != 1 || q->stride[1] != kMlaDqk)
    return fail(PA_ERR_INVALID_ARG, "q must have contiguous heads (stride[1] == 576, stride[2] == 1)");
  if ((q->stride[0] * 2) % 16 != 0 || !aligned(q->data, 16)) return fail(PA_ERR_INVALID_ARG, "q rows must be 16-byte aligned");
  if (out->stride[2] != 1 || (out->stride[1] % 4) != 0 || (out->stride[0] % 4) != 0 || !aligned(out->data, 8))
    return fail(PA_ERR_INVALID_ARG, "out must have a contiguous last dim, strides multiple of 4 elements, 8-byte alignment");
  const int esz = kc->dtype == PA_FP8_E4M3 ? 1 : 2;
  if (kc->stride[2] != 1) return fail(PA_ERR_INVALID_ARG, "kv_cache last dim must be contiguous");
  for (int d = 0; d < 2; ++d)
    if ((kc->stride[d] * esz) % 16 != 0) return fail(PA_ERR_INVALID_ARG, "kv_cache strides must be multiples of 16 bytes");
  if (!aligned(kc->data, 16)) return fail(PA_ERR_INVALID_ARG, "kv_cache data must be 16-byte aligned");
  if (!std::isfinite(scale) || !std::isfinite(kv_scale)) return fail(PA_ERR_INVALID_ARG, "scale and kv_scale must be finite");
  if ((st = check_mla_shape(static_cast<int>(std::min<int64_t>(B, kMaxSeqs + 1)), static_cast<int>(Hq), kc->dtype,
                            max_qlen, opts)) != PA_OK)
    return st;

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds, nullptr)) != PA_OK) return st;
  MlaPlan pl{};
  if ((st = make_mla_plan(static_cast<int>(std::min<int64_t>(B, kMaxSeqs + 1)), static_cast<int>(Hq), kc->dtype,
                          max_qlen, opts, ds->num_sms, ds->smem_optin, &pl)) != PA_OK)
    return st;
  void* ws = nullptr;
  if ((st = acquire_workspace(ds, opts, pl.ws_bytes, stream, "paged_attn_mla_reserve", &ws)) != PA_OK) return st;
  CUtensorMap tm, tb;
  if ((st = encode_mla_map(&tm, kc, esz, NB, kMlaDqk / 64)) != PA_OK) return st;
  if ((st = encode_mla_map(&tb, kc, esz, NB, 1)) != PA_OK) return st;

  const float kLog2e = 1.4426950408889634f;
  pa::SplitParams sp = {};
  sp.q = static_cast<const uint16_t*>(q->data);
  sp.q_stride_t = q->stride[0];
  sp.out = static_cast<uint16_t*>(out->data);
  sp.out_stride_t = out->stride[0];
  sp.out_stride_h = out->stride[1];
  sp.lse = static_cast<float*>(lse->data);
  sp.lse_stride_t = lse->data ? lse->stride[0] : 0;
  sp.lse_stride_h = lse->data ? lse->stride[1] : 0;
  sp.block_tables = static_cast<const int32_t*>(bt->data);
  sp.bt_stride = bt->stride[0];
  sp.seq_lens = static_cast<const int32_t*>(sl->data);
  sp.qsl = static_cast<const int32_t*>(qsl->data);
  sp.num_seqs = static_cast<int32_t>(B);
  sp.num_tokens = static_cast<int32_t>(T);
  sp.Hq = static_cast<int32_t>(Hq);
  sp.Hkv = 1;
  sp.G = pl.Gc;
  sp.max_qlen = max_qlen;
  sp.num_pages = static_cast<int32_t>(NB);
  sp.max_blocks = static_cast<int32_t>(MB);
  sp.HC = 1;
  sp.NC = pl.NC;
  sp.MT = pl.RT;
  sp.R_max = pl.R_max;
  sp.nstage = pl.nstage;
  sp.min_pages = pl.min_pages;
  sp.scale_log2 = scale * (esz == 1 ? kv_scale : 1.0f) * kLog2e;
  sp.v_scale = esz == 1 ? kv_scale : 1.0f;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  sp.ws_unit = reinterpret_cast<int4*>(wsb + pl.ws_unit);
  sp.ws_ml = reinterpret_cast<float2*>(wsb + pl.ws_ml);
  sp.ws_o = reinterpret_cast<float*>(wsb + pl.ws_o);
  sp.err = ds->status;
  sp.off_prefix = pl.off_prefix;
  sp.off_bar = pl.off_bar;
  sp.off_q = pl.off_q;
  sp.q_slot_bytes = pl.q_slot_bytes;
  sp.off_stage = pl.off_stage;
  sp.stage_bytes = pl.stage_bytes;
  sp.kv_bytes = pl.stage_bytes;
  sp.off_xchg = pl.off_xchg;
  sp.team_bytes = pl.team_bytes;
  sp.q_slots = pl.q_slots;
  sp.wait_ns = wait_limit_ns(opts);
  sp.starve_cta = -1;
  sp.pair_pages = pl.pair;
  sp.off_buf = pl.off_buf;
  sp.off_qring = pl.off_qring;
  sp.seg_cost = pl.tc ? pl.seg_cost : 0;

  pa::MergeParams mp = {};
  mp.out = sp.out;
  mp.out_stride_t = sp.out_stride_t;
  mp.out_stride_h = sp.out_stride_h;
  mp.lse = sp.lse;
  mp.lse_stride_t = sp.lse_stride_t;
  mp.lse_stride_h = sp.lse_stride_h;
  mp.seq_lens = sp.seq_lens;
  mp.qsl = sp.qsl;
  mp.num_seqs = sp.num_seqs;
  mp.num_tokens = sp.num_tokens;
  mp.G = pl.Gc;
  mp.HC = 1;
  mp.NC = pl.NC;
  mp.R_max = pl.R_max;
  mp.max_qlen = max_qlen;
  mp.split_grid = pl.grid * pl.nteam;
  mp.v_scale = sp.v_scale;
  mp.ws_unit = sp.ws_unit;
  mp.ws_ml = sp.ws_ml;
  mp.ws_o = sp.ws_o;
  mp.err = sp.err;

  cudaEvent_t ev0 = opts ? static_cast<cudaEvent_t>(opts->split_start_event) : nullptr;
  cudaEvent_t ev1 = opts ? static_cast<cudaEvent_t>(opts->split_stop_event) : nullptr;
  const bool pdl = !(opts && opts->disable_pdl);
  cudaError_t e;
  unsigned int rec_flags = cudaEventRecordDefault;
  if (ev0 || ev1) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if ((e = cudaStreamIsCapturing(stream, &cs)) != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cs == cudaStreamCaptureStatusActive) rec_flags = cudaEventRecordExternal;
  }
  if (ev0 && (e = cudaEventRecordWithFlags(ev0, stream, rec_flags)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord(start)");
  if (pl.tc)
    e = pa::launch_mla_tc(esz == 1, pl.rpad, tm, tb, sp, pl.grid, static_cast<int>(pl.smem), pdl && !ev0, stream);
  else
    e = pa::launch_mla(esz == 1, pl.RT, tm, sp, pl.grid, static_cast<int>(pl.smem), pdl && !ev0, stream);
  if (e != cudaSuccess) return cuda_fail(e, "MLA split kernel launch");
  if (ev1 && (e = cudaEventRecordWithFlags(ev1, stream, rec_flags)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord(stop)");
  if ((e = pa::launch_merge_mla(mp, static_cast<int>(B) * pl.NC, pl.R_max, pdl && !ev1, stream)) != cudaSuccess)
    return cuda_fail(e, "MLA merge kernel launch");
  return PA_OK;
}

}  // namespace

namespace pa {
// Lets other translation units of the library report a detailed message
// through paged_attn_last_error_message().
void set_last_error_message(const std::string& msg) { t_last_error = msg; }
}  // namespace pa

extern "C" {

int paged_attn_decode_ex(const pa_tensor_t* q, const pa_tensor_t* k_cache, const pa_tensor_t* v_cache,
                         const pa_tensor_t* block_tables, const pa_tensor_t* seq_lens,
                         const pa_tensor_t* query_start_loc, int32_t max_query_len, float scale, float k_scale,
                         float v_scale, const pa_tensor_t* out, const pa_tensor_t* lse, const pa_options_t* opts,
                         pa_stream_t stream) {
  t_last_error.clear();
  return decode_impl(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, max_query_len, scale, k_scale,
                     v_scale, out, lse, opts, reinterpret_cast<cudaStream_t>(stream));
}

int paged_attn_decode(const pa_tensor_t* q, const pa_tensor_t* k_cache, const pa_tensor_t* v_cache,
                      const pa_tensor_t* block_tables, const pa_tensor_t* seq_lens, const pa_tensor_t* query_start_loc,
                      int32_t max_query_len, float scale, float k_scale, float v_scale, const pa_tensor_t* out,
                      const pa_tensor_t* lse, pa_stream_t stream) {
  return paged_attn_decode_ex(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, max_query_len, scale,
                              k_scale, v_scale, out, lse, nullptr, stream);
}

static int cache_write_impl(const pa_tensor_t* key, const pa_tensor_t* value, const pa_tensor_t* slot_mapping,
                            const pa_tensor_t* k_cache, const pa_tensor_t* v_cache, float k_scale, float v_scale,
                            const pa_tensor_t* kts, const pa_tensor_t* vts, pa_stream_t stream) {
  t_last_error.clear();
  int st;
  if ((st = check_tensor(key, "key", 3, false)) || (st = check_tensor(value, "value", 3, false)) ||
      (st = check_tensor(slot_mapping, "slot_mapping", 1, false)) || (st = check_tensor(k_cache, "k_cache", 4, false)) ||
      (st = check_tensor(v_cache, "v_cache", 4, false)))
    return st;
  if (key->dtype != PA_BF16 || value->dtype != PA_BF16) return fail(PA_ERR_INVALID_ARG, "key and value must be bf16");
  if (slot_mapping->dtype != PA_I32) return fail(PA_ERR_INVALID_ARG, "slot_mapping must be int32");
  if (k_cache->dtype != PA_BF16 && k_cache->dtype != PA_FP8_E4M3)
    return fail(PA_ERR_INVALID_ARG, "k_cache must be bf16 or fp8 e4m3");
  if (v_cache->dtype != k_cache->dtype) return fail(PA_ERR_INVALID_ARG, "v_cache dtype differs from k_cache");
  const int64_t T = key->shape[0], Hkv = key->shape[1], D = key->shape[2];
  for (int d = 0; d < 3; ++d)
    if (value->shape[d] != key->shape[d]) return fail(PA_ERR_INVALID_ARG, "value shape differs from key");
  if (slot_mapping->shape[0] != T) return fail(PA_ERR_INVALID_ARG, "slot_mapping needs one entry per token");
  if (slot_mapping->stride[0] != 1) return fail(PA_ERR_INVALID_ARG, "slot_mapping must be contiguous");
  if (k_cache->shape[1] != kPageSize) return fail(PA_ERR_UNSUPPORTED, "page size must be 16");
  if (k_cache->shape[2] != Hkv || k_cache->shape[3] != D)
    return fail(PA_ERR_INVALID_ARG, "cache [NB, 16, Hkv, D] does not match key [T, Hkv, D]");
  for (int d = 0; d < 4; ++d)
    if (v_cache->shape[d] != k_cache->shape[d]) return fail(PA_ERR_INVALID_ARG, "v_cache shape differs from k_cache");
  if (D % 8 != 0 || D > 512) return fail(PA_ERR_UNSUPPORTED, "head_dim must be a multiple of 8 up to 512");
  if (T > (int64_t(1) << 30) || Hkv > 4096 || k_cache->shape[0] > (int64_t(1) << 31) - 1)
    return fail(PA_ERR_UNSUPPORTED, "tensor extents too large");
  for (const pa_tensor_t* t : {key, value}) {
    if (t->stride[2] != 1 || t->stride[1] % 8 != 0 || t->stride[0] % 8 != 0 || !aligned(t->data, 16))
      return fail(PA_ERR_INVALID_ARG, "key/value rows must be contiguous and 16-byte aligned (strides multiple of 8)");
  }
  const int esz = k_cache->dtype == PA_FP8_E4M3 ? 1 : 2;
  for (const pa_tensor_t* c : {k_cache, v_cache}) {
    if (c->stride[3] != 1) return fail(PA_ERR_INVALID_ARG, "KV cache last dim must be contiguous");
    for (int d = 0; d < 3; ++d)
      if ((c->stride[d] * esz) % 16 != 0) return fail(PA_ERR_INVALID_ARG, "KV cache strides must be multiples of 16 bytes");
    if (!aligned(c->data, 16)) return fail(PA_ERR_INVALID_ARG, "KV cache data must be 16-byte aligned");
  }
  const bool tok = kts != nullptr;
  if (tok) {
    if (esz != 1) return fail(PA_ERR_INVALID_ARG, "per-token quantisation needs fp8 caches");
    const pa_tensor_t* ts[2] = {kts, vts};
    const char* nm[2] = {"k_token_scales", "v_token_scales"};
    for (int x = 0; x < 2; ++x) {
      if ((st = check_tensor(ts[x], nm[x], 3, false)) != PA_OK) return st;
      if (ts[x]->dtype != PA_F32) return fail(PA_ERR_INVALID_ARG, "%s must be float32", nm[x]);
      if (ts[x]->shape[0] != k_cache->shape[0] || ts[x]->shape[1] != Hkv || ts[x]->shape[2] != kPageSize)
        return fail(PA_ERR_INVALID_ARG, "%s must have shape [NB, Hkv, 16]", nm[x]);
      if (!aligned(ts[x]->data, 4)) return fail(PA_ERR_INVALID_ARG, "%s must be 4-byte aligned", nm[x]);
    }
  } else if (esz == 1 && (!std::isfinite(k_scale) || !std::isfinite(v_scale) || k_scale == 0.f || v_scale == 0.f)) {
    return fail(PA_ERR_INVALID_ARG, "fp8 caches need finite, non-zero k_scale and v_scale");
  }
  if (T == 0) return PA_OK;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds, nullptr)) != PA_OK) return st;
  pa::CacheWriteParams p = {};
  p.key = static_cast<const uint16_t*>(key->data);
  p.value = static_cast<const uint16_t*>(value->data);
  p.k_stride_t = key->stride[0];
  p.k_stride_h = key->stride[1];
  p.v_stride_t = value->stride[0];
  p.v_stride_h = value->stride[1];
  p.slot_mapping = static_cast<const int32_t*>(slot_mapping->data);
  p.k_cache = static_cast<uint8_t*>(k_cache->data);
  p.v_cache = static_cast<uint8_t*>(v_cache->data);
  p.kc_stride_page = k_cache->stride[0];
  p.kc_stride_slot = k_cache->stride[1];
  p.kc_stride_head = k_cache->stride[2];
  p.vc_stride_page = v_cache->stride[0];
  p.vc_stride_slot = v_cache->stride[1];
  p.vc_stride_head = v_cache->stride[2];
  p.num_tokens = static_cast<int32_t>(T);
  p.num_kv_heads = static_cast<int32_t>(Hkv);
  p.head_dim = static_cast<int32_t>(D);
  p.num_pages = static_cast<int32_t>(k_cache->shape[0]);
  p.k_scale = tok ? 0.f : k_scale;
  p.v_scale = tok ? 0.f : v_scale;
  if (tok) {
    p.k_tok = static_cast<float*>(kts->data);
    p.v_tok = static_cast<float*>(vts->data);
    p.ks_stride_page = kts->stride[0];
    p.ks_stride_head = kts->stride[1];
    p.ks_stride_slot = kts->stride[2];
    p.vs_stride_page = vts->stride[0];
    p.vs_stride_head = vts->stride[1];
    p.vs_stride_slot = vts->stride[2];
  }
  p.err = ds->status;
  cudaError_t e = pa::launch_cache_write(esz == 1, p, ds->num_sms, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cache write kernel launch");
  return PA_OK;
}

int paged_attn_cache_write(const pa_tensor_t* key, const pa_tensor_t* value, const pa_tensor_t* slot_mapping,
                           const pa_tensor_t* k_cache, const pa_tensor_t* v_cache, float k_scale, float v_scale,
                           pa_stream_t stream) {
  return cache_write_impl(key, value, slot_mapping, k_cache, v_cache, k_scale, v_scale, nullptr, nullptr, stream);
}

int paged_attn_cache_write_per_token(const pa_tensor_t* key, const pa_tensor_t* value,
                                     const pa_tensor_t* slot_mapping, const pa_tensor_t* k_cache,
                                     const pa_tensor_t* v_cache, const pa_tensor_t* k_token_scales,
                                     const pa_tensor_t* v_token_scales, pa_stream_t stream) {
  if (k_token_scales == nullptr || v_token_scales == nullptr) {
    t_last_error.clear();
    return fail(PA_ERR_INVALID_ARG, "k_token_scales and v_token_scales descriptors are required");
  }
  return cache_write_impl(key, value, slot_mapping, k_cache, v_cache, 1.f, 1.f, k_token_scales, v_token_scales,
                          stream);
}

int paged_attn_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t kv_dtype,
                    int32_t max_query_len, const pa_options_t* opts, pa_plan_t* plan) {
  t_last_error.clear();
  if (plan == nullptr) return fail(PA_ERR_INVALID_ARG, "plan pointer is NULL");
  int st = check_shape_args(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype, max_query_len);
  if (st != PA_OK) return st;
  if ((st = check_variant_option(opts, kv_dtype, (num_q_heads / num_kv_heads) * static_cast<int64_t>(max_query_len))) !=
      PA_OK)
    return st;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds, nullptr)) != PA_OK) return st;
  Plan pl{};
  if ((st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype, max_query_len, opts, ds->num_sms,
                      ds->smem_optin, &pl)) != PA_OK)
    return st;
  plan->num_ctas = pl.grid;
  plan->heads_per_cta = pl.HC;
  plan->row_tiles = pl.MT;
  plan->num_stages = pl.nstage;
  plan->threads_per_cta = pl.threads;
  plan->smem_bytes = static_cast<int32_t>(pl.smem);
  plan->min_pages_per_cta = pl.min_pages;
  plan->merge_rows = pl.HC * pl.R_max;
  plan->page_pairing = pl.pair;
  plan->workspace_bytes = static_cast<int64_t>(pl.ws_bytes);
  plan->variant = pl.tc ? 1 : 0;
  plan->block_pages = pl.tc ? pl.block_pages : (pl.pair ? 2 : 1);
  return PA_OK;
}

int paged_attn_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t kv_dtype, int32_t max_query_len, size_t* bytes) {
  if (bytes == nullptr) return fail(PA_ERR_INVALID_ARG, "bytes pointer is NULL");
  pa_plan_t plan;
  const int st = paged_attn_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype, max_query_len, nullptr, &plan);
  if (st == PA_OK) *bytes = static_cast<size_t>(plan.workspace_bytes);
  return st;
}

int paged_attn_reserve(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t kv_dtype, int32_t max_query_len) {
  t_last_error.clear();
  int st = check_shape_args(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype, max_query_len);
  if (st != PA_OK) return st;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds, nullptr)) != PA_OK) return st;
  Plan pl{};
  if ((st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype, max_query_len, nullptr, ds->num_sms,
                      ds->smem_optin, &pl)) != PA_OK)
    return st;
  return grow_workspace(ds, pl.ws_bytes);
}

int paged_attn_mla_decode_ex(const pa_tensor_t* q, const pa_tensor_t* kv_cache, const pa_tensor_t* block_tables,
                             const pa_tensor_t* seq_lens, const pa_tensor_t* query_start_loc, int32_t max_query_len,
                             float scale, float kv_scale, const pa_tensor_t* out, const pa_tensor_t* lse,
                             const pa_options_t* opts, pa_stream_t stream) {
  t_last_error.clear();
  return mla_decode_impl(q, kv_cache, block_tables, seq_lens, query_start_loc, max_query_len, scale, kv_scale, out, lse,
                         opts, reinterpret_cast<cudaStream_t>(stream));
}

int paged_attn_mla_decode(const pa_tensor_t* q, const pa_tensor_t* kv_cache, const pa_tensor_t* block_tables,
                          const pa_tensor_t* seq_lens, const pa_tensor_t* query_start_loc, int32_t max_query_len,
                          float scale, float kv_scale, const pa_tensor_t* out, const pa_tensor_t* lse,
                          pa_stream_t stream) {
  return paged_attn_mla_decode_ex(q, kv_cache, block_tables, seq_lens, query_start_loc, max_query_len, scale, kv_scale,
                                  out, lse, nullptr, stream);
}

int paged_attn_mla_plan(int32_t num_seqs, int32_t num_q_heads, int32_t kv_dtype, int32_t max_query_len,
                        const pa_options_t* opts, pa_plan_t* plan) {
  t_last_error.clear();
  if (plan == nullptr) return fail(PA_ERR_INVALID_ARG, "plan pointer is NULL");
  int st = check_mla_shape(num_seqs, num_q_heads, kv_dtype, max_query_len, opts);
  if (st != PA_OK) return st;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds, nullptr)) != PA_OK) return st;
  MlaPlan pl{};
  if ((st = make_mla_plan(num_seqs, num_q_heads, kv_dtype, max_query_len, opts, ds->num_sms, ds->smem_optin, &pl)) !=
      PA_OK)
    return st;
  plan->num_ctas = pl.grid;
  plan->heads_per_cta = pl.Gc;
  plan->row_tiles = pl.RT;
  plan->num_stages = pl.nstage;
  plan->threads_per_cta = pl.threads;
  plan->smem_bytes = static_cast<int32_t>(pl.smem);
  plan->min_pages_per_cta = pl.min_pages;
  plan->merge_rows = pl.R_max;
  plan->page_pairing = pl.pair;
  plan->workspace_bytes = static_cast<int64_t>(pl.ws_bytes);
  plan->variant = pl.tc ? 3 : 2;
  plan->block_pages = pl.tc ? 3 : (pl.pair ? 2 : 1);
  return PA_OK;
}

int paged_attn_mla_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t kv_dtype, int32_t max_query_len,
                                  size_t* bytes) {
  if (bytes == nullptr) return fail(PA_ERR_INVALID_ARG, "bytes pointer is NULL");
  pa_plan_t plan;
  const int st = paged_attn_mla_plan(num_seqs, num_q_heads, kv_dtype, max_query_len, nullptr, &plan);
  if (st == PA_OK) *bytes = static_cast<size_t>(plan.workspace_bytes);
  return st;
}

int paged_attn_mla_reserve(int32_t num_seqs, int32_t num_q_heads, int32_t kv_dtype, int32_t max_query_len) {
  t_last_error.clear();
  int st = check_mla_shape(num_seqs, num_q_heads, kv_dtype, max_query_len, nullptr);
  if (st != PA_OK) return st;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds, nullptr)) != PA_OK) return st;
  MlaPlan pl{};
  if ((st = make_mla_plan(num_seqs, num_q_heads, kv_dtype, max_query_len, nullptr, ds->num_sms, ds->smem_optin,
                          &pl)) != PA_OK)
    return st;
  return grow_workspace(ds, pl.ws_bytes);
}

int paged_attn_release(void) {
  t_last_error.clear();
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  int st = device_state(&ds, nullptr);
  if (st != PA_OK) return st;
  if (ds->ws) {
    cudaError_t e = cudaFree(ds->ws);
    ds->ws = nullptr;
    ds->ws_bytes = 0;
    if (e != cudaSuccess) return cuda_fail(e, "cudaFree(workspace)");
  }
  return PA_OK;
}

int paged_attn_device_status(uint32_t* flags, int32_t clear) {
  t_last_error.clear();
  if (flags == nullptr) return fail(PA_ERR_INVALID_ARG, "flags pointer is NULL");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  int st = device_state(&ds, nullptr);
  if (st != PA_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  if ((e = cudaMemcpy(flags, ds->status, sizeof(uint32_t), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "reading the status word");
  if (clear && (e = cudaMemset(ds->status, 0, sizeof(uint32_t))) != cudaSuccess)
    return cuda_fail(e, "clearing the status word");
  if (clear && (e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  return PA_OK;
}

const char* paged_attn_error_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK: success";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG: invalid argument (shape, dtype, stride, alignment or NULL pointer)";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: outside the supported envelope";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: split workspace too small (or growth needed during capture)";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: a CUDA call or kernel launch failed";
    default: return "unknown paged_attn status";
  }
}

const char* paged_attn_last_error_message(void) { return t_last_error.c_str(); }

int32_t paged_attn_version(void) { return 100; }

}  // extern "C"
