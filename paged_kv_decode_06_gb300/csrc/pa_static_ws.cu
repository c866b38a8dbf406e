// paged_attn_decode_static_scratch: the decode entry point for callers that
// must not allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention:
// code that runs under a memory pool or allocator that owns all device memory,
// a runtime that forbids allocation once its steady state starts, or a plug-in
// that has no handle on an allocator at all.  The split kernel needs scratch
// for its partial results, so this entry point takes it from one file-scope
// device array instead of the per-device workspace the library would otherwise
// cudaMalloc.
//
// The array name is only a host-side stand-in; its device address comes from
// cudaGetSymbolAddress, taken once per device with that device current.  The
// library's per-device set-up (the first call of any entry point on a device)
// takes it, which also loads the array's module under CUDA's lazy module
// loading: from then on that GPU holds the 16 MiB until the process exits.  So
// make one call of any entry point on each device before a memory pool takes
// the device's free memory, and before any stream capture.
//
// Every call uses the same array.  Nothing in it has to start at zero (each
// call writes every scratch value before it reads it), but the array keeps the
// previous call's contents, and calls whose GPU work overlaps — on different
// streams, or on different host threads without ordering — race on it.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "paged_attn.h"

namespace pa {
void set_last_error_message(const std::string& msg);
}

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr int kMaxScratchDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

void* g_scratch_dev_ptr[kMaxScratchDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set up once).
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    pa::set_last_error_message(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    return PA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxScratchDevices) {
    pa::set_last_error_message("device ordinal out of range for the static scratch table");
    return PA_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_dev_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      pa::set_last_error_message(std::string("cudaGetSymbolAddress(static scratch): ") + cudaGetErrorString(e));
      return PA_ERR_CUDA;
    }
    g_scratch_dev_ptr[dev] = ptr;
  }
  *out = g_scratch_dev_ptr[dev];
  return PA_OK;
}

}  // namespace

namespace pa {
// Per-device set-up hook (called with the device current): resolves the
// scratch array's address now, so its module is loaded early.
int static_scratch_setup() {
  void* unused = nullptr;
  return scratch_for_current_device(&unused);
}
}  // namespace pa

extern "C" int paged_attn_decode_static_scratch(const pa_tensor_t* q, const pa_tensor_t* k_cache,
                                                const pa_tensor_t* v_cache, const pa_tensor_t* block_tables,
                                                const pa_tensor_t* seq_lens, const pa_tensor_t* query_start_loc,
                                                int32_t max_query_len, float scale, float k_scale, float v_scale,
                                                const pa_tensor_t* out, const pa_tensor_t* lse, pa_stream_t stream) {
  void* scratch = nullptr;
  int st = scratch_for_current_device(&scratch);
  if (st != PA_OK) return st;
  pa_options_t opts = {};
  opts.workspace = scratch;
  opts.workspace_bytes = kStaticScratchBytes;
  st = paged_attn_decode_ex(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, max_query_len, scale,
                            k_scale, v_scale, out, lse, &opts, stream);
  if (st == PA_ERR_WORKSPACE) {
    // Only the size check can fail this way (the workspace is given): say
    // how much the shape needs against the fixed limit.
    size_t need = 0;
    const bool known = q && k_cache && block_tables &&
                       paged_attn_workspace_size(static_cast<int32_t>(block_tables->shape[0]),
                                                 static_cast<int32_t>(q->shape[1]),
                                                 static_cast<int32_t>(k_cache->shape[2]),
                                                 static_cast<int32_t>(q->shape[2]), k_cache->dtype, max_query_len,
                                                 &need) == PA_OK;
    pa::set_last_error_message(
        "this shape needs " + (known ? std::to_string(need) : std::string("more")) +
        " bytes of split scratch; paged_attn_decode_static_scratch has a fixed " +
        std::to_string(kStaticScratchBytes) + "-byte (16 MiB) static scratch array: use paged_attn_decode instead");
    return PA_ERR_WORKSPACE;
  }
  return st;
}
