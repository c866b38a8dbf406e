// fp8 (e4m3fn) caches with per-token scales: instantiations of the split
// kernel's token-scale variant (head_dim 64 and 128, with and without a
// sliding window).
#include "pa_split.cuh"

namespace pa {

cudaError_t launch_split_fp8_tok(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                                 int grid, int threads, int smem, bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const bool win = p.window > 0;
  if (head_dim == 128)
    return win ? cudaLaunchKernelEx(&cfg, pa_split_kernel<128, true, true, true>, tk, tv, p)
               : cudaLaunchKernelEx(&cfg, pa_split_kernel<128, true, false, true>, tk, tv, p);
  if (head_dim == 64)
    return win ? cudaLaunchKernelEx(&cfg, pa_split_kernel<64, true, true, true>, tk, tv, p)
               : cudaLaunchKernelEx(&cfg, pa_split_kernel<64, true, false, true>, tk, tv, p);
  return cudaErrorInvalidValue;
}

cudaError_t set_split_smem_limits_fp8_tok(int smem) {
  const void* fns[4] = {reinterpret_cast<const void*>(pa_split_kernel<128, true, false, true>),
                        reinterpret_cast<const void*>(pa_split_kernel<128, true, true, true>),
                        reinterpret_cast<const void*>(pa_split_kernel<64, true, false, true>),
                        reinterpret_cast<const void*>(pa_split_kernel<64, true, true, true>)};
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pa
