// bf16-cache instantiations of the split kernel (head_dim 64 and 128).
#include "pa_split.cuh"

namespace pa {

cudaError_t launch_split_bf16(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
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
  if (head_dim == 128) return cudaLaunchKernelEx(&cfg, pa_split_kernel<128, false>, tk, tv, p);
  if (head_dim == 64) return cudaLaunchKernelEx(&cfg, pa_split_kernel<64, false>, tk, tv, p);
  return cudaErrorInvalidValue;
}

cudaError_t set_split_smem_limits_bf16(int smem) {
  cudaError_t e = cudaFuncSetAttribute(pa_split_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(pa_split_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace pa
