// bf16-cache instantiations of the split kernel (head_dim 64 and 128).
#include "pa_split.cuh"

namespace pa {

cudaError_t launch_split_bf16(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                              int grid, int threads, int smem, cudaStream_t stream) {
  if (head_dim == 128) {
    pa_split_kernel<128, false><<<grid, threads, smem, stream>>>(tk, tv, p);
  } else if (head_dim == 64) {
    pa_split_kernel<64, false><<<grid, threads, smem, stream>>>(tk, tv, p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t set_split_smem_limits_bf16(int smem) {
  cudaError_t e = cudaFuncSetAttribute(pa_split_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(pa_split_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace pa
