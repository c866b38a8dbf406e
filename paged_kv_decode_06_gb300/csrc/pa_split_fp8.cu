// fp8 (e4m3fn) cache instantiations of the split kernel (head_dim 64 and 128).
#include "pa_split.cuh"

namespace pa {

cudaError_t launch_split_fp8(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                             int grid, int threads, int smem, cudaStream_t stream) {
  if (head_dim == 128) {
    pa_split_kernel<128, true><<<grid, threads, smem, stream>>>(tk, tv, p);
  } else if (head_dim == 64) {
    pa_split_kernel<64, true><<<grid, threads, smem, stream>>>(tk, tv, p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t set_split_smem_limits_fp8(int smem) {
  cudaError_t e = cudaFuncSetAttribute(pa_split_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(pa_split_kernel<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace pa
