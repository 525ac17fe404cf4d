// gdr_fused.cu -- fused persistent forward (sm_103a) and the device status word.
#include "gdr_internal.cuh"

namespace gdr {

// Nonzero once a bounded wait in a fused kernel ran out; read by gdr_device_status.
__device__ int32_t g_device_status = 0;

bool fused_supported(const FusedArgs &) { return false; }

size_t fused_workspace_bytes(int64_t, int32_t, int32_t) { return 0; }

cudaError_t launch_fused(const FusedArgs &, cudaStream_t) { return cudaErrorNotSupported; }

cudaError_t read_device_status(int32_t *out) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  return cudaMemcpyFromSymbol(out, g_device_status, sizeof(int32_t));
}

cudaError_t clear_device_status() {
  const int32_t zero = 0;
  return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int32_t));
}

}  // namespace gdr
