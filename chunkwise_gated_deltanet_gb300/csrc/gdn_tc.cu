// tcgen05 tensor-core chunkwise Gated DeltaNet forward (bf16 in, fp32 state).
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {

// Set by a kernel when a bounded wait gives up; read and cleared by the host.
__device__ int g_tc_status = 0;

bool tc_supported(int, int, int, int) { return false; }

int tc_launches(const FwdArgs&) { return 0; }

cudaError_t launch_tc(const FwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }

int tc_read_and_clear_status(cudaStream_t stream, cudaError_t* err) {
  int v = 0;
  *err = cudaMemcpyFromSymbolAsync(&v, g_tc_status, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
  if (*err == cudaSuccess) *err = cudaStreamSynchronize(stream);
  if (*err != cudaSuccess || v == 0) return v;
  const int zero = 0;
  *err = cudaMemcpyToSymbolAsync(g_tc_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
  if (*err == cudaSuccess) *err = cudaStreamSynchronize(stream);
  return v;
}

}  // namespace gdn
