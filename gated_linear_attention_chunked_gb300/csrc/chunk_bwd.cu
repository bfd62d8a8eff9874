// chunk_bwd.cu -- chunked backward (placeholder until the tcgen05 kernels land).
#include <cuda_runtime.h>

#include "kernels.h"

namespace gla {

size_t chunk_bwd_workspace_bytes(int B, int T, int H) { return 0; }

cudaError_t launch_chunk_bwd(const BwdArgs& a, DevCtl ctl, cudaStream_t stream) {
  return cudaErrorNotSupported;
}

}  // namespace gla
