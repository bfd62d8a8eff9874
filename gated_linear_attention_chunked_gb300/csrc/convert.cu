// convert.cu -- fp32 -> fp16 copy used when the caller passes GLA_FP32 inputs: the chunk
// kernels stream 16-bit tiles, so fp32 q/k/v/dO are narrowed once into the workspace.
// fp16 keeps an 11-bit significand; values with |x| >= 65504 are recorded as DEV_RANGE.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace gla {
namespace {
__global__ void to_half_kernel(const float4* __restrict__ src, uint2* __restrict__ dst,
                               long long n4, DevCtl ctl) {
  bool bad = false;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 x = __ldcs(src + i);
    bad |= fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))) >= 65504.f ||
           x.x != x.x || x.y != x.y || x.z != x.z || x.w != x.w;
    __half2 a = __floats2half2_rn(x.x, x.y), b = __floats2half2_rn(x.z, x.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&a);
    o.y = *reinterpret_cast<uint32_t*>(&b);
    dst[i] = o;
  }
  if (bad) record_error(ctl, DEV_RANGE);
}
}  // namespace

cudaError_t launch_to_half(const float* src, void* dst, long long n, DevCtl ctl,
                           cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const long long n4 = n / 4;  // every tensor here has a multiple of 96 elements
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (n4 + 255) / 256;
  if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
  to_half_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(src),
                                                       reinterpret_cast<uint2*>(dst), n4, ctl);
  return cudaGetLastError();
}

}  // namespace gla
