// stage_copy.cu -- copy a decode step's inputs or outputs between page-locked host memory
// and the device with the SMs.
//
// The pages describe no such operation; it serves the step as a host program runs it: the
// step's inputs (q, the new K/V rows, slots, tables, lengths) go from one page-locked host
// buffer to the device, and the step's output comes back.  On GB300 a copy-engine transfer
// of a few hundred KiB costs about 10 us, nearly all of it latency; the SMs load page-locked
// host memory directly over the host link (it is addressed by the same pointer on both
// sides), so one wave of threads, each moving 16-byte words, finishes in a few.  The kernel
// is chained to its neighbours by programmatic dependent launch: it waits for the work
// before it and lets the next kernel's CTAs be scheduled at once.
#include <cuda_runtime.h>

#include <algorithm>

#include "decode_launch.cuh"

namespace pkv {

__global__ void __launch_bounds__(256) stage_copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                         size_t n16) {
  pdl_wait();  // the work before this copy (e.g. the kernel that wrote `src`) has completed
  pdl_launch_dependents();
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) dst[i] = src[i];
}

cudaError_t launch_stage_copy(void* dst, const void* src, size_t bytes, int sm_count, cudaStream_t stream) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  // one 16-byte word per thread up to four CTAs of 256 threads per SM, then a grid stride
  const size_t want = (n16 + 255) / 256;
  const unsigned ctas = static_cast<unsigned>(std::min<size_t>(want, static_cast<size_t>(sm_count) * 4));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stage_copy_kernel, static_cast<uint4*>(dst), static_cast<const uint4*>(src), n16);
}

}  // namespace pkv
