/* synth.cu - device fills of the seeded input generator (see synth.h). */
#include <cuda_runtime.h>
#include "synth.h"
#include "synth_core.h"

__global__ void syn_normal_blocks_kernel(uint16_t* __restrict__ out, int64_t nblk,
                                         int64_t blk_elems, int64_t blk_stride, int64_t i0,
                                         uint32_t seed, uint32_t stream, float scale) {
  int64_t total = nblk * blk_elems;
  int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += step) {
    int64_t j = e / blk_elems, r = e - j * blk_elems;
    float x = (float)syn_ih8((uint64_t)(i0 + e), seed, stream) * scale;
    out[j * blk_stride + r] = syn_f32_to_bf16_rne(x);
  }
}

extern "C" int ppsyn_normal_bf16_dev_blocks(uint16_t* out, int64_t nblk, int64_t blk_elems,
                                            int64_t blk_stride, int64_t i0, uint32_t seed,
                                            uint32_t stream, float scale, void* cuda_stream) {
  if (nblk <= 0 || blk_elems <= 0) return 0;
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  int64_t total = nblk * blk_elems;
  int64_t want = (total + 255) / 256;
  int grid = (int)(want < (int64_t)nsm * 16 ? want : (int64_t)nsm * 16);
  syn_normal_blocks_kernel<<<grid, 256, 0, (cudaStream_t)cuda_stream>>>(
      out, nblk, blk_elems, blk_stride, i0, seed, stream, scale);
  return (int)cudaGetLastError();
}

extern "C" int ppsyn_normal_bf16_dev(uint16_t* out, int64_t n, int64_t i0, uint32_t seed,
                                     uint32_t stream, float scale, void* cuda_stream) {
  return ppsyn_normal_bf16_dev_blocks(out, 1, n, n, i0, seed, stream, scale, cuda_stream);
}
