// k_rvq.cu - Mimi RVQ dequantisation, the first step after the tick: the latent of each
// frame is the sum of the codebook entries its codes select, one entry per codebook,
// added in codebook order in fp32.  One CTA row per frame; each thread owns four
// consecutive latent dims (16-byte loads of each selected entry and of the output).
#include "pp_internal.cuh"

namespace pp {

namespace {

constexpr int kRvqThreads = 128;
constexpr int kRvqMaxBooks = 32;

__global__ void __launch_bounds__(kRvqThreads)
    k_rvq(const int32_t* __restrict__ codes, int code_stride, int n_books,
          const float* __restrict__ cb, int card, int dim, float* __restrict__ out,
          uint32_t* status) {
  pdl_wait_and_trigger();
  const size_t f = blockIdx.x;
  const int d4 = blockIdx.y * kRvqThreads + threadIdx.x;   // float4 index within the frame
  if (d4 * 4 >= dim) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  bool bad = false;
  for (int k = 0; k < n_books; ++k) {
    const int32_t c = __ldg(codes + f * code_stride + k);
    if (c < 0) continue;             // a closed slot's -1: no frame, adds nothing
    if (c >= card) {
      bad = true;
      continue;
    }
    const float4 e =
        __ldg(reinterpret_cast<const float4*>(cb + ((size_t)k * card + c) * dim) + d4);
    acc.x += e.x;
    acc.y += e.y;
    acc.z += e.z;
    acc.w += e.w;
  }
  reinterpret_cast<float4*>(out + f * dim)[d4] = acc;
  if (bad && status && d4 == 0) atomicOr(status, PP_S_INDEX);
}

}  // namespace

}  // namespace pp

using namespace pp;

extern "C" int pp_rvq_dequantize(const int32_t* codes, int code_stride, int n_frames, int n_books,
                                 const float* codebooks, int card, int dim, float* out,
                                 uint32_t* status, void* stream) {
  if (n_frames < 0 || n_books < 1 || n_books > kRvqMaxBooks || card < 1 || dim < 4 ||
      dim % 4 != 0 || code_stride < n_books)
    return PP_EINVAL;
  if (n_frames == 0) return PP_OK;
  if (!codes || !codebooks || !out) return PP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(codebooks) | reinterpret_cast<uintptr_t>(out)) & 15)
    return PP_EINVAL;
  if (reinterpret_cast<uintptr_t>(codes) & 3) return PP_EINVAL;
  const dim3 grid((unsigned)n_frames, (unsigned)((dim / 4 + kRvqThreads - 1) / kRvqThreads));
  const cudaError_t err =
      launch_k(k_rvq, grid, dim3(kRvqThreads), 0, (cudaStream_t)stream, 1, codes, code_stride,
               n_books, codebooks, card, dim, out, status);
  return err == cudaSuccess ? PP_OK : PP_E_CUDA;
}
