// k_attn_noalloc.cu - pp_ring_attention for callers that cannot allocate device memory.
//
// Some callers of this library may not call cudaMalloc (or hand the library a scratch
// buffer) at the point where they need the attention: a serving host whose device
// memory is owned entirely by a pooling allocator (a framework's caching allocator or
// a pre-reserved arena) that libraries must not bypass or grow, a real-time frame loop
// where an allocation (which can synchronise the device and take milliseconds) would
// break the 80 ms cadence, or a plain C caller without a device allocator.  For them
// the split-K partials and completion tickets live in one file-scope device array
// instead of caller scratch; inputs and outputs are still the caller's.
#include <math.h>

#include <mutex>

#include "pp_internal.cuh"

namespace pp {
namespace {

// Limits of the built-in scratch: slots x heads, ring window, head dim.
constexpr int kNoAllocMaxPairs = 2048;
constexpr int kNoAllocMaxWindow = 3072;
constexpr int kNoAllocMaxHeadDim = 128;
constexpr size_t kNoAllocPartBytes =
    (((size_t)kNoAllocMaxPairs *
      attn_pair_floats(kNoAllocMaxWindow / kAttnChunk, kNoAllocMaxHeadDim) * sizeof(float)) +
     255) & ~(size_t)255;
constexpr size_t kNoAllocCountBytes = (size_t)kNoAllocMaxPairs * sizeof(uint32_t);
constexpr size_t kNoAllocQopBytes = (size_t)kNoAllocMaxPairs * 2 * kNoAllocMaxHeadDim * 2;
constexpr size_t kNoAllocBytes = kNoAllocPartBytes + kNoAllocCountBytes + kNoAllocQopBytes;
// 2048 pairs x 3264 floats of partials (25.5 MiB) + 8 KiB of tickets + 1 MiB of query
// operand: the figure the header states
static_assert(kNoAllocBytes == 27795456, "the documented size of the built-in scratch");

// Every GPU that loads the library holds this array (27,795,456 bytes, about 26.5 MiB)
// until exit.
static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// The device address of g_attn_scratch on the current device (looked up once per
// device; in host code the array's name is only a host-side stand-in).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace pp

using namespace pp;

extern "C" int pp_ring_attention_noalloc(const float* q, const uint16_t* k, const uint16_t* v,
                                         int64_t slot_stride, const int32_t* n_valid, int B,
                                         int H, int head_dim, int window, float* out,
                                         uint32_t* status, void* stream) {
  if (B < 1 || H < 1 || window < 1) return PP_EINVAL;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return PP_EINVAL;
  if ((int64_t)B * H > kNoAllocMaxPairs || window > kNoAllocMaxWindow ||
      head_dim > kNoAllocMaxHeadDim)
    return PP_E_RANGE;
  if (!q || !k || !v || !n_valid || !out || slot_stride < 0) return PP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v)) & 15)
    return PP_EINVAL;
  if (slot_stride & 7) return PP_EINVAL;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return PP_E_CUDA;

  AttnArgs a{};
  a.q = q;
  a.q_ld = H * head_dim;
  a.q_scale = 1.4426950408889634f / sqrtf((float)head_dim);
  a.k = k;
  a.v = v;
  a.slot_stride = (size_t)slot_stride;
  a.n_valid = n_valid;
  a.H = H;
  a.W = window;
  a.nc_max = (window + kAttnChunk - 1) / kAttnChunk;
  a.out = out;
  a.out_ld = H * head_dim;
  a.op = nullptr;
  a.status = status;
  char* sp = reinterpret_cast<char*>(base);
  a.part = reinterpret_cast<float*>(sp);
  a.count = reinterpret_cast<uint32_t*>(sp + kNoAllocPartBytes);
  AttnMaps maps;
  if (head_dim == 128) {
    a.q_op = reinterpret_cast<uint16_t*>(sp + kNoAllocPartBytes + kNoAllocCountBytes);
    if (!attn_maps(&maps, k, v, (size_t)slot_stride, B, H, window, head_dim, a.q_op, B * H))
      return PP_EINVAL;
  }
  cudaStream_t s = (cudaStream_t)stream;
  // the array keeps the previous call's contents: the tickets must start at zero
  cudaError_t err = cudaMemsetAsync(a.count, 0, (size_t)B * H * sizeof(uint32_t), s);
  if (err == cudaSuccess && head_dim == 128) err = launch_q_split(a, B, head_dim, s);
  if (err == cudaSuccess) err = launch_attn_args(a, B, head_dim, &maps, 0, s);
  return err == cudaSuccess ? PP_OK : PP_E_CUDA;
}
