// sf_linear_noalloc: the weight-streaming GEMM of sf_linear for callers that
// cannot hand the library any scratch memory.
//
// Some callers cannot call cudaMalloc at the point where they need a
// projection: plug-ins whose host framework owns every device allocation
// through its own pool, and latency-critical loops where cudaMalloc's
// implicit device synchronisation is not acceptable. For them the split-K
// scratch lives in a file-scope device array that is part of the loaded
// library image.
//
// The array is sized for sf_linear's workspace at up to kMaxRows output rows,
// kMaxK inputs and SF_MAX_ROWS token rows (about 38 MB); every GPU that loads
// the library holds it until the process exits. All calls share it and it
// keeps the previous call's contents: the arrival counters that must start at
// zero are cleared by every call, and calls that overlap on the GPU (e.g. on
// two streams at once) race on it. The array's device address is looked up
// once per device index and kept for the life of the process, so a context
// reset (cudaDeviceReset) after the first call is not supported.
#include <mutex>

#include "sf_kernels.h"

namespace {

constexpr int kMaxRows = 1 << 20;   // largest N accepted
constexpr size_t kPartBytes = (size_t)2048 * sf::kGroupRows * sf::kBlockRows * 4;   // sf_linear's tile area
constexpr int kMaxK = 1 << 16;      // largest K accepted (fragment-ordered copy of x)
constexpr size_t kScratchBytes = kPartBytes + (size_t)(kMaxRows / sf::kBlockRows) * sf::kMaxGroups * 4 + 3 * 256 +
                                 (size_t)(kMaxK / 64) * ((sf::kRows + 3) / 4) * 1024;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per
// device (in host code the symbol itself is only a host-side stand-in).
sf_status scratch_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return sf::set_error(SF_ERR_CUDA, "sf_linear_noalloc: no usable current CUDA device");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p)
      return sf::set_error(SF_ERR_CUDA, "sf_linear_noalloc: cudaGetSymbolAddress failed: %s",
                           cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SF_OK;
}

}  // namespace

extern "C" sf_status sf_linear_noalloc(const void* d_w, int32_t N, int32_t K, int32_t ld, const float* d_x,
                                       int32_t M, float* d_y, void* cuda_stream) {
  if (N < 1 || N > kMaxRows)
    return sf::set_error(SF_ERR_ARG, "sf_linear_noalloc: N = %d is outside 1..%d, the limit of the static scratch",
                         N, kMaxRows);
  if (K < 8 || K % 8)
    return sf::set_error(SF_ERR_ARG, "sf_linear_noalloc: K = %d must be a positive multiple of 8", K);
  const size_t need = sf_linear_workspace_bytes(N, K);
  if (need > kScratchBytes)
    return sf::set_error(SF_ERR_ARG, "sf_linear_noalloc: N = %d, K = %d needs %zu scratch bytes, the static "
                         "scratch holds %zu", N, K, need, kScratchBytes);
  void* scratch = nullptr;
  const sf_status s = scratch_ptr(&scratch);
  if (s != SF_OK) return s;
  // sf_linear clears the arrival counters on the stream before its launch
  // and allocates nothing; it only receives the static array as workspace.
  return sf_linear(d_w, N, K, ld, d_x, M, d_y, scratch, cuda_stream);
}
