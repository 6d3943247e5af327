// permute_noalloc.cu -- ft_permute_noalloc: the permute step without any
// device allocation and without a caller-supplied workspace.
//
// Some callers cannot allocate device memory at the moment they call this
// step.  Examples: a serving loop that keeps cudaMalloc/cudaFree off its hot
// path, because those calls can synchronise the whole device and stall other
// streams; or a host framework whose device memory belongs entirely to its own
// pool allocator, with no way to lend scratch to a library.  This entry point
// gives them the same result as ft_permute.  Its scratch (per-chunk expert
// counts and per-chunk starting positions) lives in one file-scope device
// array of fixed size, which every GPU that loads the library keeps until the
// process exits.
#include <mutex>
#include <string>

#include "../../include/ft_moe.h"
#include "ft_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;

// The shared scratch.  Host code must not pass this name to a kernel: on the
// host it is only a stand-in symbol, not a device address.  Its device address
// comes from cudaGetSymbolAddress, taken once per device below.
static __device__ __align__(256) int32_t g_permute_scratch[FT_PERMUTE_NOALLOC_MAX_SCRATCH_BYTES / sizeof(int32_t)];

std::mutex g_mu;
int32_t *g_scratch_addr[kMaxDevices] = {};

// Device address of g_permute_scratch on the current device, looked up on the
// first call made with that device current.
cudaError_t scratch_on_current_device(int32_t **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<int32_t *>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int ft_permute_noalloc(const int32_t *topk_idx, int T, int k, int E, int32_t *offsets, int32_t *perm,
                                  int32_t *inv, void *stream) {
  if (T < 0 || E < 1 || E > ftmoe::kMaxExperts || k < 1 || k > ftmoe::kMaxTopK) {
    ftmoe::set_stateless_error("ft_permute_noalloc: bad T/E/k");
    return FT_ERR_ARG;
  }
  if (!offsets || (T > 0 && (!topk_idx || !perm || !inv))) {
    ftmoe::set_stateless_error("ft_permute_noalloc: NULL pointer");
    return FT_ERR_ARG;
  }
  const size_t need = ftmoe::permute_scratch_ints(T, k, E) * sizeof(int32_t);
  if (need > FT_PERMUTE_NOALLOC_MAX_SCRATCH_BYTES) {
    ftmoe::set_stateless_error("ft_permute_noalloc: needs " + std::to_string(need) +
                               " bytes of scratch (2 * ceil(T/32) * E * 4), above the fixed " +
                               std::to_string((size_t)FT_PERMUTE_NOALLOC_MAX_SCRATCH_BYTES) +
                               "; use ft_permute with a workspace");
    return FT_ERR_ARG;
  }
  int32_t *ws = nullptr;
  cudaError_t e = scratch_on_current_device(&ws);
  if (e != cudaSuccess) {
    ftmoe::set_stateless_error(std::string("ft_permute_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    return FT_ERR_CUDA;
  }
  // Every scratch entry the kernels read is written earlier in the same call
  // (the chunk histograms, then the chunk bases), so nothing has to be cleared.
  const size_t half = ftmoe::permute_scratch_ints(T, k, E) / 2;
  e = ftmoe::launch_permute_only(topk_idx, T, k, E, offsets, perm, inv, ws, ws + half,
                                 reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    ftmoe::set_stateless_error(std::string("ft_permute_noalloc: ") + cudaGetErrorString(e));
    return FT_ERR_CUDA;
  }
  return FT_OK;
}
