// miss_copy.cu -- LRU misses streamed into their slots by a kernel.
//
// "FreeToken: Run Frontier MoE Models on Your Own GPU, and the RAM It Takes",
// section "Why a Huge MoE Model Fits on One Consumer GPU": an expert that is
// not in the GPU cache is streamed from host RAM over PCIe.
//
// The route kernel leaves the call's miss list {key, slot} in device memory.
// This kernel, queued on a copy stream behind the route kernel, reads each
// missed blob from pinned host memory (device-visible mapping) with 16-byte
// loads, consecutive threads on consecutive addresses, and stores it into the
// slot.  No host thread reads the miss list or issues a copy, so the call
// never waits for the GPU and can be captured in a CUDA graph.  A launch
// copies up to two byte ranges of every miss: the FFN issues the gate/up rows
// (with the global scales) first and the down rows second, so that the
// misses' gate/up kernel can start while the down rows still cross PCIe.
#include "wait_dev.cuh"

namespace ftmoe {

namespace {

constexpr int kCopyThreads = 512;

__global__ void __launch_bounds__(kCopyThreads) miss_copy_kernel(MissCopyArgs a, int s0, int s1) {
  copy_misses(a, s0, s1, (long long)blockIdx.x * blockDim.x + threadIdx.x, (long long)gridDim.x * blockDim.x);
}

}  // namespace

// One CTA per SM: 32 KB of loads in flight per SM and round (4.8 MB on 148
// SMs), far more than the PCIe link holds in flight, with room left on each
// SM for the FFN kernels that run beside it.
cudaError_t launch_miss_copy(const MissCopyArgs &a, int s0, int s1, cudaStream_t s) {
  miss_copy_kernel<<<tc_num_sms(), kCopyThreads, 0, s>>>(a, s0, s1);
  return cudaGetLastError();
}

}  // namespace ftmoe
