// la_forward_noalloc: the forward for callers that cannot allocate device
// memory while they run — for example code running inside an allocator
// callback, or under a memory-pool policy that forbids new allocations.
// The per-segment states that la_forward takes from its stream-ordered pool
// live here in one fixed, file-scope device array instead.
#include "linattn.h"

#include "internal.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

// Scratch for the per-segment states: 4 Mi floats (16 MiB) on every device
// that loads the library, held until the process exits.
constexpr size_t kScratchFloats = size_t(4) << 20;
__device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is taken
// with cudaGetSymbolAddress once per device, with that device current.
la_status scratch_on_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return LA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return LA_OK;
}

}  // namespace

extern "C" la_status la_forward_noalloc(const la_tensor* q, const la_tensor* k,
                                        const la_tensor* v, const float* decay_a,
                                        la_feature_map feature_map, const la_tensor* omega,
                                        int causal, la_tensor* out, la_stream stream) {
  la::ApiRange range_("la_forward_noalloc");
  return la::forward_in_workspace(q, k, v, decay_a, feature_map, omega, causal, out,
                                  scratch_on_current_device, kScratchFloats,
                                  reinterpret_cast<cudaStream_t>(stream));
}
