// Chunk loaders shared by the fp32 CUDA-core kernels (forward and backward):
// rows of one head into shared memory, with φ applied on the way.
#pragma once

#include "common.cuh"

namespace la {
namespace simt {

constexpr int kThreads = 256;   // threads per CTA of every CUDA-core kernel

// Loads rows [row0, row0+cs) of one head (zero beyond cs) and applies φ.
// f receives φ(x) with row stride FS.  For the Performer map ω is [D, DP]
// row-major in global memory and φ(x)_i = exp(x·ω_i − ½‖x‖²)/√m.
template <typename T, int D, int DP, bool PERF, int CS, int FS>
__device__ void load_features(const T* __restrict__ x, int cs, float* f, float* xraw,
                              float* halfsq, const T* __restrict__ omega) {
  if constexpr (!PERF) {
    for (int e = threadIdx.x; e < CS * D; e += kThreads) {
      const int t = e / D, c = e % D;
      f[t * FS + c] = (t < cs) ? elu1(to_f32(x[(int64_t)t * D + c])) : 0.f;
    }
  } else {
    for (int e = threadIdx.x; e < CS * D; e += kThreads) {
      const int t = e / D;
      xraw[e] = (t < cs) ? to_f32(x[(int64_t)t * D + (e % D)]) : 0.f;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < CS; t += kThreads) {
      float s = 0.f;
      for (int c = 0; c < D; ++c) s += xraw[t * D + c] * xraw[t * D + c];
      halfsq[t] = 0.5f * s;
    }
    __syncthreads();
    const float inv_sqrt_m = rsqrtf((float)DP);
    for (int e = threadIdx.x; e < CS * DP; e += kThreads) {
      const int t = e / DP, i = e % DP;
      float u = 0.f;
      for (int c = 0; c < D; ++c) u += xraw[t * D + c] * to_f32(omega[c * DP + i]);
      f[t * FS + i] = (t < cs) ? expf(u - halfsq[t]) * inv_sqrt_m : 0.f;
    }
  }
}

// Rows [0, cs) of one head into vv with row stride VS (zero beyond cs).
template <typename T, int D, int CS, int VS = D>
__device__ void load_values(const T* __restrict__ v, int cs, float* vv) {
  for (int e = threadIdx.x; e < CS * D; e += kThreads) {
    const int t = e / D, c = e % D;
    vv[t * VS + c] = (t < cs) ? to_f32(v[(int64_t)t * D + c]) : 0.f;
  }
}

}  // namespace simt
}  // namespace la
