// Device helpers shared by the kernels of liblinattn.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace la {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// φ(x) = elu(x) + 1 with α = 1 ("Linear Attention Research 2026", Linear
// Transformer): x + 1 for x > 0, e^x otherwise — computed as
// max(x, 0) + exp(min(x, 0)), which is the same value (exp(0) = 1 exactly)
// without a data-dependent branch.
__device__ __forceinline__ float elu1(float x) { return fmaxf(x, 0.f) + expf(fminf(x, 0.f)); }

// Weight of the newest token in eq (10)–(11): 1 − a, except a = 1 which is
// the plain running sum of eq (7)–(8).
__device__ __forceinline__ float new_token_weight(float a) { return a == 1.f ? 1.f : 1.f - a; }

// a^k for integer k ≥ 0 with 0^0 = 1.
__device__ __forceinline__ float decay_pow(float a, int64_t k) {
  return k == 0 ? 1.f : powf(a, (float)k);
}

// Status code of a failed device-side check of the LA_DEBUG build (the same
// value as LA_ERR_DEVICE_CHECK in the public header).
constexpr int kStatusDeviceCheck = 6;

// LA_DCHECK(status, cond, site) guards an index, offset or TMA coordinate the
// kernel is about to use.  In an LA_DEBUG build it evaluates cond; when cond
// is false it records kStatusDeviceCheck in status[0] and the site number in
// status[1] (the first failure wins, and a recorded timeout is kept) and
// yields false, so that the caller skips the access.  In the release build it
// is `true` and cond is not evaluated.  Sites are numbered per kernel file.
#ifdef LA_DEBUG
__device__ __noinline__ inline bool dcheck_failed(int* status, int site) {
  if (status && atomicCAS(status, 0, kStatusDeviceCheck) == 0) atomicExch(status + 1, site);
  return false;
}
#define LA_DCHECK(status, cond, site) ((cond) || ::la::dcheck_failed((status), (site)))
#else
#define LA_DCHECK(status, cond, site) true
#endif

}  // namespace la
