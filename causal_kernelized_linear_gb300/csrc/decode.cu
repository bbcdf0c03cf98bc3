// Recurrent decode step ("Efficient Transformers II" §2.2, eq (10)–(11) and
// the causal readout of eq (9)) for B·H independent heads.  elu+1 map (d' = d):
//   k' = φ(k), q' = φ(q);  μ ← a·μ + w·k'ᵀv;  ν ← a·ν + w·k';  o = q'μ / q'ν.
// The decay a is the head's (w = 1 − a, or 1 when a = 1), or this token's own
// a and weight w = b (default 1 − a) — eq (4) of the same page with a and b
// indexed by the token.
//
// The step is bound by HBM: every head streams its d×d fp32 μ in and out once
// (128 KiB of traffic at d = 128) against ~5·d² flops.  One CTA per head; each
// thread owns a float4 column group and a strided set of rows, so that a warp
// touches one contiguous 512-byte row segment per access (128-bit, coalesced).
// All μ loads of a thread are issued before any arithmetic to keep enough
// bytes in flight; loads and stores use the streaming (evict-first) hints
// because μ is touched once per step.  q'·μ is reduced over rows through
// shared memory and q'·ν with warp shuffles.
#include "common.cuh"
#include "internal.h"

namespace la {
namespace {

constexpr int kDecThreads = 256;

// Where a step's decay and new-token weight come from: per head (a [H], or
// none for a = 1) or, with TOKD, per token (a [B·H] and b [B·H] or none for
// b = 1 − a).  TOKD is a template parameter so that the per-head kernels
// carry no code of the per-token form.
struct StepDecay {
  const float* a;
  const float* b;
  int64_t H;
};

template <bool TOKD>
__device__ __forceinline__ void step_decay(const StepDecay& sd, int64_t bh, float& a, float& w) {
  if (TOKD) {
    a = sd.a[bh];
    w = sd.b ? sd.b[bh] : 1.f - a;
  } else {
    a = sd.a ? sd.a[bh % sd.H] : 1.f;
    w = new_token_weight(a);
  }
}

template <typename T>
__device__ __forceinline__ float load_elem(const T* p, int64_t i) { return to_f32(p[i]); }

template <typename T, int D, bool TOKD>
__global__ void __launch_bounds__(kDecThreads)
decode_step_kernel(float* __restrict__ mu, float* __restrict__ nu, const T* __restrict__ q,
                   const T* __restrict__ k, const T* __restrict__ v, T* __restrict__ out,
                   const StepDecay sd) {
  constexpr int CG = D / 4;                 // float4 column groups per row
  constexpr int RG = kDecThreads / CG;      // row groups
  constexpr int RPT = D / RG;               // rows per thread
  static_assert(RPT >= 1 && D % RG == 0, "decode layout");
  __shared__ float qf[D], kf[D], vv[D];
  __shared__ float4 part[RG][CG];
  __shared__ float red[kDecThreads / 32];

  const int64_t bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int cg = tid % CG;
  const int rg = tid / CG;
  float4* mrow = reinterpret_cast<float4*>(mu + bh * (int64_t)(D * D));

  // issue every μ load of this thread first (rows rg, rg+RG, ...)
  float4 m[RPT];
#pragma unroll
  for (int r = 0; r < RPT; ++r) m[r] = __ldcs(mrow + (int64_t)(rg + r * RG) * CG + cg);

  float a, w;
  step_decay<TOKD>(sd, bh, a, w);
  for (int i = tid; i < D; i += kDecThreads) {
    qf[i] = elu1(load_elem(q, bh * D + i));
    kf[i] = elu1(load_elem(k, bh * D + i));
    vv[i] = load_elem(v, bh * D + i);
  }
  __syncthreads();

  const float4 vc = make_float4(vv[4 * cg], vv[4 * cg + 1], vv[4 * cg + 2], vv[4 * cg + 3]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
    const int i = rg + r * RG;
    const float wk = w * kf[i];
    float4 x = m[r];
    x.x = a * x.x + wk * vc.x;
    x.y = a * x.y + wk * vc.y;
    x.z = a * x.z + wk * vc.z;
    x.w = a * x.w + wk * vc.w;
    __stcs(mrow + (int64_t)i * CG + cg, x);
    const float qi = qf[i];
    acc.x += qi * x.x;
    acc.y += qi * x.y;
    acc.z += qi * x.z;
    acc.w += qi * x.w;
  }
  part[rg][cg] = acc;

  // ν update and q'·ν (first D threads, then a block reduction)
  float dpart = 0.f;
  if (tid < D) {
    float* nb = nu + bh * D;
    const float x = a * nb[tid] + w * kf[tid];
    nb[tid] = x;
    dpart = qf[tid] * x;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dpart += __shfl_xor_sync(0xffffffffu, dpart, off);
  if ((tid & 31) == 0) red[tid >> 5] = dpart;
  __syncthreads();

  if (tid < D) {
    float den = 0.f;
#pragma unroll
    for (int wv = 0; wv < kDecThreads / 32; ++wv) den += red[wv];
    const int c = tid;
    float num = 0.f;
#pragma unroll 8
    for (int g = 0; g < RG; ++g) {
      const float4 pv = part[g][c / 4];
      num += (c % 4 == 0) ? pv.x : (c % 4 == 1) ? pv.y : (c % 4 == 2) ? pv.z : pv.w;
    }
    out[bh * D + c] = from_f32<T>(num / den);
  }
}

// The same step with the Performer map ("Linear Attention Research 2026",
// Performer random features): k' = φ(k), q' = φ(q) with
// φ(x)_f = exp(x·ω_f − ½‖x‖²)/√m, so the state μ is [m × d] and ν is [m].
// Thread f < m projects feature f (ω read through the read-only cache: every
// head of the launch reads the same [d × m] matrix, which stays in L1/L2);
// the state update then follows the elu+1 kernel with the m feature rows as
// the state rows.  All μ loads are issued before the projection so that
// their latency overlaps it.
template <typename T, int D, int M>
struct PerfDecodeCfg {
  static constexpr int NT = (D * M / 64 > 256) ? D * M / 64 : 256;   // ≤ 16 float4 rows per thread
  static constexpr int CG = D / 4;
  static constexpr int RG = NT / CG;
  static constexpr int RPT = M / RG;
  static_assert(RPT >= 1 && M % RG == 0 && RPT <= 16 && NT >= M, "Performer decode layout");
};

template <typename T, int D, int M, bool TOKD>
__global__ void __launch_bounds__((PerfDecodeCfg<T, D, M>::NT))
decode_performer_kernel(float* __restrict__ mu, float* __restrict__ nu, const T* __restrict__ q,
                        const T* __restrict__ k, const T* __restrict__ v, T* __restrict__ out,
                        const StepDecay sd, const T* __restrict__ omega) {
  using Cfg = PerfDecodeCfg<T, D, M>;
  constexpr int NT = Cfg::NT, CG = Cfg::CG, RG = Cfg::RG, RPT = Cfg::RPT;
  __shared__ float xq[D], xk[D], vv[D];
  __shared__ float phq[M], phk[M];
  __shared__ float4 part[RG][CG];
  __shared__ float red[NT / 32];
  __shared__ float half_sq[2];

  const int64_t bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int cg = tid % CG;
  const int rg = tid / CG;
  float4* mrow = reinterpret_cast<float4*>(mu + bh * (int64_t)(M * D));

  float4 m[RPT];
#pragma unroll
  for (int r = 0; r < RPT; ++r) m[r] = __ldcs(mrow + (int64_t)(rg + r * RG) * CG + cg);

  float a, w;
  step_decay<TOKD>(sd, bh, a, w);
  for (int i = tid; i < D; i += NT) {
    xq[i] = load_elem(q, bh * D + i);
    xk[i] = load_elem(k, bh * D + i);
    vv[i] = load_elem(v, bh * D + i);
  }
  __syncthreads();
  // ½‖q‖² (warp 0) and ½‖k‖² (warp 1)
  if (tid < 64) {
    const float* x = tid < 32 ? xq : xk;
    float s2 = 0.f;
    for (int c = tid & 31; c < D; c += 32) s2 += x[c] * x[c];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
    if ((tid & 31) == 0) half_sq[tid >> 5] = 0.5f * s2;
  }
  __syncthreads();
  if (tid < M) {
    float uq = 0.f, uk = 0.f;
#pragma unroll 8
    for (int c = 0; c < D; ++c) {
      const float wc = to_f32(__ldg(omega + c * M + tid));
      uq += xq[c] * wc;
      uk += xk[c] * wc;
    }
    const float log_sqrt_m = 0.5f * logf((float)M);
    phq[tid] = expf(uq - half_sq[0] - log_sqrt_m);
    phk[tid] = expf(uk - half_sq[1] - log_sqrt_m);
  }
  __syncthreads();

  const float4 vc = make_float4(vv[4 * cg], vv[4 * cg + 1], vv[4 * cg + 2], vv[4 * cg + 3]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
    const int i = rg + r * RG;
    const float wk = w * phk[i];
    float4 x = m[r];
    x.x = a * x.x + wk * vc.x;
    x.y = a * x.y + wk * vc.y;
    x.z = a * x.z + wk * vc.z;
    x.w = a * x.w + wk * vc.w;
    __stcs(mrow + (int64_t)i * CG + cg, x);
    const float qi = phq[i];
    acc.x += qi * x.x;
    acc.y += qi * x.y;
    acc.z += qi * x.z;
    acc.w += qi * x.w;
  }
  part[rg][cg] = acc;

  // ν update and q'·ν
  float dpart = 0.f;
  if (tid < M) {
    float* nb = nu + bh * M;
    const float x = a * nb[tid] + w * phk[tid];
    nb[tid] = x;
    dpart = phq[tid] * x;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dpart += __shfl_xor_sync(0xffffffffu, dpart, off);
  if ((tid & 31) == 0) red[tid >> 5] = dpart;
  __syncthreads();

  if (tid < D) {
    float den = 0.f;
#pragma unroll
    for (int wv = 0; wv < NT / 32; ++wv) den += red[wv];
    const int c = tid;
    float num = 0.f;
#pragma unroll 8
    for (int g = 0; g < RG; ++g) {
      const float4 pv = part[g][c / 4];
      num += (c % 4 == 0) ? pv.x : (c % 4 == 1) ? pv.y : (c % 4 == 2) ? pv.z : pv.w;
    }
    out[bh * D + c] = from_f32<T>(num / den);
  }
}

StepDecay step_decay_of(const DecodeArgs& a) {
  StepDecay sd;
  sd.a = a.decay;
  sd.b = a.weight;
  sd.H = a.H;
  return sd;
}

template <typename T, int D, int M>
cudaError_t launch_perf_decode(const DecodeArgs& a, cudaStream_t s) {
  using Cfg = PerfDecodeCfg<T, D, M>;
  auto kern = a.per_token ? decode_performer_kernel<T, D, M, true>
                          : decode_performer_kernel<T, D, M, false>;
  kern<<<(unsigned)(a.B * a.H), Cfg::NT, 0, s>>>(
      a.mu, a.nu, static_cast<const T*>(a.q), static_cast<const T*>(a.k),
      static_cast<const T*>(a.v), static_cast<T*>(a.out), step_decay_of(a),
      static_cast<const T*>(a.omega));
  count_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t run_perf_decode(const DecodeArgs& a, cudaStream_t s) {
#define LA_PD_CASE(DD, MM) \
  if (a.d == DD && a.m == MM) return launch_perf_decode<T, DD, MM>(a, s);
  LA_PD_CASE(32, 64) LA_PD_CASE(32, 128) LA_PD_CASE(32, 256)
  LA_PD_CASE(64, 64) LA_PD_CASE(64, 128) LA_PD_CASE(64, 256)
  LA_PD_CASE(128, 64) LA_PD_CASE(128, 128) LA_PD_CASE(128, 256)
#undef LA_PD_CASE
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t run_decode(const DecodeArgs& a, cudaStream_t s) {
  const unsigned grid = (unsigned)(a.B * a.H);
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  T* o = static_cast<T*>(a.out);
  switch (a.d) {
    case 32:
      (a.per_token ? decode_step_kernel<T, 32, true> : decode_step_kernel<T, 32, false>)
          <<<grid, kDecThreads, 0, s>>>(a.mu, a.nu, q, k, v, o, step_decay_of(a));
      break;
    case 64:
      (a.per_token ? decode_step_kernel<T, 64, true> : decode_step_kernel<T, 64, false>)
          <<<grid, kDecThreads, 0, s>>>(a.mu, a.nu, q, k, v, o, step_decay_of(a));
      break;
    case 128:
      (a.per_token ? decode_step_kernel<T, 128, true> : decode_step_kernel<T, 128, false>)
          <<<grid, kDecThreads, 0, s>>>(a.mu, a.nu, q, k, v, o, step_decay_of(a));
      break;
    default:
      return cudaErrorInvalidValue;
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t decode_step(const DecodeArgs& a, cudaStream_t stream) {
  if (a.performer) {
    if (a.bf16) return run_perf_decode<__nv_bfloat16>(a, stream);
    return run_perf_decode<float>(a, stream);
  }
  if (a.bf16) return run_decode<__nv_bfloat16>(a, stream);
  return run_decode<float>(a, stream);
}

}  // namespace la
