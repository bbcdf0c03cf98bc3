// fp32 CUDA-core chunked forward of causal / non-causal kernelized linear
// attention, and the decayed segment scan.
//
// Method ("Efficient Transformers II" §2.2, eq (6)–(11)): per head, with the
// state (μ, ν) at the start of a chunk of cs tokens (local positions t, s):
//   o_t = [ Σ_{s≤t} w·a^{t−s}(q'_t·k'_s) v_s + a^{t+1} q'_t μ ]
//       / [ Σ_{s≤t} w·a^{t−s}(q'_t·k'_s)     + a^{t+1} q'_t ν ]
//   μ ← a^{cs} μ + Σ_s w·a^{cs−1−s} k'_sᵀ v_s,   ν ← a^{cs} ν + Σ_s w·a^{cs−1−s} k'_sᵀ
// which is eq (10)–(11) unrolled over the chunk (eq (7)–(8) when a = 1, w = 1),
// with the causal readout of eq (9) that includes token t.  The intra-chunk part
// is the quadratic form of "Efficient Transformers I" eq (25)–(26) restricted to
// the chunk.  Everything is computed in fp32 on CUDA cores: this is the path
// for fp32 inputs, where the parity bound (1e-4) rules out bf16 tensor-core
// operands.
//
// Per-token decay (the same page's eq (4), z_i = a·z_{i−1} + b·s_i, with a and
// b indexed by the token): with L_t = Σ_{j≤t} log2 a_j over the chunk,
//   a^{t−s} → 2^{L_t − L_s},  a^{t+1} → 2^{L_t},  a^{cs} → 2^{L_{cs−1}},
// and the weight w of token s becomes b_s (1 − a_s unless given).  log2 a_j is
// clamped at −64, so a_j = 0 attenuates the past by 2^{−64} instead of
// erasing it.
//
// Long sequences are cut into segments (one CTA per (segment, head)).  Pass 1
// computes each segment's own decayed aggregate, segment_scan turns them into
// exclusive prefixes (the state entering each segment), pass 2 produces the
// outputs.  Non-causal mode: pass 1 + scan give μ_n, ν_n, then a readout pass.
#include "common.cuh"
#include "internal.h"
#include "simt.cuh"

#include <algorithm>

namespace la {
namespace {

using simt::kThreads;
using simt::load_features;
using simt::load_values;

template <int D, int DP, bool PERF>
struct SimtCfg {
  // tokens per chunk: 32 unless the fp32 state plus chunk buffers would not fit
  static constexpr int CS = (DP * D >= 256 * 128) ? 16 : 32;
  static constexpr int FS = DP + 1;  // padded row stride of feature tiles
  // shared-memory layout (floats)
  static constexpr int oS = 0;                      // μ  [DP][D]
  static constexpr int oZ = oS + DP * D;            // ν  [DP]
  static constexpr int oQF = oZ + DP;               // q' [CS][FS]
  static constexpr int oKF = oQF + CS * FS;         // k' [CS][FS]
  static constexpr int oV = oKF + CS * FS;          // v  [CS][D]
  static constexpr int oX = oV + CS * D;            // raw rows for Performer [CS][D]
  static constexpr int oP = oX + (PERF ? CS * D : 0);  // masked weights [CS][CS]
  static constexpr int oPW = oP + CS * CS;          // a^k, k = 0..CS
  static constexpr int oSQ = oPW + CS + 1;          // ½‖x‖² per row (Performer)
  static constexpr int oDEN = oSQ + CS;             // denominators [CS]
  static constexpr int oLC = oDEN + CS;             // per-token decay: L_t [CS]
  static constexpr int oBW = oLC + CS;              // per-token decay: b_t [CS]
  static constexpr int total = oBW + CS;
  static constexpr size_t bytes = size_t(total) * sizeof(float);
};

// μ ← a^{cs} μ + Σ_s w·a^{cs−1−s} k'_sᵀ v_s ; ν likewise (eq (10)–(11) over a chunk).
template <int D, int DP, int CS, int FS>
__device__ void update_state(float* S, float* z, const float* kf, const float* vv,
                             const float* pw, float w, int cs) {
  const float acs = pw[cs];
  for (int e = threadIdx.x; e < DP * D; e += kThreads) {
    const int i = e / D, c = e % D;
    float acc = 0.f;
    for (int s = 0; s < cs; ++s) acc += (w * pw[cs - 1 - s]) * kf[s * FS + i] * vv[s * D + c];
    S[e] = acs * S[e] + acc;
  }
  for (int i = threadIdx.x; i < DP; i += kThreads) {
    float acc = 0.f;
    for (int s = 0; s < cs; ++s) acc += (w * pw[cs - 1 - s]) * kf[s * FS + i];
    z[i] = acs * z[i] + acc;
  }
}

// Per-token decay of one chunk, computed by warp 0: Lc[t] = Σ_{j≤t} log2 a_j
// (within the chunk, log2 clamped at −64; tokens t ≥ cs add 0, so Lc[CS−1]
// is the chunk's total) and Bw[t] = b_t (0 for t ≥ cs).
template <int CS>
__device__ void tok_chunk_prep(const float* __restrict__ a, const float* __restrict__ b, int cs,
                               float* Lc, float* Bw) {
  static_assert(CS <= 32, "one warp per chunk");
  if (threadIdx.x >= 32) return;
  const int t = threadIdx.x;
  const bool live = t < cs;
  const float at = live ? a[t] : 1.f;
  float lg = live ? fmaxf(log2f(at), -64.f) : 0.f;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float u = __shfl_up_sync(0xffffffffu, lg, o);
    if (t >= o) lg += u;
  }
  if (t < CS) {
    Lc[t] = lg;
    Bw[t] = live ? (b ? b[t] : 1.f - at) : 0.f;
  }
}

// Per-token form of update_state: μ ← 2^{L_{cs−1}} μ + Σ_s b_s·2^{L_{cs−1}−L_s} k'_sᵀ v_s.
template <int D, int DP, int CS, int FS>
__device__ void update_state_tok(float* S, float* z, const float* kf, const float* vv,
                                 const float* Lc, const float* Bw, int cs) {
  const float ltot = Lc[CS - 1];
  const float acs = exp2f(ltot);
  for (int e = threadIdx.x; e < DP * D; e += kThreads) {
    const int i = e / D, c = e % D;
    float acc = 0.f;
    for (int s = 0; s < cs; ++s) acc += (Bw[s] * exp2f(ltot - Lc[s])) * kf[s * FS + i] * vv[s * D + c];
    S[e] = acs * S[e] + acc;
  }
  for (int i = threadIdx.x; i < DP; i += kThreads) {
    float acc = 0.f;
    for (int s = 0; s < cs; ++s) acc += (Bw[s] * exp2f(ltot - Lc[s])) * kf[s * FS + i];
    z[i] = acs * z[i] + acc;
  }
}

struct SimtParams {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  const float* decay;
  const float* tok_decay;   // [BH][n] or nullptr
  const float* tok_weight;  // [BH][n] or nullptr
  float* ws_ld;             // [BH][nseg] log2 decay of each segment (per-token decay)
  const void* omega;
  int64_t H, n, seg_len;
  int nseg;
  float* ws_state;   // [BH][nseg][DP*D]
  float* ws_z;       // [BH][nseg][DP]
  const float* init_state;   // causal: state entering token 0 [BH][DP*D], or nullptr
  const float* init_z;       // [BH][DP]
  const float* tot_state;  // non-causal: [BH][DP*D]
  const float* tot_z;
  float* fin_state;  // causal single-segment: final state out (or nullptr)
  float* fin_z;
};

// Pass 1: the decayed aggregate of one segment, starting from zero state
// (and, with a per-token decay, the segment's total log2 decay).
template <typename T, int D, int DP, bool PERF, bool TOK>
__global__ void __launch_bounds__(kThreads)
simt_segment_state(SimtParams p) {
  using C = SimtCfg<D, DP, PERF>;
  constexpr int CS = C::CS, FS = C::FS;
  extern __shared__ float sm[];
  float* S = sm + C::oS;
  float* z = sm + C::oZ;
  float* kf = sm + C::oKF;
  float* vv = sm + C::oV;
  float* xr = sm + C::oX;
  float* pw = sm + C::oPW;
  float* hs = sm + C::oSQ;
  float* Lc = sm + C::oLC;
  float* Bw = sm + C::oBW;
  const int g = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int64_t t_begin = (int64_t)g * p.seg_len;
  const int64_t t_end = min(p.n, t_begin + p.seg_len);
  const float a = p.decay ? p.decay[bh % p.H] : 1.f;
  const float w = new_token_weight(a);
  for (int e = threadIdx.x; e < DP * D; e += kThreads) S[e] = 0.f;
  for (int i = threadIdx.x; i < DP; i += kThreads) z[i] = 0.f;
  for (int kk = threadIdx.x; kk <= CS; kk += kThreads) pw[kk] = decay_pow(a, kk);
  const T* kb = static_cast<const T*>(p.k) + bh * p.n * D;
  const T* vb = static_cast<const T*>(p.v) + bh * p.n * D;
  const T* om = static_cast<const T*>(p.omega);
  const float* ab = TOK ? p.tok_decay + bh * p.n : nullptr;
  const float* bb = (TOK && p.tok_weight) ? p.tok_weight + bh * p.n : nullptr;
  float seg_ld = 0.f;
  for (int64_t t0 = t_begin; t0 < t_end; t0 += CS) {
    const int cs = (int)min((int64_t)CS, t_end - t0);
    __syncthreads();
    load_features<T, D, DP, PERF, CS, FS>(kb + t0 * D, cs, kf, xr, hs, om);
    load_values<T, D, CS>(vb + t0 * D, cs, vv);
    if (TOK) tok_chunk_prep<CS>(ab + t0, bb ? bb + t0 : nullptr, cs, Lc, Bw);
    __syncthreads();
    if (TOK) {
      seg_ld += Lc[CS - 1];
      update_state_tok<D, DP, CS, FS>(S, z, kf, vv, Lc, Bw, cs);
    } else {
      update_state<D, DP, CS, FS>(S, z, kf, vv, pw, w, cs);
    }
  }
  __syncthreads();
  float* dS = p.ws_state + (bh * p.nseg + g) * (int64_t)(DP * D);
  float* dz = p.ws_z + (bh * p.nseg + g) * (int64_t)DP;
  for (int e = threadIdx.x; e < DP * D; e += kThreads) dS[e] = S[e];
  for (int i = threadIdx.x; i < DP; i += kThreads) dz[i] = z[i];
  if (TOK && threadIdx.x == 0) p.ws_ld[bh * p.nseg + g] = seg_ld;
}

// Pass 2 (causal): outputs of one segment from the state entering it.
template <typename T, int D, int DP, bool PERF, bool TOK>
__global__ void __launch_bounds__(kThreads)
simt_causal_output(SimtParams p) {
  using C = SimtCfg<D, DP, PERF>;
  constexpr int CS = C::CS, FS = C::FS;
  extern __shared__ float sm[];
  float* S = sm + C::oS;
  float* z = sm + C::oZ;
  float* qf = sm + C::oQF;
  float* kf = sm + C::oKF;
  float* vv = sm + C::oV;
  float* xr = sm + C::oX;
  float* P = sm + C::oP;
  float* pw = sm + C::oPW;
  float* hs = sm + C::oSQ;
  float* den = sm + C::oDEN;
  float* Lc = sm + C::oLC;
  float* Bw = sm + C::oBW;
  const int g = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int64_t t_begin = (int64_t)g * p.seg_len;
  const int64_t t_end = min(p.n, t_begin + p.seg_len);
  const float a = p.decay ? p.decay[bh % p.H] : 1.f;
  const float w = new_token_weight(a);
  // the state entering the segment: its exclusive prefix from the scan
  // (which starts from the initial state), or the initial state itself
  const float* sS = nullptr;
  const float* sz = nullptr;
  if (p.nseg > 1) {
    sS = p.ws_state + (bh * p.nseg + g) * (int64_t)(DP * D);
    sz = p.ws_z + (bh * p.nseg + g) * (int64_t)DP;
  } else if (p.init_state) {
    sS = p.init_state + bh * (int64_t)(DP * D);
    sz = p.init_z + bh * (int64_t)DP;
  }
  if (sS) {
    for (int e = threadIdx.x; e < DP * D; e += kThreads) S[e] = sS[e];
    for (int i = threadIdx.x; i < DP; i += kThreads) z[i] = sz[i];
  } else {
    for (int e = threadIdx.x; e < DP * D; e += kThreads) S[e] = 0.f;
    for (int i = threadIdx.x; i < DP; i += kThreads) z[i] = 0.f;
  }
  for (int kk = threadIdx.x; kk <= CS; kk += kThreads) pw[kk] = decay_pow(a, kk);
  const T* qb = static_cast<const T*>(p.q) + bh * p.n * D;
  const T* kb = static_cast<const T*>(p.k) + bh * p.n * D;
  const T* vb = static_cast<const T*>(p.v) + bh * p.n * D;
  T* ob = static_cast<T*>(p.out) + bh * p.n * D;
  const T* om = static_cast<const T*>(p.omega);
  const float* ab = TOK ? p.tok_decay + bh * p.n : nullptr;
  const float* bb = (TOK && p.tok_weight) ? p.tok_weight + bh * p.n : nullptr;
  for (int64_t t0 = t_begin; t0 < t_end; t0 += CS) {
    const int cs = (int)min((int64_t)CS, t_end - t0);
    __syncthreads();
    load_features<T, D, DP, PERF, CS, FS>(kb + t0 * D, cs, kf, xr, hs, om);
    __syncthreads();
    load_features<T, D, DP, PERF, CS, FS>(qb + t0 * D, cs, qf, xr, hs, om);
    load_values<T, D, CS>(vb + t0 * D, cs, vv);
    if (TOK) tok_chunk_prep<CS>(ab + t0, bb ? bb + t0 : nullptr, cs, Lc, Bw);
    __syncthreads();
    // masked, decayed weights P[t][s] = w·a^{t−s}(q'_t·k'_s), s ≤ t
    // (per-token decay: b_s·2^{L_t − L_s}(q'_t·k'_s))
    for (int e = threadIdx.x; e < CS * CS; e += kThreads) {
      const int t = e / CS, s = e % CS;
      float acc = 0.f;
      if (s <= t) {
        for (int i = 0; i < DP; ++i) acc += qf[t * FS + i] * kf[s * FS + i];
        acc *= TOK ? Bw[s] * exp2f(Lc[t] - Lc[s]) : w * pw[t - s];
      }
      P[e] = acc;
    }
    __syncthreads();
    // decay of the entering state at token t: a^{t+1} (per-token: 2^{L_t})
    for (int t = threadIdx.x; t < CS; t += kThreads) {
      float intra = 0.f, inter = 0.f;
      for (int s = 0; s <= t; ++s) intra += P[t * CS + s];
      for (int i = 0; i < DP; ++i) inter += qf[t * FS + i] * z[i];
      den[t] = intra + (TOK ? exp2f(Lc[t]) : pw[t + 1]) * inter;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < CS * D; e += kThreads) {
      const int t = e / D, c = e % D;
      if (t < cs) {
        float intra = 0.f, inter = 0.f;
        for (int s = 0; s <= t; ++s) intra += P[t * CS + s] * vv[s * D + c];
        for (int i = 0; i < DP; ++i) inter += qf[t * FS + i] * S[i * D + c];
        const float num = intra + (TOK ? exp2f(Lc[t]) : pw[t + 1]) * inter;
        ob[(t0 + t) * D + c] = from_f32<T>(num / den[t]);
      }
    }
    __syncthreads();
    if (TOK) update_state_tok<D, DP, CS, FS>(S, z, kf, vv, Lc, Bw, cs);
    else update_state<D, DP, CS, FS>(S, z, kf, vv, pw, w, cs);
  }
  if (p.fin_state) {
    __syncthreads();
    for (int e = threadIdx.x; e < DP * D; e += kThreads) p.fin_state[bh * (DP * D) + e] = S[e];
    for (int i = threadIdx.x; i < DP; i += kThreads) p.fin_z[bh * DP + i] = z[i];
  }
}

// Non-causal readout: o_j = q'_j μ_n / q'_j ν_n (eq (6) / eq (9)).
template <typename T, int D, int DP, bool PERF>
__global__ void __launch_bounds__(kThreads)
simt_noncausal_readout(SimtParams p) {
  using C = SimtCfg<D, DP, PERF>;
  constexpr int CS = C::CS, FS = C::FS;
  extern __shared__ float sm[];
  float* S = sm + C::oS;
  float* z = sm + C::oZ;
  float* qf = sm + C::oQF;
  float* xr = sm + C::oX;
  float* hs = sm + C::oSQ;
  float* den = sm + C::oDEN;
  const int g = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int64_t t_begin = (int64_t)g * p.seg_len;
  const int64_t t_end = min(p.n, t_begin + p.seg_len);
  for (int e = threadIdx.x; e < DP * D; e += kThreads) S[e] = p.tot_state[bh * (DP * D) + e];
  for (int i = threadIdx.x; i < DP; i += kThreads) z[i] = p.tot_z[bh * DP + i];
  const T* qb = static_cast<const T*>(p.q) + bh * p.n * D;
  T* ob = static_cast<T*>(p.out) + bh * p.n * D;
  const T* om = static_cast<const T*>(p.omega);
  for (int64_t t0 = t_begin; t0 < t_end; t0 += CS) {
    const int cs = (int)min((int64_t)CS, t_end - t0);
    __syncthreads();
    load_features<T, D, DP, PERF, CS, FS>(qb + t0 * D, cs, qf, xr, hs, om);
    __syncthreads();
    for (int t = threadIdx.x; t < CS; t += kThreads) {
      float acc = 0.f;
      for (int i = 0; i < DP; ++i) acc += qf[t * FS + i] * z[i];
      den[t] = acc;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < CS * D; e += kThreads) {
      const int t = e / D, c = e % D;
      if (t < cs) {
        float acc = 0.f;
        for (int i = 0; i < DP; ++i) acc += qf[t * FS + i] * S[i * D + c];
        ob[(t0 + t) * D + c] = from_f32<T>(acc / den[t]);
      }
    }
  }
}

__global__ void __launch_bounds__(256)
segment_scan_kernel(float* ws_state, float* ws_z, float* tot_state, float* tot_z, int64_t H,
                    int nseg, int nagg, int64_t seg_len, int64_t n, int dpd, int dp,
                    const float* decay, const float* seg_ld, const float* init_state,
                    const float* init_z) {
  constexpr int kBatch = 8;  // aggregates loaded together to keep loads in flight
  // launched as a programmatic dependent of the launch that wrote the
  // aggregates (tensor-core paths): let the next launch start, then wait for
  // the aggregates (both are no-ops in an ordinary launch)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t bh = blockIdx.x;
  const int e = blockIdx.y * 256 + threadIdx.x;
  if (e >= dpd + dp) return;
  const float a = decay ? decay[bh % H] : 1.f;
  const float a_full = decay_pow(a, seg_len);  // every segment but the last is full
  float* base;
  int64_t stride;
  if (e < dpd) {
    base = ws_state + bh * nseg * (int64_t)dpd + e;
    stride = dpd;
  } else {
    base = ws_z + bh * nseg * (int64_t)dp + (e - dpd);
    stride = dp;
  }
  float acc = 0.f;  // state entering segment g
  if (init_state) acc = e < dpd ? init_state[bh * dpd + e] : init_z[bh * dp + (e - dpd)];
  for (int g0 = 0; g0 < nseg; g0 += kBatch) {
    float agg[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) agg[j] = (g0 + j < nagg) ? base[(g0 + j) * stride] : 0.f;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int g = g0 + j;
      if (g < nseg) {
        base[g * stride] = acc;
        const int64_t len = min(seg_len, n - (int64_t)g * seg_len);
        // per-token decay: the segment's own total, written with its aggregate
        const float fac = seg_ld ? (g < nagg ? exp2f(seg_ld[bh * nseg + g]) : 0.f)
                                 : (len == seg_len ? a_full : decay_pow(a, len));
        acc = fac * acc + agg[j];
      }
    }
  }
  if (tot_state && nagg == nseg) {
    if (e < dpd) tot_state[bh * dpd + e] = acc;
    else tot_z[bh * dp + (e - dpd)] = acc;
  }
}

// segment_scan_kernel with four consecutive state elements per thread
// (float4 loads and stores; dp a multiple of 4 and every pointer 16-byte
// aligned).
__global__ void __launch_bounds__(256)
segment_scan4_kernel(float* ws_state, float* ws_z, float* tot_state, float* tot_z, int64_t H,
                     int nseg, int nagg, int64_t seg_len, int64_t n, int dpd, int dp,
                     const float* decay, const float* seg_ld, const float* init_state,
                     const float* init_z) {
  constexpr int kBatch = 8;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t bh = blockIdx.x;
  const int e4 = (blockIdx.y * 256 + threadIdx.x) * 4;
  if (e4 >= dpd + dp) return;
  const bool mat = e4 < dpd;
  float* base = mat ? ws_state + bh * nseg * (int64_t)dpd + e4 : ws_z + bh * nseg * (int64_t)dp + (e4 - dpd);
  const int64_t stride = mat ? dpd : dp;
  const float a = decay ? decay[bh % H] : 1.f;
  const float a_full = decay_pow(a, seg_len);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);   // state entering segment g
  if (init_state)
    acc = mat ? *reinterpret_cast<const float4*>(init_state + bh * dpd + e4)
              : *reinterpret_cast<const float4*>(init_z + bh * dp + (e4 - dpd));
  for (int g0 = 0; g0 < nseg; g0 += kBatch) {
    float4 agg[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      agg[j] = (g0 + j < nagg) ? *reinterpret_cast<const float4*>(base + (g0 + j) * stride)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int g = g0 + j;
      if (g < nseg) {
        *reinterpret_cast<float4*>(base + g * stride) = acc;
        const int64_t len = min(seg_len, n - (int64_t)g * seg_len);
        const float fac = seg_ld ? (g < nagg ? exp2f(seg_ld[bh * nseg + g]) : 0.f)
                                 : (len == seg_len ? a_full : decay_pow(a, len));
        acc = make_float4(fac * acc.x + agg[j].x, fac * acc.y + agg[j].y, fac * acc.z + agg[j].z,
                          fac * acc.w + agg[j].w);
      }
    }
  }
  if (tot_state && nagg == nseg) {
    if (mat) *reinterpret_cast<float4*>(tot_state + bh * dpd + e4) = acc;
    else *reinterpret_cast<float4*>(tot_z + bh * dp + (e4 - dpd)) = acc;
  }
}

// The total of every head's segment aggregates alone (no exclusive prefixes):
// acc ← init, then acc ← fac_g·acc + A_g over the segments g, four
// consecutive state elements per thread, all of a head's aggregates loaded
// together (up to 16 in flight per thread).
__global__ void __launch_bounds__(256)
segment_total_kernel(const float* __restrict__ ws_state, const float* __restrict__ ws_z,
                     float* __restrict__ tot_state, float* __restrict__ tot_z, int64_t H, int nseg,
                     int64_t seg_len, int64_t n, int dpd, int dp, const float* decay,
                     const float* seg_ld, const float* init_state, const float* init_z) {
  constexpr int kBatch = 16;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t bh = blockIdx.x;
  const int e4 = (blockIdx.y * 256 + threadIdx.x) * 4;
  if (e4 >= dpd + dp) return;
  const bool mat = e4 < dpd;   // dpd is a multiple of 4: no float4 straddles the two parts
  const float* base = mat ? ws_state + bh * nseg * (int64_t)dpd + e4
                          : ws_z + bh * nseg * (int64_t)dp + (e4 - dpd);
  const int64_t stride = mat ? dpd : dp;
  const float a = decay ? decay[bh % H] : 1.f;
  const float a_full = decay_pow(a, seg_len);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (init_state)
    acc = mat ? *reinterpret_cast<const float4*>(init_state + bh * dpd + e4)
              : *reinterpret_cast<const float4*>(init_z + bh * dp + (e4 - dpd));
  for (int g0 = 0; g0 < nseg; g0 += kBatch) {
    float4 agg[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      agg[j] = g0 + j < nseg ? *reinterpret_cast<const float4*>(base + (g0 + j) * stride)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int g = g0 + j;
      if (g < nseg) {
        const int64_t len = min(seg_len, n - (int64_t)g * seg_len);
        const float fac = seg_ld ? exp2f(seg_ld[bh * nseg + g])
                                 : (len == seg_len ? a_full : decay_pow(a, len));
        acc = make_float4(fac * acc.x + agg[j].x, fac * acc.y + agg[j].y, fac * acc.z + agg[j].z,
                          fac * acc.w + agg[j].w);
      }
    }
  }
  if (mat) *reinterpret_cast<float4*>(tot_state + bh * dpd + e4) = acc;
  else *reinterpret_cast<float4*>(tot_z + bh * dp + (e4 - dpd)) = acc;
}

template <typename T, int D, int DP, bool PERF, bool TOK>
cudaError_t run_simt_impl(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                          float* tot_state, float* tot_z, const SegmentPlan& plan) {
  using C = SimtCfg<D, DP, PERF>;
  static_assert(C::bytes <= 227 * 1024, "SIMT chunk buffers exceed shared memory");
  const size_t smem = C::bytes;
  cudaError_t err;
  err = cudaFuncSetAttribute(simt_segment_state<T, D, DP, PERF, TOK>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(simt_causal_output<T, D, DP, PERF, TOK>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  if (!TOK) {
    err = cudaFuncSetAttribute(simt_noncausal_readout<T, D, DP, PERF>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }

  SimtParams p{};
  p.q = a.q;
  p.k = a.k;
  p.v = a.v;
  p.out = a.out;
  p.decay = a.decay;
  p.tok_decay = a.tok_decay;
  p.tok_weight = a.tok_weight;
  p.ws_ld = a.ws_ld;
  p.omega = a.omega;
  p.H = a.H;
  p.n = a.n;
  p.seg_len = plan.seg_len;
  p.nseg = plan.nseg;
  p.ws_state = ws_state;
  p.ws_z = ws_z;
  p.init_state = a.init_state;
  p.init_z = a.init_z;
  const int64_t BH = a.B * a.H;
  const dim3 grid((unsigned)plan.nseg, (unsigned)BH);
  const bool need_scan = !a.causal || plan.nseg > 1;
  if (need_scan) {
    simt_segment_state<T, D, DP, PERF, TOK><<<grid, kThreads, smem, stream>>>(p);
    count_launches(1);
    err = segment_scan(ws_state, ws_z, tot_state, tot_z, BH, a.H, plan.nseg, plan.nseg,
                       plan.seg_len, a.n, DP, D, a.decay, TOK ? a.ws_ld : nullptr, stream, false,
                       a.causal ? a.init_state : nullptr, a.causal ? a.init_z : nullptr);
    if (err != cudaSuccess) return err;
  }
  if (a.causal) {
    if (plan.nseg == 1) {
      p.fin_state = a.mu_out;
      p.fin_z = a.nu_out;
    }
    simt_causal_output<T, D, DP, PERF, TOK><<<grid, kThreads, smem, stream>>>(p);
    count_launches(1);
  } else if (!TOK) {
    p.tot_state = tot_state;
    p.tot_z = tot_z;
    simt_noncausal_readout<T, D, DP, PERF><<<grid, kThreads, smem, stream>>>(p);
    count_launches(1);
  } else {
    return cudaErrorInvalidValue;   // the per-token decay is causal only
  }
  return cudaGetLastError();
}

template <typename T, int D, int DP, bool PERF>
cudaError_t run_simt(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                     float* tot_state, float* tot_z, const SegmentPlan& plan) {
  if (a.tok_decay)
    return run_simt_impl<T, D, DP, PERF, true>(a, stream, ws_state, ws_z, tot_state, tot_z, plan);
  return run_simt_impl<T, D, DP, PERF, false>(a, stream, ws_state, ws_z, tot_state, tot_z, plan);
}

template <typename T>
cudaError_t dispatch_simt(const FwdArgs& a, cudaStream_t s, float* ws, float* wz, float* ts,
                          float* tz, const SegmentPlan& pl) {
  if (!a.performer) {
    switch (a.d) {
      case 32: return run_simt<T, 32, 32, false>(a, s, ws, wz, ts, tz, pl);
      case 64: return run_simt<T, 64, 64, false>(a, s, ws, wz, ts, tz, pl);
      case 128: return run_simt<T, 128, 128, false>(a, s, ws, wz, ts, tz, pl);
    }
    return cudaErrorInvalidValue;
  }
#define LA_PERF_CASE(DD, MM) \
  if (a.d == DD && a.m == MM) return run_simt<T, DD, MM, true>(a, s, ws, wz, ts, tz, pl);
  LA_PERF_CASE(32, 64) LA_PERF_CASE(32, 128) LA_PERF_CASE(32, 256)
  LA_PERF_CASE(64, 64) LA_PERF_CASE(64, 128) LA_PERF_CASE(64, 256)
  LA_PERF_CASE(128, 64) LA_PERF_CASE(128, 128) LA_PERF_CASE(128, 256)
#undef LA_PERF_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t segment_total(float* ws_state, float* ws_z, float* tot_state, float* tot_z,
                          int64_t BH, int64_t H, int nseg, int64_t seg_len, int64_t n, int dp, int d,
                          const float* decay, const float* seg_ld, cudaStream_t stream,
                          bool dependent, const float* init_state, const float* init_z) {
  const int dpd = dp * d;
  auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  if (dp % 4 || !a16(ws_state) || !a16(ws_z) || !a16(tot_state) || !a16(tot_z) ||
      (init_state && (!a16(init_state) || !a16(init_z))))
    return segment_scan(ws_state, ws_z, tot_state, tot_z, BH, H, nseg, nseg, seg_len, n, dp, d,
                        decay, seg_ld, stream, dependent, init_state, init_z);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)BH, (unsigned)(((dpd + dp) / 4 + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, segment_total_kernel, (const float*)ws_state,
                                     (const float*)ws_z, tot_state, tot_z, H, nseg, seg_len, n, dpd,
                                     dp, decay, seg_ld, init_state, init_z);
  count_launches(1);
  return e;
}

cudaError_t segment_scan(float* ws_state, float* ws_z, float* tot_state, float* tot_z,
                         int64_t BH, int64_t H, int nseg, int nagg, int64_t seg_len, int64_t n,
                         int dp, int d, const float* decay, const float* seg_ld,
                         cudaStream_t stream, bool dependent, const float* init_state,
                         const float* init_z) {
  const int dpd = dp * d;
  auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  const bool vec = dp % 4 == 0 && a16(ws_state) && a16(ws_z) && a16(tot_state) && a16(tot_z) &&
                   a16(init_state) && a16(init_z);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)BH, (unsigned)(((vec ? (dpd + dp) / 4 : dpd + dp) + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, vec ? segment_scan4_kernel : segment_scan_kernel,
                                     ws_state, ws_z, tot_state, tot_z, H, nseg, nagg, seg_len, n,
                                     dpd, dp, decay, seg_ld, init_state, init_z);
  count_launches(1);
  return e;
}

namespace {

template <typename T, int D, int DP, bool PERF>
cudaError_t run_simt_state(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                           const SegmentPlan& plan) {
  using C = SimtCfg<D, DP, PERF>;
  const size_t smem = C::bytes;
  cudaError_t err = cudaFuncSetAttribute(simt_segment_state<T, D, DP, PERF, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  SimtParams p{};
  p.k = a.k;
  p.v = a.v;
  p.decay = a.decay;
  p.omega = a.omega;
  p.H = a.H;
  p.n = a.n;
  p.seg_len = plan.seg_len;
  p.nseg = plan.nseg;
  p.ws_state = ws_state;
  p.ws_z = ws_z;
  const dim3 grid((unsigned)plan.nseg, (unsigned)(a.B * a.H));
  simt_segment_state<T, D, DP, PERF, false><<<grid, kThreads, smem, stream>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_simt_state(const FwdArgs& a, cudaStream_t s, float* ws, float* wz,
                                const SegmentPlan& pl) {
  if (!a.performer) {
    switch (a.d) {
      case 32: return run_simt_state<T, 32, 32, false>(a, s, ws, wz, pl);
      case 64: return run_simt_state<T, 64, 64, false>(a, s, ws, wz, pl);
      case 128: return run_simt_state<T, 128, 128, false>(a, s, ws, wz, pl);
    }
    return cudaErrorInvalidValue;
  }
#define LA_PERF_CASE(DD, MM) \
  if (a.d == DD && a.m == MM) return run_simt_state<T, DD, MM, true>(a, s, ws, wz, pl);
  LA_PERF_CASE(32, 64) LA_PERF_CASE(32, 128) LA_PERF_CASE(32, 256)
  LA_PERF_CASE(64, 64) LA_PERF_CASE(64, 128) LA_PERF_CASE(64, 256)
  LA_PERF_CASE(128, 64) LA_PERF_CASE(128, 128) LA_PERF_CASE(128, 256)
#undef LA_PERF_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t simt_state_only(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                            const SegmentPlan& plan) {
  if (a.bf16) return dispatch_simt_state<__nv_bfloat16>(a, stream, ws_state, ws_z, plan);
  return dispatch_simt_state<float>(a, stream, ws_state, ws_z, plan);
}

cudaError_t simt_forward(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                         float* tot_state, float* tot_z, const SegmentPlan& plan) {
  if (a.bf16) return dispatch_simt<__nv_bfloat16>(a, stream, ws_state, ws_z, tot_state, tot_z, plan);
  return dispatch_simt<float>(a, stream, ws_state, ws_z, tot_state, tot_z, plan);
}

}  // namespace la
