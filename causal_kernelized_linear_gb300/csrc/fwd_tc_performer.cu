// Tensor-core (tcgen05 + TMA + TMEM) chunked forward of kernelized linear
// attention with the Performer positive random feature map, bf16 inputs,
// fp32 state, d = 64, m ∈ {128, 256} features, no decay (a = 1).
//
// Method ("Linear Attention Research 2026", Performer random features:
// φ(x) = exp(xω − ½‖x‖²)/√m; "Efficient Transformers II" §2.2 eq (6)–(9):
// the running sums μ, ν, the causal readout o_j = q'_j·μ_j / q'_j·ν_j and the
// non-causal D⁻¹(Q'(K'ᵀV)) of eq (6)).  Per head and 128-token chunk
// (local t, s; cs valid rows) with state (S, z) at the chunk start:
//   U = X·ω (the projection, on the tensor core, X = the raw q or k rows)
//   φ(x)_i = 2^(u_i·log2 e − ½‖x‖²·log2 e − ½·log2 m)       (fp32 exponent)
//   causal:     P_ts = q'_t·k'_s for s ≤ t, else 0
//               num_t = Σ_s P_ts v_s + q'_t·S,   den_t = Σ_s P_ts + q'_t·z
//   non-causal: num_t = q'_t·S_n,   den_t = q'_t·z_n   (S_n, z_n: the sums
//               over the whole sequence, eq (6) regrouped as eq (9))
//   S ← S + Σ_s k'_sᵀ v_s,   z ← z + Σ_s k'_s
//
// Launch modes (one CTA per (head, segment), 16 warps):
//   state    the aggregate (S, z) of one segment, from zero
//   causal   o over one segment, starting from the sum of the aggregates of
//            the segments before it (the last segment also writes the final
//            state)
//   readout  o = q'·S_n / q'·z_n over one segment, S_n the sum of all the
//            aggregates
// Between the state launch and the other one, segment_scan turns the
// aggregates into those sums (exclusive prefixes, and the total, which is
// also the non-causal final state).  The scan and the launch after it are
// programmatic dependents: they start while the launch before drains, and
// only the reads of its results wait for it.
//
// Roles:
//   warp 0       TMA producer (ω once; raw q and k tiles one stage each, v two)
//   warps 1–3    tcgen05 MMA issuers: output products (warp 1, TMEM owner),
//                state products (warp 2), projections (warp 3)
//   warps 4–7    initial state; state operand tile per chunk; masked P;
//                epilogue o = num/den stored row by row; final state
//   warps 8–15   φ: each 64-feature projection block of U comes through one
//                of two TMEM buffers; warps 8–11 take its first 32 features,
//                warps 12–15 the other 32; φ(K) goes to shared memory (the
//                operand of the scores and state products), φ(Q) to TMEM
// tcgen05 products: U = X·ω (M 128, N 64, K 64), scores = φ(Q)·φ(K)ᵀ
// (K = m), ΔS = φ(K)ᵀV and Δz = φ(K)ᵀ1 per 128-feature block, num = φ(Q)·S,
// den = φ(Q)·z, num += P·V, den += P·1.  Every wait is bounded in time and
// reports LA_ERR_TIMEOUT through the device status word.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace la {
namespace {

using namespace tc;

constexpr int kC = 128;        // tokens per chunk
constexpr int kD = 64;         // input and value width
constexpr int kThreads = 512;
constexpr float kLog2e = 1.4426950408889634f;

enum Mode { kState = 0, kCausal = 1, kReadout = 2 };

template <int DP>
struct PCfg {
  static constexpr int NB = DP / 64;             // 64-feature blocks
  static constexpr int NP = DP / 128;            // 128-feature projection steps per operand
  static constexpr int MB = DP / 128;            // 128-feature blocks (state lane blocks)
  static constexpr int TILE = kC * kD * 2;       // [128 × 64] bf16 = 16 KB
  static constexpr int WATOM = 64 * 128;         // ω block [64 (d) × 64 (features)] = 8 KB
  // shared memory (offsets from a 1024-aligned base)
  static constexpr int oW = 0;                   // ω, NB blocks
  // raw q and k, one stage each: only the projection and the row norms read
  // them, early in a chunk, so the next chunk's load has most of a chunk to land
  static constexpr int oQ0 = oW + NB * WATOM;
  static constexpr int oK0 = oQ0 + TILE;
  static constexpr int oV0 = oK0 + TILE;         // v stages
  static constexpr int oV1 = oV0 + TILE;
  // an all-ones [128 × 64] block one descriptor stride after either v stage:
  // the B operand [V | 1] (N = 80) gives Σ_s φ(k_s)ᵀ·1 next to ΔS and Σ_s P
  // next to P·V, without separate N = 16 products
  static constexpr int oVONE = oV1 + TILE;
  static constexpr int oKP = oVONE + TILE;       // φ(K): NB column blocks of [128 × 64]
  static constexpr int oS = oKP + NB * TILE;     // state operand, bf16 [DP × 64]
  static constexpr int oZF = oS + DP * kD * 2;   // z of the state operand, fp32 [DP]
  static constexpr int oQZ = oZF + DP * 4;       // q'·z partials [chunk parity][half][128 rows]
  static constexpr int oBAR = oQZ + 2 * 2 * kC * 4;
  static constexpr int NBAR = 40;
  static constexpr int oMISC = oBAR + NBAR * 8;  // tmem slot, abort flag
  static constexpr int BYTES = oMISC + 16;
  static constexpr int SMEM_ALLOC = (BYTES + 1024 > 118 * 1024) ? BYTES + 1024 : 118 * 1024;
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
  // tensor memory columns
  static constexpr uint32_t TST = 0;             // [S | z]: MB blocks of 80 columns (lanes =
                                                 // features; z in column 64 of a block)
  static constexpr uint32_t TN = 160;            // [num | Σ P]: 64 + 16 columns
  static constexpr uint32_t TR = TN + 64;        // Σ_s P_ts (16 equal columns, zeroed by the row
                                                 // warps before each chunk's products)
  static constexpr uint32_t TS = 256;            // scores / P; the q projection buffer (128 columns)
  static constexpr uint32_t TQ = 384;            // φ(Q) as bf16 pairs (DP/2 columns); the k
                                                 // projection buffer (128 columns)
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(TST + MB * 80 <= TN && TN + 80 <= TS && TQ + 128 <= TMEM_COLS, "TMEM");
  __host__ __device__ static constexpr uint32_t tst(int mb) { return TST + 80 * mb; }
  __host__ __device__ static constexpr uint32_t tz(int mb) { return TST + 80 * mb + 64; }
  // [V | 1] descriptor stride for v stage s: the distance to the ones block
  __host__ __device__ static constexpr int vone_lbo(int s) { return oVONE - (s ? oV1 : oV0); }
};

enum {
  B_W = 0,
  B_QFULL0, B_QFULL1, B_QEMPTY0, B_QEMPTY1,
  B_KFULL0, B_KFULL1, B_KEMPTY0, B_KEMPTY1,
  B_VFULL0, B_VFULL1, B_VEMPTY0, B_VEMPTY1,
  B_PKFULL, B_PKEMPTY,     // projection buffer of k (in the φ(Q) columns)
  B_PQFULL, B_PQEMPTY,     // projection buffer of q (in the scores columns)
  B_KREADY, B_KPEMPTY, B_QREADY, B_QPEMPTY,
  B_SCORES, B_PREADY, B_NUMFULL, B_NUMEMPTY,
  B_DSFULL, B_SCONV, B_SREADY, B_SEMPTY, B_MMADONE, B_COUNT
};
static_assert(B_COUNT <= PCfg<128>::NBAR, "barrier slots");

struct PParams {
  __nv_bfloat16* out;      // [BH, n, 64]
  int64_t n, seg_len;
  int nseg;
  float* ws_state;         // [BH][nseg][DP·64] segment aggregates → exclusive prefixes (scan)
  float* ws_z;             // [BH][nseg][DP]
  float* tot_state;        // non-causal: the sum of all aggregates [BH][DP·64] (scan)
  float* tot_z;
  float* fin_state;        // causal: final state [BH][DP·64] or nullptr
  float* fin_z;
  const float* init_state; // causal: state entering token 0 [BH][DP·64], or nullptr (zero)
  const float* init_z;     // [BH][DP]
  float half_log2m;        // ½·log2 m
  int* status;
};

struct PCtx {
  uint8_t* sm;
  uint32_t sbase;
  uint64_t* bar;
  volatile int* abort_flag;
  uint32_t tmem;
  int* status;
  int64_t bh, t_begin, t_end;
  int g, nchunks;
};

template <int MODE> struct Loads {
  static constexpr bool Q = MODE != kState;
  static constexpr bool K = MODE != kReadout;
  static constexpr bool V = MODE != kReadout;
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ roles

template <int DP, int MODE>
__device__ __forceinline__ void role_producer(const PCtx& x, const CUtensorMap* mq,
                                              const CUtensorMap* mk, const CUtensorMap* mv,
                                              const CUtensorMap* mw) {
  using Cfg = PCfg<DP>;
  using LD = Loads<MODE>;
  uint64_t* bar = x.bar;
  mbar_arrive_expect_tx(&bar[B_W], Cfg::NB * Cfg::WATOM);
  for (int f = 0; f < Cfg::NB; ++f) tma_load_2d(x.sm + Cfg::oW + f * Cfg::WATOM, mw, &bar[B_W], 64 * f, 0);
  int last[3] = {-1, -1, -1};   // last chunk loaded per operand (k, q, v)
  // ring of `stages` (1 or 2) buffers; stage s of chunk c = c % stages
  auto load = [&](const CUtensorMap* map, int off0, int off1, int full, int empty, int c, int y,
                  int which, int stages) -> bool {
    const int s = stages == 2 ? (c & 1) : 0;
    const int u = stages == 2 ? (c >> 1) : c;          // use index of the stage
    if (c >= stages && !mbar_wait(&bar[empty + s], (u - 1) & 1, x.status, x.abort_flag))
      return false;
    // the tile's first row lies in this CTA's token range
    if (!LA_DCHECK(x.status, y >= x.t_begin && y < x.t_end, 41)) return false;
    mbar_arrive_expect_tx(&bar[full + s], Cfg::TILE);
    tma_load_3d(x.sm + (s ? off1 : off0), map, &bar[full + s], 0, y, (int)x.bh);
    last[which] = c;
    return true;
  };
  for (int c = 0; c < x.nchunks && !*x.abort_flag; ++c) {
    const int y = (int)(x.t_begin + (int64_t)c * kC);
    if (LD::K && !load(mk, Cfg::oK0, Cfg::oK0, B_KFULL0, B_KEMPTY0, c, y, 0, 1)) break;
    if (LD::Q && !load(mq, Cfg::oQ0, Cfg::oQ0, B_QFULL0, B_QEMPTY0, c, y, 1, 1)) break;
    if (LD::V && !load(mv, Cfg::oV0, Cfg::oV1, B_VFULL0, B_VEMPTY0, c, y, 2, 2)) break;
  }
  if (*x.abort_flag) {
    // drain the loads still in flight before the CTA's shared memory goes away
    mbar_wait_drain(&bar[B_W], 0);
    const int full[3] = {B_KFULL0, B_QFULL0, B_VFULL0};
    const int stages[3] = {1, 1, 2};
    for (int w = 0; w < 3; ++w)
      for (int c = max(0, last[w] - stages[w] + 1); c <= last[w]; ++c)
        mbar_wait_drain(&bar[full[w] + (stages[w] == 2 ? (c & 1) : 0)],
                        (stages[w] == 2 ? (c >> 1) : c) & 1);
  }
}

// Three MMA issuers, one thread each (tcgen05.commit tracks the MMAs of
// the issuing thread, so each chain commits its own barriers; a tile read
// by two chains is released by a commit from each):
//   projections (warp 3):  U = X·ω per 64-feature block into two TMEM
//                          buffers per operand: k's in the φ(Q) columns (free
//                          once φ(Q)·S of the previous chunk is done, so they
//                          overlap its P mask and P·V), q's in the scores
//                          columns (free once P·V of the previous chunk is done)
//   state (warp 2):        ΔS = φ(K)ᵀV, Δz = φ(K)ᵀ1 onto the TMEM state
//   output (warp 1):       scores = φ(Q)·φ(K)ᵀ; num = φ(Q)·S, den = φ(Q)·z;
//                          num += P·V, den += P·1
// Operand descriptors are built once per tile and advanced by address.
template <int DP, int MODE>
__device__ __forceinline__ void role_mma_proj(const PCtx& x) {
  using Cfg = PCfg<DP>;
  using LD = Loads<MODE>;
  uint64_t* bar = x.bar;
  const uint32_t sb = x.sbase;
  constexpr uint32_t idP = idesc_bf16_f32(128, 128, false, true);   // U = X·ω, 128 features
  int* st = x.status;
  volatile int* ab = x.abort_flag;
  const uint64_t dW = smem_desc(sb + Cfg::oW, Cfg::WATOM, 1024, kSwizzle128B);
  bool ok = mbar_wait(&bar[B_W], 0, st, ab);
  int pk = 0, pq = 0;   // projection steps issued into the k / q buffer
  // U for features 128·f … 128·f + 127 of the raw tile at sX into the k
  // buffer (φ(Q) columns) or the q buffer (scores columns)
  auto project = [&](uint32_t sX, int f, bool is_k) -> bool {
    int& pj = is_k ? pk : pq;
    if (pj >= 1 && !mbar_wait(&bar[is_k ? B_PKEMPTY : B_PQEMPTY], (pj - 1) & 1, st, ab))
      return false;
    tc_fence_after();
    const uint64_t dX = smem_desc(sX, 16, 1024, kSwizzle128B);
    const uint32_t d = x.tmem + (is_k ? Cfg::TQ : Cfg::TS);
#pragma unroll
    for (int k = 0; k < kD / 16; ++k)
      mma_ss(d, desc_at(dX, k * 32), desc_at(dW, 2 * f * Cfg::WATOM + k * 2048), idP, k > 0);
    mma_commit(&bar[is_k ? B_PKFULL : B_PQFULL]);
    ++pj;
    return true;
  };
  for (int c = 0; ok && c < x.nchunks; ++c) {
    const int s = c & 1;
    if (LD::K) {
      // causal: the k buffers sit in the φ(Q) columns of chunk c − 1, free
      // once φ(Q)·S of that chunk (after its scores) has completed
      if (MODE == kCausal && c >= 1 && !mbar_wait(&bar[B_QPEMPTY], (c - 1) & 1, st, ab)) break;
      if (!mbar_wait(&bar[B_KFULL0], c & 1, st, ab)) break;
      for (int f = 0; ok && f < Cfg::NP; ++f) ok = project(sb + Cfg::oK0, f, true);
      if (!ok) break;
      mma_commit(&bar[B_KEMPTY0]);
    }
    if (LD::Q) {
      // causal: the q buffers sit in the scores columns, free once P·V of
      // chunk c − 1 has completed
      if (MODE == kCausal && c >= 1 && !mbar_wait(&bar[B_NUMFULL], (c - 1) & 1, st, ab)) break;
      if (!mbar_wait(&bar[B_QFULL0], c & 1, st, ab)) break;
      for (int f = 0; ok && f < Cfg::NP; ++f) ok = project(sb + Cfg::oQ0, f, false);
      if (!ok) break;
      mma_commit(&bar[B_QEMPTY0]);
    }
  }
  mma_commit(&bar[B_MMADONE]);
  mbar_wait_drain(&bar[B_MMADONE], 0);
}

template <int DP, int MODE>
__device__ __forceinline__ void role_mma_state(const PCtx& x) {
  using Cfg = PCfg<DP>;
  uint64_t* bar = x.bar;
  const uint32_t sb = x.sbase;
  constexpr uint32_t idD = idesc_bf16_f32(128, 80, true, true);     // [ΔS | Δz] = φ(K)ᵀ [V | 1]
  const uint64_t dKP = smem_desc(sb + Cfg::oKP, Cfg::TILE, 1024, kSwizzle128B);
  int* st = x.status;
  volatile int* ab = x.abort_flag;
  for (int c = 0; c < x.nchunks; ++c) {
    const int s = c & 1;
    const uint64_t dV =
        smem_desc(sb + (s ? Cfg::oV1 : Cfg::oV0), Cfg::vone_lbo(s), 1024, kSwizzle128B);
    if (!mbar_wait(&bar[B_KREADY], c & 1, st, ab)) break;
    if (!mbar_wait(&bar[B_VFULL0 + s], (c >> 1) & 1, st, ab)) break;
    if ((MODE == kCausal || c == 0) &&
        !mbar_wait(&bar[B_SCONV], MODE == kCausal ? (c & 1) : 0, st, ab))
      break;
    tc_fence_after();
#pragma unroll
    for (int mb = 0; mb < Cfg::MB; ++mb)
#pragma unroll
      for (int k = 0; k < kC / 16; ++k) {
        mma_ss(x.tmem + Cfg::tst(mb), desc_at(dKP, mb * 2 * Cfg::TILE + k * 2048),
               desc_at(dV, k * 2048), idD, 1);
      }
    mma_commit(&bar[B_DSFULL]);
    mma_commit(&bar[B_KPEMPTY]);
    mma_commit(&bar[B_VEMPTY0 + s]);
  }
  mma_commit(&bar[B_MMADONE]);
  mbar_wait_drain(&bar[B_MMADONE], 0);
}

template <int DP, int MODE>
__device__ __forceinline__ void role_mma_out(const PCtx& x) {
  using Cfg = PCfg<DP>;
  uint64_t* bar = x.bar;
  const uint32_t tmem = x.tmem;
  const uint32_t sb = x.sbase;
  constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);  // scores
  constexpr uint32_t idN = idesc_bf16_f32(128, 64, false, true);    // num (+)= A·{S, V}
  constexpr uint32_t idV = idesc_bf16_f32(128, 80, false, true);    // [num | den] += P·[V | 1]
  const uint64_t dKP = smem_desc(sb + Cfg::oKP, 16, 1024, kSwizzle128B);
  const uint64_t dS = smem_desc(sb + Cfg::oS, DP * 128, 1024, kSwizzle128B);
  int* st = x.status;
  volatile int* ab = x.abort_flag;
  for (int c = 0; c < x.nchunks; ++c) {
    const int s = c & 1;
    if (MODE == kCausal) {
      // scores = φ(Q)·φ(K)ᵀ over the m features
      if (!mbar_wait(&bar[B_KREADY], c & 1, st, ab)) break;
      if (!mbar_wait(&bar[B_QREADY], c & 1, st, ab)) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < DP / 16; ++k)
        mma_ts(tmem + Cfg::TS, tmem + Cfg::TQ + k * 8,
               desc_at(dKP, (k >> 2) * Cfg::TILE + (k & 3) * 32), idS, k > 0);
      mma_commit(&bar[B_SCORES]);
      mma_commit(&bar[B_KPEMPTY]);                 // φ(K) also read by ΔS (state chain)
    } else {
      if (!mbar_wait(&bar[B_QREADY], c & 1, st, ab)) break;
    }
    // num = φ(Q)·S (φ(Q)·z is summed by the φ warps)
    if ((MODE == kCausal || c == 0) &&
        !mbar_wait(&bar[B_SREADY], MODE == kCausal ? (c & 1) : 0, st, ab))
      break;
    if (c >= 1 && !mbar_wait(&bar[B_NUMEMPTY], (c - 1) & 1, st, ab)) break;
    tc_fence_after();
#pragma unroll
    for (int k = 0; k < DP / 16; ++k)
      mma_ts(tmem + Cfg::TN, tmem + Cfg::TQ + k * 8, desc_at(dS, k * 2048), idN, k > 0);
    if (MODE == kCausal) mma_commit(&bar[B_SEMPTY]);
    mma_commit(&bar[B_QPEMPTY]);                   // φ(Q) read by scores and num
    if (MODE == kReadout) {
      mma_commit(&bar[B_NUMFULL]);
      continue;
    }
    // [num | den] += P·[V | 1]
    const uint64_t dV =
        smem_desc(sb + (s ? Cfg::oV1 : Cfg::oV0), Cfg::vone_lbo(s), 1024, kSwizzle128B);
    if (!mbar_wait(&bar[B_PREADY], c & 1, st, ab)) break;
    if (!mbar_wait(&bar[B_VFULL0 + s], (c >> 1) & 1, st, ab)) break;
    tc_fence_after();
#pragma unroll
    for (int k = 0; k < kC / 16; ++k)
      mma_ts(tmem + Cfg::TN, tmem + Cfg::TS + k * 8, desc_at(dV, k * 2048), idV, 1);
    mma_commit(&bar[B_NUMFULL]);
    mma_commit(&bar[B_VEMPTY0 + s]);
  }
  mma_commit(&bar[B_MMADONE]);
  mbar_wait_drain(&bar[B_MMADONE], 0);
}

// Warps 8–15: φ.  Thread r: token row / TMEM lane r; `half` selects 64 of
// the 128 features of each projection step.  For q the warps also sum
// φ(q_r)·z over their features (the q'·z term of the denominator) into a
// per-row partial that the epilogue adds.
template <int DP, int MODE>
__device__ __forceinline__ void role_phi(const PCtx& x, const PParams& p, int warp, int lane) {
  using Cfg = PCfg<DP>;
  using LD = Loads<MODE>;
  uint64_t* bar = x.bar;
  int* st = x.status;
  volatile int* ab = x.abort_flag;
  const int half = (warp - 8) >> 2;
  const int r = (warp & 3) * 32 + lane;
  const uint32_t lane_base = (uint32_t)(warp & 3) * 32;
  const float* zf = reinterpret_cast<const float*>(x.sm + Cfg::oZF);
  float* qzbuf = reinterpret_cast<float*>(x.sm + Cfg::oQZ);
  int pk = 0, pq = 0;   // projection steps consumed from the k / q buffer
  // ½‖x_r‖²·log2 e + ½·log2 m for row r of a raw tile (the exponent offset)
  auto row_offset = [&](int off) -> float {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 u = lds128(x.sbase + off + sw_chunk(kC, r, 0, j));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = bf16lo_to_f32(w[e]), hi = bf16hi_to_f32(w[e]);
        ss = fmaf(lo, lo, ss);
        ss = fmaf(hi, hi, ss);
      }
    }
    return 0.5f * ss * kLog2e + p.half_log2m;
  };
  // one projection step f: φ of features 128·f + 64·half … + 63 of row r
  // (zero for dead rows); q also adds its features' φ·z to `qz`
  auto step = [&](bool is_k, int f, float off, bool live, float& qz) -> bool {
    int& pj = is_k ? pk : pq;
    if (!warp_wait(&bar[is_k ? B_PKFULL : B_PQFULL], pj & 1, st, ab)) return false;
    tc_fence_after();
    uint32_t u[64];
    const uint32_t src = tmem_addr(x.tmem, lane_base, (is_k ? Cfg::TQ : Cfg::TS) + 64 * half);
    tmem_ld32(src, u);
    tmem_ld32(src + 32, u + 32);
    tmem_ld_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[is_k ? B_PKEMPTY : B_PQEMPTY]);
    ++pj;
    const int f0 = 128 * f + 64 * half;            // first feature of this thread's 64
    uint32_t pkd[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float a0 = ex2_approx(fmaf(__uint_as_float(u[2 * j]), kLog2e, -off));
      const float a1 = ex2_approx(fmaf(__uint_as_float(u[2 * j + 1]), kLog2e, -off));
      pkd[j] = live ? pack_bf16x2(a0, a1) : 0u;
    }
    if (!is_k) {
      // q'·z with the bf16 values the tensor core sees in φ(Q)·S; z by 16-byte
      // broadcast loads (f0 is a multiple of 64)
#pragma unroll
      for (int j4 = 0; j4 < 16; ++j4) {
        const float4 z4 = *reinterpret_cast<const float4*>(zf + f0 + 4 * j4);
        qz += bf16lo_to_f32(pkd[2 * j4]) * z4.x + bf16hi_to_f32(pkd[2 * j4]) * z4.y +
              bf16lo_to_f32(pkd[2 * j4 + 1]) * z4.z + bf16hi_to_f32(pkd[2 * j4 + 1]) * z4.w;
      }
    }
    if (is_k) {
      const uint32_t base = x.sbase + Cfg::oKP + (2 * f + half) * Cfg::TILE;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        sts128(base + sw_chunk(kC, r, 0, q),
               make_uint4(pkd[4 * q], pkd[4 * q + 1], pkd[4 * q + 2], pkd[4 * q + 3]));
    } else {
      tmem_st32(tmem_addr(x.tmem, lane_base, Cfg::TQ + 64 * f + 32 * half), pkd);
    }
    return true;
  };
  for (int c = 0; c < x.nchunks; ++c) {
    const int s = c & 1;
    const int cs = (int)min((int64_t)kC, x.t_end - (x.t_begin + (int64_t)c * kC));
    if (LD::K) {
      if (!warp_wait(&bar[B_KFULL0], c & 1, st, ab)) return;
      const float off = row_offset(Cfg::oK0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_KEMPTY0]);
      // the φ(K) tile of the previous chunk must have been consumed
      if (c >= 1 && !warp_wait(&bar[B_KPEMPTY], (c - 1) & 1, st, ab)) return;
      float unused = 0.f;
      for (int f = 0; f < Cfg::NP; ++f)
        if (!step(true, f, off, r < cs, unused)) return;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_KREADY]);
    }
    if (LD::Q) {
      if (!warp_wait(&bar[B_QFULL0], c & 1, st, ab)) return;
      const float off = row_offset(Cfg::oQ0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_QEMPTY0]);
      if (c >= 1 && !warp_wait(&bar[B_QPEMPTY], (c - 1) & 1, st, ab)) return;
      // z of this chunk's state (written with the state operand)
      if ((MODE == kCausal || c == 0) &&
          !warp_wait(&bar[B_SREADY], MODE == kCausal ? (c & 1) : 0, st, ab))
        return;
      float qz = 0.f;
      for (int f = 0; f < Cfg::NP; ++f)
        if (!step(false, f, off, true, qz)) return;
      qzbuf[((c & 1) * 2 + half) * kC + r] = qz;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_QREADY]);
    }
  }
}

// Warps 4–7: thread r owns feature rows r and 128 + r of the state (TMEM
// lane r of each 128-feature block) and token row / TMEM lane r of a chunk.
template <int DP, int MODE>
__device__ __forceinline__ void role_rows(const PCtx& x, const PParams& p, int warp, int lane) {
  using Cfg = PCfg<DP>;
  uint64_t* bar = x.bar;
  const uint32_t tmem = x.tmem;
  int* st = x.status;
  volatile int* ab = x.abort_flag;
  const int r = (warp - 4) * 32 + lane;
  const int wq = warp - 4;
  const uint32_t lane_base = (uint32_t)wq * 32;
  const uint32_t stile = x.sbase + Cfg::oS;
  float* zf = reinterpret_cast<float*>(x.sm + Cfg::oZF);
  const float* qzbuf = reinterpret_cast<const float*>(x.sm + Cfg::oQZ);
  const int64_t agg0 = x.bh * p.nseg;
  // zero the Σ P columns of the accumulator (P·[V | 1] accumulates into them)
  auto zero_rowsum = [&]() {
    uint32_t zz[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) zz[j] = 0u;
    tmem_st16(tmem_addr(tmem, lane_base, Cfg::TR), zz);
  };

  // State row f = 128·mb + r is handled in two 32-column halves hh.
  // bf16 operand: 32 values of state-tile row f (16-byte chunks 4hh … 4hh+3)
  auto put_tile_half = [&](int f, int hh, const float* v) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = v[8 * q + e];
      sts128(stile + sw_chunk(DP, f, 0, 4 * hh + q), pack8(w));
    }
  };
  auto write_half = [&](float* dst_S, int f, int hh, const float* v) {
#pragma unroll
    for (int j = 0; j < 32; j += 4)
      *reinterpret_cast<float4*>(dst_S + (int64_t)f * kD + 32 * hh + j) =
          make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
  };
  // the fp32 state of block mb from TMEM → `sink(f, hh, v)` per half; returns z
  auto drain_state = [&](int mb, auto sink) -> float {
    uint32_t zr = 0;
    tmem_ld1(tmem_addr(tmem, lane_base, Cfg::tz(mb)), zr);
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t u[32];
      tmem_ld32(tmem_addr(tmem, lane_base, Cfg::tst(mb) + 32 * hh), u);
      tmem_ld_wait();
      sink(128 * mb + r, hh, reinterpret_cast<const float*>(u));
    }
    return __uint_as_float(zr);
  };

  // ---- initial state: the prefix of the aggregates before this segment
  // (causal, from the scan, which starts from the caller's initial state),
  // the caller's initial state (causal, first segment), the total
  // (readout), or zero (state)
  {
    const float* srcS = nullptr;
    const float* srcZ = nullptr;
    if (MODE == kCausal && x.g > 0) {
      srcS = p.ws_state + (agg0 + x.g) * (int64_t)(DP * kD);
      srcZ = p.ws_z + (agg0 + x.g) * DP;
    } else if (MODE == kCausal && p.init_state) {
      srcS = p.init_state + x.bh * (int64_t)(DP * kD);
      srcZ = p.init_z + x.bh * DP;
    } else if (MODE == kReadout) {
      srcS = p.tot_state + x.bh * (int64_t)(DP * kD);
      srcZ = p.tot_z + x.bh * DP;
    }
    if (srcS) grid_dependency_wait();
    for (int mb = 0; mb < Cfg::MB; ++mb) {
      const int f = 128 * mb + r;
      const float zsum = srcS ? srcZ[f] : 0.f;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float v[32];
        if (srcS) {
          const float4* src4 = reinterpret_cast<const float4*>(srcS + f * kD + 32 * hh);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 t = src4[j];
            v[4 * j] = t.x; v[4 * j + 1] = t.y; v[4 * j + 2] = t.z; v[4 * j + 3] = t.w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        if (MODE != kReadout)
          tmem_st32(tmem_addr(tmem, lane_base, Cfg::tst(mb) + 32 * hh),
                    reinterpret_cast<const uint32_t*>(v));
        if (MODE != kState) put_tile_half(f, hh, v);
      }
      if (MODE != kReadout) {
        const uint32_t zo = __float_as_uint(zsum);
        asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(
                         tmem_addr(tmem, lane_base, Cfg::tz(mb))),
                     "r"(zo)
                     : "memory");
      }
      if (MODE != kState) zf[f] = zsum;
    }
    if (MODE == kCausal) zero_rowsum();
    if (MODE != kReadout) tmem_st_wait();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&bar[B_SCONV]);
      mbar_arrive(&bar[B_SREADY]);
    }
  }

  if (MODE == kState) {
    bool ok = true;
    for (int c = 0; ok && c < x.nchunks; ++c) ok = warp_wait(&bar[B_DSFULL], c & 1, st, ab);
    if (!ok) return;
    tc_fence_after();
    float* dS = p.ws_state + (agg0 + x.g) * (int64_t)(DP * kD);
    for (int mb = 0; mb < Cfg::MB; ++mb) {
      const float zsum =
          drain_state(mb, [&](int f, int hh, const float* v) { write_half(dS, f, hh, v); });
      p.ws_z[(agg0 + x.g) * DP + 128 * mb + r] = zsum;
    }
    return;
  }

  for (int c = 0; c < x.nchunks; ++c) {
    if (MODE == kCausal) {
      if (c >= 1) {
        // operand tile for chunk c: S_c, accumulated by ΔS of chunk c−1
        if (!warp_wait(&bar[B_DSFULL], (c - 1) & 1, st, ab)) return;
        if (!warp_wait(&bar[B_SEMPTY], (c - 1) & 1, st, ab)) return;
        tc_fence_after();
        for (int mb = 0; mb < Cfg::MB; ++mb) {
          zf[128 * mb + r] =
              drain_state(mb, [&](int f, int hh, const float* v) { put_tile_half(f, hh, v); });
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bar[B_SCONV]);
          mbar_arrive(&bar[B_SREADY]);
        }
      }
      // ---- P: causal mask of the scores
      if (!warp_wait(&bar[B_SCORES], c & 1, st, ab)) return;
      tc_fence_after();
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        uint32_t pk[16];
        if (b > wq) {
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = 0u;
        } else {
          uint32_t sc[32];
          tmem_ld32(tmem_addr(tmem, lane_base, Cfg::TS + b * 32), sc);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int s0 = b * 32 + j;
            const float p0 = (s0 <= r) ? __uint_as_float(sc[j]) : 0.f;
            const float p1 = (s0 + 1 <= r) ? __uint_as_float(sc[j + 1]) : 0.f;
            pk[j / 2] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st16(tmem_addr(tmem, lane_base, Cfg::TS + b * 16), pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_PREADY]);
    }
    // ---- epilogue: o = num / den → bf16, row r straight to global memory
    if (!warp_wait(&bar[B_NUMFULL], c & 1, st, ab)) return;
    tc_fence_after();
    uint32_t psum = 0;
    if (MODE == kCausal) {
      tmem_ld1(tmem_addr(tmem, lane_base, Cfg::TR), psum);
      tmem_ld_wait();
    }
    // q'·z: the φ warps' partials, published with q_ready of this chunk
    if (!warp_wait(&bar[B_QREADY], c & 1, st, ab)) return;
    const float qz = qzbuf[((c & 1) * 2) * kC + r] + qzbuf[((c & 1) * 2 + 1) * kC + r];
    const float inv_den = 1.f / (__uint_as_float(psum) + qz);
    const int64_t row = x.t_begin + (int64_t)c * kC + r;
    const bool valid = row < x.t_end && LA_DCHECK(x.status, x.t_end <= p.n, 42);
    uint4* orow = reinterpret_cast<uint4*>(p.out + (x.bh * p.n + (valid ? row : 0)) * kD);
#pragma unroll 1
    for (int j0 = 0; j0 < kD; j0 += 32) {
      uint32_t nv[32];
      tmem_ld32(tmem_addr(tmem, lane_base, Cfg::TN + j0), nv);
      tmem_ld_wait();
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(nv[q8 * 8 + e]) * inv_den;
        if (valid) __stcs(orow + (j0 + q8 * 8) / 8, pack8(f));
      }
    }
    if (MODE == kCausal) {
      zero_rowsum();
      tmem_st_wait();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_NUMEMPTY]);
  }
  // ---- final state of the sequence (causal, last segment)
  if (MODE == kCausal && p.fin_state && x.g == p.nseg - 1) {
    if (!warp_wait(&bar[B_DSFULL], (x.nchunks - 1) & 1, st, ab)) return;
    tc_fence_after();
    float* dS = p.fin_state + x.bh * (int64_t)(DP * kD);
    for (int mb = 0; mb < Cfg::MB; ++mb) {
      const float zsum =
          drain_state(mb, [&](int f, int hh, const float* v) { write_half(dS, f, hh, v); });
      p.fin_z[x.bh * DP + 128 * mb + r] = zsum;
    }
  }
}

template <int DP, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
tcp_forward_kernel(const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v,
                   const __grid_constant__ CUtensorMap map_w, const PParams p) {
  using Cfg = PCfg<DP>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  PCtx x;
  x.sm = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  x.sbase = smem_u32(x.sm);
  x.bar = reinterpret_cast<uint64_t*>(x.sm + Cfg::oBAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(x.sm + Cfg::oMISC);
  x.abort_flag = reinterpret_cast<volatile int*>(x.sm + Cfg::oMISC + 4);
  x.status = p.status;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // a launch that depends on this state launch may start now
  if (MODE == kState) grid_dependents_launch();
  // grid (heads, segments)
  x.bh = blockIdx.x;
  x.g = blockIdx.y;
  x.t_begin = (int64_t)x.g * p.seg_len;
  x.t_end = min(p.n, x.t_begin + p.seg_len);
  x.nchunks = (int)((x.t_end - x.t_begin + kC - 1) / kC);

  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      if (i == B_QEMPTY0 || i == B_QEMPTY1 || i == B_KEMPTY0 || i == B_KEMPTY1) cnt = 1 + 8;
      if (i == B_PKEMPTY || i == B_PQEMPTY || i == B_KREADY || i == B_QREADY) cnt = 8;
      if (i == B_PREADY || i == B_NUMEMPTY || i == B_SCONV || i == B_SREADY) cnt = 4;
      // released by two MMA chains in the causal mode: φ(K) (scores, ΔS), V (ΔS, P·V)
      if ((i == B_KPEMPTY || i == B_VEMPTY0 || i == B_VEMPTY1) && MODE == kCausal) cnt = 2;
      if (i == B_MMADONE) cnt = MODE == kCausal ? 3 : 2;
      mbar_init(&x.bar[i], cnt);
    }
    *x.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  {
    uint32_t* vone = reinterpret_cast<uint32_t*>(x.sm + Cfg::oVONE);
    for (int i = tid; i < Cfg::TILE / 4; i += kThreads) vone[i] = 0x3F803F80u;   // bf16 1.0 pairs
    fence_proxy_async_smem();                     // read by the tensor core
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_w);
    if (Loads<MODE>::Q) tma_prefetch_desc(&map_q);
    if (Loads<MODE>::K) tma_prefetch_desc(&map_k);
    if (Loads<MODE>::V) tma_prefetch_desc(&map_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  x.tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) role_producer<DP, MODE>(x, &map_q, &map_k, &map_v, &map_w);
  } else if (warp == 1) {
    if (MODE != kState && lane == 0) role_mma_out<DP, MODE>(x);
  } else if (warp == 2) {
    if (MODE != kReadout && lane == 0) role_mma_state<DP, MODE>(x);
  } else if (warp == 3) {
    if (lane == 0) role_mma_proj<DP, MODE>(x);
  } else if (warp >= 4 && warp < 8) {
    role_rows<DP, MODE>(x, p, warp, lane);
  } else if (warp >= 8) {
    role_phi<DP, MODE>(x, p, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(x.tmem, Cfg::TMEM_COLS);
  }
  // a dependent launch completes only after the launch it depends on
  if (MODE != kState) grid_dependency_wait();
}

template <int DP, int MODE>
cudaError_t launch(const PParams& p, dim3 grid, bool dependent, const CUtensorMap& mq,
                   const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mw,
                   cudaStream_t stream) {
  using Cfg = PCfg<DP>;
  cudaError_t e = cudaFuncSetAttribute(tcp_forward_kernel<DP, MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg::SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, tcp_forward_kernel<DP, MODE>, mq, mk, mv, mw, p);
  count_launches(1);
  return e;
}

template <int DP>
cudaError_t run(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                float* tot_state, float* tot_z, const SegmentPlan& plan) {
  const int64_t BH = a.B * a.H;
  CUtensorMap mq, mk, mv, mw;
  cudaError_t e;
  if ((e = tmap_rows(&mq, a.q, BH, a.n, kD, kC)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mk, a.k, BH, a.n, kD, kC)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mv, a.v, BH, a.n, kD, kC)) != cudaSuccess) return e;
  if ((e = tmap_matrix(&mw, a.omega, kD, DP, 64)) != cudaSuccess) return e;
  PParams p{};
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.n = a.n;
  p.seg_len = plan.seg_len;
  p.nseg = plan.nseg;
  p.ws_state = ws_state;
  p.ws_z = ws_z;
  p.tot_state = tot_state;
  p.tot_z = tot_z;
  p.fin_state = a.mu_out;
  p.fin_z = a.nu_out;
  p.init_state = a.causal ? a.init_state : nullptr;
  p.init_z = a.causal ? a.init_z : nullptr;
  p.half_log2m = 0.5f * log2f((float)DP);
  p.status = a.status;
  const unsigned ubh = (unsigned)BH;
  if (a.causal) {
    if (plan.nseg > 1) {
      // aggregates of segments 0 … nseg−2 (nothing follows the last one),
      // then their exclusive prefixes in place
      e = launch<DP, kState>(p, dim3(ubh, (unsigned)(plan.nseg - 1)), false, mq, mk, mv, mw, stream);
      if (e != cudaSuccess) return e;
      e = segment_scan(ws_state, ws_z, nullptr, nullptr, a.B * a.H, a.H, plan.nseg, plan.nseg - 1,
                       plan.seg_len, a.n, DP, kD, nullptr, nullptr, stream, true, p.init_state,
                       p.init_z);
      if (e != cudaSuccess) return e;
    }
    return launch<DP, kCausal>(p, dim3(ubh, (unsigned)plan.nseg), plan.nseg > 1, mq, mk, mv, mw,
                               stream);
  }
  // non-causal: all the aggregates, then their total (the final state)
  e = launch<DP, kState>(p, dim3(ubh, (unsigned)plan.nseg), false, mq, mk, mv, mw, stream);
  if (e != cudaSuccess) return e;
  e = segment_total(ws_state, ws_z, tot_state, tot_z, a.B * a.H, a.H, plan.nseg, plan.seg_len,
                    a.n, DP, kD, nullptr, nullptr, stream, true);
  if (e != cudaSuccess) return e;
  return launch<DP, kReadout>(p, dim3(ubh, (unsigned)plan.nseg), true, mq, mk, mv, mw, stream);
}

// The aggregate of every segment (the state launch over all of them).
template <int DP>
cudaError_t run_state(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                      const SegmentPlan& plan) {
  const int64_t BH = a.B * a.H;
  CUtensorMap mq, mk, mv, mw;
  cudaError_t e;
  // the state launch never reads q; its map describes k
  if ((e = tmap_rows(&mq, a.k, BH, a.n, kD, kC)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mk, a.k, BH, a.n, kD, kC)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mv, a.v, BH, a.n, kD, kC)) != cudaSuccess) return e;
  if ((e = tmap_matrix(&mw, a.omega, kD, DP, 64)) != cudaSuccess) return e;
  PParams p{};
  p.n = a.n;
  p.seg_len = plan.seg_len;
  p.nseg = plan.nseg;
  p.ws_state = ws_state;
  p.ws_z = ws_z;
  p.half_log2m = 0.5f * log2f((float)DP);
  p.status = a.status;
  return launch<DP, kState>(p, dim3((unsigned)BH, (unsigned)plan.nseg), false, mq, mk, mv, mw,
                            stream);
}

}  // namespace

bool tc_performer_supported(const FwdArgs& a) {
  return a.bf16 && a.performer && a.d == kD && (a.m == 128 || a.m == 256) && a.decay == nullptr &&
         a.tok_decay == nullptr &&
         a.n >= kC;
}

cudaError_t tc_performer_state_only(const FwdArgs& a, cudaStream_t stream, float* ws_state,
                                    float* ws_z, const SegmentPlan& plan) {
  if (a.m == 256) return run_state<256>(a, stream, ws_state, ws_z, plan);
  if (a.m == 128) return run_state<128>(a, stream, ws_state, ws_z, plan);
  return cudaErrorInvalidValue;
}

cudaError_t tc_performer_forward(const FwdArgs& a, cudaStream_t stream, float* ws_state,
                                 float* ws_z, float* tot_state, float* tot_z,
                                 const SegmentPlan& plan) {
  if (a.m == 256) return run<256>(a, stream, ws_state, ws_z, tot_state, tot_z, plan);
  if (a.m == 128) return run<128>(a, stream, ws_state, ws_z, tot_state, tot_z, plan);
  return cudaErrorInvalidValue;
}

}  // namespace la
