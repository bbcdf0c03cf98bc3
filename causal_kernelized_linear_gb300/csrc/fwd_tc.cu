// Tensor-core (tcgen05 + TMA + TMEM) chunked forward of causal kernelized
// linear attention, elu+1 feature map, bf16 inputs, fp32 state, d = d' ∈ {64, 128}.
//
// Method ("Efficient Transformers II" §2.2, eq (7)–(11) with the causal
// readout of eq (9)); per head, a chunk of C = 128 tokens (local t, s), cs of
// them valid, with state (μ, ν) = (S, z) at its start:
//   P_ts  = w·a^{t−s}·(q'_t·k'_s) for s ≤ t, else 0
//   num_t = Σ_s P_ts v_s + a^{t+1} q'_t·S,   den_t = Σ_s P_ts + a^{t+1} q'_t·z
//   o_t   = num_t / den_t
//   S ← a^{cs}·S + Σ_s w·a^{cs−1−s} k'_sᵀ v_s,   z likewise
// i.e. eq (10)–(11) unrolled over the chunk; the intra-chunk part is the
// quadratic form of "Efficient Transformers I" eq (25)–(26) on the chunk.
//
// The decay is folded into the bf16 tensor-core operands.  Two foldings:
//   centered (a ≥ 0.5 or a = 1):  Q'' = a^{t−63}·q',  K'' = w·a^{63−s}·k'
//       Q''K''ᵀ = w·a^{t−s}·Q'K'ᵀ, so P is the causally masked product itself;
//       num = P·V + Q''·(a^{64}S);  ΔS'' = K''ᵀV,  S ← a^{cs}S + a^{cs−64}ΔS''.
//       Every power stays within a^{±64}, inside bf16/fp32 range for a ≥ 0.5.
//       Only Q'' (TMEM) and K'' (smem; the K-major view feeds Q''K''ᵀ, the
//       MN-major view feeds K''ᵀV) are needed, so the raw Q/K tiles are
//       released as soon as φ has read them.
//   general (any a ∈ [0, 1]):  Q' = q' (TMEM), K' (smem), K'' = w·a^{cs−1−s}k';
//       P = (w·a^{t−s}) ⊙ Q'K'ᵀ with a table of w·a^k; the product Q'·S is
//       scaled by a^{t+1} row by row in fp32 before P·V accumulates onto it:
//       num = P·V + a^{t+1}(Q'·S);  S ← a^{cs}S + K''ᵀV.
// Each CTA picks the folding for its head's a.
// Per-token decay (the same page's eq (4) with a and b indexed by the token):
//   the general folding with L_t = Σ_{j≤t} log2 a_j over the chunk (log2
//   clamped at −64):  K' = b_s·k',  K'' = b_s·2^{L_{cs−1}−L_s}k',
//   P = 2^{L_t−L_s} ⊙ Q'K'ᵀ (computed per element), the row scale 2^{L_t},
//   TMEM = 2^{L_{cs−1}}·S_c; the segment aggregates carry their total log2
//   decay to the combine.
//
// One CTA per (segment, head), 16 warps:
//   warp 0        TMA producer
//   warp 1        tcgen05 MMA issuer for the output products, TMEM owner
//   warp 2        tcgen05 MMA issuer for the state products
//   warps 4–7     masked P; epilogue o = num/den stored row by row
//                 (state-only launch: a share of φ(K))
//   warps 8–15    φ(K) → K'' (and K') one chunk ahead; the state update (fp32
//                 state in TMEM); φ(Q) → Q'' in TMEM (and Q'); one column
//                 half per warpgroup (d = 64: warps 8–11 all columns, warps
//                 12–15 compute φ(Q), or in the state-only launch a share of φ(K))
// tcgen05 products: scores = Q''K''ᵀ (or Q'K'ᵀ), ΔS = K''ᵀV, Δz = K''ᵀ1,
// num = Q''S + P·V, den = Q''z + P·1 — fp32 accumulators in TMEM; S and z
// enter the products as bf16 operands.
// Long sequences are split into segments: a state-only launch of this kernel
// computes the decayed aggregate of every segment but the last; the full
// launch combines the aggregates before each segment into its entering state
// and produces o (and, from the last segment, the final state).  The full
// launch is a programmatic dependent of the state-only one: it starts on the
// SMs the state-only launch leaves free (and as its CTAs finish), and only
// the reads of the aggregates wait for it to complete.
// Every wait is bounded in time: on expiry the kernel records LA_ERR_TIMEOUT
// in the device status word, stops issuing work, drains what it issued and
// frees its TMEM.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

#include <cuda.h>

namespace la {
namespace {

using namespace tc;

constexpr int kC = 128;                  // tokens per chunk (MMA M)
constexpr int kThreadsTc = 512;          // 16 warps
constexpr float kCenteredMinDecay = 0.5f;

template <int D>
struct TcCfg {
  static constexpr int HALVES = D / 64;          // 64-column (128-byte) swizzle atoms per row
  static constexpr int TILE = kC * D * 2;        // one [128 × D] bf16 tile
  static constexpr int STILE = D * D * 2;        // state tile [D × D] bf16
  // shared memory (offsets from a 1024-aligned base): seven [128 × D] tiles
  // (see Layout for their roles), the bf16 state operand and small tables.
  static constexpr int oT0 = 0;
  static constexpr int oT1 = oT0 + TILE;
  static constexpr int oT2 = oT1 + TILE;
  static constexpr int oKP = oT2 + TILE;
  static constexpr int oV0 = oKP + TILE;
  static constexpr int oV1 = oV0 + TILE;
  static constexpr int oS = oV1 + TILE;          // state operand, bf16 [D' × D]
  static constexpr int oONES = oS + STILE;       // 8×8 bf16 ones (128 B; every core matrix aliases it)
  // normalizer operand z, bf16 [D'] followed by 112 readable bytes: the B
  // operand of den = Q''·z is K-major with its core matrices 16 bytes apart,
  // so row 0 of each holds z and rows 1–7 (output columns never read) overlap
  // the next ones
  static constexpr int oZB = oONES + 128;
  static constexpr int oPW = oZB + 2 * D + 128;  // w·a^k, k = 0..127 (general folding)
  static constexpr int oBAR = oPW + 132 * 4;     // mbarriers
  static constexpr int NBAR = 33;
  static constexpr int oMISC = oBAR + NBAR * 8;  // tmem slot, abort flag
  static constexpr int BYTES = oMISC + 16;
  // + alignment slack; at least half of the SM's shared memory so that one
  // CTA (which owns all 512 TMEM columns) runs per SM
  static constexpr int SMEM_ALLOC = (BYTES + 1024 > 118 * 1024) ? BYTES + 1024 : 118 * 1024;
  // tensor memory columns
  static constexpr uint32_t TS = 0;              // scores (fp32) / P (bf16 pairs)
  static constexpr uint32_t TN = 128;            // numerator [128 × D]
  static constexpr uint32_t TD = TN + D;         // ΔS [D' × D] (lanes = feature)
  static constexpr uint32_t TZ = TD + D;         // Δz (16 columns, column 0 used)
  static constexpr uint32_t TR = TZ + 16;        // q''·z + Σ_s P_ts (16 columns, column 0 used)
  static constexpr uint32_t TQ = (D == 128) ? 448 : 320;  // Q'' (bf16 pairs, D/2 columns)
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(TR + 16 <= TQ, "TMEM layout");
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

enum {
  B_QFULL0 = 0, B_QFULL1, B_QEMPTY0, B_QEMPTY1,
  B_KFULL0, B_KFULL1, B_KFULL2, B_KEMPTY0, B_KEMPTY1, B_KEMPTY2,
  B_VFULL0, B_VFULL1, B_VFULL2, B_VEMPTY0, B_VEMPTY1, B_VEMPTY2,
  B_KREADY0, B_KREADY1, B_KREADY2,   // one per K stage: φ(K) may run a chunk ahead
  B_QREADY0, B_QREADY1,              // one per Q stage: Q'' (centered) or Q' (general) ready
  B_KPEMPTY, B_SREADY, B_SEMPTY, B_SCORES, B_PREADY, B_NUMFULL, B_NUMEMPTY,
  B_DSFULL, B_DSEMPTY, B_QPEMPTY, B_MMADONE, B_COUNT
};
static_assert(B_COUNT <= TcCfg<64>::NBAR, "barrier slots");

// Roles of the seven tiles T0, T1, T2, KP, V0, V1 (and S) per kernel mode:
//   centered, full:  Q stages T0, T1 | K stages T2, KP (φ(K) writes K'' in place) | V V0, V1
//   general, full:   Q T0 | K stages T1, T2 (K' in place) | K'' in KP | V V0, V1
// In both full modes the raw Q tile is released as soon as φ(Q) has read it
// (the products read φ(Q) from TMEM).
//   state-only:      K stages T0, T1, T2 (K'' in place) | V stages KP, V0, V1
template <int D, bool FULL, bool CEN>
struct Layout {
  using Cfg = TcCfg<D>;
  static constexpr int QST = (FULL && CEN) ? 2 : 1;
  static constexpr int KST = FULL ? 2 : 3;
  static constexpr int VST = FULL ? 2 : 3;
  static constexpr bool K_IN_PLACE = !(FULL && !CEN);   // K'' overwrites the raw K tile
  __device__ static int q_off(int s) { return s ? Cfg::oT1 : Cfg::oT0; }
  __device__ static int k_off(int s) {
    if (FULL && CEN) return s ? Cfg::oKP : Cfg::oT2;
    if (FULL) return s ? Cfg::oT2 : Cfg::oT1;
    return s == 0 ? Cfg::oT0 : (s == 1 ? Cfg::oT1 : Cfg::oT2);
  }
  __device__ static int kpp_off(int s) { return K_IN_PLACE ? k_off(s) : Cfg::oKP; }
  __device__ static int v_off(int s) {
    if (FULL) return s ? Cfg::oV1 : Cfg::oV0;
    return s == 0 ? Cfg::oKP : (s == 1 ? Cfg::oV0 : Cfg::oV1);
  }
};

struct TcParams {
  __nv_bfloat16* out;      // [BH, n, D]
  const float* decay;      // [H] or nullptr
  const float* tok_decay;  // per-token decay [BH, n] or nullptr
  const float* tok_weight; // per-token weight [BH, n] or nullptr (1 − a)
  float* ws_ld;            // per-token decay: [BH][nseg] log2 decay of each segment
  const float* tok_L;      // per-token decay: [BH, n] log2 prefix of a within each chunk
  const float* tok_B;      // per-token decay: [BH, n] weight b (or 1 − a)
  int64_t H, n, seg_len;
  int nseg;
  float* ws_state;         // [BH][nseg][D*D]
  float* ws_z;             // [BH][nseg][D]
  float* fin_state;        // final state (single-segment full launch) or nullptr
  float* fin_z;
  int init_slot;           // 1: slot 0 of every head's aggregates holds the state
                           // entering token 0, segment g's aggregate is in slot
                           // g + 1 (nseg + 1 slots per head); 0: no initial state
  int* status;
};


// a^e for integer e of either sign (a > 0, or e ≥ 0).
__device__ __forceinline__ float decay_pow_signed(float a, int e) {
  return e == 0 ? 1.f : powf(a, (float)e);
}

struct Ctx {
  uint8_t* sm;
  uint32_t sbase;
  uint64_t* bar;
  volatile int* abort_flag;
  __nv_bfloat16* zb;
  float* pw;
  uint32_t tmem;
  int* status;
  int64_t bh, t_begin, t_end;
  int g, nchunks;
  float a, w;
  float lg;    // log2 a (centered folding; 0 for a = 1)
  int R;       // centered folding: the TMEM state is rescaled every R chunks
  const float* ta;   // per-token decay of this head (token 0 of the head), or nullptr
  const float* tl;   // its chunk prefixes L (tok_prefix_kernel), or nullptr
  const float* tw;   // its weights B (tok_prefix_kernel), or nullptr
};

// Per-token decay of chunk c, computed by one warp (hardware lg2/ex2
// approximations: their relative error, ≈ 2^-22, is far below the bf16
// rounding the factors get as tensor-core operands): lane j gets, for each
// 32-token block i of the chunk, L[i] = Σ_{s ≤ 32i+j} log2 a_s (the running
// sum from the chunk's first token, log2 clamped at −64; tokens past the
// end add 0) and B[i] = b_{32i+j} (0 past the end); tot is the chunk's sum.
struct TokChunk {
  float L[4];
  float B[4];
  float tot;
};

__device__ __forceinline__ float pick4(const float (&v)[4], int i) {
  return i == 0 ? v[0] : (i == 1 ? v[1] : (i == 2 ? v[2] : v[3]));
}

// The precomputed L and B of one chunk for a warp (lane j: tokens 32i + j),
// loaded one chunk ahead of their use so that their latency overlaps a
// chunk's work.  The loads are unconditional (tokens past the end read the
// chunk's last token) and the values stay as loaded until tok_chunk uses
// them: masking them here would make each load wait for its data at once.
struct TokPipe {
  float L[4];
  float B[4];
  int cs;       // valid tokens of the chunk
  int c;        // the chunk they belong to, −1 for none
};

__device__ __forceinline__ void tok_load(const Ctx& x, int c, int lane, TokPipe& pp) {
  const int64_t t0 = x.t_begin + (int64_t)c * kC;
  const int cs = (int)min((int64_t)kC, x.t_end - t0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int s = min(32 * i + lane, cs - 1);
    pp.L[i] = __ldg(x.tl + t0 + s);
    pp.B[i] = __ldg(x.tw + t0 + s);
  }
  pp.cs = cs;
  pp.c = c;
}

// Chunk c's decay from the pipe (loading it now if the pipe holds another
// chunk), then the loads of chunk c + 1 are issued.  L past the end is the
// last token's (those tokens add no decay), so the chunk total is lane 31's
// value of the last block.
__device__ __forceinline__ TokChunk tok_chunk(const Ctx& x, int c, int lane, TokPipe& pp) {
  TokChunk t;
  if (pp.c != c) tok_load(x, c, lane, pp);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    t.L[i] = pp.L[i];
    t.B[i] = 32 * i + lane < pp.cs ? pp.B[i] : 0.f;
  }
  t.tot = __shfl_sync(0xffffffffu, pp.L[3], 31);
  if (c + 1 < x.nchunks) tok_load(x, c + 1, lane, pp);
  return t;
}

// The per-token decay of every 128-token chunk of every head, once before the
// tensor-core launches (one warp per chunk): L_t = Σ_{s ≤ t} max(log2 a_s, −64)
// from the chunk's first token (hardware lg2; its relative error, ≈ 2^-22, is
// far below the bf16 rounding the factors get as tensor-core operands), and
// B_t = b_t (1 − a_t without a weight array).  tok_load / tok_chunk read them.
__global__ void __launch_bounds__(128)
tok_prefix_kernel(const float* __restrict__ ta, const float* __restrict__ tb,
                  float* __restrict__ L, float* __restrict__ B, int64_t n, int64_t nch,
                  int64_t chunks) {
  const int64_t wid = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= chunks) return;
  const int64_t bh = wid / nch;
  const int64_t t0 = (wid % nch) * kC;
  const int cs = (int)min((int64_t)kC, n - t0);
  const int64_t base = bh * n + t0;
  float av[4], bv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int s = 32 * i + lane;
    av[i] = s < cs ? ta[base + s] : 1.f;
    bv[i] = s < cs ? (tb ? tb[base + s] : 1.f - av[i]) : 0.f;
  }
  float run = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float v = fmaxf(lg2_f32(av[i]), -64.f);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    const int s = 32 * i + lane;
    if (s < cs) {
      L[base + s] = run + v;
      B[base + s] = bv[i];
    }
    run += __shfl_sync(0xffffffffu, v, 31);
  }
}

// Per-warp running state of the per-token decay, advanced by φ(K) chunk by
// chunk: the load pipe, and for the chunk φ(K) last ran on L_r (this thread's
// row), L_{cs−1} and L_63.  The centered folding (Q̃ = 2^{L_t − L_63}φ(q),
// K̃ = σ·b_s·2^{L_63 − L_s}φ(k)) also keeps log2 ρ of that chunk and, for the
// state update of the chunk before it, whether its TMEM state is renormalised
// and by which factor.  With Δ_c = L_63(c+1) + L_{cs−1}(c) − L_63(c) (the decay
// from token 63 of chunk c to token 63 of chunk c + 1), log2 ρ_{c+1} =
// log2 ρ_c + Δ_c, reset to 0 (a renormalisation) once it falls below −32, so
// that σ = 1/ρ never exceeds 2^32.
struct TokTrack {
  TokPipe pipe;
  float lr, tot, mid;
  float lrho;
  bool renorm_prev;
  float alpha_prev;
};

__device__ __forceinline__ void tok_track_init(TokTrack& tt) {
  tt.pipe.c = -1;
  tt.lr = tt.tot = tt.mid = tt.lrho = 0.f;
  tt.renorm_prev = false;
  tt.alpha_prev = 1.f;
}

// Centered folding, lazy rescaling: K'' of chunk c carries σ_c = a^{−128·(c mod R)}
// (all chunks but the last are full), so that the state MMA can keep
// accumulating onto the TMEM state for R chunks before it is rescaled.
__device__ __forceinline__ float lazy_sigma(const Ctx& x, int c) {
  return exp2f(-128.f * (float)(c % x.R) * x.lg);
}

// ------------------------------------------------------------------ roles

template <int D, bool FULL, bool CEN>
__device__ __forceinline__ void role_producer(const Ctx& x, const CUtensorMap* map_q,
                                              const CUtensorMap* map_k,
                                              const CUtensorMap* map_v) {
  using Cfg = TcCfg<D>;
  using L = Layout<D, FULL, CEN>;
  uint64_t* bar = x.bar;
  int last_q = -1, last_k = -1, last_v = -1;
  auto load = [&](const CUtensorMap* map, int off, uint64_t* b, int y) {
    // the tile's first row lies in this CTA's token range
    if (!LA_DCHECK(x.status, y >= x.t_begin && y < x.t_end, 11)) return;
    mbar_arrive_expect_tx(b, Cfg::TILE);
    for (int h = 0; h < Cfg::HALVES; ++h)
      tma_load_3d(x.sm + off + h * kC * 128, map, b, h * 64, y, (int)x.bh);
  };
  // Every wait below is for a chunk at least two behind, so the producer runs
  // up to one full stage ring ahead of the consumers.
  for (int c = 0; c < x.nchunks && !*x.abort_flag; ++c) {
    const int y = (int)(x.t_begin + (int64_t)c * kC);
    if (FULL) {
      const int qs = c % L::QST;
      if (c >= L::QST &&
          !mbar_wait(&bar[B_QEMPTY0 + qs], ((c - L::QST) / L::QST) & 1, x.status, x.abort_flag))
        break;
      load(map_q, L::q_off(qs), &bar[B_QFULL0 + qs], y);
      last_q = c;
    }
    const int ks = c % L::KST;
    if (c >= L::KST &&
        !mbar_wait(&bar[B_KEMPTY0 + ks], ((c - L::KST) / L::KST) & 1, x.status, x.abort_flag))
      break;
    load(map_k, L::k_off(ks), &bar[B_KFULL0 + ks], y);
    last_k = c;
    const int vs = c % L::VST;
    if (c >= L::VST &&
        !mbar_wait(&bar[B_VEMPTY0 + vs], ((c - L::VST) / L::VST) & 1, x.status, x.abort_flag))
      break;
    load(map_v, L::v_off(vs), &bar[B_VFULL0 + vs], y);
    last_v = c;
  }
  if (*x.abort_flag) {
    // drain the loads still in flight before the CTA's shared memory goes away
    if (FULL)
      for (int c = max(0, last_q - L::QST + 1); c <= last_q; ++c)
        mbar_wait_drain(&bar[B_QFULL0 + c % L::QST], (c / L::QST) & 1);
    for (int c = max(0, last_k - L::KST + 1); c <= last_k; ++c)
      mbar_wait_drain(&bar[B_KFULL0 + c % L::KST], (c / L::KST) & 1);
    for (int c = max(0, last_v - L::VST + 1); c <= last_v; ++c)
      mbar_wait_drain(&bar[B_VFULL0 + c % L::VST], (c / L::VST) & 1);
  }
}

// Two MMA issuers, each a single thread; tcgen05.commit tracks the
// operations of the issuing thread, so each chain commits its own barriers.
// Output chain (warp 1): scores, num = Q''·S and den = Q''·z, then
// num += P·V and den += P·1.  State chain (warp 2): ΔS = K''ᵀV, Δz = K''ᵀ1.
// Tiles read by both chains (K'' in the centered folding, V) are released
// by a commit from each.
template <int D, bool CEN, bool QIP>
__device__ __forceinline__ void role_mma_out(const Ctx& x) {
  using Cfg = TcCfg<D>;
  using L = Layout<D, true, CEN>;
  uint64_t* bar = x.bar;
  const uint32_t tmem = x.tmem;
  const uint32_t sONES = x.sbase + Cfg::oONES;
  const uint64_t dS = smem_desc(x.sbase + Cfg::oS, D * 128, 1024, kSwizzle128B);
  const uint64_t dZ = smem_desc(x.sbase + Cfg::oZB, 16, 0, kSwizzleNone);
  constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);   // scores
  constexpr uint32_t idN = idesc_bf16_f32(128, D, false, true);      // num (+)= A·{S, V}
  constexpr uint32_t idR = idesc_bf16_f32(128, 16, false, false);    // den: Q''·z, P·1
  constexpr int KD = D / 16;                                         // K-steps over D'
  const uint64_t ones = smem_desc(sONES, 0, 0, kSwizzleNone);        // all core matrices alias
  int* st = x.status;
  volatile int* ab = x.abort_flag;
  for (int c = 0; c < x.nchunks; ++c) {
    const int ks = c % L::KST, vs = c % L::VST, qs = c % L::QST;
    const uint32_t sK = x.sbase + L::k_off(ks);
    const uint32_t sV = x.sbase + L::v_off(vs);
    // K-step k of a K-major [128 × D] operand tile (64-column atoms)
    auto kstep = [](int k) { return (uint32_t)((k >> 2) * (kC * 128) + (k & 3) * 32); };
    // QIP: Q'' in place of the raw Q tile (A from shared memory); otherwise
    // Q'' (Q') in TMEM
    const uint64_t dQ = smem_desc(x.sbase + L::q_off(qs), 16, 1024, kSwizzle128B);
    // scores = Q''K''ᵀ (centered; K'' in place of K) or Q'K'ᵀ (general; K'
    // in place of K); P(c−1) in the same columns must have been consumed by
    // P·V of chunk c−1
    if (!mbar_wait(&bar[B_KREADY0 + ks], (c / L::KST) & 1, st, ab)) break;
    if (!mbar_wait(&bar[B_QREADY0 + qs], (c / L::QST) & 1, st, ab)) break;
    if (c >= 1 && !mbar_wait(&bar[B_NUMFULL], (c - 1) & 1, st, ab)) break;
    tc_fence_after();
    {
      const uint64_t dK = smem_desc(sK, 16, 1024, kSwizzle128B);
#pragma unroll
      for (int k = 0; k < KD; ++k) {
        if constexpr (QIP)
          mma_ss(tmem + Cfg::TS, desc_at(dQ, kstep(k)), desc_at(dK, kstep(k)), idS, k > 0);
        else
          mma_ts(tmem + Cfg::TS, tmem + Cfg::TQ + k * 8, desc_at(dK, kstep(k)), idS, k > 0);
      }
      mma_commit(&bar[B_SCORES]);
    }
    mma_commit(&bar[B_KEMPTY0 + ks]);
    // num = Q''·S ; den = Q''·z (general: Q'·S, Q'·z, row-scaled by warps 4–7)
    if (!mbar_wait(&bar[B_SREADY], c & 1, st, ab)) break;
    if (c >= 1 && !mbar_wait(&bar[B_NUMEMPTY], (c - 1) & 1, st, ab)) break;
    tc_fence_after();
#pragma unroll
    for (int k = 0; k < KD; ++k) {
      if constexpr (QIP) {
        mma_ss(tmem + Cfg::TN, desc_at(dQ, kstep(k)), desc_at(dS, k * 2048), idN, k > 0);
        mma_ss(tmem + Cfg::TR, desc_at(dQ, kstep(k)), desc_at(dZ, k * 32), idR, k > 0);
      } else {
        mma_ts(tmem + Cfg::TN, tmem + Cfg::TQ + k * 8, desc_at(dS, k * 2048), idN, k > 0);
        mma_ts(tmem + Cfg::TR, tmem + Cfg::TQ + k * 8, desc_at(dZ, k * 32), idR, k > 0);
      }
    }
    mma_commit(&bar[B_SEMPTY]);
    // Q'' (its stage) or Q' (its TMEM columns) read by both of its products
    mma_commit(&bar[QIP ? B_QEMPTY0 + qs : B_QPEMPTY]);
    // num += P·V ; den += P·1
    if (!mbar_wait(&bar[B_PREADY], c & 1, st, ab)) break;
    if (!mbar_wait(&bar[B_VFULL0 + vs], (c / L::VST) & 1, st, ab)) break;
    tc_fence_after();
    const uint64_t dV = smem_desc(sV, kC * 128, 1024, kSwizzle128B);
#pragma unroll
    for (int k = 0; k < kC / 16; ++k) {
      mma_ts(tmem + Cfg::TN, tmem + Cfg::TS + k * 8, desc_at(dV, k * 2048), idN, 1);
      mma_ts(tmem + Cfg::TR, tmem + Cfg::TS + k * 8, ones, idR, 1);
    }
    mma_commit(&bar[B_NUMFULL]);
    mma_commit(&bar[B_VEMPTY0 + vs]);
  }
  // every issued MMA must finish before TMEM is released
  mma_commit(&bar[B_MMADONE]);
  mbar_wait_drain(&bar[B_MMADONE], 0);
}

template <int D, bool FULL, bool CEN>
__device__ __forceinline__ void role_mma_state(const Ctx& x) {
  using Cfg = TcCfg<D>;
  using L = Layout<D, FULL, CEN>;
  uint64_t* bar = x.bar;
  const uint32_t tmem = x.tmem;
  constexpr uint32_t idD = idesc_bf16_f32(128, D, true, true);       // ΔS = K''ᵀ V
  constexpr uint32_t idZ = idesc_bf16_f32(128, 16, true, false);     // Δz = K''ᵀ 1
  const uint32_t lbo_kp = (D == 128) ? kC * 128 : 0;                 // M blocks of K''ᵀ
  const uint64_t ones = smem_desc(x.sbase + Cfg::oONES, 0, 0, kSwizzleNone);
  int* st = x.status;
  volatile int* ab = x.abort_flag;
  for (int c = 0; c < x.nchunks; ++c) {
    const int ks = c % L::KST, vs = c % L::VST;
    const uint32_t sKP = x.sbase + L::kpp_off(ks);
    const uint32_t sV = x.sbase + L::v_off(vs);
    if (!mbar_wait(&bar[B_KREADY0 + ks], (c / L::KST) & 1, st, ab)) break;
    if (!mbar_wait(&bar[B_VFULL0 + vs], (c / L::VST) & 1, st, ab)) break;
    if (!mbar_wait(&bar[B_DSEMPTY], c & 1, st, ab)) break;   // state in TMEM read out
    tc_fence_after();
    const uint64_t dA = smem_desc(sKP, lbo_kp, 1024, kSwizzle128B);
    const uint64_t dV = smem_desc(sV, kC * 128, 1024, kSwizzle128B);
#pragma unroll
    for (int k = 0; k < kC / 16; ++k) {
      const uint64_t ad = desc_at(dA, k * 2048);
      mma_ss(tmem + Cfg::TD, ad, desc_at(dV, k * 2048), idD, 1);
      mma_ss(tmem + Cfg::TZ, ad, ones, idZ, 1);
    }
    mma_commit(&bar[B_DSFULL]);
    mma_commit(&bar[L::K_IN_PLACE ? B_KEMPTY0 + ks : B_KPEMPTY]);
    mma_commit(&bar[B_VEMPTY0 + vs]);
  }
  mma_commit(&bar[B_MMADONE]);
  mbar_wait_drain(&bar[B_MMADONE], 0);
}

// φ(Q) of chunk c for the 64 columns of half h of row r (TMEM lane r):
// Q'' = a_row·φ(q) (centered; Q' = φ(q) in the general folding).  QIP
// (per-head decay, centered): Q'' replaces the raw q tile in its stage,
// which the output MMAs release; otherwise Q'' (Q') goes to TMEM and the
// raw tile is released at once.  Signals the stage's q_ready (the scores MMA
// may start).  Returns false if a wait gave up.
template <int D, bool CEN, bool QIP>
__device__ __forceinline__ bool phi_q_half(const Ctx& x, int c, int h, int r, int lane,
                                           uint32_t lane_base, float a_row) {
  using Cfg = TcCfg<D>;
  using L = Layout<D, true, CEN>;
  uint64_t* bar = x.bar;
  int* st = x.status;
  volatile int* ab = x.abort_flag;
  const int qs = c % L::QST;
  if (!warp_wait(&bar[B_QFULL0 + qs], (c / L::QST) & 1, st, ab)) return false;
  const uint32_t a2 = splat_bf16x2(a_row);
  if constexpr (QIP) {
    // Q'' in place of the raw tile (the A operand of the scores and of Q''·S);
    // the output MMAs release the stage, so φ(Q) may run a stage ahead
    uint8_t* qw = x.sm + L::q_off(qs);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint4* p4 = reinterpret_cast<uint4*>(qw + sw_chunk(kC, r, h, j));
      uint4 u = *p4;
      u.x = mul_bf16x2(elu1_bf16x2(u.x), a2);
      u.y = mul_bf16x2(elu1_bf16x2(u.y), a2);
      u.z = mul_bf16x2(elu1_bf16x2(u.z), a2);
      u.w = mul_bf16x2(elu1_bf16x2(u.w), a2);
      *p4 = u;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_QREADY0 + qs]);
    return true;
  }
  if (c >= 1 && !warp_wait(&bar[B_QPEMPTY], (c - 1) & 1, st, ab)) return false;
  const uint8_t* qt = x.sm + L::q_off(qs);
  uint32_t packed[32];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint4 u = *reinterpret_cast<const uint4*>(qt + sw_chunk(kC, r, h, j));
    u.x = elu1_bf16x2(u.x); u.y = elu1_bf16x2(u.y);
    u.z = elu1_bf16x2(u.z); u.w = elu1_bf16x2(u.w);
    packed[j * 4 + 0] = CEN ? mul_bf16x2(u.x, a2) : u.x;
    packed[j * 4 + 1] = CEN ? mul_bf16x2(u.y, a2) : u.y;
    packed[j * 4 + 2] = CEN ? mul_bf16x2(u.z, a2) : u.z;
    packed[j * 4 + 3] = CEN ? mul_bf16x2(u.w, a2) : u.w;
  }
  tmem_st32(tmem_addr(x.tmem, lane_base, Cfg::TQ + h * 32), packed);
  tmem_st_wait();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    mbar_arrive(&bar[B_QREADY0 + qs]);
    mbar_arrive(&bar[B_QEMPTY0 + qs]);   // raw Q tile no longer needed
  }
  return true;
}

// φ(K) of chunk c for the 16-byte column chunks [j0, j1) of token row r →
// K'' = gs·φ(k) (rows ≥ cs get weight 0), written in place into the K tile
// except for the general full kernel, which keeps K' = m·φ(k) in place and
// writes K'' into its own tile.  φ is computed for every row so that no
// per-element branch splits the warp.  Signals k_ready for the warp.
// Per-token decay: general folding m = b_r, gs = b_r·2^{L_{cs−1} − L_r};
// centered folding gs = σ_c·b_r·2^{L_63 − L_r}; tt advances to this chunk.
template <int D, bool FULL, bool CEN, bool TOK>
__device__ __forceinline__ bool phi_k_chunk(const Ctx& x, int c, int r, int j0, int j1, int lane,
                                            float k_scale_cen, TokTrack& tt) {
  using L = Layout<D, FULL, CEN>;
  uint64_t* bar = x.bar;
  int* st = x.status;
  volatile int* ab = x.abort_flag;
  const int ks = c % L::KST;
  const int cs = (int)min((int64_t)kC, x.t_end - (x.t_begin + (int64_t)c * kC));
  TokChunk tk;
  if (TOK) tk = tok_chunk(x, c, lane, tt.pipe);
  if (!warp_wait(&bar[B_KFULL0 + ks], (c / L::KST) & 1, st, ab)) return false;
  if (!L::K_IN_PLACE && c >= 1 && !warp_wait(&bar[B_KPEMPTY], (c - 1) & 1, st, ab)) return false;
  const bool live = r < cs;
  uint32_t m2, g2;
  if (TOK) {
    const float lr = pick4(tk.L, r >> 5), br = pick4(tk.B, r >> 5);
    const float mid = __shfl_sync(0xffffffffu, tk.L[1], 31);   // L_63
    if (CEN) {
      if (c == 0) {
        tt.lrho = 0.f;
        tt.renorm_prev = false;
      } else {
        const float l = tt.lrho + (mid + tt.tot - tt.mid);
        tt.renorm_prev = l < -32.f;
        tt.alpha_prev = exp2f(l);
        tt.lrho = tt.renorm_prev ? 0.f : l;
      }
      m2 = 0u;
      g2 = splat_bf16x2(br * ex2_f32(mid - lr - tt.lrho));
    } else {
      m2 = splat_bf16x2(br);
      g2 = splat_bf16x2(br * ex2_f32(tk.tot - lr));
    }
    tt.lr = lr;
    tt.tot = tk.tot;
    tt.mid = mid;
  } else {
    m2 = live ? 0x3F803F80u : 0u;   // bf16 1.0 / 0.0 pairs
    g2 = live ? splat_bf16x2(CEN ? k_scale_cen * lazy_sigma(x, c) : x.pw[max(cs - 1 - r, 0)]) : 0u;
  }
  uint8_t* kt = x.sm + L::k_off(ks);
  uint8_t* kpp = x.sm + L::kpp_off(ks);
  // full launch: always 8 chunks (one 64-column half), fully unrolled so that
  // all eight loads are in flight together
  constexpr int UNROLL = FULL ? 8 : 4;
#pragma unroll UNROLL
  for (int jj = j0; jj < (FULL ? j0 + 8 : j1); ++jj) {
    const uint32_t off = sw_chunk(kC, r, jj >> 3, jj & 7);
    uint4 u = *reinterpret_cast<const uint4*>(kt + off);
    u.x = elu1_bf16x2(u.x); u.y = elu1_bf16x2(u.y);
    u.z = elu1_bf16x2(u.z); u.w = elu1_bf16x2(u.w);
    if (!L::K_IN_PLACE)
      *reinterpret_cast<uint4*>(kt + off) =
          make_uint4(mul_bf16x2(u.x, m2), mul_bf16x2(u.y, m2), mul_bf16x2(u.z, m2), mul_bf16x2(u.w, m2));
    *reinterpret_cast<uint4*>(kpp + off) =
        make_uint4(mul_bf16x2(u.x, g2), mul_bf16x2(u.y, g2), mul_bf16x2(u.z, g2), mul_bf16x2(u.w, g2));
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) mbar_arrive(&bar[B_KREADY0 + ks]);
  return true;
}

// φ(K) column ranges (16-byte chunks of a row, 8 per 64 columns) per
// warpgroup wg.  Full launch: the state warpgroups, one 64-column half each.
// State-only launch: the otherwise idle warpgroups take a share — d = 128:
// warps 4–7 chunks 0–7, the state warpgroups 8–11 and 12–15; d = 64: warps
// 4–7 chunks 0–2, warps 12–15 chunks 3–5, the state warps 6–7.
template <int D, bool FULL>
struct KSplit {
  __device__ static void range(int wg, int& j0, int& j1) {
    if (FULL) {
      j0 = (wg - 2) * 8; j1 = j0 + 8;
    } else if (D == 128) {
      j0 = wg == 1 ? 0 : (wg == 2 ? 8 : 12); j1 = wg == 1 ? 8 : (wg == 2 ? 12 : 16);
    } else {
      j0 = wg == 1 ? 0 : (wg == 3 ? 3 : 6); j1 = wg == 1 ? 3 : (wg == 3 ? 6 : 8);
    }
  }
  static constexpr int ARRIVALS = FULL ? 4 * TcCfg<D>::HALVES : 12;
};

// Warps 4–7: masked P and the epilogue.  Thread r owns token row / TMEM lane r.
template <int D, bool CEN, bool TOK>
__device__ __forceinline__ void role_rows(const Ctx& x, __nv_bfloat16* out, int64_t p_n, int warp,
                                          int lane) {
  using Cfg = TcCfg<D>;
  using L = Layout<D, true, CEN>;
  uint64_t* bar = x.bar;
  const uint32_t tmem = x.tmem;
  int* st = x.status;
  volatile int* ab = x.abort_flag;
  const int r = (warp - 4) * 32 + lane;
  const int wq = warp - 4;                        // lane quarter
  const uint32_t lane_base = (uint32_t)wq * 32;
  const float f_row = CEN ? 1.f : decay_pow(x.a, r + 1);   // general: a^{t+1}
  TokPipe pipe;
  pipe.c = -1;
  for (int c = 0; c < x.nchunks; ++c) {
    // ---- P: causal mask (and, general folding, the decay w·a^{t−s}; per-token
    // decay: 2^{L_t − L_s}, L_s of block b taken from lane s − 32b)
    TokChunk tk;
    if (TOK && !CEN) tk = tok_chunk(x, c, lane, pipe);
    if (!warp_wait(&bar[B_SCORES], c & 1, st, ab)) break;
    tc_fence_after();
    const float l_t = (TOK && !CEN) ? pick4(tk.L, wq) : 0.f;
    // 32-column blocks b: b > wq lies above the diagonal for the whole warp
    // (zeros, scores not read), b < wq below it (no mask), b == wq straddles it.
    // Loops over blocks and output columns stay rolled: the roles of this
    // kernel share each SM's instruction cache.
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
        if (CEN) {
          if (b < wq) {
#pragma unroll
            for (int j = 0; j < 32; j += 2)
              pk[j / 2] = pack_bf16x2(__uint_as_float(sc[j]), __uint_as_float(sc[j + 1]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const int s0 = b * 32 + j;
              const float p0 = (s0 <= r) ? __uint_as_float(sc[j]) : 0.f;
              const float p1 = (s0 + 1 <= r) ? __uint_as_float(sc[j + 1]) : 0.f;
              pk[j / 2] = pack_bf16x2(p0, p1);
            }
          }
        } else if (TOK) {
          const float l_b = pick4(tk.L, b);   // lane j: L of token 32b + j
          if (b < wq) {
            // below the diagonal: 2^{L_t − L_s} = 2^{L_t − L_e}·2^{L_e − L_s} with
            // e the block's last token; both factors are ≤ 1
            const float l_e = __shfl_sync(0xffffffffu, l_b, 31);
            const float rf = ex2_f32(l_t - l_e);
            const float cf = ex2_f32(l_e - l_b);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float c0 = __shfl_sync(0xffffffffu, cf, j);
              const float c1 = __shfl_sync(0xffffffffu, cf, j + 1);
              pk[j / 2] = pack_bf16x2(rf * c0 * __uint_as_float(sc[j]),
                                      rf * c1 * __uint_as_float(sc[j + 1]));
            }
          } else {
            // the diagonal block: one exponential per entry s ≤ t
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const int s0 = b * 32 + j;
              const float l0 = __shfl_sync(0xffffffffu, l_b, j);
              const float l1 = __shfl_sync(0xffffffffu, l_b, j + 1);
              const float p0 = (s0 <= r) ? ex2_f32(l_t - l0) * __uint_as_float(sc[j]) : 0.f;
              const float p1 = (s0 + 1 <= r) ? ex2_f32(l_t - l1) * __uint_as_float(sc[j + 1]) : 0.f;
              pk[j / 2] = pack_bf16x2(p0, p1);
            }
          }
        } else {
          const float* wp = x.pw + (r - b * 32);   // wp[-j] = w·a^{r-(32b+j)}
          if (b < wq) {
#pragma unroll
            for (int j = 0; j < 32; j += 2)
              pk[j / 2] = pack_bf16x2(wp[-j] * __uint_as_float(sc[j]),
                                      wp[-j - 1] * __uint_as_float(sc[j + 1]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const int s0 = b * 32 + j;
              const float p0 = (s0 <= r) ? wp[-j] * __uint_as_float(sc[j]) : 0.f;
              const float p1 = (s0 + 1 <= r) ? wp[-j - 1] * __uint_as_float(sc[j + 1]) : 0.f;
              pk[j / 2] = pack_bf16x2(p0, p1);
            }
          }
        }
      }
      tmem_st16(tmem_addr(tmem, lane_base, Cfg::TS + b * 16), pk);
    }
    if (!CEN) {
      // general folding: the row's Q'·S and Q'·z (complete once Q' is
      // released) are scaled by a^{t+1} (per-token decay: 2^{L_t}) before
      // P·V and P·1 accumulate onto them
      if (!warp_wait(&bar[B_QPEMPTY], c & 1, st, ab)) break;
      tc_fence_after();
      const float f = TOK ? exp2f(l_t) : f_row;
#pragma unroll 1
      for (int j0 = 0; j0 < D; j0 += 32) {
        uint32_t nv[32];
        tmem_ld32(tmem_addr(tmem, lane_base, Cfg::TN + j0), nv);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) nv[e] = __float_as_uint(f * __uint_as_float(nv[e]));
        tmem_st32(tmem_addr(tmem, lane_base, Cfg::TN + j0), nv);
      }
      uint32_t dz = 0;
      tmem_ld1(tmem_addr(tmem, lane_base, Cfg::TR), dz);
      tmem_ld_wait();
      dz = __float_as_uint(f * __uint_as_float(dz));
      asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};"
                   ::"r"(tmem_addr(tmem, lane_base, Cfg::TR)), "r"(dz) : "memory");
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_PREADY]);

    // ---- epilogue: o = num / den → bf16, row r written straight to global memory
    if (!warp_wait(&bar[B_NUMFULL], c & 1, st, ab)) break;
    tc_fence_after();
    uint32_t den = 0;
    tmem_ld1(tmem_addr(tmem, lane_base, Cfg::TR), den);
    tmem_ld_wait();
    const float inv_den = 1.f / __uint_as_float(den);
    const int64_t row = x.t_begin + (int64_t)c * kC + r;
    const bool valid = row < x.t_end && LA_DCHECK(x.status, x.t_end <= p_n, 12);
    uint4* orow = reinterpret_cast<uint4*>(out + (x.bh * p_n + (valid ? row : 0)) * D);
#pragma unroll 1
    for (int j0 = 0; j0 < D; j0 += 32) {
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
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_NUMEMPTY]);
  }
}


// Warps 8–15: φ(K), the fp32 state, and (D = 128) φ(Q).  Thread r: token
// row r for φ(K) and φ(Q) (the columns of its half), feature row r / TMEM
// lane r for the state (the 64 state columns of its half).
//
// The fp32 state lives in TMEM (columns TD, and TZ for z), scaled so that
// the state MMA accumulates onto it:
//   centered:  TMEM holds U_c with a^{64}·S_c = ρ_c·U_c, ρ_c = a^{128·(c mod R)}.
//              K''_c carries σ_c = 1/ρ_c, so the MMA leaves U_{c+1} = U_c + σ_c·ΔS''
//              and a^{64}S_{c+1} = a^{cs}(a^{64}S_c + ΔS'') = ρ_{c+1}U_{c+1}.
//              Every output term of chunk c — P·V, P·1 (through K'') and the
//              inter-chunk part — is then scaled by the same σ_c, which
//              cancels in num/den, so the operand tile is U_c itself.  Every
//              R chunks U is multiplied by a^{128R} (ρ back to 1); R keeps
//              σ ≤ 2^{32}.  a = 1: ρ = σ = 1 throughout.
//   general:   TMEM = a^{cs}·S_c, so after the MMA v = S_{c+1}; the tile gets
//              S_{c+1} and TMEM a^{cs'}·S_{c+1} for the next chunk (cs').
template <int D, bool FULL, bool CEN, bool TOK>
__device__ __forceinline__ void role_state(const Ctx& x, const TcParams& p, int warp, int lane) {
  using Cfg = TcCfg<D>;
  using L = Layout<D, FULL, CEN>;
  uint64_t* bar = x.bar;
  const uint32_t tmem = x.tmem;
  int* st = x.status;
  volatile int* ab = x.abort_flag;
  const int half = (warp - 8) >> 2;
  const int r = ((warp - 8) & 3) * 32 + lane;
  const uint32_t lane_base = (uint32_t)((warp - 8) & 3) * 32;
  const bool srow = r < D;
  const float a = x.a, w = x.w;
  const float k_scale_cen = CEN ? w * decay_pow_signed(a, 63 - r) : 0.f;
  const uint32_t td = tmem_addr(tmem, lane_base, Cfg::TD + half * 64);
  const uint32_t tz = tmem_addr(tmem, lane_base, Cfg::TZ);
  const uint32_t stile = x.sbase + Cfg::oS;
  auto chunk_len = [&](int c) {
    return (int)min((int64_t)kC, x.t_end - (x.t_begin + (int64_t)c * kC));
  };
  // final-state destination (state-only pass: the segment aggregate)
  float* out_S = nullptr;
  float* out_z = nullptr;
  if (!FULL) {
    const int64_t slot = x.bh * (p.nseg + p.init_slot) + x.g + p.init_slot;
    if (LA_DCHECK(x.status, x.bh < gridDim.x && x.g < p.nseg, 13)) {
      out_S = p.ws_state + slot * (int64_t)(D * D);
      out_z = p.ws_z + slot * (int64_t)D;
    }
  } else if (p.fin_state && x.g == p.nseg - 1) {
    out_S = p.fin_state + x.bh * (int64_t)(D * D);
    out_z = p.fin_z + x.bh * (int64_t)D;
  }

  // Writes one state value v (this thread's 64 columns, in 32-column steps
  // produced by `fetch`) as: tile ← α·v (full kernel), TMEM ← β·v (when
  // to_tmem), global ← γ·v (last chunk).  z is handled by the half-0 warps.
  // tile, to_tmem and to_global are warp-uniform.
  auto put_state = [&](auto fetch, float zv, float alpha, float beta, float gamma, bool tile,
                       bool to_tmem, bool to_global) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float v[32];
      fetch(hh, v);
      if (tile && srow) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = alpha * v[q * 8 + e];
          sts128(stile + sw_chunk(D, r, half, hh * 4 + q), pack8(f));
        }
      }
      if (to_global && srow) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(out_S + r * D + half * 64 + hh * 32 + j) =
              make_float4(gamma * v[j], gamma * v[j + 1], gamma * v[j + 2], gamma * v[j + 3]);
      }
      if (to_tmem) {
        uint32_t o[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(beta * v[j]);
        tmem_st32(td + hh * 32, o);
      }
    }
    if (half == 0) {
      if (to_tmem) {
        const uint32_t zo = __float_as_uint(beta * zv);
        asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tz), "r"(zo)
                     : "memory");
      }
      if (srow && tile) x.zb[r] = __float2bfloat16_rn(alpha * zv);
      if (srow && to_global) out_z[r] = gamma * zv;
    }
    if (to_tmem) tmem_st_wait();
    tc_fence_before();
    if (tile) fence_proxy_async_smem();
    __syncwarp();
  };

  int kj0, kj1;
  KSplit<D, FULL>::range((warp - 8) / 4 + 2, kj0, kj1);
  // per-token decay: the running state of the chunks φ(K) has seen, and the
  // running log2 decay of the segment (state-only launch)
  TokTrack tt;
  tok_track_init(tt);
  float seg_ld = 0.f;
  auto phi_k = [&](int c) {
    const bool r_ok = phi_k_chunk<D, FULL, CEN, TOK>(x, c, r, kj0, kj1, lane, k_scale_cen, tt);
    if (TOK) seg_ld += tt.tot;
    return r_ok;
  };

  // D = 128: these warps also compute φ(Q) for their half of the columns;
  // φ(Q) of the first chunk does not depend on the state, so it goes first.
  // Centered: Q'' = a^{t−63}φ(q) (per-token: 2^{L_t − L_63}, from the chunk
  // φ(K) last ran on); general: Q' unscaled.
  constexpr bool DO_Q = FULL && Cfg::HALVES == 2;
  const float a_row_head = CEN ? decay_pow_signed(a, r - 63) : 1.f;
  auto q_row_scale = [&]() { return (CEN && TOK) ? ex2_f32(tt.lr - tt.mid) : a_row_head; };
  bool ok = x.nchunks > 0 && phi_k(0);
  if (DO_Q && ok) ok = phi_q_half<D, CEN, CEN && !TOK>(x, 0, half, r, lane, lane_base, q_row_scale());

  // ---- initial state: S_in = a^{L·g}·S_0 + Σ_{j<g} a^{L·(g−1−j)}·A_j over
  // the caller's initial state S_0 (zero when none is given) and the
  // aggregates A_j of the earlier segments of this head (all of length L),
  // written by the state-only launch that precedes this one.  In Horner
  // form over the head's slots (S_0 first when given, then A_0, A_1, …):
  // S ← 0, then S ← a^L·S + slot_j for the nin slots before this segment
  if (ok) {
    const int nin = x.g + p.init_slot;
    const bool have_in = FULL && nin > 0 && LA_DCHECK(x.status, x.g < p.nseg, 14);
    if (have_in) grid_dependency_wait();
    // segment j carries the state through it with aL (per-token decay: its
    // own total 2^{ws_ld})
    const float aL = (have_in && !TOK) ? decay_pow(a, p.seg_len) : 0.f;
    const int64_t agg0 = x.bh * (p.nseg + p.init_slot);
    auto seg_fac = [&](int j) { return TOK ? exp2f(p.ws_ld[agg0 + j]) : aL; };
    float zin = 0.f;
    if (have_in && srow && half == 0)
      for (int j = 0; j < nin; ++j) zin = seg_fac(j) * zin + p.ws_z[(agg0 + j) * D + r];
    // centered: tile and TMEM hold a^{64}·S_in (per-token: 2^{L_63}·S_in);
    // general: tile S_in, TMEM a^{cs}·S_in (per-token: 2^{L_{cs−1}}·S_in)
    const float alpha0 = CEN ? (TOK ? exp2f(tt.mid) : decay_pow_signed(a, 64)) : 1.f;
    const float beta0 = CEN ? alpha0 : (TOK ? exp2f(tt.tot) : decay_pow(a, chunk_len(0)));
    put_state([&](int hh, float* v) {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0.f;
                if (have_in && srow) {
                  const float* src = p.ws_state + agg0 * (int64_t)(D * D) + r * D + half * 64 + hh * 32;
#pragma unroll 2
                  for (int j = 0; j < nin; ++j) {
                    const float4* s4 = reinterpret_cast<const float4*>(src + j * (int64_t)(D * D));
                    const float f = seg_fac(j);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                      const float4 t = s4[e];
                      v[4 * e] = f * v[4 * e] + t.x;
                      v[4 * e + 1] = f * v[4 * e + 1] + t.y;
                      v[4 * e + 2] = f * v[4 * e + 2] + t.z;
                      v[4 * e + 3] = f * v[4 * e + 3] + t.w;
                    }
                  }
                }
              },
              zin, alpha0, beta0, 1.f, FULL, true, false);
    if (lane == 0) {
      mbar_arrive(&bar[B_DSEMPTY]);                // TMEM state ready for the first MMA
      if (FULL) mbar_arrive(&bar[B_SREADY]);       // operand tile ready
    }
  }

  for (int c = 0; ok && c < x.nchunks; ++c) {
    if (c + 1 < x.nchunks && !phi_k(c + 1)) break;
    // centered, per-head decay: Q'' of the next chunk goes to its own stage,
    // so it needs no product of this chunk and is formed before the state
    // update (with a per-token decay Q'' stays in TMEM: measured faster)
    if (CEN && !TOK && DO_Q && c + 1 < x.nchunks &&
        !phi_q_half<D, CEN, CEN && !TOK>(x, c + 1, half, r, lane, lane_base, q_row_scale()))
      break;
    // ---- state update from the accumulated TMEM value v
    const int cs = chunk_len(c);
    const bool last = c + 1 == x.nchunks;
    if (!warp_wait(&bar[B_DSFULL], c & 1, st, ab)) break;
    if (FULL && !last && !warp_wait(&bar[B_SEMPTY], c & 1, st, ab)) break;   // tile free
    tc_fence_after();
    float alpha, beta, gamma;
    bool to_tmem;
    if (CEN && TOK) {
      // tt describes chunk c + 1 here (φ(K) of c + 1 ran above), or chunk c
      // when c is the last one
      const bool renorm = !last && tt.renorm_prev;
      alpha = beta = renorm ? tt.alpha_prev : 1.f;
      gamma = exp2f(tt.tot - tt.mid + tt.lrho);   // 2^{L_{cs−1} − L_63}·ρ_c (last chunk)
      to_tmem = renorm;
    } else if (CEN) {
      const bool renorm = !last && (c + 1) % x.R == 0;
      alpha = beta = renorm ? exp2f(128.f * (float)x.R * x.lg) : 1.f;
      gamma = exp2f(x.lg * (float)(cs - 64 + 128 * (c % x.R)));   // a^{cs−64}·ρ_c
      to_tmem = renorm;
    } else {
      alpha = 1.f;
      // tt holds chunk c + 1's totals here (φ(K) of c + 1 ran above)
      beta = last ? 1.f : (TOK ? exp2f(tt.tot) : decay_pow(a, chunk_len(c + 1)));
      gamma = 1.f;
      to_tmem = !last;
    }
    const bool tile = FULL && !last;
    const bool to_global = last && out_S != nullptr;
    if (tile || to_tmem || to_global) {
      uint32_t zraw = 0;
      uint32_t u[64];
      tmem_ld32(td, u);
      tmem_ld32(td + 32, u + 32);
      if (half == 0) tmem_ld1(tz, zraw);
      tmem_ld_wait();
      put_state([&](int hh, float* v) {
#pragma unroll
                  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(u[hh * 32 + j]);
                },
                __uint_as_float(zraw), alpha, beta, gamma, tile, to_tmem, to_global);
    } else {
      tc_fence_before();
      __syncwarp();
    }
    if (lane == 0) {
      mbar_arrive(&bar[B_DSEMPTY]);
      if (FULL && !last) mbar_arrive(&bar[B_SREADY]);
    }
    if (!(CEN && !TOK) && DO_Q && c + 1 < x.nchunks &&
        !phi_q_half<D, CEN, CEN && !TOK>(x, c + 1, half, r, lane, lane_base, q_row_scale()))
      break;
  }
  // state-only launch, per-token decay: the segment's total log2 decay
  if (TOK && !FULL && ok && warp == 8 && lane == 0) p.ws_ld[x.bh * p.nseg + x.g] = seg_ld;
}

template <int D, bool FULL, bool CEN, bool TOK>
__device__ __forceinline__ void run_roles(const Ctx& x, const TcParams& p, const CUtensorMap* mq,
                                          const CUtensorMap* mk, const CUtensorMap* mv, int warp,
                                          int lane) {
  using Cfg = TcCfg<D>;
  if (warp == 0) {
    if (lane == 0) role_producer<D, FULL, CEN>(x, mq, mk, mv);
  } else if (warp == 1) {
    if (FULL && lane == 0) role_mma_out<D, CEN, CEN && !TOK>(x);
  } else if (warp == 2) {
    if (lane == 0) role_mma_state<D, FULL, CEN>(x);
  } else if (warp >= 4 && warp < 8 && FULL) {
    role_rows<D, CEN, TOK>(x, p.out, p.n, warp, lane);
  } else if (warp >= 8 && warp < 8 + 4 * Cfg::HALVES) {
    role_state<D, FULL, CEN, TOK>(x, p, warp, lane);
  } else if (!FULL && warp >= 4) {
    // state-only launch: a share of φ(K) on the otherwise idle warpgroups
    const int r = (warp & 3) * 32 + lane;
    const float k_scale_cen = CEN ? x.w * decay_pow_signed(x.a, 63 - r) : 0.f;
    int j0, j1;
    KSplit<D, false>::range(warp / 4, j0, j1);
    TokTrack tt;
    tok_track_init(tt);
    for (int c = 0; c < x.nchunks; ++c)
      if (!phi_k_chunk<D, false, CEN, TOK>(x, c, r, j0, j1, lane, k_scale_cen, tt)) break;
  } else if (FULL && Cfg::HALVES == 1 && warp >= 12) {
    // D = 64: the fourth warpgroup computes φ(Q)
    const int r = (warp - 12) * 32 + lane;
    const float a_row = CEN ? decay_pow_signed(x.a, r - 63) : 1.f;   // general: Q' unscaled
    TokPipe pipe;
    pipe.c = -1;
    for (int c = 0; c < x.nchunks; ++c) {
      float ar = a_row;
      if (CEN && TOK) {   // 2^{L_r − L_63} of this chunk
        const TokChunk tk = tok_chunk(x, c, lane, pipe);
        ar = ex2_f32(pick4(tk.L, r >> 5) - __shfl_sync(0xffffffffu, tk.L[1], 31));
      }
      if (!phi_q_half<D, CEN, CEN && !TOK>(x, c, 0, r, lane, (uint32_t)(warp - 12) * 32, ar)) break;
    }
  }
}

// Per-token decay: whether every chunk of this CTA's segment fits the
// centered folding — each half of a chunk (tokens 1–63 and 64–127) spans at
// most 2^64 of decay, so that 2^{±(L_t − L_63)} and σ ≤ 2^32 stay far inside
// the bf16/fp32 range.  All threads take part (one warp per chunk, 64
// chunks' loads in flight per round); the answer is the CTA's.
__device__ bool tok_centered_ok(const Ctx& x, int warp, int lane) {
  bool bad = false;
  for (int c0 = warp; c0 < x.nchunks; c0 += 16 * 4) {
    float av[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + 16 * j;
      const int64_t t0 = x.t_begin + (int64_t)c * kC;
      const int cs = c < x.nchunks ? (int)min((int64_t)kC, x.t_end - t0) : 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int s = 32 * i + lane;
        av[j][i] = s < cs ? __ldg(x.ta + t0 + s) : 1.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float s1 = 0.f, s2 = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int s = 32 * i + lane;
        const float l = fmaxf(lg2_f32(av[j][i]), -64.f);
        if (s >= 64) s2 -= l;
        else if (s >= 1) s1 -= l;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      }
      if (s1 > 64.f || s2 > 64.f) bad = true;
    }
  }
  return __syncthreads_or(bad) == 0;
}

template <int D, bool FULL, bool TOK>
__global__ void __launch_bounds__(kThreadsTc, 1)
tc_forward_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const TcParams p) {
  using Cfg = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  Ctx x;
  x.sm = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  x.sbase = smem_u32(x.sm);
  x.bar = reinterpret_cast<uint64_t*>(x.sm + Cfg::oBAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(x.sm + Cfg::oMISC);
  x.abort_flag = reinterpret_cast<volatile int*>(x.sm + Cfg::oMISC + 4);
  x.zb = reinterpret_cast<__nv_bfloat16*>(x.sm + Cfg::oZB);
  x.pw = reinterpret_cast<float*>(x.sm + Cfg::oPW);
  x.status = p.status;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // the full launch that depends on this state-only one may start now
  if (!FULL) grid_dependents_launch();
  // grid (heads, segments): the CTAs of the first segments, which need no
  // aggregate, come first in launch order
  x.bh = blockIdx.x;
  x.g = blockIdx.y;
  x.t_begin = (int64_t)x.g * p.seg_len;
  x.t_end = min(p.n, x.t_begin + p.seg_len);
  x.nchunks = (int)((x.t_end - x.t_begin + kC - 1) / kC);
  x.a = p.decay ? p.decay[x.bh % p.H] : 1.f;
  x.w = new_token_weight(x.a);
  x.ta = TOK ? p.tok_decay + x.bh * p.n : nullptr;
  x.tl = TOK ? p.tok_L + x.bh * p.n : nullptr;
  x.tw = TOK ? p.tok_B + x.bh * p.n : nullptr;
  // the per-token decay takes the centered folding when the whole segment
  // fits it, the general folding otherwise
  const bool cen = TOK ? tok_centered_ok(x, warp, lane)
                       : ((x.a == 1.f) || (x.a >= kCenteredMinDecay));
  x.lg = (cen && x.a != 1.f) ? log2f(x.a) : 0.f;
  // largest R with 128·(R−1)·|log2 a| ≤ 32 − 128·|log2 a|, at least 1
  x.R = x.lg == 0.f ? (1 << 30) : max(1, (int)fminf(32.f / (128.f * -x.lg), 1e9f));

  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      if (i == B_PREADY || i == B_NUMEMPTY) cnt = 4;
      // released by both MMA chains: K'' (centered, full), V (full)
      if (i >= B_KEMPTY0 && i <= B_KEMPTY2 && FULL && cen) cnt = 2;
      if (((i >= B_VEMPTY0 && i <= B_VEMPTY2) || i == B_MMADONE) && FULL) cnt = 2;
      if (i == B_SREADY || i == B_DSEMPTY) cnt = 4 * Cfg::HALVES;
      if (i >= B_KREADY0 && i <= B_KREADY2) cnt = KSplit<D, FULL>::ARRIVALS;
      // φ(Q) warps: 8 for D = 128 (the state warps), 4 for D = 64
      if (i == B_QREADY0 || i == B_QREADY1) cnt = 4 * Cfg::HALVES;
      // Q stages are released by the φ(Q) warps (Q'' or Q' goes to TMEM),
      // or by the output MMAs that read Q'' in place (centered, per-head decay)
      if (i == B_QEMPTY0 || i == B_QEMPTY1) cnt = (FULL && cen && !TOK) ? 1 : 4 * Cfg::HALVES;
      mbar_init(&x.bar[i], cnt);
    }
    *x.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) {
    uint32_t* ones = reinterpret_cast<uint32_t*>(x.sm + Cfg::oONES);
    for (int i = lane; i < 32; i += 32) ones[i] = 0x3F803F80u;   // bf16 1.0 pairs
    // z operand and its read-past bytes (columns never read, kept finite)
    uint32_t* zw = reinterpret_cast<uint32_t*>(x.sm + Cfg::oZB);
    for (int i = lane; i < (2 * D + 128) / 4; i += 32) zw[i] = 0u;
    fence_proxy_async_smem();
  }
  if (warp == 3) {
    for (int k = lane; k < kC; k += 32) x.pw[k] = x.w * decay_pow(x.a, k);  // w·a^k
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    if (FULL) tma_prefetch_desc(&map_q);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  x.tmem = *tmem_slot;

  if (TOK && cen) run_roles<D, FULL, true, true>(x, p, &map_q, &map_k, &map_v, warp, lane);
  else if (TOK) run_roles<D, FULL, false, true>(x, p, &map_q, &map_k, &map_v, warp, lane);
  else if (cen) run_roles<D, FULL, true, false>(x, p, &map_q, &map_k, &map_v, warp, lane);
  else run_roles<D, FULL, false, false>(x, p, &map_q, &map_k, &map_v, warp, lane);

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(x.tmem, Cfg::TMEM_COLS);
  }
  // a dependent full launch completes only after the launch it depends on
  if (FULL) grid_dependency_wait();
}

// ------------------------------------------------------------------ host side

template <int D, bool TOK>
cudaError_t run_tc(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                   const SegmentPlan& plan) {
  using Cfg = TcCfg<D>;
  cudaError_t e;
  const int64_t BH = a.B * a.H;
  CUtensorMap mq, mk, mv;
  if ((e = tmap_rows(&mq, a.q, BH, a.n, D, kC)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mk, a.k, BH, a.n, D, kC)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mv, a.v, BH, a.n, D, kC)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_forward_kernel<D, true, TOK>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_forward_kernel<D, false, TOK>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  TcParams p{};
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.decay = a.decay;
  p.tok_decay = a.tok_decay;
  p.tok_weight = a.tok_weight;
  p.ws_ld = a.ws_ld;
  p.tok_L = a.ws_tok;
  p.tok_B = a.ws_tok ? a.ws_tok + (size_t)BH * a.n : nullptr;
  p.H = a.H;
  p.n = a.n;
  p.seg_len = plan.seg_len;
  p.nseg = plan.nseg;
  p.ws_state = ws_state;
  p.ws_z = ws_z;
  p.status = a.status;
  // the last segment's CTA of the full launch writes the final state
  p.fin_state = a.mu_out;
  p.fin_z = a.nu_out;
  p.init_slot = a.init_state ? 1 : 0;
  if (a.init_state) {
    // the initial state into slot 0 of every head's aggregates
    const size_t nslot = (size_t)plan.nseg + 1;
    e = cudaMemcpy2DAsync(ws_state, nslot * D * D * sizeof(float), a.init_state,
                          (size_t)D * D * sizeof(float), (size_t)D * D * sizeof(float), (size_t)BH,
                          cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpy2DAsync(ws_z, nslot * D * sizeof(float), a.init_z, (size_t)D * sizeof(float),
                          (size_t)D * sizeof(float), (size_t)BH, cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return e;
  }
  if (TOK) {
    // the per-token chunk prefixes and weights, read by every role that needs them
    if (!a.ws_tok) return cudaErrorInvalidValue;
    const int64_t nch = (a.n + kC - 1) / kC, chunks = BH * nch;
    tok_prefix_kernel<<<(unsigned)((chunks + 3) / 4), 128, 0, stream>>>(
        a.tok_decay, a.tok_weight, a.ws_tok, a.ws_tok + (size_t)BH * a.n, a.n, nch, chunks);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (plan.nseg > 1) {
    // aggregates of segments 0 … nseg−2 (nothing follows the last one)
    const dim3 grid_state((unsigned)BH, (unsigned)(plan.nseg - 1));
    tc_forward_kernel<D, false, TOK><<<grid_state, kThreadsTc, Cfg::SMEM_ALLOC, stream>>>(mq, mk, mv, p);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // The full launch overlaps the state-only one only when it directly
  // follows it: it reads q, k, v before waiting, so it must never overlap a
  // caller's kernel.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)BH, (unsigned)plan.nseg);
  cfg.blockDim = dim3(kThreadsTc);
  cfg.dynamicSmemBytes = Cfg::SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = plan.nseg > 1 ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, tc_forward_kernel<D, true, TOK>, mq, mk, mv, p);
  count_launches(1);
  return e;
}

// The aggregate of every segment (the state-only launch over all of them).
template <int D>
cudaError_t run_tc_state(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                         const SegmentPlan& plan) {
  using Cfg = TcCfg<D>;
  cudaError_t e;
  const int64_t BH = a.B * a.H;
  CUtensorMap mq, mk, mv;
  // the state-only launch never reads q; its map describes k
  if ((e = tmap_rows(&mq, a.k, BH, a.n, D, kC)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mk, a.k, BH, a.n, D, kC)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mv, a.v, BH, a.n, D, kC)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_forward_kernel<D, false, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  TcParams p{};
  p.decay = a.decay;
  p.H = a.H;
  p.n = a.n;
  p.seg_len = plan.seg_len;
  p.nseg = plan.nseg;
  p.ws_state = ws_state;
  p.ws_z = ws_z;
  p.status = a.status;
  const dim3 grid((unsigned)BH, (unsigned)plan.nseg);
  tc_forward_kernel<D, false, false><<<grid, kThreadsTc, Cfg::SMEM_ALLOC, stream>>>(mq, mk, mv, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

bool tc_forward_supported(const FwdArgs& a) {
  return a.bf16 && !a.performer && a.causal && (a.d == 64 || a.d == 128) && a.n >= kC;
}

int64_t tc_segment_granule() { return kC; }

cudaError_t tc_state_only(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                          const SegmentPlan& plan) {
  if (a.d == 128) return run_tc_state<128>(a, stream, ws_state, ws_z, plan);
  if (a.d == 64) return run_tc_state<64>(a, stream, ws_state, ws_z, plan);
  return cudaErrorInvalidValue;
}

cudaError_t tc_forward(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                       float* tot_state, float* tot_z, const SegmentPlan& plan) {
  (void)tot_state;   // causal only: the final state goes straight to a.mu_out
  (void)tot_z;
  if (a.tok_decay) {
    if (a.d == 128) return run_tc<128, true>(a, stream, ws_state, ws_z, plan);
    if (a.d == 64) return run_tc<64, true>(a, stream, ws_state, ws_z, plan);
    return cudaErrorInvalidValue;
  }
  if (a.d == 128) return run_tc<128, false>(a, stream, ws_state, ws_z, plan);
  if (a.d == 64) return run_tc<64, false>(a, stream, ws_state, ws_z, plan);
  return cudaErrorInvalidValue;
}

}  // namespace la
