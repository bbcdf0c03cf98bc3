// Tensor-core (tcgen05 + TMA + TMEM) chunked forward of causal kernelized
// linear attention, elu+1 feature map, bf16 inputs, fp32 state, d = d' ∈ {64, 128}.
//
// Method ("Efficient Transformers II" §2.2, eq (7)–(11) with the causal
// readout of eq (9)); per head, a chunk of C = 128 tokens (local t, s) with
// state (μ, ν) = (S, z) at its start:
//   scores  A = Q'K'ᵀ                                  (tcgen05, fp32 in TMEM)
//   P_ts    = w·a^{t−s}·A_ts for s ≤ t, else 0         (registers → bf16 in TMEM)
//   num     = P·V + Q''·S,  Q'' = diag(a^{t+1})·Q'     (two tcgen05 MMAs, one accumulator)
//   den     = Σ_s P_ts + q''_t·z                       (P·1 by tcgen05; q''·z in registers)
//   o_t     = num_t / den_t                            (epilogue, bf16, TMA store)
//   ΔS      = K''ᵀ·V, Δz = K''ᵀ·1, K'' = diag(w·a^{cs−1−s})·K'   (tcgen05)
//   S ← a^{cs}·S + ΔS,  z ← a^{cs}·z + Δz              (fp32 registers)
// i.e. eq (10)–(11) unrolled over the chunk; the intra-chunk part is the
// quadratic form of "Efficient Transformers I" eq (25)–(26) on the chunk.
//
// One CTA per (segment, head), 16 warps:
//   warp 0        TMA producer (Q, K, V tiles; one Q buffer, two K/V stages)
//   warp 1        tcgen05 MMA issuer, TMEM owner
//   warps 4–7     φ(Q) → Q' (smem) and Q'' (TMEM); masked decayed P; epilogue
//   warps 8–15    φ(K) → K' and K''; fp32 state S (64 columns per warpgroup)
// Long sequences are split into segments; a state-only launch of the same
// kernel computes each segment's decayed aggregate, segment_scan turns them
// into the states entering each segment, and the full launch produces o.
// Every wait is bounded in time: on expiry the kernel records LA_ERR_TIMEOUT
// in the device status word, stops issuing work, drains what it issued and
// frees its TMEM.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace la {
namespace {

using namespace tc;

constexpr int kC = 128;          // tokens per chunk (MMA M)
constexpr int kThreadsTc = 512;  // 16 warps

template <int D>
struct TcCfg {
  static constexpr int HALVES = D / 64;          // 64-column (128-byte) swizzle atoms per row
  static constexpr int TILE = kC * D * 2;        // one [128 × D] bf16 tile
  static constexpr int STILE = D * D * 2;        // state tile [D × D] bf16
  // shared memory (offsets from a 1024-aligned base)
  static constexpr int oQ = 0;
  static constexpr int oK0 = oQ + TILE;
  static constexpr int oK1 = oK0 + TILE;
  static constexpr int oKP = oK1 + TILE;
  static constexpr int oV0 = oKP + TILE;
  static constexpr int oV1 = oV0 + TILE;
  static constexpr int oS = oV1 + TILE;
  static constexpr int oONES = oS + STILE;       // 16×16 bf16 ones (512 B)
  // z [D] fp32.  One copy suffices: φ(Q) of chunk c reads z_c before it
  // signals q_ready(c), and z_{c+1} is written only after MMA3(c) — issued
  // after MMA1(c), which waits for q_ready(c) — has completed.
  static constexpr int oZ = oONES + 512;
  static constexpr int oPW = oZ + D * 4;         // w·a^k, k = 0..127 (+pad)
  static constexpr int oBAR = oPW + 132 * 4;     // mbarriers
  static constexpr int NBAR = 24;  // ≥ B_COUNT
  static constexpr int oMISC = oBAR + NBAR * 8;  // tmem slot, abort flag
  static constexpr int BYTES = oMISC + 16;
  // + alignment slack; at least half of the SM's shared memory so that one
  // CTA (which owns all 512 TMEM columns) runs per SM
  static constexpr int SMEM_ALLOC = (BYTES + 1024 > 118 * 1024) ? BYTES + 1024 : 118 * 1024;
  // tensor memory columns
  static constexpr uint32_t TS = 0;              // scores (fp32) / P (bf16 pairs, cols 0..63)
  static constexpr uint32_t TN = 128;            // numerator [128 × D]
  static constexpr uint32_t TD = TN + D;         // ΔS [D' × D] (lanes = feature)
  static constexpr uint32_t TZ = TD + D;         // Δz (16 columns, column 0 used)
  static constexpr uint32_t TR = TZ + 16;        // Σ_s P_ts (16 columns, column 0 used)
  static constexpr uint32_t TQ = (D == 128) ? 448 : 320;  // Q'' (bf16 pairs, D/2 columns)
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(TR + 16 <= TQ, "TMEM layout");
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

// barrier indices
enum {
  B_QFULL = 0, B_QEMPTY, B_KFULL0, B_KFULL1, B_KEMPTY0, B_KEMPTY1, B_VFULL0, B_VFULL1,
  B_VEMPTY0, B_VEMPTY1, B_QREADY, B_KREADY, B_KPEMPTY, B_SREADY, B_SEMPTY, B_SCORES,
  B_PREADY, B_NUMFULL, B_NUMEMPTY, B_DSFULL, B_DSEMPTY, B_QPEMPTY, B_MMADONE, B_STAGED, B_COUNT
};

struct TcParams {
  const float* decay;      // [H] or nullptr
  int64_t H, n, seg_len;
  int nseg;
  float* ws_state;         // [BH][nseg][D*D]
  float* ws_z;             // [BH][nseg][D]
  float* fin_state;        // final state (single-segment full launch) or nullptr
  float* fin_z;
  int* status;
};

// 16-byte chunk j (8 bf16, columns h*64 + 8j …) of row `row` in a swizzled tile.
__device__ __forceinline__ uint32_t sw_chunk(int rows, int row, int half, int j) {
  return (uint32_t)(half * rows * 128 + row * 128 + ((j ^ (row & 7)) << 4));
}

// φ(x) = elu(x) + 1 with the fast exponential: the result is rounded to bf16,
// so the intrinsic's few-ulp error is far below the output precision.
__device__ __forceinline__ float elu1_fast(float x) { return x > 0.f ? x + 1.f : __expf(x); }

// Every lane of the warp waits (bounded); the warp then agrees on the
// outcome so that control flow — and the .sync.aligned tcgen05 operations
// after it — stays warp-uniform even if the limit expires mid-wait.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* status,
                                          volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, status, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = bf16lo_to_f32(u.x); f[1] = bf16hi_to_f32(u.x);
  f[2] = bf16lo_to_f32(u.y); f[3] = bf16hi_to_f32(u.y);
  f[4] = bf16lo_to_f32(u.z); f[5] = bf16hi_to_f32(u.z);
  f[6] = bf16lo_to_f32(u.w); f[7] = bf16hi_to_f32(u.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

template <int D, bool FULL>
__global__ void __launch_bounds__(kThreadsTc, 1)
tc_forward_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                  const TcParams p) {
  using Cfg = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t sbase = smem_u32(sm);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Cfg::oBAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Cfg::oMISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Cfg::oMISC + 4);
  float* zbuf = reinterpret_cast<float*>(sm + Cfg::oZ);
  float* pw = reinterpret_cast<float*>(sm + Cfg::oPW);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int64_t t_begin = (int64_t)g * p.seg_len;
  const int64_t t_end = min(p.n, t_begin + p.seg_len);
  const int nchunks = (int)((t_end - t_begin + kC - 1) / kC);
  const float a = p.decay ? p.decay[bh % p.H] : 1.f;
  const float w = new_token_weight(a);

  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      if (i == B_QREADY || i == B_PREADY || i == B_NUMEMPTY || i == B_STAGED) cnt = 4;  // WG1 warps
      if (i == B_KREADY) cnt = 4 * Cfg::HALVES;                                // φK warps
      if (i == B_SREADY || i == B_DSEMPTY) cnt = 4 * Cfg::HALVES;              // state warps
      mbar_init(&bar[i], cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) {
    uint32_t* ones = reinterpret_cast<uint32_t*>(sm + Cfg::oONES);
    for (int i = lane; i < 128; i += 32) ones[i] = 0x3F803F80u;  // bf16 1.0 pairs
    fence_proxy_async_smem();
  }
  if (warp == 3) {
    for (int k = lane; k < kC; k += 32) pw[k] = w * decay_pow(a, k);  // w·a^k
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    if (FULL) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_o);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int* status = p.status;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued_q = -1, issued_kv = -1;
      for (int c = 0; c < nchunks && !*abort_flag; ++c) {
        const int st = c & 1;
        const int y = (int)(t_begin + (int64_t)c * kC);
        if (c >= 2 && !mbar_wait(&bar[B_KEMPTY0 + st], ((c - 2) >> 1) & 1, status, abort_flag)) break;
        mbar_arrive_expect_tx(&bar[B_KFULL0 + st], Cfg::TILE);
        for (int h = 0; h < Cfg::HALVES; ++h)
          tma_load_3d(sm + (st ? Cfg::oK1 : Cfg::oK0) + h * kC * 128, &map_k, &bar[B_KFULL0 + st],
                      h * 64, y, (int)bh);
        if (c >= 2 && !mbar_wait(&bar[B_VEMPTY0 + st], ((c - 2) >> 1) & 1, status, abort_flag)) break;
        mbar_arrive_expect_tx(&bar[B_VFULL0 + st], Cfg::TILE);
        for (int h = 0; h < Cfg::HALVES; ++h)
          tma_load_3d(sm + (st ? Cfg::oV1 : Cfg::oV0) + h * kC * 128, &map_v, &bar[B_VFULL0 + st],
                      h * 64, y, (int)bh);
        issued_kv = c;
        if (FULL) {
          if (c >= 1 && !mbar_wait(&bar[B_QEMPTY], (c - 1) & 1, status, abort_flag)) break;
          mbar_arrive_expect_tx(&bar[B_QFULL], Cfg::TILE);
          for (int h = 0; h < Cfg::HALVES; ++h)
            tma_load_3d(sm + Cfg::oQ + h * kC * 128, &map_q, &bar[B_QFULL], h * 64, y, (int)bh);
          issued_q = c;
        }
      }
      if (*abort_flag) {
        // drain the loads still in flight before the CTA's shared memory goes away
        for (int c = max(0, issued_kv - 1); c <= issued_kv; ++c) {
          mbar_wait_drain(&bar[B_KFULL0 + (c & 1)], (c >> 1) & 1);
          mbar_wait_drain(&bar[B_VFULL0 + (c & 1)], (c >> 1) & 1);
        }
        if (issued_q >= 0) mbar_wait_drain(&bar[B_QFULL], issued_q & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sQ = sbase + Cfg::oQ, sKP = sbase + Cfg::oKP, sS = sbase + Cfg::oS;
      const uint32_t sONES = sbase + Cfg::oONES;
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);   // scores
      constexpr uint32_t idD = idesc_bf16_f32(128, D, true, true);       // ΔS = K''ᵀ V
      constexpr uint32_t idZ = idesc_bf16_f32(128, 16, true, false);     // Δz = K''ᵀ 1
      constexpr uint32_t idN = idesc_bf16_f32(128, D, false, true);      // num (+)= A·{S,V}
      constexpr uint32_t idR = idesc_bf16_f32(128, 16, false, false);    // Σ_s P = P·1
      constexpr int KD = D / 16;                                         // K-steps over D'
      const uint32_t lbo_kp = (D == 128) ? 64 * 128 * 2 : 0;             // M blocks of K''ᵀ
      for (int c = 0; c < nchunks; ++c) {
        const int st = c & 1;
        const uint32_t sK = sbase + (st ? Cfg::oK1 : Cfg::oK0);
        const uint32_t sV = sbase + (st ? Cfg::oV1 : Cfg::oV0);
        if (FULL) {
          // scores = Q' K'ᵀ
          if (!mbar_wait(&bar[B_QREADY], c & 1, status, abort_flag)) break;
          if (!mbar_wait(&bar[B_KREADY], c & 1, status, abort_flag)) break;
          if (c >= 1 && !mbar_wait(&bar[B_NUMFULL], (c - 1) & 1, status, abort_flag)) break;
          tc_fence_after();
          for (int k = 0; k < KD; ++k) {
            const uint32_t off = (k >> 2) * (kC * 128) + (k & 3) * 32;
            mma_ss(tmem + Cfg::TS, smem_desc(sQ + off, 16, 1024, kSwizzle128B),
                   smem_desc(sK + off, 16, 1024, kSwizzle128B), idS, k > 0);
          }
          mma_commit(&bar[B_SCORES]);
          mma_commit(&bar[B_QEMPTY]);
        } else {
          if (!mbar_wait(&bar[B_KREADY], c & 1, status, abort_flag)) break;
        }
        mma_commit(&bar[B_KEMPTY0 + st]);
        // ΔS = K''ᵀ V ; Δz = K''ᵀ 1
        if (!mbar_wait(&bar[B_VFULL0 + st], (c >> 1) & 1, status, abort_flag)) break;
        if (c >= 1 && !mbar_wait(&bar[B_DSEMPTY], (c - 1) & 1, status, abort_flag)) break;
        tc_fence_after();
        for (int k = 0; k < kC / 16; ++k) {
          const uint64_t ad = smem_desc(sKP + k * 2048, lbo_kp, 1024, kSwizzle128B);
          mma_ss(tmem + Cfg::TD, ad, smem_desc(sV + k * 2048, kC * 128, 1024, kSwizzle128B), idD,
                 k > 0);
          mma_ss(tmem + Cfg::TZ, ad, smem_desc(sONES, 128, 256, kSwizzleNone), idZ, k > 0);
        }
        mma_commit(&bar[B_DSFULL]);
        mma_commit(&bar[B_KPEMPTY]);
        if (!FULL) {
          mma_commit(&bar[B_VEMPTY0 + st]);
          continue;
        }
        // num = Q'' S
        if (!mbar_wait(&bar[B_SREADY], c & 1, status, abort_flag)) break;
        if (c >= 1 && !mbar_wait(&bar[B_NUMEMPTY], (c - 1) & 1, status, abort_flag)) break;
        tc_fence_after();
        for (int k = 0; k < KD; ++k)
          mma_ts(tmem + Cfg::TN, tmem + Cfg::TQ + k * 8,
                 smem_desc(sS + k * 2048, D * 128, 1024, kSwizzle128B), idN, k > 0);
        mma_commit(&bar[B_SEMPTY]);
        mma_commit(&bar[B_QPEMPTY]);
        // num += P V
        if (!mbar_wait(&bar[B_PREADY], c & 1, status, abort_flag)) break;
        tc_fence_after();
        for (int k = 0; k < kC / 16; ++k) {
          mma_ts(tmem + Cfg::TN, tmem + Cfg::TS + k * 8,
                 smem_desc(sV + k * 2048, kC * 128, 1024, kSwizzle128B), idN, 1);
          mma_ts(tmem + Cfg::TR, tmem + Cfg::TS + k * 8, smem_desc(sONES, 128, 256, kSwizzleNone),
                 idR, k > 0);
        }
        mma_commit(&bar[B_NUMFULL]);
      }
      // every issued MMA must finish before TMEM is released
      mma_commit(&bar[B_MMADONE]);
      mbar_wait_drain(&bar[B_MMADONE], 0);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ WG1: φ(Q), P, epilogue
    if (FULL) {
      const int r = tid - 128;                       // row / TMEM lane
      const uint32_t lane_base = (uint32_t)(warp - 4) * 32;
      const float a_row = decay_pow(a, r + 1);       // a^{r+1}
      const float* pwr = pw;
      for (int c = 0; c < nchunks; ++c) {
        const int st = c & 1;
        // ---- φ(Q): Q' in place (smem), Q'' = a^{r+1} Q' into TMEM, q''·z
        if (!warp_wait(&bar[B_QFULL], c & 1, status, abort_flag)) break;
        if (c >= 1 && !warp_wait(&bar[B_QPEMPTY], (c - 1) & 1, status, abort_flag)) break;
        if (!warp_wait(&bar[B_SREADY], c & 1, status, abort_flag)) break;
        const float4* zc4 = reinterpret_cast<const float4*>(zbuf);
        float qz = 0.f;
        uint8_t* qtile = sm + Cfg::oQ;
#pragma unroll
        for (int h = 0; h < Cfg::HALVES; ++h) {
          uint32_t packed[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint4* ptr = reinterpret_cast<uint4*>(qtile + sw_chunk(kC, r, h, j));
            float f[8];
            unpack8(*ptr, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = elu1_fast(f[e]);
            *ptr = pack8(f);
            const float4 z0 = zc4[(h * 64 + j * 8) / 4];
            const float4 z1 = zc4[(h * 64 + j * 8) / 4 + 1];
            const float zz[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const uint32_t pr = pack_bf16x2(a_row * f[e], a_row * f[e + 1]);
              packed[j * 4 + e / 2] = pr;
              qz += bf16lo_to_f32(pr) * zz[e] + bf16hi_to_f32(pr) * zz[e + 1];
            }
          }
          tmem_st32(tmem_addr(tmem, lane_base, Cfg::TQ + h * 32), packed);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[B_QREADY]);

        // ---- P = mask ⊙ w a^{t−s} ⊙ scores  (bf16 into TMEM columns 0..63)
        if (!warp_wait(&bar[B_SCORES], c & 1, status, abort_flag)) break;
        tc_fence_after();
        // 32-column blocks b of row r (warp quarter wq = rows 32wq..32wq+31):
        // b > wq lies above the diagonal for the whole warp (zeros, scores not
        // read), b < wq below it (no mask), b == wq straddles it.
        const int wq = warp - 4;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t pk[16];
          if (b > wq) {
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[j] = 0u;
          } else {
            uint32_t sc[32];
            tmem_ld32(tmem_addr(tmem, lane_base, Cfg::TS + b * 32), sc);
            tmem_ld_wait();
            const float* wp = pwr + (r - b * 32);      // wp[-j] = w·a^{r-(32b+j)}
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
          tmem_st16(tmem_addr(tmem, lane_base, Cfg::TS + b * 16), pk);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[B_PREADY]);

        // ---- epilogue: o = num / den → bf16 → staging (V buffer) → TMA store
        if (!warp_wait(&bar[B_NUMFULL], c & 1, status, abort_flag)) break;
        tc_fence_after();
        uint32_t rs = 0;
        tmem_ld1(tmem_addr(tmem, lane_base, Cfg::TR), rs);
        tmem_ld_wait();
        const float inv_den = 1.f / (__uint_as_float(rs) + qz);
        uint8_t* stage = sm + (st ? Cfg::oV1 : Cfg::oV0);
#pragma unroll
        for (int j0 = 0; j0 < D; j0 += 32) {
          uint32_t nv[32];
          tmem_ld32(tmem_addr(tmem, lane_base, Cfg::TN + j0), nv);
          tmem_ld_wait();
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(nv[q8 * 8 + e]) * inv_den;
            const int col = j0 + q8 * 8;
            *reinterpret_cast<uint4*>(stage + sw_chunk(kC, r, col >> 6, (col & 63) >> 3)) = pack8(f);
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bar[B_NUMEMPTY]);
          mbar_arrive(&bar[B_STAGED]);
        }
        if (r == 0) {
          // all four warps staged their rows: store the tile, then release the buffer
          if (mbar_wait(&bar[B_STAGED], c & 1, status, abort_flag)) {
            const int y = (int)(t_begin + (int64_t)c * kC);
            for (int h = 0; h < Cfg::HALVES; ++h)
              tma_store_3d(&map_o, stage + h * kC * 128, h * 64, y, (int)bh);
            tma_store_commit();
            tma_store_wait_read0();
            mbar_arrive(&bar[B_VEMPTY0 + st]);
          }
        }
        __syncwarp();
      }
      if (r == 0) tma_store_wait0();
    }
  } else if (warp >= 8 && warp < 8 + 4 * Cfg::HALVES) {
    // ------------------------------------------------------------ WG2/WG3: φ(K), state
    const int half = (warp - 8) >> 2;              // which 64 state columns
    const int r = tid - 128 * (2 + half);          // token row for φK; feature row for S
    const uint32_t lane_base = (uint32_t)((warp - 8) & 3) * 32;
    float S[64];
    float zr = 0.f;
    const bool srow = r < D;                       // this thread owns state row r
    if (p.nseg > 1) {
      const float* src = p.ws_state + (bh * p.nseg + g) * (int64_t)(D * D);
#pragma unroll
      for (int j = 0; j < 64; ++j) S[j] = (FULL && srow) ? src[r * D + half * 64 + j] : 0.f;
      if (FULL && srow && half == 0) zr = p.ws_z[(bh * p.nseg + g) * (int64_t)D + r];
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) S[j] = 0.f;
    }
    uint8_t* stile = sm + Cfg::oS;
    auto write_state = [&]() {
      if (srow) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = S[j * 8 + e];
          *reinterpret_cast<uint4*>(stile + sw_chunk(D, r, half, j)) = pack8(f);
        }
        if (half == 0) zbuf[r] = zr;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_SREADY]);
    };
    write_state();
    for (int c = 0; c < nchunks; ++c) {
      const int st = c & 1;
      const int cs = (int)min((int64_t)kC, t_end - (t_begin + (int64_t)c * kC));
      // ---- φ(K): K' in place, K'' = w a^{cs−1−s} K' (rows ≥ cs zeroed)
      if (!warp_wait(&bar[B_KFULL0 + st], (c >> 1) & 1, status, abort_flag)) break;
      if (c >= 1 && !warp_wait(&bar[B_KPEMPTY], (c - 1) & 1, status, abort_flag)) break;
      {
        uint8_t* ktile = sm + (st ? Cfg::oK1 : Cfg::oK0);
        uint8_t* kp = sm + Cfg::oKP;
        const bool live = r < cs;
        const float gs = live ? pw[cs - 1 - r] : 0.f;   // w·a^{cs−1−s}
        const int h = half;                          // D = 128: each warpgroup one half
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t off = sw_chunk(kC, r, h, j);
          uint4* ptr = reinterpret_cast<uint4*>(ktile + off);
          float f[8], f2[8];
          unpack8(*ptr, f);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            f[e] = live ? elu1_fast(f[e]) : 0.f;
            f2[e] = gs * f[e];
          }
          if (FULL) *ptr = pack8(f);
          *reinterpret_cast<uint4*>(kp + off) = pack8(f2);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_KREADY]);
      // ---- state update: S ← a^{cs} S + ΔS, z ← a^{cs} z + Δz
      if (!warp_wait(&bar[B_DSFULL], c & 1, status, abort_flag)) break;
      tc_fence_after();
      const float acs = decay_pow(a, cs);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t dv[32];
        tmem_ld32(tmem_addr(tmem, lane_base, Cfg::TD + half * 64 + hh * 32), dv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) S[hh * 32 + j] = acs * S[hh * 32 + j] + __uint_as_float(dv[j]);
      }
      uint32_t dz = 0;
      tmem_ld1(tmem_addr(tmem, lane_base, Cfg::TZ), dz);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_DSEMPTY]);
      zr = acs * zr + __uint_as_float(dz);
      if (FULL) {
        if (!warp_wait(&bar[B_SEMPTY], c & 1, status, abort_flag)) break;
        write_state();
      }
    }
    // ---- hand the state on
    if (srow && !*abort_flag) {
      float* dS = nullptr;
      float* dz = nullptr;
      if (!FULL) {
        dS = p.ws_state + (bh * p.nseg + g) * (int64_t)(D * D);
        dz = p.ws_z + (bh * p.nseg + g) * (int64_t)D;
      } else if (p.fin_state) {
        dS = p.fin_state + bh * (int64_t)(D * D);
        dz = p.fin_z + bh * (int64_t)D;
      }
      if (dS) {
#pragma unroll
        for (int j = 0; j < 64; j += 4)
          *reinterpret_cast<float4*>(dS + r * D + half * 64 + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        if (half == 0) dz[r] = zr;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

// [BH, n, D] bf16 viewed as a 3-D tensor (D innermost), box 64 × 128 × 1 with
// the 128-byte swizzle.  Rows past n read as zero and are not stored.
cudaError_t make_map(CUtensorMap* m, const void* base, int64_t BH, int64_t n, int D) {
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)n, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)n * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kC, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                        box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t run_tc(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                   float* tot_state, float* tot_z, const SegmentPlan& plan) {
  using Cfg = TcCfg<D>;
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  const int64_t BH = a.B * a.H;
  CUtensorMap mq, mk, mv, mo;
  if ((e = make_map(&mq, a.q, BH, a.n, D)) != cudaSuccess) return e;
  if ((e = make_map(&mk, a.k, BH, a.n, D)) != cudaSuccess) return e;
  if ((e = make_map(&mv, a.v, BH, a.n, D)) != cudaSuccess) return e;
  if ((e = make_map(&mo, a.out, BH, a.n, D)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_forward_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_forward_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg::SMEM_ALLOC);
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
  const dim3 grid((unsigned)plan.nseg, (unsigned)BH);
  if (plan.nseg > 1) {
    tc_forward_kernel<D, false><<<grid, kThreadsTc, Cfg::SMEM_ALLOC, stream>>>(mq, mk, mv, mo, p);
    count_launches(1);
    e = segment_scan(ws_state, ws_z, tot_state, tot_z, BH, a.H, plan.nseg, plan.seg_len, a.n, D, D,
                     a.decay, stream);
    if (e != cudaSuccess) return e;
  } else {
    p.fin_state = a.mu_out;
    p.fin_z = a.nu_out;
  }
  tc_forward_kernel<D, true><<<grid, kThreadsTc, Cfg::SMEM_ALLOC, stream>>>(mq, mk, mv, mo, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

bool tc_forward_supported(const FwdArgs& a) {
  return a.bf16 && !a.performer && a.causal && (a.d == 64 || a.d == 128) && a.n >= kC;
}

int64_t tc_segment_granule() { return kC; }

cudaError_t tc_forward(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                       float* tot_state, float* tot_z, const SegmentPlan& plan) {
  if (a.d == 128) return run_tc<128>(a, stream, ws_state, ws_z, tot_state, tot_z, plan);
  if (a.d == 64) return run_tc<64>(a, stream, ws_state, ws_z, tot_state, tot_z, plan);
  return cudaErrorInvalidValue;
}

}  // namespace la
