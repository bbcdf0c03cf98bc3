// Tensor-core (tcgen05 + TMA + TMEM) backward of the causal forward, elu+1
// map, bf16 inputs, d = d' ∈ {64, 128}: the gradients of L = Σ_t g_t·o_t.
//
// Method ("Efficient Transformers II" §2.2, eq (7)–(11) with the causal
// readout of eq (9), differentiated).  Per head, chunks of C = 128 tokens
// (local t, s; cs valid), q' = φ(q), k' = φ(k), x_ts = q'_t·k'_s,
// W_ts = w·a^{t−s} (s ≤ t), and for every chunk c
//   S_c, z_c  the forward state entering the chunk (Σ_{s<t0} w·a^{t0−1−s} k'_sᵀv_s, …),
//   M_c, N_c  the adjoint after the chunk (Σ_{t>t1} a^{t−t1} q'_tᵀĝ_t, Σ a^{t−t1} ρ_t q'_t),
// with ĝ_t = g_t/den_t and ρ_t = −(g_t·o_t)/den_t:
//   ∂q'_t = Σ_{s≤t} W_ts(ĝ_t·v_s + ρ_t) k'_s + a^{t+1}(S_c ĝ_t + ρ_t z_c)
//   ∂v_s  = Σ_{t≥s} W_ts x_ts ĝ_t + w·a^{cs−1−s} k'_s M_c
//   ∂k'_s = Σ_{t≥s} W_ts(ĝ_t·v_s + ρ_t) q'_t + w·a^{cs−1−s}(M_c v_s + N_c)
// and ∂a = Σ_{s<t}(t−s)·w·a^{t−s−1}·x_ts(ĝ_t·v_s + ρ_t), counted chunk by chunk
// over the token boundaries inside the chunk: pairs inside it, pairs from
// before it into it (weight t − t0 + 1), pairs from it to after it (weight
// t1 − s), and pairs across it (weight cs, the term cs·a^{cs−1}(⟨S_c, M_c⟩ +
// ⟨z_c, N_c⟩)) — so no position-weighted state is needed.
//
// Passes (each CTA loops over a contiguous range of (head, chunk) items; 256
// threads, two per token row r = TMEM lane r, each on one half of the row's
// columns; one thread issues the MMAs and every product is waited for before
// the rows use it; each of the next item's loads is issued as soon as its
// region is consumed):
//   1. bt_state:  ΔS_c = K''ᵀV (K'' = w·a^{cs−1−s}φ(k)), Δz_c      → workspace
//   2. scan:      S_c = exclusive decayed prefix of ΔS, as the bf16 operand
//                 tile of pass 3 (z_c in fp32)                       (CUDA cores, float4)
//   3. bt_dq:     recompute o, den; ∂q; den, ρ; ΔM_c = Q''ᵀ∂o (Q'' = a^{t+1}φ(q)/den), ΔN_c
//   4. scan:      M_c = reverse exclusive decayed suffix of ΔM, as the bf16
//                 operand tile of pass 5; the ∂a share across each chunk
//   5. bt_dkdv:   ∂k, ∂v
//   6. ∂a:        sum of the per-chunk shares                       (CUDA cores)
// The products take the ∂o tile as loaded (exact bf16) and the rows apply
// 1/den in fp32, so ĝ is never rounded to bf16.  The [128 × D] tiles arrive by
// TMA (tensor maps over the [B·H, n, D] rows) and the operand tiles of S_c and
// M_c by bulk copies, on one barrier per item; ∂q, ∂k, ∂v, ΔS_c and ΔM_c leave
// by TMA stores from swizzled staging tiles.  Every wait is bounded in time;
// on expiry the kernel records LA_ERR_TIMEOUT in the device status word and
// stops.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

#include <cuda.h>

#include <algorithm>
#include <type_traits>

namespace la {
namespace {

using namespace tc;

constexpr int kCb = 128;          // tokens per chunk
constexpr int kThreadsB = 256;    // two threads per token row / TMEM lane (one per column half)

template <int D>
struct BtCfg {
  static constexpr int TILE = kCb * D * 2;      // [128 × D] bf16, 128-byte swizzle
  static constexpr int STILE = D * D * 2;       // [D' × D] bf16 state / adjoint tile
  static constexpr int oQ = 0;
  static constexpr int oK = oQ + TILE;
  static constexpr int oV = oK + TILE;
  static constexpr int oG = oV + TILE;
  static constexpr int oS = oG + TILE;
  // staging for the TMA stores, apart from the tiles (which the next item's
  // loads may already be filling): two fp32 [D × 32] boxes or one bf16
  // [128 × D] tile, with the 128-byte swizzle
  static constexpr int oST = oS + STILE;
  static constexpr int STG_TMA = TILE > 2 * D * 128 ? TILE : 2 * D * 128;
  static constexpr int oZ = oST + STG_TMA;       // fp32 [D]: z_c or N_c
  static constexpr int oRHO = oZ + D * 4;        // fp32 [128]
  static constexpr int oDEN = oRHO + kCb * 4;    // fp32 [128]
  static constexpr int oPW = oDEN + kCb * 4;     // fp32 a^k, k = 0..128
  static constexpr int oAW = oPW + 132 * 4;      // fp32 k·w·a^{k−1}, k = 0..128
  static constexpr int oRED = oAW + 132 * 4;     // fp32 [8] warp partials
  static constexpr int oXCH = oRED + 32;         // fp32 [2][128] row partials of the two column halves
  static constexpr int oBAR = oXCH + 2 * kCb * 4;   // mbarriers: TMA, MMA
  static constexpr int oMISC = oBAR + 16;        // TMEM slot, abort flag
  static constexpr int BYTES = oMISC + 16;
  // + alignment slack; at least half of the SM's shared memory, so that one
  // CTA (which holds all 512 TMEM columns) runs per SM
  static constexpr int SMEM_ALLOC = (BYTES + 1024 > 118 * 1024) ? BYTES + 1024 : 118 * 1024;
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
  static_assert((kThreadsB / (D / 8)) * D * 4 <= STILE, "column-sum scratch in the S tile");
  static_assert(oZ % 16 == 0, "bulk-copy destination alignment");
  static_assert(oST % 1024 == 0, "swizzled staging alignment");
  static constexpr uint32_t TMEM_COLS = 512;
};

struct BtParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* g;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* decay;   // [H] or nullptr
  int64_t H, n;
  int nch;              // chunks per head
  int64_t items;        // B·H·nch
  float* S;             // [BH][nch][D*D]: ΔS_c (S_c itself only as its bf16 tile)
  float* z;             // [BH][nch][D]
  float* M;             // [BH][nch][D*D]: ΔM_c (M_c itself only as its bf16 tile)
  float* N;             // [BH][nch][D]: ΔN_c, then N_c
  const __nv_bfloat16* St;   // [BH][nch] bf16 operand tiles of S_c
  const __nv_bfloat16* Mt;   // [BH][nch] bf16 operand tiles of M_c
  float* den;           // [BH][n]
  float* rho;           // [BH][n]
  float* dapart;        // [BH][da_parts]: the ∂q pass shares (one per chunk), the
                        // ∂k/∂v pass shares, then the reverse scan's warp shares
  int da_parts;
  bool want_da;
  int* status;
};

struct Bt {
  uint8_t* sm;
  uint32_t sbase;
  uint64_t* bar;         // [0] TMA, [1] MMA
  volatile int* abort_flag;
  uint32_t tmem;
  uint32_t tma_phase, mma_phase;
  bool tma_pending;      // a tile load was issued and not yet waited for
  int* status;
};

__device__ __forceinline__ void init_bt(Bt& x, uint8_t* smem_raw, int* status, int off_bar,
                                        int off_misc) {
  const uint32_t raw = smem_u32(smem_raw);
  x.sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  x.sbase = smem_u32(x.sm);
  x.bar = reinterpret_cast<uint64_t*>(x.sm + off_bar);
  x.abort_flag = reinterpret_cast<volatile int*>(x.sm + off_misc + 4);
  x.tma_phase = x.mma_phase = 0;
  x.tma_pending = false;
  x.status = status;
}

// All threads wait for the MMAs issued since the last wait; false on timeout.
// The outcome is made the same for the whole CTA, so that every thread leaves
// the item loop together (the loop body is full of CTA barriers).
__device__ __forceinline__ bool wait_mma(Bt& x) {
  const bool ok = warp_wait(&x.bar[1], x.mma_phase & 1, x.status, x.abort_flag);
  ++x.mma_phase;
  tc_fence_after();
  return __syncthreads_and(ok) != 0;
}

// Thread 0 commits the MMAs it issued to the MMA barrier.
__device__ __forceinline__ void commit_mma(Bt& x) {
  if (threadIdx.x == 0) mma_commit(&x.bar[1]);
}

// Hand-off from the rows (TMEM and shared-memory writes) to the MMA issuer.
__device__ __forceinline__ void rows_to_mma() {
  tmem_st_wait();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// Contiguous global → shared copy on the TMA barrier (both addresses 16-byte
// aligned, bytes a multiple of 16); the caller has added the bytes to the
// barrier's expected transaction count.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Thread 0 arms the TMA barrier with the byte count of one item's copies;
// the copies may be issued later, within the same barrier phase.
__device__ __forceinline__ void arm_tiles(Bt& x, uint32_t bytes) {
  if (threadIdx.x == 0) mbar_arrive_expect_tx(&x.bar[0], bytes);
  x.tma_pending = true;
}

// Thread 0 loads the [128 × D] rows t0.. of head bh into the tile at `off`.
template <int D>
__device__ __forceinline__ void tile_load(Bt& x, const CUtensorMap* map, int off, int t0, int bh) {
  if (threadIdx.x == 0)
    for (int h = 0; h < D / 64; ++h)
      tma_load_3d(x.sm + off + h * kCb * 128, map, &x.bar[0], h * 64, t0, bh);
}

// Thread 0 copies `bytes` contiguous bytes to shared memory at `off`.
__device__ __forceinline__ void bulk_to(Bt& x, int off, const void* src, uint32_t bytes) {
  if (threadIdx.x == 0) bulk_load(x.sm + off, src, bytes, &x.bar[0]);
}

// The CTA's items: a contiguous range, so that consecutive items mostly share
// a head (and its decay tables).
__device__ __forceinline__ void item_range(int64_t items, int64_t& ib, int64_t& ie) {
  const int64_t per = (items + gridDim.x - 1) / gridDim.x;
  ib = min(items, (int64_t)blockIdx.x * per);
  ie = min(items, ib + per);
}

__device__ __forceinline__ bool wait_tiles(Bt& x) {
  const bool ok = warp_wait(&x.bar[0], x.tma_phase & 1, x.status, x.abort_flag);
  const bool all = __syncthreads_and(ok) != 0;
  if (all) {
    ++x.tma_phase;
    x.tma_pending = false;
  }
  return all;
}

// Applies f to the 16-byte chunks (8 bf16) [c0, c0 + NC) of row r of a
// [128 × D] tile (128-byte swizzle), in place: the whole row (NC = D/8, c0 = 0)
// or one column half (NC = D/16, c0 = 0 or D/16).  Every chunk is loaded
// before anything is stored, so the loads are not held back behind the stores.
template <int D, int NC = D / 8, typename F>
__device__ __forceinline__ void row_map(uint8_t* tile, int r, int c0, F f) {
  uint4 u[NC];
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int c = c0 + i;
    u[i] = *reinterpret_cast<const uint4*>(tile + sw_chunk(kCb, r, c >> 3, c & 7));
  }
#pragma unroll
  for (int i = 0; i < NC; ++i) u[i] = f(u[i]);
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int c = c0 + i;
    *reinterpret_cast<uint4*>(tile + sw_chunk(kCb, r, c >> 3, c & 7)) = u[i];
  }
}

// Column half hp of row r of a [128 × D] tile.
template <int D, typename F>
__device__ __forceinline__ void half_row_map(uint8_t* tile, int r, int hp, F f) {
  row_map<D, D / 16>(tile, r, hp * (D / 16), f);
}

// φ = elu+1 in place on row r of a [128 × D] tile; rows ≥ cs become 0 (the
// tensor map reads zeros past n, and φ(0) = 1 must not enter the sums).
template <int D>
__device__ __forceinline__ void phi_row_inplace(uint8_t* tile, int r, bool live) {
  row_map<D>(tile, r, 0, [live](uint4 u) {
    if (!live) return make_uint4(0u, 0u, 0u, 0u);
    return make_uint4(elu1_bf16x2(u.x), elu1_bf16x2(u.y), elu1_bf16x2(u.z), elu1_bf16x2(u.w));
  });
}

// 8 bf16 → 8 floats
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  f[0] = bf16lo_to_f32(u.x); f[1] = bf16hi_to_f32(u.x);
  f[2] = bf16lo_to_f32(u.y); f[3] = bf16hi_to_f32(u.y);
  f[4] = bf16lo_to_f32(u.z); f[5] = bf16hi_to_f32(u.z);
  f[6] = bf16lo_to_f32(u.w); f[7] = bf16hi_to_f32(u.w);
}

// The fp32 [D' × D] accumulator in TMEM (lane = row, columns col0..col0+D)
// to matrix `item` of `map` (fp32 [D × D] matrices, boxes of 32 columns × D
// rows with the 128-byte swizzle): staged box by box in shared memory
// (`stage`, two boxes, 1024-byte aligned) and written by TMA stores, two
// boxes per round; the two threads of a row fill one box each.  Thread 0
// issues and commits the stores; before a round reuses the stage it waits
// for the previous round's reads.  Every thread of the CTA calls it (it
// holds CTA barriers); the caller waits for the last round's reads before
// the stage is written again.
template <int D>
__device__ __forceinline__ void store_tmem_matrix_tma(uint32_t tmem, uint32_t col0, uint8_t* stage,
                                                      const CUtensorMap* map, int64_t item) {
  constexpr int BOX = D * 128;                 // bytes of one [D × 32] fp32 box
  constexpr int NBOX = D / 32;
  const int r = threadIdx.x & (kCb - 1), part = threadIdx.x / kCb;
#pragma unroll 1
  for (int b0 = 0; b0 < NBOX; b0 += 2) {
    if (b0 > 0) {
      if (threadIdx.x == 0) tma_store_wait_read0();
      __syncthreads();
    }
    if (r < D) {
      uint32_t v[32];
      tmem_ld32(tmem_addr(tmem, (uint32_t)(r >> 5) * 32, col0 + (b0 + part) * 32), v);
      tmem_ld_wait();
      uint8_t* box = stage + part * BOX;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(box + sw_chunk(D, r, 0, j)) =
            make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      tma_store_3d(map, stage, b0 * 32, 0, (int)item);
      tma_store_3d(map, stage + BOX, (b0 + 1) * 32, 0, (int)item);
      tma_store_commit();
    }
  }
}

// Weighted column sums of a [128 × D] bf16 tile (rows = tokens, 128-byte
// swizzle): out[i] = Σ_s wt(s)·T[s][i].  Thread t sums the 8 columns of chunk
// t mod (D/8) over one group of rows, so its loads and adds are independent;
// the group partials meet in `scratch` (128·8 floats).  Every thread of the
// CTA calls it (it holds a CTA barrier).
template <int D, typename Wt>
__device__ __forceinline__ void tile_colsum(const uint8_t* tile, Wt wt, float* scratch,
                                            float* __restrict__ out) {
  constexpr int NCH = D / 8;                 // 16-byte chunks per row
  constexpr int NG = kThreadsB / NCH;        // row groups
  constexpr int RPG = kCb / NG;              // rows per group
  const int ch = threadIdx.x % NCH, grp = threadIdx.x / NCH;
  const int h = ch >> 3, j = ch & 7;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
  for (int i = 0; i < RPG; ++i) {
    const int s = grp * RPG + i;
    float f[8];
    unpack8(*reinterpret_cast<const uint4*>(tile + sw_chunk(kCb, s, h, j)), f);
    const float ws = wt(s);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += ws * f[e];
  }
  float4* sc = reinterpret_cast<float4*>(scratch + grp * D + ch * 8);
  sc[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  sc[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) s += scratch[g * D + threadIdx.x];
    out[threadIdx.x] = s;
  }
}

// Per-head tables a^k and k·w·a^{k−1} (k = 0..128).
__device__ __forceinline__ void head_tables(float a, float w, float* pw, float* aw) {
  for (int k = threadIdx.x; k <= kCb; k += kThreadsB) {
    pw[k] = decay_pow(a, k);
    aw[k] = k == 0 ? 0.f : (float)k * w * decay_pow(a, k - 1);
  }
}

// Sum over the CTA (valid in every thread).
__device__ __forceinline__ float cta_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < kThreadsB / 32; ++i) t += red[i];
  return t;
}

__device__ __forceinline__ void head_decay(const BtParams& p, int64_t bh, float& a, float& w) {
  a = p.decay ? p.decay[bh % p.H] : 1.f;
  w = new_token_weight(a);
}

template <int D>
struct BtSetup {
  using Cfg = BtCfg<D>;
  __device__ static void run(Bt& x) {
    if (threadIdx.x == 0) {
      mbar_init(&x.bar[0], 1);
      mbar_init(&x.bar[1], 1);
      *x.abort_flag = 0;
      fence_barrier_init();
    }
    if (threadIdx.x < 32) {
      tmem_alloc(reinterpret_cast<uint32_t*>(x.sm + Cfg::oMISC), Cfg::TMEM_COLS);
      tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    x.tmem = *reinterpret_cast<uint32_t*>(x.sm + Cfg::oMISC);
  }
  __device__ static void teardown(Bt& x) {
    // nothing issued may still run when TMEM and shared memory are released
    if (threadIdx.x == 0 && *x.abort_flag) {
      if (x.tma_pending) mbar_wait_drain(&x.bar[0], x.tma_phase & 1);
      mma_commit(&x.bar[1]);
      mbar_wait_drain(&x.bar[1], x.mma_phase & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
      tc_fence_after();
      tmem_dealloc(x.tmem, Cfg::TMEM_COLS);
    }
  }
};

// ------------------------------------------------------------------ pass 1

// ΔS_c = K''ᵀV with K'' = w·a^{cs−1−s}φ(k) (rows ≥ cs zero), Δz_c = Σ_s K''_s.
template <int D>
__global__ void __launch_bounds__(kThreadsB, 1)
bt_state_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                const __grid_constant__ CUtensorMap map_ds, const BtParams p) {
  using Cfg = BtCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  Bt x;
  init_bt(x, smem_raw, p.status, Cfg::oBAR, Cfg::oMISC);
  BtSetup<D>::run(x);
  float* pw = reinterpret_cast<float*>(x.sm + Cfg::oPW);
  float* aw = reinterpret_cast<float*>(x.sm + Cfg::oAW);
  const int r = threadIdx.x & (kCb - 1), hp = threadIdx.x / kCb;   // row, column half
  int64_t ib, ie;
  item_range(p.items, ib, ie);
  // the K and V tiles of item `it` (issued while the previous item finishes)
  auto issue = [&](int64_t it) {
    if (it >= ie || !LA_DCHECK(p.status, it < p.items, 21)) return;
    const int ibh = (int)(it / p.nch), it0 = (int)(it % p.nch) * kCb;
    arm_tiles(x, 2 * Cfg::TILE);
    tile_load<D>(x, &map_k, Cfg::oK, it0, ibh);
    tile_load<D>(x, &map_v, Cfg::oV, it0, ibh);
  };
  issue(ib);
  int64_t last_bh = -1;
  float a = 1.f, w = 1.f;   // the decay of head last_bh and its new-token weight
  for (int64_t item = ib; item < ie && !*x.abort_flag; ++item) {
    const int64_t bh = item / p.nch;
    const int c = (int)(item % p.nch);
    const int t0 = c * kCb;
    const int cs = (int)min((int64_t)kCb, p.n - t0);
    __syncthreads();   // the previous item's tables are no longer read
    if (bh != last_bh) {
      head_decay(p, bh, a, w);
      head_tables(a, w, pw, aw);
    }
    last_bh = bh;
    __syncthreads();
    if (!wait_tiles(x)) break;
    // K'' in place
    {
      uint8_t* kt = x.sm + Cfg::oK;
      const bool live = r < cs;
      const uint32_t g2 = live ? splat_bf16x2(w * pw[cs - 1 - r]) : 0u;
      half_row_map<D>(kt, r, hp, [g2](uint4 u) {
        return make_uint4(mul_bf16x2(elu1_bf16x2(u.x), g2), mul_bf16x2(elu1_bf16x2(u.y), g2),
                          mul_bf16x2(elu1_bf16x2(u.z), g2), mul_bf16x2(elu1_bf16x2(u.w), g2));
      });
    }
    rows_to_mma();
    if (threadIdx.x == 0) {
      const uint64_t dA = smem_desc(x.sbase + Cfg::oK, (D == 128) ? kCb * 128 : 0, 1024, kSwizzle128B);
      const uint64_t dB = smem_desc(x.sbase + Cfg::oV, kCb * 128, 1024, kSwizzle128B);
      constexpr uint32_t id = idesc_bf16_f32(128, D, true, true);
#pragma unroll
      for (int k = 0; k < kCb / 16; ++k)
        mma_ss(x.tmem, desc_at(dA, k * 2048), desc_at(dB, k * 2048), id, k > 0);
    }
    commit_mma(x);
    // Δz on the CUDA cores meanwhile (rows ≥ cs of K'' are zero)
    tile_colsum<D>(x.sm + Cfg::oK, [](int) { return 1.f; },
                   reinterpret_cast<float*>(x.sm + Cfg::oS), p.z + item * D);
    if (threadIdx.x == 0) tma_store_wait_read0();   // the previous item's ΔS left the stage
    if (!wait_mma(x)) break;
    issue(item + 1);   // K'' and V are consumed
    store_tmem_matrix_tma<D>(x.tmem, 0, x.sm + Cfg::oST, &map_ds, item);
    tc_fence_before();
  }
  if (threadIdx.x == 0) tma_store_wait0();   // ΔS is in global memory
  BtSetup<D>::teardown(x);
}

// ------------------------------------------------------------------ pass 3

template <int D>
__global__ void __launch_bounds__(kThreadsB, 1)
bt_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
             const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_g,
             const __grid_constant__ CUtensorMap map_dq, const __grid_constant__ CUtensorMap map_dm,
             const BtParams p) {
  using Cfg = BtCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  Bt x;
  init_bt(x, smem_raw, p.status, Cfg::oBAR, Cfg::oMISC);
  BtSetup<D>::run(x);
  float* zc = reinterpret_cast<float*>(x.sm + Cfg::oZ);
  float* srho = reinterpret_cast<float*>(x.sm + Cfg::oRHO);
  float* pw = reinterpret_cast<float*>(x.sm + Cfg::oPW);
  float* aw = reinterpret_cast<float*>(x.sm + Cfg::oAW);
  float* red = reinterpret_cast<float*>(x.sm + Cfg::oRED);
  float* xch = reinterpret_cast<float*>(x.sm + Cfg::oXCH);
  uint8_t* qt = x.sm + Cfg::oQ;
  uint8_t* gt = x.sm + Cfg::oG;
  // thread (r, hp): token row r = TMEM lane r, column half hp (the 32-column
  // blocks hp, hp + 2 of the [128 × 128] score tiles; columns [hp·D/2,
  // (hp + 1)·D/2) of the [128 × D] ones); row sums meet in xch
  const int r = threadIdx.x & (kCb - 1), hp = threadIdx.x / kCb, wq = r >> 5;
  const uint32_t lane_base = (uint32_t)wq * 32;
  constexpr int HB = D / 2;
  // TMEM columns: X [0,128) | P, later E (bf16) [128,192) | Y, later U, then ∂q'
  // [192, 192+D) | PV, later ĜVᵀ, then ΔM [192+D, 320+D)
  constexpr uint32_t RX = 0, RP = 128, RY = 192, RN = 192 + D;
  int64_t ib, ie;
  item_range(p.items, ib, ie);
  // the Q, K, V, ∂o tiles, the S_c operand tile and z_c of item `it`, issued
  // while the previous item finishes, each as soon as its region is free: V
  // (arming the barrier for all of them), then K, then the rest
  auto issue_v = [&](int64_t it) {
    if (it >= ie || !LA_DCHECK(p.status, it < p.items, 22)) return;
    arm_tiles(x, 4 * Cfg::TILE + Cfg::STILE + D * 4);
    tile_load<D>(x, &map_v, Cfg::oV, (int)(it % p.nch) * kCb, (int)(it / p.nch));
  };
  auto issue_k = [&](int64_t it) {
    if (it < ie) tile_load<D>(x, &map_k, Cfg::oK, (int)(it % p.nch) * kCb, (int)(it / p.nch));
  };
  auto issue_rest = [&](int64_t it) {
    if (it >= ie) return;
    const int ibh = (int)(it / p.nch), it0 = (int)(it % p.nch) * kCb;
    tile_load<D>(x, &map_q, Cfg::oQ, it0, ibh);
    tile_load<D>(x, &map_g, Cfg::oG, it0, ibh);
    bulk_to(x, Cfg::oS, p.St + it * (int64_t)(D * D), Cfg::STILE);
    bulk_to(x, Cfg::oZ, p.z + it * D, D * 4);
  };
  issue_v(ib);
  issue_k(ib);
  issue_rest(ib);
  int64_t last_bh = -1;
  float a = 1.f, w = 1.f;   // the decay of head last_bh and its new-token weight
  for (int64_t item = ib; item < ie && !*x.abort_flag; ++item) {
    const int64_t bh = item / p.nch;
    const int c = (int)(item % p.nch);
    const int t0 = c * kCb;
    const int cs = (int)min((int64_t)kCb, p.n - t0);
    const bool live = r < cs;
    __syncthreads();   // the previous item's tables are no longer read
    if (bh != last_bh) {
      head_decay(p, bh, a, w);
      head_tables(a, w, pw, aw);
    }
    last_bh = bh;
    __syncthreads();
    if (!wait_tiles(x)) break;
    phi_row_inplace<D>(x.sm + (hp ? Cfg::oK : Cfg::oQ), r, live);   // φ(Q) | φ(K)
    rows_to_mma();
    // X = Q'K'ᵀ, Y = Q'·S_c
    if (threadIdx.x == 0) {
      const uint64_t dQ = smem_desc(x.sbase + Cfg::oQ, 16, 1024, kSwizzle128B);
      const uint64_t dK = smem_desc(x.sbase + Cfg::oK, 16, 1024, kSwizzle128B);
      const uint64_t dS = smem_desc(x.sbase + Cfg::oS, D * 128, 1024, kSwizzle128B);
      constexpr uint32_t idX = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idY = idesc_bf16_f32(128, D, false, true);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * (kCb * 128) + (k & 3) * 32;
        mma_ss(x.tmem + RX, desc_at(dQ, off), desc_at(dK, off), idX, k > 0);
        mma_ss(x.tmem + RY, desc_at(dQ, off), desc_at(dS, k * 2048), idY, k > 0);
      }
    }
    commit_mma(x);
    // q'_r·z_c over the column half meanwhile
    float qz = 0.f;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      const int cc = hp * (D / 16) + i;   // 16-byte chunk of the row
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(qt + sw_chunk(kCb, r, cc >> 3, cc & 7)), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) qz += f[e] * zc[cc * 8 + e];
    }
    if (!wait_mma(x)) break;
    // ---- rows 1: P = W ⊙ X (bf16, for P·V), den
    float den = 0.f;
#pragma unroll 1
    for (int b = hp; b < 4; b += 2) {
      uint32_t pk[16];
      if (b > wq) {
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = 0u;
      } else {
        uint32_t sc[32];
        tmem_ld32(tmem_addr(x.tmem, lane_base, RX + b * 32), sc);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int s0 = b * 32 + j;
          const float p0 = (s0 <= r) ? w * pw[r - s0] * __uint_as_float(sc[j]) : 0.f;
          const float p1 = (s0 + 1 <= r) ? w * pw[r - s0 - 1] * __uint_as_float(sc[j + 1]) : 0.f;
          den += p0 + p1;
          pk[j / 2] = pack_bf16x2(p0, p1);
        }
      }
      tmem_st16(tmem_addr(x.tmem, lane_base, RP + b * 16), pk);
    }
    xch[hp * kCb + r] = den + pw[r + 1] * qz;
    rows_to_mma();
    den = xch[r] + xch[kCb + r];
    if (threadIdx.x == 0) {
      const uint64_t dV = smem_desc(x.sbase + Cfg::oV, kCb * 128, 1024, kSwizzle128B);
      constexpr uint32_t idN = idesc_bf16_f32(128, D, false, true);
#pragma unroll
      for (int k = 0; k < kCb / 16; ++k)
        mma_ts(x.tmem + RN, x.tmem + RP + k * 8, desc_at(dV, k * 2048), idN, k > 0);
    }
    commit_mma(x);
    if (!wait_mma(x)) break;
    // ---- rows 2: o = (P·V + a^{t+1} Y)/den, ρ.  The ∂o tile stays as it is
    // (exact bf16): the products below use it and the rows divide by den in
    // fp32, so that ĝ = ∂o/den is never rounded to bf16
    const float inv_den = live ? 1.f / den : 0.f;
    float go = 0.f;
#pragma unroll 1
    for (int j0 = hp * HB; j0 < (hp + 1) * HB; j0 += 32) {
      uint32_t nv[32], yv[32];
      tmem_ld32(tmem_addr(x.tmem, lane_base, RN + j0), nv);
      tmem_ld32(tmem_addr(x.tmem, lane_base, RY + j0), yv);
      tmem_ld_wait();
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        const int h = (j0 + q8 * 8) >> 6, j = ((j0 + q8 * 8) & 63) >> 3;
        float gf[8];
        unpack8(*reinterpret_cast<const uint4*>(gt + sw_chunk(kCb, r, h, j)), gf);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float o = (__uint_as_float(nv[q8 * 8 + e]) + pw[r + 1] * __uint_as_float(yv[q8 * 8 + e])) * inv_den;
          go += gf[e] * o;
        }
      }
    }
    xch[hp * kCb + r] = go;
    rows_to_mma();
    const float go_r = xch[r] + xch[kCb + r];
    const float rho = -go_r * inv_den;
    if (hp == 0) {
      srho[r] = live ? -go_r : 0.f;   // ρ_t·den_t, the ΔN weight of Q'' (which carries 1/den_t)
      if (live) {
        p.den[bh * p.n + t0 + r] = den;
        p.rho[bh * p.n + t0 + r] = rho;
      }
    }
    // ∂o·Vᵀ, ∂o·S_cᵀ (rows scaled by 1/den in rows 3)
    if (threadIdx.x == 0) {
      const uint64_t dG = smem_desc(x.sbase + Cfg::oG, 16, 1024, kSwizzle128B);
      const uint64_t dVk = smem_desc(x.sbase + Cfg::oV, 16, 1024, kSwizzle128B);
      const uint64_t dSk = smem_desc(x.sbase + Cfg::oS, 16, 1024, kSwizzle128B);
      constexpr uint32_t idGV = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idU = idesc_bf16_f32(128, D, false, false);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * (kCb * 128) + (k & 3) * 32;
        const uint32_t offS = (k >> 2) * (D * 128) + (k & 3) * 32;
        mma_ss(x.tmem + RN, desc_at(dG, off), desc_at(dVk, off), idGV, k > 0);
        mma_ss(x.tmem + RY, desc_at(dG, off), desc_at(dSk, offS), idU, k > 0);
      }
    }
    commit_mma(x);
    if (!wait_mma(x)) break;
    issue_v(item + 1);   // V is consumed
    // ---- rows 3: E = W ⊙ (ĜVᵀ + ρ) (bf16, for E·K'), ∂a shares; ∂q' starts
    // as a^{t+1}·u_t, u_t = S_c ĝ_t + ρ_t z_c (ĜVᵀ = ∂o·Vᵀ/den, S_c ĝ = S_c∂o/den)
    float da = 0.f;
#pragma unroll 1
    for (int b = hp; b < 4; b += 2) {
      uint32_t pk[16];
      if (b > wq) {
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = 0u;
      } else {
        uint32_t xv[32], gv[32];
        tmem_ld32(tmem_addr(x.tmem, lane_base, RX + b * 32), xv);
        tmem_ld32(tmem_addr(x.tmem, lane_base, RN + b * 32), gv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int s0 = b * 32 + j;
          float e2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int s = s0 + u;
            const float f = __uint_as_float(gv[j + u]) * inv_den + rho;
            e2[u] = (s <= r && live) ? w * pw[r - s] * f : 0.f;
            if (s < r && live) da += aw[r - s] * __uint_as_float(xv[j + u]) * f;
          }
          pk[j / 2] = pack_bf16x2(e2[0], e2[1]);
        }
      }
      tmem_st16(tmem_addr(x.tmem, lane_base, RP + b * 16), pk);
    }
    // ... and Q'' = a^{t+1}φ(q)/den in place (ΔM = Q''ᵀ∂o = Σ_t a^{t+1}q'_tᵀĝ_t),
    // keeping min(φ(q), 1) of this thread's columns (bf16 pairs) for ∂q
    float qu = 0.f;
    uint32_t qmask[HB / 2];
    const float q2s = pw[r + 1] * inv_den;
#pragma unroll
    for (int jj = 0; jj < HB / 32; ++jj) {
      const int j0 = hp * HB + jj * 32;
      uint32_t uv[32];
      tmem_ld32(tmem_addr(x.tmem, lane_base, RY + j0), uv);
      tmem_ld_wait();
      float qf[32];
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        const int h = (j0 + q8 * 8) >> 6, j = ((j0 + q8 * 8) & 63) >> 3;
        unpack8(*reinterpret_cast<const uint4*>(qt + sw_chunk(kCb, r, h, j)), qf + q8 * 8);
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float u = __uint_as_float(uv[e]) * inv_den + rho * zc[j0 + e];
        qu += qf[e] * u;
        uv[e] = __float_as_uint(pw[r + 1] * u);
      }
      tmem_st32(tmem_addr(x.tmem, lane_base, RY + j0), uv);
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        const int h = (j0 + q8 * 8) >> 6, j = ((j0 + q8 * 8) & 63) >> 3;
        float m[8], sc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          m[e] = fminf(qf[q8 * 8 + e], 1.f);
          sc[e] = q2s * qf[q8 * 8 + e];
        }
        const uint4 mk = pack8(m);
        qmask[jj * 16 + q8 * 4 + 0] = mk.x;
        qmask[jj * 16 + q8 * 4 + 1] = mk.y;
        qmask[jj * 16 + q8 * 4 + 2] = mk.z;
        qmask[jj * 16 + q8 * 4 + 3] = mk.w;
        *reinterpret_cast<uint4*>(qt + sw_chunk(kCb, r, h, j)) = pack8(sc);
      }
    }
    if (live) da += (float)(r + 1) * pw[r] * qu;
    rows_to_mma();
    // ∂q' += E·K'; ΔM = Q''ᵀ∂o (over the columns of ĜVᵀ, read by rows 3)
    if (threadIdx.x == 0) {
      const uint64_t dKm = smem_desc(x.sbase + Cfg::oK, kCb * 128, 1024, kSwizzle128B);
      constexpr uint32_t idN = idesc_bf16_f32(128, D, false, true);
#pragma unroll
      for (int k = 0; k < kCb / 16; ++k)
        mma_ts(x.tmem + RY, x.tmem + RP + k * 8, desc_at(dKm, k * 2048), idN, 1);
      const uint64_t dA = smem_desc(x.sbase + Cfg::oQ, (D == 128) ? kCb * 128 : 0, 1024, kSwizzle128B);
      const uint64_t dB = smem_desc(x.sbase + Cfg::oG, kCb * 128, 1024, kSwizzle128B);
      constexpr uint32_t id = idesc_bf16_f32(128, D, true, true);
#pragma unroll
      for (int k = 0; k < kCb / 16; ++k)
        mma_ss(x.tmem + RN, desc_at(dA, k * 2048), desc_at(dB, k * 2048), id, k > 0);
    }
    commit_mma(x);
    // ΔN_i = Σ_t a^{t+1} ρ_t q'_ti = Σ_t ρ_t den_t q''_ti meanwhile (rows ≥ cs
    // of Q'' and of the weights are zero; the S_c tile is free since ∂o·S_cᵀ
    // completed)
    tile_colsum<D>(qt, [&](int t) { return srho[t]; }, reinterpret_cast<float*>(x.sm + Cfg::oS),
                   p.N + item * D);
    if (threadIdx.x == 0) tma_store_wait_read0();   // the previous item's ΔM left the stage
    if (!wait_mma(x)) break;
    issue_k(item + 1);      // every tile, z_c and the scratch are consumed
    issue_rest(item + 1);
    // ---- rows 4: ∂q = ∂q' ⊙ min(φ(q), 1), staged as a swizzled tile and stored
    // by TMA (rows past n are not written)
    uint8_t* dq_stage = x.sm + Cfg::oST;
#pragma unroll
    for (int jj = 0; jj < HB / 32; ++jj) {
      const int j0 = hp * HB + jj * 32;
      uint32_t dv[32];
      tmem_ld32(tmem_addr(x.tmem, lane_base, RY + j0), dv);
      tmem_ld_wait();
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        const int h = (j0 + q8 * 8) >> 6, j = ((j0 + q8 * 8) & 63) >> 3;
        float f[8];
        unpack8(make_uint4(qmask[jj * 16 + q8 * 4 + 0], qmask[jj * 16 + q8 * 4 + 1],
                           qmask[jj * 16 + q8 * 4 + 2], qmask[jj * 16 + q8 * 4 + 3]),
                f);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] *= __uint_as_float(dv[q8 * 8 + e]);
        *reinterpret_cast<uint4*>(dq_stage + sw_chunk(kCb, r, h, j)) = pack8(f);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();   // ∂q is staged
    tc_fence_after();
    // stores start at a non-negative row of the tensor (rows past n are clipped)
    if (threadIdx.x == 0 && LA_DCHECK(p.status, t0 >= 0 && t0 < p.n && bh * p.nch < p.items, 24)) {
#pragma unroll
      for (int h = 0; h < D / 64; ++h) tma_store_3d(&map_dq, dq_stage + h * kCb * 128, h * 64, t0, (int)bh);
      tma_store_commit();
      tma_store_wait_read0();   // the stage is reused for ΔM
    }
    __syncthreads();
    store_tmem_matrix_tma<D>(x.tmem, RN, x.sm + Cfg::oST, &map_dm, item);
    tc_fence_before();
    if (p.want_da) {
      const float s = cta_sum(da, red);
      if (threadIdx.x == 0) p.dapart[bh * p.da_parts + c] = s;
    }
  }
  if (threadIdx.x == 0) tma_store_wait0();   // ∂q and ΔM are in global memory
  BtSetup<D>::teardown(x);
}

// ------------------------------------------------------------------ pass 5

template <int D>
__global__ void __launch_bounds__(kThreadsB, 1)
bt_dkdv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_g,
               const __grid_constant__ CUtensorMap map_dk, const __grid_constant__ CUtensorMap map_dv,
               const BtParams p) {
  using Cfg = BtCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  Bt x;
  init_bt(x, smem_raw, p.status, Cfg::oBAR, Cfg::oMISC);
  BtSetup<D>::run(x);
  float* nc = reinterpret_cast<float*>(x.sm + Cfg::oZ);
  float* srho = reinterpret_cast<float*>(x.sm + Cfg::oRHO);
  float* sinv = reinterpret_cast<float*>(x.sm + Cfg::oDEN);   // 1/den_t (0 past the chunk)
  float* pw = reinterpret_cast<float*>(x.sm + Cfg::oPW);
  float* aw = reinterpret_cast<float*>(x.sm + Cfg::oAW);
  float* red = reinterpret_cast<float*>(x.sm + Cfg::oRED);
  uint8_t* kt = x.sm + Cfg::oK;
  uint8_t* gt = x.sm + Cfg::oG;
  // thread (r, hp): row r = TMEM lane r, column half hp (as in the ∂q pass)
  const int r = threadIdx.x & (kCb - 1), hp = threadIdx.x / kCb, wq = r >> 5;
  const uint32_t lane_base = (uint32_t)wq * 32;
  constexpr int HB = D / 2;
  // TMEM columns: Xᵀ, later K'M [0,128) | Pᵀ [128,192) | Eᵀ [192,256) (both
  // later V·Mᵀ [128, 128+D)) | ∂v [256, 256+D) | V∂oᵀ, later ∂k' [384, 512)
  constexpr uint32_t RX = 0, RP = 128, RE = 192, RF = 128, RV = 256, RK = 384;
  int64_t ib, ie;
  item_range(p.items, ib, ie);
  // item `it`'s inputs, issued while the previous item finishes: first the
  // Q, V, ∂o tiles and the M_c operand tile, then (once the K tile and N_c
  // have been read) the K tile and N_c; ρ and den of its rows into registers
  auto issue_a = [&](int64_t it) {
    if (it >= ie || !LA_DCHECK(p.status, it < p.items, 23)) return;
    const int ibh = (int)(it / p.nch), it0 = (int)(it % p.nch) * kCb;
    arm_tiles(x, 4 * Cfg::TILE + Cfg::STILE + D * 4);
    tile_load<D>(x, &map_q, Cfg::oQ, it0, ibh);
    tile_load<D>(x, &map_v, Cfg::oV, it0, ibh);
    tile_load<D>(x, &map_g, Cfg::oG, it0, ibh);
    bulk_to(x, Cfg::oS, p.Mt + it * (int64_t)(D * D), Cfg::STILE);
  };
  auto issue_b = [&](int64_t it) {
    if (it >= ie) return;
    const int ibh = (int)(it / p.nch), it0 = (int)(it % p.nch) * kCb;
    tile_load<D>(x, &map_k, Cfg::oK, it0, ibh);
    bulk_to(x, Cfg::oZ, p.N + it * D, D * 4);
  };
  float rho_n = 0.f, den_n = 1.f;
  auto rows_of = [&](int64_t it) {
    if (it >= ie) return;
    const int64_t ibh = it / p.nch, it0 = (it % p.nch) * kCb;
    const bool l = r < min((int64_t)kCb, p.n - it0);
    rho_n = l ? p.rho[ibh * p.n + it0 + r] : 0.f;
    den_n = l ? p.den[ibh * p.n + it0 + r] : 1.f;
  };
  issue_a(ib);
  issue_b(ib);
  rows_of(ib);
  int64_t last_bh = -1;
  float a = 1.f, w = 1.f;   // the decay of head last_bh and its new-token weight
  for (int64_t item = ib; item < ie && !*x.abort_flag; ++item) {
    const int64_t bh = item / p.nch;
    const int c = (int)(item % p.nch);
    const int t0 = c * kCb;
    const int cs = (int)min((int64_t)kCb, p.n - t0);
    const bool live = r < cs;
    __syncthreads();   // the previous item's tables are no longer read
    // (the share of the pairs across the chunk comes from the reverse scan)
    float da = 0.f;
    if (hp == 0) {
      srho[r] = rho_n;
      sinv[r] = live ? 1.f / den_n : 0.f;
    }
    if (bh != last_bh) {
      head_decay(p, bh, a, w);
      head_tables(a, w, pw, aw);
    }
    last_bh = bh;
    __syncthreads();
    if (!wait_tiles(x)) break;
    // φ(Q) | φ(K); the ∂o tile stays as it is (exact bf16): the products use
    // it and the rows carry 1/den_t, so that ĝ = ∂o/den is never rounded
    phi_row_inplace<D>(hp ? kt : x.sm + Cfg::oQ, r, live);
    rows_to_mma();
    // Xᵀ = K'Q'ᵀ, V∂oᵀ (column t of it is den_t·(ĜVᵀ)ᵀ)
    if (threadIdx.x == 0) {
      const uint64_t dQ = smem_desc(x.sbase + Cfg::oQ, 16, 1024, kSwizzle128B);
      const uint64_t dK = smem_desc(x.sbase + Cfg::oK, 16, 1024, kSwizzle128B);
      const uint64_t dV = smem_desc(x.sbase + Cfg::oV, 16, 1024, kSwizzle128B);
      const uint64_t dG = smem_desc(x.sbase + Cfg::oG, 16, 1024, kSwizzle128B);
      constexpr uint32_t id = idesc_bf16_f32(128, 128, false, false);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * (kCb * 128) + (k & 3) * 32;
        mma_ss(x.tmem + RX, desc_at(dK, off), desc_at(dQ, off), id, k > 0);
        mma_ss(x.tmem + RK, desc_at(dV, off), desc_at(dG, off), id, k > 0);
      }
    }
    commit_mma(x);
    if (!wait_mma(x)) break;
    // ---- rows 1 (thread s = r): Pᵀ_st = W_ts x_ts/den_t (so that Pᵀ∂o = PᵀĜ),
    // Eᵀ_st = W_ts(ĝ_t·v_s + ρ_t), ĝ_t·v_s = (V∂oᵀ)_st/den_t, t ≥ s
#pragma unroll 1
    for (int b = hp; b < 4; b += 2) {
      uint32_t pk[16], ek[16];
      if (b < wq) {   // every t of the block is before every s of the warp
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = ek[j] = 0u;
      } else {
        uint32_t xv[32], gv[32];
        tmem_ld32(tmem_addr(x.tmem, lane_base, RX + b * 32), xv);
        tmem_ld32(tmem_addr(x.tmem, lane_base, RK + b * 32), gv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float p2[2], e2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int t = b * 32 + j + u;
            const bool on = t >= r && t < cs;
            const float wts = on ? w * pw[t - r] : 0.f;
            p2[u] = wts * sinv[t] * __uint_as_float(xv[j + u]);
            e2[u] = wts * (__uint_as_float(gv[j + u]) * sinv[t] + srho[t]);
          }
          pk[j / 2] = pack_bf16x2(p2[0], p2[1]);
          ek[j / 2] = pack_bf16x2(e2[0], e2[1]);
        }
      }
      tmem_st16(tmem_addr(x.tmem, lane_base, RP + b * 16), pk);
      tmem_st16(tmem_addr(x.tmem, lane_base, RE + b * 16), ek);
    }
    rows_to_mma();
    // ∂v = Pᵀ∂o (= PᵀĜ), ∂k' = EᵀQ'
    if (threadIdx.x == 0) {
      const uint64_t dGm = smem_desc(x.sbase + Cfg::oG, kCb * 128, 1024, kSwizzle128B);
      const uint64_t dQm = smem_desc(x.sbase + Cfg::oQ, kCb * 128, 1024, kSwizzle128B);
      constexpr uint32_t idN = idesc_bf16_f32(128, D, false, true);
#pragma unroll
      for (int k = 0; k < kCb / 16; ++k) {
        mma_ts(x.tmem + RV, x.tmem + RP + k * 8, desc_at(dGm, k * 2048), idN, k > 0);
        mma_ts(x.tmem + RK, x.tmem + RE + k * 8, desc_at(dQm, k * 2048), idN, k > 0);
      }
    }
    commit_mma(x);
    if (!wait_mma(x)) break;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // K'·M_c, V·M_cᵀ (into the columns of Xᵀ, Pᵀ and Eᵀ, all consumed)
    if (threadIdx.x == 0) {
      const uint64_t dK = smem_desc(x.sbase + Cfg::oK, 16, 1024, kSwizzle128B);
      const uint64_t dV = smem_desc(x.sbase + Cfg::oV, 16, 1024, kSwizzle128B);
      const uint64_t dMm = smem_desc(x.sbase + Cfg::oS, D * 128, 1024, kSwizzle128B);
      const uint64_t dMk = smem_desc(x.sbase + Cfg::oS, 16, 1024, kSwizzle128B);
      constexpr uint32_t idMN = idesc_bf16_f32(128, D, false, true);
      constexpr uint32_t idKK = idesc_bf16_f32(128, D, false, false);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * (kCb * 128) + (k & 3) * 32;
        const uint32_t offS = (k >> 2) * (D * 128) + (k & 3) * 32;
        mma_ss(x.tmem + RX, desc_at(dK, off), desc_at(dMm, k * 2048), idMN, k > 0);
        mma_ss(x.tmem + RF, desc_at(dV, off), desc_at(dMk, offS), idKK, k > 0);
      }
    }
    commit_mma(x);
    if (threadIdx.x == 0) tma_store_wait_read0();   // the previous item's ∂v left the stage
    if (!wait_mma(x)) break;
    issue_a(item + 1);   // Q, V, ∂o and M_c are consumed
    rows_of(item + 1);
    // ---- rows 2: ∂k'_s = (EᵀQ')_s + w·a^{cs−1−s}((VMᵀ)_s + N); ∂a share
    // (t1 − s)·w·a^{t1−s−1}·k'_s·((VMᵀ)_s + N); then ∂v_s = (PᵀĜ)_s +
    // w·a^{cs−1−s}(K'M)_s.  ∂k goes first: it is the last reader of the K tile
    // and N_c, whose next loads then start.  The TMEM loads are warp-collective,
    // so every row takes part.  ∂k, then ∂v, are staged as swizzled tiles and
    // stored by TMA (rows past n are not written).
    uint8_t* stage = x.sm + Cfg::oST;
    const float fut = live ? w * pw[cs - 1 - r] : 0.f;
    {
      float kfut = 0.f;
#pragma unroll 1
      for (int j0 = hp * HB; j0 < (hp + 1) * HB; j0 += 32) {
        uint32_t va[32], vb[32];
        tmem_ld32(tmem_addr(x.tmem, lane_base, RK + j0), va);
        tmem_ld32(tmem_addr(x.tmem, lane_base, RF + j0), vb);
        tmem_ld_wait();
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          const int h = (j0 + q8 * 8) >> 6, j = ((j0 + q8 * 8) & 63) >> 3;
          float kf[8], f[8];
          unpack8(*reinterpret_cast<const uint4*>(kt + sw_chunk(kCb, r, h, j)), kf);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float m = __uint_as_float(vb[q8 * 8 + e]) + nc[j0 + q8 * 8 + e];
            kfut += kf[e] * m;
            f[e] = (__uint_as_float(va[q8 * 8 + e]) + fut * m) * fminf(kf[e], 1.f);
          }
          *reinterpret_cast<uint4*>(stage + sw_chunk(kCb, r, h, j)) = pack8(f);
        }
      }
      if (live) da += aw[cs - 1 - r] * kfut;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    issue_b(item + 1);   // the K tile and N_c are consumed
    if (threadIdx.x == 0 && LA_DCHECK(p.status, t0 >= 0 && t0 < p.n && bh * p.nch < p.items, 25)) {
#pragma unroll
      for (int h = 0; h < D / 64; ++h) tma_store_3d(&map_dk, stage + h * kCb * 128, h * 64, t0, (int)bh);
      tma_store_commit();
      tma_store_wait_read0();   // the stage is reused for ∂v
    }
    __syncthreads();
#pragma unroll 1
    for (int j0 = hp * HB; j0 < (hp + 1) * HB; j0 += 32) {
      uint32_t va[32], vb[32];
      tmem_ld32(tmem_addr(x.tmem, lane_base, RV + j0), va);
      tmem_ld32(tmem_addr(x.tmem, lane_base, RX + j0), vb);
      tmem_ld_wait();
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        const int h = (j0 + q8 * 8) >> 6, j = ((j0 + q8 * 8) & 63) >> 3;
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          f[e] = __uint_as_float(va[q8 * 8 + e]) + fut * __uint_as_float(vb[q8 * 8 + e]);
        *reinterpret_cast<uint4*>(stage + sw_chunk(kCb, r, h, j)) = pack8(f);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && LA_DCHECK(p.status, t0 >= 0 && t0 < p.n && bh * p.nch < p.items, 26)) {
#pragma unroll
      for (int h = 0; h < D / 64; ++h) tma_store_3d(&map_dv, stage + h * kCb * 128, h * 64, t0, (int)bh);
      tma_store_commit();
    }
    if (p.want_da) {
      const float s = cta_sum(da, red);
      if (threadIdx.x == 0) p.dapart[bh * p.da_parts + p.nch + c] = s;
    }
  }
  if (threadIdx.x == 0) tma_store_wait0();   // ∂k and ∂v are in global memory
  BtSetup<D>::teardown(x);
}

// The chunk scans, four consecutive state elements per thread (the matrix
// part [D' × D], then the vector part [D']):
//   forward (S, z): out[c] = acc, acc ← a^{cs_c}·acc + ΔS_c — the state
//     entering chunk c; the matrix part goes only to its bf16 operand tile
//     (for the ∂q pass), the vector part z_c stays fp32 in place;
//   reverse (M, N): walking down, out[c] = acc, acc ← ΔM_c + a^{cs_c}·acc —
//     the adjoint after chunk c, stored the same way (M_c as the operand tile
//     of the ∂k/∂v pass, N_c in fp32).  With ∂a, every thread also sums its
//     part of the pairs across the chunks, Σ_c cs_c·a^{cs_c−1}(⟨S_c, M_c⟩ +
//     ⟨z_c, N_c⟩), with S_c read from its bf16 operand tile (the value the
//     ∂q pass uses) and z_c in fp32; each warp stores one total in da_out.
// The operand tile is [D' × 64]-column blocks with the 128-byte swizzle, the
// layout the tensor-core passes copy into shared memory as is.  The next
// chunks' values are loaded before the current results are stored, so that
// loads stay in flight.
template <int D, bool REV>
__global__ void __launch_bounds__(256, 2)
bt_chunk_scan(float* __restrict__ S, float* __restrict__ z, __nv_bfloat16* __restrict__ tiles,
              const __nv_bfloat16* __restrict__ fS, const float* __restrict__ fz, float* __restrict__ da_out,
              int da_parts, int64_t H, int nch, int64_t n, const float* __restrict__ decay) {
  constexpr int DPD = D * D;
  static_assert(DPD % 1024 == 0, "a block holds matrix elements only or vector elements only");
  const int64_t bh = blockIdx.x;
  const float a = decay ? decay[bh % H] : 1.f;
  const float a_full = decay_pow(a, kCb);
  const float wfull = (float)kCb * decay_pow(a, kCb - 1);
  const bool fwd_state = REV && da_out;
  const int slot = blockIdx.y * 8 + (threadIdx.x >> 5);
  auto idx = [&](int i) { return REV ? nch - 1 - i : i; };   // i-th chunk visited
  auto clen = [&](int c) { return (int)min((int64_t)kCb, n - (int64_t)c * kCb); };
  auto fac = [&](int c) {
    const int len = clen(c);
    return len == kCb ? a_full : decay_pow(a, len);
  };
  // The scan of four consecutive elements: of the matrix part (MAT; every
  // thread of the block) or of the vector part (the first D/4 threads of the
  // last block).
  auto run = [&](auto mat_tag) {
    constexpr bool MAT = decltype(mat_tag)::value;
    // the ∂a stream (S_c from its operand tile, z_c in fp32) is kept as raw
    // bits and widened only where it is used, so that the prefetching loads
    // do not wait for their data
    using Raw = std::conditional_t<MAT, uint2, uint4>;
    constexpr int kB = REV ? 6 : 8;   // chunks in flight (the reverse scan loads two streams)
    const int e4 = (blockIdx.y * 256 + threadIdx.x) * 4 - (MAT ? 0 : DPD);
    const bool valid = MAT || e4 < D;
    const int64_t off = MAT ? bh * nch * (int64_t)DPD + e4 : bh * nch * (int64_t)D + e4;
    float* base = (MAT ? S : z) + off;
    constexpr int64_t stride = MAT ? DPD : D;
    // byte offset of this thread's four elements inside an operand tile
    const int row = e4 / D, col = e4 % D;
    const uint32_t toff = MAT ? sw_chunk(D, row, col >> 6, (col & 63) >> 3) + (col & 7) * 2 : 0u;
    uint8_t* tbase = reinterpret_cast<uint8_t*>(tiles + bh * nch * (int64_t)DPD) + toff;
    const uint8_t* fbase = nullptr;
    if (fwd_state)
      fbase = MAT ? reinterpret_cast<const uint8_t*>(fS + bh * nch * (int64_t)DPD) + toff
                  : reinterpret_cast<const uint8_t*>(fz + off);
    auto ld = [&](int i) {
      return (valid && i < nch) ? *reinterpret_cast<const float4*>(base + idx(i) * stride)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto ld_state = [&](int i) {
      Raw u{};
      if (valid && i < nch)
        u = *reinterpret_cast<const Raw*>(fbase + idx(i) * stride * (MAT ? 2 : 4));
      return u;
    };
    auto state_val = [](const Raw& u) {
      if constexpr (MAT)
        return make_float4(bf16lo_to_f32(u.x), bf16hi_to_f32(u.x), bf16lo_to_f32(u.y),
                           bf16hi_to_f32(u.y));
      else
        return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                           __uint_as_float(u.w));
    };
    float da_acc = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 cur[kB], nxt[kB];
    Raw fcur[kB], fnxt[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      cur[j] = ld(j);
      if (fwd_state) fcur[j] = ld_state(j);
    }
    for (int i0 = 0; i0 < nch; i0 += kB) {
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        nxt[j] = ld(i0 + kB + j);
        if (fwd_state) fnxt[j] = ld_state(i0 + kB + j);
      }
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int i = i0 + j;
        if (i < nch) {
          const int c = idx(i);
          if (valid) {
            if (MAT)
              *reinterpret_cast<uint2*>(tbase + c * (int64_t)DPD * 2) =
                  make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
            else
              *reinterpret_cast<float4*>(base + c * stride) = acc;
          }
          if (fwd_state) {
            const int len = clen(c);
            const float w_c = len == kCb ? wfull : (float)len * decay_pow(a, len - 1);
            const float4 sv = state_val(fcur[j]);
            da_acc += w_c * (acc.x * sv.x + acc.y * sv.y + acc.z * sv.z + acc.w * sv.w);
          }
          const float f = fac(c);
          acc = make_float4(f * acc.x + cur[j].x, f * acc.y + cur[j].y, f * acc.z + cur[j].z,
                            f * acc.w + cur[j].w);
        }
      }
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        cur[j] = nxt[j];
        if (fwd_state) fcur[j] = fnxt[j];
      }
    }
    return da_acc;
  };
  const bool mat_block = (blockIdx.y + 1) * 1024 <= DPD;
  float da_acc = mat_block ? run(std::true_type{}) : run(std::false_type{});
  if (fwd_state) {   // block-uniform: every lane takes part
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) da_acc += __shfl_xor_sync(0xffffffffu, da_acc, o);
    if ((threadIdx.x & 31) == 0) da_out[bh * (int64_t)da_parts + slot] = da_acc;
  }
}

template <int D>
cudaError_t run_bt(const BwdArgs& a, float* ws, int num_sms, int* status, cudaStream_t stream) {
  using Cfg = BtCfg<D>;
  cudaError_t e;
  const int64_t BH = a.B * a.H;
  const int nch = (int)((a.n + kCb - 1) / kCb);
  BtParams p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k);
  p.g = static_cast<const __nv_bfloat16*>(a.g);
  p.dq = static_cast<__nv_bfloat16*>(a.dq);
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.decay = a.decay;
  p.H = a.H;
  p.n = a.n;
  p.nch = nch;
  p.items = BH * nch;
  p.want_da = a.da != nullptr;
  p.status = status;
  const size_t ns = (size_t)BH * nch;
  const dim3 sgrid((unsigned)BH, (unsigned)((D * D + D) / 4 + 255) / 256);
  float* cur = ws;
  p.S = cur; cur += ns * D * D;
  p.z = cur; cur += ns * D;
  p.M = cur; cur += ns * D * D;
  p.N = cur; cur += ns * D;
  __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(cur); cur += ns * D * D / 2;
  __nv_bfloat16* mt = reinterpret_cast<__nv_bfloat16*>(cur); cur += ns * D * D / 2;
  p.St = st;
  p.Mt = mt;
  p.den = cur; cur += (size_t)BH * a.n;
  p.rho = cur; cur += (size_t)BH * a.n;
  p.dapart = cur;
  p.da_parts = 2 * nch + (int)sgrid.y * 8;
  CUtensorMap mq, mk, mv, mg, mdq, mdk, mdv, mdm, mds;
  if ((e = tmap_f32_mats(&mds, p.S, (int64_t)ns, D)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mdq, a.dq, BH, a.n, D, kCb)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mdk, a.dk, BH, a.n, D, kCb)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mdv, a.dv, BH, a.n, D, kCb)) != cudaSuccess) return e;
  if ((e = tmap_f32_mats(&mdm, p.M, (int64_t)ns, D)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mq, a.q, BH, a.n, D, kCb)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mk, a.k, BH, a.n, D, kCb)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mv, a.v, BH, a.n, D, kCb)) != cudaSuccess) return e;
  if ((e = tmap_rows(&mg, a.g, BH, a.n, D, kCb)) != cudaSuccess) return e;
  const int smem = Cfg::SMEM_ALLOC;
  if ((e = cudaFuncSetAttribute(bt_state_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(bt_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(bt_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem)) != cudaSuccess)
    return e;
  const unsigned grid = (unsigned)std::min<int64_t>(p.items, (int64_t)num_sms);
  bt_state_kernel<D><<<grid, kThreadsB, smem, stream>>>(mk, mv, mds, p);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bt_chunk_scan<D, false><<<sgrid, 256, 0, stream>>>(p.S, p.z, st, nullptr, nullptr, nullptr, 0, a.H,
                                                     nch, a.n, a.decay);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bt_dq_kernel<D><<<grid, kThreadsB, smem, stream>>>(mq, mk, mv, mg, mdq, mdm, p);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bt_chunk_scan<D, true><<<sgrid, 256, 0, stream>>>(p.M, p.N, mt, st, p.z,
                                                    p.want_da ? p.dapart + 2 * nch : nullptr, p.da_parts,
                                                    a.H, nch, a.n, a.decay);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bt_dkdv_kernel<D><<<grid, kThreadsB, smem, stream>>>(mq, mk, mv, mg, mdk, mdv, p);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.want_da) return backward_da_reduce(p.dapart, a.da, a.B, a.H, p.da_parts, stream);
  return cudaSuccess;
}

}  // namespace

bool tc_backward_supported(const BwdArgs& a) {
  return a.bf16 && !a.performer && (a.d == 64 || a.d == 128) && a.n >= 1;
}

size_t tc_backward_ws_floats(const BwdArgs& a) {
  const size_t BH = (size_t)(a.B * a.H);
  const size_t nch = (size_t)((a.n + kCb - 1) / kCb);
  const size_t D = (size_t)a.d;
  const size_t scan_warps = 8 * (((D * D + D) / 4 + 255) / 256);
  return BH * nch * (3 * D * D + 2 * D) + 2 * BH * (size_t)a.n + BH * (2 * nch + scan_warps);
}

cudaError_t tc_backward(const BwdArgs& a, float* ws, int num_sms, int* status,
                        cudaStream_t stream) {
  if (a.d == 128) return run_bt<128>(a, ws, num_sms, status, stream);
  if (a.d == 64) return run_bt<64>(a, ws, num_sms, status, stream);
  return cudaErrorInvalidValue;
}

}  // namespace la
