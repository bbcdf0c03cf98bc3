// Tensor-core (tcgen05 + TMA + TMEM) readout of non-causal kernelized linear
// attention with the elu+1 feature map, bf16 inputs, fp32 state,
// d = d' ∈ {64, 128}.
//
// Method ("Efficient Transformers II" §2.2 eq (6), "Efficient Transformers I"
// eq (27)): o = D⁻¹(Q'(K'ᵀV)) with D = diag(Q'(K'ᵀ1)).  Regrouped as in eq (9),
// every token reads out the same totals S = Σ_s k'_sᵀv_s [d' × d] and
// z = Σ_s k'_sᵀ [d']:  o_t = q'_t·S / q'_t·z.  The totals come from the
// state-only launch of the causal kernel over all segments and the segment
// scan's total; this kernel applies them to the queries.
//
// One CTA per (head, segment), 16 warps; per 128-token chunk:
//   warp 0        TMA producer: the raw q tile into one of NQ stages
//   warp 1        tcgen05 MMA issuer (TMEM owner): num = Q'·S (M 128, N d,
//                 K d) into one of two TMEM buffers
//   warps 4–7     epilogue: o = num / den → bf16, row by row
//   warps 8–15    φ(Q) → Q' in place (bf16, the MMA's A operand), and the
//                 normaliser den_t = q'_t·z in fp32 from the same bf16 Q'
//                 and the fp32 z (one column half per warpgroup)
// S enters the product as a bf16 operand tile (the same operand and layout
// as the causal kernel's inter-chunk product); z stays fp32.  Every wait is
// bounded in time and reports LA_ERR_TIMEOUT through the device status word.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

#include <cuda.h>

namespace la {
namespace {

using namespace tc;

constexpr int kC = 128;          // tokens per chunk (MMA M)
constexpr int kThreads = 512;

template <int D>
struct RCfg {
  static constexpr int HALVES = D / 64;            // 64-column swizzle atoms per row
  static constexpr int TILE = kC * D * 2;          // one [128 × D] bf16 q tile
  static constexpr int STILE = D * D * 2;          // the bf16 state operand [D' × D]
  static constexpr int NQ = D == 128 ? 4 : 8;      // q stages
  static constexpr int oQ0 = 0;
  static constexpr int oS = oQ0 + NQ * TILE;
  static constexpr int oZ = oS + STILE;            // z, fp32 [D']
  static constexpr int oDEN = oZ + D * 4;          // den partials [stage][half][128 rows]
  static constexpr int oBAR = oDEN + NQ * 2 * kC * 4;
  static constexpr int NBAR = 2 * NQ + NQ + 4 + 1;
  static constexpr int oMISC = oBAR + NBAR * 8;    // tmem slot, abort flag
  static constexpr int BYTES = oMISC + 16;
  // at least half the SM's shared memory: one CTA per SM
  static constexpr int SMEM_ALLOC = (BYTES + 1024 > 118 * 1024) ? BYTES + 1024 : 118 * 1024;
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
  // tensor memory: two numerator buffers of D columns
  static constexpr uint32_t TMEM_COLS = 2 * D;
};

// barrier indices (offsets into the CTA's barrier array)
template <int D>
struct RBar {
  static constexpr int QFULL = 0;                   // NQ: q tile landed
  static constexpr int QREADY = RCfg<D>::NQ;        // NQ: Q' and den written
  static constexpr int QEMPTY = 2 * RCfg<D>::NQ;    // NQ: Q' read by the MMA, den by the epilogue
  static constexpr int NFULL = 3 * RCfg<D>::NQ;     // 2: numerator buffer ready
  static constexpr int NEMPTY = NFULL + 2;          // 2: numerator buffer read
  static constexpr int DONE = NEMPTY + 2;           // every MMA finished
  static_assert(DONE + 1 <= RCfg<D>::NBAR, "barrier slots");
};

struct RParams {
  __nv_bfloat16* out;        // [BH, n, D]
  const float* tot_state;    // [BH][D·D] S (row = feature)
  const float* tot_z;        // [BH][D]
  int64_t n, seg_len;
  int* status;
};

struct RCtx {
  uint8_t* sm;
  uint32_t sbase;
  uint64_t* bar;
  volatile int* abort_flag;
  uint32_t tmem;
  int* status;
  int64_t bh, t_begin, t_end;
  int nchunks;
};

template <int D>
__device__ __forceinline__ void role_producer(const RCtx& x, const CUtensorMap* mq) {
  using Cfg = RCfg<D>;
  using Bar = RBar<D>;
  uint64_t* bar = x.bar;
  int c = 0;
  for (; c < x.nchunks && !*x.abort_flag; ++c) {
    const int s = c % Cfg::NQ;
    const int u = c / Cfg::NQ;   // use of the stage
    if (u >= 1 && !mbar_wait(&bar[Bar::QEMPTY + s], (u - 1) & 1, x.status, x.abort_flag)) break;
    const int y = (int)(x.t_begin + (int64_t)c * kC);
    // the tile's first row lies in this CTA's token range
    if (!LA_DCHECK(x.status, y >= x.t_begin && y < x.t_end, 31)) break;
    mbar_arrive_expect_tx(&bar[Bar::QFULL + s], Cfg::TILE);
    for (int h = 0; h < Cfg::HALVES; ++h)
      tma_load_3d(x.sm + Cfg::oQ0 + s * Cfg::TILE + h * kC * 128, mq, &bar[Bar::QFULL + s], h * 64,
                  y, (int)x.bh);
  }
  if (*x.abort_flag) {
    // drain the loads still in flight before the CTA's shared memory goes away
    for (int j = max(0, c - Cfg::NQ); j < c; ++j)
      mbar_wait_drain(&bar[Bar::QFULL + j % Cfg::NQ], (j / Cfg::NQ) & 1);
  }
}

template <int D>
__device__ __forceinline__ void role_mma(const RCtx& x) {
  using Cfg = RCfg<D>;
  using Bar = RBar<D>;
  uint64_t* bar = x.bar;
  constexpr uint32_t idN = idesc_bf16_f32(128, D, false, true);   // A K-major, B MN-major
  const uint64_t dS = smem_desc(x.sbase + Cfg::oS, D * 128, 1024, kSwizzle128B);
  for (int c = 0; c < x.nchunks; ++c) {
    const int s = c % Cfg::NQ;
    const int b = c & 1;
    if (!mbar_wait(&bar[Bar::QREADY + s], (c / Cfg::NQ) & 1, x.status, x.abort_flag)) break;
    if (c >= 2 && !mbar_wait(&bar[Bar::NEMPTY + b], ((c >> 1) - 1) & 1, x.status, x.abort_flag))
      break;
    tc_fence_after();
    const uint64_t dQ = smem_desc(x.sbase + Cfg::oQ0 + s * Cfg::TILE, 16, 1024, kSwizzle128B);
#pragma unroll
    for (int k = 0; k < D / 16; ++k)
      mma_ss(x.tmem + b * D, desc_at(dQ, (k >> 2) * (kC * 128) + (k & 3) * 32),
             desc_at(dS, k * 2048), idN, k > 0);
    mma_commit(&bar[Bar::NFULL + b]);
    mma_commit(&bar[Bar::QEMPTY + s]);
  }
  // every issued MMA must finish before TMEM is released
  mma_commit(&bar[Bar::DONE]);
  mbar_wait_drain(&bar[Bar::DONE], 0);
}

// Warps 8–15: φ(Q) in place and the den partials of one column half.
template <int D>
__device__ __forceinline__ void role_phi(const RCtx& x, int warp, int lane) {
  using Cfg = RCfg<D>;
  using Bar = RBar<D>;
  uint64_t* bar = x.bar;
  const int half = (warp - 8) >> 2;
  const int r = ((warp - 8) & 3) * 32 + lane;
  constexpr int NJ = D / 16;          // 16-byte chunks of a row per column half
  const int j0 = half * NJ;
  const uint32_t zbase = x.sbase + Cfg::oZ;
  float* den = reinterpret_cast<float*>(x.sm + Cfg::oDEN);
  for (int c = 0; c < x.nchunks; ++c) {
    const int s = c % Cfg::NQ;
    if (!warp_wait(&bar[Bar::QFULL + s], (c / Cfg::NQ) & 1, x.status, x.abort_flag)) return;
    uint8_t* qt = x.sm + Cfg::oQ0 + s * Cfg::TILE;
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int jj = j0 + j;
      const uint32_t off = sw_chunk(kC, r, jj >> 3, jj & 7);
      uint4 u = *reinterpret_cast<const uint4*>(qt + off);
      u.x = elu1_bf16x2(u.x);
      u.y = elu1_bf16x2(u.y);
      u.z = elu1_bf16x2(u.z);
      u.w = elu1_bf16x2(u.w);
      *reinterpret_cast<uint4*>(qt + off) = u;
      // z[8jj … 8jj+7]: the same address in every lane (a broadcast)
      const float4 z0 = lds128f(zbase + jj * 32);
      const float4 z1 = lds128f(zbase + jj * 32 + 16);
      acc = fmaf(bf16lo_to_f32(u.x), z0.x, acc);
      acc = fmaf(bf16hi_to_f32(u.x), z0.y, acc);
      acc = fmaf(bf16lo_to_f32(u.y), z0.z, acc);
      acc = fmaf(bf16hi_to_f32(u.y), z0.w, acc);
      acc = fmaf(bf16lo_to_f32(u.z), z1.x, acc);
      acc = fmaf(bf16hi_to_f32(u.z), z1.y, acc);
      acc = fmaf(bf16lo_to_f32(u.w), z1.z, acc);
      acc = fmaf(bf16hi_to_f32(u.w), z1.w, acc);
    }
    den[(s * 2 + half) * kC + r] = acc;
    fence_proxy_async_smem();   // Q' is read by the tensor core
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[Bar::QREADY + s]);
  }
}

// Warps 4–7: o = num / den for token row r of every chunk.
template <int D>
__device__ __forceinline__ void role_epilogue(const RCtx& x, const RParams& p, int warp, int lane) {
  using Cfg = RCfg<D>;
  using Bar = RBar<D>;
  uint64_t* bar = x.bar;
  const int wq = warp - 4;
  const int r = wq * 32 + lane;
  const uint32_t lane_base = (uint32_t)wq * 32;
  const float* den = reinterpret_cast<const float*>(x.sm + Cfg::oDEN);
  for (int c = 0; c < x.nchunks; ++c) {
    const int s = c % Cfg::NQ;
    const int b = c & 1;
    // the den partials of the stage (written before its Q' was handed over)
    // and the numerator
    if (!warp_wait(&bar[Bar::QREADY + s], (c / Cfg::NQ) & 1, x.status, x.abort_flag) ||
        !warp_wait(&bar[Bar::NFULL + b], (c >> 1) & 1, x.status, x.abort_flag))
      return;
    tc_fence_after();
    const float inv = 1.f / (den[(s * 2) * kC + r] + den[(s * 2 + 1) * kC + r]);
    uint32_t ob[D / 2];
#pragma unroll
    for (int j0 = 0; j0 < D; j0 += 32) {
      uint32_t nv[32];
      tmem_ld32(tmem_addr(x.tmem, lane_base, b * D + j0), nv);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; e += 2)
        ob[j0 / 2 + e / 2] =
            pack_bf16x2(__uint_as_float(nv[e]) * inv, __uint_as_float(nv[e + 1]) * inv);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&bar[Bar::NEMPTY + b]);
      mbar_arrive(&bar[Bar::QEMPTY + s]);   // the den partials of this stage are read
    }
    const int64_t t = x.t_begin + (int64_t)c * kC + r;
    if (t < x.t_end && LA_DCHECK(x.status, x.t_end <= p.n, 32)) {
      uint4* orow = reinterpret_cast<uint4*>(p.out + (x.bh * p.n + t) * D);
#pragma unroll
      for (int q = 0; q < D / 8; ++q)
        __stcs(orow + q, make_uint4(ob[4 * q], ob[4 * q + 1], ob[4 * q + 2], ob[4 * q + 3]));
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
tcr_readout_kernel(const __grid_constant__ CUtensorMap map_q, const RParams p) {
  using Cfg = RCfg<D>;
  using Bar = RBar<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  RCtx x;
  x.sm = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  x.sbase = smem_u32(x.sm);
  x.bar = reinterpret_cast<uint64_t*>(x.sm + Cfg::oBAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(x.sm + Cfg::oMISC);
  x.abort_flag = reinterpret_cast<volatile int*>(x.sm + Cfg::oMISC + 4);
  x.status = p.status;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  x.bh = blockIdx.x;
  x.t_begin = (int64_t)blockIdx.y * p.seg_len;
  x.t_end = min(p.n, x.t_begin + p.seg_len);
  x.nchunks = (int)((x.t_end - x.t_begin + kC - 1) / kC);

  if (tid == 0) {
    for (int i = 0; i < Cfg::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i >= Bar::QREADY && i < Bar::QREADY + Cfg::NQ) cnt = 8;        // φ warps
      if (i >= Bar::QEMPTY && i < Bar::QEMPTY + Cfg::NQ) cnt = 1 + 4;    // MMA + epilogue warps
      if (i == Bar::NEMPTY || i == Bar::NEMPTY + 1) cnt = 4;
      mbar_init(&x.bar[i], cnt);
    }
    *x.abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&map_q);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  // the totals come from the launch before this one (the segment scan)
  grid_dependency_wait();
  // S → bf16 operand tile (row = feature, 64-column swizzle atoms), z → fp32
  {
    const float* S = p.tot_state + x.bh * (int64_t)(D * D);
    uint32_t* zs = reinterpret_cast<uint32_t*>(x.sm + Cfg::oZ);
    for (int i = tid; i < D; i += kThreads)
      zs[i] = __float_as_uint(p.tot_z[x.bh * D + i]);
    // one thread per 8 consecutive elements of a row
    for (int i = tid; i < D * D / 8; i += kThreads) {
      const int row = i / (D / 8), j = i % (D / 8);
      const float4 a = reinterpret_cast<const float4*>(S + row * D + j * 8)[0];
      const float4 b = reinterpret_cast<const float4*>(S + row * D + j * 8)[1];
      const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      sts128(x.sbase + Cfg::oS + sw_chunk(D, row, j >> 3, j & 7), pack8(f));
    }
    fence_proxy_async_smem();   // read by the tensor core
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  x.tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) role_producer<D>(x, &map_q);
  } else if (warp == 1) {
    if (lane == 0) role_mma<D>(x);
  } else if (warp >= 4 && warp < 8) {
    role_epilogue<D>(x, p, warp, lane);
  } else if (warp >= 8) {
    role_phi<D>(x, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(x.tmem, Cfg::TMEM_COLS);
  }
}

template <int D>
cudaError_t run_readout(const FwdArgs& a, const float* tot_state, const float* tot_z,
                        const SegmentPlan& plan, bool dependent, cudaStream_t stream) {
  using Cfg = RCfg<D>;
  const int64_t BH = a.B * a.H;
  CUtensorMap mq;
  cudaError_t e;
  if ((e = tmap_rows(&mq, a.q, BH, a.n, D, kC)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tcr_readout_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  RParams p{};
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.tot_state = tot_state;
  p.tot_z = tot_z;
  p.n = a.n;
  p.seg_len = plan.seg_len;
  p.status = a.status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)BH, (unsigned)plan.nseg);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg::SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, tcr_readout_kernel<D>, mq, p);
  count_launches(1);
  return e;
}

}  // namespace

bool tc_readout_supported(const FwdArgs& a) {
  return a.bf16 && !a.performer && !a.causal && (a.d == 64 || a.d == 128) && a.n >= kC;
}

cudaError_t tc_noncausal_forward(const FwdArgs& a, cudaStream_t stream, float* ws_state,
                                 float* ws_z, float* tot_state, float* tot_z,
                                 const SegmentPlan& plan) {
  // the aggregate of every segment, their total, then the readout
  cudaError_t e = tc_state_only(a, stream, ws_state, ws_z, plan);
  if (e != cudaSuccess) return e;
  e = segment_total(ws_state, ws_z, tot_state, tot_z, a.B * a.H, a.H, plan.nseg, plan.seg_len,
                    a.n, a.d, a.d, nullptr, nullptr, stream, true);
  if (e != cudaSuccess) return e;
  if (a.d == 128) return run_readout<128>(a, tot_state, tot_z, plan, true, stream);
  if (a.d == 64) return run_readout<64>(a, tot_state, tot_z, plan, true, stream);
  return cudaErrorInvalidValue;
}

}  // namespace la
