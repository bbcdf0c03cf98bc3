// The exchange step of a sequence split across devices ("Efficient
// Transformers II" §2.2, eq (10)–(11) unrolled over a shard): shard j of a
// head holds L_j consecutive tokens and, run from zero, reaches its aggregate
// A_j (the state la_forward_state returns).  The state entering shard r is
//   S_in(r) = Σ_{j<r} a^{L_{j+1} + … + L_{r−1}} A_j,
// i.e. S ← 0, then S ← a^{L_j}·S + A_j for j = 0 … r−1 (ν likewise; a = 1
// without a decay).  la_shard_entering_state computes it from the aggregates
// of all shards gathered in one buffer.
#include "common.cuh"
#include "internal.h"

#include <cuda_runtime.h>

namespace la {
namespace {

constexpr int kMaxShards = 256;

struct ShardLens {
  int64_t len[kMaxShards];
};

// One thread per state element e of head bh (e < d'·d: μ, else ν).
__global__ void __launch_bounds__(256)
shard_prefix_kernel(const float* __restrict__ gathered, int rank, ShardLens lens, const float* decay,
                    int64_t H, int64_t BH, int dpd, int dp, float* mu_in, float* nu_in) {
  const int64_t bh = blockIdx.x;
  const int e = blockIdx.y * 256 + threadIdx.x;
  if (e >= dpd + dp) return;
  const float a = decay ? decay[bh % H] : 1.f;
  // one shard's block: μ [BH][dpd], then ν [BH][dp]
  const int64_t block = BH * (int64_t)(dpd + dp);
  const int64_t off = e < dpd ? bh * dpd + e : BH * (int64_t)dpd + bh * dp + (e - dpd);
  float acc = 0.f;
  for (int j = 0; j < rank; ++j) acc = decay_pow(a, lens.len[j]) * acc + gathered[j * block + off];
  if (e < dpd) mu_in[bh * dpd + e] = acc;
  else nu_in[bh * dp + (e - dpd)] = acc;
}

}  // namespace
}  // namespace la

la_status la_shard_entering_state(const float* gathered, int nshards, int rank,
                                  const int64_t* shard_len, const float* decay_a, int64_t B,
                                  int64_t H, int dp, int d, float* mu_in, float* nu_in,
                                  la_stream stream) {
  la::ApiRange range_("la_shard_entering_state");
  if (!gathered || !shard_len || !mu_in || !nu_in) return LA_ERR_INVALID_ARG;
  if (nshards < 1 || rank < 0 || rank >= nshards || B < 1 || H < 1 || dp < 1 || d < 1)
    return LA_ERR_INVALID_ARG;
  if (nshards > la::kMaxShards) return LA_ERR_UNSUPPORTED;
  if (decay_a && (reinterpret_cast<uintptr_t>(decay_a) & 3u)) return LA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(gathered) | reinterpret_cast<uintptr_t>(mu_in) |
       reinterpret_cast<uintptr_t>(nu_in)) & 3u)
    return LA_ERR_INVALID_ARG;
  la::ShardLens lens{};
  for (int j = 0; j < nshards; ++j) {
    if (shard_len[j] < 0) return LA_ERR_INVALID_ARG;
    lens.len[j] = shard_len[j];
  }
  const int64_t BH = B * H;
  const int dpd = dp * d;
  const dim3 grid((unsigned)BH, (unsigned)((dpd + dp + 255) / 256));
  la::shard_prefix_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      gathered, rank, lens, decay_a, H, BH, dpd, dp, mu_in, nu_in);
  la::count_launches(1);
  return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}
