// Internal host-side interfaces between the translation units of liblinattn.
// Not part of the public ABI (include/linattn.h is).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "linattn.h"

namespace la {

// Everything a forward launcher needs, already validated by the API layer.
struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  const float* decay;   // device [H] or nullptr (a = 1)
  const float* tok_decay;   // device [B,H,n] per-token decay, or nullptr
  const float* tok_weight;  // device [B,H,n] per-token input weight, or nullptr (1 − a)
  float* ws_ld;         // per-token decay, nseg > 1: [B·H][nseg] log2 decay of each segment
  float* ws_tok;        // per-token decay, tensor-core path: [2][B·H][n], the log2 prefix of
                        // a within each 128-token chunk, then the weight b (or 1 − a)
  const void* omega;    // device [d, m] (Performer) or nullptr
  int64_t B, H, n;
  int d;                // value / input width
  int m;                // Performer feature count (0 for elu+1)
  int dp;               // feature width d' (d for elu+1, m for Performer)
  bool bf16;            // element type of q, k, v, out, omega
  bool performer;
  bool causal;
  float* mu_out;        // optional final state [B,H,dp,d]
  float* nu_out;        // optional final state [B,H,dp]
  const float* init_state;  // causal: state entering token 0 [B,H,dp,d], or nullptr (zero)
  const float* init_z;      // [B,H,dp] (given together with init_state)
  int* status;          // device status word (bounded waits report here)
  int num_sms;
};

struct DecodeArgs {
  float* mu;            // [B,H,d',d]
  float* nu;            // [B,H,d']
  const void* q;
  const void* k;
  const void* v;
  void* out;
  const float* decay;   // [H] (or nullptr: a = 1), or [B·H] when per_token
  const float* weight;  // per_token: new-token weights [B·H], or nullptr for 1 − a
  bool per_token;
  const void* omega;    // Performer: [d, m]; else nullptr
  int64_t B, H;
  int d;
  int m;                // Performer feature count (0 for elu+1)
  bool bf16;
  bool performer;
};

// Everything the backward needs, already validated by the API layer.
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* g;        // ∂L/∂o [B,H,n,d]
  void* dq;
  void* dk;
  void* dv;
  const float* decay;   // [H] or nullptr (a = 1)
  float* da;            // [H] or nullptr
  const void* omega;
  int64_t B, H, n;
  int d, m, dp;
  bool bf16;
  bool performer;
};

// Segment plan shared by the forward paths: the sequence of every head is cut
// into nseg segments of seg_len tokens (the last one ragged); per-segment
// states are combined by segment_scan.
struct SegmentPlan {
  int nseg;
  int64_t seg_len;
};

// fp32 CUDA-core chunked forward (fp32 or bf16 inputs).
cudaError_t simt_forward(const FwdArgs& a, cudaStream_t stream, float* ws_state,
                         float* ws_z, float* tot_state, float* tot_z,
                         const SegmentPlan& plan);

// The aggregate (the state reached from zero) of every segment of the plan,
// into ws_state / ws_z [BH][nseg]: the state-only kernels of each family.
cudaError_t simt_state_only(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                            const SegmentPlan& plan);
cudaError_t tc_state_only(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                          const SegmentPlan& plan);
cudaError_t tc_performer_state_only(const FwdArgs& a, cudaStream_t stream, float* ws_state,
                                    float* ws_z, const SegmentPlan& plan);

// tcgen05/TMA chunked forward (bf16, elu+1, causal, d ∈ {64, 128}, n ≥ 128).
bool tc_forward_supported(const FwdArgs& a);
int64_t tc_segment_granule();
cudaError_t tc_forward(const FwdArgs& a, cudaStream_t stream, float* ws_state, float* ws_z,
                       float* tot_state, float* tot_z, const SegmentPlan& plan);

// tcgen05/TMA non-causal forward with the elu+1 map (bf16, d ∈ {64, 128},
// n ≥ 128): the state-only launch over all segments, the scan's total (into
// tot_state / tot_z), then the readout o = q'·S / q'·z.
bool tc_readout_supported(const FwdArgs& a);
cudaError_t tc_noncausal_forward(const FwdArgs& a, cudaStream_t stream, float* ws_state,
                                 float* ws_z, float* tot_state, float* tot_z,
                                 const SegmentPlan& plan);

// tcgen05/TMA chunked forward with the Performer feature map (bf16, d = 64,
// m ∈ {128, 256}, no decay, n ≥ 128; causal and non-causal).
bool tc_performer_supported(const FwdArgs& a);
cudaError_t tc_performer_forward(const FwdArgs& a, cudaStream_t stream, float* ws_state,
                                 float* ws_z, float* tot_state, float* tot_z,
                                 const SegmentPlan& plan);

// TMA tensor maps (128-byte swizzle, boxes 128 bytes wide):
//   tmap_rows:     bf16 [BH, n, D] as a 3-D tensor, box 64 × rows × 1 (rows
//                  past n read as zero and are not written);
//   tmap_matrix:   a bf16 row-major [rows, cols] matrix, box 64 × box_rows;
//   tmap_f32_mats: `count` fp32 row-major [D × D] matrices, contiguous, as a
//                  3-D tensor, box 32 × D × 1.
cudaError_t tmap_rows(CUtensorMap* m, const void* base, int64_t BH, int64_t n, int D, int rows);
cudaError_t tmap_matrix(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows);
cudaError_t tmap_f32_mats(CUtensorMap* m, const void* base, int64_t count, int D);

// Exclusive decayed prefix over the per-segment aggregates of every head, in
// place.  Segment g's aggregate is carried past it with the factor
// decay^{its length} (per-head decay), or 2^{seg_ld[bh·nseg + g]} when seg_ld
// (the per-token decay's log2 total of each segment) is given.
// Only the first nagg aggregates are read (nagg = nseg − 1 when the
// last segment's aggregate was not computed: the exclusive prefixes do not
// need it); the inclusive total (final state) is written when tot_state !=
// nullptr and nagg == nseg.  init_state / init_z ([BH][dp·d], [BH][dp], or
// nullptr for zero) is the state entering segment 0.  `dependent` launches it as a programmatic
// dependent of the preceding launch (which must be this library's kernel
// that wrote the aggregates); the launch after it may then start early too.
cudaError_t segment_scan(float* ws_state, float* ws_z, float* tot_state, float* tot_z,
                         int64_t BH, int64_t H, int nseg, int nagg, int64_t seg_len, int64_t n,
                         int dp, int d, const float* decay, const float* seg_ld,
                         cudaStream_t stream, bool dependent, const float* init_state = nullptr,
                         const float* init_z = nullptr);

// The total of the same recurrence over all nseg aggregates of every head
// (acc ← init, then acc ← a^{L_g}·acc + A_g) into tot_state / tot_z, without
// the exclusive prefixes; the aggregates are left as they are.  float4
// loads (the scalar segment_scan when a pointer is not 16-byte aligned).
cudaError_t segment_total(float* ws_state, float* ws_z, float* tot_state, float* tot_z,
                          int64_t BH, int64_t H, int nseg, int64_t seg_len, int64_t n, int dp, int d,
                          const float* decay, const float* seg_ld, cudaStream_t stream,
                          bool dependent, const float* init_state = nullptr,
                          const float* init_z = nullptr);

// la_forward with a fixed workspace of ws_floats floats, fetched through
// get_ws only when the plan needs it, instead of stream-ordered allocations
// (see la_forward_noalloc).
la_status forward_in_workspace(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                               const float* decay_a, la_feature_map feature_map,
                               const la_tensor* omega, int causal, la_tensor* out,
                               la_status (*get_ws)(float**), size_t ws_floats,
                               cudaStream_t stream);

// Records `k` kernel launches in the process-wide launch counter.
void count_launches(int k);

// An NVTX range named after a C entry point for the lifetime of the object,
// when the environment variable LA_NVTX is set to a non-zero value (read
// once); otherwise nothing.  Profilers that record NVTX show each call's
// host-side span and the kernels it queued inside it.
class ApiRange {
 public:
  explicit ApiRange(const char* name);
  ~ApiRange();
  ApiRange(const ApiRange&) = delete;
  ApiRange& operator=(const ApiRange&) = delete;

 private:
  bool on_;
};

// One CTA of bounded waits on a barrier nothing signals (la_selftest_wait_timeout).
cudaError_t selftest_wait(int* status, uint64_t limit_ns, cudaStream_t stream);
// One guarded access whose LA_DEBUG check fails (la_selftest_device_check).
cudaError_t selftest_check(int* status, cudaStream_t stream);

// Backward of the causal forward (fp32 CUDA cores): ∂q, ∂k, ∂v and ∂a.
bool backward_supported(int d, int m, bool performer);
size_t backward_workspace_floats(const BwdArgs& a, const SegmentPlan& plan);
cudaError_t backward(const BwdArgs& a, float* ws, const SegmentPlan& plan, cudaStream_t stream);

// Scans of the backward over consecutive blocks (segments or chunks) of
// seg_len tokens, in place: forward (S, z) → the state entering each block;
// reverse (M, N) → the adjoint after each block.  Only the pointers of the
// chosen direction are used.
cudaError_t backward_scan(float* S, float* z, float* M, float* N, int64_t BH, int64_t H,
                          int nseg, int64_t seg_len, int64_t n, int dp, int d, const float* decay,
                          bool reverse, cudaStream_t stream);
// ∂a[h] = Σ over b and the nparts per-(b, h) partial sums (fp64 accumulation).
cudaError_t backward_da_reduce(const float* parts, float* da, int64_t B, int64_t H, int nparts,
                               cudaStream_t stream);

// Tensor-core backward (bf16, elu+1, d ∈ {64, 128}): chunk states, the ∂q
// pass and the ∂k/∂v pass on tcgen05; workspace of tc_backward_ws_floats.
bool tc_backward_supported(const BwdArgs& a);
size_t tc_backward_ws_floats(const BwdArgs& a);
cudaError_t tc_backward(const BwdArgs& a, float* ws, int num_sms, int* status, cudaStream_t stream);

// Memory-bound recurrent decode step.
cudaError_t decode_step(const DecodeArgs& a, cudaStream_t stream);

}  // namespace la
