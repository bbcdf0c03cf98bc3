/*
 * linattn.h — C ABI of the GB300 (sm_103a) causal kernelized linear attention
 * library (liblinattn.so).
 *
 * The method (cited by page title and equation):
 *   "Efficient Transformers II", §2.2 Linear Attention:
 *     eq (6)   Att = D⁻¹(Q'(K'ᵀV)),  Q' = φ(Q), K' = φ(K) ∈ R^{n×d'}
 *     eq (7)   μ_j = μ_{j−1} + k'_jᵀ v_j          (μ ∈ R^{d'×d})
 *     eq (8)   ν_j = ν_{j−1} + k'_jᵀ              (ν ∈ R^{d'})
 *     eq (9)   o_j = q'_j·μ / q'_j·ν  — μ_n, ν_n non-causal; μ_j, ν_j causal
 *     eq (10)  μ_j = a·μ_{j−1} + (1−a)·k'_jᵀ v_j
 *     eq (11)  ν_j = a·ν_{j−1} + (1−a)·k'_jᵀ
 *   "Linear Attention Research 2026", "Linear Transformer": φ(x) = elu(x)+1
 *     (α = 1), and "Performer random features": φ(x) = exp(xω − ½‖x‖²)/√m.
 *   "Efficient Transformers I", kernelized attention eq (25)–(27): the same
 *     output written as normalized weights (the quadratic form).
 *
 * Conventions shared by every entry point
 *   - Tensors are dense, row-major [B, H, n, d] with d innermost and no
 *     padding (element (b,h,t,c) at ((b·H + h)·n + t)·d + c).
 *   - All tensor data, decay values and state buffers are DEVICE pointers on
 *     the current CUDA device, owned by the caller.  The library never frees
 *     or retains them after a call returns.
 *   - A decay a = 1 (or decay_a == NULL) selects the plain sums of eq (7)–(8)
 *     (weight 1 on the new token); any other a ∈ [0, 1] selects eq (10)–(11)
 *     with weight (1 − a).  Values are read on the device only; values outside
 *     [0, 1] give unspecified (but finite-time, fault-free) results.
 *   - The exported state is μ [B, H, d', d] and ν [B, H, d'] in fp32,
 *     row i of μ being feature i of φ.
 *   - Work is queued on `stream` and the call returns without synchronising.
 *     Arguments are validated on the host before anything is queued: a call
 *     that returns an error queued no kernel and wrote nothing.
 *   - Temporary device workspace (per-segment states of long sequences) is
 *     taken stream-ordered on `stream` (cudaMallocFromPoolAsync /
 *     cudaFreeAsync) from a memory pool the library creates per device; the
 *     pool keeps its reservation (the largest workspace in flight at once)
 *     until the process exits, so repeated calls do not map memory again.
 *   - The library keeps per-device state only for cached device attributes,
 *     the device status word and cached kernel attributes.
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  LA_ERR_CUDA carries a CUDA runtime error from a launch or an
 * allocation; LA_ERR_TIMEOUT reports a bounded device-side wait that gave up;
 * LA_ERR_DEVICE_CHECK exists only in the LA_DEBUG build of the library. */
typedef enum {
  LA_OK = 0,
  LA_ERR_INVALID_ARG = 1,   /* null pointer, shape or dtype mismatch, misalignment */
  LA_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels implement */
  LA_ERR_CUDA = 3,          /* a CUDA runtime call failed */
  LA_ERR_TIMEOUT = 4,       /* a device-side bounded wait expired (see la_get_last_device_status) */
  LA_ERR_OUT_OF_MEMORY = 5, /* workspace allocation failed */
  LA_ERR_DEVICE_CHECK = 6   /* LA_DEBUG build: a kernel's index check failed and the
                               access was skipped (see la_get_last_device_check) */
} la_status;

typedef enum { LA_BF16 = 0, LA_F32 = 1 } la_dtype;

/* φ: elu(x)+1 ("Linear Transformer", d' = d) or Performer positive random
 * features ("Performer random features", d' = m). */
typedef enum { LA_FM_ELU1 = 0, LA_FM_PERFORMER = 1 } la_feature_map;

/* A dense [B, H, n, d] tensor (see conventions above).  `data` must be
 * 16-byte aligned. */
typedef struct {
  void* data;
  la_dtype dtype;
  int64_t B, H, n, d;
} la_tensor;

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* la_stream;

/*
 * la_forward — prefill / training forward of the whole sequence.
 *
 * Computes, for every (b, h) head independently:
 *   causal != 0 : o_j = q'_j·μ_j / q'_j·ν_j with μ, ν from eq (7)–(8) (a = 1)
 *                 or eq (10)–(11) (per-head a), starting from zero state and
 *                 including token j itself;
 *   causal == 0 : eq (6), o_j = q'_j·μ_n / q'_j·ν_n (no decay).
 *
 *   q, k, v      [B, H, n, d], same shape and dtype (LA_BF16 or LA_F32);
 *                d ∈ {32, 64, 128}; n ≥ 0 (n = 0 is a no-op).
 *   decay_a      device [H] fp32, or NULL for a = 1.  Must be NULL when
 *                causal == 0 (eq (6) has no decay) → LA_ERR_UNSUPPORTED.
 *   feature_map  LA_FM_ELU1 (omega must be NULL) or LA_FM_PERFORMER.
 *   omega        Performer only: tensor with B = H = 1, n = d, d = m,
 *                i.e. ω stored [d, m] row-major, same dtype as q;
 *                m ∈ {64, 128, 256}.  Column i of ω is the i-th random
 *                direction.  Scaling of ω (e.g. N(0, 1/d)) is the caller's.
 *   causal       non-zero for the causal (autoregressive) form.
 *   out          [B, H, n, d], same dtype as q.  Written in full.
 *   stream       CUDA stream for all work.
 *
 * bf16 inputs run on the tcgen05 tensor-core path with fp32 state; fp32
 * inputs run on an fp32 CUDA-core path.
 * Errors: LA_ERR_INVALID_ARG (null/shape/dtype/alignment), LA_ERR_UNSUPPORTED
 * (d, m, or decay with causal == 0), LA_ERR_OUT_OF_MEMORY, LA_ERR_CUDA.
 */
la_status la_forward(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                     const float* decay_a, la_feature_map feature_map,
                     const la_tensor* omega, int causal, la_tensor* out,
                     la_stream stream);

/*
 * la_forward_with_state — la_forward that also exports the final state
 * (μ_n, ν_n) of eq (7)–(11) for every head, e.g. to continue with
 * la_decode_step ("Efficient Transformers II" §2.2: μ and ν are the fixed-size
 * memory of the sequence).
 *   mu_out  device fp32 [B, H, d', d], 16-byte aligned, written in full.
 *   nu_out  device fp32 [B, H, d'], 16-byte aligned, written in full.
 * Other arguments and errors as la_forward.
 */
la_status la_forward_with_state(const la_tensor* q, const la_tensor* k,
                                const la_tensor* v, const float* decay_a,
                                la_feature_map feature_map, const la_tensor* omega,
                                int causal, la_tensor* out, float* mu_out,
                                float* nu_out, la_stream stream);

/*
 * la_forward_host — la_forward on host buffers: q, k, v, out (and decay_a
 * [H], omega when given) are page-locked host memory (cudaHostAlloc or
 * cudaHostRegister).  The library copies the inputs to device memory it
 * takes from its pool, runs la_forward, and copies o back; the heads are cut
 * into up to eight groups (along B, or along H when B = 1) so that the copies
 * of one group overlap the compute of the others.  The call is asynchronous:
 * the input copies may start as soon as it is made (on the library's own
 * copy stream, so the inputs must already be in host memory, not still being
 * written by device work), while the compute and the copy of o back are
 * ordered after the work already queued on `stream`, which resumes after the
 * last copy.  The host buffers must stay valid, and the inputs unchanged,
 * until then (synchronise `stream` before reading out).  The method
 * and the other arguments are those of la_forward ("Efficient Transformers
 * II" eq (6)–(11)).
 * Errors: those of la_forward; LA_ERR_INVALID_ARG also when a buffer is not
 * page-locked host memory.
 */
la_status la_forward_host(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                          const float* decay_a, la_feature_map feature_map, const la_tensor* omega,
                          int causal, la_tensor* out, la_stream stream);

/*
 * la_forward_from_state — the causal forward of la_forward continued from a
 * given state: the recurrence of eq (7)–(11) ("Efficient Transformers II"
 * §2.2) starts from μ_{−1} = mu0, ν_{−1} = nu0 instead of zero, so that
 * o_j = q'_j·μ_j / q'_j·ν_j with μ_j = a·μ_{j−1} + (1 − a)·k'_jᵀv_j (a = 1:
 * the plain sums).  Running a sequence as two calls, the second from the
 * first one's final state, gives the same outputs as one call.
 *   mu0, nu0        device fp32 [B, H, d', d] and [B, H, d'], 16-byte
 *                   aligned; both NULL for the zero state.
 *   mu_out, nu_out  final state as in la_forward_with_state, or both NULL.
 *                   Must not overlap mu0 / nu0.
 * Other arguments and errors as la_forward with causal != 0 (one NULL of a
 * pair, misalignment or overlap → LA_ERR_INVALID_ARG).  n = 0 copies the
 * initial state to the final one.
 */
la_status la_forward_from_state(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                                const float* decay_a, la_feature_map feature_map,
                                const la_tensor* omega, const float* mu0, const float* nu0,
                                la_tensor* out, float* mu_out, float* nu_out, la_stream stream);

/*
 * la_forward_state — the state (μ_n, ν_n) that the recurrence of eq (7)–(11)
 * reaches from zero over the whole sequence, without the outputs (no q, no
 * o): for a = 1 these are the sums Σ_j k'_jᵀv_j and Σ_j k'_jᵀ of eq (6).
 *   k, v            [B, H, n, d] as in la_forward.
 *   mu_out, nu_out  device fp32 [B, H, d', d] and [B, H, d'], 16-byte
 *                   aligned, written in full (zero for n = 0).
 * Other arguments and errors as la_forward with causal != 0.
 */
la_status la_forward_state(const la_tensor* k, const la_tensor* v, const float* decay_a,
                           la_feature_map feature_map, const la_tensor* omega, float* mu_out,
                           float* nu_out, la_stream stream);

/*
 * la_shard_entering_state — the exchange step of a causal sequence split
 * into consecutive shards (one per device): eq (10)–(11) unrolled over shard
 * j, whose aggregate A_j (la_forward_state of its L_j tokens) and length
 * are known to every device, give the state entering shard `rank`:
 *   S_in(rank) = Σ_{j<rank} a^{L_{j+1} + … + L_{rank−1}}·A_j
 * (ν likewise; a = 1 without a decay).  la_forward_from_state of the shard
 * from S_in then equals la_forward of the whole sequence on those tokens.
 *   gathered   device fp32, nshards consecutive blocks, block j = shard j's
 *              μ [B, H, d', d] followed by its ν [B, H, d']; 4-byte aligned.
 *   nshards    1 … 256; rank in [0, nshards).
 *   shard_len  host int64 [nshards], tokens per shard (≥ 0).
 *   decay_a    device [H] fp32, or NULL for a = 1.
 *   B, H, dp, d  the state's shape (dp = d' = d for elu+1, m for Performer).
 *   mu_in, nu_in  device fp32 [B, H, d', d] and [B, H, d'], written in full
 *              (zero for rank 0).
 * Errors: LA_ERR_INVALID_ARG (null pointer, bad count, rank or length,
 * misalignment), LA_ERR_UNSUPPORTED (more than 256 shards), LA_ERR_CUDA.
 */
la_status la_shard_entering_state(const float* gathered, int nshards, int rank,
                                  const int64_t* shard_len, const float* decay_a, int64_t B,
                                  int64_t H, int dp, int d, float* mu_in, float* nu_in,
                                  la_stream stream);

/*
 * la_decode_step — one recurrent step for B·H heads ("Efficient Transformers
 * II" eq (10)–(11) followed by the causal readout of eq (9)), elu+1 map:
 *   k' = φ(k), μ ← a·μ + w·k'ᵀv, ν ← a·ν + w·k', o = q'μ / q'ν,
 * with w = 1 − a (w = 1 when a = 1 or decay_a == NULL).
 *   mu      device fp32 [B, H, d, d], updated in place (d' = d).
 *   nu      device fp32 [B, H, d], updated in place.
 *   q, k, v [B, H, 1, d] LA_BF16 or LA_F32 (all the same dtype), d ∈ {32, 64, 128}.
 *   decay_a device [H] fp32 or NULL.
 *   out     [B, H, 1, d], same dtype as q.
 * Errors: LA_ERR_INVALID_ARG (null/shape/dtype/alignment, mu/nu not 16-byte
 * aligned), LA_ERR_UNSUPPORTED (d), LA_ERR_CUDA.
 */
la_status la_decode_step(float* mu, float* nu, const la_tensor* q,
                         const la_tensor* k, const la_tensor* v,
                         const float* decay_a, la_tensor* out, la_stream stream);

/*
 * la_decode_step_fm — la_decode_step with either feature map
 * ("Linear Attention Research 2026"): feature_map = LA_FM_ELU1 (omega must be
 * NULL; identical to la_decode_step) or LA_FM_PERFORMER, φ(x) =
 * exp(x·ω − ½‖x‖²)/√m with omega a [1, 1, d, m] tensor of the same dtype as
 * q (m ∈ {64, 128, 256}, 16-byte aligned).  The state is then mu [B, H, m, d]
 * and nu [B, H, m] (fp32, updated in place); everything else — shapes,
 * decay, readout o = q'·μ / q'·ν after the update, ownership, asynchrony and
 * errors — is as for la_decode_step.  Invalid or unsupported arguments
 * (unknown map, omega missing or with the wrong shape, dtype or alignment,
 * omega given for elu+1) are rejected before any launch.
 */
la_status la_decode_step_fm(float* mu, float* nu, const la_tensor* q, const la_tensor* k,
                            const la_tensor* v, const float* decay_a, la_feature_map feature_map,
                            const la_tensor* omega, la_tensor* out, la_stream stream);

/*
 * la_forward_token_decay — causal forward with a decay and an input weight
 * for every token: "Efficient Transformers II" eq (4), z_i = a·z_{i−1} + b·s_i,
 * with a and b indexed by the token (the input-dependent, "selective" state
 * update of the Mamba section of "Linear Attention Research 2026"), applied
 * to the state of eq (7)–(8):
 *   μ_i = a_i·μ_{i−1} + b_i·k'_iᵀv_i,  ν_i = a_i·ν_{i−1} + b_i·k'_iᵀ,
 *   o_i = q'_i·μ_i / q'_i·ν_i  (token i included, zero initial state).
 *   q, k, v, out, feature_map, omega  as la_forward (causal).
 *   decay_a   device fp32 [B, H, n] (the layout of q without d), 4-byte
 *             aligned, a_i ∈ [0, 1].  Required when B·H·n > 0.
 *   weight_b  device fp32 [B, H, n], 4-byte aligned, b_i ≥ 0 — or NULL for
 *             b_i = 1 − a_i (eq (10)–(11) per token; unlike la_forward there
 *             is no special case at a_i = 1: such a token gets weight 0).
 *   mu_out, nu_out  final state as in la_forward_with_state, or both NULL.
 * Decays are applied as powers of two of per-chunk running sums of log2 a_i,
 * with log2 a_i clamped at −64: a_i = 0 scales everything before token i by
 * 2^−64 rather than removing it exactly.  Values of a outside [0, 1] or
 * negative b give unspecified (finite-time, fault-free) results.
 * bf16 inputs with elu+1 and d ∈ {64, 128} run on the tcgen05 path, all
 * others on the fp32 CUDA-core path.
 * Errors: as la_forward; LA_ERR_INVALID_ARG also for a missing or misaligned
 * decay_a, a misaligned weight_b, or only one of mu_out / nu_out.
 */
la_status la_forward_token_decay(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                                 const float* decay_a, const float* weight_b,
                                 la_feature_map feature_map, const la_tensor* omega,
                                 la_tensor* out, float* mu_out, float* nu_out,
                                 la_stream stream);

/*
 * la_decode_step_token_decay — one recurrent step with this token's own
 * decay and weight (the step of la_forward_token_decay):
 *   μ ← a·μ + b·k'ᵀv,  ν ← a·ν + b·k',  o = q'μ / q'ν,
 *   decay_a   device fp32 [B, H], 4-byte aligned (required);
 *   weight_b  device fp32 [B, H], or NULL for b = 1 − a.
 * Everything else (state, shapes, feature maps, ownership, asynchrony,
 * errors) is as for la_decode_step_fm.
 */
la_status la_decode_step_token_decay(float* mu, float* nu, const la_tensor* q,
                                     const la_tensor* k, const la_tensor* v,
                                     const float* decay_a, const float* weight_b,
                                     la_feature_map feature_map, const la_tensor* omega,
                                     la_tensor* out, la_stream stream);

/*
 * la_backward — gradients of the causal forward (la_forward with causal != 0)
 * for training: given ∂L/∂o = grad_out, writes ∂L/∂q, ∂L/∂k, ∂L/∂v and,
 * when da != NULL, ∂L/∂a for the per-head decay ("Efficient Transformers II"
 * eq (7)–(11) and the causal readout after eq (9), differentiated; the pages
 * train a "as usual").  With ĝ_j = g_j/den_j and ρ_j = −(g_j·o_j)/den_j:
 *   ∂q'_j = Σ_{s≤j} w·a^{j−s}(ĝ_j·v_s + ρ_j) k'_s,
 *   ∂k'_s = Σ_{j≥s} w·a^{j−s}(ĝ_j·v_s + ρ_j) q'_j,
 *   ∂v_s  = Σ_{j≥s} w·a^{j−s}(q'_j·k'_s) ĝ_j,
 *   ∂a    = Σ_{s<j} (j−s)·w·a^{j−s−1}(q'_j·k'_s)(ĝ_j·v_s + ρ_j)  (summed over the batch),
 * then ∂q, ∂k through φ (elu+1: φ' = 1 for x > 0, e^x otherwise; Performer:
 * ∂φ_i/∂x = φ_i·(ω_i − x)).  The forward's outputs and normalizers are
 * recomputed; nothing from the forward call needs to be kept.
 *   q, k, v, decay_a, feature_map, omega  as la_forward (causal).
 *   grad_out      [B, H, n, d], same dtype as q.
 *   dq, dk, dv    [B, H, n, d], same dtype as q, written in full.
 *   da            device fp32 [H] or NULL; needs decay_a (INVALID_ARG otherwise).
 *                 At a = 1 it is the derivative of the plain sums' extension
 *                 a ↦ w(a)·a^{j−s} from below.
 * bf16 inputs with elu+1 and d ∈ {64, 128} run on tcgen05 tensor cores
 * (per-chunk forward states and adjoints are kept in the workspace: about
 * 2·(d² + d)·4 bytes per 128 tokens per head, plus 8 bytes per token); all
 * other cases run on fp32 CUDA cores.  d ∈ {32, 64, 128}, and for the
 * Performer map d·m ≤ 16384 (else LA_ERR_UNSUPPORTED).  Temporary workspace
 * as for la_forward (stream-ordered, from the library's pool).
 */
la_status la_backward(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                      const float* decay_a, la_feature_map feature_map, const la_tensor* omega,
                      const la_tensor* grad_out, la_tensor* dq, la_tensor* dk, la_tensor* dv,
                      float* da, la_stream stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* la_status_string(la_status status);

/*
 * la_get_last_device_status — synchronises `stream`, then reports and clears
 * the current device's status word, which kernels set when a bounded wait on
 * another CTA or on the tensor-core/TMA pipeline expires (LA_ERR_TIMEOUT).
 * Returns LA_ERR_CUDA if the synchronisation itself fails.
 */
la_status la_get_last_device_status(la_stream stream);

/*
 * la_forward_noalloc — la_forward for callers that cannot allocate device
 * memory during the call: code running inside an allocator or out-of-memory
 * handler, under a memory pool whose policy forbids growth, or in a setting
 * where cudaMalloc / cudaMallocAsync would deadlock or be refused.  It
 * allocates nothing: the per-segment states that la_forward takes from
 * its stream-ordered pool live in a fixed scratch array of 4 Mi floats (16 MiB),
 * which every GPU that loads the library holds until the process exits.
 * The method is the same as la_forward; the pages have no counterpart of
 * this entry point, it only changes where the temporary states live.
 *
 *   Arguments, output and validation are those of la_forward.
 *   Segments are planned as for la_forward, then merged (fewer, longer
 *   segments, so less parallelism) until their states fit the scratch.  A
 *   request whose states do not fit even as one segment per head (a
 *   non-causal call with B·H·2·(d'·d + d') > 4 Mi floats) returns
 *   LA_ERR_UNSUPPORTED and queues nothing.  Causal requests that fit in one
 *   segment per head use no scratch at all.
 *   The first call on a device looks up the scratch array's device address
 *   (cudaGetSymbolAddress) once; later calls reuse it.
 *   Every call overwrites the part of the scratch it uses and nothing needs
 *   to be zeroed, but all calls share the one array: calls that overlap on
 *   the GPU (e.g. on two streams) race on it and give wrong results.
 *   Serialise them (one stream, or events).
 */
la_status la_forward_noalloc(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                             const float* decay_a, la_feature_map feature_map,
                             const la_tensor* omega, int causal, la_tensor* out,
                             la_stream stream);

/*
 * la_launch_count — instrumentation: the number of CUDA kernels this process
 * has queued through the library so far (all devices, all entry points).
 * The difference across a region counts the library's own launches in it.
 * Host-only; never fails.  No counterpart on the pages: it exists so that
 * benchmarks can report how many of this library's kernels they timed.
 */
uint64_t la_launch_count(void);

/*
 * la_selftest_wait_timeout — test hook for the failure path of the bounded
 * waits.  Queues on `stream` one small kernel that runs the same bounded
 * wait the tensor-core kernels use (single-thread and whole-warp forms) on a
 * shared-memory barrier that nothing ever signals, with a limit of
 * `limit_ns` nanoseconds (1 000 … 100 000 000).  The waits give up, record
 * LA_ERR_TIMEOUT in the device status word and the kernel exits normally: no
 * trap, no fault, no hang.  A following la_get_last_device_status(stream)
 * returns LA_ERR_TIMEOUT (and clears the word).  Returns LA_ERR_INVALID_ARG
 * for a limit outside the range (nothing queued), LA_ERR_CUDA if the launch
 * fails, else LA_OK.  No counterpart on the pages.
 */
la_status la_selftest_wait_timeout(uint64_t limit_ns, la_stream stream);

/*
 * The LA_DEBUG build.  Compiled with -DLA_DEBUG (`python -m
 * causal_kernelized_linear_gb300.build --debug`, into a library of its own),
 * the kernels check the indices, workspace slots and TMA coordinates they are
 * about to use — that a tile's first row lies in the CTA's token range, that
 * an output row lies inside the tensor, that a workspace slot belongs to the
 * head, that a TMA store starts at a non-negative row.  A failed check
 * records LA_ERR_DEVICE_CHECK and the check's site number in the device
 * status word (the first error of either kind wins) and skips the access;
 * nothing traps.  Kernels waiting on a skipped load then give up through
 * their bounded waits.  The release build compiles the checks away and
 * otherwise runs the same arithmetic, so both give identical results.
 *
 * la_debug_build — 1 in the LA_DEBUG build, 0 otherwise.  Never fails.
 */
int la_debug_build(void);

/*
 * la_get_last_device_check — la_get_last_device_status that also reports,
 * in *site, the site number of the first failed check when the status is
 * LA_ERR_DEVICE_CHECK (0 otherwise).  Synchronises `stream`, then clears the
 * word.  Site numbers: 11–14 the tcgen05 elu+1 forward (tile rows, output
 * rows, the aggregate slot, the entering-state slots), 21–26 the tcgen05
 * backward (item ranges of the loads, rows of the ∂q, ∂k, ∂v stores), 31–32
 * the non-causal readout, 41–42 the Performer forward, 90 the self-test.
 * Errors: LA_ERR_INVALID_ARG (site is NULL), LA_ERR_CUDA.
 */
la_status la_get_last_device_check(la_stream stream, int* site);

/*
 * la_selftest_device_check — test hook for the LA_DEBUG checks.  Queues one
 * small kernel whose guarded access has an index one past its 4-element
 * shared-memory buffer: the check fails, records LA_ERR_DEVICE_CHECK with
 * site 90 and the access is skipped (the index is also masked into the
 * buffer, so no build can touch memory outside it).  A following
 * la_get_last_device_check(stream, &site) returns LA_ERR_DEVICE_CHECK and
 * site 90.  Returns LA_ERR_UNSUPPORTED in the release build (nothing
 * queued), LA_ERR_CUDA if the launch fails, else LA_OK.
 */
la_status la_selftest_device_check(la_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H */
