// C ABI of liblinattn (declared in include/linattn.h): argument validation,
// path selection, segment planning and workspace, device status word.
#include "linattn.h"

#include "common.cuh"
#include "internal.h"

#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <cstdint>
#include <mutex>

namespace la {

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

void count_launches(int k) { g_launches.fetch_add((uint64_t)k, std::memory_order_relaxed); }

namespace {
bool nvtx_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("LA_NVTX");
    return e != nullptr && *e != '\0' && std::strcmp(e, "0") != 0;
  }();
  return on;
}
}  // namespace

ApiRange::ApiRange(const char* name) : on_(nvtx_enabled()) {
  if (on_) nvtxRangePushA(name);
}
ApiRange::~ApiRange() {
  if (on_) nvtxRangePop();
}

namespace {

// Per-device status word: [0] the first error a kernel recorded (a bounded
// wait that expired; in LA_DEBUG builds also a failed device-side check),
// [1] the site number of a failed check.
__device__ int g_device_status[2];

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  int* status = nullptr;  // device address of g_device_status[0]
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

la_status device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return LA_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return LA_ERR_CUDA;
    di.num_sms = sms;
    di.status = static_cast<int*>(p);
    di.ready = true;
  }
  *out = di;
  return LA_OK;
}

// Workspace memory: stream-ordered allocations from one pool per device owned
// by the library.  The pool keeps what it has reserved (unlimited release
// threshold), so repeated calls reuse the same device memory instead of
// mapping and unmapping it at every synchronisation; the reservation is the
// largest workspace that calls had in flight at once, held until exit.
cudaMemPool_t g_pool[kMaxDevices] = {};

cudaError_t ws_alloc(void** p, size_t bytes, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_pool[dev]) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t np;
      if ((e = cudaMemPoolCreate(&np, &props)) != cudaSuccess) return e;
      uint64_t keep = UINT64_MAX;
      if ((e = cudaMemPoolSetAttribute(np, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
        cudaMemPoolDestroy(np);
        return e;
      }
      g_pool[dev] = np;
    }
    pool = g_pool[dev];
  }
  return cudaMallocFromPoolAsync(p, bytes, pool, s);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype(la_dtype t) { return t == LA_BF16 || t == LA_F32; }

bool same_shape(const la_tensor* a, const la_tensor* b) {
  return a->B == b->B && a->H == b->H && a->n == b->n && a->d == b->d;
}

bool supported_width(int64_t d) { return d == 32 || d == 64 || d == 128; }

bool supported_features(int64_t m) { return m == 64 || m == 128 || m == 256; }

// Checks shared by la_forward and la_forward_with_state; fills `a`.
la_status validate_forward(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                           const float* decay_a, la_feature_map fm, const la_tensor* omega,
                           int causal, la_tensor* out, FwdArgs* a) {
  if (!q || !k || !v || !out) return LA_ERR_INVALID_ARG;
  if (!valid_dtype(q->dtype) || k->dtype != q->dtype || v->dtype != q->dtype ||
      out->dtype != q->dtype)
    return LA_ERR_INVALID_ARG;
  if (!same_shape(q, k) || !same_shape(q, v) || !same_shape(q, out)) return LA_ERR_INVALID_ARG;
  if (q->B < 1 || q->H < 1 || q->n < 0 || q->d < 1) return LA_ERR_INVALID_ARG;
  if (q->B > (int64_t)1 << 24 || q->H > (int64_t)1 << 16 || q->n > (int64_t)1 << 31)
    return LA_ERR_UNSUPPORTED;
  if (!supported_width(q->d)) return LA_ERR_UNSUPPORTED;
  if (fm != LA_FM_ELU1 && fm != LA_FM_PERFORMER) return LA_ERR_INVALID_ARG;
  if (!causal && decay_a) return LA_ERR_UNSUPPORTED;  // eq (6) carries no decay
  const int64_t elems = q->B * q->H * q->n * q->d;
  if (elems > 0) {
    if (!q->data || !k->data || !v->data || !out->data) return LA_ERR_INVALID_ARG;
    if (!aligned16(q->data) || !aligned16(k->data) || !aligned16(v->data) ||
        !aligned16(out->data))
      return LA_ERR_INVALID_ARG;
  }
  if (decay_a && (reinterpret_cast<uintptr_t>(decay_a) & 3u)) return LA_ERR_INVALID_ARG;
  int m = 0;
  if (fm == LA_FM_PERFORMER) {
    if (!omega || !omega->data) return LA_ERR_INVALID_ARG;
    if (omega->dtype != q->dtype || omega->B != 1 || omega->H != 1 || omega->n != q->d)
      return LA_ERR_INVALID_ARG;
    if (!aligned16(omega->data)) return LA_ERR_INVALID_ARG;
    if (!supported_features(omega->d)) return LA_ERR_UNSUPPORTED;
    m = (int)omega->d;
  } else if (omega) {
    return LA_ERR_INVALID_ARG;
  }
  a->q = q->data;
  a->k = k->data;
  a->v = v->data;
  a->out = out->data;
  a->decay = decay_a;
  a->tok_decay = nullptr;
  a->tok_weight = nullptr;
  a->ws_ld = nullptr;
  a->ws_tok = nullptr;
  a->omega = omega ? omega->data : nullptr;
  a->B = q->B;
  a->H = q->H;
  a->n = q->n;
  a->d = (int)q->d;
  a->m = m;
  a->dp = fm == LA_FM_PERFORMER ? m : (int)q->d;
  a->bf16 = q->dtype == LA_BF16;
  a->performer = fm == LA_FM_PERFORMER;
  a->causal = causal != 0;
  a->mu_out = nullptr;
  a->nu_out = nullptr;
  a->init_state = nullptr;
  a->init_z = nullptr;
  return LA_OK;
}

// [p, p + bytes) and [q, q + bytes2) share a byte
bool overlaps(const void* p, size_t bytes, const void* q, size_t bytes2) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), b0 = reinterpret_cast<uintptr_t>(q);
  return a0 < b0 + bytes2 && b0 < a0 + bytes;
}

// Cut every head into segments so that all CTAs fit in one wave
// (num_sms · ctas_per_sm); with more heads than that, one segment per head.
SegmentPlan plan_segments(int64_t BH, int64_t n, int num_sms, int64_t granule,
                          int ctas_per_sm) {
  SegmentPlan p;
  const int64_t target = (int64_t)num_sms * ctas_per_sm;
  int64_t g = target / BH;
  const int64_t max_g = std::max<int64_t>(1, (n + granule - 1) / granule);
  g = std::max<int64_t>(1, std::min(g, max_g));
  int64_t len = (n + g - 1) / g;
  len = ((len + granule - 1) / granule) * granule;
  p.seg_len = std::max<int64_t>(len, granule);
  p.nseg = (int)std::max<int64_t>(1, (n + p.seg_len - 1) / p.seg_len);
  return p;
}

la_status to_status(cudaError_t e) {
  if (e == cudaSuccess) return LA_OK;
  if (e == cudaErrorMemoryAllocation) return LA_ERR_OUT_OF_MEMORY;
  return LA_ERR_CUDA;
}

// Kernel family for a validated request and its segment plan: the tcgen05
// path for what it supports, the fp32 CUDA-core path otherwise.
struct PathPlan {
  bool tensor_cores;
  SegmentPlan plan;
  int64_t granule;
};

PathPlan choose_path(const FwdArgs& a) {
  PathPlan pp;
  pp.tensor_cores = tc_forward_supported(a) || tc_performer_supported(a) || tc_readout_supported(a);
  // tcgen05 path: one 512-thread CTA per SM, 128-token chunks; CUDA-core
  // path: two CTAs per SM, 32-token chunks
  pp.granule = pp.tensor_cores ? tc_segment_granule() : 32;
  pp.plan = plan_segments(a.B * a.H, a.n, a.num_sms, pp.granule, pp.tensor_cores ? 1 : 2);
  return pp;
}

cudaError_t dispatch_forward(const FwdArgs& a, const PathPlan& pp, cudaStream_t stream,
                             float* ws_state, float* ws_z, float* tot_state, float* tot_z) {
  if (pp.tensor_cores && a.performer)
    return tc_performer_forward(a, stream, ws_state, ws_z, tot_state, tot_z, pp.plan);
  if (pp.tensor_cores && !a.causal)
    return tc_noncausal_forward(a, stream, ws_state, ws_z, tot_state, tot_z, pp.plan);
  if (pp.tensor_cores) return tc_forward(a, stream, ws_state, ws_z, tot_state, tot_z, pp.plan);
  return simt_forward(a, stream, ws_state, ws_z, tot_state, tot_z, pp.plan);
}

la_status run_forward(FwdArgs& a, cudaStream_t stream) {
  DeviceInfo di;
  la_status st = device_info(&di);
  if (st != LA_OK) return st;
  a.status = di.status;
  a.num_sms = di.num_sms;
  const int64_t BH = a.B * a.H;
  const size_t state_elems = (size_t)a.dp * a.d;
  if (a.n == 0) {
    // empty sequence: nothing to write but the state, which is the initial
    // one (zero when none is given)
    if (a.init_state) {
      if (a.mu_out && cudaMemcpyAsync(a.mu_out, a.init_state, BH * state_elems * sizeof(float),
                                      cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
        return LA_ERR_CUDA;
      if (a.nu_out && cudaMemcpyAsync(a.nu_out, a.init_z, BH * a.dp * sizeof(float),
                                      cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
        return LA_ERR_CUDA;
      return LA_OK;
    }
    if (a.mu_out && cudaMemsetAsync(a.mu_out, 0, BH * state_elems * sizeof(float), stream) != cudaSuccess)
      return LA_ERR_CUDA;
    if (a.nu_out && cudaMemsetAsync(a.nu_out, 0, BH * a.dp * sizeof(float), stream) != cudaSuccess)
      return LA_ERR_CUDA;
    return LA_OK;
  }
  const PathPlan pp = choose_path(a);
  const SegmentPlan& plan = pp.plan;
  // state slots per head: one per segment; the causal elu+1 tensor-core path
  // keeps an initial state in one more, ahead of the segments' aggregates
  const int slots = plan.nseg + ((a.init_state && tc_forward_supported(a)) ? 1 : 0);
  const bool need_ws = !a.causal || slots > 1;
  // the inclusive total is an input of the non-causal readout; the causal
  // paths write the final state only when the caller asks for it
  const bool need_tot = !a.causal && (a.mu_out == nullptr);
  size_t ws_floats = 0;
  if (need_ws) ws_floats += (size_t)BH * slots * (state_elems + a.dp);
  if (need_tot) ws_floats += (size_t)BH * (state_elems + a.dp);
  // per-token decay: the log2 decay of every segment, beside its aggregate
  const bool need_ld = a.tok_decay != nullptr && plan.nseg > 1;
  if (need_ld) ws_floats += (size_t)BH * plan.nseg;
  // per-token decay on the tensor-core elu+1 path: the per-token chunk prefixes
  const bool need_tok = a.tok_decay != nullptr && tc_forward_supported(a);
  const size_t tok_at = ws_floats + (need_tok ? (4 - ws_floats % 4) % 4 : 0);   // 16-byte aligned
  if (need_tok) ws_floats = tok_at + 2 * (size_t)BH * a.n;
  float* ws = nullptr;
  if (ws_floats) {
    cudaError_t e = ws_alloc(reinterpret_cast<void**>(&ws), ws_floats * sizeof(float), stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return e == cudaErrorMemoryAllocation ? LA_ERR_OUT_OF_MEMORY : LA_ERR_CUDA;
    }
  }
  float* ws_state = ws;
  float* ws_z = ws ? ws + (size_t)BH * slots * state_elems : nullptr;
  float* tot_state = a.mu_out;
  float* tot_z = a.nu_out;
  if (need_tot) {
    tot_state = ws + (size_t)BH * slots * (state_elems + a.dp);
    tot_z = tot_state + (size_t)BH * state_elems;
  }
  if (need_ld) a.ws_ld = ws + (size_t)BH * slots * (state_elems + a.dp);
  if (need_tok) a.ws_tok = ws + tok_at;
  cudaError_t e = dispatch_forward(a, pp, stream, ws_state, ws_z, tot_state, tot_z);
  if (ws) {
    cudaError_t f = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = f;
  }
  return to_status(e);
}

// The final state from zero without the outputs: the aggregate of every
// segment, then their decayed sum (segment_total) into mu_out / nu_out.
la_status run_state(FwdArgs& a, cudaStream_t stream) {
  DeviceInfo di;
  la_status st = device_info(&di);
  if (st != LA_OK) return st;
  a.status = di.status;
  a.num_sms = di.num_sms;
  const int64_t BH = a.B * a.H;
  const size_t state_elems = (size_t)a.dp * a.d;
  if (a.n == 0) {
    if (cudaMemsetAsync(a.mu_out, 0, BH * state_elems * sizeof(float), stream) != cudaSuccess ||
        cudaMemsetAsync(a.nu_out, 0, BH * a.dp * sizeof(float), stream) != cudaSuccess)
      return LA_ERR_CUDA;
    return LA_OK;
  }
  const PathPlan pp = choose_path(a);
  const SegmentPlan& plan = pp.plan;
  float* ws = nullptr;
  const size_t ws_floats = (size_t)BH * plan.nseg * (state_elems + a.dp);
  cudaError_t e = ws_alloc(reinterpret_cast<void**>(&ws), ws_floats * sizeof(float), stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? LA_ERR_OUT_OF_MEMORY : LA_ERR_CUDA;
  }
  float* ws_state = ws;
  float* ws_z = ws + (size_t)BH * plan.nseg * state_elems;
  if (pp.tensor_cores && a.performer) e = tc_performer_state_only(a, stream, ws_state, ws_z, plan);
  else if (pp.tensor_cores) e = tc_state_only(a, stream, ws_state, ws_z, plan);
  else e = simt_state_only(a, stream, ws_state, ws_z, plan);
  if (e == cudaSuccess)
    e = segment_total(ws_state, ws_z, a.mu_out, a.nu_out, BH, a.H, plan.nseg, plan.seg_len, a.n,
                      a.dp, a.d, a.decay, nullptr, stream, false);
  const cudaError_t f = cudaFreeAsync(ws, stream);
  if (e == cudaSuccess) e = f;
  return to_status(e);
}

// Copy streams of the host-buffer forward (one per input tensor and one for
// the output), per device, created on first use and kept until exit.
struct HostStreams {
  cudaStream_t in[3] = {nullptr, nullptr, nullptr};
  cudaStream_t out = nullptr;
};
HostStreams g_hs[kMaxDevices];

cudaError_t host_streams(HostStreams* hs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_hs[dev].out) {
    HostStreams n;
    cudaStream_t* all[4] = {&n.in[0], &n.in[1], &n.in[2], &n.out};
    for (int i = 0; i < 4; ++i) {
      if ((e = cudaStreamCreateWithFlags(all[i], cudaStreamNonBlocking)) != cudaSuccess) {
        for (int j = 0; j < i; ++j) cudaStreamDestroy(*all[j]);
        return e;
      }
    }
    g_hs[dev] = n;
  }
  *hs = g_hs[dev];
  return cudaSuccess;
}

// Page-locked host memory (cudaHostAlloc / cudaHostRegister).
bool pinned_host(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost;
}

// la_forward on page-locked host buffers (validated into `a`, whose data
// pointers are host pointers), in up to eight pieces whose copies overlap
// the compute of the others:
//   causal, n ≥ 2048: pieces along the sequence; piece g's rows of q, k, v
//     go to dense device staging (one strided copy per tensor), its forward
//     continues from the state piece g − 1 ended with (la_forward_from_state's
//     path), and its rows of o go back with one strided copy;
//   otherwise: groups of heads along B (or H when B = 1), each a forward of
//     its own.
// The q, k, v copies run on three copy-in streams and start at once (the
// staging is taken on the first of them, so they need not wait for the work
// already on `stream`); each piece's compute waits for its copies on
// `stream`, its output copy waits for its compute on the copy-out stream,
// and `stream` resumes after the last output copy, where the staging goes
// back to the pool.
la_status run_forward_host(FwdArgs& a, const float* decay_host, const void* omega_host,
                           size_t omega_bytes, cudaStream_t stream) {
  HostStreams hs;
  if (host_streams(&hs) != cudaSuccess) return LA_ERR_CUDA;
  const size_t esize = a.bf16 ? 2 : 4;
  const int64_t BH = a.B * a.H;
  const size_t row_bytes = (size_t)a.d * esize;
  const size_t tensor_bytes = (size_t)BH * a.n * row_bytes;
  const size_t decay_bytes = decay_host ? (size_t)a.H * sizeof(float) : 0;
  const bool by_seq = a.causal && a.n >= 2048;
  const size_t state_floats = (size_t)BH * ((size_t)a.dp * a.d + a.dp);
  auto round16 = [](size_t x) { return (x + 15) & ~(size_t)15; };
  const size_t states_bytes = by_seq ? 2 * round16(state_floats * sizeof(float)) : 0;
  const size_t total =
      4 * round16(tensor_bytes) + round16(omega_bytes) + round16(decay_bytes) + states_bytes;
  char* stg = nullptr;
  cudaError_t e = ws_alloc(reinterpret_cast<void**>(&stg), total, hs.in[0]);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? LA_ERR_OUT_OF_MEMORY : LA_ERR_CUDA;
  }
  char* dbuf[4];   // q, k, v, o staging
  for (int i = 0; i < 4; ++i) dbuf[i] = stg + i * round16(tensor_bytes);
  char* domega = stg + 4 * round16(tensor_bytes);
  float* ddecay = reinterpret_cast<float*>(domega + round16(omega_bytes));
  float* dstate[2];
  dstate[0] = reinterpret_cast<float*>(reinterpret_cast<char*>(ddecay) + round16(decay_bytes));
  dstate[1] = reinterpret_cast<float*>(reinterpret_cast<char*>(dstate[0]) +
                                       round16(state_floats * sizeof(float)));
  const char* hin[3] = {static_cast<const char*>(a.q), static_cast<const char*>(a.k),
                        static_cast<const char*>(a.v)};
  char* hout = static_cast<char*>(a.out);
  la_status st = LA_OK;
  auto ok = [&](cudaError_t r) {
    if (r != cudaSuccess && st == LA_OK) st = LA_ERR_CUDA;
    return r == cudaSuccess;
  };
  if (omega_bytes) ok(cudaMemcpyAsync(domega, omega_host, omega_bytes, cudaMemcpyHostToDevice, hs.in[0]));
  if (decay_bytes) ok(cudaMemcpyAsync(ddecay, decay_host, decay_bytes, cudaMemcpyHostToDevice, hs.in[0]));
  // the other copy-in streams may use the staging once it is allocated
  cudaEvent_t ev_alloc = nullptr;
  if (ok(cudaEventCreateWithFlags(&ev_alloc, cudaEventDisableTiming))) {
    ok(cudaEventRecord(ev_alloc, hs.in[0]));
    ok(cudaStreamWaitEvent(hs.in[1], ev_alloc, 0));
    ok(cudaStreamWaitEvent(hs.in[2], ev_alloc, 0));
    cudaEventDestroy(ev_alloc);
  }
  // pieces: rows [t0, t1) of every head (by_seq), or heads [u0, u1)
  const int64_t outer = by_seq ? a.n : (a.B > 1 ? a.B : a.H);
  int64_t npieces = by_seq ? std::min<int64_t>(8, a.n / 1024) : std::min<int64_t>(outer, 8);
  int64_t piece_len = (outer + npieces - 1) / npieces;
  if (by_seq) piece_len = (piece_len + 127) / 128 * 128;
  npieces = (outer + piece_len - 1) / piece_len;
  const size_t unit_bytes = by_seq ? row_bytes : (a.B > 1 ? (size_t)a.H : 1) * a.n * row_bytes;
  for (int64_t gi = 0; gi < npieces && st == LA_OK; ++gi) {
    const int64_t u0 = gi * piece_len, u1 = std::min(outer, u0 + piece_len);
    cudaEvent_t ev_in[3] = {nullptr, nullptr, nullptr}, ev_comp = nullptr;
    bool made = ok(cudaEventCreateWithFlags(&ev_comp, cudaEventDisableTiming));
    for (int i = 0; i < 3 && made; ++i) made = ok(cudaEventCreateWithFlags(&ev_in[i], cudaEventDisableTiming));
    if (!made) {
      for (int i = 0; i < 3; ++i)
        if (ev_in[i]) cudaEventDestroy(ev_in[i]);
      if (ev_comp) cudaEventDestroy(ev_comp);
      break;
    }
    // dense staging of the piece: [BH][u1 − u0 rows] (by_seq) or its heads
    const size_t off = by_seq ? (size_t)BH * u0 * row_bytes : (size_t)u0 * unit_bytes;
    const size_t width = (size_t)(u1 - u0) * unit_bytes;
    for (int i = 0; i < 3; ++i) {
      if (by_seq)
        ok(cudaMemcpy2DAsync(dbuf[i] + off, width, hin[i] + (size_t)u0 * row_bytes,
                             (size_t)a.n * row_bytes, width, (size_t)BH, cudaMemcpyHostToDevice,
                             hs.in[i]));
      else
        ok(cudaMemcpyAsync(dbuf[i] + off, hin[i] + off, width, cudaMemcpyHostToDevice, hs.in[i]));
      ok(cudaEventRecord(ev_in[i], hs.in[i]));
      ok(cudaStreamWaitEvent(stream, ev_in[i], 0));
    }
    if (st == LA_OK) {
      FwdArgs g = a;
      g.q = dbuf[0] + off;
      g.k = dbuf[1] + off;
      g.v = dbuf[2] + off;
      g.out = dbuf[3] + off;
      g.omega = omega_bytes ? domega : nullptr;
      g.decay = decay_bytes ? ddecay : nullptr;
      g.mu_out = nullptr;
      g.nu_out = nullptr;
      g.init_state = nullptr;
      g.init_z = nullptr;
      if (by_seq) {
        g.n = u1 - u0;
        // the state piece gi − 1 ended with, into piece gi; every piece but
        // the last leaves its own in the other buffer
        const size_t zoff = (size_t)BH * a.dp * a.d;
        if (gi > 0) {
          g.init_state = dstate[(gi - 1) & 1];
          g.init_z = dstate[(gi - 1) & 1] + zoff;
        }
        if (gi + 1 < npieces) {
          g.mu_out = dstate[gi & 1];
          g.nu_out = dstate[gi & 1] + zoff;
        }
      } else if (a.B > 1) {
        g.B = u1 - u0;
      } else {
        g.H = u1 - u0;
        g.decay = decay_bytes ? ddecay + u0 : nullptr;
      }
      const la_status fs = run_forward(g, stream);
      if (fs != LA_OK) st = fs;
    }
    ok(cudaEventRecord(ev_comp, stream));
    ok(cudaStreamWaitEvent(hs.out, ev_comp, 0));
    if (by_seq)
      ok(cudaMemcpy2DAsync(hout + (size_t)u0 * row_bytes, (size_t)a.n * row_bytes, dbuf[3] + off,
                           width, width, (size_t)BH, cudaMemcpyDeviceToHost, hs.out));
    else
      ok(cudaMemcpyAsync(hout + off, dbuf[3] + off, width, cudaMemcpyDeviceToHost, hs.out));
    for (int i = 0; i < 3; ++i) cudaEventDestroy(ev_in[i]);
    cudaEventDestroy(ev_comp);
  }
  // the caller's stream resumes after the last copy out; the staging goes
  // back to the pool after every use of it
  cudaEvent_t ev_done = nullptr;
  bool waited = false;
  if (cudaEventCreateWithFlags(&ev_done, cudaEventDisableTiming) == cudaSuccess) {
    waited = cudaEventRecord(ev_done, hs.out) == cudaSuccess &&
             cudaStreamWaitEvent(stream, ev_done, 0) == cudaSuccess;
    cudaEventDestroy(ev_done);
  }
  if (!waited) {
    // order the release behind the copy streams the slow way
    cudaStreamSynchronize(hs.out);
    for (int i = 0; i < 3; ++i) cudaStreamSynchronize(hs.in[i]);
    st = LA_ERR_CUDA;
  }
  if (cudaFreeAsync(stg, stream) != cudaSuccess && st == LA_OK) st = LA_ERR_CUDA;
  return st;
}

}  // namespace

// Forward into a workspace of `ws_floats` floats obtained from `get_ws`
// after validation (no allocation).  Segments are planned as for la_forward,
// then reduced until the per-segment states fit; a request whose smallest
// plan does not fit is rejected with LA_ERR_UNSUPPORTED before anything is
// queued.
la_status forward_in_workspace(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                               const float* decay_a, la_feature_map feature_map,
                               const la_tensor* omega, int causal, la_tensor* out,
                               la_status (*get_ws)(float**), size_t ws_floats,
                               cudaStream_t stream) {
  FwdArgs a;
  la_status st = validate_forward(q, k, v, decay_a, feature_map, omega, causal, out, &a);
  if (st != LA_OK) return st;
  DeviceInfo di;
  st = device_info(&di);
  if (st != LA_OK) return st;
  a.status = di.status;
  a.num_sms = di.num_sms;
  if (a.n == 0) return LA_OK;
  const int64_t BH = a.B * a.H;
  const size_t per_state = (size_t)a.dp * a.d + a.dp;
  PathPlan pp = choose_path(a);
  SegmentPlan& plan = pp.plan;
  auto need = [&](const SegmentPlan& p) -> size_t {
    const bool use_ws = !a.causal || p.nseg > 1;
    if (!use_ws) return 0;
    return (size_t)BH * per_state * (size_t)p.nseg + (a.causal ? 0 : (size_t)BH * per_state);
  };
  while (need(plan) > ws_floats && plan.nseg > 1) {
    const int g = plan.nseg - 1;
    int64_t len = (a.n + g - 1) / g;
    len = ((len + pp.granule - 1) / pp.granule) * pp.granule;
    plan.seg_len = len;
    plan.nseg = (int)((a.n + len - 1) / len);
  }
  if (need(plan) > ws_floats) return LA_ERR_UNSUPPORTED;
  float* ws = nullptr;
  if (need(plan) > 0) {
    st = get_ws(&ws);
    if (st != LA_OK) return st;
  }
  const size_t state_elems = (size_t)a.dp * a.d;
  float* ws_state = ws;
  float* ws_z = ws ? ws + (size_t)BH * plan.nseg * state_elems : nullptr;
  float* tot_state = nullptr;
  float* tot_z = nullptr;
  if (!a.causal) {
    tot_state = ws + (size_t)BH * plan.nseg * per_state;
    tot_z = tot_state + (size_t)BH * state_elems;
  }
  return to_status(dispatch_forward(a, pp, stream, ws_state, ws_z, tot_state, tot_z));
}

}  // namespace la

extern "C" {

la_status la_forward(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                     const float* decay_a, la_feature_map feature_map,
                     const la_tensor* omega, int causal, la_tensor* out, la_stream stream) {
  la::ApiRange range_("la_forward");
  la::FwdArgs a;
  la_status st = la::validate_forward(q, k, v, decay_a, feature_map, omega, causal, out, &a);
  if (st != LA_OK) return st;
  return la::run_forward(a, reinterpret_cast<cudaStream_t>(stream));
}

la_status la_forward_host(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                          const float* decay_a, la_feature_map feature_map, const la_tensor* omega,
                          int causal, la_tensor* out, la_stream stream) {
  la::ApiRange range_("la_forward_host");
  la::FwdArgs a;
  la_status st = la::validate_forward(q, k, v, decay_a, feature_map, omega, causal, out, &a);
  if (st != LA_OK) return st;
  if (a.B * a.H * a.n * a.d == 0) return LA_OK;
  // every host array must be page-locked (the copies are asynchronous)
  if (!la::pinned_host(a.q) || !la::pinned_host(a.k) || !la::pinned_host(a.v) ||
      !la::pinned_host(a.out) || (decay_a && !la::pinned_host(decay_a)) ||
      (a.omega && !la::pinned_host(a.omega)))
    return LA_ERR_INVALID_ARG;
  const size_t omega_bytes = a.omega ? (size_t)a.d * a.m * (a.bf16 ? 2 : 4) : 0;
  return la::run_forward_host(a, decay_a, a.omega, omega_bytes,
                              reinterpret_cast<cudaStream_t>(stream));
}

la_status la_forward_from_state(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                                const float* decay_a, la_feature_map feature_map,
                                const la_tensor* omega, const float* mu0, const float* nu0,
                                la_tensor* out, float* mu_out, float* nu_out, la_stream stream) {
  la::ApiRange range_("la_forward_from_state");
  la::FwdArgs a;
  la_status st = la::validate_forward(q, k, v, decay_a, feature_map, omega, 1, out, &a);
  if (st != LA_OK) return st;
  if ((mu0 == nullptr) != (nu0 == nullptr) || (mu_out == nullptr) != (nu_out == nullptr))
    return LA_ERR_INVALID_ARG;
  const size_t BH = (size_t)(a.B * a.H);
  const size_t sbytes = BH * (size_t)a.dp * a.d * sizeof(float);
  const size_t zbytes = BH * (size_t)a.dp * sizeof(float);
  if (mu0 && (!la::aligned16(mu0) || !la::aligned16(nu0))) return LA_ERR_INVALID_ARG;
  if (mu_out && (!la::aligned16(mu_out) || !la::aligned16(nu_out))) return LA_ERR_INVALID_ARG;
  if (mu0 && mu_out &&
      (la::overlaps(mu0, sbytes, mu_out, sbytes) || la::overlaps(mu0, sbytes, nu_out, zbytes) ||
       la::overlaps(nu0, zbytes, mu_out, sbytes) || la::overlaps(nu0, zbytes, nu_out, zbytes)))
    return LA_ERR_INVALID_ARG;
  a.init_state = mu0;
  a.init_z = nu0;
  a.mu_out = mu_out;
  a.nu_out = nu_out;
  return la::run_forward(a, reinterpret_cast<cudaStream_t>(stream));
}

la_status la_forward_state(const la_tensor* k, const la_tensor* v, const float* decay_a,
                           la_feature_map feature_map, const la_tensor* omega, float* mu_out,
                           float* nu_out, la_stream stream) {
  la::ApiRange range_("la_forward_state");
  if (!k || !v) return LA_ERR_INVALID_ARG;
  // the checks of la_forward, with k standing in for q and for the output
  la_tensor kk = *k;
  la::FwdArgs a;
  la_status st = la::validate_forward(&kk, k, v, decay_a, feature_map, omega, 1, &kk, &a);
  if (st != LA_OK) return st;
  if (!mu_out || !nu_out || !la::aligned16(mu_out) || !la::aligned16(nu_out))
    return LA_ERR_INVALID_ARG;
  a.q = nullptr;
  a.out = nullptr;
  a.mu_out = mu_out;
  a.nu_out = nu_out;
  return la::run_state(a, reinterpret_cast<cudaStream_t>(stream));
}

la_status la_forward_with_state(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                                const float* decay_a, la_feature_map feature_map,
                                const la_tensor* omega, int causal, la_tensor* out,
                                float* mu_out, float* nu_out, la_stream stream) {
  la::ApiRange range_("la_forward_with_state");
  la::FwdArgs a;
  la_status st = la::validate_forward(q, k, v, decay_a, feature_map, omega, causal, out, &a);
  if (st != LA_OK) return st;
  if (!mu_out || !nu_out || !la::aligned16(mu_out) || !la::aligned16(nu_out))
    return LA_ERR_INVALID_ARG;
  a.mu_out = mu_out;
  a.nu_out = nu_out;
  return la::run_forward(a, reinterpret_cast<cudaStream_t>(stream));
}

la_status la_forward_token_decay(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                                 const float* decay_a, const float* weight_b,
                                 la_feature_map feature_map, const la_tensor* omega,
                                 la_tensor* out, float* mu_out, float* nu_out, la_stream stream) {
  la::ApiRange range_("la_forward_token_decay");
  la::FwdArgs a;
  la_status st = la::validate_forward(q, k, v, nullptr, feature_map, omega, 1, out, &a);
  if (st != LA_OK) return st;
  if (q->B * q->H * q->n > 0 && !decay_a) return LA_ERR_INVALID_ARG;
  if (decay_a && (reinterpret_cast<uintptr_t>(decay_a) & 3u)) return LA_ERR_INVALID_ARG;
  if (weight_b && (reinterpret_cast<uintptr_t>(weight_b) & 3u)) return LA_ERR_INVALID_ARG;
  if ((mu_out == nullptr) != (nu_out == nullptr)) return LA_ERR_INVALID_ARG;
  if (mu_out && (!la::aligned16(mu_out) || !la::aligned16(nu_out))) return LA_ERR_INVALID_ARG;
  a.tok_decay = decay_a;
  a.tok_weight = weight_b;
  a.mu_out = mu_out;
  a.nu_out = nu_out;
  return la::run_forward(a, reinterpret_cast<cudaStream_t>(stream));
}

la_status la_backward(const la_tensor* q, const la_tensor* k, const la_tensor* v,
                      const float* decay_a, la_feature_map feature_map, const la_tensor* omega,
                      const la_tensor* grad_out, la_tensor* dq, la_tensor* dk, la_tensor* dv,
                      float* da, la_stream stream) {
  la::ApiRange range_("la_backward");
  la::FwdArgs f;
  // q, k, v, ω and the decay are checked as for the causal forward (with dq
  // standing in for the output)
  la_status st = la::validate_forward(q, k, v, decay_a, feature_map, omega, 1, dq, &f);
  if (st != LA_OK) return st;
  if (!grad_out || !dk || !dv) return LA_ERR_INVALID_ARG;
  for (const la_tensor* t : {grad_out, static_cast<const la_tensor*>(dk),
                             static_cast<const la_tensor*>(dv)}) {
    if (t->dtype != q->dtype || !la::same_shape(q, t)) return LA_ERR_INVALID_ARG;
    if (f.B * f.H * f.n > 0 && (!t->data || !la::aligned16(t->data))) return LA_ERR_INVALID_ARG;
  }
  if (da && !decay_a) return LA_ERR_INVALID_ARG;   // ∂a needs a decay to differentiate
  if (da && (reinterpret_cast<uintptr_t>(da) & 3u)) return LA_ERR_INVALID_ARG;
  if (!la::backward_supported(f.d, f.m, f.performer)) return LA_ERR_UNSUPPORTED;
  la::DeviceInfo di;
  st = la::device_info(&di);
  if (st != LA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (f.n == 0) {
    if (da && cudaMemsetAsync(da, 0, (size_t)f.H * sizeof(float), s) != cudaSuccess)
      return LA_ERR_CUDA;
    return LA_OK;
  }
  la::BwdArgs b;
  b.q = f.q;
  b.k = f.k;
  b.v = f.v;
  b.g = grad_out->data;
  b.dq = dq->data;
  b.dk = dk->data;
  b.dv = dv->data;
  b.decay = decay_a;
  b.da = da;
  b.omega = f.omega;
  b.B = f.B;
  b.H = f.H;
  b.n = f.n;
  b.d = f.d;
  b.m = f.m;
  b.dp = f.dp;
  b.bf16 = f.bf16;
  b.performer = f.performer;
  // tensor-core kernels (bf16, elu+1, d ∈ {64, 128}): per-chunk states;
  // CUDA-core kernels otherwise: 32-token chunks, two CTAs per SM
  const bool tc = la::tc_backward_supported(b);
  const la::SegmentPlan plan = la::plan_segments(f.B * f.H, f.n, di.num_sms, 32, 2);
  const size_t ws_floats = tc ? la::tc_backward_ws_floats(b) : la::backward_workspace_floats(b, plan);
  float* ws = nullptr;
  cudaError_t e = la::ws_alloc(reinterpret_cast<void**>(&ws), ws_floats * sizeof(float), s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? LA_ERR_OUT_OF_MEMORY : LA_ERR_CUDA;
  }
  e = tc ? la::tc_backward(b, ws, di.num_sms, di.status, s) : la::backward(b, ws, plan, s);
  cudaError_t fe = cudaFreeAsync(ws, s);
  if (e == cudaSuccess) e = fe;
  return la::to_status(e);
}

namespace la {
namespace {

// Checks shared by the decode entry points; fills everything in `a` but the
// decay fields.
la_status validate_decode(float* mu, float* nu, const la_tensor* q, const la_tensor* k,
                          const la_tensor* v, la_feature_map feature_map, const la_tensor* omega,
                          la_tensor* out, DecodeArgs* a) {
  if (!mu || !nu || !q || !k || !v || !out) return LA_ERR_INVALID_ARG;
  if (!valid_dtype(q->dtype) || k->dtype != q->dtype || v->dtype != q->dtype ||
      out->dtype != q->dtype)
    return LA_ERR_INVALID_ARG;
  if (!same_shape(q, k) || !same_shape(q, v) || !same_shape(q, out)) return LA_ERR_INVALID_ARG;
  if (q->B < 1 || q->H < 1 || q->n != 1) return LA_ERR_INVALID_ARG;
  if (q->B * q->H > ((int64_t)1 << 31) - 1) return LA_ERR_UNSUPPORTED;
  if (!supported_width(q->d)) return LA_ERR_UNSUPPORTED;
  if (!q->data || !k->data || !v->data || !out->data) return LA_ERR_INVALID_ARG;
  if (!aligned16(mu) || !aligned16(nu) || !aligned16(q->data) || !aligned16(k->data) ||
      !aligned16(v->data) || !aligned16(out->data))
    return LA_ERR_INVALID_ARG;
  int m = 0;
  if (feature_map == LA_FM_PERFORMER) {
    if (!omega || !omega->data) return LA_ERR_INVALID_ARG;
    if (omega->dtype != q->dtype || omega->B != 1 || omega->H != 1 || omega->n != q->d)
      return LA_ERR_INVALID_ARG;
    if (!aligned16(omega->data)) return LA_ERR_INVALID_ARG;
    if (!supported_features(omega->d)) return LA_ERR_UNSUPPORTED;
    m = (int)omega->d;
  } else if (feature_map == LA_FM_ELU1) {
    if (omega) return LA_ERR_INVALID_ARG;
  } else {
    return LA_ERR_INVALID_ARG;
  }
  a->mu = mu;
  a->nu = nu;
  a->q = q->data;
  a->k = k->data;
  a->v = v->data;
  a->out = out->data;
  a->decay = nullptr;
  a->weight = nullptr;
  a->per_token = false;
  a->omega = omega ? omega->data : nullptr;
  a->B = q->B;
  a->H = q->H;
  a->d = (int)q->d;
  a->m = m;
  a->bf16 = q->dtype == LA_BF16;
  a->performer = feature_map == LA_FM_PERFORMER;
  return LA_OK;
}

}  // namespace
}  // namespace la

la_status la_decode_step_token_decay(float* mu, float* nu, const la_tensor* q,
                                     const la_tensor* k, const la_tensor* v,
                                     const float* decay_a, const float* weight_b,
                                     la_feature_map feature_map, const la_tensor* omega,
                                     la_tensor* out, la_stream stream) {
  la::ApiRange range_("la_decode_step_token_decay");
  la::DecodeArgs a;
  la_status st = la::validate_decode(mu, nu, q, k, v, feature_map, omega, out, &a);
  if (st != LA_OK) return st;
  if (!decay_a || (reinterpret_cast<uintptr_t>(decay_a) & 3u)) return LA_ERR_INVALID_ARG;
  if (weight_b && (reinterpret_cast<uintptr_t>(weight_b) & 3u)) return LA_ERR_INVALID_ARG;
  a.decay = decay_a;
  a.weight = weight_b;
  a.per_token = true;
  return la::to_status(la::decode_step(a, reinterpret_cast<cudaStream_t>(stream)));
}

la_status la_decode_step_fm(float* mu, float* nu, const la_tensor* q, const la_tensor* k,
                            const la_tensor* v, const float* decay_a, la_feature_map feature_map,
                            const la_tensor* omega, la_tensor* out, la_stream stream) {
  la::ApiRange range_("la_decode_step_fm");
  la::DecodeArgs a;
  la_status st = la::validate_decode(mu, nu, q, k, v, feature_map, omega, out, &a);
  if (st != LA_OK) return st;
  if (decay_a && (reinterpret_cast<uintptr_t>(decay_a) & 3u)) return LA_ERR_INVALID_ARG;
  a.decay = decay_a;
  return la::to_status(la::decode_step(a, reinterpret_cast<cudaStream_t>(stream)));
}

la_status la_decode_step(float* mu, float* nu, const la_tensor* q, const la_tensor* k,
                         const la_tensor* v, const float* decay_a, la_tensor* out,
                         la_stream stream) {
  la::ApiRange range_("la_decode_step");
  return la_decode_step_fm(mu, nu, q, k, v, decay_a, LA_FM_ELU1, nullptr, out, stream);
}

static_assert(la::kStatusDeviceCheck == LA_ERR_DEVICE_CHECK, "device check status code");

const char* la_status_string(la_status status) {
  switch (status) {
    case LA_OK: return "LA_OK";
    case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG";
    case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED";
    case LA_ERR_CUDA: return "LA_ERR_CUDA";
    case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT";
    case LA_ERR_OUT_OF_MEMORY: return "LA_ERR_OUT_OF_MEMORY";
    case LA_ERR_DEVICE_CHECK: return "LA_ERR_DEVICE_CHECK";
  }
  return "LA_ERR_UNKNOWN";
}

uint64_t la_launch_count(void) { return la::g_launches.load(std::memory_order_relaxed); }

la_status la_selftest_wait_timeout(uint64_t limit_ns, la_stream stream) {
  la::ApiRange range_("la_selftest_wait_timeout");
  if (limit_ns < 1000ull || limit_ns > 100000000ull) return LA_ERR_INVALID_ARG;
  la::DeviceInfo di;
  la_status st = la::device_info(&di);
  if (st != LA_OK) return st;
  return la::to_status(la::selftest_wait(di.status, limit_ns, reinterpret_cast<cudaStream_t>(stream)));
}

// Synchronises the stream, reads and clears the device status word; *site
// gets the site of a failed device-side check (0 if none).
static la_status read_device_status(la_stream stream, int* site) {
  la::DeviceInfo di;
  la_status st = la::device_info(&di);
  if (st != LA_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return LA_ERR_CUDA;
  int word[2] = {0, 0};
  if (cudaMemcpy(word, di.status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return LA_ERR_CUDA;
  if (site) *site = word[0] == la::kStatusDeviceCheck ? word[1] : 0;
  if (word[0] != 0 || word[1] != 0) {
    const int zero[2] = {0, 0};
    if (cudaMemcpy(di.status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return LA_ERR_CUDA;
  }
  return static_cast<la_status>(word[0]);
}

la_status la_get_last_device_status(la_stream stream) {
  la::ApiRange range_("la_get_last_device_status");
  return read_device_status(stream, nullptr);
}

la_status la_get_last_device_check(la_stream stream, int* site) {
  la::ApiRange range_("la_get_last_device_check");
  if (!site) return LA_ERR_INVALID_ARG;
  *site = 0;
  return read_device_status(stream, site);
}

int la_debug_build(void) {
#ifdef LA_DEBUG
  return 1;
#else
  return 0;
#endif
}

la_status la_selftest_device_check(la_stream stream) {
  la::ApiRange range_("la_selftest_device_check");
#ifdef LA_DEBUG
  la::DeviceInfo di;
  la_status st = la::device_info(&di);
  if (st != LA_OK) return st;
  return la::to_status(la::selftest_check(di.status, reinterpret_cast<cudaStream_t>(stream)));
#else
  (void)stream;
  return LA_ERR_UNSUPPORTED;
#endif
}

}  // extern "C"
