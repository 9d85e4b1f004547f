// Host side of the C ABI declared in include/la.h: argument validation,
// sequence segmentation, workspace layout and kernel dispatch. Nothing here
// allocates device memory or synchronises the stream.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "la_internal.cuh"
#include "la_variants.cuh"

namespace la {

// Set to LA_ERR_TIMEOUT by a kernel whose bounded wait gave up; read and
// cleared by la_device_status. One per device (module-scope device variable).
__device__ int g_la_device_status = 0;

namespace {

thread_local char g_last_error[256] = "";
std::atomic<int> g_path{LA_PATH_AUTO};
std::atomic<int> g_timeout_test{0};

la_status fail(la_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

la_status cuda_fail(cudaError_t e, const char* where) {
  return fail(LA_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e),
              cudaGetErrorString(e));
}

bool head_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Common size checks. Returns LA_OK and sets *empty when there is nothing to do.
la_status check_sizes(int B, int H, int N, int dk, int dv, la_dtype dtype,
                      float eps, bool* empty) {
  if (B < 0 || H < 0 || N < 0) return fail(LA_ERR_INVALID_ARG, "negative size B=%d H=%d N=%d", B, H, N);
  if (dtype != LA_F32 && dtype != LA_BF16) return fail(LA_ERR_UNSUPPORTED, "dtype %d not supported", (int)dtype);
  if (!head_ok(dk) || !head_ok(dv))
    return fail(LA_ERR_UNSUPPORTED, "head sizes dk=%d dv=%d not in {16,32,64,128}", dk, dv);
  if (!(eps >= 0.f) || isinf(eps)) return fail(LA_ERR_INVALID_ARG, "eps must be finite and >= 0");
  const long long BH = (long long)B * H;
  if (BH > 0x7fffffffLL) return fail(LA_ERR_INVALID_ARG, "B*H too large");
  const long long elems = BH * (long long)N * (dk > dv ? dk : dv);
  if (elems > (1LL << 40)) return fail(LA_ERR_INVALID_ARG, "problem too large");
  *empty = (BH == 0 || N == 0);
  return LA_OK;
}

// Workspace layout for a plan: [state records][reverse records][token scalars],
// each region 256-byte aligned.
struct WsLayout {
  size_t state_off, rev_off, tok_off, total;
};

WsLayout layout(long long BH, int N, int dk, int dv, const SegPlan& plan, bool backward) {
  WsLayout w{};
  const size_t rec = sizeof(float) * (size_t)record_slot_words(dk, dv) * (size_t)plan.P * (size_t)BH;
  // forward records: one per piece, or F per segment
  const size_t frec = plan.NP > 0 ? sizeof(float) * (size_t)record_slot_words(dk, dv) * (size_t)plan.NP
                                  : rec * (size_t)plan.F;
  w.state_off = 0;
  size_t off = align_up(frec, 256);
  if (backward) {
    w.rev_off = off;
    off += align_up(rec, 256);
    w.tok_off = off;
    off += align_up(sizeof(float) * 2 * (size_t)BH * (size_t)N, 256);
  }
  w.total = off;
  return w;
}

struct Span {
  int label;
  cudaEvent_t start, stop;
  bool closed;
};

std::mutex g_prof_mu;
std::atomic<bool> g_prof_on{false};
std::vector<Span> g_spans;
std::vector<cudaEvent_t> g_free_events;
std::atomic<long long> g_launches{0};

cudaEvent_t take_event() {
  if (!g_free_events.empty()) {
    cudaEvent_t e = g_free_events.back();
    g_free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return e;
}

void recycle_spans_locked() {
  for (Span& s : g_spans) {
    if (s.start) g_free_events.push_back(s.start);
    if (s.stop) g_free_events.push_back(s.stop);
  }
  g_spans.clear();
}

// Record `e` on `stream`; while the stream is being captured into a CUDA graph
// the record must be an external event-record node to take effect at replay.
void record_event(cudaEvent_t e, cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, stream, cudaEventRecordExternal);
  else
    cudaEventRecord(e, stream);
}

}  // namespace

void prof_begin(int label, cudaStream_t stream) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  Span s{label, take_event(), take_event(), false};
  if (s.start) record_event(s.start, stream);
  (void)cudaGetLastError();  // a failed record must not surface as a later launch error
  g_spans.push_back(s);
}

void prof_end(int label, cudaStream_t stream) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto it = g_spans.rbegin(); it != g_spans.rend(); ++it) {
    if (it->label == label && !it->closed) {
      if (it->stop) record_event(it->stop, stream);
      (void)cudaGetLastError();
      it->closed = true;
      return;
    }
  }
}

void note_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

la_status set_error(la_status s, const char* msg) { return fail(s, "%s", msg); }

int* device_status_ptr() {
  static std::mutex mu;
  static int* cache[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_la_device_status) == cudaSuccess)
      cache[dev] = static_cast<int*>(p);
    else
      (void)cudaGetLastError();
  }
  return cache[dev];
}

bool take_timeout_test() { return g_timeout_test.exchange(0) != 0; }

// Pick the number of segments per sequence. Cost model in units of one
// kSegGranule-token chunk: every CTA pays its chunks plus about one chunk of
// prologue (loading its starting state); CTAs run in waves of `slots`; the
// segment scan adds a little per segment, and `record_cost` per state record
// the costliest segment sums before its first chunk (P - 1 records causal,
// P non-causal). Pure function of the sizes, so the workspace query and the
// call agree.
static SegPlan plan_segments_cost(long long BH, int N, int slots, double record_cost, bool causal) {
  SegPlan best{1, N > 0 ? N : 1};
  if (BH <= 0 || N <= 0) return best;
  const int nch = (N + kSegGranule - 1) / kSegGranule;
  double best_cost = 1e300;
  for (int P = 1; P <= nch && P <= 4096; ++P) {
    const int L = (nch + P - 1) / P;           // chunks per segment
    if ((nch + L - 1) / L != P) continue;      // P not reachable with equal segments
    const long long ctas = BH * P;
    const long long waves = (ctas + slots - 1) / slots;
    const double cost = (double)waves * (L + 1) + 0.02 * P + record_cost * (causal ? P - 1 : P);
    if (cost < best_cost) {
      best_cost = cost;
      best.P = P;
      best.seg_len = L * kSegGranule;
    }
  }
  return best;
}

SegPlan plan_segments(long long BH, int N, int slots) { return plan_segments_cost(BH, N, slots, 0.0, true); }

// A state record summed at the start of a tensor-core chunk loop or backward
// sweep costs about half a chunk: one thread per state row reads it from L2
// with 16 loads in flight, ~2.1 us per 128 x 128 record against ~3.9 us per
// chunk with every SM streaming (measured at d = 128; a d = 64 record and
// chunk are both about half). With few heads the record sums decide the
// plan: one head of 32768 tokens in 128 segments of 2 chunks took 278 us in
// its chunk loop, 127 records for the last segment.
constexpr double kRecordCost = 0.5;

static SegPlan plan_segments_tc(long long BH, int N, bool causal) {
  return plan_segments_cost(BH, N, kSlots, kRecordCost, causal);
}

// The forward's segment plan (one CTA per SM for the output kernels). On the
// tensor-core path the state pass may split each segment over F CTAs (F
// records per segment) while it still fits in one CTA per SM: the output
// kernel's CTAs, which need a whole SM, start on the SMs the state pass
// leaves free (measured: a state pass spread over every SM delays them more
// than its shorter CTAs save).
// The causal tensor-core forward at d = 128 without a final state takes
// balanced pieces instead (SegPlan) when they cost less: with B*H heads the
// segments give B*H*P CTAs of whole segments, which leaves SMs idle whenever
// B*H does not divide the SM count (32 heads: 128 CTAs on 152 SMs), while
// pieces give every SM the same number of chunks.
SegPlan forward_plan(long long BH, int N, int dk, int dv, la_dtype dtype, bool causal, bool final_state) {
  const bool tc = g_path.load() == LA_PATH_AUTO && tc_forward_supported(dk, dv, dtype, causal);
  SegPlan plan = tc ? plan_segments_tc(BH, N, causal) : plan_segments(BH, N, kSlots);
  if (tc && causal && dk == 128 && dv == 128 && !final_state) {
    const long long nch = (N + kSegGranule - 1) / kSegGranule;
    const long long total = BH * nch;
    const long long np0 = std::min<long long>(kSlots, total);
    const long long len = (total + np0 - 1) / np0;          // chunks per piece
    const long long np = (total + len - 1) / len;
    const long long L = (plan.seg_len + kSegGranule - 1) / kSegGranule;
    const long long waves = (BH * plan.P + kSlots - 1) / kSlots;
    // a piece sums the records of the pieces before it in its head (at most
    // ceil(nch / len)), a segment those of the segments before it
    const double piece_cost = (double)(len + 1) + kRecordCost * (double)((nch + len - 1) / len);
    const double seg_cost = (double)(waves * (L + 1)) + kRecordCost * (plan.P - 1);
    // a piece spans at most two heads (len <= chunks per head)
    if (len <= nch && piece_cost <= seg_cost) {
      plan.NP = (int)np;
      plan.piece_len = (int)len;
      return plan;
    }
  }
  // segments the state pass sums: the earlier ones (causal) or all of them
  const int nseg = causal ? plan.P - 1 : plan.P;
  if (!tc || nseg < 1) return plan;
  const int L = plan.seg_len / kSegGranule;
  double best = 1e300;
  for (int F = 1; F <= 8 && F <= L; ++F) {
    const int sub = (L + F - 1) / F;
    if ((F - 1) * sub >= L) continue;          // every part must hold a chunk
    const long long ctas = BH * nseg * F;
    if (F > 1 && ctas > kSlots) break;
    // every part is a record the costliest chunk-loop CTA sums
    const double cost = (double)((ctas + kSlots - 1) / kSlots) * (sub + 1) +
                        kRecordCost * (causal ? plan.P - 1 : plan.P) * F;
    if (cost < best) {
      best = cost;
      plan.F = F;
    }
  }
  return plan;
}

// la_forward_host: internal copy streams and events per device, created on
// first use on that device and reused under its lock (enqueueing is short).
struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in[2] = {nullptr, nullptr}, done[2] = {nullptr, nullptr}, freed[2] = {nullptr, nullptr};
};
constexpr int kMaxDevices = 64;
HostPipe g_pipes[kMaxDevices];

// With p.mu held and `device` current.
cudaError_t host_pipe_ready_locked(HostPipe& p) {
  if (p.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking);
  cudaEvent_t* evs[8] = {&p.start, &p.end, &p.in[0], &p.in[1], &p.done[0], &p.done[1], &p.freed[0], &p.freed[1]};
  for (int i = 0; i < 8 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming);
  if (e == cudaSuccess) p.ready = true;
  return e;
}

// Staging layout of la_forward_host: two slots of [q | k | v | out] for the
// largest slice, then one la_forward workspace; regions 256-byte aligned.
struct HostLayout {
  int S, base, extra;            // slices; sequences per slice: base (+1 for the first `extra`)
  size_t qb, vb, slot, fwd_off, fwd_bytes, total;
};

HostLayout host_layout(long long BH, int N, int dk, int dv, int causal, la_dtype dtype, int slices) {
  HostLayout L{};
  L.S = (int)(slices < 1 ? 1 : (slices > BH ? BH : slices));
  if (L.S < 1) L.S = 1;
  L.base = (int)(BH / L.S);
  L.extra = (int)(BH % L.S);
  const long long maxcnt = L.base + (L.extra ? 1 : 0);
  const size_t elt = dtype == LA_BF16 ? 2 : 4;
  L.qb = align_up((size_t)maxcnt * N * dk * elt, 256);
  L.vb = align_up((size_t)maxcnt * N * dv * elt, 256);
  L.slot = 2 * L.qb + 2 * L.vb;
  size_t fw = 0;
  for (int extra = 0; extra <= (L.extra ? 1 : 0); ++extra) {
    const int cnt = L.base + extra;
    if (cnt <= 0) continue;
    const size_t w = la_forward_workspace_size(1, cnt, N, dk, dv, causal, dtype);
    fw = w > fw ? w : fw;
  }
  L.fwd_off = 2 * L.slot;
  L.fwd_bytes = fw;
  L.total = L.fwd_off + align_up(fw, 256);
  return L;
}

}  // namespace la

using namespace la;

extern "C" {

const char* la_status_string(la_status s) {
  switch (s) {
    case LA_OK: return "LA_OK";
    case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG";
    case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED";
    case LA_ERR_CUDA: return "LA_ERR_CUDA";
    case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT";
  }
  return "LA_ERR_UNKNOWN";
}

const char* la_last_error(void) { return g_last_error; }

int la_version(void) { return 100; }

int la_set_path(int path) {
  if (path != LA_PATH_AUTO && path != LA_PATH_SIMT) return -1;
  return g_path.exchange(path);
}

int la_forward_path(int dk, int dv, la_dtype dtype, int causal) {
  if (!head_ok(dk) || !head_ok(dv) || (dtype != LA_F32 && dtype != LA_BF16)) return -1;
  return (g_path.load() == LA_PATH_AUTO && tc_forward_supported(dk, dv, dtype, causal != 0)) ? 1 : 0;
}

int la_decode_path(int dk, int dv, la_dtype dtype, int T) {
  if (!head_ok(dk) || !head_ok(dv) || (dtype != LA_F32 && dtype != LA_BF16) || T < 0) return -1;
  return (g_path.load() == LA_PATH_AUTO && tc_decode_supported(dk, dv, dtype, T)) ? 1 : 0;
}

int la_backward_path(int dk, int dv, la_dtype dtype, int causal) {
  if (!head_ok(dk) || !head_ok(dv) || (dtype != LA_F32 && dtype != LA_BF16)) return -1;
  return (g_path.load() == LA_PATH_AUTO && tc_backward_supported(dk, dv, dtype, causal != 0)) ? 1 : 0;
}

size_t la_forward_workspace_size(int B, int H, int N, int dk, int dv, int causal, la_dtype dtype) {
  if (B <= 0 || H <= 0 || N <= 0 || !head_ok(dk) || !head_ok(dv)) return 0;
  const long long BH = (long long)B * H;
  // with or without a final state (the plan may differ): the larger
  const size_t a = layout(BH, N, dk, dv, forward_plan(BH, N, dk, dv, dtype, causal != 0, false), false).total;
  const size_t b = layout(BH, N, dk, dv, forward_plan(BH, N, dk, dv, dtype, causal != 0, true), false).total;
  return std::max(a, b);
}

la_status la_forward_plan(int B, int H, int N, int dk, int dv, int causal, la_dtype dtype, int final_state,
                          int* out) {
  if (out == nullptr) return fail(LA_ERR_INVALID_ARG, "out must be non-NULL");
  if (B <= 0 || H <= 0 || N <= 0) return fail(LA_ERR_INVALID_ARG, "B, H, N must be positive");
  if (!head_ok(dk) || !head_ok(dv)) return fail(LA_ERR_INVALID_ARG, "head sizes dk=%d dv=%d", dk, dv);
  if (dtype != LA_F32 && dtype != LA_BF16) return fail(LA_ERR_INVALID_ARG, "dtype %d", (int)dtype);
  const SegPlan p = forward_plan((long long)B * H, N, dk, dv, dtype, causal != 0, final_state != 0);
  out[0] = p.P;
  out[1] = p.seg_len;
  out[2] = p.F;
  out[3] = p.NP;
  out[4] = p.piece_len;
  return LA_OK;
}

size_t la_backward_workspace_size(int B, int H, int N, int dk, int dv, int causal, la_dtype dtype) {
  (void)dtype;
  if (B <= 0 || H <= 0 || N <= 0 || !head_ok(dk) || !head_ok(dv)) return 0;
  const long long BH = (long long)B * H;
  // the CUDA-core and the tensor-core plans (the path is chosen at the call): the larger
  const size_t a = layout(BH, N, dk, dv, plan_segments(BH, N), true).total;
  const size_t b = layout(BH, N, dk, dv, plan_segments_tc(BH, N, causal != 0), true).total;
  return std::max(a, b);
}

la_status la_forward(const void* q, const void* k, const void* v, void* out,
                     int B, int H, int N, int dk, int dv, int causal, float eps,
                     la_dtype dtype, float* S_final, float* z_final,
                     void* workspace, size_t workspace_bytes, la_stream_t stream_) {
  bool empty = false;
  la_status st = check_sizes(B, H, N, dk, dv, dtype, eps, &empty);
  if (st != LA_OK) return st;
  if ((S_final == nullptr) != (z_final == nullptr))
    return fail(LA_ERR_INVALID_ARG, "S_final and z_final must be both given or both NULL");
  if ((S_final && !aligned16(S_final)) || (z_final && !aligned16(z_final)))
    return fail(LA_ERR_INVALID_ARG, "S_final/z_final must be 16-byte aligned");
  cudaStream_t stream = (cudaStream_t)stream_;
  const long long BH = (long long)B * H;
  if (empty) {
    if (S_final != nullptr && BH > 0) {
      cudaError_t e = cudaMemsetAsync(S_final, 0, sizeof(float) * BH * dk * dv, stream);
      if (e == cudaSuccess) e = cudaMemsetAsync(z_final, 0, sizeof(float) * BH * dk, stream);
      if (e != cudaSuccess) return cuda_fail(e, "la_forward (zero final state)");
    }
    return LA_OK;
  }
  if (!q || !k || !v || !out) return fail(LA_ERR_INVALID_ARG, "q, k, v, out must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(LA_ERR_INVALID_ARG, "q, k, v, out must be 16-byte aligned");
  const SegPlan plan = forward_plan(BH, N, dk, dv, dtype, causal != 0, S_final != nullptr);
  const WsLayout w = layout(BH, N, dk, dv, plan, false);
  if (workspace == nullptr || workspace_bytes < w.total)
    return fail(LA_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", w.total,
                workspace == nullptr ? (size_t)0 : workspace_bytes);
  if (!aligned16(workspace)) return fail(LA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");

  FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.BH = (int)BH; a.N = N; a.dk = dk; a.dv = dv; a.causal = causal != 0;
  a.eps = eps; a.dtype = dtype; a.S_final = S_final; a.z_final = z_final;
  a.ws_state = (float*)((char*)workspace + w.state_off);
  a.plan = plan; a.stream = stream;

  const bool use_tc = g_path.load() == LA_PATH_AUTO && tc_forward_supported(dk, dv, dtype, a.causal);
  if (use_tc && device_status_ptr() == nullptr)
    return fail(LA_ERR_CUDA, "la_forward: device status word unavailable");
  prof_begin(LA_SPAN_FWD_STATE, stream);
  cudaError_t e = use_tc ? tc_segment_state(a) : simt_segment_state(a);
  prof_end(LA_SPAN_FWD_STATE, stream);
  if (e != cudaSuccess) return cuda_fail(e, "la_forward (segment state)");
  if (!use_tc) {
    // the tensor-core output kernel sums the earlier segments' records itself
    // and writes the final state from its last segment
    prof_begin(LA_SPAN_FWD_SCAN, stream);
    e = segment_scan(a.ws_state, a.BH, plan.P, state_words(dk, dv),
                     a.causal ? SCAN_EXCLUSIVE_FWD : SCAN_TOTAL, S_final, z_final,
                     dk, dv, stream);
    prof_end(LA_SPAN_FWD_SCAN, stream);
    if (e != cudaSuccess) return cuda_fail(e, "la_forward (segment scan)");
  }
  prof_begin(LA_SPAN_FWD_OUTPUT, stream);
  e = use_tc ? tc_forward_output(a) : simt_forward_output(a);
  prof_end(LA_SPAN_FWD_OUTPUT, stream);
  if (e != cudaSuccess) return cuda_fail(e, "la_forward (output)");
  return LA_OK;
}

size_t la_forward_host_workspace_size(int B, int H, int N, int dk, int dv, int causal, la_dtype dtype,
                                      int slices) {
  if (B <= 0 || H <= 0 || N <= 0 || !head_ok(dk) || !head_ok(dv) || (dtype != LA_F32 && dtype != LA_BF16))
    return 0;
  return host_layout((long long)B * H, N, dk, dv, causal, dtype, slices).total;
}

la_status la_forward_host(const void* q, const void* k, const void* v, void* out, int B, int H, int N, int dk,
                          int dv, int causal, float eps, la_dtype dtype, int slices, void* workspace,
                          size_t workspace_bytes, la_stream_t stream_) {
  bool empty = false;
  la_status st = check_sizes(B, H, N, dk, dv, dtype, eps, &empty);
  if (st != LA_OK) return st;
  if (slices < 1) return fail(LA_ERR_INVALID_ARG, "slices must be >= 1");
  if (empty) return LA_OK;
  if (!q || !k || !v || !out) return fail(LA_ERR_INVALID_ARG, "q, k, v, out must be non-NULL");
  const long long BH = (long long)B * H;
  const HostLayout L = host_layout(BH, N, dk, dv, causal, dtype, slices);
  if (workspace == nullptr || workspace_bytes < L.total)
    return fail(LA_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", L.total,
                workspace == nullptr ? (size_t)0 : workspace_bytes);
  if (!aligned16(workspace)) return fail(LA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "la_forward_host (device)");
  if (dev < 0 || dev >= kMaxDevices) return fail(LA_ERR_UNSUPPORTED, "la_forward_host: device %d", dev);
  HostPipe& g_pipe = g_pipes[dev];
  std::lock_guard<std::mutex> lk(g_pipe.mu);
  e = host_pipe_ready_locked(g_pipe);
  if (e != cudaSuccess) return cuda_fail(e, "la_forward_host (copy streams)");
  cudaStream_t s = (cudaStream_t)stream_;
  const size_t elt = dtype == LA_BF16 ? 2 : 4;
  char* ws = (char*)workspace;
  // the copy streams start after the work already on `stream`
  e = cudaEventRecord(g_pipe.start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(g_pipe.h2d, g_pipe.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(g_pipe.d2h, g_pipe.start, 0);
  if (e != cudaSuccess) return cuda_fail(e, "la_forward_host (start)");
  la_status result = LA_OK;
  long long seq0 = 0;
  for (int i = 0; i < L.S; ++i) {
    const int cnt = L.base + (i < L.extra ? 1 : 0);
    const int slot = i & 1;
    char* sq = ws + slot * L.slot;
    char* sk = sq + L.qb;
    char* sv = sk + L.qb;
    char* so = sv + L.vb;
    const size_t nq = (size_t)cnt * N * dk * elt, nv = (size_t)cnt * N * dv * elt;
    const size_t oq = (size_t)seq0 * N * dk * elt, ov = (size_t)seq0 * N * dv * elt;
    // the slot was last read by slice i - 2's compute and output copy
    if (i >= 2) e = cudaStreamWaitEvent(g_pipe.h2d, g_pipe.freed[slot], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(sq, (const char*)q + oq, nq, cudaMemcpyHostToDevice, g_pipe.h2d);
    if (e == cudaSuccess) e = cudaMemcpyAsync(sk, (const char*)k + oq, nq, cudaMemcpyHostToDevice, g_pipe.h2d);
    if (e == cudaSuccess) e = cudaMemcpyAsync(sv, (const char*)v + ov, nv, cudaMemcpyHostToDevice, g_pipe.h2d);
    if (e == cudaSuccess) e = cudaEventRecord(g_pipe.in[slot], g_pipe.h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, g_pipe.in[slot], 0);
    if (e != cudaSuccess) {
      result = cuda_fail(e, "la_forward_host (input copies)");
      break;
    }
    st = la_forward(sq, sk, sv, so, 1, cnt, N, dk, dv, causal, eps, dtype, nullptr, nullptr, ws + L.fwd_off,
                    L.fwd_bytes, stream_);
    if (st != LA_OK) {
      result = st;
      break;
    }
    e = cudaEventRecord(g_pipe.done[slot], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(g_pipe.d2h, g_pipe.done[slot], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync((char*)out + ov, so, nv, cudaMemcpyDeviceToHost, g_pipe.d2h);
    if (e == cudaSuccess) e = cudaEventRecord(g_pipe.freed[slot], g_pipe.d2h);
    if (e != cudaSuccess) {
      result = cuda_fail(e, "la_forward_host (output copy)");
      break;
    }
    seq0 += cnt;
  }
  // join: `stream` continues after the last output copy (also on an error,
  // so that nothing enqueued here outlives the caller's view of the stream)
  e = cudaEventRecord(g_pipe.end, g_pipe.d2h);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, g_pipe.end, 0);
  if (e == cudaSuccess) e = cudaEventRecord(g_pipe.end, g_pipe.h2d);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, g_pipe.end, 0);
  if (e != cudaSuccess && result == LA_OK) result = cuda_fail(e, "la_forward_host (join)");
  return result;
}

la_status la_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (on) recycle_spans_locked();
  g_prof_on.store(on != 0);
  return LA_OK;
}

int la_profile_read(int* labels, float* ms, int max) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  const int n = (int)g_spans.size();
  for (int i = 0; i < n && i < max; ++i) {
    const Span& s = g_spans[i];
    float t = -1.f;
    if (s.start && s.stop && s.closed && cudaEventSynchronize(s.stop) == cudaSuccess) {
      if (cudaEventElapsedTime(&t, s.start, s.stop) != cudaSuccess) t = -1.f;
    }
    if (labels) labels[i] = s.label;
    if (ms) ms[i] = t;
  }
  (void)cudaGetLastError();
  return n;
}

long long la_launch_count(void) { return g_launches.load(); }

void la_test_timeout_next_forward(void) { la::g_timeout_test.store(1); }

la_status la_device_status(int clear) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_la_device_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "la_device_status");
  if (clear && v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_la_device_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "la_device_status (clear)");
  }
  if (v != 0) return fail(LA_ERR_TIMEOUT, "a kernel's bounded wait gave up (status %d)", v);
  return LA_OK;
}

la_status la_decode_step(float* S, float* z, const void* q, const void* k,
                         const void* v, void* out, int B, int H, int dk, int dv,
                         float eps, la_dtype dtype, la_stream_t stream) {
  bool empty = false;
  la_status st = check_sizes(B, H, 1, dk, dv, dtype, eps, &empty);
  if (st != LA_OK) return st;
  if (empty) return LA_OK;
  if (!S || !z || !q || !k || !v || !out)
    return fail(LA_ERR_INVALID_ARG, "S, z, q, k, v, out must be non-NULL");
  if (!aligned16(S) || !aligned16(z) || !aligned16(q) || !aligned16(k) ||
      !aligned16(v) || !aligned16(out))
    return fail(LA_ERR_INVALID_ARG, "all pointers must be 16-byte aligned");
  DecodeArgs a{};
  a.S = S; a.z = z; a.q = q; a.k = k; a.v = v; a.out = out;
  a.BH = B * H; a.dk = dk; a.dv = dv; a.eps = eps; a.dtype = dtype;
  a.stream = (cudaStream_t)stream;
  prof_begin(LA_SPAN_DECODE, a.stream);
  cudaError_t e = la::decode_step(a);
  prof_end(LA_SPAN_DECODE, a.stream);
  if (e != cudaSuccess) return cuda_fail(e, "la_decode_step");
  return LA_OK;
}

la_status la_decode_steps(float* S, float* z, const void* q, const void* k,
                          const void* v, void* out, int B, int H, int T, int dk,
                          int dv, float eps, la_dtype dtype, la_stream_t stream) {
  if (T < 0) return fail(LA_ERR_INVALID_ARG, "T must be >= 0");
  bool empty = false;
  la_status st = check_sizes(B, H, T, dk, dv, dtype, eps, &empty);
  if (st != LA_OK) return st;
  if (empty) return LA_OK;
  if (!S || !z || !q || !k || !v || !out)
    return fail(LA_ERR_INVALID_ARG, "S, z, q, k, v, out must be non-NULL");
  if (!aligned16(S) || !aligned16(z) || !aligned16(q) || !aligned16(k) ||
      !aligned16(v) || !aligned16(out))
    return fail(LA_ERR_INVALID_ARG, "all pointers must be 16-byte aligned");
  DecodeArgs a{};
  a.S = S; a.z = z; a.q = q; a.k = k; a.v = v; a.out = out;
  a.BH = B * H; a.dk = dk; a.dv = dv; a.eps = eps; a.dtype = dtype;
  a.stream = (cudaStream_t)stream;
  a.ntok = T;
  const bool use_tc = g_path.load() == LA_PATH_AUTO && tc_decode_supported(dk, dv, dtype, T);
  if (use_tc && device_status_ptr() == nullptr)
    return fail(LA_ERR_CUDA, "la_decode_steps: device status word unavailable");
  prof_begin(LA_SPAN_DECODE, a.stream);
  cudaError_t e = use_tc ? la::tc_decode_steps(a) : la::decode_step(a);
  prof_end(LA_SPAN_DECODE, a.stream);
  if (e != cudaSuccess) return cuda_fail(e, "la_decode_steps");
  return LA_OK;
}

la_status la_forward_decay(const void* q, const void* k, const void* v, void* out,
                           int B, int H, int N, int dk, int dv, const float* alpha, float eps,
                           la_dtype dtype, float* S_final, float* z_final,
                           void* workspace, size_t workspace_bytes, la_stream_t stream_) {
  bool empty = false;
  la_status st = check_sizes(B, H, N, dk, dv, dtype, eps, &empty);
  if (st != LA_OK) return st;
  if (dtype != LA_BF16 || dk != 64 || dv != 64)
    return fail(LA_ERR_UNSUPPORTED, "la_forward_decay: bf16 with dk = dv = 64 only");
  if ((S_final == nullptr) != (z_final == nullptr))
    return fail(LA_ERR_INVALID_ARG, "S_final and z_final must be both given or both NULL");
  if ((S_final && !aligned16(S_final)) || (z_final && !aligned16(z_final)))
    return fail(LA_ERR_INVALID_ARG, "S_final/z_final must be 16-byte aligned");
  cudaStream_t stream = (cudaStream_t)stream_;
  const long long BH = (long long)B * H;
  if (empty) {
    if (S_final != nullptr && BH > 0) {
      cudaError_t e = cudaMemsetAsync(S_final, 0, sizeof(float) * BH * dk * dv, stream);
      if (e == cudaSuccess) e = cudaMemsetAsync(z_final, 0, sizeof(float) * BH * dk, stream);
      if (e != cudaSuccess) return cuda_fail(e, "la_forward_decay (zero final state)");
    }
    return LA_OK;
  }
  if (!q || !k || !v || !out || !alpha) return fail(LA_ERR_INVALID_ARG, "q, k, v, out, alpha must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(LA_ERR_INVALID_ARG, "q, k, v, out must be 16-byte aligned");
  const SegPlan plan = forward_plan(BH, N, dk, dv, dtype, true, true);
  const WsLayout w = layout(BH, N, dk, dv, plan, false);
  if (workspace == nullptr || workspace_bytes < w.total)
    return fail(LA_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", w.total,
                workspace == nullptr ? (size_t)0 : workspace_bytes);
  if (!aligned16(workspace)) return fail(LA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (device_status_ptr() == nullptr) return fail(LA_ERR_CUDA, "la_forward_decay: device status word unavailable");
  FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.BH = (int)BH; a.N = N; a.dk = dk; a.dv = dv; a.causal = 1;
  a.eps = eps; a.dtype = dtype; a.S_final = S_final; a.z_final = z_final;
  a.ws_state = (float*)((char*)workspace + w.state_off);
  a.plan = plan; a.stream = stream;
  cudaError_t e = tc_forward_decay(a, alpha, H);
  if (e != cudaSuccess) return cuda_fail(e, "la_forward_decay");
  return LA_OK;
}

la_status la_decode_steps_decay(float* S, float* z, const void* q, const void* k,
                                const void* v, void* out, int B, int H, int T, int dk,
                                int dv, const float* alpha, float eps, la_dtype dtype,
                                la_stream_t stream) {
  if (T < 0) return fail(LA_ERR_INVALID_ARG, "T must be >= 0");
  bool empty = false;
  la_status st = check_sizes(B, H, T, dk, dv, dtype, eps, &empty);
  if (st != LA_OK) return st;
  if (empty) return LA_OK;
  if (!S || !z || !q || !k || !v || !out || !alpha)
    return fail(LA_ERR_INVALID_ARG, "S, z, q, k, v, out, alpha must be non-NULL");
  if (!aligned16(S) || !aligned16(z) || !aligned16(q) || !aligned16(k) ||
      !aligned16(v) || !aligned16(out))
    return fail(LA_ERR_INVALID_ARG, "S, z, q, k, v, out must be 16-byte aligned");
  if (g_path.load() == LA_PATH_AUTO && tc_decode_supported(dk, dv, dtype, T)) {
    // the tensor-core multi-token decode with the decay weights
    if (device_status_ptr() == nullptr)
      return fail(LA_ERR_CUDA, "la_decode_steps_decay: device status word unavailable");
    DecodeArgs d{};
    d.S = S; d.z = z; d.q = q; d.k = k; d.v = v; d.out = out;
    d.BH = B * H; d.dk = dk; d.dv = dv; d.eps = eps; d.dtype = dtype;
    d.stream = (cudaStream_t)stream;
    d.ntok = T;
    cudaError_t e = la::tc_decode_steps_decay(d, alpha, H);
    if (e != cudaSuccess) return cuda_fail(e, "la_decode_steps_decay");
    return LA_OK;
  }
  VariantArgs a{};
  a.S = S; a.z = z; a.q = q; a.k = k; a.v = v; a.out = out; a.alpha = alpha;
  a.H = H; a.BH = B * H; a.ntok = T; a.dk = dk; a.dv = dv; a.eps = eps; a.dtype = dtype;
  a.stream = (cudaStream_t)stream;
  cudaError_t e = la::decode_steps_decay(a);
  if (e != cudaSuccess) return cuda_fail(e, "la_decode_steps_decay");
  return LA_OK;
}

la_status la_decode_steps_delta(float* S, const void* q, const void* k, const void* v,
                                void* out, int B, int H, int T, int dk, int dv,
                                la_dtype dtype, la_stream_t stream) {
  if (T < 0) return fail(LA_ERR_INVALID_ARG, "T must be >= 0");
  bool empty = false;
  la_status st = check_sizes(B, H, T, dk, dv, dtype, 0.f, &empty);
  if (st != LA_OK) return st;
  if (empty) return LA_OK;
  if (!S || !q || !k || !v || !out) return fail(LA_ERR_INVALID_ARG, "S, q, k, v, out must be non-NULL");
  if (!aligned16(S) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(LA_ERR_INVALID_ARG, "all pointers must be 16-byte aligned");
  if (g_path.load() == LA_PATH_AUTO && tc_decode_supported(dk, dv, dtype, T)) {
    // on the tensor cores: pair products, the state read (hi + lo) and the
    // update as MMAs, the triangular solve per value index
    if (device_status_ptr() == nullptr)
      return fail(LA_ERR_CUDA, "la_decode_steps_delta: device status word unavailable");
    DecodeArgs d{};
    d.S = S; d.q = q; d.k = k; d.v = v; d.out = out;
    d.BH = B * H; d.dk = dk; d.dv = dv; d.dtype = dtype;
    d.stream = (cudaStream_t)stream;
    d.ntok = T;
    cudaError_t e = la::tc_decode_steps_delta(d);
    if (e != cudaSuccess) return cuda_fail(e, "la_decode_steps_delta");
    return LA_OK;
  }
  VariantArgs a{};
  a.S = S; a.q = q; a.k = k; a.v = v; a.out = out;
  a.H = H; a.BH = B * H; a.ntok = T; a.dk = dk; a.dv = dv; a.dtype = dtype;
  a.stream = (cudaStream_t)stream;
  cudaError_t e = la::decode_steps_delta(a);
  if (e != cudaSuccess) return cuda_fail(e, "la_decode_steps_delta");
  return LA_OK;
}

la_status la_forward_delta(float* S, const void* q, const void* k, const void* v, void* out,
                           int B, int H, int N, int dk, int dv, la_dtype dtype,
                           la_stream_t stream) {
  if (N < 0) return fail(LA_ERR_INVALID_ARG, "N must be >= 0");
  bool empty = false;
  la_status st = check_sizes(B, H, N, dk, dv, dtype, 0.f, &empty);
  if (st != LA_OK) return st;
  if (dk != dv) return fail(LA_ERR_UNSUPPORTED, "la_forward_delta needs dk == dv");
  if (empty) return LA_OK;
  if (!S || !q || !k || !v || !out) return fail(LA_ERR_INVALID_ARG, "S, q, k, v, out must be non-NULL");
  if (!aligned16(S) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(LA_ERR_INVALID_ARG, "all pointers must be 16-byte aligned");
  // with at least 64 heads the tensor-core group kernel (one head per team
  // of a persistent CTA, 16 tokens per group) fills the GPU and is faster
  // than the column-split CUDA-core kernel (measured: 32 heads level, 128
  // heads 3.2x at d = 128)
  if (g_path.load() == LA_PATH_AUTO && tc_decode_supported(dk, dv, dtype, N) && (long long)B * H >= 64) {
    if (device_status_ptr() == nullptr)
      return fail(LA_ERR_CUDA, "la_forward_delta: device status word unavailable");
    DecodeArgs d{};
    d.S = S; d.q = q; d.k = k; d.v = v; d.out = out;
    d.BH = B * H; d.dk = dk; d.dv = dv; d.dtype = dtype;
    d.stream = (cudaStream_t)stream;
    d.ntok = N;
    cudaError_t e = la::tc_decode_steps_delta(d);
    if (e != cudaSuccess) return cuda_fail(e, "la_forward_delta");
    return LA_OK;
  }
  VariantArgs a{};
  a.S = S; a.q = q; a.k = k; a.v = v; a.out = out;
  a.H = H; a.BH = B * H; a.ntok = N; a.dk = dk; a.dv = dv; a.dtype = dtype;
  a.stream = (cudaStream_t)stream;
  cudaError_t e = la::forward_delta_chunked(a);
  if (e != cudaSuccess) return cuda_fail(e, "la_forward_delta");
  return LA_OK;
}

la_status la_state_copy(float* dst_S, float* dst_z, const float* src_S, const float* src_z,
                        int B, int H, int dk, int dv, la_stream_t stream) {
  bool empty = false;
  la_status st = check_sizes(B, H, 1, dk, dv, LA_F32, 0.f, &empty);
  if (st != LA_OK) return st;
  if ((dst_z == nullptr) != (src_z == nullptr))
    return fail(LA_ERR_INVALID_ARG, "dst_z and src_z must be both given or both NULL");
  if (empty) return LA_OK;
  if (!dst_S || !src_S) return fail(LA_ERR_INVALID_ARG, "dst_S and src_S must be non-NULL");
  if (!aligned16(dst_S) || !aligned16(src_S) || !aligned16(dst_z) || !aligned16(src_z))
    return fail(LA_ERR_INVALID_ARG, "all pointers must be 16-byte aligned");
  const long long BH = (long long)B * H;
  cudaError_t e = la::copy_floats(dst_S, src_S, BH * dk * dv, (cudaStream_t)stream);
  if (e == cudaSuccess && dst_z) e = la::copy_floats(dst_z, src_z, BH * dk, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "la_state_copy");
  return LA_OK;
}

}  // extern "C"

namespace la {
namespace {

// la_backward and la_backward_saved: `saved` (nullable) is the workspace a
// matching la_forward call left its state-pass records in.
la_status backward_impl(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk_,
                        void* dv_, int B, int H, int N, int dk, int dv, int causal, float eps, la_dtype dtype,
                        const void* saved, size_t saved_bytes, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream, const char* name, const float* alpha = nullptr) {
  bool empty = false;
  la_status st = check_sizes(B, H, N, dk, dv, dtype, eps, &empty);
  if (st != LA_OK) return st;
  if (empty) return LA_OK;
  if (!q || !k || !v || !dout || !dq || !dk_ || !dv_)
    return fail(LA_ERR_INVALID_ARG, "q, k, v, dout, dq, dk, dv must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk_) || !aligned16(dv_))
    return fail(LA_ERR_INVALID_ARG, "all pointers must be 16-byte aligned");
  const long long BH = (long long)B * H;
  // decay gating runs on the CUDA-core kernels
  const bool use_tc = alpha == nullptr && g_path.load() == LA_PATH_AUTO &&
                      tc_backward_supported(dk, dv, dtype, causal != 0);
  // the tensor-core sweeps take the forward's record-aware segments
  const SegPlan plan = use_tc ? plan_segments_tc(BH, N, causal != 0) : plan_segments(BH, N);
  const WsLayout w = layout(BH, N, dk, dv, plan, true);
  if (workspace == nullptr || workspace_bytes < w.total)
    return fail(LA_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", w.total,
                workspace == nullptr ? (size_t)0 : workspace_bytes);
  if (!aligned16(workspace)) return fail(LA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  BwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.dout = dout; a.dq = dq; a.dk_ = dk_; a.dv_ = dv_;
  a.BH = (int)BH; a.N = N; a.dk = dk; a.dv = dv; a.causal = causal != 0;
  a.eps = eps; a.dtype = dtype;
  a.ws_state = (float*)((char*)workspace + w.state_off);
  a.ws_rev = (float*)((char*)workspace + w.rev_off);
  a.ws_tok = (float*)((char*)workspace + w.tok_off);
  a.plan = plan; a.stream = stream;
  a.alpha = alpha; a.H = H;
  if (saved != nullptr) {
    const SegPlan fplan = forward_plan(BH, N, dk, dv, dtype, a.causal, true);
    const size_t need = layout(BH, N, dk, dv, fplan, false).total;
    if (saved_bytes < need)
      return fail(LA_ERR_INVALID_ARG, "saved forward workspace of %zu bytes needed, %zu given", need, saved_bytes);
    if (!aligned16(saved)) return fail(LA_ERR_INVALID_ARG, "saved workspace must be 16-byte aligned");
    // the tensor-core backward reads the forward's records as they are (the
    // same segments, F parts each); the CUDA-core path recomputes them
    if (use_tc && fplan.P == plan.P && fplan.seg_len == plan.seg_len) {
      a.ws_state = (float*)saved;
      a.plan.F = fplan.F;
      a.state_ready = true;
    }
  }
  if (use_tc && device_status_ptr() == nullptr)
    return fail(LA_ERR_CUDA, "%s: device status word unavailable", name);
  cudaError_t e = use_tc ? tc_backward(a) : simt_backward(a);
  if (e != cudaSuccess) return cuda_fail(e, name);
  return LA_OK;
}

}  // namespace
}  // namespace la

extern "C" {

la_status la_backward(const void* q, const void* k, const void* v,
                      const void* dout, void* dq, void* dk_, void* dv_, int B,
                      int H, int N, int dk, int dv, int causal, float eps,
                      la_dtype dtype, void* workspace, size_t workspace_bytes,
                      la_stream_t stream) {
  return backward_impl(q, k, v, dout, dq, dk_, dv_, B, H, N, dk, dv, causal, eps, dtype, nullptr, 0, workspace,
                       workspace_bytes, (cudaStream_t)stream, "la_backward");
}

la_status la_backward_saved(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk_,
                            void* dv_, int B, int H, int N, int dk, int dv, int causal, float eps, la_dtype dtype,
                            const void* saved, size_t saved_bytes, void* workspace, size_t workspace_bytes,
                            la_stream_t stream) {
  if (saved == nullptr) return fail(LA_ERR_INVALID_ARG, "saved must be the forward's workspace (non-NULL)");
  return backward_impl(q, k, v, dout, dq, dk_, dv_, B, H, N, dk, dv, causal, eps, dtype, saved, saved_bytes,
                       workspace, workspace_bytes, (cudaStream_t)stream, "la_backward_saved");
}

la_status la_backward_decay(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk_,
                            void* dv_, int B, int H, int N, int dk, int dv, const float* alpha, float eps,
                            la_dtype dtype, void* workspace, size_t workspace_bytes, la_stream_t stream) {
  if (alpha == nullptr && (long long)B * H * N > 0) return fail(LA_ERR_INVALID_ARG, "alpha must be non-NULL");
  return backward_impl(q, k, v, dout, dq, dk_, dv_, B, H, N, dk, dv, 1, eps, dtype, nullptr, 0, workspace,
                       workspace_bytes, (cudaStream_t)stream, "la_backward_decay", alpha);
}

}  // extern "C"
