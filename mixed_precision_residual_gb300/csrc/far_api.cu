// C ABI of the fused residual-add + RMSNorm (and LayerNorm) library (declared in include/far.h):
// host-side validation, the launch plan, the device error word, the
// host-buffer (end-to-end) pipeline and the bounded-wait self test.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "far.h"
#include "far_device.cuh"
#include "far_params.h"

namespace far {

// Device error word: bit FAR_ERR_TIMEOUT is set by a kernel that gave up a
// bounded wait.  Read and cleared by far_device_status.
__device__ unsigned int g_status;

// Row counters of the staged kernel's claimed rows: pairs {next claim, CTAs done}, zero
// while free (each launch's last CTA zeroes its pair).
constexpr int kSchedSlots = 64;
__device__ unsigned long long g_sched[kSchedSlots][2];

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxHidden = int64_t(1) << 24;  // (float)hidden must be exact

struct DeviceState {
  bool ready = false;
  int sms = 0;
  unsigned int* status = nullptr;  // device address of g_status on this device
  // host-buffer pipeline: two internal streams and the events that fork/join them
  bool pipe_ready = false;
  cudaStream_t pipe[2] = {nullptr, nullptr};
  cudaEvent_t fork = nullptr, wready = nullptr, join[2] = {nullptr, nullptr};
  std::mutex pipe_mu;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// The counter pairs of a device (claimed rows, an opt-in row schedule). A launch on stream S
// may take a pair whose launches still pending are all on S: S runs them in order, so each
// has left the pair zero before the next starts. Otherwise it takes a pair with no launch
// pending whose event (recorded after its last launch) has completed. So launches that can
// run side by side (different streams) never share a pair, while a stream with many
// launches queued keeps claiming rows. Streams are told apart by their context-unique id,
// not their handle (a destroyed stream's handle can come back; every thread's per-thread
// default stream has one handle). No pair during stream capture (a captured event cannot
// be polled) or when all are busy: the launch takes fixed-stride rows.
//
// PoolBook is that bookkeeping alone, apart from CUDA (the event's state is asked through
// a callback), so that the host-only model far_sched_pool_model can drive it.
struct PoolBook {
  unsigned long long stream_id[kSchedSlots] = {};  // the stream of its pending launches
  int pending[kSchedSlots] = {};   // handed out, not yet released after the launch
  bool used[kSchedSlots] = {};     // launched at least once: its event shows the last launch
  bool retired[kSchedSlots] = {};  // no trustworthy event: never handed out again
  int next = 0;

  // a pair for a launch on stream `sid`, or -1; event_done(s) is 1 when the event recorded
  // after pair s's last launch has completed, else 0
  template <typename Done>
  int acquire(unsigned long long sid, Done event_done) {
    int got = -1;
    // a pair last given to this stream (whatever is pending on it runs before this launch)
    for (int s = 0; s < kSchedSlots && got < 0; ++s)
      if (!retired[s] && (used[s] || pending[s] > 0) && stream_id[s] == sid) got = s;
    // else a pair nothing is pending on, whose last launch has finished
    for (int i = 0; i < kSchedSlots && got < 0; ++i) {
      const int s = (next + i) % kSchedSlots;
      if (pending[s] > 0 || retired[s]) continue;
      if (used[s] && event_done(s) != 1) continue;
      got = s;
      next = (s + 1) % kSchedSlots;
    }
    if (got >= 0) {
      stream_id[got] = sid;
      ++pending[got];
    }
    return got;
  }

  // after the launch that used pair s: launched (the kernel was enqueued) and recorded (an
  // event was recorded after it, outside any capture); a launched pair without such an
  // event is retired
  void release(int s, bool launched, bool recorded) {
    if (launched) {
      if (recorded) used[s] = true;
      else retired[s] = true;
    }
    --pending[s];
  }
};

struct SchedPool {
  std::mutex mu;
  bool ready = false, broken = false;
  unsigned long long* pairs = nullptr;  // device address of g_sched on this device
  cudaEvent_t ev[kSchedSlots] = {};
  PoolBook book;
};
SchedPool g_sched_pool[kMaxDevices];

// programmatic dependent launch of the norm kernels: 1 (default) on, 0 off
std::atomic<int> g_programmatic{1};

// row schedule: 1 fixed stride always (the default: no state kept between calls),
// 0 claimed rows by the automatic rule, 2 claimed rows whenever a pair is free
std::atomic<int> g_row_schedule{1};
thread_local int g_last_claimed = 0;  // this thread's last staged launch claimed rows

bool stream_capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return true;  // unknown: treat as capturing (no pair)
  }
  return cs != cudaStreamCaptureStatusNone;
}

// a counter pair for a launch on `stream`, or -1
int sched_acquire(int dev, cudaStream_t stream) {
  // a capturing stream gets no pair, and no other call: one (the stream's id) was seen to
  // invalidate the capture
  if (stream_capturing(stream)) return -1;
  SchedPool& sp = g_sched_pool[dev];
  std::lock_guard<std::mutex> lk(sp.mu);
  if (sp.broken) return -1;
  // polling events is a call that a capture in global mode on another thread forbids:
  // relax this thread's mode for the pool's own calls
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  cudaThreadExchangeStreamCaptureMode(&mode);
  unsigned long long sid = 0;
  if (cudaStreamGetId(stream, &sid) != cudaSuccess) {
    cudaGetLastError();
    cudaThreadExchangeStreamCaptureMode(&mode);
    return -1;
  }
  if (!sp.ready) {
    void* addr = nullptr;
    bool ok = cudaGetSymbolAddress(&addr, g_sched) == cudaSuccess;
    for (int i = 0; ok && i < kSchedSlots; ++i)
      ok = cudaEventCreateWithFlags(&sp.ev[i], cudaEventDisableTiming) == cudaSuccess;
    if (ok) {
      sp.pairs = static_cast<unsigned long long*>(addr);
      sp.ready = true;
    } else {
      cudaGetLastError();
      sp.broken = true;
    }
  }
  int got = -1;
  if (sp.ready) {
    got = sp.book.acquire(sid, [&](int s) {
      const cudaError_t e = cudaEventQuery(sp.ev[s]);
      if (e == cudaSuccess) return 1;
      if (e != cudaErrorNotReady) cudaGetLastError();
      return 0;
    });
  }
  cudaThreadExchangeStreamCaptureMode(&mode);
  return got;
}

// after the launch that used pair `s` (launched: the kernel was enqueued). The event is
// recorded after the launch, so once no launch is pending it follows all of them. A stream
// that began capturing after the launch would take the record into its graph, where the
// pool could never see it: such a pair is retired instead.
void sched_release(int dev, int s, cudaStream_t stream, bool launched) {
  SchedPool& sp = g_sched_pool[dev];
  std::lock_guard<std::mutex> lk(sp.mu);
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  cudaThreadExchangeStreamCaptureMode(&mode);
  bool recorded = false;
  if (launched && !stream_capturing(stream)) {
    recorded = cudaEventRecord(sp.ev[s], stream) == cudaSuccess;
    if (!recorded) cudaGetLastError();
  }
  sp.book.release(s, launched, recorded);
  cudaThreadExchangeStreamCaptureMode(&mode);
}

thread_local char g_cuda_msg[256] = "CUDA error";

int cuda_fail(cudaError_t e) {
  snprintf(g_cuda_msg, sizeof g_cuda_msg, "CUDA error %d: %s", (int)e, cudaGetErrorString(e));
  return FAR_ERR_CUDA;
}

int current_device(DeviceState*& st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
  st = &g_dev[dev];
  std::lock_guard<std::mutex> lk(g_mu);
  if (!st->ready) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_status);
    if (e != cudaSuccess) return cuda_fail(e);
    st->sms = sms;
    st->status = static_cast<unsigned int*>(addr);
    st->ready = true;
  }
  return FAR_OK;
}

// tuning override of the staged plan (0 = automatic), process-wide
std::atomic<int> g_force_nch{0}, g_force_groups{0}, g_force_stages{0}, g_force_kind{-1};

int decode(int dtype, int& act, int& wd, int& od) {
  if (dtype < 0 || (dtype >> 8) != 0) return FAR_ERR_DTYPE;
  act = dtype & 0xf;
  wd = (dtype >> 4) & 0xf;
  auto known = [](int d) { return d == FAR_F32 || d == FAR_F16 || d == FAR_BF16; };
  if (!known(act) || !known(wd)) return FAR_ERR_DTYPE;
  if ((act == FAR_F16 && wd == FAR_BF16) || (act == FAR_BF16 && wd == FAR_F16)) return FAR_ERR_DTYPE_MIX;
  od = promote(act, wd);
  return FAR_OK;
}

int dsize(int dt) { return dt == FAR_F32 ? 4 : 2; }

// Row strides in elements (each >= hidden); the contiguous entry points pass hidden.
struct Strides {
  int64_t x, r, out, res;
};

// A strided tensor in memory: `rows` rows of `width` bytes, `stride` bytes apart.
struct Region {
  uint64_t base;
  int64_t rows, width, stride;
};

Region region(const void* p, int64_t rows, int64_t width, int64_t stride) {
  return Region{(uint64_t)(uintptr_t)p, rows, width, stride};
}

int64_t floor_div(int64_t a, int64_t b) {  // b > 0
  return a >= 0 ? a / b : -((-a + b - 1) / b);
}

// Do any bytes of A and B coincide?  Exact for equal strides (rows of two column
// slices of one matrix interleave without touching); otherwise any overlap of the
// spanned byte ranges counts.
bool regions_overlap(const Region& A, const Region& B) {
  if (A.rows == 0 || B.rows == 0 || A.width == 0 || B.width == 0) return false;
  const uint64_t a_end = A.base + (uint64_t)((A.rows - 1) * A.stride + A.width);
  const uint64_t b_end = B.base + (uint64_t)((B.rows - 1) * B.stride + B.width);
  if (!(A.base < b_end && B.base < a_end)) return false;
  if (A.stride != B.stride || A.rows == 1 || B.rows == 1) return true;
  // row i of A and row j of B meet iff -B.width < d + (j - i) * s < A.width, d = B.base - A.base
  const int64_t s = A.stride;
  const int64_t d = (int64_t)(B.base - A.base);
  const int64_t kmin = floor_div(-B.width - d, s) + 1;
  const int64_t kmax = -floor_div(-(A.width - d), s) - 1;  // ceil((A.width - d) / s) - 1
  const int64_t lo = kmin > -(B.rows - 1) ? kmin : -(B.rows - 1);
  const int64_t hi = kmax < (A.rows - 1) ? kmax : (A.rows - 1);
  return lo <= hi;
}

bool same_region(const Region& A, const Region& B) {
  return A.base == B.base && A.rows == B.rows && A.width == B.width && A.stride == B.stride;
}

// an output may be exactly an input region (in place); no other byte may be shared
bool bad_overlap(const Region& out, const Region& in) { return regions_overlap(out, in) && !same_region(out, in); }

struct Call {
  const void* x;
  const void* r;
  const void* w;
  float eps;
  void* out;
  void* res_out;
  int64_t tokens, hidden;
  int act, wd, od;
  bool residual;
  Strides st;  // elements
  int quant = kQuantNone;  // quantised output: q [tokens, hidden] bytes and scale [tokens]
  void* q = nullptr;
  float* scale = nullptr;
  bool ln = false;            // LayerNorm: gamma in w, beta [hidden] in the weight dtype
  const void* beta = nullptr;
  bool fixed_stride = false;  // never claim rows (no counter pair, no event: the
                              // allocation-free entry point creates and records none)
};

// Set while a host-only plan query validates its stand-in addresses: the plan depends on
// shapes and alignment alone, and stand-ins spread over the address space for the largest
// accepted shapes could wrap past 2^64 and read as overlapping, so no overlap is checked.
thread_local bool t_plan_query = false;
struct PlanQuery {
  PlanQuery() { t_plan_query = true; }
  ~PlanQuery() { t_plan_query = false; }
};

int validate(const void* x, const void* r, const void* w, float eps, void* out, void* res_out,
             int64_t tokens, int64_t hidden, int dtype, bool residual, Call& c, const Strides* strides = nullptr) {
  int st = decode(dtype, c.act, c.wd, c.od);
  if (st != FAR_OK) return st;
  if (hidden <= 0 || hidden > kMaxHidden || tokens < 0) return FAR_ERR_SHAPE;
  const Strides sd = strides ? *strides : Strides{hidden, hidden, hidden, hidden};
  const int64_t widest = residual ? (sd.x > sd.r ? sd.x : sd.r) : sd.x;
  const int64_t wider = residual ? (sd.out > sd.res ? sd.out : sd.res) : sd.out;
  if (sd.x < hidden || sd.out < hidden || (residual && (sd.r < hidden || sd.res < hidden))) return FAR_ERR_SHAPE;
  // byte offsets must fit in int64 (and in the kernels' 64-bit offsets)
  const int64_t max_stride = widest > wider ? widest : wider;
  if (tokens > (INT64_MAX / 8) / max_stride) return FAR_ERR_SHAPE;
  if (!(eps >= 0.0f) || eps == INFINITY) return FAR_ERR_EPS;
  c = Call{x, r, w, eps, out, res_out, tokens, hidden, c.act, c.wd, c.od, residual, sd, c.quant, c.q, c.scale,
           c.ln, c.beta};
  if (tokens == 0) return FAR_OK;
  if (!x || !w || !out || (residual && (!r || !res_out))) return FAR_ERR_NULL;
  if (c.ln && !c.beta) return FAR_ERR_NULL;
  if (t_plan_query) return FAR_OK;
  const int64_t sa = dsize(c.act), so = c.quant ? 1 : dsize(c.od);  // a quantised output is one byte
  const Region X = region(x, tokens, hidden * sa, sd.x * sa);
  const Region O = region(out, tokens, hidden * so, sd.out * so);
  const Region W = region(w, 1, hidden * dsize(c.wd), hidden * dsize(c.wd));
  if (bad_overlap(O, X) || regions_overlap(O, W)) return FAR_ERR_ALIAS;
  if (residual) {
    const Region R = region(r, tokens, hidden * sa, sd.r * sa);
    const Region RO = region(res_out, tokens, hidden * sa, sd.res * sa);
    if (bad_overlap(O, R) || regions_overlap(O, RO)) return FAR_ERR_ALIAS;
    if (bad_overlap(RO, X) || bad_overlap(RO, R) || regions_overlap(RO, W)) return FAR_ERR_ALIAS;
  }
  if (c.ln) {  // LayerNorm's shift: read-only, so no output may touch it
    const Region B = region(c.beta, 1, hidden * dsize(c.wd), hidden * dsize(c.wd));
    if (regions_overlap(O, B)) return FAR_ERR_ALIAS;
    if (residual && regions_overlap(region(res_out, tokens, hidden * sa, sd.res * sa), B)) return FAR_ERR_ALIAS;
  }
  return FAR_OK;
}

// the LayerNorm entry points: gamma in the weight's place, plus beta
int validate_ln(const void* x, const void* r, const void* gamma, const void* beta, float eps, void* out,
                void* res_out, int64_t tokens, int64_t hidden, int dtype, bool residual, Call& c,
                const Strides* strides = nullptr) {
  c.ln = true;
  c.beta = beta;
  return validate(x, r, gamma, eps, out, res_out, tokens, hidden, dtype, residual, c, strides);
}

// the quantised entry points: q and scale replace out and must share no byte with anything
int validate_quant(const void* x, const void* r, const void* w, float eps, void* q, float* scale, void* res_out,
                   int64_t tokens, int64_t hidden, int dtype, int qtype, bool residual, Call& c,
                   const Strides* strides = nullptr) {
  if (qtype != kQuantInt8 && qtype != kQuantFp8) return FAR_ERR_DTYPE;
  c.quant = qtype;
  c.q = q;
  c.scale = scale;
  // q is always contiguous ([tokens, hidden] bytes); x, the residual and residual_out may
  // have row strides
  Strides sd = strides ? *strides : Strides{hidden, hidden, hidden, hidden};
  sd.out = hidden;
  // validate the rest with q standing in for out (the out checks then cover q's bytes too)
  int st = validate(x, r, w, eps, q, res_out, tokens, hidden, dtype, residual, c, &sd);
  if (st != FAR_OK || tokens == 0) return st;
  if (!scale) return FAR_ERR_NULL;
  if (t_plan_query) {
    c.out = nullptr;
    return FAR_OK;
  }
  const int64_t sa = dsize(c.act);
  const Region Q = region(q, tokens, hidden, hidden);
  const Region S = region(scale, 1, tokens * 4, tokens * 4);
  const Region X = region(x, tokens, hidden * sa, sd.x * sa);
  const Region W = region(w, 1, hidden * dsize(c.wd), hidden * dsize(c.wd));
  // q: one byte an element, never an exact alias of an input
  if (regions_overlap(Q, X) || regions_overlap(S, X) || regions_overlap(S, Q) || regions_overlap(S, W))
    return FAR_ERR_ALIAS;
  if (residual) {
    const Region R = region(r, tokens, hidden * sa, sd.r * sa);
    const Region RO = region(res_out, tokens, hidden * sa, sd.res * sa);
    if (regions_overlap(Q, R) || regions_overlap(S, R) || regions_overlap(S, RO)) return FAR_ERR_ALIAS;
  }
  c.out = nullptr;
  return FAR_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// the launch plan for a validated call on a device with `sms` SMs (pure host logic)
int plan(const Call& c, int sms, unsigned int* status, cudaStream_t stream, Launch& L) {
  memset(&L, 0, sizeof L);
  Params& p = L.p;
  p.x = c.x;
  p.r = c.r;
  p.w = c.w;
  p.beta = c.beta;
  L.ln = c.ln;
  p.out = c.out;
  p.res_out = c.res_out;
  p.tokens = c.tokens;
  p.hidden = (int32_t)c.hidden;
  p.hidden_f = (float)c.hidden;
  p.eps = c.eps;
  p.q = c.q;
  p.scale = c.scale;
  L.quant = c.quant;
  p.status = status;
  p.timeout_ns = kWaitTimeoutNs;
  L.stream = stream;
  L.programmatic = g_programmatic.load() != 0;

  const int sa = dsize(c.act), sw = dsize(c.wd);
  const int64_t row_bytes = c.hidden * sa;
  const int so = dsize(c.od);
  p.x_stride = c.st.x * sa;
  p.r_stride = c.st.r * sa;
  p.out_stride = c.st.out * so;
  p.res_stride = c.st.res * sa;
  // the bulk-copy path needs every row start on a 16-byte boundary
  const bool rows_aligned = p.x_stride % 16 == 0 && p.out_stride % 16 == 0 &&
                            (!c.residual || (p.r_stride % 16 == 0 && p.res_stride % 16 == 0));
  const void* out_ptr = c.quant ? c.q : c.out;
  bool staged = g_force_kind.load() != kGeneric && row_bytes % 16 == 0 && rows_aligned && aligned16(c.x) &&
                aligned16(c.w) && (!c.ln || aligned16(c.beta)) && aligned16(out_ptr) &&
                (!c.residual || (aligned16(c.r) && aligned16(c.res_out))) &&
                (!c.quant || ((uintptr_t)c.scale & 3u) == 0);
  int nch = 0, G = 0, groups = 0, stages = 0;
  uint32_t stage_bytes = 0, w_bytes = (uint32_t)((c.hidden * sw + 15) / 16 * 16);
  if (c.ln) w_bytes *= 2;  // gamma, then beta at the next 16-byte boundary
  size_t smem = 0;
  if (staged) {
    // Launch table, from sweeps of chunks a thread x groups x ring slots on GB300, timed
    // after an L2 flush and back to back (where each launch writes back its predecessor's
    // output still in L2):
    //  - at most 2 rows an SM: one group spreading each row over as many warps as it has chunks;
    //  - otherwise 8 chunks a thread (64 values of 16-bit data) keeps the per-row work
    //    (reductions, IEEE divide and square root, waits) small against the per-element
    //    work, with 5, 6, 10 or 4 chunks where 8 would leave lanes idle;
    //  - the groups keep a measured amount of rows in flight per SM: ~70 KB (fused RMSNorm),
    //    ~64 KB (fused LayerNorm), 128 / 120 KB (fp32 output, fused / variant), a fitted
    //    count for the no-residual RMSNorm variant; the quantised output as many groups as
    //    the warps hold;
    //  - the warp budget: 12 warps at 8 chunks (128 registers), 16 below, 19 for the
    //    no-residual variant on 16-bit rows (x kept packed: 96 registers).
    // Each branch below states its own rule and measurements.
    const int64_t C = row_bytes / 16;
    // packed x leaves room for 19 warps (96 registers a thread), also with a quantised
    // output, whose kept outputs take the registers of the consumed x; LayerNorm keeps the
    // binary32 deviations s - mean instead
    const bool packed = packed_rows(c.residual, c.act) && !c.ln;
    int slots_per_group = c.residual ? 1 : 2;
    nch = 8;
    G = (int)((C + 255) / 256);
    if (C <= 128) {  // one warp covers the row with fewer chunks a thread
      nch = 1;
      while (32LL * nch < C) nch *= 2;
      G = 1;
    }
    bool one_group = false;
    int group_cap = 1 << 30;
    const int64_t rows_per_sm = (c.tokens + sms - 1) / sms;
    if (rows_per_sm <= 2) {
      // a batch this small is latency-bound: spread each row over as many warps as it has
      // chunks (one chunk a thread) instead of minimising the per-row overhead
      nch = 1;
      while ((C + 32LL * nch - 1) / (32LL * nch) > kMaxConsumerWarps && nch < 8) nch *= 2;
      G = (int)((C + 32LL * nch - 1) / (32LL * nch));
      one_group = true;
    } else if (c.ln && C > 128) {
      // LayerNorm (two reductions a row, the mean's then the squared deviations', and
      // more arithmetic an element than RMSNorm): measured best were 8 chunks a thread
      // and as many groups as 12 warps hold, one ring slot each; with an fp32 output of
      // 16-bit activations 3 groups for fused rows of 4+ warps, 5 for shorter fused rows
      // (10 for one-warp rows) and 5 for the variant; the fused op otherwise as below
      nch = 8;
      G = (int)((C + 255) / 256);
      const bool wide_out = c.od == FAR_F32 && c.act != FAR_F32;
      if (c.residual && !wide_out) {
        // the fused op, from sweeps timed after an L2 flush and back to back: 4 chunks a
        // thread where 8 would leave lanes idle and 4 cover the row exactly, and as many
        // groups of one slot as keep about 64 KB of x and residual in flight per SM (a slot
        // more where an SM has at most 32 rows), but at least 2 (bf16 32768 x 3072: 130 us
        // against 156; 16384 x 7168: 160 against 177)
        if (C % 256 != 0 && C % 128 == 0 && C / 128 <= kMaxConsumerWarps) {
          nch = 4;
          G = (int)(C / 128);
        }
        const int64_t slot = 2 * ((row_bytes + 127) / 128 * 128);
        const int64_t want = (64 * 1024 + (rows_per_sm <= 32 ? slot : 0) + slot / 2) / slot;
        group_cap = (int)(want < 2 ? 2 : want);
      } else if (c.residual) {
        group_cap = G >= 4 ? 3 : (G == 1 ? 10 : 5);
      } else {
        // the variant: one-warp rows at most 10 groups (12 measured 9 % slower in a stream,
        // bf16 16384 x 2048); rows of 4+ warps two ring slots a group (fp16 65536 x 8192:
        // 424 us against 436 with claimed rows, 458 against 467 at the fixed stride); with
        // a 16-bit output, rows that 8 chunks a thread would cover with idle lanes take 5 or
        // 6 chunks where those cover them exactly (hidden 2560, 3072, 5120 in 16-bit)
        if (!wide_out && C % 256 != 0) {
          for (int cand : {5, 6})
            if (C % (32LL * cand) == 0 && C / (32LL * cand) <= kMaxConsumerWarps) {
              nch = cand;
              G = (int)(C / (32LL * cand));
              break;
            }
        }
        group_cap = wide_out ? 5 : (G == 1 ? 10 : kMaxConsumerWarps);
      }
      slots_per_group = (!c.residual && !wide_out && G >= 4) ? 2 : 1;
    } else if (c.ln) {
      // LayerNorm on rows of one warp at up to 4 chunks a thread (hidden up to 1024 in
      // 16-bit): 7 groups (measured 5-50 % faster than a rows-per-group cap), of two slots
      // for the fused op (9 % faster back to back than one)
      group_cap = 7;
      slots_per_group = c.residual ? 2 : 1;
    } else if (c.quant) {
      // quantised output (a second per-row reduction, the row maximum, lengthens each
      // row's critical path, so as many groups as possible must overlap it), from a sweep
      // of every plan on 20 shapes per op (hidden 1024 to 8192, 512 to 32768 tokens; mean
      // 0.6-0.9 % above the best plan of each, against 14-16 % for the previous table):
      // 8 chunks a thread where they cover the row exactly (the non-exact quantised kernels
      // spill registers) and need at most 12 warps but not 3, else 4 chunks; as many
      // groups of one slot as the warps hold, but at most 11 (fused) or 12 (variant) on
      // one-warp rows and 7 (fused) or 10 (variant) on rows of up to 128 chunks. The fused
      // op on rows of 2+ warps at 8 chunks keeps to 8 warps: with 12 it is 5-10 % faster
      // after an L2 flush but 3-10 % slower when the previous launch's output is still
      // being written back (back-to-back launches, as in the bench)
      // (5 chunks where 8 do not cover the row exactly but 5 do: hidden 2560 and 5120 in
      // 16-bit run 5 chunks on 2 or 4 warps instead of 4 on 3 or 5; measured in a stream,
      // bf16 16384 x 5120 int8 variant 73.1 us against 83.9, E4M3 71.8 against 85.4, fused
      // 92.3 / 88.8 against 93.8 / 92.8; fp16 32768 x 2560 int8 variant 70.0 against 85.0,
      // fused 88.9 against 102.3)
      if (C > 128) {
        nch = (C % 256 == 0 && C / 256 <= 12 && C / 256 != 3) ? 8 : 4;
        if (nch == 4 && C % 160 == 0 && C / 160 <= 12) nch = 5;
        G = (int)((C + 32LL * nch - 1) / (32LL * nch));
        if (G > kMaxConsumerWarps) {
          nch = 8;
          G = (int)((C + 255) / 256);
        }
        if (G == 1) group_cap = c.residual ? 11 : 12;
        else if (c.residual && nch == 8) group_cap = 8 / G > 0 ? 8 / G : 1;
        else group_cap = 1 << 30;
      } else {
        group_cap = c.residual ? 7 : 10;
      }
      // (the variant on 16-bit rows holds up to 19 warps: measured 5-10 % faster than 12 on
      // hidden 4096 and 8192); the variant on rows of 4+ warps takes two ring slots a group
      // (int8, fp16 65536 x 8192: 347 us against 359 in a stream; 16384 x 8192: 94.5 / 97.1)
      slots_per_group = (!c.residual && G >= 4) ? 2 : 1;
    } else if (c.od == FAR_F32 && !c.quant) {
      // fp32 output (or fp32 activations): rows are long in bytes; keep about 128 KB
      // (fused) or 120 KB (variant) of rows in progress per SM, one ring slot per group.
      // The variant of 16-bit activations, from a sweep timed in a stream (launches back to
      // back) and after an L2 flush: 72 KB in progress above 64 rows an SM, and 3 slots a
      // group on one-warp rows, 2 on two-warp rows (bf16 / fp32 weight 4096 x 4096: 18.1 us
      // against 19.2; 16384 x 4096: 66.0 against 67.5; 32768 x 2048: ~65 against 69.0)
      const int64_t row_total = c.hidden * (c.residual ? (3 * sa + dsize(c.od)) : (sa + dsize(c.od)));
      const bool variant16 = !c.residual && c.act != FAR_F32;
      const int64_t budget = c.residual ? 128 * 1024 : ((variant16 && rows_per_sm > 64) ? 72 : 120) * 1024;
      const int64_t want = (budget + row_total / 2) / row_total;
      group_cap = (int)(want < 1 ? 1 : want);
      slots_per_group = variant16 ? (G == 1 ? 3 : (G == 2 ? 2 : 1)) : 1;
    } else if (c.residual && C > 128 && G <= max_consumer_warps(nch, false)) {
      // fused rows, one ring slot per group, from sweeps of every plan timed both after an
      // L2 flush and back to back (where each launch writes back the previous one's output
      // still in L2, as in a stream of launches): rows that 8 chunks a thread cover exactly
      // (and one-warp rows) at 8 chunks with about 70 KB of x and residual in flight per
      // SM, a slot more where an SM has at most 32 rows; longer rows that 8 chunks would
      // cover with idle lanes at 5 or 6 chunks where they cover the row exactly, else 4,
      // with about 64 KB in flight (96 KB at most 32 rows an SM)
      if (C > 256 && C % 256 != 0) {
        int n = 0;
        for (int cand : {5, 6, 4})
          if (C % (32LL * cand) == 0 && C / (32LL * cand) <= kMaxConsumerWarps) {
            n = cand;
            break;
          }
        if (n == 0 && (C + 127) / 128 <= kMaxConsumerWarps) n = 4;
        if (n != 0) {
          nch = n;
          G = (int)((C + 32LL * nch - 1) / (32LL * nch));
        }
      }
      const int64_t slot = 2 * ((row_bytes + 127) / 128 * 128);
      const int64_t target = nch != 8 ? (rows_per_sm <= 32 ? 96 : 64) * 1024
                                      : 70 * 1024 + (rows_per_sm <= 32 ? slot : 0);
      const int64_t want = (target + slot / 2) / slot;
      group_cap = (int)(want < 1 ? 1 : want);
      // rows of 4+ warps at up to 4 rows an SM: 2 groups (fp16 512 x 8192: 7.7 us against
      // 8.1 for 3 in a stream, 12.3 against 12.8 after an L2 flush; rows of 2 warps were
      // slower so, bf16 600 x 4096)
      if (rows_per_sm <= 4 && G >= 4 && group_cap > 2) group_cap = 2;
      slots_per_group = 1;
    } else if (packed && c.od != FAR_F32) {
      // the no-residual variant on 16-bit rows (x kept packed), from a sweep of every plan
      // on 59 shapes (hidden 1024 to 16384, 512 to 65536 tokens): rows of up to 192 chunks
      // 7 groups of 2 slots; one warp a row 7 groups of 3 slots (1 below 100 rows an SM);
      // three warps 6 groups of one slot; four 4; more, 16 warps in groups of 2 slots (of one
      // slot at 8+ warps a row, measured back to back).  Two warps a row: 5 groups of 2
      // slots, from a later sweep timed in a stream (programmatic launch) and after an L2
      // flush (fp16 16384 x 4096: 44.6 us against 47.8 for 8 groups of one slot); three
      // warps with idle lanes (hidden 5120 at 8 chunks, taken above 128 rows an SM, see
      // below) 5 groups of 2 slots as well
      if (C <= 192) {
        group_cap = 7;
        slots_per_group = 2;
      } else if (G <= 4) {
        const bool idle3 = G == 3 && C % 256 != 0;
        const int caps[5] = {0, 7, 5, 6, 4};
        group_cap = idle3 ? 5 : caps[G];
        slots_per_group = G == 1 ? (rows_per_sm >= 100 ? 3 : 1) : ((G == 2 || idle3) ? 2 : 1);
      } else {
        group_cap = kMaxConsumerWarps / G;
        slots_per_group = G >= 8 ? 1 : 2;
      }
    } else if (c.residual && C <= 128) {
      // fused rows of one warp at up to 4 chunks a thread (hidden up to 1024 in 16-bit):
      // 7 groups of 2 slots (one slot at most 16 rows an SM), measured 7-10 % faster than
      // a cap of 5 rows a group an SM, back to back and after a flush
      group_cap = 7;
      slots_per_group = rows_per_sm <= 16 ? 1 : 2;
    } else if (c.residual) {
      // fused rows longer than 12 warps at 8 chunks (hidden above 24576 in 16-bit): beyond
      // the 12-warp budget of 8 chunks, so the check below sends them to the generic kernel
      nch = 1;
      while ((C + 32LL * nch - 1) / (32LL * nch) > kMaxConsumerWarps && nch < 8) nch *= 2;
      G = (int)((C + 32LL * nch - 1) / (32LL * nch));
      one_group = true;
    } else {
      // (every variant is taken above; kept as a safe default) 4 groups of one slot
      group_cap = 4;
      slots_per_group = 1;
    }
    // A row that 8 chunks a thread cover with idle lanes but 6 or 5 chunks cover exactly with
    // the same number of warps (hidden 2560 or 3072 in 16-bit) takes the exact plan: measured
    // 3-8 % faster (at most 6 groups fused, 7 for the variant); plain RMSNorm only.
    // The packed variant on rows of 640 chunks (hidden 5120 in 16-bit), which 8 chunks cover
    // with 3 warps and idle lanes: up to 128 rows an SM it runs 10 chunks on 2 warps, 5
    // groups of one slot (two above 32 rows an SM); above, 8 chunks on 3 warps in 5 groups
    // of 2 slots, as the rule above gives.  Timed in a stream (programmatic launch) and
    // after an L2 flush, bf16: 4096 tokens 15.6 us against 17.2 (9 groups of one slot);
    // 8192 30.4 against 33.1; 65536 196.7 against 208.4 (10 chunks, 7 groups).  At 16384
    // tokens (108 rows an SM) 8 chunks on 3 warps were faster in a stream (55.9 against
    // 58.2 us) but slower from a clean L2 (57.4 against 53.5; under ncu 56.2 against
    // 52.5), so 10 chunks stay there.
    if (nch == 8 && packed && C == 640 && c.od != FAR_F32 && !one_group && rows_per_sm <= 128) {
      nch = 10;
      G = 2;
      group_cap = 5;
      slots_per_group = rows_per_sm > 32 ? 2 : 1;
    }
    if (nch == 8 && !c.quant && !c.ln && C % 256 != 0 && !one_group) {
      for (int cand : {6, 5}) {
        if (C % (32LL * cand) == 0 && C / (32LL * cand) == G) {
          nch = cand;
          const int cap = c.residual ? 6 : 7;  // measured best: 6 groups (fused), 7 (variant)
          if (group_cap > cap) group_cap = cap;
          if (packed) slots_per_group = 2;  // the variant: 2 slots a group
          break;
        }
      }
    }
    // a variant batch of at most 16 rows an SM is latency-bound: one slot a group
    if (packed && c.od != FAR_F32 && rows_per_sm <= 16 && G > 1) slots_per_group = 1;
    if (g_force_nch.load() > 0) {
      nch = g_force_nch.load();
      G = (int)((C + 32LL * nch - 1) / (32LL * nch));
      one_group = false;
    }
    staged = G <= max_consumer_warps(nch, packed);
    // 5 or 6 chunks a thread exist only as exact kernels (6 without a quantised output)
    if ((nch == 5 || nch == 6) && (C != 32LL * nch * G || (c.quant && nch == 6))) staged = false;
    // 10 chunks a thread exist only as exact kernels of the packed no-residual variant
    if (nch == 10 && (C != 320LL * G || !packed)) staged = false;
    if (staged) {
      // the default plans keep to 16 consumer warps but for the packed variant with a 16-bit
      // output (19); more are reachable through overrides
      const int cap_warps = max_consumer_warps(nch, packed);
      const int plan_warps =
          ((packed && c.od != FAR_F32) || cap_warps < kMaxConsumerWarps) ? cap_warps : kMaxConsumerWarps;
      groups = one_group ? 1 : plan_warps / G;
      if (groups > group_cap) groups = group_cap;
      if (groups > rows_per_sm) groups = (int)(rows_per_sm > 0 ? rows_per_sm : 1);
      if (g_force_groups.load() > 0 && g_force_groups.load() * G <= max_consumer_warps(nch, packed))
        groups = g_force_groups.load();
      stage_bytes = (uint32_t)(((row_bytes + 127) / 128 * 128) * (c.residual ? 2 : 1));
      int want = one_group ? 4 : groups * slots_per_group;
      if (want < 2) want = 2;
      // as many ring slots as wanted and as fit in shared memory
      stages = want > 32 ? 32 : want;
      while (stages >= 2 && staged_smem_bytes(stages, groups, G, w_bytes, stage_bytes, c.quant, c.ln) > (size_t)kMaxDynamicSmem)
        --stages;
      const int forced = g_force_stages.load();
      if (forced >= 2) {
        stages = forced;
        while (stages >= 2 && staged_smem_bytes(stages, groups, G, w_bytes, stage_bytes, c.quant, c.ln) > (size_t)kMaxDynamicSmem)
          --stages;
      }
      if (groups > stages) groups = stages;
      // Each ring slot must belong to one group (stages a multiple of groups):
      // then every wait on a slot's barriers is for the phase right after the
      // one its waiter saw complete, which is all a parity wait can tell apart.
      stages -= stages % groups;
      if (stages < 2) {
        staged = false;
      } else {
        smem = staged_smem_bytes(stages, groups, G, w_bytes, stage_bytes, c.quant, c.ln);
      }
    }
  }
  if (staged) {
    L.kind = kStaged;
    L.nch = nch;
    L.exact = (row_bytes / 16) == (int64_t)nch * G * 32;
    p.chunks = (int32_t)(row_bytes / 16);
    p.warps_per_row = G;
    p.groups = groups;
    p.stages = stages;
    p.row_bytes = (uint32_t)row_bytes;
    p.w_smem_bytes = w_bytes;
    p.stage_bytes = stage_bytes;
    int64_t grid = (c.tokens + groups - 1) / groups;
    if (grid > sms) grid = sms;
    L.grid = dim3((unsigned)grid);
    L.block = dim3((unsigned)((1 + groups * G) * 32));
    L.smem = smem;
  } else {
    L.kind = kGeneric;
    int64_t grid = c.tokens < (int64_t)sms * 8 ? c.tokens : (int64_t)sms * 8;
    L.grid = dim3((unsigned)grid);
    L.block = dim3(kGenericThreads);
    L.smem = 0;
  }
  return FAR_OK;
}

// Rows a claim for a call's launch under schedule `mode`, or 0 for the fixed stride (host
// logic only; whether a counter pair is free, or the stream capturing, is decided at
// launch). Rows a claim: as few as keep the claims below ~150 M/s at the copy rate
// (~6.8 TB/s), well under the ~250 M/s that one counter's atomics were measured to sustain
// on GB300. Claimed rows by the automatic rule where that is one or two rows (rows moving
// 23 KB or more) and at least three times as many rows are left after every CTA's first
// ring-full as those take: on shorter rows the fixed stride was as fast or faster, and on
// launches of fewer ring-fulls the claims' round trips delay the loads more than the
// balance gains (bf16 / fp32-weight 4096 x 4096 variant, 2.7 ring-fulls a CTA: 19.7 us
// against 18.0 at the fixed stride); forced, wherever rows are left.
// Also three rows a claim for the packed no-residual kernels on 16-bit rows (RMSNorm with a
// 16-bit out, or a quantised out) with at least eight ring-fulls of rows and a row that is
// not a whole number of 256 chunks: there the fixed stride loses 7-16 % when the launch
// follows another on the stream (dirty lines of the one ahead written back meanwhile)
// and claims cost at most ~1.5 % after an L2 flush (bf16 16384 x 5120: 53.3 us against 59.9
// in a stream, 53.7 against 52.9 after a flush; 32768 x 4608 90.9 against 105.8 and 94.2
// against 94.7; fp16 24576 x 5120 76.7 against 88.2 and 76.1 against 80.5; int8 out within
// -0.1 / +2.6 % either way). Rows of whole 256-chunk multiples keep the stride (hidden
// 4096: claims 2.8 % slower in a stream, 10 % after a flush).
int64_t claim_rows_for(const Call& c, const Launch& L, int mode) {
  if (L.kind != kStaged || c.fixed_stride || mode == 1) return 0;
  // bytes a row moves: x (and the residual and residual_out), then out, or the quantised
  // codes plus the row's binary32 scale (LayerNorm's beta, like the weight, is read once a
  // launch, not a row)
  const int64_t row_traffic = c.hidden * (dsize(c.act) * (c.residual ? 3 : 1) + (c.quant ? 1 : dsize(c.od))) +
                              (c.quant ? 4 : 0);
  const int64_t claim_rows = (45333 + row_traffic - 1) / row_traffic;
  const int64_t r0 = (int64_t)L.grid.x * L.p.stages;
  const bool packed16 = !c.residual && !c.ln && c.act != FAR_F32 && (c.quant || c.od != FAR_F32);
  const int64_t chunks = c.hidden * dsize(c.act) / 16;
  if (mode == 2 ? c.tokens > r0
                : ((claim_rows <= 2 && c.tokens >= 4 * r0) ||
                   (packed16 && claim_rows == 3 && c.tokens >= 8 * r0 && chunks % 256 != 0)))
    return claim_rows < (1 << 20) ? claim_rows : (1 << 20);
  return 0;
}

// Rows a CTA takes at the fixed stride before it claims (with claimed rows): its first
// ring-full, except for the automatic rule's three-row claims of the packed kernels, which
// claim only the last quarter of a CTA's share. bf16 16384 x 5120, after an L2 flush / in a
// stream: 52.8 / 54.2 us against 53.4 / 54.2 claiming from the first ring-full and 53.4 /
// 59.7 at the fixed stride. (Claims from the first ring-full stay best where they take one
// or two rows: fp16 65536 x 8192 variant 303 us against 307 with the last quarter claimed.)
int64_t static_rows_for(const Call& c, const Launch& L, int mode) {
  const int64_t ring = L.p.stages;
  if (mode != 0 || claim_rows_for(c, L, mode) != 3) return ring;
  const int64_t per = c.tokens / (int64_t)L.grid.x;
  const int64_t s = per - (per + 3) / 4;
  return s > ring ? (s < (1 << 30) ? s : (1 << 30)) : ring;
}

int launch(const Call& c, const DeviceState& dev, cudaStream_t stream) {
  g_last_claimed = 0;
  if (c.tokens == 0) return FAR_OK;
  Launch L;
  int st = plan(c, dev.sms, dev.status, stream, L);
  if (st != FAR_OK) return st;
  const int mode = g_row_schedule.load();
  const int64_t claim_rows = claim_rows_for(c, L, mode);
  int pair = -1;
  const int devno = (int)(&dev - g_dev);
  if (claim_rows > 0) {
    pair = sched_acquire(devno, stream);
    // a capture begun on another thread since the pair was taken: give it back unused
    if (pair >= 0 && stream_capturing(stream)) {
      sched_release(devno, pair, stream, false);
      pair = -1;
    }
    if (pair >= 0) {
      L.p.sched = g_sched_pool[devno].pairs + 2 * pair;
      L.p.sched_run = (int32_t)claim_rows;
      L.p.sched_static = (int32_t)static_rows_for(c, L, mode);
    }
  }
  cudaError_t e;
  if (c.ln) {
    switch (c.act) {
      case FAR_F16: e = launch_ln_act_f16(c.wd, c.residual, L); break;
      case FAR_BF16: e = launch_ln_act_bf16(c.wd, c.residual, L); break;
      default: e = launch_ln_act_f32(c.wd, c.residual, L); break;
    }
  } else if (c.quant) {
    switch (c.act) {
      case FAR_F16: e = launch_q_act_f16(c.wd, c.residual, L); break;
      case FAR_BF16: e = launch_q_act_bf16(c.wd, c.residual, L); break;
      default: e = launch_q_act_f32(c.wd, c.residual, L); break;
    }
  } else {
    switch (c.act) {
      case FAR_F16: e = launch_act_f16(c.wd, c.residual, L); break;
      case FAR_BF16: e = launch_act_bf16(c.wd, c.residual, L); break;
      default: e = launch_act_f32(c.wd, c.residual, L); break;
    }
  }
  if (pair >= 0) sched_release(devno, pair, stream, e == cudaSuccess);
  g_last_claimed = pair >= 0 && e == cudaSuccess;
  return e == cudaSuccess ? FAR_OK : cuda_fail(e);
}

int run(const void* x, const void* r, const void* w, float eps, void* out, void* res_out, int64_t tokens,
        int64_t hidden, int dtype, bool residual, void* stream, const Strides* strides = nullptr,
        bool fixed_stride = false) {
  Call c;
  int st = validate(x, r, w, eps, out, res_out, tokens, hidden, dtype, residual, c, strides);
  if (st != FAR_OK || tokens == 0) return st;
  c.fixed_stride = fixed_stride;
  DeviceState* dev = nullptr;
  st = current_device(dev);
  if (st != FAR_OK) return st;
  return launch(c, *dev, static_cast<cudaStream_t>(stream));
}

int run_quant(const void* x, const void* r, const void* w, float eps, void* q, float* scale, void* res_out,
              int64_t tokens, int64_t hidden, int dtype, int qtype, bool residual, void* stream,
              const Strides* strides = nullptr) {
  Call c;
  int st = validate_quant(x, r, w, eps, q, scale, res_out, tokens, hidden, dtype, qtype, residual, c, strides);
  if (st != FAR_OK || tokens == 0) return st;
  DeviceState* dev = nullptr;
  st = current_device(dev);
  if (st != FAR_OK) return st;
  return launch(c, *dev, static_cast<cudaStream_t>(stream));
}

int run_ln(const void* x, const void* r, const void* gamma, const void* beta, float eps, void* out, void* res_out,
           int64_t tokens, int64_t hidden, int dtype, bool residual, void* stream, const Strides* strides = nullptr) {
  Call c;
  int st = validate_ln(x, r, gamma, beta, eps, out, res_out, tokens, hidden, dtype, residual, c, strides);
  if (st != FAR_OK || tokens == 0) return st;
  DeviceState* dev = nullptr;
  st = current_device(dev);
  if (st != FAR_OK) return st;
  return launch(c, *dev, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// host-buffer pipeline
// ---------------------------------------------------------------------------

int64_t align256(int64_t n) { return (n + 255) / 256 * 256; }

struct HostLayout {
  int64_t w_bytes, x_bytes, o_bytes;  // per chunk of `rows` rows
  int64_t total;
};

enum HostOp { kHostRms = 0, kHostLn = 1, kHostQuant = 2 };

HostLayout host_layout(int64_t rows, int64_t hidden, int act, int wd, int od, bool residual, int op = kHostRms) {
  HostLayout h;
  h.w_bytes = align256(hidden * dsize(wd)) * (op == kHostLn ? 2 : 1);  // the weight (LayerNorm: gamma, beta)
  h.x_bytes = align256(rows * hidden * dsize(act));
  // out, or for a quantised output q (one byte an element) and the per-row scales
  h.o_bytes = op == kHostQuant ? align256(rows * hidden) + align256(rows * 4) : align256(rows * hidden * dsize(od));
  // per slot: x, (residual, residual_out), out
  int64_t slot = h.x_bytes * (residual ? 3 : 1) + h.o_bytes;
  h.total = h.w_bytes + 2 * slot;
  return h;
}

int ensure_pipe(DeviceState& d) {
  if (d.pipe_ready) return FAR_OK;
  for (int i = 0; i < 2; ++i) {
    cudaError_t e = cudaStreamCreateWithFlags(&d.pipe[i], cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaEventCreateWithFlags(&d.join[i], cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  cudaError_t e = cudaEventCreateWithFlags(&d.fork, cudaEventDisableTiming);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaEventCreateWithFlags(&d.wready, cudaEventDisableTiming);
  if (e != cudaSuccess) return cuda_fail(e);
  d.pipe_ready = true;
  return FAR_OK;
}

// The host-buffer pipeline for a validated call `c` whose pointers are host buffers:
// row chunks stream through the two slots of `workspace` on two internal streams (copy in,
// kernel, copy out), after the weight (and LayerNorm's beta) is copied once.
int run_host_call(const Call& c, void* workspace, int64_t ws_bytes, void* stream) {
  if (c.tokens == 0) return FAR_OK;
  if (!workspace) return FAR_ERR_NULL;
  if (!aligned16(workspace)) return FAR_ERR_WORKSPACE;
  const int op = c.ln ? kHostLn : c.quant ? kHostQuant : kHostRms;
  const int64_t tokens = c.tokens, hidden = c.hidden;
  const bool residual = c.residual;
  // the largest chunk of rows whose two slots fit the workspace (the layout grows with rows)
  if (host_layout(1, hidden, c.act, c.wd, c.od, residual, op).total > ws_bytes) return FAR_ERR_WORKSPACE;
  int64_t lo = 1, hi = tokens;
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo + 1) / 2;
    if (host_layout(mid, hidden, c.act, c.wd, c.od, residual, op).total <= ws_bytes) lo = mid;
    else hi = mid - 1;
  }
  const int64_t rows = lo;
  DeviceState* dev = nullptr;
  int st = current_device(dev);
  if (st != FAR_OK) return st;
  std::lock_guard<std::mutex> lk(dev->pipe_mu);
  st = ensure_pipe(*dev);
  if (st != FAR_OK) return st;

  const HostLayout lay = host_layout(rows, hidden, c.act, c.wd, c.od, residual, op);
  char* base = static_cast<char*>(workspace);
  char* w_dev = base;
  char* beta_dev = base + align256(hidden * dsize(c.wd));
  char* slot_base[2] = {base + lay.w_bytes, base + lay.w_bytes + (lay.total - lay.w_bytes) / 2};
  const int64_t sa = dsize(c.act), so = op == kHostQuant ? 1 : dsize(c.od);
  cudaStream_t caller = static_cast<cudaStream_t>(stream);

  cudaError_t e = cudaEventRecord(dev->fork, caller);
  for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(dev->pipe[i], dev->fork, 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(w_dev, c.w, hidden * dsize(c.wd), cudaMemcpyHostToDevice, dev->pipe[0]);
  if (e == cudaSuccess && op == kHostLn)
    e = cudaMemcpyAsync(beta_dev, c.beta, hidden * dsize(c.wd), cudaMemcpyHostToDevice, dev->pipe[0]);
  if (e == cudaSuccess) e = cudaEventRecord(dev->wready, dev->pipe[0]);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(dev->pipe[1], dev->wready, 0);
  if (e != cudaSuccess) return cuda_fail(e);

  int64_t chunk = 0;
  for (int64_t t0 = 0; t0 < tokens; t0 += rows, ++chunk) {
    const int64_t n = (tokens - t0 < rows) ? tokens - t0 : rows;
    const int s = (int)(chunk & 1);
    cudaStream_t ps = dev->pipe[s];
    char* xd = slot_base[s];
    char* od = xd + lay.x_bytes;                         // out, or q then the scales
    char* scd = od + align256(rows * hidden);            // the scales (quantised output)
    char* rd = od + lay.o_bytes;
    char* rod = rd + lay.x_bytes;
    const int64_t in_off = t0 * hidden * sa, out_off = t0 * hidden * so;
    e = cudaMemcpyAsync(xd, static_cast<const char*>(c.x) + in_off, n * hidden * sa, cudaMemcpyHostToDevice, ps);
    if (e == cudaSuccess && residual)
      e = cudaMemcpyAsync(rd, static_cast<const char*>(c.r) + in_off, n * hidden * sa, cudaMemcpyHostToDevice, ps);
    if (e != cudaSuccess) return cuda_fail(e);
    Call cc = c;
    cc.x = xd;
    cc.r = residual ? rd : nullptr;
    cc.w = w_dev;
    cc.beta = op == kHostLn ? beta_dev : nullptr;
    cc.out = op == kHostQuant ? nullptr : od;
    cc.q = op == kHostQuant ? od : nullptr;
    cc.scale = op == kHostQuant ? reinterpret_cast<float*>(scd) : nullptr;
    cc.res_out = residual ? rod : nullptr;
    cc.tokens = n;
    cc.st = Strides{hidden, hidden, hidden, hidden};  // the workspace slots are contiguous
    st = launch(cc, *dev, ps);
    if (st != FAR_OK) return st;
    void* out_host = op == kHostQuant ? c.q : c.out;
    e = cudaMemcpyAsync(static_cast<char*>(out_host) + out_off, od, n * hidden * so, cudaMemcpyDeviceToHost, ps);
    if (e == cudaSuccess && op == kHostQuant)
      e = cudaMemcpyAsync(c.scale + t0, scd, n * 4, cudaMemcpyDeviceToHost, ps);
    if (e == cudaSuccess && residual)
      e = cudaMemcpyAsync(static_cast<char*>(c.res_out) + in_off, rod, n * hidden * sa, cudaMemcpyDeviceToHost, ps);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  for (int i = 0; i < 2; ++i) {
    e = cudaEventRecord(dev->join[i], dev->pipe[i]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(caller, dev->join[i], 0);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return FAR_OK;
}

int run_host(const void* x, const void* r, const void* w, float eps, void* out, void* res_out, int64_t tokens,
             int64_t hidden, int dtype, bool residual, void* workspace, int64_t ws_bytes, void* stream) {
  Call c;
  int st = validate(x, r, w, eps, out, res_out, tokens, hidden, dtype, residual, c);
  if (st != FAR_OK || tokens == 0) return st;
  return run_host_call(c, workspace, ws_bytes, stream);
}

// ---------------------------------------------------------------------------
// bounded-wait self test
// ---------------------------------------------------------------------------

__global__ void wait_selftest_kernel(unsigned int* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: the wait runs out and records the time-out
  if (threadIdx.x == 0) mbar_wait(smem_addr(&bar), 0u, timeout_ns, status);
}

std::mutex g_attr_mu;
std::set<std::pair<const void*, int>> g_attr_done;

}  // namespace

cudaError_t ensure_smem_attribute(const void* func, size_t bytes) {
  (void)bytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (g_attr_done.count({func, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynamicSmem);
  if (e == cudaSuccess) g_attr_done.insert({func, dev});
  return e;
}

int check_call(const void* x, const void* r, const void* w, float eps, void* out, void* res_out, int64_t tokens,
               int64_t hidden, int dtype, bool residual, int* act, int* wd, int* od) {
  Call c;
  const int st = validate(x, r, w, eps, out, res_out, tokens, hidden, dtype, residual, c);
  if (st == FAR_OK) {
    *act = c.act;
    *wd = c.wd;
    *od = c.od;
  }
  return st;
}

// the allocation-free entry point's launches: fixed-stride rows, so no counter pair and no
// event is created or recorded for them
int enqueue_device_call(const void* x, const void* r, const void* w, float eps, void* out, void* res_out,
                        int64_t tokens, int64_t hidden, int dtype, bool residual, cudaStream_t stream) {
  return run(x, r, w, eps, out, res_out, tokens, hidden, dtype, residual, stream, nullptr, true);
}

int device_info(unsigned int** status, int* sms) {
  DeviceState* dev = nullptr;
  int st = current_device(dev);
  if (st != FAR_OK) return st;
  *status = dev->status;
  *sms = dev->sms;
  return FAR_OK;
}

int cuda_error_status(cudaError_t e) { return cuda_fail(e); }

cudaError_t launch_wait_selftest(unsigned int* status, uint64_t timeout_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace far

using namespace far;

extern "C" {

int fused_add_rmsnorm(const void* x, const void* residual, const void* weight, float eps, void* out,
                      void* residual_out, int64_t tokens, int64_t hidden, int dtype, void* stream) {
  return run(x, residual, weight, eps, out, residual_out, tokens, hidden, dtype, true, stream);
}

int rmsnorm(const void* x, const void* weight, float eps, void* out, int64_t tokens, int64_t hidden, int dtype,
            void* stream) {
  return run(x, nullptr, weight, eps, out, nullptr, tokens, hidden, dtype, false, stream);
}

int fused_add_rmsnorm_strided(const void* x, int64_t x_row_stride, const void* residual,
                              int64_t residual_row_stride, const void* weight, float eps, void* out,
                              int64_t out_row_stride, void* residual_out, int64_t residual_out_row_stride,
                              int64_t tokens, int64_t hidden, int dtype, void* stream) {
  const Strides sd{x_row_stride, residual_row_stride, out_row_stride, residual_out_row_stride};
  return run(x, residual, weight, eps, out, residual_out, tokens, hidden, dtype, true, stream, &sd);
}

int far_validate_strided(const void* x, int64_t x_row_stride, const void* residual, int64_t residual_row_stride,
                         const void* weight, float eps, const void* out, int64_t out_row_stride,
                         const void* residual_out, int64_t residual_out_row_stride, int64_t tokens, int64_t hidden,
                         int dtype, int has_residual) {
  const Strides sd{x_row_stride, has_residual ? residual_row_stride : hidden, out_row_stride,
                   has_residual ? residual_out_row_stride : hidden};
  Call c;
  return validate(x, has_residual ? residual : nullptr, weight, eps, const_cast<void*>(out),
                  has_residual ? const_cast<void*>(residual_out) : nullptr, tokens, hidden, dtype, has_residual != 0, c,
                  &sd);
}

int rmsnorm_strided(const void* x, int64_t x_row_stride, const void* weight, float eps, void* out,
                    int64_t out_row_stride, int64_t tokens, int64_t hidden, int dtype, void* stream) {
  const Strides sd{x_row_stride, hidden, out_row_stride, hidden};
  return run(x, nullptr, weight, eps, out, nullptr, tokens, hidden, dtype, false, stream, &sd);
}

int fused_add_rmsnorm_quant(const void* x, const void* residual, const void* weight, float eps, void* q,
                            float* scale, void* residual_out, int64_t tokens, int64_t hidden, int dtype, int qtype,
                            void* stream) {
  return run_quant(x, residual, weight, eps, q, scale, residual_out, tokens, hidden, dtype, qtype, true, stream);
}

int rmsnorm_quant(const void* x, const void* weight, float eps, void* q, float* scale, int64_t tokens,
                  int64_t hidden, int dtype, int qtype, void* stream) {
  return run_quant(x, nullptr, weight, eps, q, scale, nullptr, tokens, hidden, dtype, qtype, false, stream);
}

int fused_add_layernorm(const void* x, const void* residual, const void* gamma, const void* beta, float eps,
                        void* out, void* residual_out, int64_t tokens, int64_t hidden, int dtype, void* stream) {
  return run_ln(x, residual, gamma, beta, eps, out, residual_out, tokens, hidden, dtype, true, stream);
}

int layernorm(const void* x, const void* gamma, const void* beta, float eps, void* out, int64_t tokens,
              int64_t hidden, int dtype, void* stream) {
  return run_ln(x, nullptr, gamma, beta, eps, out, nullptr, tokens, hidden, dtype, false, stream);
}

int fused_add_layernorm_strided(const void* x, int64_t x_row_stride, const void* residual,
                                int64_t residual_row_stride, const void* gamma, const void* beta, float eps, void* out,
                                int64_t out_row_stride, void* residual_out, int64_t residual_out_row_stride,
                                int64_t tokens, int64_t hidden, int dtype, void* stream) {
  const Strides sd{x_row_stride, residual_row_stride, out_row_stride, residual_out_row_stride};
  return run_ln(x, residual, gamma, beta, eps, out, residual_out, tokens, hidden, dtype, true, stream, &sd);
}

int layernorm_strided(const void* x, int64_t x_row_stride, const void* gamma, const void* beta, float eps, void* out,
                      int64_t out_row_stride, int64_t tokens, int64_t hidden, int dtype, void* stream) {
  const Strides sd{x_row_stride, hidden, out_row_stride, hidden};
  return run_ln(x, nullptr, gamma, beta, eps, out, nullptr, tokens, hidden, dtype, false, stream, &sd);
}

int fused_add_rmsnorm_quant_strided(const void* x, int64_t x_row_stride, const void* residual,
                                    int64_t residual_row_stride, const void* weight, float eps, void* q, float* scale,
                                    void* residual_out, int64_t residual_out_row_stride, int64_t tokens,
                                    int64_t hidden, int dtype, int qtype, void* stream) {
  const Strides sd{x_row_stride, residual_row_stride, hidden, residual_out_row_stride};
  return run_quant(x, residual, weight, eps, q, scale, residual_out, tokens, hidden, dtype, qtype, true, stream, &sd);
}

int rmsnorm_quant_strided(const void* x, int64_t x_row_stride, const void* weight, float eps, void* q, float* scale,
                          int64_t tokens, int64_t hidden, int dtype, int qtype, void* stream) {
  const Strides sd{x_row_stride, hidden, hidden, hidden};
  return run_quant(x, nullptr, weight, eps, q, scale, nullptr, tokens, hidden, dtype, qtype, false, stream, &sd);
}

int far_output_dtype(int dtype) {
  int act, wd, od;
  int st = decode(dtype, act, wd, od);
  return st == FAR_OK ? od : -st;
}

const char* far_status_string(int status) {
  switch (status) {
    case FAR_OK: return "ok";
    case FAR_ERR_DTYPE_MIX: return "fp16 mixed with bf16 is rejected by the dtype policy";
    case FAR_ERR_DTYPE: return "unknown dtype code";
    case FAR_ERR_NULL: return "a required pointer is NULL";
    case FAR_ERR_SHAPE: return "invalid shape (hidden must be 1..2^24, tokens >= 0)";
    case FAR_ERR_ALIAS: return "an output overlaps another buffer (only exact in-place aliasing is allowed)";
    case FAR_ERR_EPS: return "eps must be finite and non-negative";
    case FAR_ERR_CUDA: return g_cuda_msg;
    case FAR_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out; its outputs are incomplete";
    case FAR_ERR_WORKSPACE: return "workspace too small or misaligned for one row";
    case FAR_ERR_SCRATCH:
      return "one row (plus the weight) does not fit the fixed device scratch of the allocation-free entry point";
    default: return "unknown status";
  }
}

int far_device_status(void* stream) {
  DeviceState* dev = nullptr;
  int st = current_device(dev);
  if (st != FAR_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int word = 0;
  e = cudaMemcpy(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (word != 0) {
    e = cudaMemset(dev->status, 0, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (word & (1u << FAR_ERR_TIMEOUT)) return FAR_ERR_TIMEOUT;
  return word ? FAR_ERR_SHAPE : FAR_OK;  // a kernel refused an inconsistent launch plan
}

int64_t far_host_workspace_bytes(int64_t chunk_tokens, int64_t hidden, int dtype, int has_residual) {
  int act, wd, od;
  int st = decode(dtype, act, wd, od);
  if (st != FAR_OK) return -st;
  if (chunk_tokens <= 0 || hidden <= 0 || hidden > kMaxHidden) return -FAR_ERR_SHAPE;
  return host_layout(chunk_tokens, hidden, act, wd, od, has_residual != 0).total;
}

int64_t far_host_workspace_bytes_op(int64_t chunk_tokens, int64_t hidden, int dtype, int has_residual, int op) {
  int act, wd, od;
  int st = decode(dtype, act, wd, od);
  if (st != FAR_OK) return -st;
  if (chunk_tokens <= 0 || hidden <= 0 || hidden > kMaxHidden || op < 0 || op > 2) return -FAR_ERR_SHAPE;
  return host_layout(chunk_tokens, hidden, act, wd, od, has_residual != 0, op).total;
}

int fused_add_layernorm_host(const void* x, const void* residual, const void* gamma, const void* beta, float eps,
                             void* out, void* residual_out, int64_t tokens, int64_t hidden, int dtype,
                             void* workspace, int64_t workspace_bytes, void* stream) {
  Call c;
  int st = validate_ln(x, residual, gamma, beta, eps, out, residual_out, tokens, hidden, dtype, true, c);
  return (st != FAR_OK || tokens == 0) ? st : run_host_call(c, workspace, workspace_bytes, stream);
}

int layernorm_host(const void* x, const void* gamma, const void* beta, float eps, void* out, int64_t tokens,
                   int64_t hidden, int dtype, void* workspace, int64_t workspace_bytes, void* stream) {
  Call c;
  int st = validate_ln(x, nullptr, gamma, beta, eps, out, nullptr, tokens, hidden, dtype, false, c);
  return (st != FAR_OK || tokens == 0) ? st : run_host_call(c, workspace, workspace_bytes, stream);
}

int fused_add_rmsnorm_quant_host(const void* x, const void* residual, const void* weight, float eps, void* q,
                                 float* scale, void* residual_out, int64_t tokens, int64_t hidden, int dtype,
                                 int qtype, void* workspace, int64_t workspace_bytes, void* stream) {
  Call c;
  int st = validate_quant(x, residual, weight, eps, q, scale, residual_out, tokens, hidden, dtype, qtype, true, c);
  return (st != FAR_OK || tokens == 0) ? st : run_host_call(c, workspace, workspace_bytes, stream);
}

int rmsnorm_quant_host(const void* x, const void* weight, float eps, void* q, float* scale, int64_t tokens,
                       int64_t hidden, int dtype, int qtype, void* workspace, int64_t workspace_bytes,
                       void* stream) {
  Call c;
  int st = validate_quant(x, nullptr, weight, eps, q, scale, nullptr, tokens, hidden, dtype, qtype, false, c);
  return (st != FAR_OK || tokens == 0) ? st : run_host_call(c, workspace, workspace_bytes, stream);
}

int fused_add_rmsnorm_host(const void* x, const void* residual, const void* weight, float eps, void* out,
                           void* residual_out, int64_t tokens, int64_t hidden, int dtype, void* workspace,
                           int64_t workspace_bytes, void* stream) {
  return run_host(x, residual, weight, eps, out, residual_out, tokens, hidden, dtype, true, workspace,
                  workspace_bytes, stream);
}

int rmsnorm_host(const void* x, const void* weight, float eps, void* out, int64_t tokens, int64_t hidden,
                 int dtype, void* workspace, int64_t workspace_bytes, void* stream) {
  return run_host(x, nullptr, weight, eps, out, nullptr, tokens, hidden, dtype, false, workspace,
                  workspace_bytes, stream);
}

int far_selftest_wait_timeout(uint32_t timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 10000000u) return FAR_ERR_SHAPE;
  DeviceState* dev = nullptr;
  int st = current_device(dev);
  if (st != FAR_OK) return st;
  cudaError_t e = launch_wait_selftest(dev->status, (uint64_t)timeout_us * 1000ull, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FAR_OK : cuda_fail(e);
}

int far_set_launch_override(int kind, int nch, int groups, int stages) {
  if (kind < -1 || kind > 1 || (nch != 0 && nch != 1 && nch != 2 && nch != 4 && nch != 5 && nch != 6 && nch != 8 &&
                                   nch != 10) ||
      groups < 0 ||
      groups > kMaxPackedWarps || stages < 0 || stages > 32)
    return FAR_ERR_SHAPE;
  g_force_kind = kind;
  g_force_nch = nch;
  g_force_groups = groups;
  g_force_stages = stages;
  return FAR_OK;
}

int far_set_row_schedule(int mode) {
  if (mode < 0 || mode > 2) return FAR_ERR_SHAPE;
  g_row_schedule = mode;
  return FAR_OK;
}

int far_get_row_schedule(void) { return g_row_schedule.load(); }

int far_set_programmatic_launch(int enable) {
  if (enable != 0 && enable != 1) return FAR_ERR_SHAPE;
  g_programmatic = enable;
  return FAR_OK;
}

int far_get_programmatic_launch(void) { return g_programmatic.load(); }

int far_last_launch_claimed_rows(void) { return g_last_claimed; }

int far_sched_pool_model(const int64_t* ops, int n, int* results) {
  if (n < 0 || (n > 0 && (!ops || !results))) return FAR_ERR_SHAPE;
  PoolBook book;
  for (int i = 0; i < n; ++i) {
    const int64_t op = ops[3 * i], a = ops[3 * i + 1], b = ops[3 * i + 2];
    if (op == 1) {
      const uint64_t done = (uint64_t)b;
      results[i] = book.acquire((unsigned long long)a, [&](int s) { return (int)((done >> s) & 1u); });
    } else if (op == 2) {
      if (a < 0 || a >= kSchedSlots || book.pending[a] <= 0) return FAR_ERR_SHAPE;
      book.release((int)a, (b & 1) != 0, (b & 2) != 0);
      results[i] = 0;
    } else {
      return FAR_ERR_SHAPE;
    }
  }
  return FAR_OK;
}

int far_plan_for_sms(int64_t tokens, int64_t hidden, int dtype, int has_residual, int sms, int* out8) {
  // kind, nch, warps per row, groups, stages, grid, threads per CTA, dynamic shared bytes
  if (sms < 1 || !out8) return FAR_ERR_SHAPE;
  PlanQuery query;  // stand-in addresses: no overlap check
  Call c;
  // distinct, aligned, non-overlapping stand-in addresses: only the plan is computed
  const char* base = reinterpret_cast<const char*>((uintptr_t)1 << 40);
  const uint64_t span = (uint64_t)tokens * hidden * 4 + 4096;
  const void* x = base;
  const void* r = base + span;
  const void* w = base + 2 * span;
  void* o = const_cast<char*>(base + 3 * span);
  void* ro = const_cast<char*>(base + 4 * span);
  int st = validate(x, has_residual ? r : nullptr, w, 1e-6f, o, has_residual ? ro : nullptr, tokens, hidden,
                    dtype, has_residual != 0, c);
  if (st != FAR_OK) return st;
  if (tokens == 0) return FAR_ERR_SHAPE;
  Launch L;
  st = plan(c, sms, nullptr, nullptr, L);
  if (st != FAR_OK) return st;
  out8[0] = L.kind;
  out8[1] = L.nch;
  out8[2] = L.p.warps_per_row;
  out8[3] = L.p.groups;
  out8[4] = L.p.stages;
  out8[5] = (int)L.grid.x;
  out8[6] = (int)L.block.x;
  out8[7] = (int)L.smem;
  return FAR_OK;
}

int far_row_schedule_for_sms(int64_t tokens, int64_t hidden, int dtype, int has_residual, int op, int sms,
                             int* rows_per_claim) {
  if (sms < 1 || !rows_per_claim || op < 0 || op > 2) return FAR_ERR_SHAPE;
  PlanQuery query;  // stand-in addresses: no overlap check
  Call c;
  const char* base = reinterpret_cast<const char*>((uintptr_t)1 << 40);
  char* mb = const_cast<char*>(base);
  const uint64_t span = (uint64_t)tokens * hidden * 4 + 4096;
  const void* r = has_residual ? base + span : nullptr;
  void* ro = has_residual ? mb + 4 * span : nullptr;
  int st;
  if (op == 0)
    st = validate(base, r, base + 2 * span, 1e-6f, mb + 3 * span, ro, tokens, hidden, dtype, has_residual != 0, c);
  else if (op == 1)
    st = validate_ln(base, r, base + 2 * span, base + 5 * span, 1e-6f, mb + 3 * span, ro, tokens, hidden, dtype,
                     has_residual != 0, c);
  else
    st = validate_quant(base, r, base + 2 * span, 1e-6f, mb + 3 * span, reinterpret_cast<float*>(mb + 5 * span), ro,
                        tokens, hidden, dtype, FAR_Q_INT8, has_residual != 0, c);
  if (st != FAR_OK) return st;
  if (tokens == 0) return FAR_ERR_SHAPE;
  Launch L;
  st = plan(c, sms, nullptr, nullptr, L);
  if (st != FAR_OK) return st;
  *rows_per_claim = (int)claim_rows_for(c, L, g_row_schedule.load());
  return FAR_OK;
}

int far_plan_quant_for_sms(int64_t tokens, int64_t hidden, int dtype, int has_residual, int qtype, int sms,
                           int* out8) {
  if (sms < 1 || !out8) return FAR_ERR_SHAPE;
  PlanQuery query;  // stand-in addresses: no overlap check
  Call c;
  const char* base = reinterpret_cast<const char*>((uintptr_t)1 << 40);
  const uint64_t span = (uint64_t)tokens * hidden * 4 + 4096;
  int st = validate_quant(base, has_residual ? base + span : nullptr, base + 2 * span, 1e-6f,
                          const_cast<char*>(base + 3 * span), reinterpret_cast<float*>(const_cast<char*>(base + 5 * span)),
                          has_residual ? const_cast<char*>(base + 4 * span) : nullptr, tokens, hidden, dtype, qtype,
                          has_residual != 0, c);
  if (st != FAR_OK) return st;
  if (tokens == 0) return FAR_ERR_SHAPE;
  Launch L;
  st = plan(c, sms, nullptr, nullptr, L);
  if (st != FAR_OK) return st;
  int vals[8] = {L.kind, L.nch, L.p.warps_per_row, L.p.groups, L.p.stages, (int)L.grid.x, (int)L.block.x, (int)L.smem};
  for (int i = 0; i < 8; ++i) out8[i] = vals[i];
  return FAR_OK;
}

int far_plan_ln_for_sms(int64_t tokens, int64_t hidden, int dtype, int has_residual, int beta_offset, int sms,
                        int* out8) {
  if (sms < 1 || !out8 || beta_offset < 0 || beta_offset > 15) return FAR_ERR_SHAPE;
  PlanQuery query;  // stand-in addresses: no overlap check
  Call c;
  const char* base = reinterpret_cast<const char*>((uintptr_t)1 << 40);
  const uint64_t span = (uint64_t)tokens * hidden * 4 + 4096;
  int st = validate_ln(base, has_residual ? base + span : nullptr, base + 2 * span, base + 5 * span + beta_offset, 1e-6f,
                       const_cast<char*>(base + 3 * span), has_residual ? const_cast<char*>(base + 4 * span) : nullptr,
                       tokens, hidden, dtype, has_residual != 0, c);
  if (st != FAR_OK) return st;
  if (tokens == 0) return FAR_ERR_SHAPE;
  Launch L;
  st = plan(c, sms, nullptr, nullptr, L);
  if (st != FAR_OK) return st;
  int vals[8] = {L.kind, L.nch, L.p.warps_per_row, L.p.groups, L.p.stages, (int)L.grid.x, (int)L.block.x, (int)L.smem};
  for (int i = 0; i < 8; ++i) out8[i] = vals[i];
  return FAR_OK;
}

int far_describe_launch(int64_t tokens, int64_t hidden, int dtype, int has_residual, int* out6) {
  DeviceState* dev = nullptr;
  int st = current_device(dev);
  if (st != FAR_OK) return st;
  int o8[8];
  st = far_plan_for_sms(tokens, hidden, dtype, has_residual, dev->sms, o8);
  if (st != FAR_OK) return st;
  for (int i = 0; i < 6; ++i) out6[i] = o8[i];
  return FAR_OK;
}

}  // extern "C"
