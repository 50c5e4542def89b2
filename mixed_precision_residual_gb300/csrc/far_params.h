// Kernel parameters and the per-activation-dtype launchers shared between the
// C-ABI translation unit and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace far {

// shapes of the staged kernel: a CTA = 1 producer warp + groups x warps_per_row consumer warps.
// 16 consumer warps leave 96 registers a thread (17 warps: 5 on one SM sub-partition);
// 8 chunks a thread (64 values of s) need more, so those CTAs stop at 12 (128 registers).
// The no-residual variant on 16-bit data keeps x packed (s = x exactly), half the
// registers, so it keeps 16 warps at 8 chunks a thread.
constexpr int kMaxConsumerWarps = 16;
__host__ __device__ constexpr bool packed_rows(bool residual, int act) { return !residual && act != 0; }
// Consumer warps a CTA may hold: 12 at 8 chunks a thread (up to 128 registers), 16 below.
// A packed no-residual row (RMSNorm, or RMSNorm with a quantised output, whose kept
// outputs reuse the consumed x's registers) needs at most 96 registers a thread: 19
// consumer warps and the producer put at most 5 warps on each of the SM's four register
// file quarters (16384 registers each), which leaves 96 a thread.
constexpr int kMaxPackedWarps = 19;
__host__ __device__ constexpr int max_consumer_warps(int nch, bool packed = false) {
  return packed ? kMaxPackedWarps : (nch >= 8 ? 12 : 16);
}
__host__ __device__ constexpr int max_threads(int nch, bool packed = false) {
  return (max_consumer_warps(nch, packed) + 1) * 32;
}
constexpr int kMaxDynamicSmem = 227 * 1024;
constexpr int kGenericThreads = 256;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

struct Params {
  const void* x;
  const void* r;         // residual (unused by the no-residual variant)
  const void* w;         // weight [hidden] (gamma of LayerNorm)
  const void* beta;      // LayerNorm shift [hidden], weight dtype
  void* out;             // [tokens, hidden] od
  void* res_out;         // [tokens, hidden] act (unused by the no-residual variant)
  int64_t tokens;
  int32_t hidden;
  float hidden_f;        // (float)hidden, exact for hidden <= 2^24
  float eps;
  int32_t chunks;        // 16-byte chunks per activation row (staged kernel)
  int32_t warps_per_row; // G (staged kernel)
  int32_t groups;        // rows processed concurrently per CTA (staged kernel)
  int32_t stages;        // shared-memory ring slots (staged kernel)
  uint32_t row_bytes;    // hidden * sizeof(act)
  int64_t x_stride;      // bytes between consecutive rows of x
  int64_t r_stride;      // ... of the residual
  int64_t out_stride;    // ... of out
  int64_t res_stride;    // ... of residual_out
  uint32_t w_smem_bytes; // hidden * sizeof(wd), rounded up to 16 (twice that for LayerNorm: gamma, beta)
  uint32_t stage_bytes;  // bytes of one ring slot (x row, then residual row), 128-aligned
  void* q;               // quantised output [tokens, hidden] bytes (quantised variants)
  float* scale;          // per-row scale [tokens] (quantised variants)
  unsigned int* status;  // device error word
  uint64_t timeout_ns;
  // staged kernel: this launch's row counter pair {next row claim, CTAs done}, zero at
  // launch and left zero by the launch's last CTA; null: every CTA takes a fixed stride
  unsigned long long* sched;
  int32_t sched_run;     // rows taken per claim from sched (>= 1)
  int32_t sched_static;  // with sched: rows a CTA takes at the fixed stride before it claims
};

enum Kind { kStaged = 0, kGeneric = 1 };

enum QuantKind { kQuantNone = 0, kQuantInt8 = 1, kQuantFp8 = 2 };

struct Launch {
  Params p;
  int kind;
  int quant;   // QuantKind
  bool ln;     // LayerNorm instead of RMSNorm
  int nch;     // 16-byte chunks per thread (staged kernel): 1, 2, 4 or 8
  bool exact;  // chunks == nch * warps_per_row * 32: no per-chunk bounds test
  dim3 grid, block;
  size_t smem;
  cudaStream_t stream;
  bool programmatic;  // launched as a programmatic dependent launch
};

// cross-warp reduction buffers per group: two (the sum of squares, double-buffered over
// rows), four with a quantised output (the row maximum too) or for LayerNorm (the sum
// for the mean, then the sum of the squared deviations)
__host__ __device__ constexpr int reduce_buffers(int q, bool ln = false) { return (q || ln) ? 4 : 2; }

// shared-memory bytes the staged kernel needs for a plan
inline size_t staged_smem_bytes(int stages, int groups, int warps_per_row, uint32_t w_smem_bytes,
                                uint32_t stage_bytes, int q = 0, bool ln = false) {
  const int nred = reduce_buffers(q, ln);
  size_t bars = (size_t)(2 * stages + nred * groups) * 8;
  size_t red = (size_t)groups * nred * warps_per_row * 8;
  size_t rows = (size_t)stages * 8;  // the row held by each ring slot
  size_t head = (bars + red + rows + 127) / 128 * 128;
  return head + (w_smem_bytes + 127) / 128 * 128 + (size_t)stages * stage_bytes;
}

// one launcher per activation dtype (each in its own translation unit)
cudaError_t launch_act_f16(int wd, bool residual, const Launch& L);
cudaError_t launch_act_bf16(int wd, bool residual, const Launch& L);
cudaError_t launch_act_f32(int wd, bool residual, const Launch& L);
cudaError_t launch_q_act_f16(int wd, bool residual, const Launch& L);
cudaError_t launch_q_act_bf16(int wd, bool residual, const Launch& L);
cudaError_t launch_q_act_f32(int wd, bool residual, const Launch& L);
cudaError_t launch_ln_act_f16(int wd, bool residual, const Launch& L);
cudaError_t launch_ln_act_bf16(int wd, bool residual, const Launch& L);
cudaError_t launch_ln_act_f32(int wd, bool residual, const Launch& L);

// the argument checks and the device-buffer launch behind the public entry points (far_api.cu)
int check_call(const void* x, const void* r, const void* w, float eps, void* out, void* res_out, int64_t tokens,
               int64_t hidden, int dtype, bool residual, int* act, int* wd, int* od);
int enqueue_device_call(const void* x, const void* r, const void* w, float eps, void* out, void* res_out,
                        int64_t tokens, int64_t hidden, int dtype, bool residual, cudaStream_t stream);

// the current device's error word and SM count, and a CUDA error as a status (far_api.cu)
int device_info(unsigned int** status, int* sms);
int cuda_error_status(cudaError_t e);

// the bounded-wait self test (far_api.cu)
cudaError_t launch_wait_selftest(unsigned int* status, uint64_t timeout_ns, cudaStream_t stream);

}  // namespace far
