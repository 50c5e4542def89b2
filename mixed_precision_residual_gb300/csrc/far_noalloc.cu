// fused_add_rmsnorm_host_noalloc: the host-buffer fused op for callers that
// cannot allocate device memory (see include/far.h).  Its device staging area is
// the fixed array below instead of a caller-provided workspace; it creates no
// stream, event or allocation and runs on the caller's stream alone.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "far.h"
#include "far_params.h"

namespace far {
namespace {

constexpr int kMaxDevices = 64;

// The staging area.  In host code this name is only a stand-in for the device
// symbol, never a device address: the address is looked up per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FAR_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// The scratch's device address on the current device (looked up once per device).
int scratch_address(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FAR_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return FAR_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return FAR_OK;
}

int64_t round256(int64_t n) { return (n + 255) / 256 * 256; }

int elem(int dt) { return dt == FAR_F32 ? 4 : 2; }

}  // namespace
}  // namespace far

extern "C" int fused_add_rmsnorm_host_noalloc(const void* x, const void* residual, const void* weight, float eps,
                                              void* out, void* residual_out, int64_t tokens, int64_t hidden,
                                              int dtype, void* stream) {
  using namespace far;
  int act = 0, wd = 0, od = 0;
  int st = check_call(x, residual, weight, eps, out, residual_out, tokens, hidden, dtype, true, &act, &wd, &od);
  if (st != FAR_OK || tokens == 0) return st;
  const int64_t sa = elem(act), so = elem(od);
  // layout of the scratch: weight | x rows | residual rows | out rows | residual_out rows
  const int64_t w_bytes = round256(hidden * elem(wd));
  const int64_t row_bytes = 3 * round256(hidden * sa) + round256(hidden * so);  // per-row bound, padding included
  if (w_bytes + row_bytes > FAR_NOALLOC_SCRATCH_BYTES) return FAR_ERR_SCRATCH;
  int64_t rows = (FAR_NOALLOC_SCRATCH_BYTES - w_bytes) / row_bytes;
  if (rows > tokens) rows = tokens;
  void* base = nullptr;
  st = scratch_address(&base);
  if (st != FAR_OK) return st;
  char* wdev = static_cast<char*>(base);
  char* xdev = wdev + w_bytes;
  char* rdev = xdev + round256(rows * hidden * sa);
  char* odev = rdev + round256(rows * hidden * sa);
  char* rodev = odev + round256(rows * hidden * so);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (cudaMemcpyAsync(wdev, weight, hidden * elem(wd), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return FAR_ERR_CUDA;
  for (int64_t t0 = 0; t0 < tokens; t0 += rows) {
    const int64_t n = (tokens - t0 < rows) ? tokens - t0 : rows;
    const int64_t in_off = t0 * hidden * sa, out_off = t0 * hidden * so;
    if (cudaMemcpyAsync(xdev, static_cast<const char*>(x) + in_off, n * hidden * sa, cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(rdev, static_cast<const char*>(residual) + in_off, n * hidden * sa, cudaMemcpyHostToDevice,
                        s) != cudaSuccess)
      return FAR_ERR_CUDA;
    st = enqueue_device_call(xdev, rdev, wdev, eps, odev, rodev, n, hidden, dtype, true, s);
    if (st != FAR_OK) return st;
    if (cudaMemcpyAsync(static_cast<char*>(out) + out_off, odev, n * hidden * so, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(static_cast<char*>(residual_out) + in_off, rodev, n * hidden * sa, cudaMemcpyDeviceToHost,
                        s) != cudaSuccess)
      return FAR_ERR_CUDA;
  }
  return FAR_OK;
}
