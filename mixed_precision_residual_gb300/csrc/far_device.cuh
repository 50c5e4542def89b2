// Device helpers for the fused residual-add + RMSNorm kernels (sm_103a).
//
// - dtype traits and exact widening / round-to-nearest-even narrowing,
// - the binary32 double-word accumulator for the row's sum of squares,
// - mbarrier and bulk-copy (cp.async.bulk) wrappers in inline PTX,
// - the bounded wait every kernel uses on every barrier.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "far.h"
#include "far_params.h"

namespace far {

// ---------------------------------------------------------------------------
// dtypes
// ---------------------------------------------------------------------------

template <int DT> struct dtype_size { static constexpr int value = (DT == FAR_F32) ? 4 : 2; };

// the promoted output dtype: fp32 if either operand is fp32, else the common 16-bit type
__host__ __device__ constexpr int promote(int act, int wd) {
  return (act == FAR_F32 || wd == FAR_F32) ? FAR_F32 : act;
}

// widen two packed 16-bit values (low half first) to binary32: exact
template <int DT> __device__ __forceinline__ float2 widen2(uint32_t w);
template <> __device__ __forceinline__ float2 widen2<FAR_F16>(uint32_t w) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}
template <> __device__ __forceinline__ float2 widen2<FAR_BF16>(uint32_t w) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
  return __bfloat1622float2(h);
}

// round two binary32 values to a 16-bit dtype, to nearest even, packed (low half first)
template <int DT> __device__ __forceinline__ uint32_t narrow2(float a, float b);
template <> __device__ __forceinline__ uint32_t narrow2<FAR_F16>(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <> __device__ __forceinline__ uint32_t narrow2<FAR_BF16>(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// V consecutive elements of dtype DT held in 32-bit words, widened to binary32
template <int DT, int V>
__device__ __forceinline__ void widen(const uint32_t* words, float* f) {
  if constexpr (DT == FAR_F32) {
#pragma unroll
    for (int i = 0; i < V; ++i) f[i] = __uint_as_float(words[i]);
  } else {
#pragma unroll
    for (int i = 0; i < V / 2; ++i) {
      float2 p = widen2<DT>(words[i]);
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
}

// V binary32 values rounded to dtype DT (identity for fp32) into 32-bit words
template <int DT, int V>
__device__ __forceinline__ void narrow(const float* f, uint32_t* words) {
  if constexpr (DT == FAR_F32) {
#pragma unroll
    for (int i = 0; i < V; ++i) words[i] = __float_as_uint(f[i]);
  } else {
#pragma unroll
    for (int i = 0; i < V / 2; ++i) words[i] = narrow2<DT>(f[2 * i], f[2 * i + 1]);
  }
}

// a binary32 value rounded to dtype DT and widened back (RNE_DT as a binary32 value)
template <int DT, int V>
__device__ __forceinline__ void round_through(float* f) {
  if constexpr (DT != FAR_F32) {
#pragma unroll
    for (int i = 0; i < V / 2; ++i) {
      float2 p = widen2<DT>(narrow2<DT>(f[2 * i], f[2 * i + 1]));
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
}

// vector memory access of N bytes (N = 8, 16 or 32), N-aligned
template <int N> __device__ __forceinline__ void load_bytes(const void* p, uint32_t* w) {
  if constexpr (N == 8) {
    uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int k = 0; k < N / 16; ++k) {
      uint4 v = reinterpret_cast<const uint4*>(p)[k];
      w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
    }
  }
}

// streaming store (evict-first in L2: the outputs are not re-read by this kernel)
template <int N> __device__ __forceinline__ void store_bytes_stream(void* p, const uint32_t* w) {
  if constexpr (N == 8) {
    asm volatile("st.global.cs.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(w[0]), "r"(w[1]) : "memory");
  } else {
#pragma unroll
    for (int k = 0; k < N / 16; ++k)
      asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(reinterpret_cast<char*>(p) + 16 * k),
                   "r"(w[4 * k]), "r"(w[4 * k + 1]), "r"(w[4 * k + 2]), "r"(w[4 * k + 3])
                   : "memory");
  }
}

// ---------------------------------------------------------------------------
// the row's sum of squares: a binary32 double-word (hi + lo) accumulator
// ---------------------------------------------------------------------------
//
// The contract fixes binary32 accumulation but not the order.  Adding each
// square with an error-free transformation (Knuth's TwoSum, TAOCP vol. 2,
// 4.2.2) and carrying the rounding errors in `lo` keeps hi + lo within about
// 2^-44 (relative) of the exact sum, so the final hi + lo rounded to binary32
// is the correctly rounded sum -- the one order-free binary32 value -- except
// in the astronomically rare rows whose exact sum lies within that distance of
// a binary32 rounding boundary.  Every operation is a binary32 add with an
// explicit rounding intrinsic, so nothing is contracted into an FMA.

struct DW {
  float hi, lo;
};

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bv = __fsub_rn(s, a);
  float av = __fsub_rn(s, bv);
  e = __fadd_rn(__fsub_rn(a, av), __fsub_rn(b, bv));
}

// acc += p for a non-negative binary32 p
__device__ __forceinline__ void dw_add(DW& acc, float p) {
  float s, e;
  two_sum(acc.hi, p, s, e);
  acc.hi = s;
  acc.lo = __fadd_rn(acc.lo, e);
}

// a + b, renormalised; commutative bit for bit, so butterfly partners agree.
// An infinite or NaN sum stands as it is (its error terms are NaN and must not
// leak into it: a row with an infinite square has S = inf, not NaN).
__device__ __forceinline__ DW dw_combine(DW a, DW b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  if (!isfinite(s)) return DW{s, 0.f};
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  float hi = __fadd_rn(s, e);
  float lo = __fsub_rn(e, __fsub_rn(hi, s));
  return DW{hi, lo};
}

// the binary32 sum: hi + lo rounded once; an infinite or NaN hi stands
__device__ __forceinline__ float dw_value(DW a) {
  return isfinite(a.hi) ? __fadd_rn(a.hi, a.lo) : a.hi;
}

__device__ __forceinline__ DW dw_warp_allreduce(DW a) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    DW o{__shfl_xor_sync(0xffffffffu, a.hi, off), __shfl_xor_sync(0xffffffffu, a.lo, off)};
    a = dw_combine(a, o);
  }
  return a;
}

// rstd from the row's sum of squares, IEEE-rounded at every step:
// var = S / hidden, rstd = 1 / sqrt(var + eps)
__device__ __forceinline__ float row_rstd(float S, float hidden_f, float eps) {
  float var = __fdiv_rn(S, hidden_f);
  float tv = __fadd_rn(var, eps);
  float root = __fsqrt_rn(tv);
  return __fdiv_rn(1.0f, root);
}

// ---------------------------------------------------------------------------
// mbarrier, bulk copy, timer (inline PTX)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `bar` with the given parity to complete, for at most
// timeout_ns.  On time-out, record FAR_ERR_TIMEOUT in the device error word and
// return false: the caller then stops (after draining its own copies, if any).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                          unsigned int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > timeout_ns) {
      atomicOr(status, 1u << FAR_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// global -> this CTA's shared memory, completion counted in bytes on `bar`
// (plain copy into the CTA's own shared memory: no multicast)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

}  // namespace far
