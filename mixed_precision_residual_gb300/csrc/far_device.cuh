// Device helpers for the fused residual-add + RMSNorm kernels (sm_103a).
//
// - dtype traits and exact widening / round-to-nearest-even narrowing,
// - the binary32 double-word accumulator for the row's sum of squares,
// - mbarrier and bulk-copy (cp.async.bulk) wrappers in inline PTX,
// - the bounded wait every kernel uses on every barrier.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
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

// two packed 16-bit products, each rounded once to nearest even (IEEE binary16 /
// bfloat16 multiply, subnormals kept).  For 16-bit n and w the binary32 product
// n * w is exact, so this equals RNE_DT(fl32(n * w)) with one instruction per pair.
template <int DT> __device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b);
template <> __device__ __forceinline__ uint32_t mul2<FAR_F16>(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <> __device__ __forceinline__ uint32_t mul2<FAR_BF16>(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// fl32(x + r) for the two 16-bit x values packed in xw and binary32 r0, r1:
// the mixed-precision add widens x exactly and rounds the sum once.
template <int DT> __device__ __forceinline__ float2 add2_mixed(uint32_t xw, float r0, float r1);
template <> __device__ __forceinline__ float2 add2_mixed<FAR_F16>(uint32_t xw, float r0, float r1) {
  float s0, s1;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.f16 %0, lo, %3;\n\tadd.rn.f32.f16 %1, hi, %4;\n\t}"
      : "=f"(s0), "=f"(s1) : "r"(xw), "f"(r0), "f"(r1));
  return make_float2(s0, s1);
}
template <> __device__ __forceinline__ float2 add2_mixed<FAR_BF16>(uint32_t xw, float r0, float r1) {
  float s0, s1;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.bf16 %0, lo, %3;\n\tadd.rn.f32.bf16 %1, hi, %4;\n\t}"
      : "=f"(s0), "=f"(s1) : "r"(xw), "f"(r0), "f"(r1));
  return make_float2(s0, s1);
}

// fl32(x * x) for the two 16-bit x values packed in xw: the mixed-precision fma
// widens both factors exactly and rounds once; x * x of a 16-bit x is exact in
// binary32, so this is the binary32 square of s = x.  (Adding -0 keeps +0 for x = 0.)
template <int DT> __device__ __forceinline__ float2 square2_mixed(uint32_t xw);
template <> __device__ __forceinline__ float2 square2_mixed<FAR_F16>(uint32_t xw) {
  float q0, q1;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "fma.rn.f32.f16 %0, lo, lo, 0f80000000;\n\tfma.rn.f32.f16 %1, hi, hi, 0f80000000;\n\t}"
      : "=f"(q0), "=f"(q1) : "r"(xw));
  return make_float2(q0, q1);
}
template <> __device__ __forceinline__ float2 square2_mixed<FAR_BF16>(uint32_t xw) {
  float q0, q1;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "fma.rn.f32.bf16 %0, lo, lo, 0f80000000;\n\tfma.rn.f32.bf16 %1, hi, hi, 0f80000000;\n\t}"
      : "=f"(q0), "=f"(q1) : "r"(xw));
  return make_float2(q0, q1);
}

// LayerNorm's affine step on two lanes, fl32(fl32(n * g) + b), for n, g and b of one
// 16-bit dtype packed in pairs: the mixed fma with a -0 addend rounds the exact product
// once (so it is fl32(n * g), underflow and overflow included), and the mixed add widens
// b exactly and rounds the sum once.
template <int DT> __device__ __forceinline__ float2 affine2_mixed(uint32_t n2, uint32_t g2, uint32_t b2);
template <> __device__ __forceinline__ float2 affine2_mixed<FAR_F16>(uint32_t n2, uint32_t g2, uint32_t b2) {
  float o0, o1;
  asm("{\n\t.reg .b16 n0, n1, g0, g1, b0, b1;\n\t.reg .f32 t0, t1;\n\t"
      "mov.b32 {n0, n1}, %2;\n\tmov.b32 {g0, g1}, %3;\n\tmov.b32 {b0, b1}, %4;\n\t"
      "fma.rn.f32.f16 t0, n0, g0, 0f80000000;\n\tfma.rn.f32.f16 t1, n1, g1, 0f80000000;\n\t"
      "add.rn.f32.f16 %0, b0, t0;\n\tadd.rn.f32.f16 %1, b1, t1;\n\t}"
      : "=f"(o0), "=f"(o1) : "r"(n2), "r"(g2), "r"(b2));
  return make_float2(o0, o1);
}
template <> __device__ __forceinline__ float2 affine2_mixed<FAR_BF16>(uint32_t n2, uint32_t g2, uint32_t b2) {
  float o0, o1;
  asm("{\n\t.reg .b16 n0, n1, g0, g1, b0, b1;\n\t.reg .f32 t0, t1;\n\t"
      "mov.b32 {n0, n1}, %2;\n\tmov.b32 {g0, g1}, %3;\n\tmov.b32 {b0, b1}, %4;\n\t"
      "fma.rn.f32.bf16 t0, n0, g0, 0f80000000;\n\tfma.rn.f32.bf16 t1, n1, g1, 0f80000000;\n\t"
      "add.rn.f32.bf16 %0, b0, t0;\n\tadd.rn.f32.bf16 %1, b1, t1;\n\t}"
      : "=f"(o0), "=f"(o1) : "r"(n2), "r"(g2), "r"(b2));
  return make_float2(o0, o1);
}

// ---------------------------------------------------------------------------
// packed binary32 pairs (add / sub / mul .f32x2): each half rounds exactly as the
// scalar instruction does (to nearest even, subnormals kept), two lanes an issue.
// Unlike the scalar forms with an explicit rounding mode, a packed multiply (or a
// packed fma with a -0 addend) whose result feeds a packed add is fused into one
// multiply-add by the compiler, --fmad=false notwithstanding (measured: the outputs
// then equal the single-rounding result).  So a product that a packed add consumes
// is always formed by the scalar mul.rn, which is never fused.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pk(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 unpk(uint64_t v) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return make_float2(a, b);
}
__device__ __forceinline__ uint64_t add_x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub_x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
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

// vector store of N bytes (N = 8, 16 or 32), N-aligned; default L2 policy, so a
// following kernel can still find the tail of the output in L2
template <int N> __device__ __forceinline__ void store_bytes(void* p, const uint32_t* w) {
  if constexpr (N == 8) {
    asm volatile("st.global.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(w[0]), "r"(w[1]) : "memory");
  } else {
#pragma unroll
    for (int k = 0; k < N / 16; ++k)
      asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(reinterpret_cast<char*>(p) + 16 * k),
                   "r"(w[4 * k]), "r"(w[4 * k + 1]), "r"(w[4 * k + 2]), "r"(w[4 * k + 3])
                   : "memory");
  }
}

// ---------------------------------------------------------------------------
// the row's sum of squares: a binary32 double-word (hi + lo) accumulator
// ---------------------------------------------------------------------------
//
// The contract fixes binary32 accumulation but not the order.  Each square is
// added with an error-free transformation and the exact rounding errors are
// carried in `lo`; hi + lo then stays within about 2^-44 (relative) of the
// exact sum, so hi + lo rounded once to binary32 is the correctly rounded sum
// -- the one order-free binary32 value -- except in astronomically rare rows
// whose exact sum lies within that distance of a binary32 rounding boundary.
// All terms are non-negative, so ordering the pair with max/min makes Dekker's
// Fast2Sum exact (|a| >= |b|); the NaN-propagating max/min keep a NaN square
// from being dropped.  Every add carries an explicit rounding intrinsic, so
// nothing is contracted into an FMA.  (The generic kernel adds its squares this
// way, one at a time; the staged kernel, which holds a thread's values in
// registers, uses the packed chains offset by the largest square further below,
// which need no ordering.)

struct DW {
  float hi, lo;
};

__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

__device__ __forceinline__ float min_nan(float a, float b) {
  float d;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// s + e == a + b exactly, for non-negative a, b (or inf / NaN, which stand in s)
__device__ __forceinline__ void fast_two_sum_ordered(float a, float b, float& s, float& e) {
  const float big = max_nan(a, b), small = min_nan(a, b);
  s = __fadd_rn(big, small);
  e = __fsub_rn(small, __fsub_rn(s, big));
}

// acc += p for a non-negative binary32 p
__device__ __forceinline__ void dw_add(DW& acc, float p) {
  float s, e;
  fast_two_sum_ordered(acc.hi, p, s, e);
  acc.hi = s;
  acc.lo = __fadd_rn(acc.lo, e);
}

// a + b; commutative bit for bit, so butterfly partners agree.  hi carries the
// rounded sum of the his, lo every exact error so far (an infinite or NaN hi
// makes lo NaN, and dw_value then lets hi stand).
__device__ __forceinline__ DW dw_combine(DW a, DW b) {
  float s, e;
  fast_two_sum_ordered(a.hi, b.hi, s, e);
  return DW{s, __fadd_rn(__fadd_rn(a.lo, b.lo), e)};
}

// the binary32 sum: hi + lo rounded once; an infinite or NaN hi stands
__device__ __forceinline__ float dw_value(DW a) {
  return isfinite(a.hi) ? __fadd_rn(a.hi, a.lo) : a.hi;
}

// TwoSum (Knuth): s + e == a + b exactly, for any signs and any order of a and b
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bv = __fsub_rn(s, a);
  const float av = __fsub_rn(s, bv);
  e = __fadd_rn(__fsub_rn(a, av), __fsub_rn(b, bv));
}

// acc += v for a binary32 v of any sign (the LayerNorm mean's sum)
__device__ __forceinline__ void dw_add_signed(DW& acc, float v) {
  float s, e;
  two_sum(acc.hi, v, s, e);
  acc.hi = s;
  acc.lo = __fadd_rn(acc.lo, e);
}

// a + b for signed double words; commutative bit for bit (the TwoSum error is exact)
__device__ __forceinline__ DW dw_combine_signed(DW a, DW b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  return DW{s, __fadd_rn(__fadd_rn(a.lo, b.lo), e)};
}

__device__ __forceinline__ DW dw_shfl_xor(DW a, int off) {
  return DW{__shfl_xor_sync(0xffffffffu, a.hi, off), __shfl_xor_sync(0xffffffffu, a.lo, off)};
}

__device__ __forceinline__ DW dw_warp_allreduce(DW a) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) a = dw_combine(a, dw_shfl_xor(a, off));
  return a;
}

// Two independent double-word chains in the two halves of packed pairs: TwoSum in each
// half (any signs, any order), so a pair of values costs seven packed instructions.
struct DW2 {
  uint64_t hi, lo;
};
__device__ __forceinline__ void dw2_add(DW2& acc, uint64_t v) {
  const uint64_t s = add_x2(acc.hi, v);
  const uint64_t bv = sub_x2(s, acc.hi);
  const uint64_t av = sub_x2(s, bv);
  const uint64_t e = add_x2(sub_x2(acc.hi, av), sub_x2(v, bv));
  acc.hi = s;
  acc.lo = add_x2(acc.lo, e);
}
// The same two chains by the ordered Fast2Sum: the operand of larger magnitude first
// (a compare and two selects, on the integer pipe), then three packed operations; exact
// for any signs.  Half the floating-point work of TwoSum.
__device__ __forceinline__ void dw2_add_ordered(DW2& acc, float v0, float v1) {
  const float2 h = unpk(acc.hi);
  const bool p0 = fabsf(h.x) >= fabsf(v0), p1 = fabsf(h.y) >= fabsf(v1);
  const uint64_t big = pk(p0 ? h.x : v0, p1 ? h.y : v1);
  const uint64_t small = pk(p0 ? v0 : h.x, p1 ? v1 : h.y);
  const uint64_t s = add_x2(big, small);
  acc.hi = s;
  acc.lo = add_x2(acc.lo, sub_x2(small, sub_x2(s, big)));
}

// Sums of non-negative terms whose largest term is known before the first addition: each
// chain starts at B, the largest power of two not above that term (its exponent, the
// mantissa cleared; 0 for a subnormal term), and only grows.  So a chain's exponent is
// never below a term's, and Dekker's Fast2Sum -- s = a + b, t = b - (s - a) -- is exact
// without ordering the operands (its condition is e_a >= e_b): three packed operations and
// the low-part add a pair, nothing on the integer pipe.  At the end hi - B is exact (hi and
// B are multiples of ulp(hi) while hi < 2^24 B, i.e. fewer than 2^22 terms a chain), and
// (hi - B) + lo is the chain's sum as a double word.  Each rounding error carried in lo is
// relative to B + the chain's sum, where B is at most the largest term of the whole sum:
// the row's double word stays within a few units of 2^-44 (relative) of the exact sum.
__device__ __forceinline__ float pow2_floor(float q) {
  return __uint_as_float(__float_as_uint(q) & 0x7f800000u);  // NaN -> +inf, inf stays
}
__device__ __forceinline__ void dwb_add(DW2& acc, uint64_t v) {
  const uint64_t s = add_x2(acc.hi, v);
  acc.lo = add_x2(acc.lo, sub_x2(v, sub_x2(s, acc.hi)));
  acc.hi = s;
}
// the two chains of an offset DW2 as double words, B taken off: exact.  B infinite (an
// infinite or NaN term, so the chains are infinite or NaN): hi stands
__device__ __forceinline__ void dwb_split(DW2 a, float B, DW& c0, DW& c1) {
  const float2 h = unpk(isfinite(B) ? sub_x2(a.hi, pk(B, B)) : a.hi), l = unpk(a.lo);
  c0 = DW{h.x, l.x};
  c1 = DW{h.y, l.y};
}

// the two chains of a DW2 folded into one double word
__device__ __forceinline__ DW dw2_fold(DW2 a) {
  const float2 h = unpk(a.hi), l = unpk(a.lo);
  return dw_combine_signed(DW{h.x, l.x}, DW{h.y, l.y});
}

// the same butterfly for sums of either sign (TwoSum in place of the ordered Fast2Sum)
__device__ __forceinline__ DW dw_warp_allreduce_signed(DW a) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) a = dw_combine_signed(a, dw_shfl_xor(a, off));
  return a;
}

// ---------------------------------------------------------------------------
// quantised output: per-row maximum, scale, and the two byte formats
// ---------------------------------------------------------------------------

__device__ __forceinline__ float warp_max_allreduce(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// running max of |v| over packed 16-bit pairs, NaN-propagating
template <int DT> __device__ __forceinline__ uint32_t habs_max2(uint32_t m, uint32_t v);
template <> __device__ __forceinline__ uint32_t habs_max2<FAR_F16>(uint32_t m, uint32_t v) {
  __half2 r = __hmax2_nan(*reinterpret_cast<__half2*>(&m), __habs2(*reinterpret_cast<__half2*>(&v)));
  return *reinterpret_cast<uint32_t*>(&r);
}
template <> __device__ __forceinline__ uint32_t habs_max2<FAR_BF16>(uint32_t m, uint32_t v) {
  __nv_bfloat162 r =
      __hmax2_nan(*reinterpret_cast<__nv_bfloat162*>(&m), __habs2(*reinterpret_cast<__nv_bfloat162*>(&v)));
  return *reinterpret_cast<uint32_t*>(&r);
}

// four values scaled into quantised bytes, packed little-endian into one word
//   Q = 1: int8, nearest integer with ties to even, saturated (the scaled values never
//          pass +-127.5, so the saturation bound of -128 is never reached); NaN -> 0
//   Q = 2: FP8 E4M3, nearest with ties to even, finite values saturated to +-448
template <int Q> __device__ __forceinline__ uint32_t quantise4(float a, float b, float c, float d);
template <> __device__ __forceinline__ uint32_t quantise4<1>(float a, float b, float c, float d) {
  uint32_t qa, qb, qc, qd;
  asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(qa) : "f"(a));
  asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(qb) : "f"(b));
  asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(qc) : "f"(c));
  asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(qd) : "f"(d));
  return __byte_perm(__byte_perm(qa, qb, 0x0040), __byte_perm(qc, qd, 0x0040), 0x5410);
}
template <> __device__ __forceinline__ uint32_t quantise4<2>(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return __byte_perm(lo, hi, 0x5410);
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
// programmatic dependent launch (inline PTX; both are no-ops in a kernel launched without
// the programmatic-stream-serialization attribute)
// ---------------------------------------------------------------------------

// Let the next kernel on the stream, if it was launched with the attribute, be dispatched
// now: its CTAs take SMs as this grid's CTAs leave them.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until every kernel before this one on the stream has completed and its memory
// operations are visible.  Every kernel here calls it before its first access to global
// memory, so stream order holds whatever the launch attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// One bounded attempt: the thread may be suspended until the phase completes or
// kSuspendHintNs passes, so a waiting warp sleeps instead of spinning on issue slots.
constexpr uint32_t kSuspendHintNs = 20000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
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
    for (int i = 0; i < 8; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > timeout_ns) {
      atomicOr(status, 1u << FAR_ERR_TIMEOUT);
      return false;
    }
  }
}

// global -> this CTA's shared memory, completion counted in bytes on `bar`
// (plain copy into the CTA's own shared memory: no multicast)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

}  // namespace far
