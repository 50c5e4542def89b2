// Kernels for fused residual-add + RMSNorm and its no-residual variant (and, under
// the same rounding contract, fused residual-add + LayerNorm and its variant).
//
// staged_kernel -- the hot path.  Persistent (one CTA per SM), warp-specialised:
//   warp 0, lane 0 (producer) bulk-copies each row of x and of the residual into
//   a ring of shared-memory slots (cp.async.bulk, mbarrier completion, plain
//   copies into the CTA's own shared memory), at a fixed stride over the rows
//   for the first ring-full and then, given a row counter, in runs claimed from
//   it, so that CTAs served faster take more rows;
//   `groups` groups of G consumer warps each take a row from the ring: every
//   thread widens its 16-byte chunks, forms s = fl32(x + r) and keeps s in
//   registers, accumulates the squares, releases the slot, reduces across the
//   warp (shuffles) and the group (shared memory + mbarrier), then normalises
//   from the registers and streams residual_out and out to HBM.
//   So every input byte is read from HBM once and the binary32 sum is never
//   re-read; every output byte is written once.
//
// generic_kernel -- any alignment and any hidden size: one CTA per row
//   (grid-stride), scalar accesses, the row re-read in the second pass (from
//   L1/L2).  Same arithmetic, same results.
//
// The rounding steps are the ones the case study "Aligning fused RMSNorm
// rounding across vLLM backends" fixes (stage table of "Finding the rounding
// boundary"): s kept in binary32, residual rounded only on store, variance and
// normalisation from s, the normalised value cast to the weight dtype before
// the weight multiply.
#pragma once

#include <type_traits>

#include "far_device.cuh"

namespace far {

// Reduce a double word across the G warps of a group: every warp publishes its
// value in buffer `buf`, then all combine the G values with the same butterfly over
// lanes 0..G8-1, so every lane of every warp ends with the same bits.  False when
// the bounded wait ran out (the caller then stops).
template <typename Combine>
__device__ __forceinline__ bool group_reduce(DW& v, float2* partials, uint64_t* bars, int red_base, int g,
                                             int nred, int buf, int G, int G8, int wg, int lane, uint32_t use,
                                             const Params& p, Combine combine) {
  float2* part = partials + (size_t)(g * nred + buf) * G;
  const uint32_t rbar = smem_addr(&bars[red_base + g * nred + buf]);
  if (lane == 0) {
    part[wg] = make_float2(v.hi, v.lo);
    mbar_arrive(rbar);
  }
  if (!mbar_wait(rbar, (use >> 1) & 1u, p.timeout_ns, p.status)) return false;
  const int src = lane & (G8 - 1);
  const float2 mine = src < G ? part[src] : make_float2(0.f, 0.f);
  DW t{mine.x, mine.y};
  for (int off = G8 >> 1; off > 0; off >>= 1) t = combine(t, dw_shfl_xor(t, off));
  v = t;
  return true;
}

template <int ACT, int WD, bool RES, int NCH, bool EXACT, int Q = kQuantNone, bool LN = false>
__global__ void __launch_bounds__(max_threads(NCH, packed_rows(RES, ACT) && !LN), 1)
    staged_kernel(const Params p) {
  constexpr int SA = dtype_size<ACT>::value;
  constexpr int SW = dtype_size<WD>::value;
  constexpr int OD = promote(ACT, WD);
  constexpr int SO = dtype_size<OD>::value;
  constexpr int V = 16 / SA;   // elements per 16-byte activation chunk
  constexpr int WB = V * SW;   // weight bytes per chunk: 8, 16 or 32
  constexpr int OB = V * SO;   // output bytes per chunk: 16 or 32
  // no residual and 16-bit x: s = x exactly, so x stays packed between the passes
  // (LayerNorm needs the binary32 deviations s - mean instead)
  constexpr bool PACKED = packed_rows(RES, ACT) && !LN;
  // 16-bit activations with a binary32 out: a thread's chunk j is two 8-byte pieces of the
  // row, 32 lanes apart (pieces 2b + lane and 2b + 32 + lane of the warp's window of 32
  // chunks starting at chunk b), so that every warp-wide access is contiguous: out in
  // 512-byte runs (one 16-byte store of 4 binary32 values a lane), residual_out in 256-byte
  // runs.  Lanes of a 16-byte chunk instead would leave each out store covering every
  // other 16 bytes of 1 KB (32 half-written sectors a request instead of 16).  (A
  // quantised output stores no binary32 values: its stores are contiguous already.)
  constexpr bool PIECE = (SA == 2 && SO == 4 && Q == kQuantNone);

  constexpr int NRED = reduce_buffers(Q, LN);  // cross-warp reduction buffers per group

  extern __shared__ __align__(128) unsigned char smem[];
  // the next kernel on the stream may be dispatched now; nothing of global memory is touched
  // before the kernels ahead of this one have completed
  pdl_launch_dependents();
  pdl_wait();
  const int stages = p.stages, groups = p.groups, G = p.warps_per_row;
  // layout: full[stages] | empty[stages] | reduce[groups][NRED] | partials[groups][NRED][G] |
  //         slot_row[stages] | w | ring
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  float2* partials = reinterpret_cast<float2*>(smem + (size_t)(2 * stages + NRED * groups) * 8);
  int64_t* slot_row = reinterpret_cast<int64_t*>(partials + (size_t)groups * NRED * G);  // -1: no more rows
  const size_t head =
      ((size_t)(2 * stages + NRED * groups) * 8 + (size_t)groups * NRED * G * 8 + (size_t)stages * 8 + 127) /
      128 * 128;
  unsigned char* wsm = smem + head;
  unsigned char* ring = wsm + (p.w_smem_bytes + 127) / 128 * 128;
  const uint32_t r_off = (p.row_bytes + 127u) & ~127u;  // residual row inside a slot

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The ring's phase bookkeeping needs every slot owned by one group (stages a
  // multiple of groups) and a warp count that matches the plan; refuse anything
  // else before any barrier or copy exists (the host never launches it).
  if (stages < 2 || groups < 1 || stages % groups != 0 || (int)blockDim.x != (1 + groups * G) * 32) {
    if (threadIdx.x == 0) atomicOr(p.status, 1u << FAR_ERR_SHAPE);
    return;
  }
  // Rows enter the ring in this order: first the CTA's fixed-stride rows b + k * nb (all of
  // them; or, with a row counter, only those with k < S, S = sched_static), then runs of n
  // rows R0 + c .. R0 + c + n - 1, R0 = nb * S, n = sched_run, each claimed by one atomic add
  // of n to the launch's counter (which returns c), until the claims pass the last row. The
  // CTAs that are served faster take more rows, all finish within a run of each other, and
  // while they claim they all work in one window of neighbouring rows.
  const int64_t b = blockIdx.x, nb = gridDim.x;
  int64_t n_static = (p.tokens > b) ? (p.tokens - b + nb - 1) / nb : 0;
  if (p.sched != nullptr && n_static > p.sched_static) n_static = p.sched_static;
  const uint32_t tx = RES ? 2u * p.row_bytes : p.row_bytes;
  const int64_t first = n_static < stages ? n_static : stages;  // rows issued before the consumers start

  // producer: the row number into slot_row[slot] (read by the slot's consumers after the
  // full barrier), then one bulk copy of the row's x (and residual) into the slot
  auto issue = [&](int64_t row, int slot) {
    slot_row[slot] = row;
    const uint32_t full = smem_addr(&bars[slot]);
    const uint32_t dst = smem_addr(ring + (size_t)slot * p.stage_bytes);
    mbar_arrive_expect_tx(full, tx);
    bulk_load(dst, static_cast<const char*>(p.x) + row * p.x_stride, p.row_bytes, full);
    if constexpr (RES) bulk_load(dst + r_off, static_cast<const char*>(p.r) + row * p.r_stride, p.row_bytes, full);
  };

  // LayerNorm's shift row sits right after the scale row in shared memory
  unsigned char* bsm = wsm + (size_t)((p.hidden * SW + 15) / 16 * 16);
  // The weight row (and LayerNorm's shift row), once per CTA (16-byte aligned; hidden * SW is
  // even), read before the first ring-full of rows is requested: issued after it, these
  // loads queue behind every CTA's first rows (measured: bf16 / fp32-weight 4096 x 4096
  // variant 17.3 us against 18.4 in a stream, fp16 512 x 8192 fused 7.8 against 8.2).
  {
    const int nbytes = p.hidden * SW;
    const int n16 = nbytes >> 4;
    for (int k = 0; k < (LN ? 2 : 1); ++k) {
      const void* srcp = k == 0 ? p.w : p.beta;
      unsigned char* dstp = k == 0 ? wsm : bsm;
      const uint4* src = reinterpret_cast<const uint4*>(srcp);
      for (int i = threadIdx.x; i < n16; i += blockDim.x) reinterpret_cast<uint4*>(dstp)[i] = src[i];
      const uint16_t* src2 = reinterpret_cast<const uint16_t*>(srcp);
      for (int i = (n16 << 3) + threadIdx.x; i < (nbytes >> 1); i += blockDim.x)
        reinterpret_cast<uint16_t*>(dstp)[i] = src2[i];
    }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(smem_addr(&bars[i]), 1);           // full: the producer's arrive + bytes
      mbar_init(smem_addr(&bars[stages + i]), G);  // empty: one arrive per consumer warp
    }
    for (int i = 0; i < NRED * groups; ++i) mbar_init(smem_addr(&bars[2 * stages + i]), G);
    fence_barrier_init();
    // the first `stages` rows need no free slot: start them now
    for (int64_t k = 0; k < first; ++k) issue(b + k * nb, (int)k);
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int64_t k = first;  // ring positions filled: position k goes to slot k % stages
      int slot = (int)(first % stages);
      uint32_t phase = (uint32_t)(first / stages) & 1u;  // (k / stages) & 1
      // fill position k with `row` (-1: the end marker of the group that owns position k)
      auto put = [&](int64_t row) -> bool {
        // slot k % stages last held position k - stages: wait until its consumers released it
        if (k >= stages && !mbar_wait(smem_addr(&bars[stages + slot]), phase ^ 1u, p.timeout_ns, p.status))
          return false;
        if (row >= 0) {
          issue(row, slot);
        } else {
          slot_row[slot] = -1;
          mbar_arrive(smem_addr(&bars[slot]));  // completes the phase: no bytes to wait for
        }
        ++k;
        if (++slot == stages) {
          slot = 0;
          phase ^= 1u;
        }
        return true;
      };
      bool ok = true;
      for (int64_t i = first; ok && i < n_static; ++i) ok = put(b + i * nb);
      if (p.sched != nullptr) {
        const int64_t R0 = nb * (int64_t)p.sched_static;
        const unsigned long long n = p.sched_run > 1 ? (unsigned long long)p.sched_run : 1ull;
        // the next run is claimed while this one is issued (its atomic's latency hidden); a
        // thread's adds to one address are ordered, so every run after a spent one is spent
        unsigned long long c0 = atomicAdd(p.sched, n), c1 = atomicAdd(p.sched, n);
        while (ok && R0 + (int64_t)c0 < p.tokens) {
          int64_t end = R0 + (int64_t)(c0 + n);
          if (end > p.tokens) end = p.tokens;
          for (int64_t row = R0 + (int64_t)c0; ok && row < end; ++row) ok = put(row);
          c0 = c1;
          if (R0 + (int64_t)c0 >= p.tokens) break;
          c1 = atomicAdd(p.sched, n);
        }
        // this CTA claims no more: count it done; the last one leaves the pair zero for the
        // next launch that is given it (every claim of this launch precedes the reset)
        __threadfence();
        if (atomicAdd(p.sched + 1, 1ull) == (unsigned long long)nb - 1) {
          atomicExch(p.sched, 0ull);
          atomicExch(p.sched + 1, 0ull);
        }
      }
      // an end marker at each group's next position (positions k .. k + groups - 1 belong
      // to distinct groups: stages is a multiple of groups)
      for (int i = 0; ok && i < groups; ++i) ok = put(-1);
      // the copies of the last (at most `stages`) positions must have landed before the CTA
      // may exit
      for (int64_t j = (k > stages ? k - stages : 0); j < k; ++j)
        mbar_wait(smem_addr(&bars[j % stages]), (uint32_t)(j / stages) & 1u, p.timeout_ns, p.status);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int cw = warp - 1;
  const int g = cw / G, wg = cw - g * G;
  const int C = p.chunks;
  int G8 = 1;  // G rounded up to a power of two (<= 16): the lanes of the cross-warp butterfly
  while (G8 < G) G8 <<= 1;
  int slot = g;          // k % stages for this group's positions k = g, g + groups, ...
  uint32_t phase = 0;    // (k / stages) & 1
  uint32_t it = 0;       // this group's row count, for the reduction buffers
  // This thread's chunk j: its pieces (in PB-byte units of the activation row: one piece, the
  // chunk itself, unless PIECE) and whether each lies inside the row.  Elements 0 .. V/2 - 1
  // of the chunk come from piece pa, V/2 .. V - 1 from piece pb (the same piece unless PIECE).
  struct Where {
    int pa, pb;
    bool va, vb;
  };
  auto where = [&](int j) {
    const int c = (j * G + wg) * 32 + lane;
    Where w;
    if constexpr (PIECE) {
      w.pa = 2 * c - lane;  // piece 2b + lane of the window of chunks b = c - lane ..
      w.pb = w.pa + 32;
      w.va = EXACT || w.pa < 2 * C;
      w.vb = EXACT || w.pb < 2 * C;
    } else {
      w.pa = w.pb = c;
      w.va = w.vb = EXACT || c < C;
    }
    return w;
  };
  // the chunk's 16 activation bytes from a shared-memory row (zeros for a piece past the row)
  auto load_act = [&](const unsigned char* base, const Where& w, uint32_t* v) {
    if constexpr (PIECE) {
      uint32_t a[2] = {0u, 0u}, b2[2] = {0u, 0u};
      if (w.va) load_bytes<8>(base + (size_t)w.pa * 8, a);
      if (w.vb) load_bytes<8>(base + (size_t)w.pb * 8, b2);
      v[0] = a[0];
      v[1] = a[1];
      v[2] = b2[0];
      v[3] = b2[1];
    } else {
      load_bytes<16>(base + (size_t)w.pa * 16, v);
    }
  };
  // the chunk's NB bytes of a per-element vector held in shared memory (the weight, beta):
  // NB / 2 bytes a piece; zeros for a piece past the row
  auto load_vec = [&](const unsigned char* base, const Where& w, uint32_t* v, auto nb) {
    constexpr int NB = decltype(nb)::value;
    if constexpr (PIECE) {
#pragma unroll
      for (int i = 0; i < NB / 4; ++i) v[i] = 0u;
      if (w.va) load_bytes<NB / 2>(base + (size_t)w.pa * (NB / 2), v);
      if (w.vb) load_bytes<NB / 2>(base + (size_t)w.pb * (NB / 2), v + NB / 8);
    } else {
      load_bytes<NB>(base + (size_t)w.pa * NB, v);
    }
  };
  // the chunk's NB bytes of an output row (NB / 2 a piece; pieces past the row not written)
  auto store_row = [&](char* rowp, const Where& w, const uint32_t* v, auto nb) {
    constexpr int NB = decltype(nb)::value;
    if constexpr (PIECE) {
      if (w.va) store_bytes<NB / 2>(rowp + (size_t)w.pa * (NB / 2), v);
      if (w.vb) store_bytes<NB / 2>(rowp + (size_t)w.pb * (NB / 2), v + NB / 8);
    } else {
      store_bytes<NB>(rowp + (size_t)w.pa * NB, v);
    }
  };
  for (;; ++it) {
    if (!mbar_wait(smem_addr(&bars[slot]), phase, p.timeout_ns, p.status)) return;
    const int64_t row = slot_row[slot];  // read before the slot is released
    if (row < 0) return;                 // the group's end marker
    const unsigned char* xs = ring + (size_t)slot * p.stage_bytes;

    // pass 1 (from shared memory): s = fl32(x + r) into registers, squares into the accumulator
    float s[PACKED ? 1 : NCH][PACKED ? 1 : V];
    uint32_t xk[PACKED ? NCH : 1][PACKED ? V / 2 : 1];  // the packed x of the no-residual variant
    DW acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};  // four independent chains
    DW2 accp[2] = {{0ull, 0ull}, {0ull, 0ull}};  // LayerNorm: four chains in packed pairs
    if constexpr (PACKED) {
      // s = x exactly, kept packed.  The first sweep brings the thread's chunks into
      // registers with their largest magnitude M; the second sums the squares in chains
      // that start at the largest square's power of two (Fast2Sum exact without ordering)
      uint32_t m2 = 0u;  // packed running max of |x|
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const Where w = where(j);
        if (w.va) {
          load_act(xs, w, xk[j]);
#pragma unroll
          for (int e = 0; e < V / 2; ++e) m2 = habs_max2<ACT>(m2, xk[j][e]);
        }
      }
      const float2 mq = square2_mixed<ACT>(m2);  // fl32(M * M), the largest square
      const float B = pow2_floor(max_nan(mq.x, mq.y));
      DW2 sq[2] = {{pk(B, B), 0ull}, {pk(B, B), 0ull}};
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        if (where(j).va) {
#pragma unroll
          for (int e = 0; e < V / 2; ++e) {
            const float2 q = square2_mixed<ACT>(xk[j][e]);
            dwb_add(sq[e & 1], pk(q.x, q.y));
          }
        }
      }
      dwb_split(sq[0], B, acc[0], acc[1]);
      dwb_split(sq[1], B, acc[2], acc[3]);
    } else {
      float smax = 0.f;  // RMSNorm: the largest |s| of the thread's chunks (NaN-propagating)
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const Where w = where(j);
        if (w.va) {
          uint32_t xw[4];
          load_act(xs, w, xw);
          if constexpr (RES) {
            uint32_t rv[4];
            load_act(xs + r_off, w, rv);
            float rf[V];
            widen<ACT, V>(rv, rf);
            if constexpr (ACT == FAR_F32) {
#pragma unroll
              for (int e = 0; e < V; ++e) s[j][e] = __fadd_rn(__uint_as_float(xw[e]), rf[e]);
            } else {
#pragma unroll
              for (int e = 0; e < V / 2; ++e) {
                const float2 t = add2_mixed<ACT>(xw[e], rf[2 * e], rf[2 * e + 1]);
                s[j][2 * e] = t.x;
                s[j][2 * e + 1] = t.y;
              }
            }
          } else {
            widen<ACT, V>(xw, s[j]);
          }
          if constexpr (LN) {
#pragma unroll
            for (int e = 0; e < V / 2; ++e) {
              // for the mean, exact for any signs: one packed chain by the ordered Fast2Sum
              // (a compare and two selects on the integer pipe), the other by TwoSum (on the
              // FMA pipe), which keeps both pipes busy (LayerNorm variant bf16 16384 x 5120:
              // 84.0 against 85.5 us with every pair ordered)
              if (e & 1) dw2_add(accp[1], pk(s[j][2 * e], s[j][2 * e + 1]));
              else dw2_add_ordered(accp[0], s[j][2 * e], s[j][2 * e + 1]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < V; ++e) smax = max_nan(smax, fabsf(s[j][e]));
          }
        } else {
#pragma unroll
          for (int e = 0; e < V; ++e) s[j][e] = 0.f;
        }
      }
      if constexpr (!LN) {
        // the squares fl32(s * s) (scalar mul.rn: never fused into the adds) in chains that
        // start at the largest square's power of two, as in the packed variant
        const float B = pow2_floor(__fmul_rn(smax, smax));
        DW2 sq[2] = {{pk(B, B), 0ull}, {pk(B, B), 0ull}};
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          if (where(j).va) {
#pragma unroll
            for (int e = 0; e < V / 2; ++e)
              dwb_add(sq[e & 1], pk(__fmul_rn(s[j][2 * e], s[j][2 * e]), __fmul_rn(s[j][2 * e + 1], s[j][2 * e + 1])));
          }
        }
        dwb_split(sq[0], B, acc[0], acc[1]);
        dwb_split(sq[1], B, acc[2], acc[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&bars[stages + slot]));  // the slot may be refilled
    slot += groups;
    if (slot >= stages) {
      slot -= stages;
      phase ^= 1u;
    }

    float rstd;
    if constexpr (LN) {
      // LayerNorm: mean from the exact-per-addition signed sum (each addition is exact, but the
      // low parts are plain binary32 sums: where values of opposite sign cancel to a sum far
      // below the row's partial sums, their rounding can leave the sum some ulps from the
      // correctly rounded one; on rows without such cancellation it is that value); then d = s - mean in place,
      // residual_out stored from s on the way, and the sum of the squared deviations
      DW tot = dw_warp_allreduce_signed(dw_combine_signed(dw2_fold(accp[0]), dw2_fold(accp[1])));
      if (G > 1 && !group_reduce(tot, partials, bars, 2 * stages, g, NRED, (int)(it & 1u), G, G8, wg, lane, it, p,
                                 dw_combine_signed))
        return;
      const float mean = __fdiv_rn(dw_value(tot), p.hidden_f);
      const uint64_t mean2 = pk(mean, mean);
      char* rrow = RES ? static_cast<char*>(p.res_out) + row * p.res_stride : nullptr;
      float dmax = 0.f;  // the largest |d| of the thread's chunks (NaN-propagating)
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const Where w = where(j);
        if (w.va) {
          if constexpr (RES) {
            uint32_t rw[4];
            narrow<ACT, V>(s[j], rw);
            store_row(rrow, w, rw, std::integral_constant<int, 16>{});
          }
#pragma unroll
          for (int e = 0; e < V / 2; ++e) {
            const uint64_t dv = sub_x2(pk(s[j][2 * e], s[j][2 * e + 1]), mean2);  // d = fl32(s - mean)
            const float2 df = unpk(dv);
            s[j][2 * e] = df.x;
            s[j][2 * e + 1] = df.y;
            // (a piece past the row holds zeros, not values of s: no deviation of it is summed)
            if (!PIECE || e < V / 4 || w.vb) dmax = max_nan(dmax, max_nan(fabsf(df.x), fabsf(df.y)));
          }
        }
      }
      // the squares fl32(d * d) (scalar mul.rn: never fused into the adds) in chains offset by
      // the largest square, as RMSNorm's (fp16 65536 x 8192 variant: 415 against 426 us with
      // chains ordered by a max / min pair)
      const float Bq = pow2_floor(__fmul_rn(dmax, dmax));
      DW2 accq[2] = {{pk(Bq, Bq), 0ull}, {pk(Bq, Bq), 0ull}};
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const Where w = where(j);
        if (w.va) {
#pragma unroll
          for (int e = 0; e < V / 2; ++e)
            if (!PIECE || e < V / 4 || w.vb)
              dwb_add(accq[e & 1], pk(__fmul_rn(s[j][2 * e], s[j][2 * e]), __fmul_rn(s[j][2 * e + 1], s[j][2 * e + 1])));
        }
      }
      DW q0, q1, q2, q3;
      dwb_split(accq[0], Bq, q0, q1);
      dwb_split(accq[1], Bq, q2, q3);
      DW tot2 = dw_warp_allreduce(dw_combine(dw_combine(q0, q1), dw_combine(q2, q3)));
      if (G > 1 && !group_reduce(tot2, partials, bars, 2 * stages, g, NRED, 2 + (int)(it & 1u), G, G8, wg, lane,
                                 it, p, dw_combine))
        return;
      rstd = row_rstd(dw_value(tot2), p.hidden_f, p.eps);
    } else {
      DW tot = dw_warp_allreduce(dw_combine(dw_combine(acc[0], acc[1]), dw_combine(acc[2], acc[3])));
      if (G > 1 && !group_reduce(tot, partials, bars, 2 * stages, g, NRED, (int)(it & 1u), G, G8, wg, lane, it, p,
                                 dw_combine))
        return;
      rstd = row_rstd(dw_value(tot), p.hidden_f, p.eps);
    }

    // pass 2 (from registers): residual_out = RNE_act(s); out = RNE_od(RNE_wd(s * rstd) * w).
    // With a quantised output the out values stay in registers (packed) until the
    // row's largest |out| is known.
    char* orow = Q ? nullptr : static_cast<char*>(p.out) + row * p.out_stride;
    char* rrow = (RES && !LN) ? static_cast<char*>(p.res_out) + row * p.res_stride : nullptr;
    uint32_t okeep[Q ? NCH : 1][Q ? OB / 4 : 1];
    float amax = 0.f;
    uint32_t amax2 = 0u;  // packed running max of |out| for a 16-bit out
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const Where w = where(j);
      if (w.va) {
        float sj[V];  // s for this chunk: kept in registers, or widened from the packed x
        if constexpr (PACKED) widen<ACT, V>(xk[j], sj);
        else {
#pragma unroll
          for (int e = 0; e < V; ++e) sj[e] = s[j][e];
        }
        uint32_t ww[WB / 4];
        load_vec(wsm, w, ww, std::integral_constant<int, WB>{});
        uint32_t ow[OB / 4];
        if constexpr (LN) {
          // out = RNE_od(fl32(fl32(RNE_wd(d * rstd) * gamma) + beta)), two lanes at a time
          uint32_t bw[WB / 4];
          load_vec(bsm, w, bw, std::integral_constant<int, WB>{});
          const uint64_t rstd2 = pk(rstd, rstd);
          float o[V];
#pragma unroll
          for (int e = 0; e < V / 2; ++e) {
            const float2 a = unpk(mul_x2(pk(sj[2 * e], sj[2 * e + 1]), rstd2));
            float2 u;
            if constexpr (WD == FAR_F32) {
              // binary32 gamma and beta (the cast is the identity): scalar multiply and add
              u.x = __fadd_rn(__fmul_rn(a.x, __uint_as_float(ww[2 * e])), __uint_as_float(bw[2 * e]));
              u.y = __fadd_rn(__fmul_rn(a.y, __uint_as_float(ww[2 * e + 1])), __uint_as_float(bw[2 * e + 1]));
            } else {
              u = affine2_mixed<WD>(narrow2<WD>(a.x, a.y), ww[e], bw[e]);  // cast to the weight dtype first
            }
            o[2 * e] = u.x;
            o[2 * e + 1] = u.y;
          }
          narrow<OD, V>(o, ow);
        } else if constexpr (WD == OD && WD != FAR_F32) {
          // 16-bit weight and output (then act == wd): cast to the weight dtype, then one
          // packed multiply rounds the exact product once.  With a quantised output s * rstd
          // is formed two lanes at a time (each half rounded as the scalar multiply; it feeds
          // only the cast, never an add); the plain kernels keep the scalar form, whose
          // registers fit without spilling
          if constexpr (Q != kQuantNone) {
            const uint64_t rstd2 = pk(rstd, rstd);
#pragma unroll
            for (int e = 0; e < V / 2; ++e) {
              const float2 a = unpk(mul_x2(pk(sj[2 * e], sj[2 * e + 1]), rstd2));
              ow[e] = mul2<WD>(narrow2<WD>(a.x, a.y), ww[e]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < V / 2; ++e)
              ow[e] = mul2<WD>(narrow2<WD>(__fmul_rn(sj[2 * e], rstd), __fmul_rn(sj[2 * e + 1], rstd)), ww[e]);
          }
        } else {
          float wf[V];
          widen<WD, V>(ww, wf);
          float o[V];
#pragma unroll
          for (int e = 0; e < V; ++e) o[e] = __fmul_rn(sj[e], rstd);
          round_through<WD, V>(o);  // cast to the weight dtype first
#pragma unroll
          for (int e = 0; e < V; ++e) o[e] = __fmul_rn(o[e], wf[e]);
          narrow<OD, V>(o, ow);
        }
        if constexpr (Q) {
          if constexpr (OD == FAR_F32) {
#pragma unroll
            for (int e = 0; e < V; ++e) amax = max_nan(amax, fabsf(__uint_as_float(ow[e])));
          } else {
            // |out| of two 16-bit values at a time (max of 16-bit values is exact)
#pragma unroll
            for (int e = 0; e < OB / 4; ++e) amax2 = habs_max2<OD>(amax2, ow[e]);
          }
#pragma unroll
          for (int e = 0; e < OB / 4; ++e) okeep[j][e] = ow[e];
        } else {
          store_row(orow, w, ow, std::integral_constant<int, OB>{});
        }
        if constexpr (RES && !LN) {
          uint32_t rw[4];
          narrow<ACT, V>(sj, rw);
          store_row(rrow, w, rw, std::integral_constant<int, 16>{});
        }
      }
    }
    if constexpr (Q) {
      if constexpr (OD != FAR_F32) {
        const float2 m2 = widen2<OD>(amax2);
        amax = max_nan(m2.x, m2.y);
      }
      // the row's largest |out|: warp, then group (its own pair of buffers), all lanes agree
      amax = warp_max_allreduce(amax);
      if (G > 1) {
        const int buf = 2 + (int)(it & 1u);
        float2* part = partials + (size_t)(g * NRED + buf) * G;
        const uint32_t rbar = smem_addr(&bars[2 * stages + g * NRED + buf]);
        if (lane == 0) {
          part[wg] = make_float2(amax, 0.f);
          mbar_arrive(rbar);
        }
        if (!mbar_wait(rbar, (it >> 1) & 1u, p.timeout_ns, p.status)) return;
        float m = part[lane < G ? lane : 0].x;
        amax = warp_max_allreduce(m);
      }
      // scale = amax / QMAX; q = Q(out * (QMAX / amax)), 0 for an all-zero row
      constexpr float QMAX = Q == kQuantInt8 ? 127.0f : 448.0f;
      const float inv = amax == 0.f ? 0.f : __fdiv_rn(QMAX, amax);
      if (wg == 0 && lane == 0) p.scale[row] = __fdiv_rn(amax, QMAX);
      unsigned char* qrow = static_cast<unsigned char*>(p.q) + row * (int64_t)p.hidden;
      // int8 of a row whose largest |out| is finite: every v = fl32(out * inv) lies within
      // +-(127 + 2^-17), so adding 1.5 * 2^23 in binary32 rounds it to the nearest integer,
      // ties to even, and leaves that integer (two's complement) in the low byte: the
      // saturating conversion's result, on the FMA pipe and two lanes an instruction.  A row
      // whose largest |out| is NaN or infinite has every v NaN or +-0: all codes 0.
      const bool finite_row = isfinite(amax);
      const uint64_t magic2 = pk(12582912.0f, 12582912.0f);
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const Where w = where(j);
        if (w.va) {
          float of[V];
          widen<OD, V>(okeep[j], of);
          uint32_t qw[V / 4];
          if constexpr (Q == kQuantInt8) {
#pragma unroll
            for (int e = 0; e < V / 4; ++e) {
              // the products by the scalar multiply (never contracted into the add)
              const uint64_t t01 = add_x2(pk(__fmul_rn(of[4 * e], inv), __fmul_rn(of[4 * e + 1], inv)), magic2);
              uint32_t hi;
              if constexpr (RES) {
                const uint64_t t23 = add_x2(pk(__fmul_rn(of[4 * e + 2], inv), __fmul_rn(of[4 * e + 3], inv)), magic2);
                hi = __byte_perm((uint32_t)t23, (uint32_t)(t23 >> 32), 0x0040);
              } else {
                // The issue-bound no-residual kernel converts one value in four with the
                // saturating conversion instead: it runs on another pipe than the adds, which
                // the FMA pipe's other work keeps busy (fp16 65536 x 8192: 302 us against 338
                // with every code from the add, 313 with two in four converted, 310 with three)
                const uint32_t t2 = __float_as_uint(__fadd_rn(__fmul_rn(of[4 * e + 2], inv), 12582912.0f));
                uint32_t q3;
                asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(q3) : "f"(__fmul_rn(of[4 * e + 3], inv)));
                hi = __byte_perm(t2, q3, 0x0040);
              }
              const uint32_t lo = __byte_perm((uint32_t)t01, (uint32_t)(t01 >> 32), 0x0040);
              qw[e] = finite_row ? __byte_perm(lo, hi, 0x5410) : 0u;
            }
          } else {
#pragma unroll
            for (int e = 0; e < V / 4; ++e)
              qw[e] = quantise4<Q>(__fmul_rn(of[4 * e], inv), __fmul_rn(of[4 * e + 1], inv),
                                   __fmul_rn(of[4 * e + 2], inv), __fmul_rn(of[4 * e + 3], inv));
          }
          if constexpr (V == 8) {
            store_bytes<8>(qrow + (size_t)w.pa * 8, qw);
          } else {
            asm volatile("st.global.b32 [%0], %1;" ::"l"(qrow + (size_t)w.pa * 4), "r"(qw[0]) : "memory");
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// generic path: any alignment, any hidden size
// ---------------------------------------------------------------------------

template <int DT> __device__ __forceinline__ float load_elem(const void* base, int64_t i) {
  if constexpr (DT == FAR_F16) return __half2float(static_cast<const __half*>(base)[i]);
  else if constexpr (DT == FAR_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
  else return static_cast<const float*>(base)[i];
}

// store a binary32 value rounded to nearest even in dtype DT
template <int DT> __device__ __forceinline__ void store_elem(void* base, int64_t i, float v) {
  if constexpr (DT == FAR_F16) static_cast<__half*>(base)[i] = __float2half_rn(v);
  else if constexpr (DT == FAR_BF16) static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  else static_cast<float*>(base)[i] = v;
}

template <int DT> __device__ __forceinline__ float round_one(float v) {
  if constexpr (DT == FAR_F16) return __half2float(__float2half_rn(v));
  else if constexpr (DT == FAR_BF16) return __bfloat162float(__float2bfloat16_rn(v));
  else return v;
}

// a double word summed over the CTA: warps first, then the warp values in a fixed order
// (every thread ends with the same bits); `part` is free again on return
template <int NW, typename Combine, typename WarpReduce>
__device__ __forceinline__ DW block_reduce(DW acc, float2* part, int warp, int lane, Combine combine,
                                           WarpReduce warp_reduce) {
  acc = warp_reduce(acc);
  if (lane == 0) part[warp] = make_float2(acc.hi, acc.lo);
  __syncthreads();
  DW tot{part[0].x, part[0].y};
  for (int i = 1; i < NW; ++i) tot = combine(tot, DW{part[i].x, part[i].y});
  __syncthreads();
  return tot;
}

// LayerNorm, one row per CTA in three passes over the row (the re-reads come from L1/L2):
// the signed sum of s for the mean, the sum of the squared deviations, then the outputs
template <int ACT, int WD, bool RES>
__device__ __forceinline__ void generic_ln_row(const Params& p, int64_t row, float2* part, int warp, int lane) {
  constexpr int OD = promote(ACT, WD);
  constexpr int NW = kGenericThreads / 32;
  const int64_t H = p.hidden;
  const char* xr = static_cast<const char*>(p.x) + row * p.x_stride;
  const char* rr = RES ? static_cast<const char*>(p.r) + row * p.r_stride : nullptr;
  auto s_at = [&](int64_t i) {
    float s = load_elem<ACT>(xr, i);
    if constexpr (RES) s = __fadd_rn(s, load_elem<ACT>(rr, i));
    return s;
  };
  DW acc{0.f, 0.f};
  for (int64_t i = threadIdx.x; i < H; i += blockDim.x) dw_add_signed(acc, s_at(i));
  const DW tot = block_reduce<NW>(acc, part, warp, lane, dw_combine_signed, dw_warp_allreduce_signed);
  const float mean = __fdiv_rn(dw_value(tot), p.hidden_f);
  DW acc2{0.f, 0.f};
  for (int64_t i = threadIdx.x; i < H; i += blockDim.x) {
    const float d = __fsub_rn(s_at(i), mean);
    dw_add(acc2, __fmul_rn(d, d));
  }
  const DW tot2 = block_reduce<NW>(acc2, part, warp, lane, dw_combine, dw_warp_allreduce);
  const float rstd = row_rstd(dw_value(tot2), p.hidden_f, p.eps);
  char* orow = static_cast<char*>(p.out) + row * p.out_stride;
  char* rrow = RES ? static_cast<char*>(p.res_out) + row * p.res_stride : nullptr;
  for (int64_t i = threadIdx.x; i < H; i += blockDim.x) {
    const float s = s_at(i);  // each element is read and written by the same thread
    if constexpr (RES) store_elem<ACT>(rrow, i, s);
    const float n = round_one<WD>(__fmul_rn(__fsub_rn(s, mean), rstd));
    store_elem<OD>(orow, i, __fadd_rn(__fmul_rn(n, load_elem<WD>(p.w, i)), load_elem<WD>(p.beta, i)));
  }
}

template <int ACT, int WD, bool RES, int Q = kQuantNone, bool LN = false>
__global__ void __launch_bounds__(kGenericThreads) generic_kernel(const Params p) {
  constexpr int OD = promote(ACT, WD);
  constexpr int NW = kGenericThreads / 32;
  __shared__ float2 part[NW];
  __shared__ float mpart[NW];
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t H = p.hidden;
  for (int64_t row = blockIdx.x; row < p.tokens; row += gridDim.x) {
    if constexpr (LN) {
      generic_ln_row<ACT, WD, RES>(p, row, part, warp, lane);
      continue;
    }
    const char* xr = static_cast<const char*>(p.x) + row * p.x_stride;
    const char* rr = RES ? static_cast<const char*>(p.r) + row * p.r_stride : nullptr;
    DW acc{0.f, 0.f};
    for (int64_t i = threadIdx.x; i < H; i += blockDim.x) {
      float s = load_elem<ACT>(xr, i);
      if constexpr (RES) s = __fadd_rn(s, load_elem<ACT>(rr, i));
      dw_add(acc, __fmul_rn(s, s));
    }
    acc = dw_warp_allreduce(acc);
    if (lane == 0) part[warp] = make_float2(acc.hi, acc.lo);
    __syncthreads();
    DW tot{part[0].x, part[0].y};
    for (int i = 1; i < NW; ++i) tot = dw_combine(tot, DW{part[i].x, part[i].y});
    __syncthreads();  // `part` is reused by the next row
    const float rstd = row_rstd(dw_value(tot), p.hidden_f, p.eps);
    char* orow = Q ? nullptr : static_cast<char*>(p.out) + row * p.out_stride;
    char* rrow = RES ? static_cast<char*>(p.res_out) + row * p.res_stride : nullptr;
    float amax = 0.f;
    for (int64_t i = threadIdx.x; i < H; i += blockDim.x) {
      float s = load_elem<ACT>(xr, i);  // each element is read and written by the same thread
      if constexpr (RES) {
        s = __fadd_rn(s, load_elem<ACT>(rr, i));
        store_elem<ACT>(rrow, i, s);
      }
      const float n = round_one<WD>(__fmul_rn(s, rstd));
      const float o = __fmul_rn(n, load_elem<WD>(p.w, i));
      if constexpr (Q) amax = max_nan(amax, fabsf(round_one<OD>(o)));
      else store_elem<OD>(orow, i, o);
    }
    if constexpr (Q) {
      // third pass: the row's largest |out|, then the quantised bytes (out recomputed)
      amax = warp_max_allreduce(amax);
      if (lane == 0) mpart[warp] = amax;
      __syncthreads();
      float m = mpart[0];
      for (int i = 1; i < NW; ++i) m = max_nan(m, mpart[i]);
      __syncthreads();  // `mpart` is reused by the next row
      constexpr float QMAX = Q == kQuantInt8 ? 127.0f : 448.0f;
      const float inv = m == 0.f ? 0.f : __fdiv_rn(QMAX, m);
      if (threadIdx.x == 0) p.scale[row] = __fdiv_rn(m, QMAX);
      unsigned char* qrow = static_cast<unsigned char*>(p.q) + row * H;
      for (int64_t i = threadIdx.x; i < H; i += blockDim.x) {
        float s = load_elem<ACT>(xr, i);
        if constexpr (RES) s = __fadd_rn(s, load_elem<ACT>(rr, i));
        const float n = round_one<WD>(__fmul_rn(s, rstd));
        const float v = __fmul_rn(round_one<OD>(__fmul_rn(n, load_elem<WD>(p.w, i))), inv);
        qrow[i] = (unsigned char)(quantise4<Q>(v, 0.f, 0.f, 0.f) & 0xffu);
      }
    }
  }
}

cudaError_t ensure_smem_attribute(const void* func, size_t bytes);

template <int ACT, int WD, bool RES, int Q, bool LN = false>
cudaError_t launch_typed(const Launch& L) {
  void (*k)(Params) = nullptr;
  if (L.kind == kGeneric) {
    k = generic_kernel<ACT, WD, RES, Q, LN>;
  } else {
    switch (L.nch * 2 + (L.exact ? 1 : 0)) {
      case 2: k = staged_kernel<ACT, WD, RES, 1, false, Q, LN>; break;
      case 3: k = staged_kernel<ACT, WD, RES, 1, true, Q, LN>; break;
      case 4: k = staged_kernel<ACT, WD, RES, 2, false, Q, LN>; break;
      case 5: k = staged_kernel<ACT, WD, RES, 2, true, Q, LN>; break;
      case 8: k = staged_kernel<ACT, WD, RES, 4, false, Q, LN>; break;
      case 9: k = staged_kernel<ACT, WD, RES, 4, true, Q, LN>; break;
      case 16: k = staged_kernel<ACT, WD, RES, 8, false, Q, LN>; break;
      case 17: k = staged_kernel<ACT, WD, RES, 8, true, Q, LN>; break;
      // 5 or 6 chunks a thread, only where they cover a row exactly (hidden 5120 or 2560 in
      // 16-bit with 4 or 2 warps a row, 3072 with 2): RMSNorm and LayerNorm; 5 chunks also
      // with a quantised output
      case 11:
        if constexpr (true) {
          k = staged_kernel<ACT, WD, RES, 5, true, Q, LN>;
          break;
        } else {
          return cudaErrorInvalidValue;
        }
      case 13:
        if constexpr (Q == kQuantNone) {
          k = staged_kernel<ACT, WD, RES, 6, true, Q, LN>;
          break;
        } else {
          return cudaErrorInvalidValue;
        }
      // 10 chunks a thread: the no-residual variant on 16-bit rows that 2 warps cover
      // exactly at 10 (hidden 5120 with x kept packed)
      case 21:
        if constexpr (Q == kQuantNone && !LN && packed_rows(RES, ACT)) {
          k = staged_kernel<ACT, WD, RES, 10, true, Q, LN>;
          break;
        } else {
          return cudaErrorInvalidValue;
        }
      default: return cudaErrorInvalidValue;
    }
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(k), L.smem);
    if (e != cudaSuccess) return e;
  }
  if (!L.programmatic) {
    k<<<L.grid, L.block, L.smem, L.stream>>>(L.p);
    return cudaGetLastError();
  }
  // programmatic dependent launch: this kernel may be dispatched while the kernel ahead of
  // it on the stream finishes (it waits for that kernel's completion before touching memory)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = L.grid;
  cfg.blockDim = L.block;
  cfg.dynamicSmemBytes = L.smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, L.p);
}

// the plain output
template <int ACT, int WD>
cudaError_t launch_res(bool residual, const Launch& L) {
  return residual ? launch_typed<ACT, WD, true, kQuantNone>(L) : launch_typed<ACT, WD, false, kQuantNone>(L);
}

// a quantised output (int8 or FP8 E4M3)
template <int ACT, int WD>
cudaError_t launch_quant(bool residual, const Launch& L) {
  if (L.quant == kQuantInt8)
    return residual ? launch_typed<ACT, WD, true, kQuantInt8>(L) : launch_typed<ACT, WD, false, kQuantInt8>(L);
  if (L.quant == kQuantFp8)
    return residual ? launch_typed<ACT, WD, true, kQuantFp8>(L) : launch_typed<ACT, WD, false, kQuantFp8>(L);
  return cudaErrorInvalidValue;
}

// LayerNorm (plain output)
template <int ACT, int WD>
cudaError_t launch_ln(bool residual, const Launch& L) {
  return residual ? launch_typed<ACT, WD, true, kQuantNone, true>(L)
                  : launch_typed<ACT, WD, false, kQuantNone, true>(L);
}

}  // namespace far
