// Device-side building blocks of the fused data-parallel step (sm_103a).
//
// Work decomposition shared by every kernel: the non-empty segments of a
// layout are cut on the global grid of TILE elements, so a tile never
// crosses a segment (owner) boundary and never crosses a TILE cell.  A
// tile's aligned hull [floor8(start), ceil8(end)) therefore stays inside
// its cell, which keeps every bulk copy 16-byte aligned.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dpstep.h"

namespace dp {

constexpr int TILE = 7680;          // elements per tile, multiple of 8 (15 KB of bf16: one bulk copy)
constexpr int SMALL_SEG = 32;       // segment-table capacity of the small kernel variants
constexpr int BIG_SEG = DP_KERNEL_SEG; // ... and of the large ones (a larger layout runs as several launches)

struct SegEntry {
  int64_t goff;   // first global element of the segment
  int64_t loff;   // first local element in the owner's shard arrays
  int32_t tile0;  // index of the segment's first tile
  int32_t owner;
};

// Passed by value inside kernel parameters (__grid_constant__): e[nseg] is a
// sentinel with goff = psi and tile0 = ntiles.
template <int MAXSEG>
struct SegTable {
  int64_t psi;
  int32_t nseg;
  int32_t ntiles;
  SegEntry e[MAXSEG + 1];
};

struct Tile {
  int64_t goff, loff, start, end;  // segment origin (global, local) and the tile's global range
  int32_t owner;
};

template <int MAXSEG>
__device__ __forceinline__ Tile tile_at(const SegTable<MAXSEG>& T, int tile) {
  int lo = 0, hi = T.nseg - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (T.e[mid].tile0 <= tile) lo = mid; else hi = mid - 1;
  }
  const int64_t goff = T.e[lo].goff;
  const int64_t gend = T.e[lo + 1].goff;
  const int64_t cell = goff / TILE + (tile - T.e[lo].tile0);
  Tile t;
  t.goff = goff;
  t.loff = T.e[lo].loff;
  t.owner = T.e[lo].owner;
  t.start = goff > cell * TILE ? goff : cell * TILE;
  t.end = gend < (cell + 1) * TILE ? gend : (cell + 1) * TILE;
  return t;
}

// Tiles of one CTA are visited in increasing order, so their segments are found by walking forward.
template <int MAXSEG>
struct TileWalker {
  int seg = 0;
  __device__ __forceinline__ Tile at(const SegTable<MAXSEG>& T, int tile) {
    while (seg + 1 < T.nseg && T.e[seg + 1].tile0 <= tile) ++seg;
    const int64_t goff = T.e[seg].goff;
    const int64_t gend = T.e[seg + 1].goff;
    const int64_t cell = goff / TILE + (tile - T.e[seg].tile0);
    Tile t;
    t.goff = goff;
    t.loff = T.e[seg].loff;
    t.owner = T.e[seg].owner;
    t.start = goff > cell * TILE ? goff : cell * TILE;
    t.end = gend < (cell + 1) * TILE ? gend : (cell + 1) * TILE;
    return t;
  }
};

// ---------------------------------------------------------------- fp32 arithmetic

__device__ __forceinline__ bool nonfinite(float x) {
  return (__float_as_uint(x) & 0x7F800000u) == 0x7F800000u;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Error-free sum: s = fl(a + b) and e with s + e = a + b exactly.  Computed as Dekker's Fast2Sum
// (Numer. Math. 18, 1971) after ordering the operands by magnitude: s = big + small, e = small - (s - big).
// For finite inputs (s, e) is unique, so this equals Knuth's TwoSum (TAOCP vol. 2, 4.2.2) except possibly
// for the sign of a zero e, which the accumulators below cannot observe (their running error terms are
// never -0: in round-to-nearest an exact zero sum is +0 unless both addends are -0).
__device__ __forceinline__ float two_sum(float a, float b, float& e) {
  const bool ge = fabsf(a) >= fabsf(b);
  const float big = ge ? a : b, small = ge ? b : a;
  const float s = __fadd_rn(big, small);
  e = __fsub_rn(small, __fsub_rn(s, big));
  return s;
}

// Packed pairs of fp32 for the sm_100+ f32x2 instructions: two independent
// round-to-nearest operations per instruction, bit-identical to the scalar ones.
typedef unsigned long long f2_t;

__device__ __forceinline__ f2_t f2_pack(float lo, float hi) {
  f2_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(f2_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
  f2_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2_t f2_sub(f2_t a, f2_t b) {
  f2_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
  f2_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// Knuth's TwoSum on a packed pair: six packed additions, no ordering (FP32 pipes only).
__device__ __forceinline__ f2_t f2_two_sum(f2_t a, f2_t b, f2_t& e) {
  const f2_t s = f2_add(a, b);
  const f2_t z = f2_sub(s, a);
  e = f2_add(f2_sub(a, f2_sub(s, z)), f2_sub(b, z));
  return s;
}
// The same error-free sum as Fast2Sum after per-lane magnitude ordering: three packed additions plus a
// compare and two selects per lane (spreads the work over the integer pipe).  Same (s, e) as f2_two_sum
// for finite inputs, up to the sign of a zero e.
__device__ __forceinline__ f2_t f2_fast_two_sum(f2_t a, f2_t b, f2_t& e) {
  float a0, a1, b0, b1;
  f2_unpack(a, a0, a1);
  f2_unpack(b, b0, b1);
  const bool g0 = fabsf(a0) >= fabsf(b0), g1 = fabsf(a1) >= fabsf(b1);
  const f2_t big = f2_pack(g0 ? a0 : b0, g1 ? a1 : b1);
  const f2_t small = f2_pack(g0 ? b0 : a0, g1 ? b1 : a1);
  const f2_t s = f2_add(big, small);
  e = f2_sub(small, f2_sub(s, big));
  return s;
}
// Two bf16 (low half = first element) widened to an fp32 pair, built directly as one 64-bit value.
__device__ __forceinline__ f2_t bf16x2_to_f2(uint32_t w) {
  return ((f2_t)(w & 0xFFFF0000u) << 32) | (f2_t)(w << 16);
}

// ---------------------------------------------------------------- Adam

struct AdamK {
  float b1, b2, omb1, omb2, eps;
  float step;   // fl32(lr / (1 - beta1^t))
  float rsbc2;  // fl32(1 / sqrt(1 - beta2^t))
};

// The hardware's approximate square root and division (one MUFU-based instruction each, PTX sqrt.approx.f32
// and div.approx.f32: relative error about 2^-23 and at most 2 ulp for divisors in [2^-126, 2^126]).
__device__ __forceinline__ float sqrt_approx(float x) {
  float r;
  asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float div_approx(float a, float b) {
  float r;
  asm("div.approx.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// One Adam update in fp32 (no contraction):
//   m' = b1 m + (1-b1) g ; v' = b2 v + ((1-b2) g) g        each operation rounded once
//   th' = th - (step m') / (sqrt(v') rsbc2 + eps)          square root and division by the approximate
// instructions above.  The update term's error is then a few ulp of itself -- at most ~3e-10 absolute for
// lr = 1e-3 -- far inside the fp32 master tolerance (1e-9 + 2e-6 |x|); the moments are exact fp32 operations.
// Every GPU path uses this function, so paths that must agree bit for bit still do.
__device__ __forceinline__ void adam1(float g, float& th, float& m, float& v, const AdamK& K) {
  const float m1 = __fmaf_rn(K.b1, m, __fmul_rn(K.omb1, g));
  const float v1 = __fmaf_rn(K.b2, v, __fmul_rn(__fmul_rn(K.omb2, g), g));
  const float den = __fmaf_rn(sqrt_approx(v1), K.rsbc2, K.eps);
  th = __fsub_rn(th, div_approx(__fmul_rn(K.step, m1), den));
  m = m1;
  v = v1;
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}
__device__ __forceinline__ uint16_t bf16_rn(float x) {
  const __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&b);
}

// ---------------------------------------------------------------- async copies and barriers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up (returns
// false) after timeout_ns of wall time, or at once when *abort is set.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                                  volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort && *abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// Global -> shared bulk copy completing on an mbarrier (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// Shared -> global bulk copy in the current bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void record_error(dp_step_state_t* st, int code) {
  atomicCAS(&st->error, 0, code);
}

// Dynamic loss-scale policy applied when a step is committed (see dp_scaler_t).
struct ScalerK {
  int32_t enabled;   // the reduction unscales by the device-resident scale
  int32_t interval;
  float growth, backoff, min_scale, max_scale;
  int32_t update;    // the commit applies the policy to the device-resident scale
};

// Commits a step once its skip decision `found` is final: unless found, t and the beta powers advance (and the
// single pass's current state set flips); the dynamic loss scale follows the decision unless a device error
// stopped the step.  Run by one thread.
__device__ __forceinline__ void commit_state(dp_step_state_t* st, int found, int err, double b1, double b2,
                                             const ScalerK* scaler, int flip_set) {
  if (!found) {
    st->t += 1;
    st->b1t *= b1;
    st->b2t *= b2;
    if (flip_set) st->cur_set ^= 1u;
  }
  if (scaler && scaler->update && err == 0) {
    float sc = st->loss_scale;
    if (found) {
      sc = fmaxf(__fmul_rn(sc, scaler->backoff), scaler->min_scale);
      st->good_steps = 0;
    } else if (st->good_steps + 1 >= scaler->interval) {
      sc = fminf(__fmul_rn(sc, scaler->growth), scaler->max_scale);
      st->good_steps = 0;
    } else {
      st->good_steps += 1;
    }
    st->loss_scale = sc;
  }
}

// End of a reduction kernel, run by thread 0 of every CTA: fold the CTA's non-finite count into the state; the
// last CTA to arrive publishes found_inf / nonfinite (merge: ORed and added into what an earlier launch of the
// same reduction published), commits the step unless the commit is deferred (advance = 0: a later launch, or
// the caller after combining found_inf across slices, commits), and clears the work fields for the next call.
__device__ __forceinline__ void finish_reduction(dp_step_state_t* st, unsigned long long cta_count, int cta_found,
                                                 int advance, double b1, double b2,
                                                 const ScalerK* scaler = nullptr, int flip_set = 0, int merge = 0) {
  if (cta_count) atomicAdd(reinterpret_cast<unsigned long long*>(&st->work_count), cta_count);
  if (cta_found) atomicOr(&st->work_found, 1u);
  __threadfence();
  const unsigned ticket = atomicAdd(&st->work_ticket, 1u);
  if (ticket == gridDim.x - 1) {
    __threadfence();
    const unsigned f = atomicExch(&st->work_found, 0u);
    unsigned long long c = atomicExch(reinterpret_cast<unsigned long long*>(&st->work_count), 0ull);
    const int err = *reinterpret_cast<volatile int*>(&st->error);
    int found = (f != 0u || err != 0) ? 1 : 0;
    if (merge) {   // a later launch of the same reduction (a layout run in several launches)
      found |= *reinterpret_cast<volatile int*>(&st->found_inf) != 0 ? 1 : 0;
      c += *reinterpret_cast<volatile unsigned long long*>(&st->nonfinite);
    }
    st->found_inf = found;
    st->nonfinite = c;
    if (advance) commit_state(st, found, err, b1, b2, scaler, flip_set);
    __threadfence();
    atomicExch(&st->work_ticket, 0u);
  }
}

}  // namespace dp
