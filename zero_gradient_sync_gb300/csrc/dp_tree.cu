// The tree reduction order (sm_103a): pass A of the step, and the staged reduce-scatter, with the ranks' sums
// added up a binomial tree instead of the ring.
//
// The second fixed order: a binomial tree over rank index rooted at rank 0, as in the tree all-reduce that
// NCCL offers beside the ring for its lower step count ("Data vs Tensor vs Pipeline Parallelism", DP
// gradient sync at scale).  Level l adds the block of ranks [j 2^(l+1) + 2^l, (j+1) 2^(l+1)) into the block
// [j 2^(l+1), j 2^(l+1) + 2^l), the lower block as the left operand; a block with no partner (n not a power
// of two) goes up a level unchanged.  The order does not depend on the shard owner (the all-reduce root is
// rank 0 for every element); each owner keeps its shard of the result.
//
// Both pass-A kernels take the ring kernel's stream: a producer warp issuing 1-D bulk copies into a ring of
// shared-memory stages, bounded mbarrier waits.
// reduce_tree_kernel (plain arithmetic): consumers keep the tree as a binary counter -- slot l holds the
// pending sum of a complete block of 2^l ranks, so at most log2(n) partial sums are live, each in registers.
// A consumer thread owns 8 elements (the ring kernel's 16), so a stage input is half a tile (3840 elements, a
// 7.5 KB copy), four inputs to a stage.  Whole half tiles take a loop without per-input guards.
// reduce_tree_rm_kernel (compensated arithmetic): a stage holds one micro-step of every rank; each thread
// carries every rank's (hi, lo) leaf and adds the leaves up a tree fixed at compile time (below).
// rs_tree_kernel: the same tree over the staged per-rank accumulators, one element per thread.
#include <type_traits>

#include "dp_device.cuh"
#include "dp_internal.h"
#include "dp_launch.h"

namespace dp {
namespace {

constexpr int TT_CWARPS = 15;
constexpr int TT_CTHREADS = TT_CWARPS * 32;
constexpr int TT_EPT = 8;                          // elements per consumer thread: one 16-byte shared load
constexpr int TT_THREADS = TT_CTHREADS + 32;       // + one producer warp
constexpr int TT_SUB = TT_CTHREADS * TT_EPT;       // elements of a stage input: half a tile
constexpr int TT_IN_BYTES = TT_SUB * 2;            // one input's half tile: a 7.5 KB bulk copy
constexpr int TT_RING_BYTES = 24 * TT_IN_BYTES;    // 180 KB of stages in flight
constexpr int TT_MAX_STAGES = 12;                  // barrier pairs reserved (either kernel)
constexpr int TT_SMEM = TT_RING_BYTES + 2 * TT_MAX_STAGES * 8 + 32;
constexpr int RT_LEVELS = 5;                       // staged kernel: slots for n <= 16 (levels 0..4)
constexpr int TT_NPS = 4;                          // binary counter: inputs per stage
constexpr int TT_STAGES = TT_RING_BYTES / (TT_NPS * TT_IN_BYTES);
static_assert(TILE == 2 * TT_SUB, "a tile is two half tiles");
static_assert(TT_IN_BYTES % 16 == 0, "bulk copies are whole 16-byte units");
static_assert(TT_STAGES <= TT_MAX_STAGES, "barriers fit");
static_assert(TT_SMEM + 64 <= 227 * 1024, "shared memory fits one CTA");

template <int MAXSEG>
struct TreeParams {
  const uint16_t* g[DP_MAX_NA];
  float* gbar[DP_MAX_N];
  dp_step_state_t* state;
  uint64_t timeout_ns;
  double beta1, beta2;
  float inv;
  int32_t n, a, advance;
  int32_t merge;     // a later launch of one reduction (see finish_reduction)
  ScalerK scaler;
  SegTable<MAXSEG> seg;
};

// Eight elements' partial sum: four packed pairs.
struct Part8 {
  f2_t h[4];
};

// left + right, left being the lower-index block.
__device__ __forceinline__ Part8 tree_add(const Part8& x, const Part8& y) {
  Part8 z;
#pragma unroll
  for (int u = 0; u < 4; ++u) z.h[u] = f2_add(x.h[u], y.h[u]);
  return z;
}

template <int NST>
struct StagePos {
  uint32_t slot = 0, phase = 0, count = 0;
  __device__ __forceinline__ void next() {
    ++count;
    if (++slot == NST) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Fold input HH of a stage (4 words = 8 bf16 of this thread) into rank r's partial sum `cur` (kfirst: its first
// micro-step).  At the rank's last micro-step (klast) the rank is complete: the slots below the lowest clear
// bit of r are all occupied and merge into it, and that bit's slot takes the sum (static slot indices keep
// every slot in registers).  When r completes a block of 2^LEVELS ranks, cur is left holding the total.
template <int LEVELS, int HH, int NW>
__device__ __forceinline__ void tree_fold(Part8 (&slot)[LEVELS], Part8& cur, const uint32_t (&w)[NW], int r,
                                          bool kfirst, bool klast) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const f2_t xx = bf16x2_to_f2(w[4 * HH + u]);
    cur.h[u] = kfirst ? xx : f2_add(cur.h[u], xx);
  }
  if (klast) {
    const int top = __ffs(~r) - 1;
#pragma unroll
    for (int lv = 0; lv < LEVELS; ++lv) {
      if (lv < top) cur = tree_add(slot[lv], cur);
      else if (lv == top) slot[lv] = cur;
    }
  }
}

// The elements [lo, hi) of a tile inside one part of its cell (a half tile here, a sub-tile below), copied as
// the 8-aligned hull [lo & ~7, min(ceil8(hi), psi & ~7)) -- the buffer's last partial 8 elements are read
// from global memory.
struct Half {
  int64_t lo, hi, sa;
  __device__ __forceinline__ bool empty() const { return lo >= hi; }
};
__device__ __forceinline__ Half half_of(const Tile& t, int h) {
  const int64_t cb = (t.start / TILE) * TILE + (int64_t)h * TT_SUB;
  Half x;
  x.lo = t.start > cb ? t.start : cb;
  x.hi = t.end < cb + TT_SUB ? t.end : cb + TT_SUB;
  x.sa = x.lo & ~int64_t(7);
  return x;
}

// LEVELS = log2 of the largest n this instance serves (3: n <= 8, 4: n <= 16); slots 0..LEVELS-1 hold
// pending blocks, and a full block of 2^LEVELS ranks is the total itself.
template <int MAXSEG, int LEVELS>
__global__ void __launch_bounds__(TT_THREADS, 1) reduce_tree_kernel(const __grid_constant__ TreeParams<MAXSEG> p) {
  constexpr int NPS = TT_NPS;
  constexpr int NST = TT_STAGES;
  constexpr int SBY = NPS * TT_IN_BYTES;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TT_RING_BYTES);
  uint64_t* empty = full + NST;
  volatile int* s_abort = reinterpret_cast<volatile int*>(empty + NST);
  unsigned long long* s_count = reinterpret_cast<unsigned long long*>(empty + NST + 1);
  __shared__ float s_inv;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = p.n, a = p.a, nin = n * a;
  const int ntiles = p.seg.ntiles;
  const int64_t psi = p.seg.psi;
  const int64_t p8 = psi & ~int64_t(7);

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), TT_CWARPS);
    }
    *s_abort = 0;
    *s_count = 0ull;
    float inv = p.inv;
    if (p.scaler.enabled) {
      // fl32(1 / (n S)) from the device-resident scale, as for the ring order.
      const float sc = *reinterpret_cast<volatile const float*>(&p.state->loss_scale);
      inv = (float)(1.0 / ((double)p.n * (double)sc));
      if (!(sc > 0.0f) || nonfinite(sc) || !(inv >= 1.17549435e-38f) || nonfinite(inv)) {
        record_error(p.state, DP_ERR_INVALID_ARG);
        *s_abort = 1;
        inv = 0.0f;
      }
    }
    s_inv = inv;
    fence_mbar_init();
  }
  __syncthreads();

  unsigned bad = 0;
  if (warp == TT_CWARPS) {
    // ------------------------------------------------------------ producer: inputs in rank order 0..n-1
    if (lane == 0) {
      StagePos<NST> sp;
      TileWalker<MAXSEG> walk;
      for (int tile = blockIdx.x; tile < ntiles && !*s_abort; tile += gridDim.x) {
        const Tile t = walk.at(p.seg, tile);
        for (int h = 0; h < 2 && !*s_abort; ++h) {
          const Half x = half_of(t, h);
          if (x.empty()) continue;
          int64_t sb = (x.hi + 7) & ~int64_t(7);
          if (sb > p8) sb = p8;
          const uint32_t bytes = sb > x.sa ? (uint32_t)(sb - x.sa) * 2u : 0u;
          for (int q = 0; q < nin && !*s_abort; q += NPS) {
            if (sp.count >= (uint32_t)NST &&
                !mbar_wait_bounded(smem_u32(&empty[sp.slot]), sp.phase ^ 1u, p.timeout_ns, s_abort)) {
              if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
              *s_abort = 1;
              break;
            }
            const int cnt = nin - q < NPS ? nin - q : NPS;
            const uint32_t fb = smem_u32(&full[sp.slot]);
            mbar_arrive_expect_tx(fb, bytes * (uint32_t)cnt);
            if (bytes)
              for (int hh = 0; hh < cnt; ++hh)
                bulk_g2s(smem_u32(stages + sp.slot * SBY + hh * TT_IN_BYTES), p.g[q + hh] + x.sa, bytes, fb);
            sp.next();
          }
        }
      }
      // Never leave with copies in flight: wait for the newest issued phase of every slot.
      if (*s_abort) {
        const uint32_t it = sp.count;
        const uint32_t first = it > (uint32_t)NST ? it - NST : 0u;
        for (uint32_t y = first; y < it; ++y)
          (void)mbar_wait_bounded(smem_u32(&full[y % NST]), (y / NST) & 1u, p.timeout_ns, nullptr);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers: 8 elements per thread
    const f2_t inv2 = f2_pack(s_inv, s_inv);
    StagePos<NST> sp;
    TileWalker<MAXSEG> walk;
    bool live = true;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const Tile t = walk.at(p.seg, tile);
      for (int h = 0; h < 2; ++h) {
        const Half x = half_of(t, h);
        if (x.empty()) continue;
        const int64_t e0 = x.sa + TT_EPT * tid;
        const bool active = e0 < x.hi;
        const bool tailgrp = active && (e0 + TT_EPT > p8);

        // One stage: wait for its bytes, take this thread's 8 values of each of its cnt inputs (input q0 + hh),
        // release the slot.  whole (a whole half tile below the buffer's last partial 8-group): shared loads
        // only.  Otherwise inactive threads take zeros and the tail group is read from global memory.
        auto take = [&](bool whole, int cnt, int q0, uint32_t (&w)[4 * TT_NPS]) {
          if (live && !mbar_wait_bounded(smem_u32(&full[sp.slot]), sp.phase, p.timeout_ns, s_abort)) {
            if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
            *s_abort = 1;
            live = false;
          }
          const unsigned char* src_s = stages + sp.slot * SBY + 2 * TT_EPT * tid;
          if (whole) {
#pragma unroll
            for (int hh = 0; hh < NPS; ++hh) {
              if (hh < cnt) {
                const uint4 v = *reinterpret_cast<const uint4*>(src_s + hh * TT_IN_BYTES);
                w[4 * hh + 0] = v.x; w[4 * hh + 1] = v.y; w[4 * hh + 2] = v.z; w[4 * hh + 3] = v.w;
              }
            }
          } else {
#pragma unroll
            for (int u = 0; u < 4 * NPS; ++u) w[u] = 0u;
            if (active && live) {
#pragma unroll
              for (int hh = 0; hh < NPS; ++hh) {
                if (hh < cnt) {
                  if (!tailgrp) {
                    const uint4 v = *reinterpret_cast<const uint4*>(src_s + hh * TT_IN_BYTES);
                    w[4 * hh + 0] = v.x; w[4 * hh + 1] = v.y; w[4 * hh + 2] = v.z; w[4 * hh + 3] = v.w;
                  } else {
                    const uint16_t* src = p.g[q0 + hh];
#pragma unroll
                    for (int u = 0; u < TT_EPT; ++u) {
                      const uint32_t b = (e0 + u < psi) ? (uint32_t)src[e0 + u] : 0u;
                      w[4 * hh + (u >> 1)] |= (u & 1) ? (b << 16) : b;
                    }
                  }
                }
              }
            }
          }
          // The slot is refilled by the async proxy: order this thread's reads of it before that write.
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&empty[sp.slot]));
          sp.next();
        };

        // Inputs in rank order, each rank's micro-steps summed before it joins the tree, NPS to a stage (the
        // last stage takes the remaining nin mod NPS).
        Part8 slot[LEVELS], cur;
        const bool whole_half = x.hi - x.lo == TT_SUB && x.hi <= p8;
        int r = 0, k = 0, q = 0;
        constexpr int H1 = NPS > 1 ? 1 : 0, H2 = NPS > 2 ? 2 : 0, H3 = NPS > 3 ? 3 : 0;
        while (q < nin) {
          const int cnt = nin - q < NPS ? nin - q : NPS;
          uint32_t w[4 * NPS];
          take(whole_half, cnt, q, w);
          tree_fold<LEVELS, 0>(slot, cur, w, r, k == 0, k == a - 1);
          if (++k == a) { k = 0; ++r; }
          if (NPS > 1 && cnt > 1) {
            tree_fold<LEVELS, H1>(slot, cur, w, r, k == 0, k == a - 1);
            if (++k == a) { k = 0; ++r; }
          }
          if (NPS > 2 && cnt > 2) {
            tree_fold<LEVELS, H2>(slot, cur, w, r, k == 0, k == a - 1);
            if (++k == a) { k = 0; ++r; }
          }
          if (NPS > 3 && cnt > 3) {
            tree_fold<LEVELS, H3>(slot, cur, w, r, k == 0, k == a - 1);
            if (++k == a) { k = 0; ++r; }
          }
          q += cnt;
        }

        // n = 2^LEVELS: the last rank completed the whole block and cur holds the total.  Otherwise the blocks
        // left without a partner join, smallest first, each the one below it on the left.
        Part8 tot = cur;
        if (n != (1 << LEVELS)) {
          bool have = false;
#pragma unroll
          for (int lv = 0; lv < LEVELS; ++lv) {
            if ((n >> lv) & 1) {
              tot = have ? tree_add(slot[lv], tot) : slot[lv];
              have = true;
            }
          }
        }
        float o[TT_EPT];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          f2_unpack(f2_mul(tot.h[u], inv2), o[2 * u], o[2 * u + 1]);
        }
        if (active) {
          float* dst = p.gbar[t.owner] + (t.loff + (e0 - t.goff));
          const bool all = e0 >= x.lo && e0 + TT_EPT <= x.hi;
          if (all && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
            *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<float4*>(dst + 4) = make_float4(o[4], o[5], o[6], o[7]);
#pragma unroll
            for (int u = 0; u < TT_EPT; ++u) bad += nonfinite(o[u]);
          } else {
#pragma unroll
            for (int u = 0; u < TT_EPT; ++u)
              if (e0 + u >= x.lo && e0 + u < x.hi) {
                dst[u] = o[u];
                bad += nonfinite(o[u]);
              }
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ CTA total, then the grid's
  unsigned long long c = bad;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
  __syncthreads();
  if (lane == 0 && c) atomicAdd(s_count, c);
  __syncthreads();
  if (tid == 0)
    finish_reduction(p.state, *s_count, (*s_count != 0ull) || *s_abort, p.advance, p.beta1, p.beta2, &p.scaler, 0,
                     p.merge);
}

// ---------------------------------------------------------------- compensated: rank-major stages
//
// reduce_tree_rm_kernel: the compensated tree for a compile-time rank count N.  The ranks go in groups of at
// most eight: [0, min(N, 8)) and, for N > 8, [8, N).  A stage holds micro-step k of every rank of a group for
// one sub-tile (one bulk copy per rank on one barrier, issued by as many producer lanes).  Each consumer
// thread carries the group's (hi, lo) leaf sums of its EPT elements across the micro-steps -- NG * EPT / 2
// independent packed lanes -- and after the last micro-step adds them up the group's binomial tree level by
// level, every merge fixed at compile time.  For N > 8 the two groups' totals then merge once, block [0, 8) on
// the left: the binomial tree restricted to ranks [8, N) is the tree of N - 8 ranks shifted by 8 (levels 0-2
// pair ranks only inside aligned blocks of eight), and its level 3 is that one merge.  Each leaf is the same
// chain and each merge the same operation on the same operands as in the tree's definition, so the result is
// the same bits.  EPT = 16, 8, 4 for groups of <= 2, <= 4, <= 8 ranks: a stage is 30 KB or less, and the leaves
// take 64 registers a thread at most.
constexpr int RM_MAX_STAGES = 12;
constexpr int RM_GROUP = 8;
template <int N>
__host__ __device__ constexpr int rm_g1() { return N < RM_GROUP ? N : RM_GROUP; }   // ranks of the first group
template <int N>
__host__ __device__ constexpr int rm_ept() { return rm_g1<N>() <= 2 ? 16 : (rm_g1<N>() <= 4 ? 8 : 4); }
template <int N>
__host__ __device__ constexpr int rm_sub() { return TT_CTHREADS * rm_ept<N>(); }      // elements of a sub-tile
template <int N>
__host__ __device__ constexpr int rm_in_bytes() { return 2 * rm_sub<N>(); }         // one input's sub-tile
template <int N>
__host__ __device__ constexpr int rm_stage_bytes() { return rm_g1<N>() * rm_in_bytes<N>(); }
template <int N>
__host__ __device__ constexpr int rm_stages() {
  return TT_RING_BYTES / rm_stage_bytes<N>() < RM_MAX_STAGES ? TT_RING_BYTES / rm_stage_bytes<N>() : RM_MAX_STAGES;
}
static_assert(RM_MAX_STAGES <= TT_MAX_STAGES, "the barriers fit the shared layout");
static_assert(TILE % rm_sub<8>() == 0 && TILE % rm_sub<4>() == 0 && TILE % rm_sub<2>() == 0,
              "a tile is a whole number of sub-tiles");
static_assert(rm_sub<8>() % 8 == 0 && rm_in_bytes<8>() % 16 == 0, "sub-tiles start on 16-byte boundaries");
static_assert(rm_stages<16>() >= 4 && rm_stages<8>() >= 4 && rm_stages<7>() >= 4, "at least four stages in flight");
static_assert(DP_MAX_N <= 2 * RM_GROUP, "two groups cover every rank count");

// The range of sub-tile h (SUB elements) of a tile, copied as the 8-aligned hull (as half_of).
__device__ __forceinline__ Half sub_of(const Tile& t, int h, int sub) {
  const int64_t cb = (t.start / TILE) * TILE + (int64_t)h * sub;
  Half x;
  x.lo = t.start > cb ? t.start : cb;
  x.hi = t.end < cb + sub ? t.end : cb + sub;
  x.sa = x.lo & ~int64_t(7);
  return x;
}

// EPT bf16 (EPT / 2 words) from shared memory: one 8- or 16-byte load, or two 16-byte loads.
template <int EPT>
__device__ __forceinline__ void rm_load(const unsigned char* s, uint32_t (&w)[EPT / 2]) {
  if constexpr (EPT == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(s);
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int c = 0; c < EPT / 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(s + 16 * c);
      w[4 * c + 0] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
    }
  }
}

// One micro-step of every rank of a group into its leaves: the first sets (h, l) = (x, 0), later ones
// (h, e) = TwoSum(h, x), l = l + e.
template <int NG, int W, bool FIRST>
__device__ __forceinline__ void rm_fold(f2_t (&h)[NG][W], f2_t (&l)[NG][W], const uint32_t (&w)[NG][W]) {
#pragma unroll
  for (int r = 0; r < NG; ++r)
#pragma unroll
    for (int u = 0; u < W; ++u) {
      const f2_t x = bf16x2_to_f2(w[r][u]);
      if (FIRST) {
        h[r][u] = x;
        l[r][u] = 0ull;
      } else {
        f2_t e;
        h[r][u] = f2_two_sum(h[r][u], x, e);
        l[r][u] = f2_add(l[r][u], e);
      }
    }
}

// left + right on W packed lanes, the lower-index block on the left: (H, e) = TwoSum(H_left, H_right),
// L = (L_left + e) + L_right.
template <int W>
__device__ __forceinline__ void rm_merge(f2_t (&hl)[W], f2_t (&ll)[W], const f2_t (&hr)[W], const f2_t (&lr)[W]) {
#pragma unroll
  for (int u = 0; u < W; ++u) {
    f2_t e;
    const f2_t H = f2_two_sum(hl[u], hr[u], e);
    ll[u] = f2_add(f2_add(ll[u], e), lr[u]);
    hl[u] = H;
  }
}

// One level of the binomial tree over a group's leaves: block r (a multiple of 2 STEP) takes block r + STEP on
// its right; a block with no partner stays.
template <int NG, int W, int STEP>
__device__ __forceinline__ void rm_level(f2_t (&h)[NG][W], f2_t (&l)[NG][W]) {
#pragma unroll
  for (int r = 0; r + STEP < NG; r += 2 * STEP) rm_merge<W>(h[r], l[r], h[r + STEP], l[r + STEP]);
}
// The group's whole tree, levels 0, 1, 2 in turn; the total is left in leaf 0.
template <int NG, int W>
__device__ __forceinline__ void rm_tree(f2_t (&h)[NG][W], f2_t (&l)[NG][W]) {
  static_assert(NG <= RM_GROUP, "a group has at most eight ranks");
  if constexpr (NG > 1) rm_level<NG, W, 1>(h, l);
  if constexpr (NG > 2) rm_level<NG, W, 2>(h, l);
  if constexpr (NG > 4) rm_level<NG, W, 4>(h, l);
}

template <int MAXSEG, int N>
__global__ void __launch_bounds__(TT_THREADS, 1) reduce_tree_rm_kernel(const __grid_constant__ TreeParams<MAXSEG> p) {
  constexpr int G1 = rm_g1<N>();               // ranks [0, G1)
  constexpr int G2 = N - G1;                   // ranks [8, N), none for N <= 8
  // Micro-steps of the second group a stage carries: 8 / G2 when that group has one or two ranks (n = 9, 10),
  // so its stages still carry up to eight copies; one otherwise (packing larger groups spilled registers).
  constexpr int PK = (G2 > 0 && G2 <= 2) ? RM_GROUP / G2 : 1;
  constexpr int G2A = G2 > 0 ? G2 : 1;             // its array extent
  constexpr int EPT = rm_ept<N>();
  constexpr int W = EPT / 2;
  constexpr int SUB = rm_sub<N>();
  constexpr int IN = rm_in_bytes<N>();
  constexpr int SBY = rm_stage_bytes<N>();
  constexpr int NST = rm_stages<N>();
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TT_RING_BYTES);
  uint64_t* empty = full + NST;
  volatile int* s_abort = reinterpret_cast<volatile int*>(empty + NST);
  unsigned long long* s_count = reinterpret_cast<unsigned long long*>(empty + NST + 1);
  __shared__ float s_inv;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int a = p.a;
  const int ntiles = p.seg.ntiles;
  const int64_t psi = p.seg.psi;
  const int64_t p8 = psi & ~int64_t(7);

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), TT_CWARPS);
    }
    *s_abort = 0;
    *s_count = 0ull;
    float inv = p.inv;
    if (p.scaler.enabled) {
      // fl32(1 / (n S)) from the device-resident scale, as for the ring order.
      const float sc = *reinterpret_cast<volatile const float*>(&p.state->loss_scale);
      inv = (float)(1.0 / ((double)p.n * (double)sc));
      if (!(sc > 0.0f) || nonfinite(sc) || !(inv >= 1.17549435e-38f) || nonfinite(inv)) {
        record_error(p.state, DP_ERR_INVALID_ARG);
        *s_abort = 1;
        inv = 0.0f;
      }
    }
    s_inv = inv;
    fence_mbar_init();
  }
  __syncthreads();

  unsigned bad = 0;
  if (warp == TT_CWARPS) {
    // ------------------------------------------------------------ producer warp: per sub-tile and group, micro-step
    // k of the group's ranks.  Lane 0 waits for the slot and posts the byte count; lane r then copies rank r.
    StagePos<NST> sp;
    TileWalker<MAXSEG> walk;
    bool stop = false;
    for (int tile = blockIdx.x; tile < ntiles && !stop; tile += gridDim.x) {
      const Tile t = walk.at(p.seg, tile);
      for (int h = 0; h < TILE / SUB && !stop; ++h) {
        const Half x = sub_of(t, h, SUB);
        if (x.empty()) continue;
        int64_t sb = (x.hi + 7) & ~int64_t(7);
        if (sb > p8) sb = p8;
        const uint32_t bytes = sb > x.sa ? (uint32_t)(sb - x.sa) * 2u : 0u;
        // The first group one micro-step a stage; the second PK micro-steps a stage, input l of the stage being
        // rank 8 + l % G2 at micro-step k + l / G2.
        for (int gq = 0; gq < (G2 > 0 ? 2 : 1) && !stop; ++gq) {
          const int r0 = gq ? RM_GROUP : 0, ng = gq ? G2 : G1, pk = gq ? PK : 1;
          for (int k = 0; k < a; k += pk) {
            const int cnt = a - k < pk ? a - k : pk;
            const int ncp = ng * cnt;
            const uint32_t fb = smem_u32(&full[sp.slot]);
            int ok = 1;
            if (lane == 0) {
              if (*s_abort) {
                ok = 0;
              } else if (sp.count >= (uint32_t)NST &&
                         !mbar_wait_bounded(smem_u32(&empty[sp.slot]), sp.phase ^ 1u, p.timeout_ns, s_abort)) {
                if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
                *s_abort = 1;
                ok = 0;
              }
              if (ok) mbar_arrive_expect_tx(fb, bytes * (uint32_t)ncp);
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            __syncwarp();
            if (!ok) {
              stop = true;
              break;
            }
            if (bytes && lane < ncp)
              bulk_g2s(smem_u32(stages + sp.slot * SBY + lane * IN),
                       p.g[(r0 + lane % ng) * a + k + lane / ng] + x.sa, bytes, fb);
            sp.next();
          }
        }
      }
    }
    // Never leave with copies in flight: wait for the newest issued phase of every slot.
    if (lane == 0 && *s_abort) {
      const uint32_t it = sp.count;
      const uint32_t first = it > (uint32_t)NST ? it - NST : 0u;
      for (uint32_t y = first; y < it; ++y)
        (void)mbar_wait_bounded(smem_u32(&full[y % NST]), (y / NST) & 1u, p.timeout_ns, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers: EPT elements of every rank per thread
    const f2_t inv2 = f2_pack(s_inv, s_inv);
    StagePos<NST> sp;
    TileWalker<MAXSEG> walk;
    bool live = true;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const Tile t = walk.at(p.seg, tile);
      for (int h = 0; h < TILE / SUB; ++h) {
        const Half x = sub_of(t, h, SUB);
        if (x.empty()) continue;
        const int64_t e0 = x.sa + EPT * tid;
        const bool active = e0 < x.hi;
        const bool tailgrp = active && (e0 + EPT > p8);

        // One stage (micro-step k of the group from rank r0): wait for its bytes, take this thread's EPT values
        // of each rank, release the slot.  WHOLE (a whole sub-tile below the buffer's last partial 8-group):
        // shared loads only.  Otherwise inactive threads take zeros and the tail group is read from global.
        auto take = [&](auto whole_tag, int r0, int k, auto& w) {
          constexpr bool WHOLE = decltype(whole_tag)::value;
          constexpr int NG = sizeof(w) / sizeof(w[0]);
          if (live && !mbar_wait_bounded(smem_u32(&full[sp.slot]), sp.phase, p.timeout_ns, s_abort)) {
            if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
            *s_abort = 1;
            live = false;
          }
          const unsigned char* src_s = stages + sp.slot * SBY + 2 * EPT * tid;
          if constexpr (WHOLE) {
#pragma unroll
            for (int r = 0; r < NG; ++r) rm_load<EPT>(src_s + r * IN, w[r]);
          } else {
#pragma unroll
            for (int r = 0; r < NG; ++r)
#pragma unroll
              for (int u = 0; u < W; ++u) w[r][u] = 0u;
            if (active && live) {
#pragma unroll
              for (int r = 0; r < NG; ++r) {
                if (!tailgrp) {
                  rm_load<EPT>(src_s + r * IN, w[r]);
                } else {
                  const uint16_t* src = p.g[(r0 + r) * a + k];
#pragma unroll
                  for (int u = 0; u < EPT; ++u) {
                    const uint32_t b = (e0 + u < psi) ? (uint32_t)src[e0 + u] : 0u;
                    w[r][u >> 1] |= (u & 1) ? (b << 16) : b;
                  }
                }
              }
            }
          }
          // The slot is refilled by the async proxy: order this thread's reads of it before that write.
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&empty[sp.slot]));
          sp.next();
        };

        // A group's leaves over the micro-steps (whole: the sub-tile takes the guard-free loads), then its tree;
        // for N > 8 the second group's total joins the first's on the right.  The total is left in leaf 0.
        auto fold_group = [&](auto whole_tag, int r0, auto& hs, auto& ls) {
          constexpr int NG = sizeof(hs) / sizeof(hs[0]);
          {
            uint32_t w[NG][W];
            take(whole_tag, r0, 0, w);
            rm_fold<NG, W, true>(hs, ls, w);
          }
          for (int k = 1; k < a; ++k) {
            uint32_t w[NG][W];
            take(whole_tag, r0, k, w);
            rm_fold<NG, W, false>(hs, ls, w);
          }
        };
        // The second group when packed: a stage holds micro-steps k .. k + cnt - 1 (cnt <= PK) of its G2 ranks,
        // folded into the leaves in micro-step order.
        auto take_packed = [&](auto whole_tag, int k, int cnt, auto& w) {
          constexpr bool WHOLE = decltype(whole_tag)::value;
          if (live && !mbar_wait_bounded(smem_u32(&full[sp.slot]), sp.phase, p.timeout_ns, s_abort)) {
            if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
            *s_abort = 1;
            live = false;
          }
          const unsigned char* src_s = stages + sp.slot * SBY + 2 * EPT * tid;
          if constexpr (WHOLE) {
#pragma unroll
            for (int kk = 0; kk < PK; ++kk)
#pragma unroll
              for (int r = 0; r < G2; ++r) rm_load<EPT>(src_s + (kk * G2 + r) * IN, w[kk][r]);
          } else {
#pragma unroll
            for (int kk = 0; kk < PK; ++kk)
#pragma unroll
              for (int r = 0; r < G2; ++r)
#pragma unroll
                for (int u = 0; u < W; ++u) w[kk][r][u] = 0u;
            if (active && live) {
#pragma unroll
              for (int kk = 0; kk < PK; ++kk) {
                if (kk < cnt) {
#pragma unroll
                  for (int r = 0; r < G2; ++r) {
                    if (!tailgrp) {
                      rm_load<EPT>(src_s + (kk * G2 + r) * IN, w[kk][r]);
                    } else {
                      const uint16_t* src = p.g[(RM_GROUP + r) * a + k + kk];
#pragma unroll
                      for (int u = 0; u < EPT; ++u) {
                        const uint32_t b = (e0 + u < psi) ? (uint32_t)src[e0 + u] : 0u;
                        w[kk][r][u >> 1] |= (u & 1) ? (b << 16) : b;
                      }
                    }
                  }
                }
              }
            }
          }
          // The slot is refilled by the async proxy: order this thread's reads of it before that write.
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&empty[sp.slot]));
          sp.next();
        };
        auto fold_packed = [&](auto whole_tag, auto& hs, auto& ls) {
          for (int k = 0; k < a; k += PK) {
            const int cnt = a - k < PK ? a - k : PK;
            uint32_t w[PK][G2A][W];
            take_packed(whole_tag, k, cnt, w);
            if (k == 0) rm_fold<G2, W, true>(hs, ls, w[0]);
            else rm_fold<G2, W, false>(hs, ls, w[0]);
#pragma unroll
            for (int kk = 1; kk < PK; ++kk)
              if (kk < cnt) rm_fold<G2, W, false>(hs, ls, w[kk]);
          }
        };
        const bool whole = x.hi - x.lo == SUB && x.hi <= p8;
        f2_t hs[G1][W], ls[G1][W];
        if (whole) fold_group(std::true_type{}, 0, hs, ls);
        else fold_group(std::false_type{}, 0, hs, ls);
        rm_tree<G1, W>(hs, ls);
        if constexpr (G2 > 0) {
          f2_t hs2[G2][W], ls2[G2][W];
          if constexpr (PK > 1) {
            if (whole) fold_packed(std::true_type{}, hs2, ls2);
            else fold_packed(std::false_type{}, hs2, ls2);
          } else {
            if (whole) fold_group(std::true_type{}, RM_GROUP, hs2, ls2);
            else fold_group(std::false_type{}, RM_GROUP, hs2, ls2);
          }
          rm_tree<G2, W>(hs2, ls2);
          rm_merge<W>(hs[0], ls[0], hs2[0], ls2[0]);
        }

        float o[EPT];
#pragma unroll
        for (int u = 0; u < W; ++u) f2_unpack(f2_mul(f2_add(hs[0][u], ls[0][u]), inv2), o[2 * u], o[2 * u + 1]);
        if (active) {
          float* dst = p.gbar[t.owner] + (t.loff + (e0 - t.goff));
          const bool all = e0 >= x.lo && e0 + EPT <= x.hi;
          if (all && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
#pragma unroll
            for (int c = 0; c < EPT / 4; ++c)
              *reinterpret_cast<float4*>(dst + 4 * c) = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
#pragma unroll
            for (int u = 0; u < EPT; ++u) bad += nonfinite(o[u]);
          } else {
#pragma unroll
            for (int u = 0; u < EPT; ++u)
              if (e0 + u >= x.lo && e0 + u < x.hi) {
                dst[u] = o[u];
                bad += nonfinite(o[u]);
              }
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ CTA total, then the grid's
  unsigned long long c = bad;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
  __syncthreads();
  if (lane == 0 && c) atomicAdd(s_count, c);
  __syncthreads();
  if (tid == 0)
    finish_reduction(p.state, *s_count, (*s_count != 0ull) || *s_abort, p.advance, p.beta1, p.beta2, &p.scaler, 0,
                     p.merge);
}

// ---------------------------------------------------------------- staged: the tree over per-rank accumulators

template <int MAXSEG>
struct RsTreeParams {
  const float* acc[DP_MAX_N];
  float* gbar[DP_MAX_N];
  dp_step_state_t* state;
  float inv;
  int32_t n, merge;
  SegTable<MAXSEG> seg;
};

// One element's partial sum: hi and (compensated) its accumulated rounding errors.
struct Part1 {
  float h, l;
};

template <bool COMP>
__device__ __forceinline__ Part1 tree_add1(Part1 x, Part1 y) {
  Part1 z;
  if (COMP) {
    float err;
    z.h = two_sum(x.h, y.h, err);
    z.l = __fadd_rn(__fadd_rn(x.l, err), y.l);
  } else {
    z.h = __fadd_rn(x.h, y.h);
    z.l = 0.0f;
  }
  return z;
}

template <int MAXSEG, bool COMP>
__global__ void __launch_bounds__(256) rs_tree_kernel(const __grid_constant__ RsTreeParams<MAXSEG> p) {
  __shared__ unsigned long long s_count;
  if (threadIdx.x == 0) s_count = 0ull;
  __syncthreads();
  unsigned bad = 0;
  const int n = p.n;
  for (int tile = blockIdx.x; tile < p.seg.ntiles; tile += gridDim.x) {
    const Tile t = tile_at(p.seg, tile);
    float* dst = p.gbar[t.owner];
    for (int64_t e = t.start + threadIdx.x; e < t.end; e += blockDim.x) {
      Part1 slot[RT_LEVELS];
      for (int r = 0; r < n; ++r) {
        Part1 v;
        if (COMP) {
          const float2 hl = reinterpret_cast<const float2*>(p.acc[r])[e];
          v = Part1{hl.x, hl.y};
        } else {
          v = Part1{p.acc[r][e], 0.0f};
        }
        const int top = __ffs(~r) - 1;
#pragma unroll
        for (int lv = 0; lv < RT_LEVELS; ++lv) {
          if (lv < top) v = tree_add1<COMP>(slot[lv], v);
          else if (lv == top) slot[lv] = v;
        }
      }
      Part1 tot{0.0f, 0.0f};
      bool have = false;
#pragma unroll
      for (int lv = 0; lv < RT_LEVELS; ++lv) {
        if ((n >> lv) & 1) {
          tot = have ? tree_add1<COMP>(slot[lv], tot) : slot[lv];
          have = true;
        }
      }
      const float pp = COMP ? __fadd_rn(tot.h, tot.l) : tot.h;
      const float g = __fmul_rn(pp, p.inv);
      dst[t.loff + (e - t.goff)] = g;
      if (nonfinite(g)) ++bad;
    }
  }
  unsigned long long c = bad;
  for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
  if ((threadIdx.x & 31) == 0 && c) atomicAdd(&s_count, c);
  __syncthreads();
  if (threadIdx.x == 0) finish_reduction(p.state, s_count, s_count != 0ull, 0, 1.0, 1.0, nullptr, 0, p.merge);
}

// ---------------------------------------------------------------- launchers

template <int MAXSEG>
TreeParams<MAXSEG> tree_params(const Plan& P, const uint16_t* const* g, int a, float* const* gbar,
                               const StepScalars& s, int advance, dp_step_state_t* st) {
  TreeParams<MAXSEG> prm;
  for (int q = 0; q < P.n * a; ++q) prm.g[q] = g[q];
  for (int r = 0; r < P.n; ++r) prm.gbar[r] = gbar[r];
  prm.state = st;
  prm.timeout_ns = s.timeout_ns;
  prm.beta1 = (double)s.beta1;
  prm.beta2 = (double)s.beta2;
  prm.inv = s.inv;
  prm.n = P.n;
  prm.a = a;
  prm.advance = advance;
  prm.merge = s.merge;
  prm.scaler = s.scaler;
  fill_seg(prm.seg, P);
  return prm;
}

template <auto KERN, int MAXSEG>
cudaError_t launch_tree_kernel(const TreeParams<MAXSEG>& prm, int ntiles, cudaStream_t stream) {
  // The opt-in shared-memory size is set once per device (not inside a stream capture on later calls).
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize, TT_SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  // One CTA per SM (every CTA joins the grid-wide finish, so at least one runs even with no tiles).
  KERN<<<occupancy_grid(KERN, TT_THREADS, TT_SMEM, ntiles), TT_THREADS, TT_SMEM, stream>>>(prm);
  return cudaGetLastError();
}

// Compensated: the rank-major kernel for that n.  Plain: the binary counter.
template <int MAXSEG, bool COMP>
cudaError_t launch_tree_n(const Plan& P, const uint16_t* const* g, int a, float* const* gbar,
                          const StepScalars& s, int advance, dp_step_state_t* st, cudaStream_t stream) {
  const TreeParams<MAXSEG> prm = tree_params<MAXSEG>(P, g, a, gbar, s, advance, st);
  if constexpr (COMP) {
    switch (P.n) {
      case 1: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 1>, MAXSEG>(prm, P.ntiles, stream);
      case 2: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 2>, MAXSEG>(prm, P.ntiles, stream);
      case 3: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 3>, MAXSEG>(prm, P.ntiles, stream);
      case 4: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 4>, MAXSEG>(prm, P.ntiles, stream);
      case 5: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 5>, MAXSEG>(prm, P.ntiles, stream);
      case 6: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 6>, MAXSEG>(prm, P.ntiles, stream);
      case 7: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 7>, MAXSEG>(prm, P.ntiles, stream);
      case 8: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 8>, MAXSEG>(prm, P.ntiles, stream);
      case 9: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 9>, MAXSEG>(prm, P.ntiles, stream);
      case 10: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 10>, MAXSEG>(prm, P.ntiles, stream);
      case 11: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 11>, MAXSEG>(prm, P.ntiles, stream);
      case 12: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 12>, MAXSEG>(prm, P.ntiles, stream);
      case 13: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 13>, MAXSEG>(prm, P.ntiles, stream);
      case 14: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 14>, MAXSEG>(prm, P.ntiles, stream);
      case 15: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 15>, MAXSEG>(prm, P.ntiles, stream);
      case 16: return launch_tree_kernel<reduce_tree_rm_kernel<MAXSEG, 16>, MAXSEG>(prm, P.ntiles, stream);
      default: return cudaErrorInvalidValue;
    }
  } else {
    if (P.n <= 8) return launch_tree_kernel<reduce_tree_kernel<MAXSEG, 3>, MAXSEG>(prm, P.ntiles, stream);
    return launch_tree_kernel<reduce_tree_kernel<MAXSEG, 4>, MAXSEG>(prm, P.ntiles, stream);
  }
}

template <int MAXSEG, bool COMP>
cudaError_t launch_rs_tree_t(const Plan& P, const float* const* acc, float* const* gbar, const StepScalars& s,
                             dp_step_state_t* st, cudaStream_t stream) {
  RsTreeParams<MAXSEG> prm;
  for (int r = 0; r < P.n; ++r) {
    prm.acc[r] = acc[r];
    prm.gbar[r] = gbar[r];
  }
  prm.state = st;
  prm.inv = s.inv;
  prm.n = P.n;
  prm.merge = s.merge;
  fill_seg(prm.seg, P);
  auto kern = rs_tree_kernel<MAXSEG, COMP>;
  kern<<<occupancy_grid(kern, 256, 0, P.ntiles), 256, 0, stream>>>(prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_reduce_tree(const Plan& P0, const uint16_t* const* g, int a, float* const* gbar,
                               const StepScalars& s0, int advance0, dp_step_state_t* st, cudaStream_t stream,
                               uint64_t* launches) {
  return for_each_chunk(P0, s0, [&](const Plan& P, const StepScalars& s, bool last) {
    ++*launches;
    const int advance = (advance0 && last) ? 1 : 0;
    const bool comp = s.mode == DP_SUM_COMPENSATED;
    if (P.nseg <= SMALL_SEG)
      return comp ? launch_tree_n<SMALL_SEG, true>(P, g, a, gbar, s, advance, st, stream)
                  : launch_tree_n<SMALL_SEG, false>(P, g, a, gbar, s, advance, st, stream);
    return comp ? launch_tree_n<BIG_SEG, true>(P, g, a, gbar, s, advance, st, stream)
                : launch_tree_n<BIG_SEG, false>(P, g, a, gbar, s, advance, st, stream);
  });
}

cudaError_t launch_rs_tree(const Plan& P0, const float* const* acc, float* const* gbar, const StepScalars& s0,
                           dp_step_state_t* st, cudaStream_t stream, uint64_t* launches) {
  return for_each_chunk(P0, s0, [&](const Plan& P, const StepScalars& s, bool) {
    ++*launches;
    const bool comp = s.mode == DP_SUM_COMPENSATED;
    if (P.nseg <= SMALL_SEG)
      return comp ? launch_rs_tree_t<SMALL_SEG, true>(P, acc, gbar, s, st, stream)
                  : launch_rs_tree_t<SMALL_SEG, false>(P, acc, gbar, s, st, stream);
    return comp ? launch_rs_tree_t<BIG_SEG, true>(P, acc, gbar, s, st, stream)
                : launch_rs_tree_t<BIG_SEG, false>(P, acc, gbar, s, st, stream);
  });
}

}  // namespace dp
