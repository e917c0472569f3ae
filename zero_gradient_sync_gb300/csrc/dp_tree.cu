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
// reduce_tree_kernel: each thread reduces 4 consecutive elements of all n*a inputs and keeps the tree as a
// binary counter: slot l holds the pending sum of a complete block of 2^l ranks, so at most log2(n) + 1
// partial sums are live, each in registers.  The ring kernel's shared-memory pipeline cannot hold these
// partials at 16 elements a thread, so this kernel streams with plain 8-byte loads, 8 in flight per thread.
// rs_tree_kernel: the same tree over the staged per-rank accumulators, one element per thread.
#include "dp_device.cuh"
#include "dp_internal.h"

namespace dp {
namespace {

constexpr int RT_THREADS = 256;
constexpr int RT_DEPTH = 8;   // input loads in flight per thread
constexpr int RT_LEVELS = 5;  // slots for n <= 16 = 2^4: levels 0..4

template <int MAXSEG>
struct TreeParams {
  const uint16_t* g[DP_MAX_NA];
  float* gbar[DP_MAX_N];
  dp_step_state_t* state;
  double beta1, beta2;
  float inv;
  int32_t n, a, advance;
  ScalerK scaler;
  SegTable<MAXSEG> seg;
};

// Four elements' partial sum: packed hi pairs and (compensated) their accumulated rounding errors.
struct Part4 {
  f2_t h[2], l[2];
};

// left + right, left being the lower-index block: (H, e) = TwoSum(left.H, right.H), L = (left.L + e) + right.L.
template <bool COMP>
__device__ __forceinline__ Part4 tree_add(const Part4& x, const Part4& y) {
  Part4 z;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    if (COMP) {
      f2_t e;
      z.h[u] = f2_two_sum(x.h[u], y.h[u], e);
      z.l[u] = f2_add(f2_add(x.l[u], e), y.l[u]);
    } else {
      z.h[u] = f2_add(x.h[u], y.h[u]);
      z.l[u] = 0ull;
    }
  }
  return z;
}

// Quad [e, e + 4) of one bf16 input as 4 bf16 in two words; elements at or past psi read as +0.
__device__ __forceinline__ uint2 load_quad(const uint16_t* src, int64_t e, int64_t psi) {
  if (e + 4 <= psi) return __ldcs(reinterpret_cast<const uint2*>(src + e));
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (e + u < psi) w[u >> 1] |= (uint32_t)src[e + u] << (16 * (u & 1));
  return make_uint2(w[0], w[1]);
}

template <int MAXSEG, bool COMP>
__global__ void __launch_bounds__(RT_THREADS) reduce_tree_kernel(const __grid_constant__ TreeParams<MAXSEG> p) {
  __shared__ unsigned long long s_count;
  __shared__ float s_inv;
  __shared__ int s_bad_scale;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_count = 0ull;
    float inv = p.inv;
    int bad = 0;
    if (p.scaler.enabled) {
      // fl32(1 / (n S)) from the device-resident scale, as for the ring order.
      const float sc = *reinterpret_cast<volatile const float*>(&p.state->loss_scale);
      inv = (float)(1.0 / ((double)p.n * (double)sc));
      if (!(sc > 0.0f) || nonfinite(sc) || !(inv >= 1.17549435e-38f) || nonfinite(inv)) {
        record_error(p.state, DP_ERR_INVALID_ARG);
        bad = 1;
        inv = 0.0f;
      }
    }
    s_inv = inv;
    s_bad_scale = bad;
  }
  __syncthreads();
  const int n = p.n, a = p.a, na = n * a;
  const int64_t psi = p.seg.psi;
  const f2_t inv2 = f2_pack(s_inv, s_inv);
  unsigned bad = 0;
  TileWalker<MAXSEG> walk;
  for (int tile = s_bad_scale ? p.seg.ntiles : blockIdx.x; tile < p.seg.ntiles; tile += gridDim.x) {
    const Tile t = walk.at(p.seg, tile);
    const int64_t A = t.start & ~int64_t(3), B = (t.end + 3) & ~int64_t(3);
    float* const dst = p.gbar[t.owner] + (t.loff - t.goff);
    for (int64_t e = A + 4 * (int64_t)tid; e < B; e += 4 * RT_THREADS) {
      uint2 buf[RT_DEPTH];
#pragma unroll
      for (int u = 0; u < RT_DEPTH; ++u)
        if (u < na) buf[u] = load_quad(p.g[u], e, psi);
      Part4 slot[RT_LEVELS], cur;
      int r = 0, k = 0;
      for (int q0 = 0; q0 < na; q0 += RT_DEPTH) {
#pragma unroll
        for (int u = 0; u < RT_DEPTH; ++u) {
          const int q = q0 + u;
          if (q < na) {
            const uint2 w = buf[u];
            if (q + RT_DEPTH < na) buf[u] = load_quad(p.g[q + RT_DEPTH], e, psi);
            const f2_t x0 = bf16x2_to_f2(w.x), x1 = bf16x2_to_f2(w.y);
            if (k == 0) {
              cur.h[0] = x0;
              cur.h[1] = x1;
              cur.l[0] = cur.l[1] = 0ull;
            } else if (COMP) {
              f2_t e0, e1;
              cur.h[0] = f2_fast_two_sum(cur.h[0], x0, e0);
              cur.h[1] = f2_fast_two_sum(cur.h[1], x1, e1);
              cur.l[0] = f2_add(cur.l[0], e0);
              cur.l[1] = f2_add(cur.l[1], e1);
            } else {
              cur.h[0] = f2_add(cur.h[0], x0);
              cur.h[1] = f2_add(cur.h[1], x1);
            }
            if (++k == a) {
              // Rank r is complete: add it into the counter.  Bit l of r marks an occupied slot l, which
              // holds the block just below it; merging carries the sum up until a free slot takes it.
              // The slots below the lowest clear bit of r are all occupied and merge; that bit's slot takes
              // the sum (static slot indices keep every slot in registers).
              const int top = __ffs(~r) - 1;
              Part4 v = cur;
#pragma unroll
              for (int lv = 0; lv < RT_LEVELS; ++lv) {
                if (lv < top) v = tree_add<COMP>(slot[lv], v);
                else if (lv == top) slot[lv] = v;
              }
              k = 0;
              ++r;
            }
          }
        }
      }
      // Blocks left without a partner, smallest first, each joining the one below it on the left.
      Part4 tot = cur;
      bool have = false;
#pragma unroll
      for (int lv = 0; lv < RT_LEVELS; ++lv) {
        if ((n >> lv) & 1) {
          tot = have ? tree_add<COMP>(slot[lv], tot) : slot[lv];
          have = true;
        }
      }
      float o[4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const f2_t pp = COMP ? f2_add(tot.h[u], tot.l[u]) : tot.h[u];
        f2_unpack(f2_mul(pp, inv2), o[2 * u], o[2 * u + 1]);
      }
      const bool whole = e >= t.start && e + 4 <= t.end;
      float* d = dst + e;
      if (whole && ((reinterpret_cast<uintptr_t>(d) & 15) == 0)) {
        *reinterpret_cast<float4*>(d) = make_float4(o[0], o[1], o[2], o[3]);
        bad += nonfinite(o[0]) + nonfinite(o[1]) + nonfinite(o[2]) + nonfinite(o[3]);
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (e + u >= t.start && e + u < t.end) {
            d[u] = o[u];
            bad += nonfinite(o[u]);
          }
      }
    }
  }
  unsigned long long c = bad;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
  if ((tid & 31) == 0 && c) atomicAdd(&s_count, c);
  __syncthreads();
  if (tid == 0)
    finish_reduction(p.state, s_count, (s_count != 0ull) || s_bad_scale, p.advance, p.beta1, p.beta2, &p.scaler, 0);
}

// ---------------------------------------------------------------- staged: the tree over per-rank accumulators

template <int MAXSEG>
struct RsTreeParams {
  const float* acc[DP_MAX_N];
  float* gbar[DP_MAX_N];
  dp_step_state_t* state;
  float inv;
  int32_t n;
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
  if (threadIdx.x == 0) finish_reduction(p.state, s_count, s_count != 0ull, 0, 1.0, 1.0);
}

// ---------------------------------------------------------------- launchers

template <int MAXSEG>
void fill_table(SegTable<MAXSEG>& T, const Plan& P) {
  T.psi = P.psi;
  T.nseg = P.nseg;
  T.ntiles = P.ntiles;
  for (int k = 0; k <= P.nseg; ++k) {
    T.e[k].goff = P.e[k].goff;
    T.e[k].loff = P.e[k].loff;
    T.e[k].tile0 = P.e[k].tile0;
    T.e[k].owner = P.e[k].owner;
  }
}

// Resident CTAs of `kernel` on every SM, capped by the tile count (at least 1: every CTA joins the finish).
template <typename K>
int resident_grid(K kernel, int threads, int ntiles) {
  int dev = 0, sms = 0, per_sm = 1;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                   cudaSuccess || sms < 1)
    sms = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  long long g = (long long)sms * per_sm;
  if (ntiles < g) g = ntiles;
  return (int)(g < 1 ? 1 : g);
}

template <int MAXSEG, bool COMP>
cudaError_t launch_tree_t(const Plan& P, const uint16_t* const* g, int a, float* const* gbar,
                          const StepScalars& s, int advance, dp_step_state_t* st, cudaStream_t stream) {
  TreeParams<MAXSEG> prm;
  for (int q = 0; q < P.n * a; ++q) prm.g[q] = g[q];
  for (int r = 0; r < P.n; ++r) prm.gbar[r] = gbar[r];
  prm.state = st;
  prm.beta1 = (double)s.beta1;
  prm.beta2 = (double)s.beta2;
  prm.inv = s.inv;
  prm.n = P.n;
  prm.a = a;
  prm.advance = advance;
  prm.scaler = s.scaler;
  fill_table(prm.seg, P);
  auto kern = reduce_tree_kernel<MAXSEG, COMP>;
  kern<<<resident_grid(kern, RT_THREADS, P.ntiles), RT_THREADS, 0, stream>>>(prm);
  return cudaGetLastError();
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
  fill_table(prm.seg, P);
  auto kern = rs_tree_kernel<MAXSEG, COMP>;
  kern<<<resident_grid(kern, 256, P.ntiles), 256, 0, stream>>>(prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_reduce_tree(const Plan& P, const uint16_t* const* g, int a, float* const* gbar,
                               const StepScalars& s, int advance, dp_step_state_t* st, cudaStream_t stream,
                               uint64_t* launches) {
  ++*launches;
  const bool comp = s.mode == DP_SUM_COMPENSATED;
  if (P.nseg <= SMALL_SEG)
    return comp ? launch_tree_t<SMALL_SEG, true>(P, g, a, gbar, s, advance, st, stream)
                : launch_tree_t<SMALL_SEG, false>(P, g, a, gbar, s, advance, st, stream);
  return comp ? launch_tree_t<BIG_SEG, true>(P, g, a, gbar, s, advance, st, stream)
              : launch_tree_t<BIG_SEG, false>(P, g, a, gbar, s, advance, st, stream);
}

cudaError_t launch_rs_tree(const Plan& P, const float* const* acc, float* const* gbar, const StepScalars& s,
                           dp_step_state_t* st, cudaStream_t stream, uint64_t* launches) {
  ++*launches;
  const bool comp = s.mode == DP_SUM_COMPENSATED;
  if (P.nseg <= SMALL_SEG)
    return comp ? launch_rs_tree_t<SMALL_SEG, true>(P, acc, gbar, s, st, stream)
                : launch_rs_tree_t<SMALL_SEG, false>(P, acc, gbar, s, st, stream);
  return comp ? launch_rs_tree_t<BIG_SEG, true>(P, acc, gbar, s, st, stream)
              : launch_rs_tree_t<BIG_SEG, false>(P, acc, gbar, s, st, stream);
}

}  // namespace dp
