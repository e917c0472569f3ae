// The single pass's shared pieces (sm_103a): the reduction kernels' thread and shared-memory layout, their
// launch parameters, and the per-tile steps every single-pass kernel takes after its reduction -- the tile's
// old optimizer state fetched into shared memory, Adam from the tile's gbar into the other state set, and the
// all-gather of the tile's bf16 image into the replicas.  Used by the ring-order kernels (dp_kernels.cu) and
// the tree-order single pass (dp_tree_sp.cu).
#pragma once

#include "dp_device.cuh"
#include "dp_internal.h"
#include "dp_launch.h"

namespace dp {

constexpr int RA_CWARPS = 15;
constexpr int RA_CTHREADS = RA_CWARPS * 32;    // consumer threads
constexpr int RA_EPT = 16;                     // elements per consumer thread: two 16-byte shared loads
constexpr int RA_THREADS = RA_CTHREADS + 32;   // + one producer warp: 16 warps, 4 per SM sub-partition
constexpr int RA_NPS = 2;                      // inputs per stage: two 15 KB bulk copies on one barrier
constexpr int RA_IN_BYTES = TILE * 2;          // one tile of one bf16 input
constexpr int RA_STAGE_BYTES = RA_NPS * RA_IN_BYTES;
constexpr int RA_GBAR_FLOATS = TILE + 16;      // single pass: the tile's gbar (+16: last group's overhang)
constexpr int RA_STATE_FLOATS = TILE + 16;     // single pass: the tile's old master / m / v, one array each
// FUSED selects the kernel's job: 0, pass A of the two-pass step (180 KB of stages in flight); 1, the single
// pass with a shared gbar tile through which the consumer warps regroup gbar into local 4-groups (three
// stages); 2, the single pass for shards whose offsets are multiples of 4, where each thread's 16 elements
// already are local 4-groups, so the gbar tile gives way to a fourth stage (chosen with at least 16 inputs a
// tile).  Both single passes also hold
// the tile's bf16 staging and its old optimizer state, fetched while its gradients stream.
template <int FUSED>
__host__ __device__ constexpr int ra_stages() { return FUSED == 2 ? 4 : FUSED ? 3 : 6; }
template <int FUSED>
__host__ __device__ constexpr int ra_gbar_bytes() { return FUSED == 1 ? RA_GBAR_FLOATS * 4 : 0; }
template <int FUSED>
__host__ __device__ constexpr int ra_extra() { return FUSED ? ra_gbar_bytes<FUSED>() + TILE * 2 + 3 * RA_STATE_FLOATS * 4 : 0; }
template <int FUSED>
__host__ __device__ constexpr int ra_bar_offset() { return ra_stages<FUSED>() * RA_STAGE_BYTES + ra_extra<FUSED>(); }
// Barriers: full/empty per stage, the single pass's state full/empty, abort, count.
template <int FUSED>
__host__ __device__ constexpr int ra_smem() { return ra_bar_offset<FUSED>() + 2 * ra_stages<FUSED>() * 8 + (FUSED ? 16 : 0) + 32; }
static_assert(ra_smem<0>() + 64 <= 227 * 1024 && ra_smem<1>() + 64 <= 227 * 1024 && ra_smem<2>() + 64 <= 227 * 1024,
              "shared memory fits one CTA");
static_assert(TILE == RA_CTHREADS * RA_EPT, "one 16-element group per consumer thread");
static_assert(RA_STATE_FLOATS >= TILE + 8, "a tile's state interior plus its head and tail groups fit one array");
static_assert(RA_IN_BYTES % 16 == 0, "bulk copies are whole 16-byte units");

template <int MAXSEG>
struct ReduceParams {
  const uint16_t* g[DP_MAX_NA];
  float* gbar[DP_MAX_N];
  dp_step_state_t* state;
  uint64_t timeout_ns;
  double beta1, beta2;
  float inv;
  int32_t n, a, advance;
  int32_t merge;     // a later launch of one reduction (see finish_reduction)
  ScalerK scaler;    // enabled: unscale by the device-resident scale, then update it
  // single pass only: the two optimizer-state sets, the replicas, Adam constants
  float* st_master[2][DP_MAX_N];
  float* st_m[2][DP_MAX_N];
  float* st_v[2][DP_MAX_N];
  uint16_t* rep[DP_MAX_N];
  int64_t state_end4[DP_MAX_N];   // each rank's shard length rounded down to a multiple of 4
  float lr, b1f, b2f, eps, omb1, omb2;
  SegTable<MAXSEG> seg;
};

// Single pass: a tile's old state in shared memory.  Each of the three arrays (RA_STATE_FLOATS apart) holds
// the tile's 4-aligned local interior [jlo, jhi) from float 4 on, and -- when the tile's local range starts or
// ends inside a 4-group that lies wholly in the shard array -- that 16-byte head group in floats 0..3 and that
// tail group right after the interior, so that local element j of the tile is always at 4 + (j - jlo).  Flags
// say which ragged groups were copied (the shard's last, partial group is read from HBM).
constexpr int RA_STATE_PAD = 4;

// Ring-buffer position of a stage: slot and the parity of its current use.
template <int NSTAGES>
struct RingPos {
  uint32_t slot = 0, phase = 0, count = 0;
  __device__ __forceinline__ void next() {
    ++count;
    if (++slot == NSTAGES) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Four bf16 values into a staging tile at element offset `off` (any alignment).
__device__ __forceinline__ void stage_bf16x4(uint16_t* sb, int64_t off, uint32_t w0, uint32_t w1) {
  if ((off & 3) == 0) {
    *reinterpret_cast<uint2*>(sb + off) = make_uint2(w0, w1);
  } else if ((off & 1) == 0) {
    *reinterpret_cast<uint32_t*>(sb + off) = w0;
    *reinterpret_cast<uint32_t*>(sb + off + 2) = w1;
  } else {
    sb[off] = (uint16_t)(w0 & 0xFFFFu);
    sb[off + 1] = (uint16_t)(w0 >> 16);
    sb[off + 2] = (uint16_t)(w1 & 0xFFFFu);
    sb[off + 3] = (uint16_t)(w1 >> 16);
  }
}

// Single pass: Adam on the tile's local 4-groups with gbar from shared memory (indexed by global position),
// old state from set `cur`, new state into the other set, bf16 of the new master into the staging tile.
template <int MAXSEG>
__device__ __forceinline__ void fused_update(const ReduceParams<MAXSEG>& p, const Tile& t, const AdamK& K, int cur,
                                             const float* s_g, uint16_t* s_stage, const float* s_state,
                                             const volatile int* s_ragged, int tid) {
  constexpr int UG = 2;
  const int64_t delta = t.loff - t.goff;
  const int64_t cb = (t.start / TILE) * TILE;
  const int64_t js = t.start + delta, je = t.end + delta;
  const int64_t jlo = (js + 3) & ~int64_t(3), jhi = je & ~int64_t(3);
  const int ngr = jhi > jlo ? (int)((jhi - jlo) >> 2) : 0;
  const float* M = p.st_master[cur][t.owner];
  const float* Mm = p.st_m[cur][t.owner];
  const float* Vv = p.st_v[cur][t.owner];
  float* M2 = p.st_master[cur ^ 1][t.owner];
  float* Mm2 = p.st_m[cur ^ 1][t.owner];
  float* Vv2 = p.st_v[cur ^ 1][t.owner];
  const bool galign = ((delta & 3) == 0);
  for (int base = 0; base < ngr; base += UG * RA_CTHREADS) {
    float4 t4[UG], m4[UG], v4[UG], g4[UG];
#pragma unroll
    for (int u = 0; u < UG; ++u) {
      const int gq = base + tid + u * RA_CTHREADS;
      if (gq < ngr) {
        const int64_t jj = jlo + 4 * (int64_t)gq;
        // The 4-aligned interior [jlo, jhi) of the old state sits in shared memory (bulk-copied by the producer).
        t4[u] = *reinterpret_cast<const float4*>(s_state + RA_STATE_PAD + 4 * gq);
        m4[u] = *reinterpret_cast<const float4*>(s_state + RA_STATE_FLOATS + RA_STATE_PAD + 4 * gq);
        v4[u] = *reinterpret_cast<const float4*>(s_state + 2 * RA_STATE_FLOATS + RA_STATE_PAD + 4 * gq);
        const float* gs = s_g + (jj - delta - cb);
        g4[u] = galign ? *reinterpret_cast<const float4*>(gs) : make_float4(gs[0], gs[1], gs[2], gs[3]);
      }
    }
#pragma unroll
    for (int u = 0; u < UG; ++u) {
      const int gq = base + tid + u * RA_CTHREADS;
      if (gq < ngr) {
        const int64_t jj = jlo + 4 * (int64_t)gq;
        adam1(g4[u].x, t4[u].x, m4[u].x, v4[u].x, K);
        adam1(g4[u].y, t4[u].y, m4[u].y, v4[u].y, K);
        adam1(g4[u].z, t4[u].z, m4[u].z, v4[u].z, K);
        adam1(g4[u].w, t4[u].w, m4[u].w, v4[u].w, K);
        *reinterpret_cast<float4*>(M2 + jj) = t4[u];
        *reinterpret_cast<float4*>(Mm2 + jj) = m4[u];
        *reinterpret_cast<float4*>(Vv2 + jj) = v4[u];
        stage_bf16x4(s_stage, jj - delta - cb, bf16x2_rn(t4[u].x, t4[u].y), bf16x2_rn(t4[u].z, t4[u].w));
      }
    }
  }
  // Ragged ends of the tile in local space (at most 3 elements each).
  int64_t jx = -1;
  if (tid < 4) {
    jx = js + tid;
    if (jx >= (jlo < je ? jlo : je)) jx = -1;
  } else if (tid < 8) {
    jx = (jhi > jlo ? jhi : jlo) + (tid - 4);
    if (jx >= je) jx = -1;
  }
  if (jx >= 0) {
    // from the copied head / tail group, or (the shard's partial last group) from HBM
    float th, mm, vv;
    if (s_ragged[jx < jlo ? 0 : 1]) {
      const int64_t o = RA_STATE_PAD + (jx - jlo);
      th = s_state[o];
      mm = s_state[RA_STATE_FLOATS + o];
      vv = s_state[2 * RA_STATE_FLOATS + o];
    } else {
      th = M[jx];
      mm = Mm[jx];
      vv = Vv[jx];
    }
    adam1(s_g[jx - delta - cb], th, mm, vv, K);
    M2[jx] = th;
    Mm2[jx] = mm;
    Vv2[jx] = vv;
    s_stage[jx - delta - cb] = bf16_rn(th);
  }
}

// Single pass, producer thread: the tile's old master/m/v -- the 4-aligned local interior of set `cur`, and
// its ragged head and tail groups where they lie wholly in the array -- into s_state, once the update of the
// previous tile has read it (sempty; sit counts this CTA's state copies).  A wait that runs out sets the abort
// flag and copies nothing.
template <int MAXSEG>
__device__ __forceinline__ void sp_issue_state(const ReduceParams<MAXSEG>& p, const Tile& t, int cur, uint32_t& sit,
                                               float* s_state, volatile int* s_ragged, uint64_t* sfull,
                                               uint64_t* sempty, volatile int* s_abort) {
  if (sit > 0 && !mbar_wait_bounded(smem_u32(sempty), (sit - 1) & 1u, p.timeout_ns, s_abort)) {
    if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
    *s_abort = 1;
    return;
  }
  const int64_t delta = t.loff - t.goff;
  const int64_t js = t.start + delta, je = t.end + delta;
  const int64_t jlo = (js + 3) & ~int64_t(3), jhi = je & ~int64_t(3);
  const int64_t end4 = p.state_end4[t.owner];
  const uint32_t sb = jhi > jlo ? (uint32_t)(jhi - jlo) * 4u : 0u;
  // The head group [jlo - 4, jlo) when the range starts inside it, the tail group [jhi, jhi + 4) when it
  // ends inside it (the same group as the head when no whole group lies inside the range), each only
  // when it lies wholly in the array.
  const bool head = (js & 3) != 0 && jlo <= end4;
  const bool tail = (je & 3) != 0 && jhi >= jlo && jhi + 4 <= end4;
  s_ragged[0] = head ? 1 : 0;
  s_ragged[1] = (tail || (jhi < jlo && head)) ? 1 : 0;
  mbar_arrive_expect_tx(smem_u32(sfull), 3u * (sb + (head ? 16u : 0u) + (tail ? 16u : 0u)));
  float* const src[3] = {p.st_master[cur][t.owner], p.st_m[cur][t.owner], p.st_v[cur][t.owner]};
  for (int k = 0; k < 3; ++k) {
    float* dst = s_state + k * RA_STATE_FLOATS;
    if (sb) bulk_g2s(smem_u32(dst + RA_STATE_PAD), src[k] + jlo, sb, smem_u32(sfull));
    if (head) bulk_g2s(smem_u32(dst + RA_STATE_PAD - 4), src[k] + (jlo - 4), 16u, smem_u32(sfull));
    if (tail) bulk_g2s(smem_u32(dst + RA_STATE_PAD + (jhi - jlo)), src[k] + jhi, 16u, smem_u32(sfull));
  }
  ++sit;
}

// Single pass, consumer threads, once a tile's bf16 image is complete in s_stage (indexed by global position
// in the cell at cb): the image into every replica -- the 16-byte-aligned interior by bulk copies that thread
// 0 issues and commits, the up to 7 elements at each end by threads 0..15 with plain stores.
template <int MAXSEG>
__device__ __forceinline__ void sp_gather(const ReduceParams<MAXSEG>& p, const Tile& t, int64_t cb,
                                          const uint16_t* s_stage, int n, int tid) {
  const int64_t ilo = (t.start + 7) & ~int64_t(7), ihi = t.end & ~int64_t(7);
  if (tid == 0) {
    if (ihi > ilo) {
      const uint32_t src = smem_u32(s_stage + (ilo - cb));
      const uint32_t bytes = (uint32_t)(ihi - ilo) * 2u;
      for (int rr = 0; rr < n; ++rr) bulk_s2g(p.rep[rr] + ilo, src, bytes);
    }
    bulk_commit();
  }
  if (tid < 16) {
    int64_t ix = -1;
    if (tid < 8) {
      ix = t.start + tid;
      if (ix >= (ilo < t.end ? ilo : t.end)) ix = -1;
    } else {
      ix = (ihi > ilo ? ihi : ilo) + (tid - 8);
      if (ix >= t.end) ix = -1;
    }
    if (ix >= 0) {
      const uint16_t b = s_stage[ix - cb];
      for (int rr = 0; rr < n; ++rr) p.rep[rr][ix] = b;
    }
  }
}

// ---------------------------------------------------------------- host side

// Single-pass inputs beyond the reduction's: optimizer-state sets and replicas.
struct FusedArgs {
  float* const* master;  // 2n pointers: set 0 then set 1
  float* const* m;
  float* const* v;
  uint16_t* const* rep;  // n
};

// The launch parameters of a reduction (fa: the single pass's state sets and replicas, or null).
template <int MAXSEG>
void fill_reduce_params(ReduceParams<MAXSEG>& prm, const Plan& P, const uint16_t* const* g, int a,
                        float* const* gbar, const StepScalars& s, int advance, dp_step_state_t* st,
                        const FusedArgs* fa) {
  for (int q = 0; q < P.n * a; ++q) prm.g[q] = g[q];
  for (int r = 0; r < P.n; ++r) prm.gbar[r] = gbar ? gbar[r] : nullptr;
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
  if (fa) {
    for (int r = 0; r < P.n; ++r) {
      for (int k = 0; k < 2; ++k) {
        prm.st_master[k][r] = fa->master[k * P.n + r];
        prm.st_m[k][r] = fa->m[k * P.n + r];
        prm.st_v[k][r] = fa->v[k * P.n + r];
      }
      prm.rep[r] = fa->rep[r];
      prm.state_end4[r] = P.shard_len[r] & ~int64_t(3);
    }
  }
  prm.lr = s.lr;
  prm.b1f = s.beta1;
  prm.b2f = s.beta2;
  prm.eps = s.eps;
  prm.omb1 = s.omb1;
  prm.omb2 = s.omb2;
  fill_seg(prm.seg, P);
}

// The tree order's single pass (dp_tree_sp.cu): one launch of a plan of at most KERNEL_SEG segments.
cudaError_t launch_tree_single(const Plan& P, const uint16_t* const* g, int a, const StepScalars& s,
                               dp_step_state_t* st, const FusedArgs& fa, cudaStream_t stream);

}  // namespace dp
