// C ABI of the fused data-parallel step: argument checks, layout plans and
// the launch sequences.  Every check runs before the first launch, so a call
// that returns an argument error has launched nothing.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include "dp_device.cuh"
#include "dp_internal.h"
#include "dpstep.h"

using dp::Plan;
using dp::StepScalars;

namespace {

thread_local char g_err[512] = "";
std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_timeout_ns{2000000000ull};

dp_status_t fail(dp_status_t s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

dp_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(DP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct LaunchCount {
  uint64_t n = 0;
  ~LaunchCount() { g_launches.fetch_add(n); }
};

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// lens (optional): elements behind each pointer; a pointer to zero elements may be NULL.
dp_status_t check_ptr_array(const void* const* arr, int count, const char* name, const int64_t* lens = nullptr) {
  if (!arr) return fail(DP_ERR_INVALID_ARG, "%s: pointer array is NULL", name);
  for (int i = 0; i < count; ++i) {
    if (!arr[i] && lens && lens[i] == 0) continue;
    if (!arr[i]) return fail(DP_ERR_INVALID_ARG, "%s[%d] is NULL", name, i);
    if (!aligned16(arr[i])) return fail(DP_ERR_ALIGNMENT, "%s[%d] is not 16-byte aligned", name, i);
  }
  return DP_OK;
}

dp_status_t check_state(const void* st) {
  if (!st) return fail(DP_ERR_INVALID_ARG, "state is NULL");
  if (((uintptr_t)st & 7u) != 0) return fail(DP_ERR_ALIGNMENT, "state is not 8-byte aligned");
  return DP_OK;
}

dp_status_t build_plan(const dp_layout_t* L, Plan& P) {
  if (!L) return fail(DP_ERR_INVALID_ARG, "layout is NULL");
  if (L->stage < 0 || L->stage > 3) return fail(DP_ERR_INVALID_ARG, "stage %d not in 0..3", L->stage);
  if (L->n < 1 || L->n > DP_MAX_N) return fail(DP_ERR_INVALID_ARG, "n = %d not in 1..%d", L->n, DP_MAX_N);
  if (L->psi < 0) return fail(DP_ERR_INVALID_ARG, "psi < 0");
  if (L->nseg < 0 || L->nseg > DP_MAX_SEG)
    return fail(DP_ERR_INVALID_ARG, "nseg = %d not in 0..%d", L->nseg, DP_MAX_SEG);
  if (L->reserved != 0) return fail(DP_ERR_INVALID_ARG, "layout.reserved must be 0");
  if (L->nseg > 0 && !L->seg) return fail(DP_ERR_INVALID_ARG, "layout.seg is NULL");
  P.n = L->n;
  P.stage = L->stage;
  P.psi = L->psi;
  for (int r = 0; r < DP_MAX_N; ++r) P.shard_len[r] = 0;
  struct LR {
    int32_t owner;
    int64_t lo, len;
  };
  std::vector<LR> locals;
  locals.reserve(L->nseg);
  P.e.resize((size_t)L->nseg + 1);
  int64_t g = 0;
  int k = 0;
  int64_t tiles = 0;
  for (int i = 0; i < L->nseg; ++i) {
    const dp_segment_t& s = L->seg[i];
    if (s.reserved != 0) return fail(DP_ERR_INVALID_ARG, "seg[%d].reserved must be 0", i);
    if (s.global_off != g)
      return fail(DP_ERR_INVALID_ARG, "seg[%d].global_off = %lld, expected %lld (segments must be contiguous)", i,
                  (long long)s.global_off, (long long)g);
    if (s.len < 0 || s.len > L->psi - g) return fail(DP_ERR_INVALID_ARG, "seg[%d].len out of range", i);
    if (s.owner < 0 || s.owner >= L->n) return fail(DP_ERR_INVALID_ARG, "seg[%d].owner = %d not in 0..n-1", i, s.owner);
    if (s.local_off < 0 || s.local_off > INT64_MAX / 2 - s.len)
      return fail(DP_ERR_INVALID_ARG, "seg[%d].local_off out of range", i);
    g += s.len;
    if (s.len == 0) continue;
    locals.push_back({s.owner, s.local_off, s.len});
    P.shard_len[s.owner] = std::max(P.shard_len[s.owner], s.local_off + s.len);
    const int64_t gend = s.global_off + s.len;
    const int64_t nt = (gend + dp::TILE - 1) / dp::TILE - s.global_off / dp::TILE;
    P.e[k].goff = s.global_off;
    P.e[k].loff = s.local_off;
    P.e[k].owner = s.owner;
    P.e[k].tile0 = (int32_t)tiles;
    tiles += nt;
    if (tiles > INT32_MAX) return fail(DP_ERR_INVALID_ARG, "too many tiles");
    ++k;
  }
  if (g != L->psi) return fail(DP_ERR_INVALID_ARG, "segments cover %lld of psi = %lld elements", (long long)g,
                               (long long)L->psi);
  std::sort(locals.begin(), locals.end(), [](const LR& x, const LR& y) {
    return x.owner != y.owner ? x.owner < y.owner : x.lo < y.lo;
  });
  for (size_t i = 1; i < locals.size(); ++i)
    if (locals[i].owner == locals[i - 1].owner && locals[i].lo < locals[i - 1].lo + locals[i - 1].len)
      return fail(DP_ERR_INVALID_ARG, "rank %d: local ranges overlap", locals[i].owner);
  P.nseg = k;
  P.ntiles = (int32_t)tiles;
  P.e.resize((size_t)k + 1);
  P.e[k].goff = L->psi;
  P.e[k].loff = 0;
  P.e[k].owner = 0;
  P.e[k].tile0 = (int32_t)tiles;
  return DP_OK;
}

dp_status_t check_adam(const dp_adam_t& A) {
  if (!std::isfinite(A.lr) || A.lr < 0.0f) return fail(DP_ERR_INVALID_ARG, "lr must be finite and >= 0");
  if (!(A.beta1 >= 0.0f && A.beta1 < 1.0f)) return fail(DP_ERR_INVALID_ARG, "beta1 must be in [0, 1)");
  if (!(A.beta2 >= 0.0f && A.beta2 < 1.0f)) return fail(DP_ERR_INVALID_ARG, "beta2 must be in [0, 1)");
  if (!std::isfinite(A.eps) || !(A.eps > 0.0f)) return fail(DP_ERR_INVALID_ARG, "eps must be finite and > 0");
  return DP_OK;
}

// The scaler argument of a commit: NULL keeps the scale as it is.
dp_status_t scaler_of(const dp_scaler_t* scaler, dp::ScalerK& k) {
  k = dp::ScalerK{0, 1, 1.0f, 1.0f, 1.0f, 1.0f, 0};
  if (!scaler) return DP_OK;
  const dp_scaler_t& c = *scaler;
  if (!(std::isfinite(c.growth_factor) && c.growth_factor >= 1.0f) ||
      !(c.backoff_factor > 0.0f && c.backoff_factor <= 1.0f) || c.growth_interval < 1 ||
      !(c.min_scale > 0.0f) || !std::isfinite(c.max_scale) || !(c.max_scale >= c.min_scale))
    return fail(DP_ERR_INVALID_ARG, "scaler: need growth >= 1, backoff in (0, 1], interval >= 1, "
                                    "0 < min_scale <= max_scale < inf");
  k = dp::ScalerK{1, c.growth_interval, c.growth_factor, c.backoff_factor, c.min_scale, c.max_scale, 1};
  return DP_OK;
}

// sum_mode = arithmetic (DP_SUM_*) | rank order (DP_ORDER_*) | step flags (DP_DEFER_COMMIT, DP_DEVICE_SCALE).
constexpr int kFlagBits = DP_DEFER_COMMIT | DP_DEVICE_SCALE;
static bool split_mode(int sum_mode, int& arith, int& order, int* flags = nullptr) {
  arith = sum_mode & 0xF;
  order = sum_mode & DP_ORDER_TREE;
  const int f = sum_mode & kFlagBits;
  if (flags) *flags = f;
  else if (f) return false;
  if (sum_mode & ~(0xF | DP_ORDER_TREE | kFlagBits)) return false;
  return (arith == DP_SUM_COMPENSATED || arith == DP_SUM_PLAIN) && (order == DP_ORDER_RING || order == DP_ORDER_TREE);
}

// allowed: the step flags this entry point accepts.  With DP_DEVICE_SCALE the reduction unscales by the
// device-resident scale (read and checked on the device) and loss_scale is not used.
dp_status_t scalars(const Plan& P, const dp_adam_t* A, float loss_scale, int sum_mode, StepScalars& s,
                    int allowed = 0) {
  int arith = 0, order = 0, flags = 0;
  if (!split_mode(sum_mode, arith, order, &flags)) return fail(DP_ERR_INVALID_ARG, "sum_mode %d unknown", sum_mode);
  if (flags & ~allowed)
    return fail(DP_ERR_INVALID_ARG, "sum_mode flag 0x%x is not accepted by this call", flags & ~allowed);
  if (flags & DP_DEVICE_SCALE) loss_scale = 1.0f;
  if (!std::isfinite(loss_scale) || !(loss_scale > 0.0f))
    return fail(DP_ERR_INVALID_ARG, "loss scale must be finite and > 0");
  const double inv = 1.0 / ((double)P.n * (double)loss_scale);
  const float inv32 = (float)inv;
  if (!std::isfinite(inv32) || !(inv32 >= 1.17549435e-38f))
    return fail(DP_ERR_INVALID_ARG, "1 / (n * loss_scale) is not a normal fp32 number");
  s.inv = inv32;
  s.mode = arith;
  s.order = order;
  s.timeout_ns = g_timeout_ns.load();
  s.scaler = dp::ScalerK{(flags & DP_DEVICE_SCALE) ? 1 : 0, 1, 1.0f, 1.0f, 1.0f, 1.0f, 0};
  s.defer = (flags & DP_DEFER_COMMIT) ? 1 : 0;
  s.merge = 0;
  if (A) {
    dp_status_t st = check_adam(*A);
    if (st != DP_OK) return st;
    s.lr = A->lr;
    s.beta1 = A->beta1;
    s.beta2 = A->beta2;
    s.eps = A->eps;
    s.omb1 = (float)(1.0 - (double)A->beta1);
    s.omb2 = (float)(1.0 - (double)A->beta2);
  } else {
    s.lr = s.beta1 = s.beta2 = s.eps = s.omb1 = s.omb2 = 0.0f;
  }
  return DP_OK;
}

size_t align256(size_t x) { return (x + 255u) & ~size_t(255u); }

// gbar shard pointers: the caller's, or carved from ws.
dp_status_t gbar_ptrs(const Plan& P, float* const* gbar_shard, void* ws, float** out) {
  if (gbar_shard) {
    for (int r = 0; r < P.n; ++r) out[r] = gbar_shard[r];
    return check_ptr_array((const void* const*)out, P.n, "gbar_shard", P.shard_len);
  }
  if (!ws) return fail(DP_ERR_INVALID_ARG, "both gbar_shard and ws are NULL");
  if (((uintptr_t)ws & 255u) != 0) return fail(DP_ERR_ALIGNMENT, "ws is not 256-byte aligned");
  size_t off = 0;
  for (int r = 0; r < P.n; ++r) {
    out[r] = reinterpret_cast<float*>(static_cast<char*>(ws) + off);
    off += align256((size_t)P.shard_len[r] * sizeof(float));
  }
  return DP_OK;
}

// Lengths of each rank's master/m/v arrays: its shard, or psi for plain data parallelism.
void state_lens(const Plan& P, int64_t* lens) {
  for (int r = 0; r < P.n; ++r) lens[r] = P.stage == 0 ? P.psi : P.shard_len[r];
}

dp_status_t check_state_arrays(const Plan& P, float* const* master, float* const* m, float* const* v) {
  int64_t lens[DP_MAX_N];
  state_lens(P, lens);
  dp_status_t st = check_ptr_array((const void* const*)master, P.n, "master", lens);
  if (st == DP_OK) st = check_ptr_array((const void* const*)m, P.n, "m", lens);
  if (st == DP_OK) st = check_ptr_array((const void* const*)v, P.n, "v", lens);
  return st;
}

dp_status_t check_full_arrays(const Plan& P, const void* const* arr, int count, const char* name) {
  int64_t lens[DP_MAX_NA];
  for (int i = 0; i < count; ++i) lens[i] = P.psi;
  return check_ptr_array(arr, count, name, lens);
}

}  // namespace

dp_status_t dp::report_error(dp_status_t s, const char* msg) { return fail(s, "%s", msg); }

extern "C" {

int32_t dp_abi_version(void) { return 2; }

const char* dp_status_str(dp_status_t s) {
  switch (s) {
    case DP_OK: return "DP_OK";
    case DP_ERR_INVALID_ARG: return "DP_ERR_INVALID_ARG";
    case DP_ERR_ALIGNMENT: return "DP_ERR_ALIGNMENT";
    case DP_ERR_CUDA: return "DP_ERR_CUDA";
    case DP_ERR_TIMEOUT: return "DP_ERR_TIMEOUT";
    case DP_ERR_IO: return "DP_ERR_IO";
  }
  return "DP_ERR_UNKNOWN";
}

const char* dp_last_error(void) { return g_err; }

dp_status_t dp_layout_validate(const dp_layout_t* layout) {
  static thread_local Plan P;
  return build_plan(layout, P);
}

dp_status_t dp_layout_even(int64_t psi, int32_t n, int64_t bucket, int32_t misalign, dp_segment_t* out,
                           int32_t* nseg) {
  if (!nseg) return fail(DP_ERR_INVALID_ARG, "nseg is NULL");
  if (psi < 0 || n < 1 || n > DP_MAX_N || misalign < 0) return fail(DP_ERR_INVALID_ARG, "bad psi, n or misalign");
  if (bucket <= 0 || bucket > psi) bucket = psi > 0 ? psi : 1;
  const int64_t nb = psi == 0 ? 0 : (psi + bucket - 1) / bucket;
  if (nb * n > DP_MAX_SEG) return fail(DP_ERR_INVALID_ARG, "%lld segments exceed %d", (long long)(nb * n), DP_MAX_SEG);
  const int32_t count = (int32_t)(nb * n);
  if (out) {
    if (*nseg < count) return fail(DP_ERR_INVALID_ARG, "capacity %d < %d segments", *nseg, count);
    std::vector<int64_t> local(n, 0), cuts(n + 1);
    int idx = 0;
    for (int64_t b = 0; b < nb; ++b) {
      const int64_t b0 = b * bucket;
      const int64_t len = std::min(bucket, psi - b0);
      const int64_t base = len / n, extra = len % n;
      for (int k = 0; k <= n; ++k) cuts[k] = k * base + std::min<int64_t>(k, extra);
      for (int k = 1; k < n; ++k) cuts[k] = std::min(len, cuts[k] + misalign);
      for (int k = 1; k <= n; ++k) cuts[k] = std::max(cuts[k], cuts[k - 1]);
      for (int s = 0; s < n; ++s) {
        dp_segment_t& e = out[idx++];
        e.global_off = b0 + cuts[s];
        e.len = cuts[s + 1] - cuts[s];
        e.owner = s;
        e.reserved = 0;
        e.local_off = local[s];
        local[s] += e.len;
      }
    }
  }
  *nseg = count;
  return DP_OK;
}

dp_status_t dp_layout_slice(const dp_layout_t* layout, int64_t lo, int64_t hi, dp_segment_t* out, int32_t* nseg,
                            int64_t* local_base) {
  static thread_local Plan P;
  if (!nseg) return fail(DP_ERR_INVALID_ARG, "nseg is NULL");
  dp_status_t st = build_plan(layout, P);
  if (st != DP_OK) return st;
  if (lo < 0 || hi < lo || hi > layout->psi)
    return fail(DP_ERR_INVALID_ARG, "slice [%lld, %lld) not inside [0, %lld)", (long long)lo, (long long)hi,
                (long long)layout->psi);
  // Pieces of the non-empty segments inside [lo, hi), and the lowest local index of each owner's pieces.
  int64_t base[DP_MAX_N];
  for (int r = 0; r < DP_MAX_N; ++r) base[r] = INT64_MAX;
  int32_t count = 0;
  for (int k = 0; k < P.nseg; ++k) {
    const int64_t g0 = std::max(P.e[k].goff, lo), g1 = std::min(P.e[k + 1].goff, hi);
    if (g0 >= g1) continue;
    const int32_t o = P.e[k].owner;
    base[o] = std::min(base[o], P.e[k].loff + (g0 - P.e[k].goff));
    ++count;
  }
  for (int r = 0; r < P.n; ++r)
    if (base[r] == INT64_MAX) base[r] = 0;   // no piece of this owner in the slice
  if (out) {
    if (*nseg < count) return fail(DP_ERR_INVALID_ARG, "capacity %d < %d segments", *nseg, count);
    int32_t idx = 0;
    for (int k = 0; k < P.nseg; ++k) {
      const int64_t g0 = std::max(P.e[k].goff, lo), g1 = std::min(P.e[k + 1].goff, hi);
      if (g0 >= g1) continue;
      dp_segment_t& e = out[idx++];
      e.global_off = g0 - lo;
      e.len = g1 - g0;
      e.owner = P.e[k].owner;
      e.reserved = 0;
      e.local_off = P.e[k].loff + (g0 - P.e[k].goff) - base[e.owner];
    }
  }
  if (local_base)
    for (int r = 0; r < P.n; ++r) local_base[r] = base[r];
  *nseg = count;
  return DP_OK;
}

int64_t dp_shard_len(const dp_layout_t* layout, int32_t rank) {
  static thread_local Plan P;
  if (build_plan(layout, P) != DP_OK || rank < 0 || rank >= P.n) return -1;
  return P.shard_len[rank];
}

size_t dp_workspace_size(const dp_layout_t* layout) {
  static thread_local Plan P;
  if (build_plan(layout, P) != DP_OK) return 0;
  size_t off = 0;
  for (int r = 0; r < P.n; ++r) off += align256((size_t)P.shard_len[r] * sizeof(float));
  return off > 0 ? off : 256;
}

size_t dp_acc_elems(int64_t psi, int32_t sum_mode) {
  if (psi < 0) return 0;
  return (size_t)psi * ((sum_mode & 0xF) == DP_SUM_COMPENSATED ? 2u : 1u);
}

int64_t dp_global_batch(int64_t b, int32_t n, int32_t a) {
  if (b < 0 || n < 0 || a < 0) return -1;
  const long double x = (long double)b * n * a;
  if (x > (long double)INT64_MAX) return -1;
  return b * (int64_t)n * (int64_t)a;
}

dp_status_t dp_memory_model(int32_t stage, int64_t psi, int32_t n, double out[4]) {
  if (!out || stage < 0 || stage > 3 || psi < 0 || n < 1) return fail(DP_ERR_INVALID_ARG, "bad memory-model args");
  const double P = (double)psi, N = (double)n;
  double params = 2.0 * P, grads = 2.0 * P, opt = 12.0 * P;
  if (stage >= 1) opt /= N;
  if (stage >= 2) grads /= N;
  if (stage >= 3) params /= N;
  out[0] = params;
  out[1] = grads;
  out[2] = opt;
  out[3] = params + grads + opt;
  return DP_OK;
}

dp_status_t dp_traffic_model(int32_t stage, int64_t psi, int32_t n, int32_t wire_bytes_grad,
                             int32_t wire_bytes_param, double out[3]) {
  if (!out || stage < 0 || stage > 3 || psi < 0 || n < 1 || wire_bytes_grad < 1 || wire_bytes_param < 1)
    return fail(DP_ERR_INVALID_ARG, "bad traffic-model args");
  const double f = (double)(n - 1) / (double)n * (double)psi;
  const double wg = wire_bytes_grad, wp = wire_bytes_param;
  double per = 0.0, units = 0.0;  // bytes per rank, and the same in units of f * wg
  int phases = 0;
  if (stage == 0) {
    per = 2.0 * f * wg;
    units = 2.0;
    phases = 2;
  } else if (stage <= 2) {
    per = f * (wg + wp);
    units = (wg + wp) / wg;
    phases = 2;
  } else {
    per = f * (wg + 2.0 * wp);
    units = (wg + 2.0 * wp) / wg;
    phases = 3;
  }
  out[0] = per;
  out[1] = (double)phases * (double)(n - 1);
  out[2] = units / 2.0;
  return DP_OK;
}

void dp_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns > 0 ? ns : 1); }
uint64_t dp_get_wait_timeout_ns(void) { return g_timeout_ns.load(); }
uint64_t dp_kernel_launches(void) { return g_launches.load(); }

dp_status_t dp_state_init(dp_step_state_t* d_state, dp_stream_t stream) {
  dp_status_t st = check_state(d_state);
  if (st != DP_OK) return st;
  LaunchCount lc;
  cudaError_t e = dp::launch_state_init(d_state, (cudaStream_t)stream, &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "state_init launch");
}

dp_status_t dp_accumulate(float* const* acc, const uint16_t* const* g, int64_t psi, int32_t n, int32_t first,
                          int32_t sum_mode, dp_stream_t stream) {
  if (psi < 0 || n < 1 || n > DP_MAX_N) return fail(DP_ERR_INVALID_ARG, "bad psi or n");
  int arith = 0, order = 0;  // the rank order plays no part in a rank's own accumulation
  if (!split_mode(sum_mode, arith, order)) return fail(DP_ERR_INVALID_ARG, "sum_mode %d unknown", sum_mode);
  dp_status_t st = check_ptr_array((const void* const*)acc, n, "acc");
  if (st == DP_OK) st = check_ptr_array((const void* const*)g, n, "g");
  if (st != DP_OK) return st;
  if (psi == 0) return DP_OK;
  LaunchCount lc;
  dp::NvtxRange range("dpstep accumulate");
  cudaError_t e = dp::launch_accumulate(acc, g, psi, n, first, arith, (cudaStream_t)stream, &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "accumulate launch");
}

dp_status_t dp_reduce_scatter_avg(float* const* gbar_shard, const float* const* acc, const dp_layout_t* layout,
                                  float loss_scale, int32_t sum_mode, dp_step_state_t* d_state, dp_stream_t stream) {
  static thread_local Plan P;
  dp_status_t st = build_plan(layout, P);
  if (st != DP_OK) return st;
  StepScalars s;
  if ((st = scalars(P, nullptr, loss_scale, sum_mode, s)) != DP_OK) return st;
  if ((st = check_ptr_array((const void* const*)gbar_shard, P.n, "gbar_shard", P.shard_len)) != DP_OK) return st;
  if ((st = check_full_arrays(P, (const void* const*)acc, P.n, "acc")) != DP_OK) return st;
  if ((st = check_state(d_state)) != DP_OK) return st;
  LaunchCount lc;
  dp::NvtxRange range("dpstep reduce-scatter + average + check");
  cudaError_t e = s.order == DP_ORDER_TREE
                      ? dp::launch_rs_tree(P, acc, gbar_shard, s, d_state, (cudaStream_t)stream, &lc.n)
                      : dp::launch_rs_avg(P, acc, gbar_shard, s, d_state, (cudaStream_t)stream, &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "reduce_scatter_avg launch");
}


dp_status_t dp_adam_shard(float* const* master, float* const* m, float* const* v, const float* const* gbar_shard,
                          const dp_layout_t* layout, dp_adam_t adam, dp_step_state_t* d_state, dp_stream_t stream) {
  static thread_local Plan P;
  dp_status_t st = build_plan(layout, P);
  if (st != DP_OK) return st;
  StepScalars s;
  if ((st = scalars(P, &adam, 1.0f, DP_SUM_COMPENSATED, s)) != DP_OK) return st;
  if ((st = check_state_arrays(P, master, m, v)) != DP_OK) return st;
  if ((st = check_ptr_array((const void* const*)gbar_shard, P.n, "gbar_shard", P.shard_len)) != DP_OK) return st;
  if ((st = check_state(d_state)) != DP_OK) return st;
  LaunchCount lc;
  dp::NvtxRange range("dpstep adam shard");
  cudaError_t e = dp::launch_advance(d_state, (double)adam.beta1, (double)adam.beta2, (cudaStream_t)stream, &lc.n);
  if (e != cudaSuccess) return cuda_fail(e, "advance launch");
  e = dp::launch_update(P, nullptr, master, m, v, gbar_shard, s, d_state, (cudaStream_t)stream, &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "adam launch");
}

dp_status_t dp_allgather_params(uint16_t* const* replicas, const float* const* master, const dp_layout_t* layout,
                                const dp_step_state_t* d_state, dp_stream_t stream) {
  static thread_local Plan P;
  dp_status_t st = build_plan(layout, P);
  if (st != DP_OK) return st;
  if ((st = check_full_arrays(P, (const void* const*)replicas, P.n, "replicas")) != DP_OK) return st;
  {
    int64_t lens[DP_MAX_N];
    state_lens(P, lens);
    if ((st = check_ptr_array((const void* const*)master, P.n, "master", lens)) != DP_OK) return st;
  }
  if ((st = check_state(d_state)) != DP_OK) return st;
  LaunchCount lc;
  dp::NvtxRange range("dpstep all-gather params");
  cudaError_t e = dp::launch_allgather(P, replicas, master, d_state, (cudaStream_t)stream, &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "allgather launch");
}

static dp_status_t prepare_reduce(const Plan& P, const uint16_t* const* grads, int32_t a, const dp_adam_t& adam,
                                  float loss_scale, int32_t sum_mode, float* const* gbar_shard, void* ws,
                                  dp_step_state_t* d_state, StepScalars& s, float** gb, int allowed = 0) {
  if (a < 1 || (int64_t)a * P.n > DP_MAX_NA)
    return fail(DP_ERR_INVALID_ARG, "a = %d: need 1 <= a and n * a <= %d", a, DP_MAX_NA);
  dp_status_t st = scalars(P, &adam, loss_scale, sum_mode, s, allowed);
  if (st == DP_OK) st = check_full_arrays(P, (const void* const*)grads, P.n * a, "grads");
  if (st == DP_OK) st = gbar_ptrs(P, gbar_shard, ws, gb);
  if (st == DP_OK) st = check_state(d_state);
  return st;
}

// Pass A in the order s names.  (With one micro-step the ring kernel and the per-micro-step kernel perform
// the same operations, p = g_{s+1} + ... + g_s then gbar; the ring kernel streams faster.)
static cudaError_t launch_pass_a(const Plan& P, const uint16_t* const* grads, int a, float* const* gb,
                                 const StepScalars& s, dp_step_state_t* st, cudaStream_t stream, uint64_t* launches) {
  dp::NvtxRange range("dpstep pass A: accumulate, reduce-scatter, average, check");
  const int advance = s.defer ? 0 : 1;
  if (s.order == DP_ORDER_TREE) return dp::launch_reduce_tree(P, grads, a, gb, s, advance, st, stream, launches);
  return dp::launch_reduce(P, grads, a, gb, s, advance, st, stream, launches);
}

static cudaError_t launch_pass_b(const Plan& P, uint16_t* const* rep, float* const* master, float* const* m,
                                 float* const* v, const float* const* gb, const StepScalars& s,
                                 const dp_step_state_t* st, cudaStream_t stream, uint64_t* launches) {
  dp::NvtxRange range("dpstep pass B: adam, all-gather");
  return dp::launch_update(P, rep, master, m, v, gb, s, st, stream, launches);
}

dp_status_t dp_step_reduce(float* const* gbar_shard, void* ws, const uint16_t* const* grads, int32_t a,
                           const dp_layout_t* layout, dp_adam_t adam, float loss_scale, int32_t sum_mode,
                           dp_step_state_t* d_state, dp_stream_t stream) {
  static thread_local Plan P;
  dp_status_t st = build_plan(layout, P);
  if (st != DP_OK) return st;
  StepScalars s;
  float* gb[DP_MAX_N];
  if ((st = prepare_reduce(P, grads, a, adam, loss_scale, sum_mode, gbar_shard, ws, d_state, s, gb,
                           DP_DEFER_COMMIT | DP_DEVICE_SCALE)) != DP_OK)
    return st;
  LaunchCount lc;
  cudaError_t e = launch_pass_a(P, grads, a, gb, s, d_state, (cudaStream_t)stream, &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "reduce launch");
}

dp_status_t dp_reduce_scatter_micro(float* const* acc_shard, float* const* gbar_shard, void* ws,
                                    const uint16_t* const* g, int32_t k, int32_t a, const dp_layout_t* layout,
                                    dp_adam_t adam, float loss_scale, int32_t sum_mode, dp_step_state_t* d_state,
                                    dp_stream_t stream) {
  static thread_local Plan P;
  dp_status_t st = build_plan(layout, P);
  if (st != DP_OK) return st;
  if (a < 1 || k < 0 || k >= a) return fail(DP_ERR_INVALID_ARG, "micro-step k = %d of a = %d", k, a);
  StepScalars s;
  if ((st = scalars(P, &adam, loss_scale, sum_mode, s, DP_DEFER_COMMIT | DP_DEVICE_SCALE)) != DP_OK) return st;
  if (s.order != DP_ORDER_RING) return fail(DP_ERR_INVALID_ARG, "dp_reduce_scatter_micro: ring order only");
  if ((st = check_full_arrays(P, (const void* const*)g, P.n, "g")) != DP_OK) return st;
  if (a > 1) {
    int64_t lens[DP_MAX_N];
    for (int r = 0; r < P.n; ++r) lens[r] = P.shard_len[r] * (s.mode == DP_SUM_COMPENSATED ? 2 : 1);
    if ((st = check_ptr_array((const void* const*)acc_shard, P.n, "acc_shard", lens)) != DP_OK) return st;
  }
  float* gb[DP_MAX_N] = {nullptr};
  if (k == a - 1 && (st = gbar_ptrs(P, gbar_shard, ws, gb)) != DP_OK) return st;
  if ((st = check_state(d_state)) != DP_OK) return st;
  LaunchCount lc;
  dp::NvtxRange range("dpstep micro-step reduce-scatter");
  cudaError_t e = dp::launch_rs_micro(P, g, a > 1 ? acc_shard : nullptr, gb, k, a, s, d_state, (cudaStream_t)stream,
                                      &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "reduce_scatter_micro launch");
}

dp_status_t dp_step_update(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                           const float* const* gbar_shard, void* ws, const dp_layout_t* layout, dp_adam_t adam,
                           const dp_step_state_t* d_state, dp_stream_t stream) {
  static thread_local Plan P;
  dp_status_t st = build_plan(layout, P);
  if (st != DP_OK) return st;
  StepScalars s;
  if ((st = scalars(P, &adam, 1.0f, DP_SUM_COMPENSATED, s)) != DP_OK) return st;
  if ((st = check_state_arrays(P, master, m, v)) != DP_OK) return st;
  if ((st = check_full_arrays(P, (const void* const*)replicas, P.n, "replicas")) != DP_OK) return st;
  float* gb[DP_MAX_N];
  if ((st = gbar_ptrs(P, (float* const*)gbar_shard, ws, gb)) != DP_OK) return st;
  if ((st = check_state(d_state)) != DP_OK) return st;
  LaunchCount lc;
  cudaError_t e = launch_pass_b(P, replicas, master, m, v, gb, s, d_state, (cudaStream_t)stream, &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "update launch");
}

}  // extern "C"

namespace {

// dp_step, optionally preceded by the host-to-device copies of its gradients and followed by the copy of its
// state to the host (dp_step_from_host).  Every argument is checked before anything is queued.
dp_status_t step_impl(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                      const uint16_t* const* host_grads, const uint16_t* const* grads, int32_t a,
                      const dp_layout_t* layout, dp_adam_t adam, float loss_scale, int32_t sum_mode,
                      float* const* gbar_shard, void* ws, dp_step_state_t* d_state, dp_step_state_t* host_state,
                      cudaStream_t stream) {
  static thread_local Plan P;
  dp_status_t st = build_plan(layout, P);
  if (st != DP_OK) return st;
  StepScalars s;
  float* gb[DP_MAX_N];
  if ((st = prepare_reduce(P, grads, a, adam, loss_scale, sum_mode, gbar_shard, ws, d_state, s, gb)) != DP_OK)
    return st;
  if ((st = check_state_arrays(P, master, m, v)) != DP_OK) return st;
  if ((st = check_full_arrays(P, (const void* const*)replicas, P.n, "replicas")) != DP_OK) return st;
  if (host_grads &&
      (st = check_full_arrays(P, (const void* const*)host_grads, P.n * a, "host_grads")) != DP_OK)
    return st;
  const size_t bytes = (size_t)P.psi * sizeof(uint16_t);
  if (host_grads && bytes) {
    dp::NvtxRange range("dpstep gradient copies to the device");
    for (int q = 0; q < P.n * a; ++q) {
      const cudaError_t e = cudaMemcpyAsync(const_cast<uint16_t*>(grads[q]), host_grads[q], bytes,
                                            cudaMemcpyHostToDevice, stream);
      if (e != cudaSuccess) return cuda_fail(e, "gradient copy to the device");
    }
  }
  LaunchCount lc;
  cudaError_t e = launch_pass_a(P, grads, a, gb, s, d_state, stream, &lc.n);
  if (e != cudaSuccess) return cuda_fail(e, "reduce launch");
  e = launch_pass_b(P, replicas, master, m, v, gb, s, d_state, stream, &lc.n);
  if (e != cudaSuccess) return cuda_fail(e, "update launch");
  if (host_state) {
    e = cudaMemcpyAsync(host_state, d_state, sizeof(dp_step_state_t), cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return cuda_fail(e, "status copy to the host");
  }
  return DP_OK;
}

}  // namespace

extern "C" {

dp_status_t dp_step(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                    const uint16_t* const* grads, int32_t a, const dp_layout_t* layout, dp_adam_t adam,
                    float loss_scale, int32_t sum_mode, float* const* gbar_shard, void* ws,
                    dp_step_state_t* d_state, dp_stream_t stream) {
  return step_impl(replicas, master, m, v, nullptr, grads, a, layout, adam, loss_scale, sum_mode, gbar_shard, ws,
                   d_state, nullptr, (cudaStream_t)stream);
}

dp_status_t dp_step_from_host(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                              const uint16_t* const* host_grads, uint16_t* const* grads, int32_t a,
                              const dp_layout_t* layout, dp_adam_t adam, float loss_scale, int32_t sum_mode,
                              float* const* gbar_shard, void* ws, dp_step_state_t* d_state,
                              dp_step_state_t* host_state, dp_stream_t stream) {
  if (!host_grads) return fail(DP_ERR_INVALID_ARG, "dp_step_from_host: host_grads is NULL");
  return step_impl(replicas, master, m, v, host_grads, (const uint16_t* const*)grads, a, layout, adam, loss_scale,
                   sum_mode, gbar_shard, ws, d_state, host_state, (cudaStream_t)stream);
}

dp_status_t dp_scaler_init(dp_step_state_t* d_state, float scale, dp_stream_t stream) {
  dp_status_t st = check_state(d_state);
  if (st != DP_OK) return st;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return fail(DP_ERR_INVALID_ARG, "scale must be finite and > 0");
  LaunchCount lc;
  cudaError_t e = dp::launch_scaler_init(d_state, scale, (cudaStream_t)stream, &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "scaler_init launch");
}

dp_status_t dp_step_scaled(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                           const uint16_t* const* grads, int32_t a, const dp_layout_t* layout, dp_adam_t adam,
                           const dp_scaler_t* scaler, int32_t sum_mode, float* const* gbar_shard, void* ws,
                           dp_step_state_t* d_state, dp_stream_t stream) {
  static thread_local Plan P;
  dp_status_t st = build_plan(layout, P);
  if (st != DP_OK) return st;
  if (!scaler) return fail(DP_ERR_INVALID_ARG, "scaler is NULL");
  dp::ScalerK k;
  if ((st = scaler_of(scaler, k)) != DP_OK) return st;
  StepScalars s;
  float* gb[DP_MAX_N];
  // The fixed-scale checks run with scale 1; the real scale is read and checked on the device.
  if ((st = prepare_reduce(P, grads, a, adam, 1.0f, sum_mode, gbar_shard, ws, d_state, s, gb)) != DP_OK)
    return st;
  if ((st = check_state_arrays(P, master, m, v)) != DP_OK) return st;
  if ((st = check_full_arrays(P, (const void* const*)replicas, P.n, "replicas")) != DP_OK) return st;
  s.scaler = k;
  LaunchCount lc;
  cudaError_t e = launch_pass_a(P, grads, a, gb, s, d_state, (cudaStream_t)stream, &lc.n);
  if (e != cudaSuccess) return cuda_fail(e, "reduce launch");
  e = launch_pass_b(P, replicas, master, m, v, gb, s, d_state, (cudaStream_t)stream, &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "update launch");
}

}  // extern "C"

namespace {

// dp_step_single_pass, optionally preceded by the host-to-device copies of its gradients and followed by the
// copy of its state to the host (dp_step_single_pass_from_host).  Every argument is checked first.
dp_status_t single_pass_impl(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                             const uint16_t* const* host_grads, const uint16_t* const* grads, int32_t a,
                             const dp_layout_t* layout, dp_adam_t adam, float loss_scale, int32_t sum_mode,
                             dp_step_state_t* d_state, dp_step_state_t* host_state, cudaStream_t stream) {
  static thread_local Plan P;
  dp_status_t st = build_plan(layout, P);
  if (st != DP_OK) return st;
  if (P.stage == 0) return fail(DP_ERR_INVALID_ARG, "dp_step_single_pass: stage 0 (full replicas) is not supported");
  if (a < 1 || (int64_t)a * P.n > DP_MAX_NA)
    return fail(DP_ERR_INVALID_ARG, "a = %d: need 1 <= a and n * a <= %d", a, DP_MAX_NA);
  StepScalars s;
  if ((st = scalars(P, &adam, loss_scale, sum_mode, s, DP_DEFER_COMMIT | DP_DEVICE_SCALE)) != DP_OK) return st;
  if ((st = check_full_arrays(P, (const void* const*)grads, P.n * a, "grads")) != DP_OK) return st;
  if ((st = check_full_arrays(P, (const void* const*)replicas, P.n, "replicas")) != DP_OK) return st;
  int64_t lens2[2 * DP_MAX_N];
  for (int r = 0; r < P.n; ++r) lens2[r] = lens2[P.n + r] = P.shard_len[r];
  if ((st = check_ptr_array((const void* const*)master, 2 * P.n, "master (2 sets)", lens2)) != DP_OK) return st;
  if ((st = check_ptr_array((const void* const*)m, 2 * P.n, "m (2 sets)", lens2)) != DP_OK) return st;
  if ((st = check_ptr_array((const void* const*)v, 2 * P.n, "v (2 sets)", lens2)) != DP_OK) return st;
  if ((st = check_state(d_state)) != DP_OK) return st;
  if (host_grads &&
      (st = check_full_arrays(P, (const void* const*)host_grads, P.n * a, "host_grads")) != DP_OK)
    return st;
  const size_t bytes = (size_t)P.psi * sizeof(uint16_t);
  if (host_grads && bytes) {
    dp::NvtxRange range("dpstep gradient copies to the device");
    for (int q = 0; q < P.n * a; ++q) {
      const cudaError_t e = cudaMemcpyAsync(const_cast<uint16_t*>(grads[q]), host_grads[q], bytes,
                                            cudaMemcpyHostToDevice, stream);
      if (e != cudaSuccess) return cuda_fail(e, "gradient copy to the device");
    }
  }
  LaunchCount lc;
  {
    dp::NvtxRange range("dpstep single pass: reduce, adam, all-gather");
    cudaError_t e = dp::launch_single_pass(P, grads, a, replicas, master, m, v, s, d_state, stream, &lc.n);
    if (e != cudaSuccess) return cuda_fail(e, "single-pass launch");
  }
  if (host_state) {
    const cudaError_t e = cudaMemcpyAsync(host_state, d_state, sizeof(dp_step_state_t), cudaMemcpyDeviceToHost,
                                          stream);
    if (e != cudaSuccess) return cuda_fail(e, "status copy to the host");
  }
  return DP_OK;
}

}  // namespace

extern "C" {

dp_status_t dp_step_single_pass(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                                const uint16_t* const* grads, int32_t a, const dp_layout_t* layout, dp_adam_t adam,
                                float loss_scale, int32_t sum_mode, dp_step_state_t* d_state, dp_stream_t stream) {
  return single_pass_impl(replicas, master, m, v, nullptr, grads, a, layout, adam, loss_scale, sum_mode, d_state,
                          nullptr, (cudaStream_t)stream);
}

dp_status_t dp_step_single_pass_from_host(uint16_t* const* replicas, float* const* master, float* const* m,
                                          float* const* v, const uint16_t* const* host_grads, uint16_t* const* grads,
                                          int32_t a, const dp_layout_t* layout, dp_adam_t adam, float loss_scale,
                                          int32_t sum_mode, dp_step_state_t* d_state, dp_step_state_t* host_state,
                                          dp_stream_t stream) {
  if (!host_grads) return fail(DP_ERR_INVALID_ARG, "dp_step_single_pass_from_host: host_grads is NULL");
  return single_pass_impl(replicas, master, m, v, host_grads, (const uint16_t* const*)grads, a, layout, adam,
                          loss_scale, sum_mode, d_state, host_state, (cudaStream_t)stream);
}

dp_status_t dp_commit_step(dp_step_state_t* d_state, dp_adam_t adam, const dp_scaler_t* scaler, dp_stream_t stream) {
  dp_status_t st = check_state(d_state);
  if (st != DP_OK) return st;
  if ((st = check_adam(adam)) != DP_OK) return st;
  dp::ScalerK k;
  if ((st = scaler_of(scaler, k)) != DP_OK) return st;
  LaunchCount lc;
  dp::NvtxRange range("dpstep commit");
  cudaError_t e = dp::launch_commit(d_state, (double)adam.beta1, (double)adam.beta2, k, 0, (cudaStream_t)stream,
                                    &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "commit launch");
}

dp_status_t dp_commit_single_pass(uint16_t* const* replicas, float* const* master, const dp_layout_t* layout,
                                  dp_adam_t adam, const dp_scaler_t* scaler, dp_step_state_t* d_state,
                                  dp_stream_t stream) {
  static thread_local Plan P;
  dp_status_t st = build_plan(layout, P);
  if (st != DP_OK) return st;
  if (P.stage == 0) return fail(DP_ERR_INVALID_ARG, "dp_commit_single_pass: stage 0 is not supported");
  if ((st = check_state(d_state)) != DP_OK) return st;
  if ((st = check_adam(adam)) != DP_OK) return st;
  if ((st = check_full_arrays(P, (const void* const*)replicas, P.n, "replicas")) != DP_OK) return st;
  int64_t lens2[2 * DP_MAX_N];
  for (int r = 0; r < P.n; ++r) lens2[r] = lens2[P.n + r] = P.shard_len[r];
  if ((st = check_ptr_array((const void* const*)master, 2 * P.n, "master (2 sets)", lens2)) != DP_OK) return st;
  dp::ScalerK k;
  if ((st = scaler_of(scaler, k)) != DP_OK) return st;
  LaunchCount lc;
  dp::NvtxRange range("dpstep commit (single pass)");
  cudaError_t e = dp::launch_commit(d_state, (double)adam.beta1, (double)adam.beta2, k, 1, (cudaStream_t)stream,
                                    &lc.n);
  if (e != cudaSuccess) return cuda_fail(e, "commit launch");
  e = dp::launch_repair(P, replicas, master, d_state, (cudaStream_t)stream, &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "repair launch");
}

dp_status_t dp_read_status(const dp_step_state_t* d_state, int32_t* skipped, int32_t* err, dp_stream_t stream) {
  dp_status_t st = check_state(d_state);
  if (st != DP_OK) return st;
  dp_step_state_t h;
  cudaError_t e = cudaMemcpyAsync(&h, d_state, sizeof(h), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "read_status copy");
  e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "read_status sync");
  if (skipped) *skipped = h.found_inf;
  if (err) *err = h.error;
  return DP_OK;
}

dp_status_t dp_selftest_wait_timeout(dp_step_state_t* d_state, uint64_t timeout_ns, dp_stream_t stream) {
  dp_status_t st = check_state(d_state);
  if (st != DP_OK) return st;
  if (timeout_ns == 0 || timeout_ns > 10000000000ull)
    return fail(DP_ERR_INVALID_ARG, "timeout_ns must be in (0, 10 s]");
  LaunchCount lc;
  cudaError_t e = dp::launch_selftest_wait(d_state, timeout_ns, (cudaStream_t)stream, &lc.n);
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "selftest launch");
}

}  // extern "C"
