/*
 * dpstep.h -- C ABI of the fused data-parallel step for one GB300 GPU (sm_103a).
 *
 * The step of data-parallel training that follows the backward passes:
 * n replicas ("ranks") each accumulate the gradients of their a micro-steps,
 * the ranks' sums are reduced in ring reduce-scatter order, averaged over n
 * and unscaled by the loss scale under a global non-finite check, a
 * ZeRO-partitioned mixed-precision Adam updates each rank's fp32 shard of
 * master weights and moments, and the bf16 parameters are all-gathered into
 * every replica.  All n ranks' buffers live in one GPU's memory.
 *
 * Sources of the operations (page title -- section or paragraph):
 *  - "Distributed Training: Split along the Four Axes of Data, Tensor,
 *    Pipeline, and State" -- data-parallelism paragraphs: every rank holds a
 *    replica; all-reduce sums the local gradients; each rank accumulates a
 *    micro-steps before one all-reduce; gbar = (sum_r g_r) / n;
 *    B_global = b x n x a; reduction order and precision change gbar.
 *  - same page -- ZeRO/FSDP paragraphs: ZeRO-1 shards optimizer state,
 *    ZeRO-2 also gradients, ZeRO-3/FSDP also parameters; reduce-scatter
 *    leaves each rank its shard's sum, all-gather collects parameters;
 *    sharding does not change the update.
 *  - same page -- memory-budget paragraph: mixed precision keeps an fp32
 *    master copy and Adam's first and second moments per parameter.
 *  - same page -- checkpoint and evaluation paragraphs: loss scaling is
 *    training state that must be kept and aligned.
 *  - "Data vs Tensor vs Pipeline Parallelism: When to Use Each" -- "Data
 *    parallelism: split the batch": ring all-reduce traffic 2(N-1)/N x the
 *    gradient bytes, 16 bytes per parameter, ZeRO-3 16 Psi / N and 1.5x
 *    traffic; "DP gradient sync at scale": 2(N-1) ring steps.
 *  The pages name Adam but do not print its equations; the library uses
 *  standard Adam (Kingma & Ba 2015) with bias correction, epsilon added to
 *  sqrt(vhat), no weight decay, in fp32 (the moments correctly rounded, the
 *  update's square root and division by the GPU's approximate instructions,
 *  within a few ulp of the update term).  Loss-scale unscaling and the skipped step
 *  are not spelled out on the pages either: gbar is multiplied by
 *  fl32(1 / (n S)) and any non-finite value skips the whole step.
 *
 * Conventions of every entry point:
 *  - "device" pointers point into memory of the current CUDA device; the
 *    caller allocates and owns every buffer (the library allocates nothing).
 *  - Arrays of pointers ("float* const* master") are HOST arrays of n (or
 *    n*a) DEVICE pointers; the host array is read during the call only.
 *  - Every device base pointer must be 16-byte aligned (DP_ERR_ALIGNMENT);
 *    element offsets inside buffers need no alignment.
 *  - bf16 values are passed as uint16_t bit patterns.
 *  - Calls are asynchronous on the caller's stream (NULL = legacy default
 *    stream) and make no host synchronisation, except dp_read_status and
 *    dp_state_init's implicit none.  A call that returns an error launched
 *    nothing.  The launch sequence of a step makes no allocation and no
 *    host synchronisation.
 *  - A skipped step is not an error: it is reported on the device in
 *    dp_step_state_t.found_inf and read with dp_read_status.
 *  - Calls on one dp_step_state_t must be ordered (one stream, or events).
 */
#ifndef DPSTEP_H
#define DPSTEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* dp_stream_t;

typedef enum {
  DP_OK = 0,
  DP_ERR_INVALID_ARG = 1, /* bad size, layout, pointer or scalar; nothing launched */
  DP_ERR_ALIGNMENT = 2,   /* a device base pointer is not 16-byte aligned; nothing launched */
  DP_ERR_CUDA = 3,        /* a CUDA runtime call failed; dp_last_error() names it */
  DP_ERR_TIMEOUT = 4,     /* a kernel gave up a bounded wait (device-side, in state.error) */
  DP_ERR_IO = 5           /* a checkpoint file could not be written, read or verified */
} dp_status_t;

/* Reduction arithmetic, the low 4 bits of every sum_mode argument. */
enum {
  DP_SUM_COMPENSATED = 0, /* fp32 with Knuth's TwoSum error terms carried alongside; in the
                             ring order of dp_step / dp_step_reduce one (hi, lo) pair is carried
                             through all n*a inputs, (hi, e) = TwoSum(hi, x), lo = lo + e */
  DP_SUM_PLAIN = 1        /* plain fp32 additions */
};

/* Order in which the ranks' sums are added, OR'd into sum_mode
 * (e.g. DP_SUM_PLAIN | DP_ORDER_TREE).  Both orders are fixed, so results are
 * bit-identical run to run; they differ from each other by rounding only.
 *   DP_ORDER_RING: for the chunk owned by s, g_{s+1} + g_{s+2} + ... + g_s
 *     left to right (the ring reduce-scatter's hops, "Data vs Tensor vs
 *     Pipeline Parallelism", data parallelism section).
 *   DP_ORDER_TREE: a binomial tree over rank index rooted at rank 0, the same
 *     for every element: level l adds the block of ranks
 *     [j 2^(l+1) + 2^l, (j+1) 2^(l+1)) into [j 2^(l+1), j 2^(l+1) + 2^l), the
 *     lower block on the left; a block without a partner (n not a power of
 *     two) moves up a level unchanged.  Compensated: (H, e) = TwoSum(H_left,
 *     H_right), L = (L_left + e) + L_right.  (NCCL's tree algorithms, named on
 *     the same page beside the ring for their 2 log2(n) instead of 2(n-1)
 *     steps.)  dp_step, dp_step_reduce, dp_step_single_pass and the staged
 *     reduce-scatter take either order; dp_reduce_scatter_micro the ring
 *     order only. */
enum { DP_ORDER_RING = 0, DP_ORDER_TREE = 16 };

/* Step flags, OR'd into sum_mode, for a step split across several GPUs, each
 * holding one contiguous slice of the parameter space with all n ranks' data
 * for it (dp_layout_slice).  Every step of the path is elementwise except the
 * skip decision, which must be global: a non-finite value in any slice skips
 * the step on every slice ("Distributed Training: Split along the Four Axes",
 * data-parallel paragraph: every rank applies the same update, so replicas
 * stay identical).  Accepted by dp_step_reduce, dp_step_single_pass(_from_host)
 * and dp_reduce_scatter_micro; the other calls refuse them.
 *   DP_DEFER_COMMIT: the reduction publishes found_inf / nonfinite for its own
 *     slice but leaves t, the beta powers, the current state set and the loss
 *     scale alone.  The caller combines found_inf (the int32 at byte offset 4
 *     of dp_step_state_t) over the slices with a maximum -- one 4-byte
 *     all-reduce -- and then calls dp_commit_step (before dp_step_update) or
 *     dp_commit_single_pass.
 *   DP_DEVICE_SCALE: the reduction unscales by d_state->loss_scale (checked on
 *     the device as dp_step_scaled checks it) instead of the loss_scale
 *     argument, which is then not used; the commit applies the scale policy. */
enum { DP_DEFER_COMMIT = 32, DP_DEVICE_SCALE = 64 };

/* ZeRO stages of the layout. */
enum { DP_STAGE_DP = 0, DP_STAGE_ZERO1 = 1, DP_STAGE_ZERO2 = 2, DP_STAGE_ZERO3 = 3 };

/* Limits: replicas, inputs (n * a), segments of a layout.  A layout of more
 * than DP_KERNEL_SEG segments runs each kernel as several launches over
 * contiguous runs of DP_KERNEL_SEG segments (results unchanged). */
enum { DP_MAX_N = 16, DP_MAX_NA = 64, DP_MAX_SEG = 1 << 20, DP_KERNEL_SEG = 1024 };

/* One contiguous piece of the flat parameter space [0, psi) and where its
 * optimizer state lives: elements [global_off, global_off + len) are owned by
 * rank `owner`, whose shard arrays hold them at [local_off, local_off + len). */
typedef struct {
  int64_t global_off;
  int64_t len;       /* >= 0; empty pieces are allowed and ignored */
  int32_t owner;     /* 0 <= owner < n */
  int32_t reserved;  /* must be 0 */
  int64_t local_off; /* >= 0 */
} dp_segment_t;

/* Shard layout (host memory).  Segments are sorted by global_off, contiguous,
 * and cover [0, psi) exactly; one owner's local ranges must not overlap.
 * stage 0 (plain data parallelism): every rank keeps full-length master/m/v
 * arrays indexed by global position and the segments only fix each chunk's
 * reduction order and where its averaged gradient is stored; stages 1-3:
 * master/m/v of rank s are its shard arrays of dp_shard_len(layout, s)
 * elements.  The stage does not change the arithmetic (ZeRO/FSDP paragraph:
 * sharding changes layout and communication, not the update). */
typedef struct {
  int32_t stage;
  int32_t n;        /* replicas, 1..DP_MAX_N */
  int64_t psi;      /* parameters, >= 0 */
  int32_t nseg;     /* 0..DP_MAX_SEG */
  int32_t reserved; /* must be 0 */
  const dp_segment_t* seg;
} dp_layout_t;

/* Adam hyper-parameters: lr >= 0, 0 <= beta < 1, eps > 0, all finite. */
typedef struct {
  float lr, beta1, beta2, eps;
} dp_adam_t;

/* Device-resident step state (64 bytes, 8-byte aligned, caller-allocated).
 * Initialise with dp_state_init before the first step. */
typedef struct {
  int32_t t;          /* Adam steps applied so far */
  int32_t found_inf;  /* 1 if the last reduction found a non-finite value: the step was skipped */
  int32_t error;      /* sticky device-side error (DP_ERR_TIMEOUT, DP_ERR_INVALID_ARG for a bad device
                         loss scale) or 0; a set error skips every step */
  int32_t good_steps; /* dynamic loss scale: applied steps since the scale last changed */
  uint64_t nonfinite; /* elements whose reduced gradient was not finite, last reduction */
  double b1t, b2t;    /* beta1^t and beta2^t, running products */
  uint64_t work_count;  /* kernel-internal, zero between calls */
  uint32_t work_found;  /* kernel-internal, zero between calls */
  uint32_t work_ticket; /* kernel-internal, zero between calls */
  float loss_scale;   /* dynamic loss scale used by dp_step_scaled (set by dp_scaler_init) */
  uint32_t cur_set;   /* dp_step_single_pass: which of the two master/m/v sets is current (0 or 1) */
} dp_step_state_t;

/* Dynamic loss-scale policy of dp_step_scaled.  After each reduction:
 *   overflow (step skipped):  scale = max(scale * backoff_factor, min_scale), good_steps = 0
 *   clean step:               good_steps += 1; when it reaches growth_interval,
 *                             scale = min(scale * growth_factor, max_scale), good_steps = 0
 * (the growth/back-off rule of common mixed-precision loss scalers, with the scale kept in
 * [min_scale, max_scale]; the pages only name loss scaling as training state to keep and align). */
typedef struct {
  float growth_factor;    /* >= 1 */
  float backoff_factor;   /* in (0, 1] */
  int32_t growth_interval; /* >= 1 */
  float min_scale;        /* > 0 */
  float max_scale;        /* >= min_scale, finite */
} dp_scaler_t;

/* ---- host helpers (no GPU needed) --------------------------------------- */

/* Version of this ABI (not on the pages). */
int32_t dp_abi_version(void);

/* Name of a status code (not on the pages). */
const char* dp_status_str(dp_status_t s);

/* Message of the last failing call on this host thread ("" if none; not on the pages). */
const char* dp_last_error(void);

/* Checks a layout against the rules of dp_layout_t.  DP_OK or DP_ERR_INVALID_ARG.
 * The shard layout follows "Distributed Training: Split along the Four Axes",
 * ZeRO/FSDP paragraph (each rank keeps only its shard of the optimizer state)
 * and "Data vs Tensor vs Pipeline Parallelism", "FSDP wrapping granularity"
 * (shards per wrapped unit); the pages fix no layout rule, these are the
 * library's. */
dp_status_t dp_layout_validate(const dp_layout_t* layout);

/* Builds the standard layouts.  bucket <= 0: one bucket of psi elements.
 * Each bucket is split n ways in rank order (the first (len mod n) pieces one
 * element longer), every interior cut moved by +misalign elements (clamped),
 * and each rank's pieces concatenated in its local space (FSDP units / DDP
 * buckets, "FSDP wrapping granularity").  out may be NULL to query the count:
 * *nseg is the capacity on entry and the number of segments on return. */
dp_status_t dp_layout_even(int64_t psi, int32_t n, int64_t bucket, int32_t misalign, dp_segment_t* out,
                           int32_t* nseg);

/* The part of a layout inside the global range [lo, hi) of its parameter
 * space, as a layout of its own: the slice one GPU holds when the space is
 * split into contiguous slices (the step flags above).  Segment pieces inside
 * [lo, hi) in order, with global_off rebased to lo and local_off rebased to
 * local_base[owner], the lowest local index of that owner's pieces in the
 * slice (0 for an owner with none); the slice layout has psi = hi - lo, the
 * same stage and n.  So the slice's shard array of rank s holds elements
 * [local_base[s], local_base[s] + dp_shard_len(slice, s)) of rank s's whole
 * shard array (stage 0: elements [lo, hi) of the full arrays), and its
 * gradient and replica buffers hold elements [lo, hi).  out may be NULL to
 * query the count: *nseg is the capacity on entry and the count on return;
 * local_base (n entries) may be NULL.  Not on the pages: a host-side layout
 * helper.  DP_ERR_INVALID_ARG for a bad layout or range. */
dp_status_t dp_layout_slice(const dp_layout_t* layout, int64_t lo, int64_t hi, dp_segment_t* out, int32_t* nseg,
                            int64_t* local_base);

/* Local length of rank's shard arrays (end of its furthest segment); -1 on
 * error.  Not on the pages: a size query of the layout above. */
int64_t dp_shard_len(const dp_layout_t* layout, int32_t rank);

/* Bytes of device workspace that dp_step needs when the caller passes ws
 * instead of gbar_shard pointers: the n averaged-gradient shards, each
 * 256-byte aligned.  0 on error.  The shards are the reduce-scatter's output
 * ("Distributed Training: Split along the Four Axes", ZeRO/FSDP paragraph:
 * the reduce-scatter leaves each rank only its own shard of the gradient). */
size_t dp_workspace_size(const dp_layout_t* layout);

/* Floats per rank in a dp_accumulate accumulator: psi (plain) or 2 psi
 * (compensated, interleaved hi, lo).  Not on the pages: a size query. */
size_t dp_acc_elems(int64_t psi, int32_t sum_mode);

/* B_global = b x n x a: tensor and pipeline degrees are not multiplied in
 * ("Distributed Training", data-parallel formula and 3D paragraph).  -1 on a
 * negative input or overflow. */
int64_t dp_global_batch(int64_t b, int32_t n, int32_t a);

/* Model-state bytes per rank for mixed-precision Adam at 16 bytes per
 * parameter (2 bf16 parameter, 2 bf16 gradient, 12 fp32 master + m + v;
 * "Data vs Tensor vs Pipeline Parallelism", 16 bytes per parameter, ZeRO-3
 * 16 Psi / N), stage 0-3 as in ZeRO: out[0] parameter bytes, out[1] gradient
 * bytes, out[2] optimizer-state bytes, out[3] total.  Even split, fractional. */
dp_status_t dp_memory_model(int32_t stage, int64_t psi, int32_t n, double out[4]);

/* Ring traffic of one training step per rank with even shards: out[0] bytes
 * sent (= received) per rank, out[1] ring steps, out[2] ratio to a plain-DP
 * all-reduce of the gradient at the same wire size.  Stage 0: all-reduce of
 * the gradient (2(N-1)/N x gradient bytes, 2(N-1) steps); stages 1-2:
 * reduce-scatter of gradients + all-gather of parameters; stage 3: plus a
 * second parameter all-gather for backward (1.5x when wire sizes match). */
dp_status_t dp_traffic_model(int32_t stage, int64_t psi, int32_t n, int32_t wire_bytes_grad,
                             int32_t wire_bytes_param, double out[3]);

/* Not on the pages: upper bound, in nanoseconds, of every device-side wait of the kernels
 * (default 2 s).  A wait that runs out records DP_ERR_TIMEOUT in
 * state.error and the kernel returns; the step is skipped. */
void dp_set_wait_timeout_ns(uint64_t ns);
uint64_t dp_get_wait_timeout_ns(void);

/* Number of kernels this library has launched in this process (not on the pages). */
uint64_t dp_kernel_launches(void);

/* ---- device entry points -------------------------------------------------- */

/* Sets *d_state to t = 0, beta powers 1, no skip, no error (one kernel).
 * Not on the pages: initialisation of the library's step state. */
dp_status_t dp_state_init(dp_step_state_t* d_state, dp_stream_t stream);

/* Staged accumulation of one micro-step (data-parallel paragraphs: each rank
 * sums its a micro-step gradients locally).  For every rank r < n:
 *   first != 0:  acc[r] := g[r]          else  acc[r] += g[r]   (left to right)
 * acc[r]: device, dp_acc_elems(psi, sum_mode) floats, element i at acc[r][i]
 * (plain) or (hi, lo) at acc[r][2i], acc[r][2i+1] (compensated, TwoSum);
 * g[r]: device, psi bf16. */
dp_status_t dp_accumulate(float* const* acc, const uint16_t* const* g, int64_t psi, int32_t n, int32_t first,
                          int32_t sum_mode, dp_stream_t stream);

/* Staged reduce-scatter + average + unscale + non-finite check ("Data vs
 * Tensor vs Pipeline Parallelism", "Data parallelism: split the batch": the
 * ring all-reduce is a reduce-scatter then an all-gather, and sharded data
 * parallelism keeps only the reduce-scatter's shard; "Distributed Training:
 * Split along the Four Axes", data-parallel averaging paragraph: gbar =
 * sum_r g_r / n).  For each segment (owner s) and element i in it:
 *   p = acc_{s+1} + acc_{s+2} + ... + acc_s   (ring order: the chunk starts at
 *       rank s+1 and reaches its owner after n-1 hops; compensated mode adds
 *       (hi, lo) pairs with TwoSum and ends with hi + lo; with DP_ORDER_TREE
 *       the acc_r are added in the tree order instead)
 *   gbar_shard[s][local_off + (i - global_off)] = fl32(p * fl32(1 / (n S)))
 * then state.found_inf / state.nonfinite report whether any gbar is inf/NaN.
 * gbar_shard[s]: device, dp_shard_len(layout, s) floats.  loss_scale S > 0. */
dp_status_t dp_reduce_scatter_avg(float* const* gbar_shard, const float* const* acc, const dp_layout_t* layout,
                                  float loss_scale, int32_t sum_mode, dp_step_state_t* d_state, dp_stream_t stream);

/* Per-micro-step reduce-scatter: the memory-saving ZeRO-2 form, in which each
 * micro-step's gradients are reduce-scattered as soon as they exist and summed
 * into the owner's shard accumulator, so no full-length per-rank gradient
 * accumulator exists ("Distributed Training: Split along the Four Axes",
 * ZeRO/FSDP paragraph: stage 2 also shards gradients; "Data vs Tensor vs
 * Pipeline Parallelism", sharded data parallelism).  Call it for k = 0..a-1,
 * in order, on one stream; then dp_step_update with the same gbar_shard / ws.
 * For an element of segment owner s:
 *   p_k = g_{s+1,k} + g_{s+2,k} + ... + g_{s,k}   (ring order, one micro-step)
 *   A   = ((p_0 + p_1) + ...) + p_{a-1}           (in the owner's accumulator)
 *   gbar_shard[s][local] = fl32(A * fl32(1 / (n S)))   (written by the k = a-1 call)
 * Compensated mode carries TwoSum error terms in both sums ((H, e) =
 * TwoSum(A_H, p_H), A_L = (A_L + e) + p_L) and ends with A_H + A_L.  This
 * order differs from dp_step's (all of a rank's micro-steps before the next
 * rank), so results agree with it to rounding, not bit for bit (for a = 1 the
 * two perform the same operations).  The k = a-1 call also
 * counts non-finite gbar values and, like dp_step_reduce, publishes found_inf
 * and advances t and the beta powers unless found.
 * g: n device pointers, micro-step k of every rank, each psi bf16.
 * acc_shard: n device shards of dp_acc_elems(dp_shard_len(layout, s),
 *   sum_mode) floats (hi, or interleaved (hi, lo) pairs when compensated) at
 *   local index; the caller's memory, overwritten at k = 0; unused (may be
 *   NULL) when a = 1.
 * gbar_shard / ws: as for dp_step_reduce; used by the k = a-1 call only.
 * Ring order only (DP_ORDER_TREE is DP_ERR_INVALID_ARG).  Accepts
 * DP_DEFER_COMMIT and DP_DEVICE_SCALE (they act on the k = a-1 call). */
dp_status_t dp_reduce_scatter_micro(float* const* acc_shard, float* const* gbar_shard, void* ws,
                                    const uint16_t* const* g, int32_t k, int32_t a, const dp_layout_t* layout,
                                    dp_adam_t adam, float loss_scale, int32_t sum_mode, dp_step_state_t* d_state,
                                    dp_stream_t stream);

/* Staged partitioned Adam ("Distributed Training: Split along the Four
 * Axes", memory-budget paragraph: an fp32 master copy and Adam's two moments
 * per parameter; ZeRO/FSDP paragraph: each rank updates only its shard, and
 * sharding does not change the update).  The Adam equations themselves are
 * not on the pages (standard Adam, see the file comment).
 * Unless state.found_inf: t += 1, beta powers
 * advance, then for every element of every shard (stage 0: of every rank's
 * full arrays, with the owner's gbar):
 *   m = b1 m + (1-b1) g ; v = b2 v + (1-b2) g^2 ;
 *   theta -= (lr / (1 - b1^t)) m / (sqrt(v) / sqrt(1 - b2^t) + eps)
 * master/m/v[s]: device fp32 shard arrays (stage 0: psi elements);
 * gbar_shard[s]: as written by dp_reduce_scatter_avg. */
dp_status_t dp_adam_shard(float* const* master, float* const* m, float* const* v, const float* const* gbar_shard,
                          const dp_layout_t* layout, dp_adam_t adam, dp_step_state_t* d_state, dp_stream_t stream);

/* Staged all-gather ("Distributed Training: Split along the Four Axes",
 * ZeRO/FSDP paragraph: the updated parameter shards are all-gathered so every
 * rank again holds the whole model; data-parallel paragraph: the replicas stay
 * identical): unless state.found_inf, replicas[r][i] = bf16_rne(theta_i)
 * for every rank r (stage 0: rank r's own master).  replicas[r]: device, psi bf16. */
dp_status_t dp_allgather_params(uint16_t* const* replicas, const float* const* master, const dp_layout_t* layout,
                                const dp_step_state_t* d_state, dp_stream_t stream);

/* The fused step: dp_step_reduce then dp_step_update (two kernels).
 * It is the whole data-parallel step of "Distributed Training: Split along the
 * Four Axes" (data-parallel paragraphs: accumulate a micro-steps, one
 * all-reduce, gbar = sum / n; ZeRO/FSDP paragraph: sharded optimizer state)
 * with the ring of "Data vs Tensor vs Pipeline Parallelism", "Data
 * parallelism: split the batch".
 * grads: host array of n*a device pointers, rank-major (grads[r*a + k] is
 * micro-step k of rank r), each psi bf16.  Per element the gradient is summed
 * in a fixed order -- ranks in ring order s+1, ..., s for the owner s, each
 * rank's micro-steps k = 0..a-1 (or in the tree order of DP_ORDER_TREE) -- so
 * results are bit-identical run to run.  Plain: each rank's micro-steps are
 * summed first, then the ranks' sums, exactly as dp_accumulate +
 * dp_reduce_scatter_avg + dp_adam_shard + dp_allgather_params compute it.
 * Compensated (ring order): one (hi, lo) pair through all n*a inputs, which
 * agrees with the staged calls (one pair per rank, then the ranks' pairs) to
 * rounding.  gbar_shard: n device shards of dp_shard_len floats, or
 * NULL to carve them from ws (dp_workspace_size bytes, 256-byte aligned).
 * If any reduced value is not finite (or a wait timed out) master, m, v,
 * replicas and t are left bit-for-bit unchanged. */
dp_status_t dp_step(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                    const uint16_t* const* grads, int32_t a, const dp_layout_t* layout, dp_adam_t adam,
                    float loss_scale, int32_t sum_mode, float* const* gbar_shard, void* ws,
                    dp_step_state_t* d_state, dp_stream_t stream);

/* dp_step with the step's gradients in host memory (same passages as dp_step;
 * the copies are not on the pages): the end-to-end call of a
 * loop whose gradients arrive on the host.  On `stream`, in order: the n*a
 * host buffers host_grads[q] (psi bf16 each, rank-major like grads) are
 * copied into the caller's device buffers grads[q] (one cudaMemcpyAsync
 * each), dp_step runs on them, and, if host_state is not NULL, the 64-byte
 * step state is copied back to host_state (read found_inf / t there after a
 * stream synchronize).  Every argument is checked before anything is
 * queued; results are those of dp_step on the same gradients.  host_grads
 * and host_state should be pinned (cudaHostAlloc / cudaHostRegister) for the
 * copies to be asynchronous and run at the link's rate; they must stay valid
 * until the stream has passed the copies.  Errors: those of dp_step, and
 * DP_ERR_CUDA if a copy cannot be queued. */
dp_status_t dp_step_from_host(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                              const uint16_t* const* host_grads, uint16_t* const* grads, int32_t a,
                              const dp_layout_t* layout, dp_adam_t adam, float loss_scale, int32_t sum_mode,
                              float* const* gbar_shard, void* ws, dp_step_state_t* d_state,
                              dp_step_state_t* host_state, dp_stream_t stream);

/* First half of dp_step (one kernel; same passages as dp_step):
 * accumulate + ring reduce-scatter +
 * average + unscale + non-finite check, gbar into the shards; the last CTA
 * publishes found_inf / nonfinite and, unless found, advances t and the
 * beta powers for the update that follows.  Accepts DP_DEFER_COMMIT and
 * DP_DEVICE_SCALE in sum_mode. */
dp_status_t dp_step_reduce(float* const* gbar_shard, void* ws, const uint16_t* const* grads, int32_t a,
                           const dp_layout_t* layout, dp_adam_t adam, float loss_scale, int32_t sum_mode,
                           dp_step_state_t* d_state, dp_stream_t stream);

/* Second half of dp_step (one kernel; same passages as dp_adam_shard and
 * dp_allgather_params): unless found_inf, Adam on every shard
 * and the bf16 all-gather into every replica, reading the gbar shards and the
 * beta powers dp_step_reduce left. */
dp_status_t dp_step_update(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                           const float* const* gbar_shard, void* ws, const dp_layout_t* layout, dp_adam_t adam,
                           const dp_step_state_t* d_state, dp_stream_t stream);

/* Sets the device-resident dynamic loss scale of *d_state to `scale` (> 0,
 * finite) and good_steps to 0 (one kernel).  Other fields are untouched.
 * ("Distributed Training: Split along the Four Axes", checkpoint and
 * evaluation paragraphs name the loss scale as training state.) */
dp_status_t dp_scaler_init(dp_step_state_t* d_state, float scale, dp_stream_t stream);

/* dp_step with a dynamic loss scale ("Distributed Training: Split along the
 * Four Axes", checkpoint and evaluation paragraphs: the loss scale is state
 * to keep and align; the growth/back-off rule is not on the pages, see
 * dp_scaler_t): the reduction unscales by the scale held
 * in d_state->loss_scale (read on the device, so no host round trip), and the
 * last CTA of the reduction updates that scale with `scaler` once the skip
 * decision is known.  A scale that is not positive and finite, or whose
 * 1 / (n S) is not a normal fp32 number, records DP_ERR_INVALID_ARG in
 * d_state->error and the step is skipped.  Other arguments as dp_step. */
dp_status_t dp_step_scaled(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                           const uint16_t* const* grads, int32_t a, const dp_layout_t* layout, dp_adam_t adam,
                           const dp_scaler_t* scaler, int32_t sum_mode, float* const* gbar_shard, void* ws,
                           dp_step_state_t* d_state, dp_stream_t stream);

/* The fused step in ONE pass over memory (same passages as dp_step; the
 * skip rule of the file comment kept by double-buffering the state, which the
 * pages do not describe) (one reduce-and-update kernel, plus a
 * repair kernel that does work only on a skipped step).  The optimizer state
 * is double-buffered: master, m and v are host arrays of 2n device pointers,
 * set 0 (entries 0..n-1) and set 1 (entries n..2n-1), each like dp_step's.
 * d_state->cur_set (0 after dp_state_init) names the current set; the kernel
 * reads it and writes the other set, and the reduction's last CTA makes the
 * other set current only if no value was non-finite.  gbar never reaches
 * memory, so the step streams the single-pass minimum 2na + 24 + 2n bytes per
 * parameter instead of dp_step's 2na + 32 + 2n.  Replicas are written in
 * place while the skip decision is still open; on a skipped step the repair
 * kernel rewrites them as bf16_rne of the (unchanged) current master, so a
 * skipped step leaves the replicas as they were provided they held
 * bf16_rne(master) before it -- the invariant every applied step
 * establishes.  Results are bit-identical to dp_step in the same order (ring
 * or DP_ORDER_TREE).  Stages 1-3 only.
 * Accepts DP_DEFER_COMMIT (then only the pass is launched; the state set is
 * not flipped and the replicas not repaired until dp_commit_single_pass) and
 * DP_DEVICE_SCALE in sum_mode. */
dp_status_t dp_step_single_pass(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                                const uint16_t* const* grads, int32_t a, const dp_layout_t* layout, dp_adam_t adam,
                                float loss_scale, int32_t sum_mode, dp_step_state_t* d_state, dp_stream_t stream);

/* dp_step_single_pass with the step's gradients in host memory, like
 * dp_step_from_host: on `stream`, the n*a host buffers host_grads[q] are
 * copied into the device buffers grads[q] (one cudaMemcpyAsync each), the
 * single pass runs on them, and, if host_state is not NULL, the 64-byte state
 * is copied back to host_state.  Arguments are checked before anything is
 * queued; host buffers should be pinned and stay valid until the stream has
 * passed the copies.  Results are those of dp_step_single_pass.  (Same
 * passages as dp_step; the copies are not on the pages.) */
dp_status_t dp_step_single_pass_from_host(uint16_t* const* replicas, float* const* master, float* const* m,
                                          float* const* v, const uint16_t* const* host_grads, uint16_t* const* grads,
                                          int32_t a, const dp_layout_t* layout, dp_adam_t adam, float loss_scale,
                                          int32_t sum_mode, dp_step_state_t* d_state, dp_step_state_t* host_state,
                                          dp_stream_t stream);

/* Commits a step whose reduction ran with DP_DEFER_COMMIT, once found_inf in
 * *d_state holds the decision of every slice (the caller's maximum over the
 * slices): unless found_inf (or a recorded device error), t += 1 and the beta
 * powers advance with adam.beta1 / beta2; with a scaler, the device-resident
 * loss scale then follows its policy (see dp_scaler_t), NULL leaves it.  One
 * kernel; call dp_step_update after it.  ("Distributed Training: Split along
 * the Four Axes", data-parallel paragraph: all ranks apply one update.) */
dp_status_t dp_commit_step(dp_step_state_t* d_state, dp_adam_t adam, const dp_scaler_t* scaler, dp_stream_t stream);

/* dp_commit_step for dp_step_single_pass with DP_DEFER_COMMIT: the commit also
 * makes the set the pass wrote current unless found_inf, and on a skipped step
 * rewrites the replicas from the (unchanged) current master, as the single
 * pass's own repair does.  replicas, master (2n pointers) and layout as for
 * dp_step_single_pass.  Two kernels. */
dp_status_t dp_commit_single_pass(uint16_t* const* replicas, float* const* master, const dp_layout_t* layout,
                                  dp_adam_t adam, const dp_scaler_t* scaler, dp_step_state_t* d_state,
                                  dp_stream_t stream);

/* Reads found_inf and error of *d_state into host ints after synchronising
 * the stream (the one blocking call).  skipped / err may be NULL.  Not on the
 * pages: a host-side read of the step's device-resident status. */
dp_status_t dp_read_status(const dp_step_state_t* d_state, int32_t* skipped, int32_t* err, dp_stream_t stream);

/* Self-test of the bounded wait (not on the pages; the failure handling of
 * every device wait): launches one block that waits on a barrier
 * nothing will complete; after timeout_ns it records DP_ERR_TIMEOUT in
 * d_state->error and returns, leaving the context usable. */
dp_status_t dp_selftest_wait_timeout(dp_step_state_t* d_state, uint64_t timeout_ns, dp_stream_t stream);

/* ---- allocation-free variant ------------------------------------------------ */

/* Size of the scratch array compiled into the library for dp_step_static. */
#define DP_STATIC_SCRATCH_BYTES (64ll * 1024 * 1024)

/* dp_step without caller-provided scratch.  The distributed-training pages
 * have no counterpart to this call; it exists for callers that cannot
 * allocate device memory themselves -- a plugin inside a runtime that owns
 * and pre-plans all device memory, a loop that must not allocate after
 * start-up, or code running while another allocator holds a lock.
 * The averaged-gradient shards live in a fixed 64 MiB array inside the
 * library (DP_STATIC_SCRATCH_BYTES, held on every GPU that loads the library
 * until the process exits): the layout's dp_workspace_size must not exceed
 * it (about 16 million parameters), else DP_ERR_INVALID_ARG and nothing is
 * launched.  Arguments, results and errors are those of dp_step; no call
 * allocates or frees memory.  Every call looks up the array's device address
 * in the current context (cudaGetSymbolAddress; the first call on a device
 * also loads the library's kernels there).  All calls share the array and it
 * keeps the last call's contents; calls whose kernels overlap on the GPU race
 * on it, so order them (one stream, or events). */
dp_status_t dp_step_static(uint16_t* const* replicas, float* const* master, float* const* m, float* const* v,
                           const uint16_t* const* grads, int32_t a, const dp_layout_t* layout, dp_adam_t adam,
                           float loss_scale, int32_t sum_mode, dp_step_state_t* d_state, dp_stream_t stream);

/* ---- sharded checkpoints ------------------------------------------------------ */

/* A checkpoint of the optimizer state, stored by shard, that loads into any
 * layout of the same psi: another n, another stage, other segments.
 * ("Distributed Training: Split along the Four Axes", checkpoint paragraphs:
 * ZeRO/FSDP state is saved in shards per rank; a restart either reshards to
 * the new world size or refuses; the write is temporary files plus an atomic
 * manifest; the loss scale and the parallel layout are saved with it.)
 *
 * On disk, under root/:
 *   <tag>/shard_<r>.bin  rank r's master, m and v, each dp_shard_len(layout, r)
 *                        fp32 values in local order (holes of the local space
 *                        as zeros), after a 24-byte header
 *   <tag>/state.bin      the dp_step_state_t: t, beta powers, error, loss scale,
 *                        good_steps; the per-step and kernel fields cleared
 *   <tag>/layout.bin     the layout it was saved with
 *   <tag>/user.bin       the caller's bytes (LR schedule, RNG, data cursor ...)
 *   <tag>/MANIFEST       each file's size and FNV-1a 64-bit checksum
 *   LATEST               the tag of the newest complete checkpoint
 * dp_checkpoint_save writes <tag>.partial/, syncs every file, renames it to
 * <tag>/ and then replaces LATEST by a rename, so a reader sees either the old
 * or the new checkpoint, never part of one.  A save that fails leaves
 * <tag>.partial/ behind (a later save of the same tag overwrites it) and
 * LATEST unchanged.
 *
 * master/m/v: arrays of n pointers laid out as for dp_step (stage 0: full
 * length on every rank, rank r's segments are saved from rank r's copy;
 * stages 1-3: shard arrays).  host_buffers = 0: they and d_state are device
 * memory; the call synchronises `stream` first, then copies through a pinned
 * host chunk on `stream` and returns when all copies are done.
 * host_buffers = 1: they are host memory and no CUDA call is made.
 * For dp_step_single_pass, pass the current set (state.cur_set); the loaded
 * state has cur_set = 0, so load into set 0.
 * Errors: DP_ERR_INVALID_ARG (bad layout, tag, NULL pointers; nothing
 * written), DP_ERR_IO (with dp_last_error() naming the file), DP_ERR_CUDA.
 * tag: 1..200 characters of [A-Za-z0-9_.-], not starting with '.'; an
 * existing <tag>/ is an error. */
dp_status_t dp_checkpoint_save(const char* root, const char* tag, const dp_layout_t* layout,
                               float* const* master, float* const* m, float* const* v,
                               const dp_step_state_t* d_state, const void* user_meta, uint64_t user_meta_bytes,
                               int32_t host_buffers, dp_stream_t stream);

/* Loads the checkpoint `tag` (NULL: the one LATEST names) into `layout`
 * (same passages as dp_checkpoint_save: a restart reshards to the new world
 * size or refuses),
 * which must have the saved psi and may differ in everything else.  Every
 * element lands at its global position's place in the new layout, so the
 * result is a bit-exact permutation of what was saved.  verify = 1 checks
 * every file against the manifest first (reads the checkpoint twice).
 * user_meta_bytes: NULL to skip the user bytes; else in: the capacity of
 * user_meta, out: the saved size (with user_meta NULL only the size is
 * returned).  Errors as for dp_checkpoint_save; DP_ERR_INVALID_ARG also for
 * a psi mismatch or a too-small user_meta.  On an error the destination may
 * be partly written. */
dp_status_t dp_checkpoint_load(const char* root, const char* tag, const dp_layout_t* layout,
                               float* const* master, float* const* m, float* const* v, dp_step_state_t* d_state,
                               void* user_meta, uint64_t* user_meta_bytes, int32_t host_buffers, int32_t verify,
                               dp_stream_t stream);

/* The saved layout of checkpoint `tag` (NULL: LATEST; same passages as
 * dp_checkpoint_save: the parallel layout is saved with the state) and the size of its
 * user bytes: any output may be NULL; seg receives the nseg segments if
 * seg_cap is large enough (else DP_ERR_INVALID_ARG).  verify as for
 * dp_checkpoint_load.  Reads no shard data unless verify is set. */
dp_status_t dp_checkpoint_info(const char* root, const char* tag, int32_t verify, int32_t* stage, int32_t* n,
                               int64_t* psi, int32_t* nseg, dp_segment_t* seg, int32_t seg_cap,
                               uint64_t* user_meta_bytes);

#ifdef __cplusplus
}
#endif

#endif /* DPSTEP_H */
