/*
 * cz.h -- C-ABI of libcz: the alpha-Balanced ZeRO-1 partition planner and the
 * local Muon step that one data-parallel rank runs on the whole tensors it owns.
 *
 * Source of the operations: "Canzona: A Unified, Asynchronous, and Load-Balanced
 * Framework for Distributed Matrix-based Optimizers" (arXiv 2602.06079), as
 * summarised on the paper-graph-ui page, section 3.4:
 *   - "Paradigm 3: Static Partitioning", Eq. 1 (start-index ownership rule);
 *   - "The DP Load-Balance Optimization Problem" (J_DP, J_Comm, Phi_i(u));
 *   - "The alpha-Balanced Greedy LPT Algorithm (Algorithm 1)";
 *   - "Runtime Static-Layout Enforcement": the optimizer step runs on each rank's
 *     intervals [s_{i,r-1}, s_{i,r}) with zero communication.
 * The Muon step itself (momentum, Frobenius normalisation, Newton-Schulz,
 * shape scale, apply) is the standard Muon update; the pages only name it
 * (section 2: Muon orthogonalises weight matrices with Newton-Schulz iterations;
 * section 4.1: Delta W = Muon_step(G, States_local)).
 *
 * Conventions for every call:
 *   - Every function returns a status: CZ_OK (0) or a negative CZ_ERR_* code.
 *     No call aborts, traps or prints.  Invalid arguments are rejected on the
 *     host before any GPU work is enqueued.
 *   - Ranks are 0-based.  Sizes are element counts (int64).
 *   - Host arrays (numels, offsets, shapes, ...) are read during the call only;
 *     the library keeps no pointer to them.
 *   - Device buffers are owned by the caller.  The library owns only cz_plan
 *     objects (host heap) and, when the caller passes no workspace, one cached
 *     device workspace per device (see cz_muon_step).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     GPU calls are asynchronous on it; CZ_OK means "enqueued".
 */
#ifndef CZ_H
#define CZ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CZ_OK                  0
#define CZ_ERR_INVALID        -1  /* bad argument (sizes, ranks, alpha, shapes, ...)   */
#define CZ_ERR_CUDA           -2  /* a CUDA runtime/driver call failed                 */
#define CZ_ERR_NOMEM          -3  /* workspace too small or allocation failed          */
#define CZ_ERR_PLAN_MISMATCH  -4  /* offsets/shapes do not describe the planned tensors */
#define CZ_ERR_TIMEOUT        -5  /* a device-side wait ran out (reported by status)   */
#define CZ_ERR_DEVICE_CHECK   -6  /* a device-side bounds/descriptor check failed      */
#define CZ_ERR_UNSUPPORTED    -7  /* no sm_103a device, or a feature not built         */

typedef struct cz_plan cz_plan;   /* opaque, immutable after creation, thread-safe to share */

/* Bucket formation (section 3.4, "Problem setup": buckets are ordered,
 * non-splittable parameter sequences).  Walks numels[0..n_params) in buffer
 * order and closes a bucket as soon as its element count is >= cap_elems; a
 * trailing partial bucket is kept.  counts_out must hold n_params entries;
 * *n_buckets_out receives the number written. */
int cz_make_buckets(const int64_t* numels, int64_t n_params, int64_t cap_elems,
                    int64_t* counts_out, int64_t* n_buckets_out);

/* Algorithm 1, alpha-Balanced Greedy LPT, cost W(p) = numel(p).
 * numels: n_params positive element counts in buffer order.
 * bucket_sizes: n_buckets positive parameter counts, consecutive, summing to n_params.
 * R >= 1 ranks, alpha in [0, 1].  Buckets are processed in LPT order (W desc,
 * index asc); per bucket, deficits d_r = max(0, mu - L_r), target
 * v* = (1-alpha)/R + alpha d_r/D (1/R when D = 0), cumulative target C, and the
 * cut s_{k,r} = argmin_{u in [s_{k,r-1}, n_k]} |Phi_k(u) - C| (ties: smaller u);
 * the last rank takes the remainder.  IEEE double, no contraction: bit-exact
 * with the reference planner.  *out receives a new plan (free with cz_plan_free). */
int cz_plan_partition(const int64_t* numels, int64_t n_params,
                      const int64_t* bucket_sizes, int64_t n_buckets,
                      int32_t R, double alpha, cz_plan** out);

/* Algorithm 1 with an explicit cost W(p) per parameter (costs[n_params], positive),
 * e.g. the Newton-Schulz FLOPs of each tensor -- the non-linear cost the pages'
 * appendix D.5 compares with numel.  Loads, deficits and cut targets are in cost
 * units; shard sizes (elem cuts, J_Comm) stay in elements.  costs = NULL is
 * cz_plan_partition. */
int cz_plan_partition_cost(const int64_t* numels, const int64_t* costs, int64_t n_params,
                           const int64_t* bucket_sizes, int64_t n_buckets,
                           int32_t R, double alpha, cz_plan** out);

/* Eq. 1, the start-index split: parameter p at element offset o inside bucket
 * B_i goes to rank floor(o * R / |B_i|), i.e. r*S <= o < (r+1)*S, S = |B_i|/R. */
int cz_plan_naive(const int64_t* numels, int64_t n_params,
                  const int64_t* bucket_sizes, int64_t n_buckets,
                  int32_t R, cz_plan** out);

void cz_plan_free(cz_plan* plan);   /* NULL is accepted */

/* Sizes of a plan, so that callers can size the query buffers below. */
int cz_plan_info(const cz_plan* plan, int64_t* n_params, int64_t* n_buckets, int32_t* R);

/* owner_out[n_params]: the 0-based rank that owns each parameter. */
int cz_plan_owner(const cz_plan* plan, int32_t* owner_out);

/* Slicing vectors s_i in physical bucket order, n_buckets*(R+1) entries each:
 * param_cuts in parameter indices within the bucket, elem_cuts = Phi_i(s_{i,r})
 * (element offsets within the bucket).  Either pointer may be NULL. */
int cz_plan_cuts(const cz_plan* plan, int64_t* param_cuts, int64_t* elem_cuts);

/* load_out[R]: load owned by each rank, sum over buckets of L_{i,r}, in cost
 * units (elements for cz_plan_partition / cz_plan_naive). */
int cz_plan_rank_load(const cz_plan* plan, int64_t* load_out);

/* elems_out[R]: elements (memory) owned by each rank. */
int cz_plan_rank_elems(const cz_plan* plan, int64_t* elems_out);

/* R_LB = max_r L_r / mean; J_DP = max_r |L_r - mu| (Eq. 2); J_Comm =
 * sum_i sum_r |S_{i,r} - |B_i|/R|.  Any pointer may be NULL. */
int cz_plan_metrics(const cz_plan* plan, double* r_lb, double* j_dp, double* j_comm);

/* TP Micro-Group Construction with Greedy Rollback and the MinHeapSolver
 * (section 3.4, "The TP Hierarchical Partitioning and Scheduling"): the
 * n_params TP-split tensors with positive costs W(p) are sorted by (W, ID)
 * descending and packed into groups in that order; a tensor joins the current
 * group if the LPT assignment of the group to R host ranks (min-heap of
 * (load, rank), ties to the smaller rank) keeps the largest rank load <= c_max,
 * otherwise the group is finalised and the tensor starts the next one (a tensor
 * whose cost alone exceeds c_max forms a group of its own).
 *   group_out[n_params]: group index of each tensor, groups numbered in order;
 *   host_out[n_params]:  host rank of each tensor within its group;
 *   *n_groups_out:       number of groups.
 * Integer arithmetic only: identical on every rank. */
int cz_plan_microgroups(const int64_t* costs, int64_t n_params, int32_t R, int64_t c_max,
                        int32_t* group_out, int32_t* host_out, int64_t* n_groups_out);

/* Variable-size collectives around the step (section 3.4, "Runtime Static-Layout
 * Enforcement": bucket B_i is reduce-scattered and all-gathered with per-rank
 * sizes S_{i,r} taken from the partition map).  Primitives that need equal
 * counts per rank take R blocks of `block` >= max_r S_{i,r} elements:
 *   cz_bucket_pack:   padded[r*block + j] = bucket[elem_cuts[r] + j] for j < S_{i,r},
 *                     0 for S_{i,r} <= j < block  (before a ReduceScatter);
 *   cz_bucket_unpack: bucket[elem_cuts[r] + j] = padded[r*block + j] for j < S_{i,r}
 *                     (after an AllGather); padding is ignored.
 * bucket / padded: device buffers of elem_bytes-byte elements (1, 2, 4 or 8;
 * values are copied bit for bit).  elem_cuts: host, R+1 element offsets within the
 * bucket (one row of cz_plan_cuts' elem_cuts), elem_cuts[0] = 0, non-decreasing.
 * R <= 1024.  Asynchronous on `stream`. */
int cz_bucket_pack(const void* bucket, int32_t elem_bytes, const int64_t* elem_cuts, int32_t R,
                   int64_t block, void* padded, void* stream);
int cz_bucket_unpack(const void* padded, int32_t elem_bytes, const int64_t* elem_cuts, int32_t R,
                     int64_t block, void* bucket, void* stream);

/* Standalone scale-and-apply of updates already in the parameters' layout: the
 * apply the Muon step fuses into its last Newton-Schulz epilogue, as a kernel of
 * its own.  Section 3.4 of the summary page gives the rule
 * W_{t+1} = W_t - eta * MatrixOp(W_t, grad W_t) ("The Atomicity Constraint ...")
 * and, as stage 4 of the TP micro-group lifecycle ("The TP Task Abstraction"),
 * the element-wise local add of received update shards, P_local += Delta W_local
 * (lr = -1, shape_scale = 0).
 *   flat_param:  fp32 device buffer (4-byte aligned), updated in place;
 *   param_bf16:  nullable bf16 device copy in the same flat layout, written as
 *                RNE(new fp32 value);
 *   flat_update: fp32 device buffer U in the same flat layout (tensor i at
 *                [offsets[i], offsets[i] + rows*cols), row-major rows x cols);
 *   offsets:     n_tensors host int64; shapes: 2*n_tensors host int64 (rows, cols).
 * Per tensor: coef = fp32(lr * sqrt(max(1, rows/cols))) (coef = fp32(lr) when
 * shape_scale = 0), then W <- fp32(W - fp32(coef * U)) element by element (two
 * roundings, the same arithmetic as the fused apply).  Bytes outside the listed
 * tensors are not touched.  Overlapping tensors, non-positive shapes, negative
 * offsets, a non-finite lr or shape_scale not 0/1 give CZ_ERR_INVALID before any
 * launch; n_tensors = 0 is a no-op.  Asynchronous on `stream`; requires an
 * sm_103a device (CZ_ERR_UNSUPPORTED otherwise). */
int cz_apply_update(float* flat_param, void* param_bf16, const float* flat_update,
                    const int64_t* offsets, const int64_t* shapes, int64_t n_tensors,
                    float lr, int32_t shape_scale, void* stream);

/* Options of the Muon step.  Fill with cz_step_opts_default, then override. */
typedef struct {
  int32_t nesterov;        /* 1: u = g + mu*m (default); 0: u = m                       */
  float   eps;             /* added to ||u||_F (default 1e-7)                           */
  float   a, b, c;         /* Newton-Schulz coefficients (default 3.4445, -4.7750, 2.0315) */
  int32_t grad_is_bf16;    /* flat_grad holds bf16 values instead of fp32              */
  void*   param_bf16;      /* nullable: bf16 copy of the parameters, same flat layout;
                              written as RNE(new fp32 master) for owned tensors        */
  void*   workspace;       /* nullable: caller-owned device scratch of workspace_bytes
                              (>= cz_workspace_size, 256-byte aligned; its first 256
                              bytes -- the status word -- must be zero before first
                              use).  NULL: the library's cached one                     */
  size_t  workspace_bytes;
  float*  debug_update_out;/* nullable: fp32 flat buffer (param layout); receives
                              lr*sqrt(max(1,rows/cols))*X_K for owned tensors          */
  const float* lr_device;  /* nullable: a device float (4-byte aligned) that the apply
                              reads in place of the lr argument, when the launch runs;
                              a step captured in a CUDA graph then follows a schedule
                              written there before each replay                         */
} cz_step_opts;

void cz_step_opts_default(cz_step_opts* opts);

/* Device scratch needed by cz_muon_step_ex for `rank`'s shard under `plan`
 * (bf16 Newton-Schulz operands, per-tensor norms, tile lists, status word).
 * shapes: 2*n_params host int64 (rows, cols per parameter). */
int cz_workspace_size(const cz_plan* plan, int32_t rank, const int64_t* shapes, size_t* bytes);

/* One Muon step over the tensors that `plan` assigns to `rank`
 * (section 3.4, "Runtime Static-Layout Enforcement", phase 2).
 *   flat_param: fp32 master weights, flat_grad: fp32 (or bf16, see opts),
 *   flat_mom: fp32 momentum -- device buffers in one flat layout, each 16-byte
 *   aligned (a bf16 gradient, the bf16 parameter copy: 8-byte aligned; the
 *   debug output: 16-byte aligned; CZ_ERR_INVALID otherwise); parameter p
 *   occupies [offsets[p], offsets[p] + rows*cols) row-major (rows x cols = out x in).
 *   offsets: n_params host int64; shapes: 2*n_params host int64.
 *   Only tensors with owner == rank are read or written; every other byte of
 *   every buffer is left untouched.  Per owned tensor (rows x cols):
 *     m <- mu*m + g;  u = g + mu*m;  X0 = u / (||u||_F + eps), transposed to
 *     min x max if rows > cols;  ns_steps x { A = X X^T; B = b A + c A A;
 *     X <- a X + B X };  W <- W - lr*sqrt(max(1, rows/cols)) * X (back in rows x cols).
 * cz_muon_step uses the defaults of cz_step_opts_default and the library's
 * cached workspace for the current device (not safe for concurrent calls on
 * different streams; pass a workspace through cz_muon_step_ex for that).
 * Requires an sm_103a device.  Errors inside kernels (bounded waits that ran out,
 * descriptor checks) are reported by cz_device_status.
 * The first call for a given (plan, rank, buffers, offsets, shapes, workspace,
 * gradient dtype) builds the step's launch tables on the host and keeps them,
 * in page-locked host memory, until the library drops its cache of them; later
 * calls copy them into the workspace with a kernel.  lr, mu, ns_steps and the
 * scalar options (eps, Nesterov, a, b, c) are launch parameters: changing them
 * from call to call (a learning-rate schedule) rebuilds nothing.
 * CUDA graphs: a call may be enqueued into a stream that is being captured,
 * once a call with the same (plan, rank, buffers, offsets, shapes, workspace,
 * gradient dtype) has run outside the capture and the workspace (the caller's,
 * or the library's cached one, already large enough) exists; otherwise the call
 * returns CZ_ERR_INVALID before enqueuing anything.  The graph replays the
 * captured scalars (lr, mu, ...) and reads the buffers in place; the library
 * keeps the captured program's page-locked tables until the process exits.
 * Kernel timing (cz_profile_enable) skips captured launches.
 * Streams: all work is ordered on `stream`; when a shard has both small
 * matrices (m <= 256, n <= 256) and tiled ones, or small matrices of both
 * on-chip kinds (m <= 128 and 128 < m <= 256), one of the launches may run on a
 * library-owned side stream (one per caller stream, never destroyed) that is
 * forked from `stream` after the momentum pass and joined back into it, so that
 * work enqueued on `stream` after the call still follows all of the step. */
int cz_muon_step(const cz_plan* plan, int32_t rank,
                 float* flat_param, const void* flat_grad, float* flat_mom,
                 const int64_t* offsets, const int64_t* shapes,
                 float lr, float mu, int32_t ns_steps, void* stream);

int cz_muon_step_ex(const cz_plan* plan, int32_t rank,
                    float* flat_param, const void* flat_grad, float* flat_mom,
                    const int64_t* offsets, const int64_t* shapes,
                    float lr, float mu, int32_t ns_steps, void* stream,
                    const cz_step_opts* opts);

/* Number of step programs (launch tables) the library has built since it was
 * loaded.  Support for checking that a training loop reuses them: it grows only
 * when a call's plan, rank, buffers, offsets, shapes, workspace or gradient
 * dtype differ from every cached program's.  No GPU work. */
int cz_step_programs_built(int64_t* count);

/* cz_muon_step without any device allocation.  The paper has no counterpart
 * to this call; it exists for callers that cannot call cudaMalloc when they run
 * the step (an allocator that owns all device memory, memory reserved up front,
 * or code that must avoid the synchronisation cudaMalloc/cudaFree can cause).
 * Same arguments, kernels and results as cz_muon_step_ex (bit for bit, for the
 * same inputs); the workspace is a static device array of
 * CZ_STATIC_WORKSPACE_BYTES (64 MiB) that every GPU loading it holds until the
 * process exits.
 *   - opts may be NULL (defaults); opts->workspace must be NULL and
 *     workspace_bytes 0, else CZ_ERR_INVALID.
 *   - A shard whose cz_workspace_size exceeds CZ_STATIC_WORKSPACE_BYTES is
 *     rejected with CZ_ERR_NOMEM before any GPU work.
 *   - The first call on each device does a set-up: it looks up the array's
 *     device address and clears the array's status word on `stream`.  Under
 *     lazy module loading (the CUDA default) that look-up is also when the
 *     runtime loads the array, so the driver reserves its 64 MiB in this first
 *     call, which can fail with CZ_ERR_CUDA when device memory is exhausted.
 *     Make the first call on a device before any stream capture.  Later calls
 *     allocate nothing.
 *   - All calls share the one array, which keeps the previous call's contents
 *     (each call re-uploads its tables and overwrites what its kernels read):
 *     calls that overlap on the GPU (other streams, other threads) race.
 *   - Device-side errors go to the array's status word; cz_device_status with a
 *     NULL workspace reads and clears it.
 * Calls no cudaMalloc, cudaFree or other allocating routine and page-locks no
 * host memory: its launch tables are uploaded from pageable memory by
 * cudaMemcpyAsync. */
#define CZ_STATIC_WORKSPACE_BYTES (64u * 1024u * 1024u)
int cz_muon_step_noalloc(const cz_plan* plan, int32_t rank,
                         float* flat_param, const void* flat_grad, float* flat_mom,
                         const int64_t* offsets, const int64_t* shapes,
                         float lr, float mu, int32_t ns_steps, void* stream,
                         const cz_step_opts* opts);

/* Synchronises `stream`, reads and clears the device status word kept in
 * `workspace`.  NULL reads and clears every library-owned scratch of the current
 * device that exists: the cached workspace of cz_muon_step(_ex) and the static
 * array of cz_muon_step_noalloc.  *status_out = CZ_OK or the first CZ_ERR_* a
 * kernel recorded (with NULL: the cached workspace's first).  The `workspace`
 * argument is an addition to the pages-derived boundary: the caller owns the
 * workspace that holds its status word, so the call must be told which one. */
int cz_device_status(void* stream, void* workspace, int* status_out);

/* Kernel timing (tracing).  While enabled, every kernel that cz_muon_step(_ex)
 * launches is bracketed by two CUDA events recorded on the caller's stream;
 * cz_profile_read synchronises on them and returns, per kernel kind, the summed
 * milliseconds and launch counts since the previous read (then clears them).
 * Kinds, in order: 0 momentum pass (including the per-tensor norm), 1 copy of the
 * step's launch tables into the workspace, 2 Gram (A = X X^T),
 * 3 Poly (B = bA + cA^2), 4 Update (X <- aX + BX), 5 Update fused with the apply,
 * 6 all Newton-Schulz products of a step in one launch (the default),
 * 7 every Newton-Schulz step of the small matrices (m <= 256, n <= 256) on chip
 *   (one CTA per matrix for m <= 128, a CTA pair above).
 * ms and launches must hold n_kinds entries (n_kinds <= CZ_KERNEL_KINDS). */
#define CZ_KERNEL_KINDS 8
int cz_profile_enable(int32_t on);
int cz_profile_read(double* ms, int64_t* launches, int32_t n_kinds);

/* Self-test of the device-side failure detection (support; no counterpart in
 * the paper).  Launches one CTA on `stream` that waits, with the same bounded
 * wait the step's kernels use, on an mbarrier that nothing ever completes; after
 * timeout_ns (0 .. 2e9) the wait gives up and records CZ_ERR_TIMEOUT in the
 * status word of `workspace` (a device buffer of >= 256 bytes whose first int
 * starts at zero), which cz_device_status then reports.  No fault, no trap: the
 * context stays usable.  Returns CZ_OK when enqueued. */
int cz_selftest_bounded_wait(int64_t timeout_ns, void* workspace, void* stream);

/* Static string for a status code. */
const char* cz_status_string(int status);

/* Library version and build target, e.g. "cz 0.1 sm_103a". */
const char* cz_version(void);

/* Support (no counterpart in the paper): name and description of the CUDA error
 * behind the most recent CZ_ERR_CUDA that a kernel launch of this thread's
 * cz_muon_step(_ex) calls returned ("cudaSuccess: no error" if none).  The
 * string is owned by the library and valid until the thread's next call. */
const char* cz_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* CZ_H */
