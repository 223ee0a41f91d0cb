/*
 * zeroadam.h -- C ABI of libzeroadam.so: the ZeRO stage-1/2 mixed-precision
 * Adam step and the ZeRO-3 unit gather on one GB300 (sm_103a).
 *
 * The method is the one in "ZeRO and FSDP: partitioning the optimizer states,
 * the gradients and the parameters" (AI infra handbooks): the parameters are
 * one flat vector of numel elements, zero-padded to world*shard with
 * shard = ceil(numel/world); rank r owns [r*shard, (r+1)*shard).  One step of
 * rank r ("Implementing ZeRO's Adam from scratch", ZeroAdam.step):
 *   1. reduce-scatter the world ranks' gradients and average them,
 *   2. Adam with bias correction on rank r's fp32 master/m/v shard,
 *   3. all-gather the updated shard back into the full parameters.
 * Here the ranks are buffers in one GPU's memory: step 1 reads the world
 * gradient buffers directly, and step 3 writes rank r's shard, cast to bf16,
 * straight into the flat bf16 parameter buffer.  One kernel does all three.
 *
 * Conventions for every call:
 *   - Status: 0 (ZERO_OK) or a negative ZERO_E_* code.  Nothing is launched
 *     when a call returns an error.  No call aborts or allocates device
 *     memory; none synchronises except zero_device_status; the only state kept
 *     between calls is a per-device status word that a kernel sets only if one
 *     of its bounded waits gives up (see zero_device_status).  Faults inside a
 *     launched kernel surface, as for any CUDA work, at the caller's next sync.
 *   - Tracing: zero_adam_step, zero_adam_step_range, zero3_unit_gather,
 *     zero3_unit_gather_rows, zero3_unit_step and zero_device_status each
 *     open an NVTX range
 *     named after the function for the duration of the call (visible to
 *     Nsight tools and any NVTX injection library; free when none is
 *     attached).
 *   - Calls on different streams may run concurrently when their output
 *     buffers are disjoint; a sequence of calls may be captured into a CUDA
 *     graph after each kernel's first call on the device (which does one-time
 *     set-up outside any capture).
 *   - Device pointers are in the current CUDA device's address space; the
 *     stream argument is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream) and must belong to the current device.
 *   - bf16 buffers are arrays of IEEE bfloat16 bit patterns (uint16_t).
 *   - The caller owns every buffer.  Host pointer arrays (grad_ptrs,
 *     shard_ptrs) are read before the call returns.
 *   - Alignment: bf16 pointers must be 2-byte and fp32 pointers 4-byte
 *     aligned (ZERO_E_ALIGN otherwise).  16-byte alignment is not required,
 *     but the fast vectorised path runs only where the buffers can be
 *     accessed 16 bytes at a time together (always so for buffers from the
 *     PyTorch/cudaMalloc allocator used as whole flat vectors).
 */
#ifndef ZEROADAM_H
#define ZEROADAM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ----------------------------------------------------------------- status */

#define ZERO_OK 0
#define ZERO_E_NULLPTR (-1) /* a required pointer is NULL                          */
#define ZERO_E_WORLD (-2)   /* world < 1 or world > ZERO_MAX_WORLD                  */
#define ZERO_E_NUMEL (-3)   /* numel < 1, or world*shard overflows int64           */
#define ZERO_E_RANK (-4)    /* rank not in [0, world) and not ZERO_ALL_RANKS        */
#define ZERO_E_STEP (-5)    /* t < 1 (t is the 1-based step count after increment)  */
#define ZERO_E_ALIGN (-6)   /* bf16 pointer odd, or fp32 pointer not 4-byte aligned */
#define ZERO_E_HPARAM (-7)  /* lr/eps negative or not finite; beta not in [0, 1)    */
#define ZERO_E_LAYOUT (-8)  /* unknown layout, or a shard layout with ALL_RANKS     */
#define ZERO_E_PLAN (-9)    /* the plan's fields are not those zero_plan computes   */
#define ZERO_E_ALIAS (-10)  /* an output buffer overlaps another buffer             */
#define ZERO_E_LAUNCH (-11) /* the CUDA launch failed; see zero_strerror            */
#define ZERO_E_DEVICE (-12) /* no usable CUDA device                                */
#define ZERO_E_RANGE (-13)  /* zero_adam_step_range: begin < 0 or end < begin       */
#define ZERO_E_SHAPE (-14)  /* zero3_unit_gather_rows: bad tensor count or shape    */
#define ZERO_E_TIMEOUT (-15) /* a kernel gave up a bounded wait (zero_device_status) */
#define ZERO_E_HOOK (-16)    /* a test hook was called without ZEROADAM_TEST_HOOKS=1 */

/* Largest tensor count of one zero3_unit_gather_rows unit. */
#define ZERO_MAX_UNIT_TENSORS 256

/* Largest world (number of emulated data-parallel ranks) accepted. */
#define ZERO_MAX_WORLD 1024

/* rank argument: step every rank's shard in one launch. */
#define ZERO_ALL_RANKS (-1)

/* grad_layout: one layout, optionally OR-ed with the flags below */
#define ZERO_GRAD_FULL 0   /* grad_ptrs[k]: rank k's whole padded flat gradient (>= numel elements) */
#define ZERO_GRAD_SHARD 1  /* grad_ptrs[k]: rank k's gradient slice of THIS rank's shard (shard elements); single rank only */
#define ZERO_GRAD_WINDOW 2 /* zero_adam_step_range only: grad_ptrs[k][i - begin], the window's gradients alone */
#define ZERO_GRAD_LAYOUT_MASK 0x0f
#define ZERO_GRAD_F32 0x10 /* flag: gradient buffers hold fp32 (default: bf16) */
#define ZERO_ACC_BF16 0x20 /* flag: round the running sum over ranks to bf16 after every addition */

/* param_layout */
#define ZERO_PARAM_FULL 0  /* param_bf16: the whole flat parameter buffer (>= numel elements) */
#define ZERO_PARAM_SHARD 1 /* param_bf16: this rank's shard only (shard elements; ZeRO-3); single rank only */

/* ------------------------------------------------------------------- plan */

/*
 * Layout and per-card memory of a flat vector of numel parameters on world
 * data-parallel ranks.
 *
 *   shard  = ceil(numel / world), pad = world*shard - numel, padded = world*shard
 *            ("Implementing ZeRO's Adam from scratch": shard size and _flatten's
 *            zero padding).
 *   bytes_* : model-state bytes per card with the padded shard: DP 16*numel,
 *            ZeRO-1 4*numel + 12*shard, ZeRO-2 2*numel + 14*shard,
 *            ZeRO-3 16*shard (mixed-precision Adam: bf16 parameter 2 B, bf16
 *            gradient 2 B, fp32 master/m/v 12 B; "The three stages" table).
 *   formula_*: the same table's real-valued expressions 16 Psi, 4 Psi + 12 Psi/N,
 *            2 Psi + 14 Psi/N, 16 Psi/N (equal to bytes_* when pad == 0).
 *   state_bytes_rank: fp32 master + m + v bytes one rank holds, 12*shard
 *            (ZeroAdam.state_bytes).
 *   comm_*: bytes sent per card per step for the bf16 gradients/parameters
 *            ("The three stages" table, last column, and "Exercises": a ring
 *            all-reduce sends 2(N-1)/N of the gradient size; ZeRO-1/2 send the
 *            same as a reduce-scatter plus an all-gather; ZeRO-3 adds one more
 *            parameter all-gather, 1.5x): comm_dp = comm_z1 = comm_z2 =
 *            2 * (N-1)/N * 2*padded, comm_z3 = 3 * (N-1)/N * 2*padded.
 *
 * Host only; no CUDA call.  Errors: ZERO_E_NULLPTR, ZERO_E_WORLD, ZERO_E_NUMEL.
 */
typedef struct {
  int64_t numel, world, shard, pad, padded;
  uint64_t bytes_dp, bytes_z1, bytes_z2, bytes_z3;
  double formula_dp, formula_z1, formula_z2, formula_z3;
  uint64_t state_bytes_rank;
  double comm_dp, comm_z1, comm_z2, comm_z3;
} zero_plan_t;

int zero_plan(int64_t numel, int32_t world, zero_plan_t* out);

/* ------------------------------------------------------------------- step */

/*
 * One ZeRO-1/2 Adam step ("Implementing ZeRO's Adam from scratch",
 * ZeroAdam.step) for rank `rank`, or for all ranks (ZERO_ALL_RANKS), on the
 * ranks' shards of the flat vector described by plan (from zero_plan).
 *
 * For every global flat index i < numel that the stepped rank(s) own:
 *   g    = (((float)g_0[i] + (float)g_1[i]) + ... + (float)g_{N-1}[i]) / N
 *          (reduce_scatter_tensor, then g /= world; fp32 sum in rank order)
 *   m    = m*b1 + (1-b1)*g ;  v = v*b2 + ((1-b2)*g)*g
 *   w    = w - (lr * (m / (1-b1^t))) / (sqrt(v / (1-b2^t)) + eps)
 *   p[i] = bf16 round-to-nearest-even of w   (all_gather_into_tensor + copy
 *          into the parameters)
 * Each operation is one IEEE binary32 operation rounded to nearest even (no
 * FMA contraction, denormals kept); the scalars 1-b1, 1-b2, 1-b1^t, 1-b2^t,
 * b1, b2, lr, eps, N are formed in double and rounded to binary32 once.
 * Indices >= numel (the zero padding) are neither read nor written.
 *
 *   plan        from zero_plan(numel, world); checked (ZERO_E_PLAN).
 *   rank        in [0, world), or ZERO_ALL_RANKS.
 *   grad_ptrs   host array of world device pointers, bf16 (fp32 with ZERO_GRAD_F32).
 *               ZERO_GRAD_FULL : grad_ptrs[k][i] for global index i.
 *               ZERO_GRAD_SHARD: grad_ptrs[k][i - rank*shard] (single rank).
 *               (ZERO_GRAD_WINDOW is zero_adam_step_range's; here ZERO_E_LAYOUT.)
 *   master,m,v  device fp32, read and written in place.
 *               ALL_RANKS: padded elements, index i (the ranks' shards back to
 *               back); single rank: shard elements, index i - rank*shard.
 *   param_bf16  device bf16, written only.
 *               ZERO_PARAM_FULL : index i, buffer of >= numel elements.
 *               ZERO_PARAM_SHARD: index i - rank*shard (single rank).
 *   lr, beta1, beta2, eps  Adam hyper-parameters (lr, eps >= 0; 0 <= beta < 1).
 *   t           1-based step number after the increment (ZeroAdam.step's
 *               self.t += 1 happens before the moments are used).
 *   stream      cudaStream_t as void*.
 * The gradient buffers must not overlap any output; master, m, v and
 * param_bf16 must not overlap one another (ZERO_E_ALIAS).
 */
int zero_adam_step(const zero_plan_t* plan, int32_t rank, const void* const* grad_ptrs,
                   int32_t grad_layout, float* master, float* m, float* v, void* param_bf16,
                   int32_t param_layout, double lr, double beta1, double beta2, double eps,
                   int64_t t, void* stream);

/*
 * The same step restricted to the global flat window [begin, end) (clipped to
 * the stepped rank's real elements): ZeRO-2's bucketed schedule ("Implementing
 * ZeRO's Adam from scratch", closing note: real ZeRO-2 reduce-scatters bucket
 * by bucket during the backward pass and frees each full-gradient bucket once
 * it has gone out).  With ZERO_GRAD_WINDOW each grad_ptrs[k] holds only the
 * bucket, element i at grad_ptrs[k][i - begin], so the full gradient never
 * needs to exist; ZERO_GRAD_FULL and ZERO_GRAD_SHARD address as in
 * zero_adam_step.  master/m/v and param_bf16 are addressed as in
 * zero_adam_step.  Buckets that tile the flat vector give exactly the result
 * of one zero_adam_step (the step is elementwise).  Errors: those of
 * zero_adam_step, and ZERO_E_RANGE.
 *
 * Gradient variants (flags in grad_layout, both calls): ZERO_GRAD_F32 takes
 * fp32 gradient buffers (the page's runnable demo keeps fp32 gradients);
 * ZERO_ACC_BF16 rounds the running sum over ranks to bf16 after every
 * addition, the result a reduce-scatter on bf16 buffers delivers (a
 * sensitivity variant, not the method).
 */
int zero_adam_step_range(const zero_plan_t* plan, int32_t rank, int64_t begin, int64_t end,
                         const void* const* grad_ptrs, int32_t grad_layout, float* master,
                         float* m, float* v, void* param_bf16, int32_t param_layout, double lr,
                         double beta1, double beta2, double eps, int64_t t, void* stream);

/* ------------------------------------------------------------ ZeRO-3 gather */

/*
 * ZeRO-3 unit all-gather ("ZeRO-3 and FSDP": before a unit is used in the
 * forward or backward pass its complete parameters are all-gathered):
 *   full_bf16[r*shard + j] = shard_ptrs[r][j]  for r < world, j < shard,
 *                                              r*shard + j < numel,
 * where unit_plan = zero_plan(U, world) of the unit's U elements.  The copy is
 * bit-exact; the padded tail of the last shard is not copied.
 *
 *   shard_ptrs  host array of world device pointers to bf16 shards of
 *               unit_plan->shard elements each.
 *   full_bf16   device bf16 buffer of >= numel elements, written only; must not
 *               overlap a shard (ZERO_E_ALIAS).
 *
 * When shard is a multiple of 8 elements and every buffer is 16-byte aligned
 * (whole cudaMalloc/PyTorch buffers) the copy runs on the TMA engine, whose
 * waits are bounded (see zero_device_status); otherwise a load/store kernel.
 */
int zero3_unit_gather(const zero_plan_t* unit_plan, const void* const* shard_ptrs,
                      void* full_bf16, void* stream);

/*
 * FSDP2-style unit gather ("ZeRO-3 and FSDP": FSDP2 represents every parameter
 * as a DTensor sharded along dimension 0, so each rank holds a block of rows of
 * each tensor).  The unit is ntensors row-major bf16 tensors, tensor i of
 * rows[i] x cols[i] elements.  With R_i = ceil(rows[i] / world), rank r holds
 * rows [r*R_i, min((r+1)*R_i, rows[i])) of tensor i, stored as R_i x cols[i]
 * elements (rows past the tensor's end are padding and are not copied); its
 * shard buffer is those blocks for i = 0..ntensors-1 back to back
 * (sum_i R_i*cols[i] elements).  The gathered unit full_bf16 is the tensors
 * back to back (sum_i rows[i]*cols[i] elements).  Bit-exact copy.  For one
 * tensor whose rows divide by world this is zero3_unit_gather's layout.
 *
 *   rows, cols  host arrays of ntensors positive sizes, read before return.
 *   shard_ptrs  host array of world device pointers (bf16 shards).
 * Errors: ZERO_E_SHAPE (ntensors not in [1, ZERO_MAX_UNIT_TENSORS], a size < 1,
 * or the unit's element count overflows), ZERO_E_WORLD, ZERO_E_NULLPTR,
 * ZERO_E_ALIGN (odd pointer), ZERO_E_ALIAS (output overlaps a shard),
 * ZERO_E_LAUNCH.
 *
 * When every tensor's offset in the unit and every R_i*cols[i] is a multiple of
 * 8 elements and every buffer is 16-byte aligned (e.g. a Llama layer's weights
 * from whole cudaMalloc/PyTorch buffers) the copy runs on the TMA engine, whose
 * waits are bounded (see zero_device_status); otherwise a load/store kernel.
 */
int zero3_unit_gather_rows(int32_t ntensors, const int64_t* rows, const int64_t* cols,
                           int32_t world, const void* const* shard_ptrs, void* full_bf16,
                           void* stream);

/*
 * One ZeRO-3 unit's gather and one rank's step in a single launch ("ZeRO-3 and
 * FSDP": a unit's parameters are all-gathered from the ranks' shards before
 * the unit is used, and each rank updates only its own shard).  The result is
 * exactly that of
 *   zero3_unit_gather(unit_plan, shard_ptrs, full_bf16, stream);
 *   zero_adam_step(unit_plan, rank, grad_ptrs, grad_layout, master, m, v,
 *                  param_bf16, param_layout, lr, beta1, beta2, eps, t, stream);
 * with the same arguments, layouts and errors as those two calls.  The step
 * does not read the gathered unit, so the two parts run side by side in one
 * grid instead of one after the other (one launch, overlapped ramps: the
 * page's small units are latency-bound).  Because they overlap, the buffers
 * of the two parts must be disjoint: full_bf16 must not overlap any gradient
 * or any step output, and no shard may overlap a step output (ZERO_E_ALIAS).
 * To update the rank's own bf16 shard in place (param_bf16 inside
 * shard_ptrs[rank]) call the two functions in sequence instead.
 *
 * When the shard is a multiple of 8 elements, every buffer of both parts is
 * 16-byte aligned at its first element, the gradients are bf16, the sum is
 * fp32 and the unit moves at most 512 MiB (gather 4 bytes per unit element +
 * step (2*world + 26) bytes per stepped element), the single launch runs (bulk copies on the TMA engine, bounded waits reported by
 * zero_device_status); otherwise the two kernels are launched in order on the
 * stream (larger units stream as fast that way, with the launch cost
 * amortised).  Errors: those of zero3_unit_gather and
 * zero_adam_step (ZERO_GRAD_WINDOW is not accepted: ZERO_E_LAYOUT).
 */
int zero3_unit_step(const zero_plan_t* unit_plan, int32_t rank, const void* const* shard_ptrs,
                    void* full_bf16, const void* const* grad_ptrs, int32_t grad_layout,
                    float* master, float* m, float* v, void* param_bf16, int32_t param_layout,
                    double lr, double beta1, double beta2, double eps, int64_t t, void* stream);

/* ------------------------------------------------------------------ misc */

/*
 * Device-side status of the library's kernels on the current device.  Some
 * launches stage data through shared memory with asynchronous bulk copies and
 * wait on hardware barriers; every such wait is bounded, and a wait that gives
 * up (one second without progress, by the GPU's global timer) ends the launch
 * early, leaving that step's outputs incomplete, and records the fact in a
 * per-device status word.
 * The call first synchronises the current device (cudaDeviceSynchronize),
 * so every kernel launched before it, on any stream of the device, has
 * finished; then it reads and clears the words with one atomic exchange on the
 * GPU each, so a word set while the call runs is reported now or by the next
 * call, never lost.  Returns ZERO_OK if no wait has given up since the previous
 * call, else ZERO_E_TIMEOUT.  ZERO_E_DEVICE if there is no usable device or the
 * synchronisation reports an error (an earlier asynchronous fault; its CUDA
 * text is in zero_strerror).  It launches a one-thread kernel on the legacy
 * default stream, so it must not be called while a stream capture is open.
 */
int zero_device_status(void);

/*
 * Test hook for the bounded waits; the pages' method has no counterpart.
 * While `on` is nonzero, every step launch that uses a TMA-staged kernel
 * (world >= 5, bf16 gradients, fp32 sum, all buffers 16-byte aligned at the
 * stepped range's first element), every zero3_unit_gather or
 * zero3_unit_gather_rows that uses the TMA copy (see those calls), and every
 * zero3_unit_step that runs as a single launch tells its producers to issue
 * no copies.  Every wait then runs out after its limit (about one second),
 * the outputs of the parts that wait are not written (at world <= 4 the
 * unit step's step part reads its gradients without staging and completes),
 * and zero_device_status reports ZERO_E_TIMEOUT; the device and its context
 * stay usable.  Launches of the other kernels are unaffected (they do not
 * wait).  The setting is process-wide and read when a call launches.  Returns
 * the previous
 * setting (0 or 1).  It exists so that tests can exercise the timeout path
 * without faulting or hanging a GPU; production code never calls it.  It is
 * off unless the environment variable ZEROADAM_TEST_HOOKS is "1" when it is
 * called; otherwise it changes nothing and returns ZERO_E_HOOK.
 */
int zero_test_withhold_copies(int on);

/* Text for a status code.  For ZERO_E_LAUNCH it includes the CUDA error text
   of this thread's last failed launch.  The pointer stays valid until this
   thread's next call into the library. */
const char* zero_strerror(int status);

/* Library version, e.g. 0x000100 for 0.1.0. */
int zero_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ZEROADAM_H */
