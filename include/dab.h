/*
 * dab.h -- C ABI of the deterministic attention backward library (libdab.so)
 * for GB300 (sm_103a).
 *
 * The operation: exact softmax attention O = softmax(scale * Q K^T, mask) V
 * and its backward pass, which produces dQ, dK and dV with the dQ partial
 * sums of all KV tiles added in a fixed order, so that the deterministic
 * schedules give bitwise-identical gradients from run to run.  The schedules
 * are those of "DASH: Deterministic Attention Scheduling for High-throughput
 * Reproducible LLM Training" (arXiv 2601.21824): the serialised baseline
 * (technical summary section 1), Descending Q-Tile Iteration (section 2.2.A)
 * and Shift Scheduling, with the symmetric variant for causal masks
 * (section 2.2.B), plus the non-deterministic atomic counterpart that the
 * abstract compares against.
 *
 * Conventions shared by every entry point
 *   Layout   Q, K, V, O, dO, dQ, dK, dV are contiguous bfloat16 tensors of
 *            shape [B][H][S][d] (row-major, d innermost); LSE is a contiguous
 *            float32 tensor [B][H][S] holding the natural log of
 *            sum_c exp(scale * q_r . k_c) over the visible keys.  Query and key
 *            sequences have the same length S.
 *   Shapes   d must be 64 or 128; S >= 0, any length (the last 128-row tile
 *            of a head may be partial); B, H >= 0; B*H*ceil(S/128)*128 < 2^31.
 *            A problem with B, H or S zero is empty: DAB_OK, no kernel runs
 *            (a backward call given a workspace clears its status word).
 *   Mask     DAB_MASK_CAUSAL hides key c from query r when c > r (the diagonal
 *            is visible, so no query row is empty).
 *   Memory   Every pointer is a device pointer, allocated and owned by the
 *            caller, 16-byte aligned (except the host-buffer path,
 *            dab_attn_bwd_host, whose tensors live in host memory).  The
 *            library never calls cudaMalloc.  State it keeps between calls:
 *            a per-device cache of kernel attributes and of the SM count;
 *            the schedule-selection cache (dab_sched_select); three
 *            library-owned CUDA streams per device, created on the first
 *            dab_attn_bwd_host call on that device (its events are created
 *            and released within each call); and the
 *            fixed scratch array of dab_attn_bwd_noalloc
 *            (DAB_NOALLOC_SCRATCH_BYTES of device memory, part of the
 *            library's image on every GPU that loads it).
 *   Streams  Every call is asynchronous on `stream` and may run concurrently
 *            with calls on other streams that use distinct workspaces.
 *   Errors   Argument errors are returned synchronously and launch nothing.
 *            DAB_ERR_CUDA reports a failed kernel launch.  Faults detected on
 *            the device (a bounded wait that ran out, an index out of range)
 *            never trap: the kernels record them in the workspace status word
 *            and return, and dab_check_status() reports them.
 */
#ifndef DAB_H_
#define DAB_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DAB_MASK_FULL = 0,
    DAB_MASK_CAUSAL = 1
} dab_mask_t;

/* Backward schedules.
 *   SERIAL        KV tile i walks its Q tiles in ascending order; dQ_j gathers
 *                 its partial sums in ascending KV order (rank(i, j) = i).
 *                 The serialised deterministic baseline (DASH summary sec. 1).
 *   DESCENDING_Q  Same dQ reduction order as SERIAL, Q tiles walked from the
 *                 last one down (DASH summary sec. 2.2.A).  dQ is bitwise equal
 *                 to SERIAL's; dK and dV accumulate along the reversed walk.
 *   SHIFT         Full mask: KV tile i walks Q tiles i, i+1, ..., N-1, 0, ...,
 *                 i-1 and dQ_j is reduced in visit order (DASH summary
 *                 sec. 2.2.B).  Causal mask: the symmetric variant, where one
 *                 CTA handles KV tiles p and N-1-p in a dense phase and a
 *                 folded phase; needs an even number of tiles N = S/128.
 *   ATOMIC        Unordered float atomics; the only schedule whose bits may
 *                 differ between runs (the non-deterministic counterpart).   */
typedef enum {
    DAB_SCHED_SERIAL = 0,
    DAB_SCHED_DESCENDING_Q = 1,
    DAB_SCHED_SHIFT = 2,
    DAB_SCHED_ATOMIC = 3,
    /* Accepted by dab_bwd_workspace_size, dab_bwd_workspace_layout,
     * dab_bwd_preprocess, dab_attn_bwd and dab_attn_bwd_ex only: the library
     * runs the deterministic schedule that dab_sched_select() picks for the
     * problem on the current device (the choice depends on mask, B*H, S and
     * the SM count, never on the data, so repeated calls give the same bits). */
    DAB_SCHED_AUTO = 4
} dab_sched_t;

typedef enum {
    DAB_OK = 0,
    DAB_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad shape or enum */
    DAB_ERR_UNSUPPORTED = 2,   /* valid but not supported here (e.g. odd N for
                                  causal SHIFT, no sm_100-family device)     */
    DAB_ERR_WORKSPACE = 3,     /* workspace missing or too small             */
    DAB_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed       */
    DAB_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out             */
    DAB_ERR_DEVICE_BOUNDS = 6  /* device: an index or alignment check failed */
} dab_status_t;

/* Attention forward: writes O (bf16 [B][H][S][d]) and LSE (f32 [B][H][S]).
 * Produces the O and LSE that the backward consumes.  `workspace` is unused
 * and may be NULL (ws_bytes 0).                                              */
dab_status_t dab_attn_fwd(const void* q, const void* k, const void* v,
                          void* o, float* lse,
                          int B, int H, int S, int d, float scale,
                          dab_mask_t mask,
                          void* workspace, size_t ws_bytes,
                          cudaStream_t stream);

/* Bytes of device workspace that dab_attn_bwd needs for this problem (0 on
 * invalid arguments).  The workspace holds the status word, the dispatch
 * counters, the semaphores (per 128-row dQ tile: one per eighth of the tile
 * and per accumulation buffer), D and -LSE*log2(e) per row, and the float32
 * dQ accumulation buffers [ways][B][H][S][d] (four interleaved buffers for
 * the ordered schedules, one for ATOMIC).  It needs no initialisation: the
 * first kernel of every backward call resets what must start at zero.      */
size_t dab_bwd_workspace_size(int B, int H, int S, int d,
                              dab_mask_t mask, dab_sched_t sched);

/* Attention backward.  Inputs Q, K, V, O, dO (bf16) and LSE (f32) as produced
 * by dab_attn_fwd; outputs dQ, dK, dV (bf16), each written in full.
 * Launches, on `stream`:
 *   1. the preprocess kernel: D_r = sum_k dO_rk O_rk (f32), -LSE*log2(e),
 *      reset of the semaphores, status word and dispatch counter (and, for
 *      ATOMIC, zeroing of the dQ accumulator);
 *   2. the persistent main kernel: per KV tile, S, P, dV, dP, dS, dK and the
 *      dQ partial on the tensor cores, then the dQ reduction in the order
 *      `sched` defines, and, for the three deterministic schedules, in the
 *      kernel's tail, dQ = bf16(scale * sum of the accumulation buffers,
 *      added in buffer order) for every 128-row tile once its contributions
 *      are in.  The deterministic reduction is semaphore-ordered: a
 *      contributor adds its partial only once every contributor of lower
 *      rank in the same buffer has published, so each element receives its
 *      additions in one fixed order.  By default that addition is a float
 *      reduction in the L2 (red.add.v4.f32: four f32 adds per 16-byte
 *      vector), issued by one contributor at a time; DAB_BWD_PLAIN_ADD
 *      replaces it with a load, an add in registers and a store, which gives
 *      the same bits and uses no float atomic;
 *   3. for ATOMIC only: the convert kernel, the same dQ formula as a separate
 *      pass (see DAB_BWD_SEPARATE_CONVERT).
 * The call returns once the kernels are queued.                              */
dab_status_t dab_attn_bwd(const void* q, const void* k, const void* v,
                          const void* o, const float* lse, const void* dout,
                          void* dq, void* dk, void* dv,
                          int B, int H, int S, int d, float scale,
                          dab_mask_t mask, dab_sched_t sched,
                          void* workspace, size_t ws_bytes,
                          cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Block masks: the block-sparse masks the DASH pages name as future work
 * (technical summary section 5).  `tiles` is a DEVICE array of N x N bytes,
 * N = S/128, row j = query tile, column i = key tile, shared by all heads and
 * caller-owned: a zero flag hides key tile i from every query of query tile
 * j.  With causal = 1 the causal mask applies too (tiles above the diagonal
 * are hidden whatever their flag, and the diagonal tiles hide keys after the
 * query).  A query row with no visible key has no softmax: O = 0 and LSE =
 * -infinity from the forward; its dQ is 0 and it adds nothing to dK, dV.
 * A key tile no query sees gets dK = dV = 0.  Errors as dab_attn_fwd /
 * dab_attn_bwd; tiles == NULL or causal not 0/1: DAB_ERR_INVALID_ARG.     */
dab_status_t dab_attn_fwd_block(const void* q, const void* k, const void* v,
                                void* o, float* lse,
                                int B, int H, int S, int d, float scale,
                                const uint8_t* tiles, int causal,
                                void* workspace, size_t ws_bytes,
                                cudaStream_t stream);

/* Workspace of dab_attn_bwd_block: that of dab_attn_bwd plus the schedule
 * tables built from the tile flags (0 for SHIFT, which is not available
 * with a block mask, or on invalid arguments).                             */
size_t dab_bwd_block_workspace_size(int B, int H, int S, int d, dab_sched_t sched);

/* The backward under a block mask.  Schedules SERIAL, DESCENDING_Q (also for
 * DAB_SCHED_AUTO) and ATOMIC: each KV tile walks its visible Q tiles only
 * (ascending, or descending for DESCENDING_Q), and dQ_j adds its visible KV
 * tiles' partial sums in ascending KV order, so SERIAL and DESCENDING_Q give
 * the same dQ bits as without a mask.  SHIFT: DAB_ERR_UNSUPPORTED.  The
 * preprocess kernel of the call builds the tables in the workspace.        */
dab_status_t dab_attn_bwd_block(const void* q, const void* k, const void* v,
                                const void* o, const float* lse, const void* dout,
                                void* dq, void* dk, void* dv,
                                int B, int H, int S, int d, float scale,
                                const uint8_t* tiles, int causal, dab_sched_t sched,
                                void* workspace, size_t ws_bytes,
                                cudaStream_t stream);

/* Synchronises `stream`, then reads the status word that the backward kernels
 * of the last call on this workspace wrote.  Returns DAB_OK, DAB_ERR_TIMEOUT
 * or DAB_ERR_DEVICE_BOUNDS (or DAB_ERR_CUDA if the synchronisation failed).  */
dab_status_t dab_check_status(const void* workspace, cudaStream_t stream);

/* Static, human-readable name of a status code.                             */
const char* dab_status_string(dab_status_t status);

/* The CUDA error behind the calling thread's last DAB_ERR_CUDA (the failing
 * step, the CUDA error name and number), or "" if there was none.  The
 * string is owned by the library and valid until the next call that fails. */
const char* dab_last_error_string(void);

/* ------------------------------------------------------------------------ */
/* Extended backward options.  dab_attn_bwd() is dab_attn_bwd_ex() with
 * opts == NULL.                                                              */
typedef struct {
    uint64_t spin_timeout_ns; /* limit of every device-side wait; 0 = default
                                 (2 s)                                         */
    uint32_t flags;           /* DAB_BWD_* bits below                         */
    int32_t grid;             /* CTAs of the main kernel; 0 = one per SM      */
} dab_bwd_opts_t;

/* Skip the preprocess kernel: the caller has run dab_bwd_preprocess() on this
 * workspace itself (used to inject faults from the host, e.g. to poison a
 * semaphore and check that the bounded wait reports DAB_ERR_TIMEOUT).       */
#define DAB_BWD_SKIP_PREPROCESS 0x1u
/* Skip the conversion of dQ to bf16, in the main kernel and as a separate
 * pass (dQ is left in the workspace accumulator).                          */
#define DAB_BWD_SKIP_CONVERT 0x2u
/* Skip the main kernel (measurement only: with DAB_BWD_SKIP_PREPROCESS it
 * runs the separate convert pass alone, so that its time can be taken; dQ,
 * dK and dV are then not the gradients).                                   */
#define DAB_BWD_SKIP_MAIN 0x4u
/* Ordered schedules: add each dQ partial to the accumulator with a load from
 * the L2, an add in registers and a store, instead of red.add.f32 in the L2
 * (the same additions in the same order, so the same bits; no float atomic
 * is then used anywhere on the deterministic path).  The default is the red,
 * which is faster.                                                          */
#define DAB_BWD_PLAIN_ADD 0x8u
/* Ordered schedules: convert dQ in a separate pass after the main kernel.
 * By default the main kernel does it itself: once a CTA has no units left it
 * converts the dQ tiles whose contributions are all in (bounded waits on the
 * dQ semaphores), with the same arithmetic as the separate pass, so both
 * give the same bits.  The atomic schedule always uses the separate pass.  */
#define DAB_BWD_SEPARATE_CONVERT 0x10u
/* Let the main kernel share the GPU: launch it without the cooperative
 * attribute when the schedule hands out units dynamically (every schedule but
 * SHIFT, whose statically placed gangs must be resident together), so that
 * its CTAs can start on SMs as other kernels release them.  The waits of
 * those schedules only point at units that running CTAs have claimed, so the
 * kernel completes whatever else occupies the GPU.  Same results.  The
 * host-buffer path uses it to overlap the kernels of consecutive chunks.   */
#define DAB_BWD_SHARE_GPU 0x20u

dab_status_t dab_attn_bwd_ex(const void* q, const void* k, const void* v,
                             const void* o, const float* lse, const void* dout,
                             void* dq, void* dk, void* dv,
                             int B, int H, int S, int d, float scale,
                             dab_mask_t mask, dab_sched_t sched,
                             void* workspace, size_t ws_bytes,
                             cudaStream_t stream, const dab_bwd_opts_t* opts);

/* The preprocess step alone (step 1 of dab_attn_bwd), for the flag above.   */
dab_status_t dab_bwd_preprocess(const void* o, const float* lse, const void* dout,
                                int B, int H, int S, int d,
                                dab_mask_t mask, dab_sched_t sched,
                                void* workspace, size_t ws_bytes,
                                cudaStream_t stream);

/* Byte offsets of the workspace regions (for tests and tools).             */
typedef struct {
    size_t status;   /* uint32 status word, uint32 error detail, uint32 counter */
    size_t sem;      /* uint32 [B*H][N][8][ways] semaphores                     */
    size_t D;        /* float  [B*H*Spad], heads padded to whole 128-row tiles  */
    size_t lse2;     /* float  [B*H*Spad] -LSE * log2(e), heads padded to tiles */
    size_t dqacc;    /* float  [ways][B*H*Spad*d]: per 128-row tile
                        [d/4][128][4] (chunk-major), except the atomic
                        schedule at d = 128: row-major [row][d]                */
    size_t total;
} dab_ws_layout_t;

dab_status_t dab_bwd_workspace_layout(int B, int H, int S, int d,
                                      dab_mask_t mask, dab_sched_t sched,
                                      dab_ws_layout_t* layout);

/* ------------------------------------------------------------------------ */
/* The backward for callers that cannot allocate device memory.
 *
 * The paper has no counterpart to this entry point.  Some callers may not
 * call cudaMalloc where they need the backward -- for example a plugin inside
 * a host framework that owns and budgets all device memory, or a
 * latency-critical loop where an allocation, which can synchronise the
 * device, is not acceptable -- and so cannot provide the workspace that
 * dab_attn_bwd needs.  dab_attn_bwd_noalloc is dab_attn_bwd with that
 * workspace taken from a fixed array inside the library
 * (DAB_NOALLOC_SCRATCH_BYTES bytes; every GPU that loads the library holds it
 * until the process exits).  The caller still passes every input and output.
 *
 *   Limit    problems whose dab_bwd_workspace_size() exceeds
 *            DAB_NOALLOC_SCRATCH_BYTES are rejected with DAB_ERR_WORKSPACE
 *            before anything is launched (roughly B*H*S*d <= 2M elements
 *            for the ordered schedules, 8M for ATOMIC).
 *   Set-up   the first call on a device, with that device current, looks up
 *            the array's device address (cudaGetSymbolAddress) and caches
 *            it; make that first call before any stream capture.  A failed
 *            lookup returns DAB_ERR_CUDA.  The cached address does not
 *            survive cudaDeviceReset(): do not use this entry point on a
 *            device after resetting it.
 *   Sharing  every call on a device uses the same array, which keeps the
 *            last call's contents; each call's first kernel clears what must
 *            start at zero.  Calls whose kernels overlap on the GPU (for
 *            instance on two streams) race on the array: serialise them.
 *   Status   the device status word lives in the array too: read it with
 *            dab_noalloc_check_status() after the call (a device-side
 *            timeout leaves the gradients undefined).
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call.    */
#define DAB_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

dab_status_t dab_attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                  const void* o, const float* lse, const void* dout,
                                  void* dq, void* dk, void* dv,
                                  int B, int H, int S, int d, float scale,
                                  dab_mask_t mask, dab_sched_t sched,
                                  cudaStream_t stream);

/* The status of the last dab_attn_bwd_noalloc call on the current device, as
 * dab_check_status() reports it for a workspace: synchronises `stream`, then
 * copies the status word out of the library's scratch array into host stack
 * memory (no allocation).  DAB_OK, DAB_ERR_TIMEOUT, DAB_ERR_DEVICE_BOUNDS, or
 * DAB_ERR_CUDA if the synchronisation or the copy failed.                   */
dab_status_t dab_noalloc_check_status(cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* The backward on HOST buffers, with the host<->device copies overlapped with
 * the computation.  Not on the pages: it is the path of a caller whose
 * tensors live in host memory.  q, k, v, o, dout (bf16 [B][H][S][d]) and lse
 * (f32 [B][H][S]) are read from host memory, dq, dk, dv (bf16) written to
 * host memory; for overlapped (asynchronous) copies all nine must be pinned
 * (cudaHostAlloc / cudaHostRegister), otherwise the copies are synchronous.
 * The heads are split into `chunks` groups of consecutive (b, h) heads (0 =
 * the default, 8; at most B*H): the inputs of all groups are copied in back
 * to back on a library-owned stream, each group's backward runs as
 * dab_attn_bwd_ex on that range of heads (so its results are those of
 * dab_attn_bwd for an explicit schedule; DAB_SCHED_AUTO picks per group
 * shape) with DAB_BWD_SHARE_GPU, even groups on `stream` and odd groups on a
 * second library-owned stream (consecutive groups overlap on the GPU), and
 * each group's gradients are copied back on a third library-owned stream
 * while later groups compute.  Everything starts after the work already
 * queued on `stream`, and `stream` waits for the last copy back: synchronise
 * `stream` before reading dq, dk, dv or reusing the inputs.  dev_ws: device
 * memory of dab_bwd_host_workspace_size() bytes, 256-byte aligned,
 * caller-owned (a status header, copies of inputs and outputs, and two
 * backward workspaces of one group); after the call, dab_check_status(dev_ws,
 * stream) reports the first device error of any group.  Errors as
 * dab_attn_bwd; on an error after the first group was queued, earlier groups
 * may still complete.                                                        */
size_t dab_bwd_host_workspace_size(int B, int H, int S, int d, dab_mask_t mask,
                                   dab_sched_t sched, int chunks);

dab_status_t dab_attn_bwd_host(const void* q, const void* k, const void* v,
                               const void* o, const float* lse, const void* dout,
                               void* dq, void* dk, void* dv,
                               int B, int H, int S, int d, float scale,
                               dab_mask_t mask, dab_sched_t sched,
                               void* dev_ws, size_t dev_ws_bytes, int chunks,
                               cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Schedule introspection (host only, no GPU needed).  N = S/128 tiles.
 * These are the same functions the main kernel evaluates on the device.     */

/* Work units per head: N, or N/2 for causal SHIFT (one unit = a KV pair).   */
int dab_sched_units_per_head(dab_sched_t sched, dab_mask_t mask, int N);
/* Steps (KV tile, Q tile) of unit u, in execution order.                    */
int dab_sched_unit_steps(dab_sched_t sched, dab_mask_t mask, int N, int u);
/* Step t of unit u: its KV tile i and Q tile j.  Returns 0, or -1 if out of
 * range.                                                                     */
int dab_sched_step(dab_sched_t sched, dab_mask_t mask, int N, int u, int t,
                   int* kv_tile, int* q_tile);
/* rank(i, j): the position of KV tile i in dQ_j's fixed reduction order
 * (0 = first), -1 if tile (i, j) is masked out or for ATOMIC.              */
int dab_sched_rank(dab_sched_t sched, dab_mask_t mask, int N, int i, int j);
/* Number of KV tiles that contribute to dQ_j.                               */
int dab_sched_contributors(dab_mask_t mask, int N, int j);
/* Units that must run at the same time for progress (1 when none must).     */
int dab_sched_gang_size(dab_sched_t sched, dab_mask_t mask, int N);

/* DAG model of one schedule (DASH summary sec. 2.1): a node per (KV tile,
 * Q tile) step made of a compute phase of weight wc and a reduction phase of
 * weight wr; edges are the KV-chain order and the dQ_j reduction order.
 * `reducer_depth` = 0 runs the reduction inside the chain (the next compute
 * waits for it); k > 0 lets up to k reductions trail the compute phases.
 * `heads` heads run on `ctas` processors that take units in dispatch order.
 * Outputs the makespan and the busy fraction (sum of weights / (ctas *
 * makespan)).  Returns 0, -1 on bad arguments, -2 if the units deadlock
 * (a gang that cannot be co-resident).                                      */
int dab_dag_simulate(dab_sched_t sched, dab_mask_t mask, int N, int heads,
                     int ctas, double wc, double wr, int reducer_depth,
                     double* makespan, double* busy_fraction);

/* The same model with `ways` interleaved accumulation buffers per dQ tile
 * (the main kernel uses four for the ordered schedules): the reduction of
 * rank r waits only for that of rank r - ways.  ways = 1 is
 * dab_dag_simulate().                                                       */
int dab_dag_simulate_ways(dab_sched_t sched, dab_mask_t mask, int N, int heads,
                          int ctas, double wc, double wr, int reducer_depth,
                          int ways, double* makespan, double* busy_fraction);

/* Schedule selection, the "palette" of DASH (technical summary section 4:
 * which schedule is best depends on the mask and the shape).  Returns the
 * deterministic schedule (SERIAL, DESCENDING_Q or SHIFT) with the smallest
 * makespan in the DAG model of dab_dag_simulate_ways() for B*H heads of
 * S/128 tiles on `ctas` CTAs, with weights fitted to this library's GB300
 * measurements (wr = wc, reducer_depth 1, 4 buffers).  SHIFT's predicted
 * makespan is multiplied by 1.025 before the comparison.  This accounts for
 * its lock-step rings, which the model does not capture; the factor was
 * fitted to the measured GB300 sweep.  Ties go to DESCENDING_Q, then SERIAL.
 * Host only, no CUDA call; -1 on bad arguments.
 * Results are cached per (mask, B*H, S, ctas); thread-safe.                 */
int dab_sched_select(dab_mask_t mask, int B, int H, int S, int ctas);

/* Longest path of one head's DAG with one processor per unit.               */
double dab_dag_critical_path(dab_sched_t sched, dab_mask_t mask, int N,
                             double wc, double wr, int reducer_depth);

#ifdef __cplusplus
}
#endif

#endif /* DAB_H_ */
