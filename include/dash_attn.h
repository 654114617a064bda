/*
 * dash_attn.h -- C ABI of the deterministic attention backward with DASH schedules.
 *
 * Source of the method: "DASH: Deterministic Attention Scheduling for High-throughput
 * Reproducible LLM Training" (ICLR 2026; arXiv 2601.21824), as summarised on its research
 * map page (sections "Problem" and "Approach") and in its Pith review ("The pith",
 * "Core claim", "What carries the argument", the referee report and Figures 1-7).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Tensors Q, K, V, O, dO, dQ, dK, dV are bf16, contiguous, BSHD: element (b, s, h, d)
 *   sits at index ((b * S + s) * H + h) * D + d. LSE is fp32 [B, H, S], natural log of
 *   the sum of exp(scale * q.k) over the keys a query may see.
 * - Supported: D in {64, 128}; S a positive multiple of 128; B, H >= 1;
 *   B * H * S * D < 2^31. Anything else returns DASH_ERR_UNSUPPORTED.
 * - The causal mask is top-left aligned (query i sees keys 0..i).
 * - All device pointers are owned by the caller and must stay valid until the work
 *   queued on `stream` has finished. The library allocates nothing per call; it keeps a
 *   cache of schedule tables per device and shape, built on first use: the task tables
 *   (O(n^2) int32 per schedule) and, for SHIFT and SYMMETRIC_SHIFT, the per-head dQ
 *   orders of the grid in use (B * H * n^2 int32, n = S / 128: 0.5 MB for 2x16 heads at
 *   S = 8192), on the device and in host memory. dash_attn_shutdown releases all of it.
 * - Calls are asynchronous on `stream`. Argument errors are returned synchronously and
 *   queue no work. Device-side failures (a reduction wait that timed out) are recorded
 *   in the workspace and reported by dash_attn_get_status.
 * - Pointers must be 16-byte aligned.
 */
#ifndef DASH_ATTN_H
#define DASH_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Attention mask. */
typedef enum { DASH_MASK_FULL = 0, DASH_MASK_CAUSAL = 1 } dash_mask_t;

/*
 * Task orders (research map page, "Approach"; Pith review, "What carries the argument";
 * Figure 3, 4, 6 and 7 captions). KV tile i always runs all of its tasks on one SM.
 * - ASCENDING: the FlashAttention-3 baseline; KV_i visits Q tiles upwards.
 * - DESCENDING: Descending Q-Tile Iteration; KV_i visits Q tiles downwards.
 * - SHIFT: Shift Scheduling (full mask only); at step t KV_i works on Q_((i+t) mod n).
 * - SYMMETRIC_SHIFT: Symmetric Shift (causal mask only, n even); one SM slot takes
 *   KV_p and KV_(n-1-p): phase 1 shifts over the dense lower-left rectangle, phase 2
 *   runs the folded triangles from the diagonal, upper-left first.
 * The dQ_j reduction order is ascending KV index for ASCENDING and DESCENDING, and the
 * arrival step for SHIFT and SYMMETRIC_SHIFT.
 */
typedef enum {
  DASH_SCHED_ASCENDING = 0,
  DASH_SCHED_DESCENDING = 1,
  DASH_SCHED_SHIFT = 2,
  DASH_SCHED_SYMMETRIC_SHIFT = 3
} dash_sched_t;

typedef enum {
  DASH_OK = 0,
  DASH_ERR_INVALID_ARG = 1,         /* null pointer, negative size, bad enum value */
  DASH_ERR_UNSUPPORTED = 2,         /* valid but not implemented (head dim, mask/schedule pair) */
  DASH_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < dash_attn_bwd_workspace_size() */
  DASH_ERR_CUDA = 4,                /* a CUDA runtime call failed; see dash_last_error() */
  DASH_ERR_SYNC_TIMEOUT = 5,        /* a wait (dQ semaphore or in-kernel pipeline) hit its limit */
  DASH_ERR_DEADLOCK_RISK = 6,       /* the schedule's waits form a cycle on this grid */
  DASH_ERR_BOUNDS = 7               /* checked build: a table index failed a device-side check */
} dash_status_t;

/*
 * Forward pass: O = softmax(scale * Q K^T [+ causal mask]) V and LSE per query row.
 * Produces the two inputs the backward recomputes P from (FlashAttention-3's forward,
 * named on the research map page under "Builds on").
 *   q, k, v : [B, S, H, D] bf16 (read)      o : [B, S, H, D] bf16 (written)
 *   lse     : [B, H, S] fp32 (written)      mask : dash_mask_t
 * Returns DASH_OK or an argument/CUDA error; nothing is queued on error. Every wait
 * inside the kernel is bounded; a CTA whose wait runs out writes NaN into its LSE rows
 * (dash_attn_fwd_ex also reports it through a status word).
 */
dash_status_t dash_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int S, int H, int D, float scale, int mask,
                            cudaStream_t stream);

/*
 * dash_attn_fwd with a device status word:
 *   status : optional device int32 (4-byte aligned; NULL = none). The call clears it on
 *            `stream` before the kernel; when any wait inside the kernel runs out (which
 *            only a fault can cause) the kernel sets it to DASH_ERR_SYNC_TIMEOUT and that
 *            CTA's O and LSE rows are undefined (LSE NaN). Read it after the stream has
 *            finished the call; the CUDA context stays usable either way.
 * Same arguments, conventions and errors as dash_attn_fwd otherwise.
 */
dash_status_t dash_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int S, int H, int D, float scale, int mask, int* status,
                               cudaStream_t stream);

/*
 * Bytes of scratch dash_attn_bwd needs for this shape: a status header, D = rowsum(dO*O)
 * and -LSE*log2(e) (two fp32 [B,H,S] arrays), two score-offset block arrays (-LSE/scale
 * and -D as three bf16 terms each, 32 bytes per row), two copies of the fp32 dQ accumulator
 * [2,B,H,S,D] (deterministic = 2 uses both), one 128-byte line of int32 semaphores per
 * 128-row dQ block, one semaphore per chain [B,H,S/128,32], 256 x 4 int32 split-tile flags
 * and the fp32 dK/dV partials of the KV tiles a grid may split over two CTAs
 * (dash_sched_deal): min(B*H*S/128 / 2, 256) tiles of [2][128][D]. Returns 0 for an
 * unsupported shape.
 */
size_t dash_attn_bwd_workspace_size(int B, int S, int H, int D);

/*
 * Backward pass (the DASH problem statement: research map page "Problem"; Pith review
 * "Core claim"). Recomputes P from Q, K and LSE, then forms dV, dP, dS, dK and dQ. Each
 * KV tile's dK/dV accumulates on one SM. Each dQ block is the sum of one partial per KV
 * tile that sees it:
 *   deterministic = 1: the partials are added in the fixed order `schedule` defines,
 *                      serialised through semaphores per dQ block. The result is
 *                      bitwise identical for identical inputs, shape and schedule on the
 *                      same GPU model and build. Different schedules may differ in the
 *                      last bits (their dQ orders differ). SHIFT and SYMMETRIC_SHIFT
 *                      order by arrival on the persistent grid of min(SMs, B*H*chains)
 *                      CTAs (dash_sched_dealt_table), so their bits also depend on the
 *                      GPU's SM count.
 *   deterministic = 2: the same fixed order run as two interleaved chains: the partial
 *                      at position p of the order is added, in order, into fp32
 *                      accumulator copy p mod 2, after the partial at position p - 2, and
 *                      dQ = copy 0 + copy 1. A partial waits only for the one two places
 *                      before it, so the hand-off between SMs leaves the critical path.
 *                      Bitwise identical run to run like 1 (its bits differ from 1's: the
 *                      additions are grouped differently).
 *   deterministic = 0: the partials are added atomically in arrival order (the speed
 *                      reference; results vary in the last bits run to run).
 *   q, k, v, o, dO : [B, S, H, D] bf16 (read);  lse : [B, H, S] fp32 (read)
 *   dq, dk, dv     : [B, S, H, D] bf16 (written; must not alias the inputs)
 *   workspace      : device scratch of at least dash_attn_bwd_workspace_size() bytes,
 *                    256-byte aligned, not shared with work running concurrently.
 *   schedule       : dash_sched_t. SHIFT needs the full mask, SYMMETRIC_SHIFT the causal
 *                    mask; other pairs return DASH_ERR_UNSUPPORTED.
 * Returns DASH_ERR_DEADLOCK_RISK (nothing queued) if the schedule's reduction waits would
 * form a cycle on the persistent grid this GPU can hold (none of the four schedules'
 * orders can: ascending KV index is the dealing order, and arrival orders follow it).
 */
dash_status_t dash_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                            const void* dO, const float* lse, void* dq, void* dk, void* dv,
                            void* workspace, size_t workspace_bytes,
                            int B, int S, int H, int D, float scale, int mask, int schedule,
                            int deterministic, cudaStream_t stream);

/*
 * Backward pass that allocates no device memory. The DASH paper has no counterpart to
 * this call; it exists for callers that cannot allocate device memory when they run the
 * backward -- for example a framework that reserves all device memory up front for its
 * own pool, or code that must not enter the CUDA allocator at that point. It computes
 * the same result as dash_attn_bwd (same kernels, same schedule, same reduction order).
 *
 * Instead of a caller-supplied workspace it uses a fixed 64 MiB array that is part of the
 * library's device image: every GPU that loads the library holds it until the process
 * exits. Shapes whose scratch (dash_attn_bwd_workspace_size() plus the schedule tables)
 * does not fit return DASH_ERR_WORKSPACE_TOO_SMALL with the sizes in dash_last_error();
 * use dash_attn_bwd for those.
 *   q .. dv, B .. stream : as for dash_attn_bwd.
 *   status_out : optional device int (may be NULL); after the kernels it receives the
 *                status word that dash_attn_get_status would report (0 = ok).
 * The first call on a device looks up the array's device address (with that device
 * current); make that first call before any stream capture. dash_attn_shutdown forgets
 * the address, and the next call looks it up again. Every call on a device shares the one
 * array and leaves its contents behind (the kernels clear what has to start at zero), so
 * calls whose work overlaps on the GPU -- on different streams or from different
 * threads -- race with each other and must be serialised by the caller.
 * No cudaMalloc, cudaFree or other allocating CUDA routine is called. The schedule tables
 * are built once per shape in host memory, kept there until dash_attn_shutdown, and
 * copied into the array with one cudaMemcpyAsync on `stream` per call. Every refusal
 * (argument, size, tensor-map, register, occupancy and deadlock checks) happens before
 * that copy, so a refused call queues nothing and leaves the array as it was.
 */
dash_status_t dash_attn_bwd_static(const void* q, const void* k, const void* v, const void* o,
                                   const void* dO, const float* lse, void* dq, void* dk,
                                   void* dv, int* status_out, int B, int S, int H, int D,
                                   float scale, int mask, int schedule, int deterministic,
                                   cudaStream_t stream);

/*
 * Synchronises `stream` and reads the status header of `workspace` written by the last
 * dash_attn_bwd on it: DASH_OK, or DASH_ERR_SYNC_TIMEOUT when a wait ran out -- a dQ
 * semaphore wait, or a hand-off between the warps of one CTA -- after which the kernel
 * abandons its remaining work and the outputs are undefined (dash_last_error() says
 * which). In the checked build (dash_bounds_checks_enabled() == 1) also
 * DASH_ERR_BOUNDS: an index read from the schedule tables failed its check, the CTA
 * stopped before using it, and dash_last_error() names the table, the head, the value
 * and the bound. Also returns DASH_ERR_CUDA if the stream reports an error.
 */
dash_status_t dash_attn_get_status(const void* workspace, cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* dash_status_string(int status);

/* Text of the last CUDA error seen by this thread inside the library ("" if none). */
const char* dash_last_error(void);

/* Frees the cached schedule tables on every device. Safe to call more than once. */
void dash_attn_shutdown(void);

/*
 * Testing hook for the failure paths. Sets, for later dash_attn_bwd and dash_attn_fwd(_ex)
 * calls in this process, the time limit of one wait (timeout_ns <= 0 restores the default
 * of 10 s) and a skew. In the backward the skew is added to every awaited dQ ordinal; in
 * the forward a skew > 0 makes the kernel load no K/V tiles. Either way no wait on them
 * can be satisfied: each one runs out its limit, the kernel records DASH_ERR_SYNC_TIMEOUT
 * (backward: in the workspace; forward: in dash_attn_fwd_ex's status word) and returns,
 * and the CUDA context stays usable. Not thread-safe against concurrent calls.
 */
void dash_debug_set_sync(long long timeout_ns, int ordinal_skew);

/*
 * Device-side bounds checks. The library is built in two forms: the product build, and a
 * checked build (libdash_attn_checked.so, compiled with DASH_BOUNDS_CHECKS=1) whose
 * backward checks every index it reads from its schedule tables before using it -- a
 * CTA's range of pieces, each piece's head, task range and split tile, each task's two
 * tile indices, each dQ ordinal -- and, on a failure, records DASH_ERR_BOUNDS in the
 * workspace header and stops that CTA's work (no trap; the context stays usable). It
 * stands in for a memory checker. Returns 1 in the checked build, 0 in the product build.
 */
int dash_bounds_checks_enabled(void);

/*
 * Testing hook of the checked build. Lowers by `tiles` the tile bound that the checks
 * compare task indices and dQ ordinals against (0 restores it), for later dash_attn_bwd
 * calls in this process; the kernel's own indexing is unchanged, so valid tables then
 * fail the checks without any access going out of bounds. Returns DASH_OK,
 * DASH_ERR_INVALID_ARG (tiles < 0), or DASH_ERR_UNSUPPORTED in the product build.
 */
dash_status_t dash_debug_narrow_checks(int tiles);

/*
 * Tracing hook. When device_counters is not NULL, later dash_attn_bwd main kernels add,
 * per CTA, the clock cycles spent in each of their waits into
 * device_counters[cta * 32 + site] (uint64). Sites with a fixed meaning in both kernels:
 *   15 : waiting for a dQ block's turn (the ordered mode's semaphore wait),
 *   16 : adding a dQ partial into the accumulator and handing the turn on,
 *   19 : the CTA's total cycles.
 * The other sites (producer, MMA-issue and softmax-gradient waits) are listed in the
 * library's sources. The buffer must hold 32 counters per SM of the device, zeroed by
 * the caller. NULL turns tracing off.
 */
void dash_debug_set_trace(void* device_counters);

/*
 * Profiling hook. With on != 0, every later dash_attn_bwd records a pair of CUDA events
 * on its stream, immediately before and after its main (compute + dQ reduction) kernel,
 * up to 1024 pairs. dash_profile_read waits for the recorded events, writes the summed
 * main-kernel milliseconds and the number of launches, and forgets them. on = 0 stops
 * recording. Returns a dash_status_t.
 */
dash_status_t dash_profile_enable(int on);
dash_status_t dash_profile_read(double* total_ms, int* launches);

/* ---- Schedule model (host only; no GPU needed) ------------------------------------ */

/*
 * Number of chains ("SM slots") per head for (mask, schedule) over n KV tiles:
 * n for ASCENDING/DESCENDING/SHIFT, n/2 for SYMMETRIC_SHIFT. Negative dash_status_t
 * value on an unsupported pair or n < 1 (or odd n for SYMMETRIC_SHIFT).
 */
int dash_sched_num_slots(int mask, int schedule, int n);

/*
 * Copies the task table the kernel follows.
 *   slot_offsets : int32[num_slots + 1]; chain p is tasks[slot_offsets[p] .. slot_offsets[p+1])
 *   tasks        : int32[cap]; each entry packs (kv_tile << 16) | q_tile, in execution order
 *   ordinals     : int32[n * n]; ordinals[i * n + j] = position of KV_i's partial in the dQ_j
 *                  reduction order, or -1 where the mask removes task (i, j). This is the
 *                  schedule's order when all chains of a head start together (one head on
 *                  n SMs); dash_sched_dealt_table gives the orders the kernel follows.
 * Returns the number of tasks, or a negative dash_status_t value (cap too small:
 * -DASH_ERR_INVALID_ARG).
 */
int dash_sched_table(int mask, int schedule, int n, int32_t* slot_offsets, int32_t* tasks,
                     int cap, int32_t* ordinals);

/*
 * How dash_attn_bwd spreads `heads` (= B * H) heads' chains over `grid` persistent CTAs
 * at head dimension `head_dim` (64 or 128). Round robin -- unit u (head u / num_slots,
 * chain slot u % num_slots) whole to CTA u % grid -- unless the schedule orders dQ by
 * arrival (SHIFT, SYMMETRIC_SHIFT) and the units overrun whole rounds of the grid (more
 * units than CTAs, not a multiple of them). Then chains are cut where their KV tile
 * changes and the pieces dealt longest first (equal lengths in head-major chain order),
 * each to the CTA with the least work dealt so far (the lower index on a tie); each CTA
 * runs its pieces in the order dealt. At head dimension 64 every unit is cut this way; at
 * 128 the first q - 1 of the q whole rounds stay round robin (whole units, keeping each
 * head's chains on concurrent CTAs and its tiles in L2) and only the units after them are
 * cut. Shift's units are single KV tiles of one length, dealt round robin all the same;
 * there, when the last partial round holds r units with 2 r <= grid (r <= 256), each of
 * those r KV tiles is split in two halves (the first ceil(len / 2) tasks, then the rest):
 * split k's first half runs on CTA k and its second half on CTA r + k, after their whole
 * units. The first half hands its fp32 dK/dV partial to the second, which adds its own (in
 * that order) and writes dK/dV. This balancing is the library's own (the pages study one
 * head on n SMs). Outputs:
 *   cta_offsets : int32[grid + 1]; CTA c runs pieces cta_offsets[c] .. cta_offsets[c + 1]
 *   pieces      : int32[5 * cap]; piece k = (head, first task, end task, part, split), the
 *                 tasks being indices into dash_sched_table's task table; part 0 = whole
 *                 KV tiles, 1 / 2 = first / second half of split tile `split` (0 for part 0)
 * Returns the number of pieces, or a negative dash_status_t value (heads or grid < 1,
 * head_dim not 64 or 128, null outputs, cap too small: -DASH_ERR_INVALID_ARG; an
 * unsupported (mask, schedule, n): the schedule's error).
 */
int dash_sched_deal(int mask, int schedule, int n, int heads, int grid, int head_dim,
                    int32_t* cta_offsets, int32_t* pieces, int cap);

/*
 * The dQ orders dash_attn_bwd follows at head dimension `head_dim` when `heads` (= B * H)
 * heads' chains are dealt onto `grid` persistent CTAs as dash_sched_deal describes:
 *   ordinals : int32[heads * n * n]; ordinals[(h * n + i) * n + j] = position of KV_i's
 *              partial in head h's dQ_j order, -1 where the mask removes the task.
 * ASCENDING and DESCENDING: ascending KV index in every head. SHIFT and SYMMETRIC_SHIFT
 * (whose order the pages define as the order of arrival): a partial's place in its
 * CTA's task sequence -- the tasks of the CTA's earlier pieces, then its step in the
 * piece -- the lower KV index first on a tie. With whole heads per round of the grid this
 * is dash_sched_table's order; when the grid splits a head over two rounds, the chains run
 * in the earlier round come first, so no partial waits for a chain that has not started.
 * Returns DASH_OK, DASH_ERR_INVALID_ARG (heads or grid < 1, head_dim not 64 or 128, null
 * ordinals), or the schedule's error for an unsupported (mask, schedule, n).
 */
dash_status_t dash_sched_dealt_table(int mask, int schedule, int n, int heads, int grid,
                                     int head_dim, int32_t* ordinals);

/*
 * Critical path of the compute/reduce DAG (Pith review, "What carries the argument"):
 * every task is a compute phase of cost c then a reduce phase of cost r; one SM runs its
 * tasks back to back; reductions into one dQ block follow the orders the kernel uses on a
 * grid of num_sms CTAs (dash_sched_dealt_table(mask, schedule, n, heads, num_sms,
 * head_dim)). `heads` heads' chains are dealt onto `num_sms` SMs as the kernel deals them
 * at head dimension `head_dim` (dash_sched_deal); the second half of a split KV tile ends
 * no earlier than its first half. Writes the makespan and, if sm_end is not NULL, each SM's
 * finish time (double[num_sms]). Returns DASH_ERR_DEADLOCK_RISK when the waits form a
 * cycle, DASH_ERR_INVALID_ARG for bad arguments (head_dim not 64 or 128).
 */
dash_status_t dash_sched_simulate(int mask, int schedule, int n, int heads, int num_sms,
                                  int head_dim, double c, double r, double* makespan,
                                  double* sm_end);

/*
 * The same critical path with synchronisation cost (the Pith review's "Where Pith is
 * reading between the lines" proposes nonzero edge costs; its Axiom & Free-Parameter
 * Ledger lists zero-cost order edges as a domain assumption):
 *   h          : cost of handing a dQ block's turn from one SM to another (the order edge's
 *                weight; 0 when consecutive reductions of the block run on one SM);
 *   overlapped : 0 = the SM runs C then R task after task (dash_sched_simulate's model);
 *                1 = two engines per SM: C phases in order, R phases in order, and the
 *                k-th task's C waits for the (k-2)-th task's R (the accumulator reuse of
 *                this library's kernels, which read one dQ partial out while the next
 *                is computed).
 * With h = 0 and overlapped = 0 the result equals dash_sched_simulate's. Same outputs and
 * errors as dash_sched_simulate; DASH_ERR_INVALID_ARG for a negative cost or overlapped
 * not in {0, 1}.
 */
dash_status_t dash_sched_simulate_ex(int mask, int schedule, int n, int heads, int num_sms,
                                     int head_dim, double c, double r, double h, int overlapped,
                                     double* makespan, double* sm_end);

/*
 * Run-time schedule selector: among the schedules defined for `mask` and n (ascending and
 * descending always; shift for the full mask; symmetric shift for the causal mask and even
 * n) whose waits are acyclic on `num_sms` SMs, the one with the smallest
 * dash_sched_simulate_ex makespan at head dimension `head_dim` (ties: the lower enum
 * value). Writes it to *schedule_out and, if makespan_out is not NULL, its makespan. The
 * pages pick schedules by configuration (Descending vs Symmetric Shift at d = 128, Shift vs
 * the baseline at long sequences); this makes that choice from the cost model. Costs
 * measured on GB300 with this library (head dim 128, cycles per 128x128 task): c ~ 6900,
 * r ~ 5600, h ~ 3000, overlapped = 1. Returns DASH_ERR_INVALID_ARG for bad arguments.
 */
dash_status_t dash_sched_select(int mask, int n, int heads, int num_sms, int head_dim, double c,
                                double r, double h, int overlapped, int* schedule_out,
                                double* makespan_out);

/*
 * Deterministic split-K GEMM with the same ordered cross-SM reduction (the Pith review's
 * section "Where Pith is reading between the lines" lists split-K GEMMs among the kernels
 * the reduction-order principle applies to): C = A B^T with
 *   a : bf16 [M, K] row-major (read);  b : bf16 [N, K] row-major (read);
 *   c : fp32 [M, N] row-major (written: zeroed, then every K chunk's partial added);
 *   workspace : device scratch of dash_gemm_splitk_workspace_size(M, N) bytes, 256-byte
 *               aligned (status header + room for one int32 semaphore per 128 x 128 block
 *               of C; the kernel's output tiles are 256 x 128 when M is a multiple of 256
 *               -- full-rate 256-wide MMAs -- else 128 x 128, one semaphore each);
 *   splits : K is cut into `splits` equal chunks, one unit of work each per output tile;
 *   deterministic = 1: a tile's chunks are added in ascending chunk order (bitwise
 *               identical run to run); 0: in arrival order.
 * Requires M, N multiples of 128, K a multiple of 64 * splits, M * N < 2^31
 * (else DASH_ERR_UNSUPPORTED). Asynchronous on `stream`; dash_attn_get_status(workspace)
 * reports a timed-out wait (DASH_ERR_SYNC_TIMEOUT) as for the backward.
 */
size_t dash_gemm_splitk_workspace_size(int M, int N);
dash_status_t dash_gemm_splitk(const void* a, const void* b, float* c, void* workspace,
                               size_t workspace_bytes, int M, int N, int K, int splits,
                               int deterministic, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DASH_ATTN_H */
