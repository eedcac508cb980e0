/*
 * dash.h - C ABI of the GB300 (sm_103a) deterministic attention library.
 *
 * The library computes softmax attention forward (O, LSE) and, above all, the
 * attention backward pass (dQ, dK, dV from Q, K, V, O, dO, LSE) with a dQ
 * reduction whose order is fixed by a schedule, so that every deterministic
 * schedule returns bit-identical gradients on every run.  The schedules are
 * those of "DASH: Deterministic Attention Scheduling for High-throughput
 * Reproducible LLM Training" as presented in the DASH overview (zskr.cn),
 * sections 2.1-3.3, and Sintesi Tecnica DASH (gist.science/it), sections
 * 1-2.2.
 *
 * Conventions shared by every entry point
 *  - Tensors are contiguous row-major [B][H][S][D] ("BHSD").  q, k, v, o, dout,
 *    dq, dk, dv are bf16 (IEEE bfloat16, 2 bytes); lse is fp32 [B][H][S],
 *    natural log with the scale inside: lse_i = log(sum_j exp(scale*q_i.k_j)).
 *  - Device pointers unless a function says "host".  The caller owns every
 *    buffer it passes; pointers must be 16-byte aligned.
 *  - D must be 64 or 128; B, H, S >= 0 (an empty problem is a no-op that
 *    returns DASH_OK).  S need not be a multiple of the tile: the ragged tail is
 *    masked.  Causal masking is square and top-left aligned (query i attends
 *    keys j <= i).  scale must be finite and > 0.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call returns after enqueueing.  A device-side failure
 *    (a bounded wait that ran out) is recorded in a status word that
 *    dash_sync_status() reads.
 *  - Errors are returned as dash_status_t; no exception crosses the ABI.
 *    dash_last_error() describes the last failure of the calling thread.
 *  - The library keeps a per-(device, stream) workspace (fp32 dQ accumulator,
 *    per-row softmax statistics, semaphores, status word) and a cache of
 *    schedule tables.  It grows the buffers that only the call's stream uses
 *    with cudaMallocAsync / cudaFreeAsync on that stream on first use of a
 *    larger shape (the status word and the tables with cudaMalloc, once);
 *    dash_release_workspace() frees them.  Two calls that run
 *    concurrently on the same stream cannot overlap, so the workspace is never
 *    shared by concurrent kernels.
 */
#ifndef DASH_H_
#define DASH_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared opaquely so that C callers need no CUDA headers. */
typedef struct CUstream_st *dash_stream_t;

/* Order in which the backward reduces dQ partials (DASH overview, section 3;
 * Sintesi Tecnica DASH, section 2.2).  A chain is the list of Q tiles that one
 * KV tile visits on one CTA; the rank of a task is its position in its dQ
 * tile's reduction order. */
typedef enum {
  DASH_SCHED_ATOMIC = 0,          /* serial chains, unordered fp32 adds: NOT deterministic (reference point) */
  DASH_SCHED_SERIAL = 1,          /* KV j visits Q tiles ascending; dQ reduced in ascending KV order (FA3's order, overview section 2.1) */
  DASH_SCHED_DESCENDING_Q = 2,    /* KV j visits Q tiles descending; ascending KV reduction order (overview section 3.1) */
  DASH_SCHED_SHIFT = 3,           /* full mask only: KV j visits Q tiles (j+t) mod n; reduced in step order (overview section 3.2) */
  DASH_SCHED_SYMMETRIC_SHIFT = 4  /* causal only, n even: slot p runs KV p then KV n-1-p, dense rectangle then folded triangle (overview section 3.3) */
} dash_schedule_t;

typedef enum {
  DASH_OK = 0,
  DASH_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad scale, misaligned pointer */
  DASH_ERR_UNSUPPORTED = 2,   /* D not 64/128, schedule invalid for the mask, odd n for symmetric shift, too few SMs,
                               * or more tasks than 32-bit task tables index (2^31 - 1) */
  DASH_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (message in dash_last_error) */
  DASH_ERR_TIMEOUT = 4,       /* a bounded device wait ran out (reported by dash_sync_status) */
  DASH_ERR_NO_MEMORY = 5,     /* workspace allocation failed */
  DASH_ERR_SCHEDULE = 6       /* the schedule simulation deadlocked or a supplied task table is malformed */
} dash_status_t;

/* Task-table encoding used by dash_build_schedule and dash_bwd_options_t:
 * four int32 per task {bh, kv_block, q_block, word} with
 * word = rank | (first ? DASH_TASK_FIRST : 0) | (last ? DASH_TASK_LAST : 0). */
#define DASH_TASK_RANK_MASK 0x00FFFFFF
#define DASH_TASK_FIRST (1 << 28) /* first task of a run on one KV tile: dK/dV accumulators start at zero */
#define DASH_TASK_LAST (1 << 29)  /* last task of a run on one KV tile: dK/dV are written out */

/* Softmax attention forward (the input side of the backward; the DASH pages
 * take it as given).  o[b,h,i,:] = sum_j P_ij v[b,h,j,:] with
 * P_ij = exp(scale*q_i.k_j - lse_i); writes o (bf16) and lse (fp32). */
dash_status_t dash_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int H, int S, int D, int causal, float scale,
                            dash_stream_t stream);

/* dash_attn_fwd with a choice of kernel.  cta_pair = 0: one CTA per 128-row Q
 * tile; 1: a pair of CTAs (a cluster of two) per two Q tiles, whose MMAs are
 * tcgen05 CTA-pair MMAs (cta_group::2, M = 256): each CTA loads half of every
 * K and V tile and the pair's first CTA issues the MMAs (D = 128 only,
 * DASH_ERR_UNSUPPORTED otherwise); -1: the library's default for D.  The
 * results agree within rounding (the same sums, formed by other MMA shapes). */
dash_status_t dash_attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                               int B, int H, int S, int D, int causal, float scale, int cta_pair,
                               dash_stream_t stream);

/* Attention backward (DASH overview, section 2.1; Sintesi Tecnica DASH,
 * section 1).  With P as above, dP = dO V^T, delta_i = dO_i.O_i,
 * dS = P*(dP - delta):  dv = P^T dO, dk = scale * dS^T Q, dq = scale * dS K,
 * written as bf16.  Each KV tile's work stays on one CTA with dK/dV
 * accumulated in tensor memory; dQ partials are added into an fp32 workspace
 * in the order `schedule` fixes, enforced by per-dQ-tile semaphores.  Every
 * schedule except DASH_SCHED_ATOMIC gives bit-identical results run to run. */
dash_status_t dash_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                            const void *dout, const float *lse,
                            void *dq, void *dk, void *dv,
                            int B, int H, int S, int D, int causal, float scale,
                            dash_schedule_t schedule, dash_stream_t stream);

/* Options of dash_attn_bwd_ex; zero-initialise and set what you need. */
typedef struct {
  int tile;                /* 0 = auto (64 when S <= 256, else 128), or 64 / 128 */
  int num_ctas;            /* 0 = choose by simulation; else exactly this many persistent CTAs */
  int cost_c, cost_r;      /* simulator costs used to place chains on CTAs (0 = 4 and 1) */
  long long spin_limit_ns; /* bound on each device wait (0 = 2 s) */
  float *dq_accum_out;     /* optional device fp32 [B,H,S,D]: receives the unscaled dQ accumulator */
  const int32_t *tasks;    /* optional HOST task table that replaces the generated one (testing) */
  const int32_t *cta_off;  /* with tasks: HOST array of num_ctas+1 offsets into tasks */
  void *main_begin_event;  /* optional cudaEvent_t recorded on `stream` just before the main kernel */
  void *main_end_event;    /* optional cudaEvent_t recorded on `stream` just after it (timing) */
  int dq_chains;           /* ordered schedules: 0 or 1 = one chain per dQ tile, the pages' order; 2 = two
                            * chains (an extension beyond the pages): the tile's even ranks add into one fp32
                            * accumulator and its odd ranks into another, each in rank order behind its own
                            * semaphore, and dQ = chain 0 + chain 1.  Deterministic, with a different
                            * summation order from 1.  With num_ctas = 0, shift then takes every SM
                            * instead of whole gangs.  Ignored by the atomic schedule. */
  int shift_fill;          /* DASH_SCHED_SHIFT and DASH_SCHED_SYMMETRIC_SHIFT, with one or two chains:
                            * 0 = the pages' schedule; 1 = with fill (an extension beyond the pages): whole
                            * gangs of CTAs run
                            * the schedule for most heads, and the CTAs they leave idle run the other heads
                            * with a fill schedule (serial or descending_q), as dash_build_shift_fill lays out.
                            * Each head keeps its own schedule's dQ order, so the result is deterministic;
                            * the filled heads' bits are the fill schedule's.  num_ctas, if set, is the CTA
                            * budget. */
  int trust_table;         /* with tasks: 0 = check the table's dQ orders on the host before the launch
                            * (dash_check_table; DASH_ERR_SCHEDULE if they could not finish); 1 = bounds
                            * checks only, so that an inconsistent table reaches the device, whose bounded
                            * waits then report DASH_ERR_TIMEOUT (testing). */
  int64_t *trace;          /* optional device int64 [n_tasks][DASH_TRACE_SLOTS], 8-byte aligned (profiling):
                            * runs the traced build of the main kernel, which stamps each task's phases
                            * (slots below) into the row of the task's position in the table.  Same
                            * results, bit for bit, as the plain kernel.  128-row tiles only
                            * (DASH_ERR_UNSUPPORTED otherwise). */
  int die_aware;           /* DASH_SCHED_SHIFT and DASH_SCHED_SYMMETRIC_SHIFT without fill or a supplied table:
                            * 0 = CTAs as the hardware places them; 1 = die-aware placement (an extension):
                            * the main kernel runs one CTA per SM, and each SM takes the task list the host
                            * gave it, so that every whole gang of chains runs on SMs of one die, and each dQ
                            * tile's semaphore sits in an L2 line homed on the die that runs most of its adds.
                            * The first such call on a (device, stream) measures the die map (a probe kernel
                            * of a few milliseconds, and a synchronisation of the stream).  The tasks, ranks
                            * and adds are those of the plain schedule, so the results are the same bits.
                            * DASH_ERR_UNSUPPORTED when the map shows no two groups of SMs. */
  int cluster_size;        /* ordered schedules with the library's own table: the persistent CTAs run in
                            * thread-block clusters of this size, and a rank whose predecessor in its dQ
                            * tile's order runs in the same cluster takes its turn from a counter in its
                            * own shared memory, which the predecessor raises after its release (the global
                            * semaphore is released as well).  The ranks and adds do not change, so neither
                            * do the results.  0 or 1 = no clusters (the hand-off through the global
                            * semaphore alone measured faster); 2, 4, 8, 16 = that size
                            * (DASH_ERR_UNSUPPORTED if it does not divide the CTA count or the GPU cannot
                            * hold that many clusters at once).  Not with die_aware. */
  int shift_split;         /* DASH_SCHED_SHIFT and DASH_SCHED_SYMMETRIC_SHIFT with the library's own table,
                            * without fill: 0 or 1 = whole gangs (the pages' order); k > 1 = each head's gang
                            * of chains runs as k sub-gangs of consecutive chains.  A dQ tile's ranks then go in
                            * (sub-gang, step) order, every head's sub-gang 0 is dispatched before any sub-gang
                            * 1, and the CTA count may be any multiple of the sub-gang.  Deterministic, with its
                            * own bits.  k must divide the gang (n, or n/2 for symmetric shift);
                            * DASH_ERR_UNSUPPORTED otherwise, and with die_aware.  -1 = the library picks k
                            * by simulated makespan (dash_choose_split), where split gangs apply; with
                            * another schedule, fill, die_aware or a supplied table it means 0. */
  int rank_order;          /* ordered schedules with the library's own table, without fill or die_aware (an
                            * extension): 0 = each dQ tile's partials in the schedule's own order (the pages');
                            * 1 = timed ranks: in the order in which the simulated schedule reaches the tile
                            * (the compute-stage end of each task in a list-scheduling run without reduction
                            * order, ties by the chain's dispatch position, then step).  Where the schedule
                            * runs as its order assumes (whole shift gangs side by side, each tile visited
                            * step by step) the two orders are the same bits; where it does not (a gang spread
                            * over time, sub-gangs of one head side by side) timed ranks keep the order from
                            * stalling.  Without a split or num_ctas the CTA count is then every SM (up to
                            * the number of chains).  Deterministic, with its own bits. */
} dash_bwd_options_t;

/* Slots of a trace row.  "clk" = the SM's clock64, "ns" = the global timer.
 *  0 clk MMA warp starts dP^T         1 clk MMA warp has P, starts dV
 *  2 clk MMA warp has dS, starts dQ   3 clk MMA warp has issued the task's last MMA
 *  4 clk pass A starts (S^T landed)   5 clk pass A done (P in tensor memory)
 *  6 clk pass B starts                7 clk pass B done (dS in shared memory)
 *  8 clk dQ partial seen by the reduction warps
 *  9 clk dQ partial in registers, its tensor memory released
 * 10 ns  start of the wait for the dQ tile's turn   11 ns  turn taken (semaphore acquired)
 * 12 clk the reduction leader's adds are issued
 * 13 ns  every add of the task is issued; the release of rank + 1 starts
 * 14 clk read next to slot 10 (puts the two clocks on one axis)
 * 15 smid * 65536 + the CTA's slot (its task list)
 * 16 ns  the release store has returned (its fence is done)
 * 17 clk the last of the eight softmax warps is done with pass A
 * 18 clk the last of the eight softmax warps is done with pass B
 * 19 clk MMA warp has issued dV (and the next S^T when it goes early)
 * 20 clk MMA warp's wait for dS has returned
 * (slots 4-7 come from softmax warp 4; slots 10, 11 and 14 from the lane of the second
 * reduction warp that waits for the turn, the other reduction stamps from the reduction leader;
 * for the atomic schedule slots 10, 11 and 13 carry no wait) */
#define DASH_TRACE_SLOTS 21

/* dash_attn_bwd with options (opt may be NULL).  A supplied task table is
 * checked on the host before the launch: indices in range, runs on one KV tile
 * each, and (for an ordered schedule, unless trust_table is set) dQ orders
 * that can finish, as dash_check_table states; DASH_ERR_SCHEDULE otherwise.
 * With trust_table set, an inconsistent table makes the device waits run out,
 * which dash_sync_status() then reports as DASH_ERR_TIMEOUT. */
dash_status_t dash_attn_bwd_ex(const void *q, const void *k, const void *v, const void *o,
                               const void *dout, const float *lse,
                               void *dq, void *dk, void *dv,
                               int B, int H, int S, int D, int causal, float scale,
                               dash_schedule_t schedule, const dash_bwd_options_t *opt,
                               dash_stream_t stream);

/* End-to-end backward from HOST buffers: copies the six inputs to the device,
 * runs dash_attn_bwd on `stream`, copies dq/dk/dv back and synchronises the
 * stream.  All pointers are host pointers (pinned memory gives full copy
 * bandwidth).  The heads go in up to eight groups: each group's inputs are
 * copied on an internal stream while the previous group's backward runs, and
 * its gradients are copied back on another while the next one runs.  Heads
 * are independent and each head's dQ order depends on that head alone, so the
 * result equals a single dash_attn_bwd call over all heads, bit for bit.
 * Device buffers and the copy streams are cached per (device, stream). */
dash_status_t dash_attn_bwd_host(const void *q, const void *k, const void *v, const void *o,
                                 const void *dout, const float *lse,
                                 void *dq, void *dk, void *dv,
                                 int B, int H, int S, int D, int causal, float scale,
                                 dash_schedule_t schedule, dash_stream_t stream);

/* dash_attn_bwd without any device allocation.  For callers that must not
 * call cudaMalloc while they run: a framework whose caching allocator owns all
 * device memory, a runtime with a fixed memory budget reserved up front, or
 * code that cannot afford an allocation that may block or fail.  (The DASH
 * pages have no counterpart; this is a property of this library.)
 * Same arguments and results as dash_attn_bwd: the same kernels and the same
 * schedule table, so a deterministic schedule returns the same bits.  The
 * workspace lives in one fixed 32 MiB array of device memory inside the
 * library, present on every GPU that loads the library until the process
 * exits; problems whose workspace does not fit (roughly B*H*S*D above 7.8 M
 * elements) return DASH_ERR_UNSUPPORTED with the required size in
 * dash_last_error().  The first call on a device does a one-time set-up: it
 * looks up the array's device address, which stays valid until the process
 * exits or the device is reset (do not use this entry point after
 * cudaDeviceReset); make that first call before any stream capture.  Every
 * call clears what must start at zero, but all calls share the array: calls
 * whose GPU work overlaps (other streams or threads) race on it.  The call
 * copies the schedule table and the status word between host and device and
 * synchronises `stream` before it returns; it reports a device wait that ran
 * out as DASH_ERR_TIMEOUT. */
dash_status_t dash_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                    const void *dout, const float *lse,
                                    void *dq, void *dk, void *dv,
                                    int B, int H, int S, int D, int causal, float scale,
                                    dash_schedule_t schedule, dash_stream_t stream);

/* Number of tasks (q-tile x kv-tile pairs) of one problem: BH*n*n for a full
 * mask, BH*n*(n+1)/2 for a causal one; -1 if the schedule is invalid for the
 * mask.  Host only. */
long long dash_schedule_num_tasks(int BH, int n, int causal, dash_schedule_t schedule);

/* Host schedule generator (DASH overview, section 2.2: chains of C and R
 * stages list-scheduled on SMs).  Builds the chains of `schedule` for BH
 * heads of n blocks, simulates them on P CTAs with integer costs c (compute)
 * and r (reduce), and writes the per-CTA task table: tasks_out (4 int32 per
 * task, dash_schedule_num_tasks entries), cta_off_out (P+1 entries) and the
 * simulated makespan.  Returns DASH_ERR_SCHEDULE if the simulation
 * deadlocks (e.g. a shift schedule on fewer CTAs than its gang of chains).
 * Host only; no GPU needed. */
dash_status_t dash_build_schedule(int BH, int n, int causal, dash_schedule_t schedule, int P,
                                  int cost_c, int cost_r, int32_t *tasks_out,
                                  int32_t *cta_off_out, long long *makespan_out);

/* Checks a task table for an ordered schedule on the host (the pages' DAG:
 * a dQ tile's reductions run in rank order, DASH overview (zskr.cn),
 * section 2.2).  tasks holds 4 int32 per task in the encoding above and
 * cta_off num_ctas + 1 offsets.  Besides indices and runs, every dQ tile's
 * ranks must be 0, 1, ... without gap or repeat (with dq_chains = 2, in each
 * parity apart), and the table must finish when each CTA performs its adds in
 * table order, each waiting for its predecessor in the tile's order (no cycle
 * of waits).  DASH_OK, DASH_ERR_SCHEDULE with the reason in
 * dash_last_error(), or DASH_ERR_INVALID_ARG.  Host only. */
dash_status_t dash_check_table(int BH, int n, int causal, int dq_chains, const int32_t *tasks, const int32_t *cta_off,
                               int num_ctas);

/* Fill, an extension beyond the pages' schedules, for DASH_SCHED_SHIFT (full
 * mask) and DASH_SCHED_SYMMETRIC_SHIFT (causal).  Each of their chains waits
 * on a neighbour in its head's gang (n chains for shift, n/2 for symmetric
 * shift), so on max_ctas SMs that are not a multiple of the gang some SMs
 * idle or a split gang stalls.  This layout runs `schedule` for the first
 * *shift_heads_out heads on whole gangs (CTAs 0 .. P1-1) and the other heads
 * with a fill schedule on the CTAs that whole gangs leave over (CTAs P1 ..
 * *ctas_out-1): serial, or for a causal mask serial or descending_q
 * (*fill_schedule_out; -1 when no head is filled).  The split is the number
 * of heads, among whole waves of gangs and BH itself, and the fill schedule
 * whose larger simulated makespan of the two parts is smallest (costs cost_c,
 * cost_r; ties to more shift heads, then to serial).  Without leftover CTAs,
 * or when every head fits in one wave, it is plain `schedule` at
 * dash_choose_ctas' count.  tasks_out takes dash_schedule_num_tasks entries
 * and cta_off_out max_ctas + 1.  The ranks of every head are those of its own
 * schedule.  Host only. */
dash_status_t dash_build_shift_fill(int BH, int n, int causal, dash_schedule_t schedule, int max_ctas, int cost_c,
                                    int cost_r, int32_t *tasks_out, int32_t *cta_off_out, int *ctas_out,
                                    int *shift_heads_out, int *fill_schedule_out, long long *makespan_out);

/* Split gangs (dash_bwd_options_t.shift_split; an extension beyond the pages'
 * schedules), host only: dash_build_schedule for shift or symmetric shift with
 * each head's gang of chains run as `split` sub-gangs of consecutive slots.  A
 * dQ tile's ranks go in (sub-gang, visiting step) order; chains are dispatched
 * sub-gang by sub-gang (every head's sub-gang 0 first).  DASH_ERR_UNSUPPORTED
 * for other schedules or a split that does not divide the gang (n, or n/2 for
 * symmetric shift); DASH_ERR_SCHEDULE if the simulation deadlocks.  The table
 * sizes are those of dash_build_schedule. */
dash_status_t dash_build_split_schedule(int BH, int n, int causal, dash_schedule_t schedule, int split, int P,
                                        int cost_c, int cost_r, int32_t *tasks_out, int32_t *cta_off_out,
                                        long long *makespan_out);

/* dash_build_schedule with both extensions of the order: `split` as
 * dash_build_split_schedule (1 = whole gangs; shift and symmetric shift only
 * above 1) and `rank_order` as dash_bwd_options_t.rank_order (0 = the
 * schedule's own ranks, 1 = timed ranks).  Same sizes and errors; host only. */
dash_status_t dash_build_schedule_ex(int BH, int n, int causal, dash_schedule_t schedule, int split, int rank_order,
                                     int P, int cost_c, int cost_r, int32_t *tasks_out, int32_t *cta_off_out,
                                     long long *makespan_out);

/* The CTA count the backward uses with split gangs when num_ctas = 0: the
 * multiple of the sub-gang up to max_ctas with the smallest simulated makespan
 * (ties to fewer CTAs); -1 if the schedule or split is invalid.  Host only. */
int dash_choose_split_ctas(int BH, int n, int causal, dash_schedule_t schedule, int split, int max_ctas,
                           int cost_c, int cost_r);

/* The split that shift_split = -1 picks (an extension): for shift and
 * symmetric shift, every k that divides the gang (n, or n/2 for symmetric
 * shift): k = 1 on the dash_choose_ctas count, k > 1 on the better of the two
 * largest candidates of dash_choose_split_ctas (on num_ctas CTAs when
 * num_ctas > 0), and the k whose simulated makespan is smallest; ties go
 * first to a k whose sub-gang divides its CTA count (sub-gangs side by side,
 * none spread over time), then to the smaller k (1 = whole gangs).  Writes
 * the CTA count and makespan; returns k,
 * or -1 for another schedule, invalid arguments, or num_ctas > max_ctas.
 * Host only. */
int dash_choose_split(int BH, int n, int causal, dash_schedule_t schedule, int max_ctas, int num_ctas, int cost_c,
                      int cost_r, int *ctas_out, long long *makespan_out);

/* The CTA count the backward uses for a problem when num_ctas = 0: the
 * candidate (max_ctas, and the multiples of the schedule's gang size up to
 * it; only those multiples for shift, whose chains wait on their gang
 * neighbours so that a gang split over time stalls) whose simulated makespan
 * is smallest, ties to fewer CTAs.  Host only. */
int dash_choose_ctas(int BH, int n, int causal, dash_schedule_t schedule, int max_ctas,
                     int cost_c, int cost_r);

/* Runtime schedule choice (DASH overview (zskr.cn), section 7: choosing the
 * strategy from the run's own parameters; section 5.2 gives a static rule of
 * thumb instead).  Among the deterministic schedules valid for the mask
 * (serial, descending_q, and shift for a full mask or symmetric_shift for a
 * causal one with n even), returns the one whose simulated makespan is
 * smallest, each simulated at the CTA count dash_choose_ctas picks for it
 * (at most max_ctas) with task costs C = cost_c and R = cost_r; ties go to the
 * lower schedule number.  Writes that CTA count and makespan when the
 * pointers are not NULL.  Returns -1 (and sets dash_last_error) when BH, n,
 * max_ctas or a cost is below 1.  Host only. */
int dash_choose_schedule(int BH, int n, int causal, int max_ctas, int cost_c, int cost_r, int *ctas_out,
                         long long *makespan_out);

/* dash_choose_schedule with split gangs (an extension) among the candidates:
 * shift or symmetric shift enters with the split and CTA count that
 * dash_choose_split picks for it, so that its simulated makespan counts every
 * SM it can use.  Writes the split as well (1 for serial, descending_q and
 * whole gangs); a caller runs the result with dash_bwd_options_t.shift_split
 * set to it (or -1) and num_ctas to the CTA count.  Same errors.  Host only. */
int dash_choose_schedule_split(int BH, int n, int causal, int max_ctas, int cost_c, int cost_r, int *ctas_out,
                               int *split_out, long long *makespan_out);

/* The runtime choice over every deterministic layout this library runs (an
 * extension of dash_choose_schedule_split): each ordered schedule valid for
 * the mask in its own order, shift or symmetric shift with the split that
 * dash_choose_split picks, and each of those with timed ranks
 * (dash_bwd_options_t.rank_order = 1; whole gangs on every SM up to max_ctas,
 * split gangs on the split's CTA count), by simulated makespan with task costs
 * C = cost_c and R = cost_r.  Ties keep the lower schedule number, then the
 * schedule's own order before split gangs before timed ranks.  Writes the CTA
 * count, the split (1 = whole gangs) and the rank order (0 or 1) to pass as
 * num_ctas, shift_split and rank_order; returns the schedule, or -1 (with
 * dash_last_error) when BH, n, max_ctas or a cost is below 1.  Host only. */
int dash_choose_layout(int BH, int n, int causal, int max_ctas, int cost_c, int cost_r, int *ctas_out,
                       int *split_out, int *rank_order_out, long long *makespan_out);

/* Task costs for dash_choose_schedule from measured times (the pages' DAG
 * model has a compute cost c and a reduce cost r per task; DASH overview
 * (zskr.cn), section 2.2).  Given the measured backward (or main-kernel)
 * times of the atomic and serial schedules for this problem, atomic_ms and
 * serial_ms, writes c = 8 and the r in {1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48,
 * 64, 96, 128, 192, 256, 384, 512} whose simulated serial / atomic makespan
 * ratio, both on min(max_ctas, chains) CTAs, is nearest the measured ratio
 * (ties to the smaller r).  DASH_ERR_INVALID_ARG for sizes below 1 or times that are not
 * positive.  Host only. */
dash_status_t dash_fit_costs(int BH, int n, int causal, int max_ctas, double atomic_ms, double serial_ms,
                             int *cost_c_out, int *cost_r_out);

/* Die-aware placement, host half (an extension; DASH news (nachedeu.com) on
 * signalling through a remote L2 segment).  lat holds [n_sms][n_lines] L2 load
 * latencies in clocks, as the library's probe measures them (one row per SM,
 * one column per 128-byte line).  Splits the SMs in two groups by two-means
 * clustering of their rows (started from the split at the line with the
 * largest spread; at most 20 rounds) and gives each line the group whose mean
 * latency to it is lower (ties to group 0): group_out[n_sms], home_out[n_lines]
 * in {0, 1}.  DASH_ERR_SCHEDULE when no split into two groups exists;
 * DASH_ERR_INVALID_ARG for null pointers or n_sms < 2.  Host only. */
dash_status_t dash_cluster_latencies(const uint32_t *lat, int n_sms, int n_lines, int32_t *group_out,
                                     int32_t *home_out);

/* Die-aware placement, tables (host only).  For a task table on P slots
 * (tasks: 4 int32 per task; cta_off: P + 1), SM ids per group (sm0[n0],
 * sm1[n1]) and pool lines per home (line0[m0], line1[m1]; 128-byte lines):
 *  - slot_of_smid_out[max_smid + 1]: the slot each SM runs, -1 for none.  Each
 *    whole gang of `gang` consecutive slots goes to the group with the most
 *    SMs left that can hold it (ties to group 0); slots that no group can take
 *    as a whole gang go to the SMs left, group 0 first;
 *  - sem_idx_out[BH * n * chains]: the int offset, from the pool base, of the
 *    semaphore of (head, dQ tile, chain): a 32-byte sector of a line homed on
 *    the group that runs most of the tile's adds (ties to group 0), taken in
 *    order, four sectors per line.
 * DASH_ERR_SCHEDULE when the SMs or pool lines do not suffice. */
dash_status_t dash_place_schedule(const int32_t *tasks, const int32_t *cta_off, int P, int gang, int BH, int n,
                                  int chains, const int32_t *sm0, int n0, const int32_t *sm1, int n1,
                                  const int32_t *line0, int m0, const int32_t *line1, int m1, int max_smid,
                                  int32_t *slot_of_smid_out, int32_t *sem_idx_out);

/* Cluster hand-offs of a task table (host only; the tables behind
 * dash_bwd_options_t.cluster_size).  For a table on P CTAs launched in clusters
 * of C, writes one word per task to links_out: bit 31 set when the task, after
 * its release, also raises a counter of its successor in its dQ tile's order,
 * whose CTA runs in the same cluster with rank (word >> 20) & 0xF; bit 30 set
 * when the task takes its turn from the counter that its predecessor's CTA,
 * of rank (word >> 16) & 0xF in the cluster, raises.  (The library merges
 * these bits into its device copy of the task words, whose ranks then take the
 * low 16 bits.)  A (producer, consumer) pair of
 * CTAs is linked only when the consumer takes its turns from the producer in
 * the order of the producer's releases.  *n_links_out receives the number of
 * linked hand-offs.  DASH_ERR_INVALID_ARG for null pointers or C outside
 * [1, 16]. */
dash_status_t dash_cluster_links(const int32_t *tasks, const int32_t *cta_off, int P, int C, int BH, int n,
                                 int chains, int32_t *links_out, long long *n_links_out);

/* The die map of the calling thread's current device as the stream's
 * workspace measures it (the probe runs on `stream` the first time, which is
 * synchronised): group_of_smid_out[max_sm + 1] receives 0 or 1 for each SM id
 * (-1 for ids the device does not have), and n0 / n1 the group sizes.
 * DASH_ERR_UNSUPPORTED if no two groups were found. */
dash_status_t dash_die_map(dash_stream_t stream, int32_t *group_of_smid_out, int max_sm, int *n0, int *n1);

/* Synchronises `stream` and returns the device status of the calling
 * thread's current device workspace for that stream: DASH_OK, or
 * DASH_ERR_TIMEOUT if a bounded wait ran out since the last call (the word is
 * then cleared). */
dash_status_t dash_sync_status(dash_stream_t stream);

/* Frees the workspaces and cached schedule tables of the current device. */
void dash_release_workspace(void);

/* Description of the calling thread's last error ("" if none). */
const char *dash_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int dash_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DASH_H_ */
