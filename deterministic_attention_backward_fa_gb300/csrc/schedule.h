// Host schedule generator: DASH chains, reduction ranks and list scheduling
// on P CTAs.  Pure host C++; see schedule.cpp.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "kernels.h"  // kLinkRelease, kLinkTurn

namespace dash {

enum Mode { kAtomic = 0, kSerial = 1, kDescendingQ = 2, kShift = 3, kSymmetricShift = 4 };

constexpr int32_t kTaskFirst = 1 << 28;
constexpr int32_t kTaskLast = 1 << 29;
constexpr int32_t kRankMask = (1 << 24) - 1;

struct Schedule {
  std::vector<int32_t> tasks;    // 4 per task: bh, kv, q, rank|flags
  std::vector<int32_t> cta_off;  // P + 1
  long long makespan = 0;
  int P = 0;
};

// Empty string when (mode, n, causal) is a valid combination, else the reason.
std::string check_mode(int mode, int n, bool causal);

// Number of chains one head contributes (the gang of a cyclic schedule).
int chains_per_head(int mode, int n);

long long num_tasks(int BH, int n, bool causal);

// Builds chains for BH heads, simulates them on P CTAs with costs (c, r) and
// fills `out`.  Returns an empty string on success, else the error.
// split (shift and symmetric shift; 1 = none): each head's gang of chains
// runs as `split` sub-gangs of consecutive chains.  A dQ tile's ranks go in
// (sub-gang, step) order, and chains are dispatched sub-gang by sub-gang:
// every head's sub-gang 0 first, then every head's sub-gang 1, and so on.  A
// sub-gang keeps shift's property that no two of its chains reach one tile at
// one step, and CTA counts that are multiples of the sub-gang become usable.
// timed (the ordered schedules): each dQ tile's ranks follow the order in
// which the simulated schedule reaches the tile (compute-stage end in a run
// without reduction order; ties by the chain's dispatch position, then step)
// instead of the schedule's own order.  Where the schedule runs as its order
// assumes (whole shift gangs side by side) the two orders agree.
std::string build_schedule(int BH, int n, bool causal, int mode, int P, int c, int r,
                           Schedule *out, int split = 1, bool timed = false);
// "" when `split` is valid for the schedule and n, else why not.
std::string check_split(int mode, int n, int split);

// Candidate CTA counts (P_max and multiples of the gang size up to it, capped
// at the number of chains; only the multiples for shift), best simulated
// makespan, ties to fewer CTAs.
int choose_ctas(int BH, int n, bool causal, int mode, int P_max, int c, int r, int split = 1);

// Split gangs chosen by simulation (shift and symmetric shift): every split k
// that divides the gang, k = 1 on choose_ctas' CTA count and k > 1 on the
// better of its two largest candidate counts (or on fixed_P CTAs when
// fixed_P > 0; for shift only
// where fixed_P is a multiple of the sub-gang), and the k of the smallest
// simulated makespan; ties go first to a k whose sub-gang divides its CTA
// count, then to the smaller k (so 1, whole gangs, wins a plain tie).
// Fills the CTA count and the makespan; returns k, or -1 on invalid arguments
// or when no k runs.
int choose_split(int BH, int n, bool causal, int mode, int P_max, int c, int r, int fixed_P, int *P_out,
                 long long *makespan_out);

// Fill (an extension beyond the pages' schedules) for shift (full mask) and
// symmetric shift (causal): whole gangs of CTAs, as many as fit in P_max, run
// `mode` for the first `shift_heads` heads; the CTAs that whole gangs leave
// idle run the other heads with a fill schedule (serial; for a causal mask
// serial or descending_q), each head keeping its own schedule's dQ order.
// The split is the number of heads, among whole waves of gangs and BH itself,
// and the fill schedule whose larger simulated makespan of the two parts is
// smallest (ties to more shift heads, then to serial).  When no CTA is left
// over, or every head fits in one wave, it is plain `mode` on choose_ctas CTAs
// (shift_heads = BH, fill_mode = -1).
std::string build_fill(int BH, int n, bool causal, int mode, int P_max, int c, int r, Schedule *out,
                       int *shift_heads, int *fill_mode);

// Checks that a task table (4 int32 per task, cta_off of P + 1 entries) runs
// to completion when each CTA performs its tasks' dQ adds in table order and a
// task's add waits for its predecessor in the tile's order: with `chains`
// chains (1 or 2), the task of rank k is position k / chains of chain
// k % chains.  Every tile's positions in each chain must be 0, 1, ... with no
// gap or repeat, and an event-driven run of the table must reach every CTA's
// end (no cycle of waits).  Bounds and run structure are checked elsewhere.
// Empty string when the table is sound, else the reason.
std::string check_table_order(const int32_t *tasks, const int32_t *cta_off, int P, int BH, int n, int chains);

// Cluster links of an ordered table (an extension of the semaphore hand-off):
// with the persistent CTAs launched in thread-block clusters of C (<= 16), a
// rank whose successor in its dQ tile's order runs in the same cluster can
// also signal it through that CTA's shared memory.  links_out[t] holds the
// bits to merge into task t's word (kernels.h):
//   kLinkRelease | (rank of the successor's CTA in the cluster << kLinkToShift):
//     task t raises the successor's counter for t's CTA after its release;
//   kLinkTurn | (rank of the predecessor's CTA in the cluster << kLinkFromShift):
//     task t takes its turn from that counter instead of the global semaphore.
// A pair of CTAs (producer a, consumer b) is linked only if b takes its turns
// from a in the order in which a releases them, so that one counter per
// producer suffices; otherwise both keep the global semaphore.  Returns the
// number of linked hand-offs.
long long cluster_links(const int32_t *tasks, const int32_t *cta_off, int P, int C, int BH, int n, int chains,
                        int32_t *links_out);

// Task costs fitted to measured times: c is fixed at kFitCostC and r is the
// value of kFitCostR whose simulated serial / atomic makespan ratio (both on
// min(P_max, chains) CTAs) is nearest the measured serial_ms / atomic_ms
// (ties to the smaller r).  Empty string on success.
constexpr int kFitCostC = 8;
constexpr int kFitCostR[] = {1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64, 96, 128, 192, 256, 384, 512};
std::string fit_costs(int BH, int n, bool causal, int P_max, double atomic_ms, double serial_ms, int *c, int *r);

// The deterministic schedule valid for the mask whose simulated makespan,
// each at its own choose_ctas CTA count, is smallest (ties to the lower mode
// number); fills its CTA count and makespan.  With allow_split, shift and
// symmetric shift enter with the split that choose_split picks (and its CTA
// count), and split_out receives it (1 for the other schedules).  -1 on
// invalid arguments.
int choose_schedule(int BH, int n, bool causal, int P_max, int c, int r, int *P_out, long long *makespan_out,
                    bool allow_split = false, int *split_out = nullptr);

// The deterministic layout with the smallest simulated makespan among every
// ordered schedule valid for the mask in its own order (choose_ctas CTAs),
// shift / symmetric shift with the split choose_split picks, and each of
// those with timed ranks (whole gangs on every SM, split gangs on the split's
// CTA count).  Ties keep the lower schedule number, then the own order before
// split gangs before timed ranks.  Fills the CTA count, split (1 = whole
// gangs) and timed flag; -1 on invalid arguments.
int choose_layout(int BH, int n, bool causal, int P_max, int c, int r, int *P_out, int *split_out, int *timed_out,
                  long long *makespan_out);

}  // namespace dash
