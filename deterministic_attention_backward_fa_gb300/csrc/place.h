// Die-aware placement (an extension for the shift schedules): which SMs share
// a die, which L2 lines are homed on which die, and the tables that put each
// gang of chains on one die with its dQ semaphores homed there.  Host C++;
// the latency probe that feeds it is in place.cu.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

namespace dash {

// Splits SMs into two groups by their L2 load-latency vectors and assigns each
// probed line the group that reaches it faster.  lat is [n_sms][n_lines]
// clocks.  group_out[n_sms] in {0, 1}; home_out[n_lines] in {0, 1}.  Two-means
// clustering from the split at the line with the largest spread, at most 20
// rounds; ties go to group 0.  Returns "" or the reason no split was found.
std::string cluster_latencies(const uint32_t *lat, int n_sms, int n_lines, int *group_out, int *home_out);

struct Placement {
  std::vector<int> slot_of_smid;  // indexed by SM id; -1 = the SM runs no slot
  std::vector<int> sem_idx;       // [BH][n][chains] int offsets into the semaphore pool
};

// Tables for a schedule on P slots (tasks: 4 int32 per task, cta_off: P + 1):
//  - slots go to SMs gang by gang: each whole gang of `gang` consecutive slots
//    goes to the group with the most SMs left that can hold it, a remainder
//    (or a gang that fits nowhere whole) to the SMs left, group 0 first;
//  - the semaphore of each (head, dQ tile, chain) goes to a free 32-byte sector
//    of a pool line homed on the group that runs most of the tile's adds.
// smids[g] lists the SM ids of group g; lines[g] the pool lines (128 bytes)
// homed on g.  Returns "" or the reason (too few SMs or pool lines).
std::string build_placement(const int32_t *tasks, const int32_t *cta_off, int P, int gang, int BH, int n, int chains,
                            const std::vector<int> (&smids)[2], const std::vector<int> (&lines)[2], int max_smid,
                            Placement *out);

}  // namespace dash
