// Die-aware placement (host half): clustering of the latency probe and the
// slot / semaphore tables.  GB300 has two dies whose L2 halves home the
// lines; the DASH pages place chains per SM and note that inter-SM signalling
// through a remote L2 segment costs 200 to more than 500 cycles (DASH news
// (nachedeu.com); DASH overview (zskr.cn), section 4.1).  This keeps each gang
// of a shift schedule on one die and homes its dQ tiles' semaphores there.
#include "place.h"

#include <algorithm>
#include <map>

namespace dash {

std::string cluster_latencies(const uint32_t *lat, int n_sms, int n_lines, int *group_out, int *home_out) {
  if (n_sms < 2 || n_lines < 1) return "need at least two SMs and one line";
  auto L = [&](int c, int a) { return (double)lat[(size_t)c * n_lines + a]; };
  std::vector<double> mu(n_lines, 0.0);
  for (int c = 0; c < n_sms; ++c)
    for (int a = 0; a < n_lines; ++a) mu[a] += L(c, a);
  for (double &m : mu) m /= n_sms;
  int a_star = 0;
  double v_star = -1.0;
  for (int a = 0; a < n_lines; ++a) {
    double v = 0.0;
    for (int c = 0; c < n_sms; ++c) v += (L(c, a) - mu[a]) * (L(c, a) - mu[a]);
    if (v > v_star) {
      v_star = v;
      a_star = a;
    }
  }
  std::vector<int> g(n_sms);
  for (int c = 0; c < n_sms; ++c) g[c] = L(c, a_star) > mu[a_star] ? 1 : 0;
  std::vector<double> cen[2] = {std::vector<double>(n_lines), std::vector<double>(n_lines)};
  for (int round = 0; round < 20; ++round) {
    int cnt[2] = {0, 0};
    for (int k = 0; k < 2; ++k) std::fill(cen[k].begin(), cen[k].end(), 0.0);
    for (int c = 0; c < n_sms; ++c) {
      ++cnt[g[c]];
      for (int a = 0; a < n_lines; ++a) cen[g[c]][a] += L(c, a);
    }
    if (cnt[0] == 0 || cnt[1] == 0) return "the latencies show a single group of SMs";
    for (int k = 0; k < 2; ++k)
      for (double &x : cen[k]) x /= cnt[k];
    int changed = 0;
    for (int c = 0; c < n_sms; ++c) {
      double d[2] = {0.0, 0.0};
      for (int k = 0; k < 2; ++k)
        for (int a = 0; a < n_lines; ++a) d[k] += (L(c, a) - cen[k][a]) * (L(c, a) - cen[k][a]);
      const int ng = d[1] < d[0] ? 1 : 0;
      changed += ng != g[c];
      g[c] = ng;
    }
    if (!changed) break;
  }
  int cnt[2] = {0, 0};
  for (int c = 0; c < n_sms; ++c) ++cnt[g[c]];
  if (cnt[0] == 0 || cnt[1] == 0) return "the latencies show a single group of SMs";
  for (int c = 0; c < n_sms; ++c) group_out[c] = g[c];
  for (int a = 0; a < n_lines; ++a) {
    double m[2] = {0.0, 0.0};
    for (int c = 0; c < n_sms; ++c) m[g[c]] += L(c, a);
    home_out[a] = (m[1] / cnt[1] < m[0] / cnt[0]) ? 1 : 0;
  }
  return "";
}

std::string build_placement(const int32_t *tasks, const int32_t *cta_off, int P, int gang, int BH, int n, int chains,
                            const std::vector<int> (&smids)[2], const std::vector<int> (&lines)[2], int max_smid,
                            Placement *out) {
  if (P < 1 || BH < 1 || n < 1 || chains < 1 || max_smid < 0) return "bad sizes";
  if ((long long)smids[0].size() + (long long)smids[1].size() < P) return "fewer SMs than slots";
  out->slot_of_smid.assign(max_smid + 1, -1);
  std::vector<int> group_of_slot(P, -1);
  size_t used[2] = {0, 0};
  auto take = [&](int grp, int slot) {
    const int sm = smids[grp][used[grp]++];
    out->slot_of_smid[sm] = slot;
    group_of_slot[slot] = grp;
  };
  int slot = 0;
  if (gang > 0) {
    for (; slot + gang <= P; slot += gang) {
      const size_t left0 = smids[0].size() - used[0], left1 = smids[1].size() - used[1];
      int grp = -1;
      if (left0 >= (size_t)gang && (left0 >= left1 || left1 < (size_t)gang)) grp = 0;
      else if (left1 >= (size_t)gang) grp = 1;
      if (grp < 0) break;  // no group holds this gang whole: the rest go where there is room
      for (int i = 0; i < gang; ++i) take(grp, slot + i);
    }
  }
  for (; slot < P; ++slot) {
    const int grp = used[0] < smids[0].size() ? 0 : 1;
    if (used[grp] >= smids[grp].size()) return "fewer SMs than slots";
    take(grp, slot);
  }
  // the group that runs most of each (head, tile, chain)'s adds
  const size_t keys = (size_t)BH * n * chains;
  std::vector<int> votes(keys * 2, 0);
  for (int c = 0; c < P; ++c)
    for (int t = cta_off[c]; t < cta_off[c + 1]; ++t) {
      const int32_t *k = tasks + 4 * (size_t)t;
      const int rank = k[3] & ((1 << 24) - 1);
      const size_t key = ((size_t)k[0] * n + k[2]) * chains + rank % chains;
      if (key < keys) ++votes[2 * key + group_of_slot[c]];
    }
  out->sem_idx.assign(keys, 0);
  size_t next[2] = {0, 0};  // next free 32-byte sector per group (four per 128-byte line)
  for (size_t key = 0; key < keys; ++key) {
    const int grp = votes[2 * key + 1] > votes[2 * key] ? 1 : 0;
    const size_t s = next[grp]++;
    if (s / 4 >= lines[grp].size()) return "too few pool lines for the semaphores";
    out->sem_idx[key] = (int)(lines[grp][s / 4] * 32 + (s % 4) * 8);  // int offsets: 32 per line, 8 per sector
  }
  return "";
}

}  // namespace dash
