// Host schedule generator for the deterministic attention backward.
//
// The DASH model (DASH overview (zskr.cn), section 2.2; Sintesi Tecnica DASH
// (gist.science/it), section 2.1): every piece of work on one KV tile runs back
// to back on one SM, forming a chain of tasks; a task is a compute stage C
// (the KV tile against one Q tile) followed by a reduction stage R (adding the
// task's dQ partial into the dQ tile).  Determinism fixes, per dQ tile, the
// order of its R stages.  This file builds the chains of each schedule, the
// rank of every task in its dQ tile's order, and places chains on the
// persistent CTAs by discrete-event list scheduling:
//   * chains are taken in (head, slot) order; at time 0 CTAs 0..P-1 take the
//     first P chains, afterwards a CTA that falls idle at time T takes the next
//     chain at T, lowest CTA id first among those idle at the same T;
//   * a task's C lasts c; its R starts once C has ended and (ordered
//     schedules) once the R of its predecessor in the dQ tile's order has
//     ended, and lasts r; the CTA stays busy while it waits.
// The resulting table is also a proof of deadlock freedom: every wait edge of
// the device execution points to a task that the simulation finished earlier,
// so the wait graph is acyclic when every CTA is resident.
//
// Schedules (DASH overview, sections 3.1-3.3):
//   serial / atomic:  KV j visits Q tiles ascending (j..n-1 when causal)
//   descending_q:     KV j visits Q tiles n-1 down to 0 (down to j when causal)
//   shift (full):     KV j visits Q tiles (j + t) mod n, t = 0..n-1
//   symmetric shift (causal, n even): slot p < n/2 runs KV p over Q tiles
//       n/2 + ((p + t) mod n/2) for t < n/2 (dense lower-left rectangle), then
//       KV p over Q tiles p..n/2-1, then KV n-1-p over Q tiles n-1 down to
//       n-1-p (the folded triangle)
// Serial, descending and atomic rank a dQ tile's partials by KV index; the two
// shift schedules rank them by the step at which their chain reaches the tile
// (conflict-free: no two chains of a head reach one tile at the same step).
#include "schedule.h"

#include <algorithm>
#include <atomic>
#include <map>
#include <string>
#include <cmath>
#include <functional>
#include <queue>
#include <thread>
#include <tuple>
#include <utility>

namespace dash {

namespace {

struct HeadPlan {
  // chains of one head, flattened: chain c holds tasks [off[c], off[c+1])
  std::vector<int> off;
  std::vector<int> kv, q, rank;
};

HeadPlan head_plan(int mode, int n, bool causal, int split = 1) {
  HeadPlan hp;
  hp.off.push_back(0);
  auto push = [&](int kv, int q) {
    hp.kv.push_back(kv);
    hp.q.push_back(q);
  };
  if (mode == kAtomic || mode == kSerial) {
    for (int j = 0; j < n; ++j) {
      for (int q = causal ? j : 0; q < n; ++q) push(j, q);
      hp.off.push_back((int)hp.kv.size());
    }
  } else if (mode == kDescendingQ) {
    for (int j = 0; j < n; ++j) {
      for (int q = n - 1; q >= (causal ? j : 0); --q) push(j, q);
      hp.off.push_back((int)hp.kv.size());
    }
  } else if (mode == kShift) {
    for (int j = 0; j < n; ++j) {
      for (int t = 0; t < n; ++t) push(j, (j + t) % n);
      hp.off.push_back((int)hp.kv.size());
    }
  } else {  // symmetric shift
    const int h = n / 2;
    for (int p = 0; p < h; ++p) {
      for (int t = 0; t < h; ++t) push(p, h + (p + t) % h);
      for (int q = p; q < h; ++q) push(p, q);
      for (int i = 0; i <= p; ++i) push(n - 1 - p, n - 1 - i);
      hp.off.push_back((int)hp.kv.size());
    }
  }
  const int nt = (int)hp.kv.size();
  hp.rank.assign(nt, 0);
  if (mode == kShift || mode == kSymmetricShift) {
    // rank = position of the visiting step among all visits of the tile; with
    // split gangs, of (sub-gang, step): sub-gang s takes the tile's ranks
    // after sub-gang s - 1 has added all of its partials
    std::vector<std::vector<std::pair<long long, int>>> visits(n);  // (order key, task)
    const int nch = (int)hp.off.size() - 1;
    const int g = nch / split;
    for (int c = 0; c < nch; ++c)
      for (int t = hp.off[c]; t < hp.off[c + 1]; ++t)
        visits[hp.q[t]].push_back({(long long)(c / g) * (n + 1) + (t - hp.off[c]), t});
    for (int q = 0; q < n; ++q) {
      auto &v = visits[q];
      std::sort(v.begin(), v.end());
      for (size_t i = 0; i < v.size(); ++i) hp.rank[v[i].second] = (int)i;
    }
  } else {
    for (int t = 0; t < nt; ++t) hp.rank[t] = hp.kv[t];
  }
  return hp;
}

// Per-head predecessor of each task in its dQ tile's order (-1 for rank 0).
std::vector<int> head_pred(const HeadPlan &hp, int n) {
  const int nt = (int)hp.kv.size();
  std::vector<std::vector<int>> by_rank(n);
  for (int t = 0; t < nt; ++t) {
    auto &v = by_rank[hp.q[t]];
    if ((int)v.size() <= hp.rank[t]) v.resize(hp.rank[t] + 1, -1);
    v[hp.rank[t]] = t;
  }
  std::vector<int> pred(nt, -1);
  for (int q = 0; q < n; ++q)
    for (size_t r = 1; r < by_rank[q].size(); ++r) pred[by_rank[q][r]] = by_rank[q][r - 1];
  return pred;
}

struct SimResult {
  bool deadlock = false;
  long long makespan = 0;
  std::vector<std::vector<int>> chains_of_cta;
};

// order (optional): the global chain id (head * chains per head + chain) of
// each dispatch, in dispatch order; identity when null.  gpred (optional):
// each task's predecessor as a global task id (head * tasks per head + task),
// in place of the per-head hpred.  c_end (optional, sized BH * tasks per
// head): receives the time each task's compute stage ends.
SimResult simulate(const HeadPlan &hp, const std::vector<int> &hpred, int BH, int P, int c, int r,
                   bool ordered, const std::vector<long long> *order = nullptr,
                   const std::vector<long long> *gpred = nullptr, std::vector<long long> *c_end = nullptr) {
  const int cph = (int)hp.off.size() - 1;   // chains per head
  const int tph = (int)hp.kv.size();        // tasks per head
  const long long nch = (long long)BH * cph;
  SimResult res;
  res.chains_of_cta.assign(P, {});
  // task id = head * tph + local task
  std::vector<char> r_done((size_t)BH * tph, 0);
  std::vector<int> waiter((size_t)BH * tph, -1);
  std::vector<long long> cta_chain(P, -1);
  std::vector<int> cta_step(P, 0);
  std::vector<char> cta_phase(P, 0);  // 'C', 'R', 'W'
  using Ev = std::pair<long long, int>;
  std::priority_queue<Ev, std::vector<Ev>, std::greater<Ev>> heap;
  long long next = 0;
  long long waiting = 0;

  auto task_id = [&](long long chain, int step) -> long long {
    const long long head = chain / cph;
    const int local_chain = (int)(chain % cph);
    return head * tph + hp.off[local_chain] + step;
  };
  auto chain_len = [&](long long chain) {
    const int lc = (int)(chain % cph);
    return hp.off[lc + 1] - hp.off[lc];
  };
  auto dispatch = [&](int s, long long T) {
    const long long ch = order ? (*order)[(size_t)next] : next;
    ++next;
    cta_chain[s] = ch;
    cta_step[s] = 0;
    cta_phase[s] = 'C';
    res.chains_of_cta[s].push_back((int)ch);
    heap.push({T + c, s});
  };

  for (int s = 0; s < P && next < nch; ++s) dispatch(s, 0);
  std::vector<int> batch, freed;
  while (!heap.empty()) {
    const long long T = heap.top().first;
    batch.clear();
    freed.clear();
    while (!heap.empty() && heap.top().first == T) {
      batch.push_back(heap.top().second);
      heap.pop();
    }
    std::sort(batch.begin(), batch.end());
    for (int s : batch) {
      const long long ch = cta_chain[s];
      const int st = cta_step[s];
      const long long tid = task_id(ch, st);
      if (cta_phase[s] == 'C') {
        if (c_end) (*c_end)[(size_t)tid] = T;
        long long p = -1;
        if (ordered && gpred) {
          p = (*gpred)[(size_t)tid];
        } else if (ordered) {
          const int lp = hpred[(size_t)(tid % tph)];
          if (lp >= 0) p = (tid / tph) * tph + lp;
        }
        if (p < 0 || r_done[(size_t)p]) {
          cta_phase[s] = 'R';
          heap.push({T + r, s});
        } else {
          cta_phase[s] = 'W';
          waiter[(size_t)p] = s;
          ++waiting;
        }
      } else {  // R finished
        r_done[(size_t)tid] = 1;
        const int w = waiter[(size_t)tid];
        if (w >= 0) {
          waiter[(size_t)tid] = -1;
          --waiting;
          cta_phase[w] = 'R';
          heap.push({T + r, w});
        }
        if (st + 1 < chain_len(ch)) {
          cta_step[s] = st + 1;
          cta_phase[s] = 'C';
          heap.push({T + c, s});
        } else {
          res.makespan = std::max(res.makespan, T);
          cta_chain[s] = -1;
          cta_phase[s] = 0;
          freed.push_back(s);
        }
      }
    }
    std::sort(freed.begin(), freed.end());
    for (int s : freed)
      if (next < nch) dispatch(s, T);
  }
  res.deadlock = (next < nch) || (waiting > 0);
  return res;
}

// Dispatch order of split gangs: every head's sub-gang 0, then every head's
// sub-gang 1, and so on, each sub-gang's chains together.
std::vector<long long> split_order(int BH, int cph, int split) {
  std::vector<long long> order;
  order.reserve((size_t)BH * cph);
  const int g = cph / split;
  for (int s = 0; s < split; ++s)
    for (int h = 0; h < BH; ++h)
      for (int k = 0; k < g; ++k) order.push_back((long long)h * cph + s * g + k);
  return order;
}

// Timed ranks: each dQ tile's order is the order in which the simulated
// schedule reaches it.  A run without reduction order gives every task's
// compute end; the tasks of one (head, q) tile are ranked by that time, ties
// by the dispatch position of their chain, then by step.  Fills the global
// rank and predecessor of every task (head * tasks per head + task).
void timed_ranks(const HeadPlan &hp, const std::vector<int> &hpred, int BH, int n, int P, int c, int r,
                 const std::vector<long long> *order, std::vector<int> *rank, std::vector<long long> *gpred) {
  const int cph = (int)hp.off.size() - 1, tph = (int)hp.kv.size();
  const size_t nt = (size_t)BH * tph;
  std::vector<long long> c_end(nt, 0);
  simulate(hp, hpred, BH, P, c, r, false, order, nullptr, &c_end);
  std::vector<long long> pos((size_t)BH * cph);
  for (long long i = 0; i < (long long)pos.size(); ++i) pos[(size_t)(order ? (*order)[(size_t)i] : i)] = i;
  std::vector<int> chain_of(tph), step_of(tph);
  for (int ch = 0; ch < cph; ++ch)
    for (int t = hp.off[ch]; t < hp.off[ch + 1]; ++t) {
      chain_of[t] = ch;
      step_of[t] = t - hp.off[ch];
    }
  rank->assign(nt, 0);
  gpred->assign(nt, -1);
  std::vector<std::vector<int>> by_q(n);
  for (int t = 0; t < tph; ++t) by_q[hp.q[t]].push_back(t);
  std::vector<std::tuple<long long, long long, int, long long>> keys;
  for (int h = 0; h < BH; ++h) {
    const long long base = (long long)h * tph;
    for (int q = 0; q < n; ++q) {
      keys.clear();
      for (int t : by_q[q])
        keys.emplace_back(c_end[(size_t)(base + t)], pos[(size_t)h * cph + chain_of[t]], step_of[t], base + t);
      std::sort(keys.begin(), keys.end());
      for (size_t i = 0; i < keys.size(); ++i) {
        const long long tid = std::get<3>(keys[i]);
        (*rank)[(size_t)tid] = (int)i;
        if (i > 0) (*gpred)[(size_t)tid] = std::get<3>(keys[i - 1]);
      }
    }
  }
}

}  // namespace

std::string check_split(int mode, int n, int split) {
  if (split <= 1) return "";
  if (mode != kShift && mode != kSymmetricShift) return "split gangs apply to shift and symmetric shift only";
  const int cph = chains_per_head(mode, n);
  if (cph % split) return "the split must divide the chains of a head's gang";
  return "";
}

std::string check_mode(int mode, int n, bool causal) {
  if (mode < kAtomic || mode > kSymmetricShift) return "unknown schedule";
  if (n < 1) return "n must be >= 1";
  if (mode == kShift && causal) return "shift scheduling is defined for full masks only";
  if (mode == kSymmetricShift && !causal) return "symmetric shift is defined for causal masks only";
  if (mode == kSymmetricShift && (n % 2)) return "symmetric shift needs an even number of blocks";
  return "";
}

int chains_per_head(int mode, int n) { return mode == kSymmetricShift ? n / 2 : n; }

long long num_tasks(int BH, int n, bool causal) {
  const long long per = causal ? (long long)n * (n + 1) / 2 : (long long)n * n;
  return per * BH;
}

std::string build_schedule(int BH, int n, bool causal, int mode, int P, int c, int r,
                           Schedule *out, int split, bool timed) {
  std::string e = check_mode(mode, n, causal);
  if (!e.empty()) return e;
  if (split < 1) split = 1;
  if (!(e = check_split(mode, n, split)).empty()) return e;
  if (BH < 1 || P < 1 || c < 1 || r < 1) return "BH, P and the costs must be >= 1";
  const HeadPlan hp = head_plan(mode, n, causal, split);
  const std::vector<int> hpred = head_pred(hp, n);
  const std::vector<long long> order = split > 1 ? split_order(BH, (int)hp.off.size() - 1, split)
                                                 : std::vector<long long>();
  const std::vector<long long> *ord = split > 1 ? &order : nullptr;
  std::vector<int> grank;
  std::vector<long long> gpred;
  if (timed && mode != kAtomic) timed_ranks(hp, hpred, BH, n, P, c, r, ord, &grank, &gpred);
  SimResult sim = simulate(hp, hpred, BH, P, c, r, mode != kAtomic, ord, grank.empty() ? nullptr : &gpred);
  if (sim.deadlock) return "schedule simulation deadlocked (too few CTAs for the chain gang?)";
  const int cph = (int)hp.off.size() - 1, tph = (int)hp.kv.size();
  out->tasks.clear();
  out->tasks.reserve((size_t)num_tasks(BH, n, causal) * 4);
  out->cta_off.assign(1, 0);
  for (int s = 0; s < P; ++s) {
    for (int ch : sim.chains_of_cta[s]) {
      const int bh = ch / cph, lc = ch % cph;
      const int a = hp.off[lc], b = hp.off[lc + 1];
      for (int t = a; t < b; ++t) {
        int32_t w = grank.empty() ? hp.rank[t] : grank[(size_t)bh * tph + t];
        if (t == a || hp.kv[t - 1] != hp.kv[t]) w |= kTaskFirst;
        if (t == b - 1 || hp.kv[t + 1] != hp.kv[t]) w |= kTaskLast;
        out->tasks.push_back(bh);
        out->tasks.push_back(hp.kv[t]);
        out->tasks.push_back(hp.q[t]);
        out->tasks.push_back(w);
      }
    }
    out->cta_off.push_back((int32_t)(out->tasks.size() / 4));
  }
  out->makespan = sim.makespan;
  out->P = P;
  return "";
}

namespace {

// choose_ctas with the winner's simulated makespan in *ms, among at most
// max_cand candidates; with fixed_P > 0 that CTA count is the only candidate
// (for shift, only if it is a multiple of the gang).
int best_ctas(int BH, int n, bool causal, int mode, int P_max, int c, int r, int split, int fixed_P, int max_cand,
              long long *ms) {
  if (split < 1) split = 1;
  if (!check_mode(mode, n, causal).empty() || !check_split(mode, n, split).empty() || BH < 1 || P_max < 1) return -1;
  const long long nch = (long long)BH * chains_per_head(mode, n);
  const int gang = chains_per_head(mode, n) / split;  // with split gangs, a sub-gang
  // Shift makes every chain of a head wait on its neighbour in the gang, so a
  // gang split over time stalls: it only takes whole gangs (the pages'
  // setting, one SM per chain of a gang).  Symmetric shift also gets the
  // full count to choose from: a split gang of it costs less than the idle
  // SMs of whole gangs, in the simulation and on the GPU.
  const bool cyclic = (mode == kShift);
  std::vector<int> cand;
  const int top = (int)std::min<long long>(P_max, nch);
  if (fixed_P > 0) {
    if (cyclic && fixed_P % gang) return -1;
    cand.push_back(fixed_P);
  } else {
    if (!cyclic) cand.push_back(top);
    for (int m = (top / gang) * gang; m >= gang && (int)cand.size() < max_cand; m -= gang)
      if (cyclic || m != top) cand.push_back(m);
  }
  const HeadPlan hp = head_plan(mode, n, causal, split);
  const std::vector<int> hpred = head_pred(hp, n);
  const std::vector<long long> order = split > 1 ? split_order(BH, (int)hp.off.size() - 1, split)
                                                 : std::vector<long long>();
  int best = -1;
  long long best_ms = 0;
  for (int P : cand) {
    SimResult sim = simulate(hp, hpred, BH, P, c, r, mode != kAtomic, split > 1 ? &order : nullptr);
    if (sim.deadlock) continue;
    if (best < 0 || sim.makespan < best_ms || (sim.makespan == best_ms && P < best)) {
      best = P;
      best_ms = sim.makespan;
    }
  }
  if (ms) *ms = best_ms;
  return best;
}

}  // namespace

int choose_ctas(int BH, int n, bool causal, int mode, int P_max, int c, int r, int split) {
  return best_ctas(BH, n, causal, mode, P_max, c, r, split, 0, 16, nullptr);
}

int choose_split(int BH, int n, bool causal, int mode, int P_max, int c, int r, int fixed_P, int *P_out,
                 long long *makespan_out) {
  if (mode != kShift && mode != kSymmetricShift) return -1;
  if (!check_mode(mode, n, causal).empty() || BH < 1 || P_max < 1 || c < 1 || r < 1) return -1;
  const int gang = chains_per_head(mode, n);
  std::vector<int> ks;
  for (int k = 1; k <= gang; ++k)
    if (gang % k == 0) ks.push_back(k);
  // Each k is simulated on its own host thread (the simulations share nothing).
  // Whole gangs (k = 1) take choose_ctas' own candidates; a split gang the two
  // largest only: its closed form has no waits, so fewer CTAs only lose SMs.
  std::vector<int> Ps(ks.size(), -1);
  std::vector<long long> spans(ks.size(), 0);
  auto run = [&](size_t i) {
    Ps[i] = best_ctas(BH, n, causal, mode, P_max, c, r, ks[i], fixed_P, ks[i] == 1 ? 16 : 2, &spans[i]);
  };
  const size_t workers = std::min<size_t>(ks.size(), std::max(1u, std::thread::hardware_concurrency()));
  std::vector<std::thread> pool;
  std::atomic<size_t> next{0};
  for (size_t w = 1; w < workers; ++w)
    pool.emplace_back([&] {
      for (size_t i; (i = next.fetch_add(1)) < ks.size();) run(i);
    });
  for (size_t i; (i = next.fetch_add(1)) < ks.size();) run(i);
  for (auto &th : pool) th.join();
  int best_k = -1, best_P = 0;
  bool best_whole = false;
  long long best_ms = 0;
  for (size_t i = 0; i < ks.size(); ++i) {
    const int k = ks[i], P = Ps[i];
    const long long ms = spans[i];
    if (P < 1) continue;
    // On a tie, sub-gangs that fill the CTAs side by side win: a sub-gang
    // spread over time waits on its neighbours' hops, which the task costs
    // do not price.
    const bool whole = P % (gang / k) == 0;
    if (best_k < 0 || ms < best_ms || (ms == best_ms && whole && !best_whole)) {
      best_k = k;
      best_P = P;
      best_ms = ms;
      best_whole = whole;
    }
  }
  if (best_k > 0) {
    if (P_out) *P_out = best_P;
    if (makespan_out) *makespan_out = best_ms;
  }
  return best_k;
}

std::string build_fill(int BH, int n, bool causal, int mode, int P_max, int c, int r, Schedule *out,
                       int *shift_heads, int *fill_mode) {
  if (mode != kShift && mode != kSymmetricShift) return "fill applies to shift and symmetric shift only";
  std::string e = check_mode(mode, n, causal);
  if (!e.empty()) return e;
  if (BH < 1 || P_max < 1 || c < 1 || r < 1) return "BH, P and the costs must be >= 1";
  const int gang = chains_per_head(mode, n);
  const int per_wave = P_max / gang;  // heads whose gangs fit side by side
  const int G = per_wave * gang, F = P_max - G;
  if (fill_mode) *fill_mode = -1;
  if (per_wave == 0 || F == 0 || BH <= per_wave) {
    const int P = choose_ctas(BH, n, causal, mode, P_max, c, r);
    if (P < 1) return "no CTA count runs this schedule without deadlock";
    if (shift_heads) *shift_heads = BH;
    return build_schedule(BH, n, causal, mode, P, c, r, out);
  }
  const HeadPlan sh_plan = head_plan(mode, n, causal);
  const std::vector<int> sh_pred = head_pred(sh_plan, n);
  std::vector<int> fill_modes = {kSerial};
  if (causal) fill_modes.push_back(kDescendingQ);
  std::vector<HeadPlan> f_plan;
  std::vector<std::vector<int>> f_pred;
  for (int m : fill_modes) {
    f_plan.push_back(head_plan(m, n, causal));
    f_pred.push_back(head_pred(f_plan.back(), n));
  }
  int best_hs = -1, best_P1 = 0, best_P2 = 0, best_fm = -1;
  long long best_ms = 0;
  const int waves = (BH + per_wave - 1) / per_wave;
  for (int k = waves; k >= 1; --k) {  // more shift heads first, so that ties keep them
    const int hs = std::min(BH, k * per_wave), rest = BH - hs;
    const int P1 = (int)std::min<long long>(G, (long long)hs * gang);
    const SimResult s1 = simulate(sh_plan, sh_pred, hs, P1, c, r, true);
    if (s1.deadlock) continue;
    for (size_t f = 0; f < fill_modes.size(); ++f) {
      long long ms = s1.makespan;
      int P2 = 0;
      if (rest > 0) {
        P2 = (int)std::min<long long>(F, (long long)rest * n);
        const SimResult s2 = simulate(f_plan[f], f_pred[f], rest, P2, c, r, true);
        if (s2.deadlock) continue;
        ms = std::max(ms, s2.makespan);
      }
      if (best_hs < 0 || ms < best_ms) {
        best_hs = hs;
        best_P1 = P1;
        best_P2 = P2;
        best_fm = rest > 0 ? fill_modes[f] : -1;
        best_ms = ms;
      }
      if (rest == 0) break;
    }
  }
  if (best_hs < 0) return "schedule simulation deadlocked";
  Schedule a, b;
  e = build_schedule(best_hs, n, causal, mode, best_P1, c, r, &a);
  if (!e.empty()) return e;
  if (best_P2 > 0) {
    e = build_schedule(BH - best_hs, n, causal, best_fm, best_P2, c, r, &b);
    if (!e.empty()) return e;
    for (size_t i = 0; i < b.tasks.size(); i += 4) b.tasks[i] += best_hs;  // those heads follow the shift heads
  }
  out->tasks = std::move(a.tasks);
  out->tasks.insert(out->tasks.end(), b.tasks.begin(), b.tasks.end());
  out->cta_off = std::move(a.cta_off);
  const int32_t base = out->cta_off.back();
  for (size_t i = 1; i < b.cta_off.size(); ++i) out->cta_off.push_back(base + b.cta_off[i]);
  out->P = best_P1 + best_P2;
  out->makespan = best_ms;
  if (shift_heads) *shift_heads = best_hs;
  if (fill_mode) *fill_mode = best_fm;
  return "";
}

std::string check_table_order(const int32_t *tasks, const int32_t *cta_off, int P, int BH, int n, int chains) {
  if (chains != 1 && chains != 2) return "chains must be 1 or 2";
  const size_t keys = (size_t)BH * n * chains;  // (head, dQ tile, chain)
  // every chain of every tile holds positions 0 .. count-1 exactly once
  std::vector<int> count(keys, 0), seen_max(keys, -1);
  std::vector<std::vector<char>> seen(keys);
  const int total = cta_off[P];
  for (int t = 0; t < total; ++t) {
    const int32_t *k = tasks + 4 * (size_t)t;
    const int rank = k[3] & kRankMask;
    const size_t key = ((size_t)k[0] * n + k[2]) * chains + rank % chains;
    const int pos = rank / chains;
    std::vector<char> &sv = seen[key];
    if ((int)sv.size() <= pos) sv.resize(pos + 1, 0);
    if (sv[pos]) return "task " + std::to_string(t) + " repeats a rank of its dQ tile";
    sv[pos] = 1;
    ++count[key];
    seen_max[key] = std::max(seen_max[key], pos);
  }
  for (size_t key = 0; key < keys; ++key)
    if (seen_max[key] + 1 != count[key]) return "a dQ tile's ranks have a gap: a reduction would wait forever";
  // run the table: a CTA's adds go in table order, each waiting for the
  // previous position of its chain; a CTA blocked on a position is resumed
  // when that position's predecessor is done
  std::vector<int> next(keys, 0), ptr(cta_off, cta_off + P);
  std::vector<int> waiter(total, -1);  // CTA blocked on the task that holds (key, pos); indexed by that task
  std::vector<int> holder;             // task index of (key, pos), built below
  std::vector<size_t> base(keys + 1, 0);
  for (size_t key = 0; key < keys; ++key) base[key + 1] = base[key] + count[key];
  holder.assign(base[keys], -1);
  for (int t = 0; t < total; ++t) {
    const int32_t *k = tasks + 4 * (size_t)t;
    const int rank = k[3] & kRankMask;
    const size_t key = ((size_t)k[0] * n + k[2]) * chains + rank % chains;
    holder[base[key] + rank / chains] = t;
  }
  std::vector<int> ready;
  for (int s = 0; s < P; ++s) ready.push_back(s);
  int finished = 0;
  while (!ready.empty()) {
    const int s = ready.back();
    ready.pop_back();
    while (ptr[s] < cta_off[s + 1]) {
      const int t = ptr[s];
      const int32_t *k = tasks + 4 * (size_t)t;
      const int rank = k[3] & kRankMask;
      const size_t key = ((size_t)k[0] * n + k[2]) * chains + rank % chains;
      const int pos = rank / chains;
      if (pos != next[key]) {  // blocked until the predecessor's add is done
        waiter[holder[base[key] + pos - 1]] = s;
        break;
      }
      ++next[key];
      ++ptr[s];
      if (waiter[t] >= 0) {  // a CTA waited for this add
        ready.push_back(waiter[t]);
        waiter[t] = -1;
      }
    }
    if (ptr[s] == cta_off[s + 1]) ++finished;
  }
  if (finished != P) return "the table's dQ orders wait on one another in a cycle: it would never finish";
  return "";
}

long long cluster_links(const int32_t *tasks, const int32_t *cta_off, int P, int C, int BH, int n, int chains,
                        int32_t *links_out) {
  const int total = cta_off[P];
  std::fill(links_out, links_out + total, 0);
  if (C < 2 || C > kMaxClusterLinks || chains < 1) return 0;
  std::vector<int> cta_of(total);
  for (int c = 0; c < P; ++c)
    for (int t = cta_off[c]; t < cta_off[c + 1]; ++t) cta_of[t] = c;
  // tasks of each (head, tile, chain) in their order of adds
  const size_t keys = (size_t)BH * n * chains;
  std::vector<std::vector<std::pair<int, int>>> order(keys);  // (position, task)
  for (int t = 0; t < total; ++t) {
    const int32_t *k = tasks + 4 * (size_t)t;
    const int rank = k[3] & kRankMask;
    const size_t key = ((size_t)k[0] * n + k[2]) * chains + rank % chains;
    if (key < keys) order[key].push_back({rank / chains, t});
  }
  // candidate hand-offs inside a cluster, grouped by (producer CTA, consumer CTA)
  std::map<std::pair<int, int>, std::vector<std::pair<int, int>>> pairs;  // -> (consumer task, producer task)
  for (auto &v : order) {
    std::sort(v.begin(), v.end());
    for (size_t i = 0; i + 1 < v.size(); ++i) {
      const int tp = v[i].second, tc = v[i + 1].second;
      const int a = cta_of[tp], b = cta_of[tc];
      if (a / C == b / C) pairs[{a, b}].push_back({tc, tp});
    }
  }
  long long linked = 0;
  for (auto &kv : pairs) {
    auto &lst = kv.second;
    std::sort(lst.begin(), lst.end());  // the consumer takes its turns in task order
    bool monotone = true;               // ... and the producer must release them in that order
    for (size_t i = 1; i < lst.size() && monotone; ++i) monotone = lst[i].second > lst[i - 1].second;
    if (!monotone) continue;
    const int a = kv.first.first, b = kv.first.second;
    for (auto &l : lst) {
      links_out[l.second] |= kLinkRelease | ((b % C) << kLinkToShift);
      links_out[l.first] |= kLinkTurn | ((a % C) << kLinkFromShift);
      ++linked;
    }
  }
  return linked;
}

std::string fit_costs(int BH, int n, bool causal, int P_max, double atomic_ms, double serial_ms, int *c, int *r) {
  if (BH < 1 || n < 1 || P_max < 1) return "BH, n and P must be >= 1";
  if (!(atomic_ms > 0) || !(serial_ms > 0)) return "the measured times must be positive";
  const int P = (int)std::min<long long>(P_max, (long long)BH * n);
  const HeadPlan ha = head_plan(kAtomic, n, causal), hs = head_plan(kSerial, n, causal);
  const std::vector<int> pa = head_pred(ha, n), ps = head_pred(hs, n);
  const double want = serial_ms / atomic_ms;
  double best_err = -1;
  for (int rr : kFitCostR) {
    const SimResult a = simulate(ha, pa, BH, P, kFitCostC, rr, false);
    const SimResult s = simulate(hs, ps, BH, P, kFitCostC, rr, true);
    if (a.deadlock || s.deadlock || a.makespan <= 0) continue;
    const double err = std::fabs((double)s.makespan / (double)a.makespan - want);
    if (best_err < 0 || err < best_err) {
      best_err = err;
      *r = rr;
    }
  }
  if (best_err < 0) return "schedule simulation deadlocked";
  *c = kFitCostC;
  return "";
}

int choose_schedule(int BH, int n, bool causal, int P_max, int c, int r, int *P_out, long long *makespan_out,
                    bool allow_split, int *split_out) {
  if (BH < 1 || n < 1 || P_max < 1 || c < 1 || r < 1) return -1;
  int best = -1, best_P = 0, best_split = 1;
  long long best_ms = 0;
  for (int mode : {kSerial, kDescendingQ, kShift, kSymmetricShift}) {
    if (!check_mode(mode, n, causal).empty()) continue;
    int P = 0, split = 1;
    long long ms = 0;
    if (allow_split && (mode == kShift || mode == kSymmetricShift)) {
      split = choose_split(BH, n, causal, mode, P_max, c, r, 0, &P, &ms);
      if (split < 1) continue;
    } else {
      P = choose_ctas(BH, n, causal, mode, P_max, c, r);
      if (P < 1) continue;
      const HeadPlan hp = head_plan(mode, n, causal);
      const SimResult sim = simulate(hp, head_pred(hp, n), BH, P, c, r, true);
      if (sim.deadlock) continue;
      ms = sim.makespan;
    }
    if (best < 0 || ms < best_ms) {  // ties keep the lower schedule number
      best = mode;
      best_P = P;
      best_ms = ms;
      best_split = split;
    }
  }
  if (best >= 0) {
    if (P_out) *P_out = best_P;
    if (makespan_out) *makespan_out = best_ms;
    if (split_out) *split_out = best_split;
  }
  return best;
}

int choose_layout(int BH, int n, bool causal, int P_max, int c, int r, int *P_out, int *split_out, int *timed_out,
                  long long *makespan_out) {
  if (BH < 1 || n < 1 || P_max < 1 || c < 1 || r < 1) return -1;
  int best = -1, best_P = 0, best_split = 1, best_timed = 0;
  long long best_ms = 0;
  auto consider = [&](int mode, int P, int split, int timed, long long ms) {
    // ties keep the earlier candidate: the lower schedule number, then the
    // pages' order before split gangs before timed ranks
    if (best < 0 || ms < best_ms) {
      best = mode;
      best_P = P;
      best_split = split;
      best_timed = timed;
      best_ms = ms;
    }
  };
  for (int mode : {kSerial, kDescendingQ, kShift, kSymmetricShift}) {
    if (!check_mode(mode, n, causal).empty()) continue;
    const bool cyclic = mode == kShift || mode == kSymmetricShift;
    const int P = choose_ctas(BH, n, causal, mode, P_max, c, r);
    Schedule sch;
    if (P >= 1 && build_schedule(BH, n, causal, mode, P, c, r, &sch).empty()) consider(mode, P, 1, 0, sch.makespan);
    int Pk = 0;
    long long msk = 0;
    const int k = cyclic ? choose_split(BH, n, causal, mode, P_max, c, r, 0, &Pk, &msk) : 1;
    if (cyclic && k > 1) consider(mode, Pk, k, 0, msk);
    // timed ranks: whole gangs on every SM, and the chosen split's gangs
    const int Pall = (int)std::min<long long>(P_max, (long long)BH * chains_per_head(mode, n));
    if (build_schedule(BH, n, causal, mode, Pall, c, r, &sch, 1, true).empty())
      consider(mode, Pall, 1, 1, sch.makespan);
    if (cyclic && k > 1 && build_schedule(BH, n, causal, mode, Pk, c, r, &sch, k, true).empty())
      consider(mode, Pk, k, 1, sch.makespan);
  }
  if (best >= 0) {
    if (P_out) *P_out = best_P;
    if (split_out) *split_out = best_split;
    if (timed_out) *timed_out = best_timed;
    if (makespan_out) *makespan_out = best_ms;
  }
  return best;
}

}  // namespace dash
