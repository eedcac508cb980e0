// C ABI of the deterministic attention library (declared in include/dash.h).
//
// Host side of the backward (DASH overview (zskr.cn), section 2.1; Sintesi
// Tecnica DASH (gist.science/it), section 1): argument checks, the
// per-(device, stream) workspace, the cache of schedule tables built by the
// generator in schedule.cpp, TMA tensor maps, and the three launches
// (preprocess, persistent main kernel, dQ convert) on the caller's stream.
#include "dash.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <climits>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "kernels.h"
#include "place.h"
#include "schedule.h"

namespace {

thread_local std::string g_last_error;

dash_status_t fail(dash_status_t code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

dash_status_t cuda_fail(cudaError_t e, const char *what) {
  return fail(DASH_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr long long kDefaultSpinNs = 2000000000LL;  // 2 s bound on every device wait
// dash_attn_fwd at D = 128: the CTA-pair kernel (tcgen05 cta_group::2) or the single-CTA one.
constexpr bool kPairForwardByDefault = false;

// ------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D map over a contiguous bf16 [BH][S][D] tensor; boxes of 64 columns x box_rows rows.
dash_status_t make_map(CUtensorMap *m, const void *base, int BH, int S, int D, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(DASH_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DASH_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return DASH_OK;
}

// ------------------------------------------------------------ workspace
struct DevBuf {
  void *ptr = nullptr;
  size_t bytes = 0;
  ~DevBuf() {
    if (ptr) cudaFree(ptr);
  }
  cudaError_t reserve(size_t want) {
    if (want <= bytes) return cudaSuccess;
    if (ptr) cudaFree(ptr);
    ptr = nullptr;
    bytes = 0;
    cudaError_t e = cudaMalloc(&ptr, want);
    if (e == cudaSuccess) bytes = want;
    return e;
  }
  // Stream-ordered growth for buffers that only work on `s` uses: the old
  // block is freed and the new one allocated in the stream's order, so the
  // call does not synchronise the device.
  cudaError_t reserve_on(size_t want, cudaStream_t s) {
    if (want <= bytes) return cudaSuccess;
    if (ptr) cudaFreeAsync(ptr, s);
    ptr = nullptr;
    bytes = 0;
    cudaError_t e = cudaMallocAsync(&ptr, want, s);
    if (e == cudaSuccess) bytes = want;
    return e;
  }
};

// Copy streams and events of dash_attn_bwd_host, which pipelines the host
// copies of one group of heads with the backward of another.
constexpr int kHostChunks = 8;
struct CopyLanes {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t landed[kHostChunks] = {}, done[kHostChunks] = {};
  bool ready = false;
  cudaError_t init() {
    if (ready) return cudaSuccess;
    cudaError_t e = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking);
    for (int c = 0; c < kHostChunks && e == cudaSuccess; ++c) {
      e = cudaEventCreateWithFlags(&landed[c], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&done[c], cudaEventDisableTiming);
    }
    ready = (e == cudaSuccess);
    return e;
  }
  ~CopyLanes() {
    for (int c = 0; c < kHostChunks; ++c) {
      if (landed[c]) cudaEventDestroy(landed[c]);
      if (done[c]) cudaEventDestroy(done[c]);
    }
    if (in) cudaStreamDestroy(in);
    if (out) cudaStreamDestroy(out);
  }
};

// Die-aware placement (an extension): the SM groups of the two dies and a
// semaphore pool whose lines' homes are known, measured once per workspace.
constexpr int kPoolLines = 4096;  // 512 KiB: four 32-byte semaphore sectors per line
struct DieMap {
  bool tried = false, ready = false;
  std::string why;                  // why it is not ready
  DevBuf pool;                      // kPoolLines lines of 128 bytes
  std::vector<int> smids[2];        // SM ids per group, ascending
  std::vector<int> lines[2];        // pool lines homed on each group
  int max_smid = 0;
};
struct PlacementEntry {
  DevBuf slot_of_smid, sem_idx;
  int n_smid = 0;
};

struct Workspace {
  DevBuf accum, lse2, delta, sem, status;
  // device copies used by dash_attn_bwd_host
  DevBuf h_in[6], h_out[3];
  CopyLanes lanes;
  DieMap die;
  std::map<std::tuple<int, int, int, int, int, int, int, int, int, int>, std::unique_ptr<PlacementEntry>> placed;
};

struct ScheduleEntry {
  DevBuf tasks, cta_off;
  std::vector<int32_t> tasks_h, cta_off_h;  // host copies (die-aware placement and cluster links read them)
  int P = 0;
  long long makespan = 0;
  std::map<std::pair<int, int>, int> cluster_for;      // (D, tile) -> cluster size that fits
  std::map<int, std::unique_ptr<DevBuf>> linked_for;   // cluster size -> device task table with the links merged
};

std::mutex g_mu;
std::map<std::pair<int, void *>, std::unique_ptr<Workspace>> g_ws;
std::map<std::tuple<int, int, int, int, int, int, int, int, int, int>, std::unique_ptr<ScheduleEntry>> g_sched;
std::map<int, int> g_sms;

int sm_count(int dev) {
  auto it = g_sms.find(dev);
  if (it != g_sms.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 0;
  g_sms[dev] = n;
  return n;
}

Workspace *workspace(int dev, cudaStream_t s) {
  auto &w = g_ws[{dev, (void *)s}];
  if (!w) w.reset(new Workspace());
  return w.get();
}

cudaError_t ensure_status(Workspace *w) {
  if (w->status.ptr) return cudaSuccess;
  cudaError_t e = w->status.reserve(16);
  if (e == cudaSuccess) e = cudaMemset(w->status.ptr, 0, 16);
  return e;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dash_status_t check_common(int B, int H, int S, int D, float scale) {
  if (B < 0 || H < 0 || S < 0) return fail(DASH_ERR_INVALID_ARG, "B, H, S must be >= 0");
  if (D != 64 && D != 128) return fail(DASH_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", D);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(DASH_ERR_INVALID_ARG, "scale must be finite and > 0");
  if ((long long)B * H > (1LL << 30) || S > (1 << 30)) return fail(DASH_ERR_INVALID_ARG, "problem too large");
  return DASH_OK;
}

dash_status_t check_ptrs(std::initializer_list<const void *> ps) {
  for (const void *p : ps) {
    if (!p) return fail(DASH_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(p)) return fail(DASH_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  }
  return DASH_OK;
}

int auto_tile(int S) { return S <= 256 ? 64 : 128; }

// Checks that a caller-supplied table is in range and that every CTA's list is
// made of runs on one (head, KV tile) bracketed by the first/last flags.
dash_status_t validate_table(const int32_t *tasks, const int32_t *off, int P, int BH, int n, bool causal) {
  if (off[0] != 0) return fail(DASH_ERR_SCHEDULE, "cta_off[0] must be 0");
  for (int s = 0; s < P; ++s) {
    if (off[s + 1] < off[s]) return fail(DASH_ERR_SCHEDULE, "cta_off must be non-decreasing");
    bool in_run = false;
    int rbh = -1, rkv = -1;
    for (int t = off[s]; t < off[s + 1]; ++t) {
      const int32_t *k = tasks + 4 * (size_t)t;
      const int bh = k[0], kv = k[1], q = k[2], w = k[3];
      if (bh < 0 || bh >= BH || kv < 0 || kv >= n || q < 0 || q >= n || (causal && q < kv))
        return fail(DASH_ERR_SCHEDULE, "task %d out of range", t);
      if ((w & dash::kRankMask) >= n) return fail(DASH_ERR_SCHEDULE, "task %d rank out of range", t);
      const bool first = w & dash::kTaskFirst, last = w & dash::kTaskLast;
      if (first == in_run) return fail(DASH_ERR_SCHEDULE, "task %d: runs must start with the first flag", t);
      if (first) {
        rbh = bh;
        rkv = kv;
      } else if (bh != rbh || kv != rkv) {
        return fail(DASH_ERR_SCHEDULE, "task %d changes KV tile inside a run", t);
      }
      in_run = !last;
    }
    if (in_run) return fail(DASH_ERR_SCHEDULE, "CTA %d ends inside a run", s);
  }
  return DASH_OK;
}

// Measures the die map of a workspace once: the latency probe on the call's
// stream (which it synchronises), then the clustering on the host.
dash_status_t ensure_die_map(Workspace *w, int sms, cudaStream_t stream) {
  DieMap &d = w->die;
  if (d.ready) return DASH_OK;
  if (d.tried) return fail(DASH_ERR_UNSUPPORTED, "die-aware placement unavailable: %s", d.why.c_str());
  d.tried = true;
  DevBuf lat, smid;
  cudaError_t e;
  if ((e = d.pool.reserve((size_t)kPoolLines * 128)) != cudaSuccess ||
      (e = lat.reserve((size_t)sms * kPoolLines * 4)) != cudaSuccess || (e = smid.reserve((size_t)sms * 4)) != cudaSuccess) {
    d.why = "allocation failed";
    return fail(DASH_ERR_NO_MEMORY, "die map: %s", cudaGetErrorString(e));
  }
  if ((e = dash::launch_probe_homes((unsigned *)d.pool.ptr, kPoolLines, (unsigned *)lat.ptr, (int *)smid.ptr, sms,
                                    stream)) != cudaSuccess) {
    d.why = "the latency probe did not launch";
    return cuda_fail(e, "die map probe");
  }
  std::vector<uint32_t> h_lat((size_t)sms * kPoolLines);
  std::vector<int> h_sm(sms);
  if ((e = cudaMemcpyAsync(h_lat.data(), lat.ptr, h_lat.size() * 4, cudaMemcpyDeviceToHost, stream)) != cudaSuccess ||
      (e = cudaMemcpyAsync(h_sm.data(), smid.ptr, h_sm.size() * 4, cudaMemcpyDeviceToHost, stream)) != cudaSuccess ||
      (e = cudaStreamSynchronize(stream)) != cudaSuccess) {
    d.why = "the latency probe failed";
    return cuda_fail(e, "die map probe");
  }
  std::vector<int> seen(h_sm);
  std::sort(seen.begin(), seen.end());
  if (std::unique(seen.begin(), seen.end()) != seen.end() || seen.front() < 0) {
    d.why = "the probe did not run one CTA on every SM";
    return fail(DASH_ERR_UNSUPPORTED, "die-aware placement unavailable: %s", d.why.c_str());
  }
  std::vector<int> grp(sms), home(kPoolLines);
  std::string why = dash::cluster_latencies(h_lat.data(), sms, kPoolLines, grp.data(), home.data());
  if (!why.empty()) {
    d.why = why;
    return fail(DASH_ERR_UNSUPPORTED, "die-aware placement unavailable: %s", why.c_str());
  }
  for (int c = 0; c < sms; ++c) d.smids[grp[c]].push_back(h_sm[c]);
  for (int g = 0; g < 2; ++g) std::sort(d.smids[g].begin(), d.smids[g].end());
  d.max_smid = seen.back();
  for (int a = 0; a < kPoolLines; ++a) d.lines[home[a]].push_back(a);
  d.ready = true;
  return DASH_OK;
}

dash_status_t bwd_impl(const void *q, const void *k, const void *v, const void *o, const void *dout,
                       const float *lse, void *dq, void *dk, void *dv, int B, int H, int S, int D, int causal,
                       float scale, dash_schedule_t schedule, const dash_bwd_options_t *opt,
                       cudaStream_t stream) {
  dash_status_t st = check_common(B, H, S, D, scale);
  if (st != DASH_OK) return st;
  const int mode = (int)schedule;
  const int T = (opt && opt->tile) ? opt->tile : auto_tile(S);
  if (T != 64 && T != 128) return fail(DASH_ERR_UNSUPPORTED, "tile %d not supported (64 or 128)", T);
  const int BH = B * H;
  if (BH == 0 || S == 0) return DASH_OK;
  st = check_ptrs({q, k, v, o, dout, lse, dq, dk, dv});
  if (st != DASH_OK) return st;
  if (opt && opt->dq_accum_out && !aligned16(opt->dq_accum_out))
    return fail(DASH_ERR_INVALID_ARG, "dq_accum_out must be 16-byte aligned");
  if (opt && opt->trace && (reinterpret_cast<uintptr_t>(opt->trace) & 7u))
    return fail(DASH_ERR_INVALID_ARG, "trace must be 8-byte aligned");
  if (opt && opt->trace && T != 128) return fail(DASH_ERR_UNSUPPORTED, "the traced kernel has 128-row tiles only");
  const int n = (S + T - 1) / T;
  std::string why = dash::check_mode(mode, n, causal != 0);
  if (!why.empty()) return fail(DASH_ERR_UNSUPPORTED, "%s", why.c_str());
  // task tables index tasks, and the semaphore buffer its words, with 32-bit ints
  if (dash::num_tasks(BH, n, causal != 0) > INT32_MAX || (long long)BH * n * (2 * dash::kSemStride + 1) > INT32_MAX)
    return fail(DASH_ERR_UNSUPPORTED, "%lld tasks: beyond the 32-bit task tables", dash::num_tasks(BH, n, causal != 0));
  const int c = (opt && opt->cost_c > 0) ? opt->cost_c : 4;
  const int r = (opt && opt->cost_r > 0) ? opt->cost_r : 1;
  const long long spin = (opt && opt->spin_limit_ns > 0) ? opt->spin_limit_ns : kDefaultSpinNs;
  if (opt && (opt->dq_chains < 0 || opt->dq_chains > 2))
    return fail(DASH_ERR_INVALID_ARG, "dq_chains must be 0, 1 or 2");
  const int chains = (mode != DASH_SCHED_ATOMIC && opt && opt->dq_chains == 2) ? 2 : 1;
  if (opt && (opt->shift_fill < 0 || opt->shift_fill > 1))
    return fail(DASH_ERR_INVALID_ARG, "shift_fill must be 0 or 1");
  const bool fill = (mode == DASH_SCHED_SHIFT || mode == DASH_SCHED_SYMMETRIC_SHIFT) && opt && opt->shift_fill == 1;
  if (opt && opt->shift_split < -1) return fail(DASH_ERR_INVALID_ARG, "shift_split must be >= -1");
  // -1: the split is chosen by simulation, where split gangs apply (shift and
  // symmetric shift on the library's own table, without fill or die-aware
  // placement); elsewhere it means whole gangs
  const bool split_auto = opt && opt->shift_split == -1 && !fill && !opt->tasks && opt->die_aware != 1 &&
                          (mode == DASH_SCHED_SHIFT || mode == DASH_SCHED_SYMMETRIC_SHIFT);
  const int split = (opt && opt->shift_split > 1) ? opt->shift_split : 1;
  if (split > 1) {
    if (fill || (opt && opt->tasks))
      return fail(DASH_ERR_UNSUPPORTED, "shift_split applies to the library's own table, without fill");
    why = dash::check_split(mode, n, split);
    if (!why.empty()) return fail(DASH_ERR_UNSUPPORTED, "%s", why.c_str());
  }
  if (opt && (opt->rank_order < 0 || opt->rank_order > 1))
    return fail(DASH_ERR_INVALID_ARG, "rank_order must be 0 or 1");
  const bool timed = opt && opt->rank_order == 1 && mode != DASH_SCHED_ATOMIC;
  if (timed && (fill || opt->tasks || opt->die_aware == 1))
    return fail(DASH_ERR_UNSUPPORTED, "rank_order = 1 applies to the library's own table, without fill or die_aware");
  if (opt && (opt->die_aware < 0 || opt->die_aware > 1)) return fail(DASH_ERR_INVALID_ARG, "die_aware must be 0 or 1");
  const bool die_aware = opt && opt->die_aware == 1;
  const bool cyclic = mode == DASH_SCHED_SHIFT || mode == DASH_SCHED_SYMMETRIC_SHIFT;
  if (die_aware && (!cyclic || fill || opt->tasks || split > 1))
    return fail(DASH_ERR_UNSUPPORTED,
                "die_aware applies to shift and symmetric shift, without fill, split gangs or a supplied table");
  const int want_cluster = opt ? opt->cluster_size : 0;
  if (want_cluster < 0 || want_cluster > 16 || (want_cluster & (want_cluster - 1)))
    return fail(DASH_ERR_INVALID_ARG, "cluster_size must be 0 (auto), 1, 2, 4, 8 or 16");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");

  std::lock_guard<std::mutex> lock(g_mu);
  const int sms = sm_count(dev);
  if (sms <= 0) return fail(DASH_ERR_CUDA, "cannot query the SM count");

  // ---- schedule table (cached per device and problem)
  const int32_t *dev_tasks = nullptr;
  const int32_t *dev_off = nullptr;
  int P = 0;
  ScheduleEntry *sched_ent = nullptr;
  std::tuple<int, int, int, int, int, int, int, int, int, int> sched_key;
  ScheduleEntry custom_holder;  // a caller-supplied table lives for this call only
  if (opt && opt->tasks) {
    if (!opt->cta_off || opt->num_ctas < 1) return fail(DASH_ERR_INVALID_ARG, "tasks needs cta_off and num_ctas");
    P = opt->num_ctas;
    if (P > sms) return fail(DASH_ERR_UNSUPPORTED, "num_ctas %d exceeds the %d SMs", P, sms);
    st = validate_table(opt->tasks, opt->cta_off, P, BH, n, causal != 0);
    if (st != DASH_OK) return st;
    if (mode != DASH_SCHED_ATOMIC && !opt->trust_table) {  // the ordered adds must be able to finish
      why = dash::check_table_order(opt->tasks, opt->cta_off, P, BH, n, chains);
      if (!why.empty()) return fail(DASH_ERR_SCHEDULE, "%s", why.c_str());
    }
    const size_t nt = (size_t)opt->cta_off[P];
    if ((e = custom_holder.tasks.reserve(std::max<size_t>(nt, 1) * 16)) != cudaSuccess ||
        (e = custom_holder.cta_off.reserve((P + 1) * 4)) != cudaSuccess)
      return cuda_fail(e, "cudaMalloc (task table)");
    if (nt && (e = cudaMemcpy(custom_holder.tasks.ptr, opt->tasks, nt * 16, cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "cudaMemcpy (task table)");
    if ((e = cudaMemcpy(custom_holder.cta_off.ptr, opt->cta_off, (P + 1) * 4, cudaMemcpyHostToDevice)) !=
        cudaSuccess)
      return cuda_fail(e, "cudaMemcpy (task table)");
    dev_tasks = (const int32_t *)custom_holder.tasks.ptr;
    dev_off = (const int32_t *)custom_holder.cta_off.ptr;
  } else {
    const int want = (opt && opt->num_ctas > 0) ? opt->num_ctas : 0;
    if (want > sms) return fail(DASH_ERR_UNSUPPORTED, "num_ctas %d exceeds the %d SMs", want, sms);
    auto key = std::make_tuple(dev, BH, n, causal ? 1 : 0, mode, want ? want : -sms, c, r, chains,
                               (fill ? -1 : split_auto ? -2 : split) * 2 + (timed ? 1 : 0));
    auto &ent = g_sched[key];
    if (!ent) {
      std::unique_ptr<ScheduleEntry> fresh(new ScheduleEntry());
      // Shift takes whole gangs of CTAs because a gang split over time stalls
      // on its single chain.  With two chains each tile's chain advances
      // every other rank, a split gang no longer stalls, and all SMs pay.
      // With fill, the SMs that whole gangs leave idle run other heads in the
      // serial order (num_ctas, if given, is the CTA budget).
      int Puse = want;
      int use_split = split;
      if (split_auto) {
        int Pk = 0;
        use_split = dash::choose_split(BH, n, causal != 0, mode, sms, c, r, want, &Pk, nullptr);
        if (use_split < 1) {
          g_sched.erase(key);
          return fail(DASH_ERR_UNSUPPORTED, "no split of the gang runs this schedule on up to %d CTAs", sms);
        }
        Puse = Pk;
      }
      if (!Puse && !fill && chains == 2 && mode == DASH_SCHED_SHIFT)
        Puse = (int)std::min<long long>(sms, (long long)BH * n);
      // With timed ranks a gang spread over time does not stall (its tiles are
      // reduced in the order the spread schedule reaches them): every SM.
      if (!Puse && timed && use_split <= 1)
        Puse = (int)std::min<long long>(sms, (long long)BH * dash::chains_per_head(mode, n));
      if (!Puse && !fill) Puse = dash::choose_ctas(BH, n, causal != 0, mode, sms, c, r, split);
      if (Puse < 1 && !fill) {
        g_sched.erase(key);
        return fail(DASH_ERR_UNSUPPORTED, "no CTA count up to %d SMs runs this schedule without deadlock", sms);
      }
      dash::Schedule sch;
      if (fill) {
        why = dash::build_fill(BH, n, causal != 0, mode, want ? want : sms, c, r, &sch, nullptr, nullptr);
        Puse = sch.P;
      } else {
        why = dash::build_schedule(BH, n, causal != 0, mode, Puse, c, r, &sch, use_split, timed);
      }
      if (!why.empty()) {
        g_sched.erase(key);
        return fail(DASH_ERR_SCHEDULE, "%s", why.c_str());
      }
      if ((e = fresh->tasks.reserve(sch.tasks.size() * 4)) != cudaSuccess ||
          (e = fresh->cta_off.reserve(sch.cta_off.size() * 4)) != cudaSuccess) {
        g_sched.erase(key);
        return cuda_fail(e, "cudaMalloc (schedule)");
      }
      cudaMemcpy(fresh->tasks.ptr, sch.tasks.data(), sch.tasks.size() * 4, cudaMemcpyHostToDevice);
      e = cudaMemcpy(fresh->cta_off.ptr, sch.cta_off.data(), sch.cta_off.size() * 4, cudaMemcpyHostToDevice);
      if (e != cudaSuccess) {
        g_sched.erase(key);
        return cuda_fail(e, "cudaMemcpy (schedule)");
      }
      fresh->P = Puse;
      fresh->makespan = sch.makespan;
      fresh->tasks_h = std::move(sch.tasks);
      fresh->cta_off_h = std::move(sch.cta_off);
      ent = std::move(fresh);
    }
    dev_tasks = (const int32_t *)ent->tasks.ptr;
    dev_off = (const int32_t *)ent->cta_off.ptr;
    P = ent->P;
    sched_ent = ent.get();
    sched_key = key;
  }

  // ---- workspace
  Workspace *w = workspace(dev, stream);
  const long long rows_padded = (long long)n * T;
  const long long total_rows = (long long)BH * rows_padded;
  const long long accum_floats = total_rows * D;
  if ((e = w->accum.reserve_on(accum_floats * chains * 4, stream)) != cudaSuccess ||
      (e = w->lse2.reserve_on(total_rows * 4, stream)) != cudaSuccess ||
      (e = w->delta.reserve_on(total_rows * 4, stream)) != cudaSuccess ||
      (e = w->sem.reserve_on((size_t)BH * n * chains * dash::kSemStride * 4, stream)) != cudaSuccess ||
      (e = ensure_status(w)) != cudaSuccess)
    return fail(DASH_ERR_NO_MEMORY, "workspace allocation failed: %s", cudaGetErrorString(e));

  // ---- cluster hand-offs: ranks whose predecessor runs in the same cluster
  // take their turn from a counter in shared memory (same ranks, same bits)
  int cluster = 1;
  const int32_t *dev_links = nullptr;
  if (sched_ent && mode != DASH_SCHED_ATOMIC && !die_aware && want_cluster > 1) {
    auto fit = sched_ent->cluster_for.find({D, T});
    if (fit == sched_ent->cluster_for.end())
      fit = sched_ent->cluster_for.emplace(std::make_pair(D, T), dash::bwd_main_cluster_size(D, T, P)).first;
    if (P % want_cluster != 0 || want_cluster > fit->second)
      return fail(DASH_ERR_UNSUPPORTED, "clusters of %d do not fit the %d CTAs of this schedule", want_cluster, P);
    const int cl = want_cluster;
    // the device words hold a rank in 16 bits beside the links
    bool ranks_fit = true;
    for (size_t t = 3; t < sched_ent->tasks_h.size() && ranks_fit; t += 4)
      ranks_fit = (sched_ent->tasks_h[t] & dash::kRankMask) <= dash::kLinkedRankMask;
    if (cl > 1 && ranks_fit) {
      auto &lk = sched_ent->linked_for[cl];
      if (!lk) {
        const size_t nt = sched_ent->tasks_h.size() / 4;
        std::vector<int32_t> words(nt), table(sched_ent->tasks_h);
        dash::cluster_links(sched_ent->tasks_h.data(), sched_ent->cta_off_h.data(), P, cl, BH, n, chains,
                            words.data());
        for (size_t t = 0; t < nt; ++t) {
          const int32_t w = table[4 * t + 3];
          table[4 * t + 3] = (w & ~dash::kRankMask) | (w & dash::kLinkedRankMask) | words[t];
        }
        std::unique_ptr<DevBuf> buf(new DevBuf());
        if ((e = buf->reserve(std::max<size_t>(table.size(), 4) * 4)) != cudaSuccess ||
            (e = cudaMemcpy(buf->ptr, table.data(), table.size() * 4, cudaMemcpyHostToDevice)) != cudaSuccess) {
          sched_ent->linked_for.erase(cl);
          return cuda_fail(e, "cluster links");
        }
        lk = std::move(buf);
      }
      cluster = cl;
      dev_links = (const int32_t *)lk->ptr;
    }
  }

  // ---- die-aware placement: each gang on one die, its semaphores homed there
  PlacementEntry *placed = nullptr;
  if (die_aware) {
    if ((st = ensure_die_map(w, sms, stream)) != DASH_OK) return st;
    auto &pe = w->placed[sched_key];
    if (!pe) {
      dash::Placement plc;
      why = dash::build_placement(sched_ent->tasks_h.data(), sched_ent->cta_off_h.data(), P,
                                  dash::chains_per_head(mode, n), BH, n, chains, w->die.smids, w->die.lines,
                                  w->die.max_smid, &plc);
      if (!why.empty()) {
        w->placed.erase(sched_key);
        return fail(DASH_ERR_UNSUPPORTED, "die-aware placement: %s", why.c_str());
      }
      std::unique_ptr<PlacementEntry> fresh(new PlacementEntry());
      if ((e = fresh->slot_of_smid.reserve(plc.slot_of_smid.size() * 4)) != cudaSuccess ||
          (e = fresh->sem_idx.reserve(plc.sem_idx.size() * 4)) != cudaSuccess ||
          (e = cudaMemcpy(fresh->slot_of_smid.ptr, plc.slot_of_smid.data(), plc.slot_of_smid.size() * 4,
                          cudaMemcpyHostToDevice)) != cudaSuccess ||
          (e = cudaMemcpy(fresh->sem_idx.ptr, plc.sem_idx.data(), plc.sem_idx.size() * 4, cudaMemcpyHostToDevice)) !=
              cudaSuccess) {
        w->placed.erase(sched_key);
        return cuda_fail(e, "die-aware placement tables");
      }
      fresh->n_smid = (int)plc.slot_of_smid.size();
      pe = std::move(fresh);
    }
    placed = pe.get();
  }

  // ---- tensor maps
  dash::BwdMaps maps;
  if ((st = make_map(&maps.q, q, BH, S, D, T)) != DASH_OK) return st;
  if ((st = make_map(&maps.dout, dout, BH, S, D, T)) != DASH_OK) return st;
  if ((st = make_map(&maps.k, k, BH, S, D, 128)) != DASH_OK) return st;
  if ((st = make_map(&maps.v, v, BH, S, D, 128)) != DASH_OK) return st;

  dash::BwdPreParams pre;
  pre.o = o;
  pre.dout = dout;
  pre.lse = lse;
  pre.lse2 = (float *)w->lse2.ptr;
  pre.delta = (float *)w->delta.ptr;
  pre.dq_accum = (float *)w->accum.ptr;
  // Ordered schedules store their rank-0 partial, so the accumulator needs no
  // zeroing; the atomic schedule (and a caller-supplied table, which need not
  // hold every rank) adds into zeros.
  const bool ordered = mode != DASH_SCHED_ATOMIC;
  // With two chains, chain 1 of a tile may receive nothing (a causal tile with
  // one partial), so its accumulator starts at zero; chain 0 always holds rank 0.
  float *accum = (float *)w->accum.ptr;
  if (ordered && !(opt && opt->tasks)) {
    pre.dq_accum = accum + accum_floats;
    pre.accum_floats = chains > 1 ? accum_floats : 0;
  } else {
    pre.accum_floats = accum_floats * chains;
  }
  pre.sem = placed ? (int *)w->die.pool.ptr : (int *)w->sem.ptr;
  pre.sem_count = placed ? kPoolLines * 32 : BH * n * chains * dash::kSemStride;
  pre.S = S;
  pre.D = D;
  pre.rows_padded = (int)rows_padded;
  pre.total_rows = total_rows;
  if ((e = dash::launch_bwd_preprocess(pre, sms, stream)) != cudaSuccess) return cuda_fail(e, "preprocess launch");

  dash::BwdMainParams mp;
  mp.tasks = (const int4 *)dev_tasks;
  mp.cta_off = dev_off;
  mp.lse2 = pre.lse2;
  mp.delta = pre.delta;
  mp.dq_accum = accum;
  mp.sem = pre.sem;
  mp.dk = (__nv_bfloat16 *)dk;
  mp.dv = (__nv_bfloat16 *)dv;
  mp.status = (int *)w->status.ptr;
  mp.S = S;
  mp.n = n;
  mp.scale = scale;
  mp.scale_log2 = scale * 1.4426950408889634f;
  mp.causal = causal ? 1 : 0;
  mp.ordered = mode != DASH_SCHED_ATOMIC;
  mp.spin_limit_ns = spin;
  mp.chains = chains;
  mp.chain_stride = accum_floats;
  mp.trace = opt ? reinterpret_cast<long long *>(opt->trace) : nullptr;
  if (dev_links) {  // the task table with the links merged into its words
    mp.tasks = (const int4 *)dev_links;
    mp.linked = 1;
  }
  if (placed) {
    mp.slot_of_smid = (const int *)placed->slot_of_smid.ptr;
    mp.n_smid = placed->n_smid;
    mp.sem_idx = (const int *)placed->sem_idx.ptr;
  }
  if (opt && opt->main_begin_event && (e = cudaEventRecord((cudaEvent_t)opt->main_begin_event, stream)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord");
  // die-aware: one CTA per SM, each running the slot of its SM
  if ((e = dash::launch_bwd_main(D, T, maps, mp, placed ? sms : P, stream, cluster)) != cudaSuccess)
    return cuda_fail(e, "main launch");
  if (opt && opt->main_end_event && (e = cudaEventRecord((cudaEvent_t)opt->main_end_event, stream)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord");
  if ((e = dash::launch_bwd_convert(D, T, accum, chains, accum_floats, dq, opt ? opt->dq_accum_out : nullptr,
                                    scale, BH, S, n, sms, stream)) != cudaSuccess)
    return cuda_fail(e, "convert launch");
  return DASH_OK;
}

}  // namespace

namespace dash {
// Lets other translation units of the library report through dash_last_error():
// formats the message, keeps it for this thread and returns the code.
dash_status_t report(dash_status_t code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}
void set_last_error(const char *msg) { g_last_error = msg; }
// The backward's tensor maps for other translation units of the library.
bool encode_bhsd_map(CUtensorMap *m, const void *base, int BH, int S, int D, int box_rows) {
  return make_map(m, base, BH, S, D, box_rows) == DASH_OK;
}
}  // namespace dash

extern "C" {

dash_status_t dash_attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                               int S, int D, int causal, float scale, int cta_pair, dash_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  dash_status_t st = check_common(B, H, S, D, scale);
  if (st != DASH_OK) return st;
  if (cta_pair < -1 || cta_pair > 1) return fail(DASH_ERR_INVALID_ARG, "cta_pair must be -1, 0 or 1");
  if (cta_pair == 1 && D != 128) return fail(DASH_ERR_UNSUPPORTED, "the CTA-pair forward needs D = 128");
  const bool pair = cta_pair == 1 || (cta_pair == -1 && D == 128 && kPairForwardByDefault);
  const int BH = B * H;
  if (BH == 0 || S == 0) return DASH_OK;
  if ((st = check_ptrs({q, k, v, o, lse})) != DASH_OK) return st;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace *w = workspace(dev, stream);
  if ((e = ensure_status(w)) != cudaSuccess) return fail(DASH_ERR_NO_MEMORY, "status word allocation failed");
  CUtensorMap mq, mk, mv;
  if ((st = make_map(&mq, q, BH, S, D, 128)) != DASH_OK) return st;
  if ((st = make_map(&mk, k, BH, S, D, pair ? 64 : 128)) != DASH_OK) return st;  // a pair's CTA loads half a K tile
  if ((st = make_map(&mv, v, BH, S, D, 128)) != DASH_OK) return st;
  dash::FwdParams p;
  p.o = (__nv_bfloat16 *)o;
  p.lse = lse;
  p.status = (int *)w->status.ptr;
  p.S = S;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  p.spin_limit_ns = kDefaultSpinNs;
  e = pair ? dash::launch_fwd_pair(mq, mk, mv, p, BH, stream) : dash::launch_fwd(D, mq, mk, mv, p, BH, stream);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return DASH_OK;
}

dash_status_t dash_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int S,
                            int D, int causal, float scale, dash_stream_t stream) {
  return dash_attn_fwd_ex(q, k, v, o, lse, B, H, S, D, causal, scale, -1, stream);
}

dash_status_t dash_attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                            const float *lse, void *dq, void *dk, void *dv, int B, int H, int S, int D, int causal,
                            float scale, dash_schedule_t schedule, dash_stream_t stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, S, D, causal, scale, schedule, nullptr,
                  (cudaStream_t)stream);
}

dash_status_t dash_attn_bwd_ex(const void *q, const void *k, const void *v, const void *o, const void *dout,
                               const float *lse, void *dq, void *dk, void *dv, int B, int H, int S, int D, int causal,
                               float scale, dash_schedule_t schedule, const dash_bwd_options_t *opt,
                               dash_stream_t stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, S, D, causal, scale, schedule, opt,
                  (cudaStream_t)stream);
}

dash_status_t dash_attn_bwd_host(const void *q, const void *k, const void *v, const void *o, const void *dout,
                                 const float *lse, void *dq, void *dk, void *dv, int B, int H, int S, int D,
                                 int causal, float scale, dash_schedule_t schedule, dash_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  dash_status_t st = check_common(B, H, S, D, scale);
  if (st != DASH_OK) return st;
  if ((long long)B * H * S == 0) return DASH_OK;
  for (const void *p : {q, k, v, o, dout, (const void *)lse, (const void *)dq, (const void *)dk, (const void *)dv})
    if (!p) return fail(DASH_ERR_INVALID_ARG, "null pointer");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const size_t tb = (size_t)B * H * S * D * 2, lb = (size_t)B * H * S * 4;
  uint8_t *d[9];
  CopyLanes *lanes = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    Workspace *w = workspace(dev, stream);
    for (int i = 0; i < 6; ++i)
      if ((e = w->h_in[i].reserve(i == 5 ? lb : tb)) != cudaSuccess)
        return fail(DASH_ERR_NO_MEMORY, "device input buffers: %s", cudaGetErrorString(e));
    for (int i = 0; i < 3; ++i)
      if ((e = w->h_out[i].reserve(tb)) != cudaSuccess)
        return fail(DASH_ERR_NO_MEMORY, "device output buffers: %s", cudaGetErrorString(e));
    for (int i = 0; i < 6; ++i) d[i] = static_cast<uint8_t *>(w->h_in[i].ptr);
    for (int i = 0; i < 3; ++i) d[6 + i] = static_cast<uint8_t *>(w->h_out[i].ptr);
    if ((e = w->lanes.init()) != cudaSuccess) return cuda_fail(e, "copy streams");
    lanes = &w->lanes;
  }
  // Heads are independent problems and each head's dQ order depends on that
  // head alone, so the heads are processed in up to kHostChunks groups: the
  // inputs of one group travel to the device while the group before it runs,
  // and its gradients travel back while the next one runs.  The results are
  // those of one call over all heads, bit for bit.
  const long long BH = (long long)B * H;
  const int nch = BH >= 2 * kHostChunks ? kHostChunks : BH >= 8 ? 4 : BH >= 2 ? 2 : 1;
  const long long per = (BH + nch - 1) / nch;
  const uint8_t *src[6] = {static_cast<const uint8_t *>(q), static_cast<const uint8_t *>(k),
                           static_cast<const uint8_t *>(v), static_cast<const uint8_t *>(o),
                           static_cast<const uint8_t *>(dout), reinterpret_cast<const uint8_t *>(lse)};
  uint8_t *dst[3] = {static_cast<uint8_t *>(dq), static_cast<uint8_t *>(dk), static_cast<uint8_t *>(dv)};
  for (int c = 0; c < nch; ++c) {
    const long long h0 = c * per, h1 = std::min(BH, h0 + per);
    if (h0 >= h1) break;
    const size_t t0 = (size_t)h0 * S * D * 2, tn = (size_t)(h1 - h0) * S * D * 2;
    const size_t l0 = (size_t)h0 * S * 4, ln = (size_t)(h1 - h0) * S * 4;
    for (int i = 0; i < 6; ++i)
      if ((e = cudaMemcpyAsync(d[i] + (i == 5 ? l0 : t0), src[i] + (i == 5 ? l0 : t0), i == 5 ? ln : tn,
                               cudaMemcpyHostToDevice, lanes->in)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpyAsync H2D");
    if ((e = cudaEventRecord(lanes->landed[c], lanes->in)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, lanes->landed[c], 0)) != cudaSuccess)
      return cuda_fail(e, "copy-in ordering");
    st = bwd_impl(d[0] + t0, d[1] + t0, d[2] + t0, d[3] + t0, d[4] + t0, reinterpret_cast<const float *>(d[5] + l0),
                  d[6] + t0, d[7] + t0, d[8] + t0, 1, (int)(h1 - h0), S, D, causal, scale, schedule, nullptr, stream);
    if (st != DASH_OK) {
      cudaStreamSynchronize(lanes->in);
      return st;
    }
    if ((e = cudaEventRecord(lanes->done[c], stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(lanes->out, lanes->done[c], 0)) != cudaSuccess)
      return cuda_fail(e, "copy-out ordering");
    for (int i = 0; i < 3; ++i)
      if ((e = cudaMemcpyAsync(dst[i] + t0, d[6 + i] + t0, tn, cudaMemcpyDeviceToHost, lanes->out)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpyAsync D2H");
  }
  if ((e = cudaStreamSynchronize(lanes->out)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  return dash_sync_status(stream_);
}

long long dash_schedule_num_tasks(int BH, int n, int causal, dash_schedule_t schedule) {
  if (BH < 0 || n < 1 || !dash::check_mode((int)schedule, n, causal != 0).empty()) return -1;
  return dash::num_tasks(BH, n, causal != 0);
}

dash_status_t dash_build_schedule(int BH, int n, int causal, dash_schedule_t schedule, int P, int cost_c, int cost_r,
                                  int32_t *tasks_out, int32_t *cta_off_out, long long *makespan_out) {
  if (!tasks_out || !cta_off_out) return fail(DASH_ERR_INVALID_ARG, "null output pointer");
  std::string why = dash::check_mode((int)schedule, n, causal != 0);
  if (!why.empty()) return fail(DASH_ERR_UNSUPPORTED, "%s", why.c_str());
  dash::Schedule s;
  why = dash::build_schedule(BH, n, causal != 0, (int)schedule, P, cost_c, cost_r, &s);
  if (!why.empty()) return fail(DASH_ERR_SCHEDULE, "%s", why.c_str());
  std::memcpy(tasks_out, s.tasks.data(), s.tasks.size() * 4);
  std::memcpy(cta_off_out, s.cta_off.data(), s.cta_off.size() * 4);
  if (makespan_out) *makespan_out = s.makespan;
  return DASH_OK;
}

dash_status_t dash_check_table(int BH, int n, int causal, int dq_chains, const int32_t *tasks, const int32_t *cta_off,
                               int num_ctas) {
  if (!tasks || !cta_off || num_ctas < 1 || BH < 1 || n < 1)
    return fail(DASH_ERR_INVALID_ARG, "dash_check_table: null table or sizes below 1");
  if (dq_chains < 0 || dq_chains > 2) return fail(DASH_ERR_INVALID_ARG, "dq_chains must be 0, 1 or 2");
  dash_status_t st = validate_table(tasks, cta_off, num_ctas, BH, n, causal != 0);
  if (st != DASH_OK) return st;
  const std::string why = dash::check_table_order(tasks, cta_off, num_ctas, BH, n, dq_chains == 2 ? 2 : 1);
  if (!why.empty()) return fail(DASH_ERR_SCHEDULE, "%s", why.c_str());
  return DASH_OK;
}

dash_status_t dash_build_shift_fill(int BH, int n, int causal, dash_schedule_t schedule, int max_ctas, int cost_c,
                                    int cost_r, int32_t *tasks_out, int32_t *cta_off_out, int *ctas_out,
                                    int *shift_heads_out, int *fill_schedule_out, long long *makespan_out) {
  if (!tasks_out || !cta_off_out) return fail(DASH_ERR_INVALID_ARG, "null output pointer");
  if (schedule != DASH_SCHED_SHIFT && schedule != DASH_SCHED_SYMMETRIC_SHIFT)
    return fail(DASH_ERR_UNSUPPORTED, "fill applies to shift and symmetric shift only");
  std::string why = dash::check_mode((int)schedule, n, causal != 0);
  if (!why.empty()) return fail(DASH_ERR_UNSUPPORTED, "%s", why.c_str());
  dash::Schedule s;
  int hs = 0, fm = -1;
  why = dash::build_fill(BH, n, causal != 0, (int)schedule, max_ctas, cost_c, cost_r, &s, &hs, &fm);
  if (!why.empty()) return fail(DASH_ERR_SCHEDULE, "%s", why.c_str());
  std::memcpy(tasks_out, s.tasks.data(), s.tasks.size() * 4);
  std::memcpy(cta_off_out, s.cta_off.data(), s.cta_off.size() * 4);
  if (ctas_out) *ctas_out = s.P;
  if (shift_heads_out) *shift_heads_out = hs;
  if (fill_schedule_out) *fill_schedule_out = fm;
  if (makespan_out) *makespan_out = s.makespan;
  return DASH_OK;
}

int dash_choose_layout(int BH, int n, int causal, int max_ctas, int cost_c, int cost_r, int *ctas_out,
                       int *split_out, int *rank_order_out, long long *makespan_out) {
  int P = 0, split = 1, timed = 0;
  long long ms = 0;
  const int s = dash::choose_layout(BH, n, causal != 0, max_ctas, cost_c, cost_r, &P, &split, &timed, &ms);
  if (s < 0) {
    dash::set_last_error("dash_choose_layout: BH, n, max_ctas and the costs must be >= 1");
    return -1;
  }
  if (ctas_out) *ctas_out = P;
  if (split_out) *split_out = split;
  if (rank_order_out) *rank_order_out = timed;
  if (makespan_out) *makespan_out = ms;
  return s;
}

dash_status_t dash_build_schedule_ex(int BH, int n, int causal, dash_schedule_t schedule, int split, int rank_order,
                                     int P, int cost_c, int cost_r, int32_t *tasks_out, int32_t *cta_off_out,
                                     long long *makespan_out) {
  if (!tasks_out || !cta_off_out) return fail(DASH_ERR_INVALID_ARG, "null output pointer");
  if (rank_order < 0 || rank_order > 1) return fail(DASH_ERR_INVALID_ARG, "rank_order must be 0 or 1");
  std::string why = dash::check_mode((int)schedule, n, causal != 0);
  if (why.empty()) why = dash::check_split((int)schedule, n, split);
  if (!why.empty()) return fail(DASH_ERR_UNSUPPORTED, "%s", why.c_str());
  dash::Schedule s;
  why = dash::build_schedule(BH, n, causal != 0, (int)schedule, P, cost_c, cost_r, &s, split, rank_order == 1);
  if (!why.empty()) return fail(DASH_ERR_SCHEDULE, "%s", why.c_str());
  std::memcpy(tasks_out, s.tasks.data(), s.tasks.size() * 4);
  std::memcpy(cta_off_out, s.cta_off.data(), s.cta_off.size() * 4);
  if (makespan_out) *makespan_out = s.makespan;
  return DASH_OK;
}

dash_status_t dash_build_split_schedule(int BH, int n, int causal, dash_schedule_t schedule, int split, int P,
                                        int cost_c, int cost_r, int32_t *tasks_out, int32_t *cta_off_out,
                                        long long *makespan_out) {
  if (!tasks_out || !cta_off_out) return fail(DASH_ERR_INVALID_ARG, "null output pointer");
  std::string why = dash::check_mode((int)schedule, n, causal != 0);
  if (why.empty()) why = dash::check_split((int)schedule, n, split);
  if (!why.empty()) return fail(DASH_ERR_UNSUPPORTED, "%s", why.c_str());
  dash::Schedule s;
  why = dash::build_schedule(BH, n, causal != 0, (int)schedule, P, cost_c, cost_r, &s, split);
  if (!why.empty()) return fail(DASH_ERR_SCHEDULE, "%s", why.c_str());
  std::memcpy(tasks_out, s.tasks.data(), s.tasks.size() * 4);
  std::memcpy(cta_off_out, s.cta_off.data(), s.cta_off.size() * 4);
  if (makespan_out) *makespan_out = s.makespan;
  return DASH_OK;
}

int dash_choose_split(int BH, int n, int causal, dash_schedule_t schedule, int max_ctas, int num_ctas, int cost_c,
                      int cost_r, int *ctas_out, long long *makespan_out) {
  if (cost_c < 1 || cost_r < 1 || num_ctas < 0 || num_ctas > max_ctas) return -1;
  return dash::choose_split(BH, n, causal != 0, (int)schedule, max_ctas, cost_c, cost_r, num_ctas, ctas_out,
                            makespan_out);
}

int dash_choose_split_ctas(int BH, int n, int causal, dash_schedule_t schedule, int split, int max_ctas, int cost_c,
                           int cost_r) {
  return dash::choose_ctas(BH, n, causal != 0, (int)schedule, max_ctas, cost_c, cost_r, split);
}

int dash_choose_ctas(int BH, int n, int causal, dash_schedule_t schedule, int max_ctas, int cost_c, int cost_r) {
  return dash::choose_ctas(BH, n, causal != 0, (int)schedule, max_ctas, cost_c, cost_r);
}

dash_status_t dash_fit_costs(int BH, int n, int causal, int max_ctas, double atomic_ms, double serial_ms,
                             int *cost_c_out, int *cost_r_out) {
  if (!cost_c_out || !cost_r_out) return fail(DASH_ERR_INVALID_ARG, "null output pointer");
  std::string why = dash::fit_costs(BH, n, causal != 0, max_ctas, atomic_ms, serial_ms, cost_c_out, cost_r_out);
  if (!why.empty()) return fail(DASH_ERR_INVALID_ARG, "dash_fit_costs: %s", why.c_str());
  return DASH_OK;
}

int dash_choose_schedule(int BH, int n, int causal, int max_ctas, int cost_c, int cost_r, int *ctas_out,
                         long long *makespan_out) {
  int P = 0;
  long long ms = 0;
  const int s = dash::choose_schedule(BH, n, causal != 0, max_ctas, cost_c, cost_r, &P, &ms);
  if (s < 0) {
    dash::set_last_error("dash_choose_schedule: BH, n, max_ctas and the costs must be >= 1");
    return -1;
  }
  if (ctas_out) *ctas_out = P;
  if (makespan_out) *makespan_out = ms;
  return s;
}

int dash_choose_schedule_split(int BH, int n, int causal, int max_ctas, int cost_c, int cost_r, int *ctas_out,
                               int *split_out, long long *makespan_out) {
  int P = 0, split = 1;
  long long ms = 0;
  const int s = dash::choose_schedule(BH, n, causal != 0, max_ctas, cost_c, cost_r, &P, &ms, true, &split);
  if (s < 0) {
    dash::set_last_error("dash_choose_schedule_split: BH, n, max_ctas and the costs must be >= 1");
    return -1;
  }
  if (ctas_out) *ctas_out = P;
  if (split_out) *split_out = split;
  if (makespan_out) *makespan_out = ms;
  return s;
}

dash_status_t dash_cluster_latencies(const uint32_t *lat, int n_sms, int n_lines, int32_t *group_out,
                                     int32_t *home_out) {
  if (!lat || !group_out || !home_out || n_sms < 2 || n_lines < 1)
    return fail(DASH_ERR_INVALID_ARG, "dash_cluster_latencies: null pointer or sizes too small");
  std::vector<int> g(n_sms), h(n_lines);
  const std::string why = dash::cluster_latencies(lat, n_sms, n_lines, g.data(), h.data());
  if (!why.empty()) return fail(DASH_ERR_SCHEDULE, "%s", why.c_str());
  std::copy(g.begin(), g.end(), group_out);
  std::copy(h.begin(), h.end(), home_out);
  return DASH_OK;
}

dash_status_t dash_place_schedule(const int32_t *tasks, const int32_t *cta_off, int P, int gang, int BH, int n,
                                  int chains, const int32_t *sm0, int n0, const int32_t *sm1, int n1,
                                  const int32_t *line0, int m0, const int32_t *line1, int m1, int max_smid,
                                  int32_t *slot_of_smid_out, int32_t *sem_idx_out) {
  if (!tasks || !cta_off || !slot_of_smid_out || !sem_idx_out || (n0 && !sm0) || (n1 && !sm1) || (m0 && !line0) ||
      (m1 && !line1) || n0 < 0 || n1 < 0 || m0 < 0 || m1 < 0)
    return fail(DASH_ERR_INVALID_ARG, "dash_place_schedule: null pointer or negative size");
  const std::vector<int> smids[2] = {std::vector<int>(sm0, sm0 + n0), std::vector<int>(sm1, sm1 + n1)};
  const std::vector<int> lines[2] = {std::vector<int>(line0, line0 + m0), std::vector<int>(line1, line1 + m1)};
  for (int g = 0; g < 2; ++g)
    for (int x : smids[g])
      if (x < 0 || x > max_smid) return fail(DASH_ERR_INVALID_ARG, "SM id %d outside [0, %d]", x, max_smid);
  dash::Placement plc;
  const std::string why = dash::build_placement(tasks, cta_off, P, gang, BH, n, chains, smids, lines, max_smid, &plc);
  if (!why.empty()) return fail(DASH_ERR_SCHEDULE, "%s", why.c_str());
  std::copy(plc.slot_of_smid.begin(), plc.slot_of_smid.end(), slot_of_smid_out);
  std::copy(plc.sem_idx.begin(), plc.sem_idx.end(), sem_idx_out);
  return DASH_OK;
}

dash_status_t dash_cluster_links(const int32_t *tasks, const int32_t *cta_off, int P, int C, int BH, int n,
                                 int chains, int32_t *links_out, long long *n_links_out) {
  if (!tasks || !cta_off || !links_out || P < 1 || C < 1 || C > dash::kMaxClusterLinks || BH < 1 || n < 1 ||
      chains < 1 || chains > 2)
    return fail(DASH_ERR_INVALID_ARG, "dash_cluster_links: null pointer or size out of range");
  const long long k = dash::cluster_links(tasks, cta_off, P, C, BH, n, chains, links_out);
  if (n_links_out) *n_links_out = k;
  return DASH_OK;
}

dash_status_t dash_die_map(dash_stream_t stream_, int32_t *group_of_smid_out, int max_sm, int *n0, int *n1) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (!group_of_smid_out || max_sm < 0) return fail(DASH_ERR_INVALID_ARG, "dash_die_map: null pointer");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_mu);
  const int sms = sm_count(dev);
  if (sms <= 0) return fail(DASH_ERR_CUDA, "cannot query the SM count");
  Workspace *w = workspace(dev, stream);
  dash_status_t st = ensure_die_map(w, sms, stream);
  if (st != DASH_OK) return st;
  for (int i = 0; i <= max_sm; ++i) group_of_smid_out[i] = -1;
  for (int g = 0; g < 2; ++g)
    for (int x : w->die.smids[g])
      if (x <= max_sm) group_of_smid_out[x] = g;
  if (n0) *n0 = (int)w->die.smids[0].size();
  if (n1) *n1 = (int)w->die.smids[1].size();
  return DASH_OK;
}

dash_status_t dash_sync_status(dash_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_ws.find({dev, (void *)stream});
  if (it == g_ws.end() || !it->second->status.ptr) return DASH_OK;
  int word = 0;
  if ((e = cudaMemcpy(&word, it->second->status.ptr, 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "reading the status word");
  if (word == 0) return DASH_OK;
  const int zero = 0;
  cudaMemcpy(it->second->status.ptr, &zero, 4, cudaMemcpyHostToDevice);
  if (word == dash::kStatusSmemMisaligned)
    return fail(DASH_ERR_CUDA, "device status %d: dynamic shared memory not 1024-byte aligned", word);
  return fail(DASH_ERR_TIMEOUT, "device status %d: a bounded wait ran out (%s)", word,
              word == dash::kStatusSemTimeout ? "dQ semaphore" : "mbarrier");
}

void dash_release_workspace(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto it = g_ws.begin(); it != g_ws.end();)
    it = (it->first.first == dev) ? g_ws.erase(it) : std::next(it);
  for (auto it = g_sched.begin(); it != g_sched.end();)
    it = (std::get<0>(it->first) == dev) ? g_sched.erase(it) : std::next(it);
}

const char *dash_last_error(void) { return g_last_error.c_str(); }

int dash_version(void) { return 200; }

}  // extern "C"
