// dash_attn_bwd_noalloc: the attention backward without any device allocation.
//
// Who needs it: code that must not call cudaMalloc (or any allocator) while it
// runs -- a framework whose caching allocator owns all device memory and forbids
// side allocations, an inference/training runtime that reserves a fixed memory
// budget up front, or a caller inside a region where an allocation could block
// or fail.  dash_attn_bwd grows a workspace with cudaMalloc on first use of a
// shape; this entry point instead uses one fixed array of device memory that is
// part of the library image and exists on every GPU that loads the library,
// until the process exits.
//
// The scratch array holds everything the backward needs besides the caller's
// inputs and outputs: the status word, the dQ semaphores, the per-row softmax
// statistics, the fp32 dQ accumulator and the schedule table.  Problems whose
// scratch would exceed kScratchBytes are rejected.  Every call shares the
// array and leaves its contents behind; the parts that must start at zero
// (the status word, the semaphores and, for the atomic schedule, the
// accumulator) are cleared by each call.  Two calls
// whose GPU work overlaps (different streams, or different host threads) race
// on the array; calls on one stream are ordered and safe.
//
// The kernels are the same ones dash_attn_bwd launches, with the same schedule
// table, so a deterministic schedule gives the same bits as dash_attn_bwd;
// only where their scratch lives differs.  The call synchronises its stream
// before it returns, so that it can report a device wait that ran out (the
// status word lives in the shared array, which a later call would clear).
//
// The array's device address is looked up once per device, by the first call
// on that device, and kept for the life of the process.  After
// cudaDeviceReset the library's module is loaded anew and that address is no
// longer valid, so the entry point must not be used after a device reset.
#include "dash.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "kernels.h"
#include "schedule.h"

namespace dash {
dash_status_t report(dash_status_t code, const char *fmt, ...);  // api.cpp: sets dash_last_error()
// TMA map over a contiguous bf16 [BH][S][D] tensor, as the backward's kernels read it (api.cpp)
bool encode_bhsd_map(CUtensorMap *m, const void *base, int BH, int S, int D, int box_rows);
}

namespace {

// 32 MiB: for example the dQ accumulator of B*H*S*D = 7.8 M elements (plus tables).
constexpr size_t kScratchBytes = 32u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device
std::map<std::tuple<int, int, int, int, int, int>, dash::Schedule> g_tables;  // host copies

template <typename... A>
dash_status_t fail(dash_status_t code, const char *fmt, A... args) {
  return dash::report(code, fmt, args...);
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" dash_status_t dash_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                               const void *dout, const float *lse, void *dq, void *dk, void *dv,
                                               int B, int H, int S, int D, int causal, float scale,
                                               dash_schedule_t schedule, dash_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (B < 0 || H < 0 || S < 0) return fail(DASH_ERR_INVALID_ARG, "B, H, S must be >= 0");
  if (D != 64 && D != 128) return fail(DASH_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", D);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(DASH_ERR_INVALID_ARG, "scale must be finite and > 0");
  const long long BH = (long long)B * H;
  if (BH > (1LL << 30) || S > (1 << 30)) return fail(DASH_ERR_INVALID_ARG, "problem too large");
  if (BH == 0 || S == 0) return DASH_OK;
  for (const void *p : {q, k, v, o, dout, (const void *)lse, (const void *)dq, (const void *)dk, (const void *)dv})
    if (!p || (reinterpret_cast<uintptr_t>(p) & 15u)) return fail(DASH_ERR_INVALID_ARG, "null or misaligned pointer");
  const int T = S <= 256 ? 64 : 128;
  const int n = (S + T - 1) / T;
  const int mode = (int)schedule;
  std::string why = dash::check_mode(mode, n, causal != 0);
  if (!why.empty()) return fail(DASH_ERR_UNSUPPORTED, "%s", why.c_str());

  // scratch layout, 256-byte aligned pieces
  const long long rows = BH * n * T;
  const size_t n_tasks = (size_t)dash::num_tasks((int)BH, n, causal != 0);
  size_t off = 0;
  const size_t o_status = off;  off += 256;
  const size_t o_sem = off;     off += up256((size_t)BH * n * dash::kSemStride * 4);
  const size_t o_lse2 = off;    off += up256((size_t)rows * 4);
  const size_t o_delta = off;   off += up256((size_t)rows * 4);
  const size_t o_accum = off;   off += up256((size_t)rows * D * 4);
  const size_t o_tasks = off;   off += up256(n_tasks * 16);
  const size_t o_off = off;     off += up256((size_t)(256 + 1) * 4);
  if (off > kScratchBytes)
    return fail(DASH_ERR_UNSUPPORTED,
                "problem needs %zu bytes of scratch; the allocation-free backward has a fixed %zu-byte array "
                "(use dash_attn_bwd for larger problems)",
                off, kScratchBytes);

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DASH_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(DASH_ERR_UNSUPPORTED, "device index %d too large", dev);

  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {  // once per device, with that device current
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr)
      return fail(DASH_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = ptr;
  }
  unsigned char *base = static_cast<unsigned char *>(g_scratch_ptr[dev]);

  int sms = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess || sms < 1)
    return fail(DASH_ERR_CUDA, "cannot query the SM count");
  const int max_ctas = sms < 256 ? sms : 256;  // the CTA-offset slot in the scratch holds 257 entries
  auto key = std::make_tuple((int)BH, n, causal ? 1 : 0, mode, max_ctas, dev);
  auto it = g_tables.find(key);
  if (it == g_tables.end()) {
    const int P = dash::choose_ctas((int)BH, n, causal != 0, mode, max_ctas, 4, 1);
    if (P < 1) return fail(DASH_ERR_UNSUPPORTED, "no CTA count runs this schedule without deadlock");
    dash::Schedule sch;
    why = dash::build_schedule((int)BH, n, causal != 0, mode, P, 4, 1, &sch);
    if (!why.empty()) return fail(DASH_ERR_SCHEDULE, "%s", why.c_str());
    it = g_tables.emplace(key, std::move(sch)).first;
  }
  const dash::Schedule &sch = it->second;

  dash::BwdMaps maps;
  if (!dash::encode_bhsd_map(&maps.q, q, (int)BH, S, D, T) ||
      !dash::encode_bhsd_map(&maps.dout, dout, (int)BH, S, D, T) ||
      !dash::encode_bhsd_map(&maps.k, k, (int)BH, S, D, 128) ||
      !dash::encode_bhsd_map(&maps.v, v, (int)BH, S, D, 128))
    return fail(DASH_ERR_CUDA, "cuTensorMapEncodeTiled failed");

  // the table goes into the scratch; the status word starts at zero
  if ((e = cudaMemcpyAsync(base + o_tasks, sch.tasks.data(), sch.tasks.size() * 4, cudaMemcpyHostToDevice,
                           stream)) != cudaSuccess ||
      (e = cudaMemcpyAsync(base + o_off, sch.cta_off.data(), sch.cta_off.size() * 4, cudaMemcpyHostToDevice,
                           stream)) != cudaSuccess ||
      (e = cudaMemsetAsync(base + o_status, 0, 4, stream)) != cudaSuccess)
    return fail(DASH_ERR_CUDA, "staging the schedule: %s", cudaGetErrorString(e));

  dash::BwdPreParams pre;
  pre.o = o;
  pre.dout = dout;
  pre.lse = lse;
  pre.lse2 = reinterpret_cast<float *>(base + o_lse2);
  pre.delta = reinterpret_cast<float *>(base + o_delta);
  pre.dq_accum = reinterpret_cast<float *>(base + o_accum);
  // Ordered schedules store the partial of rank 0, so only the atomic
  // schedule's accumulator must start at zero (as in dash_attn_bwd).
  pre.accum_floats = mode == DASH_SCHED_ATOMIC ? rows * D : 0;
  pre.sem = reinterpret_cast<int *>(base + o_sem);
  pre.sem_count = (int)(BH * n * dash::kSemStride);
  pre.S = S;
  pre.D = D;
  pre.rows_padded = n * T;
  pre.total_rows = rows;
  if ((e = dash::launch_bwd_preprocess(pre, sms, stream)) != cudaSuccess)
    return fail(DASH_ERR_CUDA, "preprocess launch: %s", cudaGetErrorString(e));

  dash::BwdMainParams mp;
  mp.tasks = reinterpret_cast<const int4 *>(base + o_tasks);
  mp.cta_off = reinterpret_cast<const int *>(base + o_off);
  mp.lse2 = pre.lse2;
  mp.delta = pre.delta;
  mp.dq_accum = pre.dq_accum;
  mp.sem = pre.sem;
  mp.dk = (__nv_bfloat16 *)dk;
  mp.dv = (__nv_bfloat16 *)dv;
  mp.status = reinterpret_cast<int *>(base + o_status);
  mp.S = S;
  mp.n = n;
  mp.scale = scale;
  mp.scale_log2 = scale * 1.4426950408889634f;
  mp.causal = causal ? 1 : 0;
  mp.ordered = mode != DASH_SCHED_ATOMIC;
  mp.spin_limit_ns = 2000000000LL;
  mp.chains = 1;
  mp.chain_stride = 0;
  if ((e = dash::launch_bwd_main(D, T, maps, mp, sch.P, stream)) != cudaSuccess)
    return fail(DASH_ERR_CUDA, "main launch: %s", cudaGetErrorString(e));
  if ((e = dash::launch_bwd_convert(D, T, pre.dq_accum, 1, 0, dq, nullptr, scale, (int)BH, S, n, sms, stream)) !=
      cudaSuccess)
    return fail(DASH_ERR_CUDA, "convert launch: %s", cudaGetErrorString(e));

  int word = 0;
  if ((e = cudaMemcpyAsync(&word, base + o_status, 4, cudaMemcpyDeviceToHost, stream)) != cudaSuccess ||
      (e = cudaStreamSynchronize(stream)) != cudaSuccess)
    return fail(DASH_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  if (word != 0) return fail(DASH_ERR_TIMEOUT, "device status %d: a bounded wait ran out", word);
  return DASH_OK;
}
