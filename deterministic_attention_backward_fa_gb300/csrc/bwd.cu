// Deterministic attention backward for sm_103a.
//
// Three kernels run on the caller's stream:
//   1. dash_bwd_preprocess: delta_i = sum_d dO_id O_id, lse2_i = LSE_i*log2(e)
//      per query row, and zeroing of the fp32 dQ accumulator and semaphores;
//   2. dash_bwd_main: persistent, one CTA per schedule slot, walking the task
//      table that the host generator built.  Each task is one KV tile against
//      one Q tile.  dK/dV of the CTA's current KV tile accumulate in tensor
//      memory; the task's dQ partial is added into the accumulator after the
//      CTA has acquired the tile's semaphore at the task's rank, and the
//      semaphore is then released at rank + 1 (DASH overview (zskr.cn),
//      section 2.1: serialised dQ reduction; sections 3.1-3.3: the orders);
//   3. dash_bwd_convert: dQ = bf16(scale * accumulator).
//
// Main-kernel roles (512 threads, four warpgroups):
//   warp 0       TMA producer: K/V once per KV run, Q and LSE per task
//   warp 2       TMA producer: dO and delta per task (a separate ring, so a
//                Q tile can land while the dO buffer is still busy)
//   warp 1       tensor-memory owner and single-lane tcgen05 MMA issuer
//   warp 3       idle (gives its registers to the other warpgroups)
//   warps 4-11   softmax: warp w handles TMEM sub-partition w % 4 (32 KV rows)
//                and half of the Q columns.  Pass A turns S^T into P and
//                stores it back packed as bf16 in tensor memory; pass B forms
//                dS = P (dP - delta) and writes it to shared memory
//   warps 12-15  dQ reduction: move the task's dQ partial from TMEM into
//                registers (tensor memory is free again at once); for an
//                ordered schedule, acquire the dQ tile's semaphore (one 32-byte
//                L2 sector each) at the task's rank, add the whole partial into
//                the fp32 accumulator from registers with vector reductions,
//                paced so that they do not clog the load/store queue
//                (rank 0 stores instead, so the accumulator needs no zeroing)
//                and release rank + 1 once every reduction is issued and
//                ordered before the release.  No shared memory is held while
//                the chain advances.  With two chains (an option) the tile's
//                even and odd ranks go to two accumulators, each its own chain.
//                A lane of the second of these warps waits for the turn, so
//                that the wait overlaps the leader's previous release.  For
//                the atomic schedule at D = 128, half the partial is staged in
//                the task's dO buffer (dV has read it) and added by the TMA
//                engine (bulk reduce-add), the other half by vector
//                reductions; at D = 64 all of it from registers.  At the end
//                of a KV run these warps write dK and dV
// setmaxnreg gives the reduction warpgroup enough registers to hold a dQ row.
//
// All MMAs are M = 128: the lanes are KV rows for S^T = K Q^T, dP^T = V dO^T,
// dV += P^T dO and dK += dS^T Q, and Q rows for dQ = dS K.  With 64-row tiles
// the KV side is padded to 128 rows (rows past the tile are masked to P = 0)
// and the Q side of dQ has 64 valid rows.
//
// Tensor memory (512 columns): S^T at 0, dP^T at 128, dV at 256, dK at 256+D.
// A softmax warp of half h turns its columns [32h + 64c, +32) of S^T into
// packed bf16 P at columns [32h + 16c, +16), inside columns it has itself
// already read, so the two halves never race; dV reads P from there as its
// TMEM A operand.  dS lives in shared memory as [q/64][kv][64 q], which is the
// MN-major A operand of dQ and the K-major A operand of dK at once.  dQ (one
// N = D MMA) goes to the dP^T columns when D = 128 and to columns 384+ when
// D = 64.
//
// Per task the MMA warp issues S^T, dP^T (once the previous dQ has left the
// dP^T columns; at D = 64 one task early, right after pass B has read the
// previous dP^T), dV, then, if the next task stays on this KV tile and its Q
// tile has landed, the next S^T, so that pass A of the next task overlaps
// this task's dQ and dK; then dQ and dK.
#include <cuda_runtime.h>

#include "kernels.h"
#include "sm103.cuh"

namespace dash {

using namespace dev;

namespace {

constexpr int kThreads = 512;
constexpr int kSoftWarp0 = 4;
constexpr int kNumSoftWarps = 8;
constexpr int kRedWarp0 = 12;
constexpr int kRedThreads = 128;
constexpr int kDrainBar = 2;          // named barrier of the dQ-reduction warps
constexpr int kNumRedWarps = 4;
// Pauses between the dQ reductions of a reduction warp (see the drain).  On
// the ordered path they lie on the tile's chain, so they are short.
constexpr unsigned kRedPauseOrderedNs = 16;  // after every reduction
constexpr unsigned kRedPauseAtomicNs = 96;   // after every third reduction
constexpr int kRegsLaunch = 128;      // 512 threads x 128 = the whole register file
constexpr int kRegsProducer = 56;     // warpgroup 0 after setmaxnreg.dec
static_assert(kRegsProducer < kRegsLaunch, "warpgroup 0 must give registers up before the others take them");
constexpr int kRegsSoftmax = 128;     // warpgroups 1, 2 (unchanged)
constexpr int kRegsReduce = 200;      // warpgroup 3 after setmaxnreg.inc (holds a dQ row)
static_assert(kRegsProducer * 128 + 2 * kRegsSoftmax * 128 + kRegsReduce * 128 <= kRegsLaunch * kThreads,
              "register split exceeds the CTA's allocation");

template <int D, int T>
struct BwdCfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kKvRows = 128;
  static constexpr int kStages = (D == 128 && T == 128) ? 2 : 3;
  static constexpr uint32_t kKvBytes = kKvRows * D * 2;   // K (and V) tile
  static constexpr uint32_t kKvPanel = kKvRows * 128;     // bytes per 64-column panel
  static constexpr uint32_t kQBytes = T * D * 2;          // Q (and dO) tile
  static constexpr uint32_t kQPanel = T * 128;
  static constexpr uint32_t kDsBytes = 128 * 128 * 2;     // dS as the A operand of dQ = dS K
  static constexpr uint32_t kDsPanel = 128 * 128;
  // shared-memory layout (offsets from a 1024-byte aligned base)
  static constexpr uint32_t oK = 0;
  static constexpr uint32_t oV = oK + kKvBytes;
  static constexpr uint32_t oQ = oV + kKvBytes;
  static constexpr uint32_t oDO = oQ + kStages * kQBytes;
  static constexpr uint32_t oDS = oDO + kStages * kQBytes;
  static constexpr uint32_t oLSE = oDS + kDsBytes;
  static constexpr uint32_t oDELTA = oLSE + kStages * T * 4;
  static constexpr uint32_t oBAR = oDELTA + kStages * T * 4;
  static constexpr int kNumBars = 12 + 4 * kStages;
  static constexpr uint32_t oMISC = oBAR + kNumBars * 8;
  static constexpr uint32_t oTURN = oMISC + 16;                  // hand-off counters, one per CTA of the cluster
  static constexpr uint32_t oSEEN = oTURN + 4 * kMaxClusterLinks;  // turns taken from each, by the poller
  static constexpr uint32_t kSmemBytes = oSEEN + 4 * kMaxClusterLinks;
  // tensor-memory columns
  static constexpr uint32_t cS = 0, cDP = 128, cDV = 256, cDK = 256 + D;
  static constexpr uint32_t cDQ = (D == 128) ? 128u : 384u;
  static constexpr bool kDqInDp = (D == 128);  // dQ reuses the dP^T columns
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kChunks = T / 64;  // 32-column chunks per softmax warp
};

// barrier indices
enum {
  bKvFull = 0, bKvEmpty, bSFull, bDpFull, bPFull, bDsFull, bDqFull, bTmemFree, bKDone, bDkvFull, bDkvEmpty, bFinal,
  bQFull0
};

// setmaxnreg towards N registers per thread: .inc may only raise and .dec only
// lower the warpgroup's count (which starts at kRegsLaunch), so the direction
// follows from N.
template <int N>
__device__ __forceinline__ void regs_set() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg takes a multiple of 8 in [24, 256]");
  if constexpr (N > kRegsLaunch) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
  } else if constexpr (N < kRegsLaunch) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
  }
}
__device__ __forceinline__ void regs_dec() { regs_set<kRegsProducer>(); }
// Phase stamp of the traced kernel (compiled out of the plain one).
template <bool kTrace>
__device__ __forceinline__ void trace_put(const BwdMainParams &p, int t, int slot, long long v) {
  if constexpr (kTrace) p.trace[(size_t)t * kTraceSlots + slot] = v;
}
// The SM clock, read where it stands in the program: the volatile asm with a
// memory clobber keeps the compiler from moving it across the waits it times.
__device__ __forceinline__ long long clk() {
  long long r;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(r) : : "memory");
  return r;
}
__device__ __forceinline__ unsigned smid() {
  unsigned r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void regs_softmax() { regs_set<kRegsSoftmax>(); }
__device__ __forceinline__ void regs_reduce() { regs_set<kRegsReduce>(); }

template <int D, int T, bool kTrace>
__global__ void __launch_bounds__(kThreads, 1)
    dash_bwd_main(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdMainParams p) {
  using C = BwdCfg<D, T>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // With die-aware placement every SM holds one CTA, which runs the slot that
  // the host gave its SM (or nothing, before any set-up).
  int slot = blockIdx.x;
  if (p.slot_of_smid) {
    const int s = (int)smid();
    slot = s < p.n_smid ? p.slot_of_smid[s] : -1;
    if (slot < 0) return;
  }

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::oBAR);
  uint64_t *qfullQ = bars + bQFull0;                   // Q tile + LSE landed
  uint64_t *qfullDO = bars + bQFull0 + C::kStages;      // dO tile + delta landed
  uint64_t *qemptyQ = bars + bQFull0 + 2 * C::kStages;  // Q buffer + LSE free
  uint64_t *qemptyDO = bars + bQFull0 + 3 * C::kStages; // dO buffer (+ staged dQ half) + delta free
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::oMISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::oMISC + 4);
  uint32_t *pass_done = reinterpret_cast<uint32_t *>(smem + C::oMISC + 8);  // traced: softmax warps done, per pass
  uint32_t *turn_count = reinterpret_cast<uint32_t *>(smem + C::oTURN);
  uint32_t *turns_seen = reinterpret_cast<uint32_t *>(smem + C::oSEEN);

  if ((smem_u32(smem) & 1023u) != 0) {  // swizzled operand tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kStatusSmemMisaligned);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars[bKvFull], 1);
    mbar_init(&bars[bKvEmpty], 1);
    mbar_init(&bars[bSFull], 1);
    mbar_init(&bars[bDpFull], 1);
    mbar_init(&bars[bPFull], kNumSoftWarps);
    mbar_init(&bars[bDsFull], kNumSoftWarps);
    mbar_init(&bars[bDqFull], 1);
    mbar_init(&bars[bTmemFree], kNumRedWarps);
    mbar_init(&bars[bKDone], 1);
    mbar_init(&bars[bDkvFull], 1);
    mbar_init(&bars[bDkvEmpty], kNumRedWarps);
    mbar_init(&bars[bFinal], 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&qfullQ[s], 1);
      mbar_init(&qfullDO[s], 1);
      mbar_init(&qemptyQ[s], 1 + kNumSoftWarps);  // dK's commit + the softmax warps (LSE)
      mbar_init(&qemptyDO[s], kNumSoftWarps + 1);   // the softmax warps (delta) + the dQ half's TMA read
    }
    *abort_flag = 0;
    pass_done[0] = pass_done[1] = 0;
    for (int i = 0; i < kMaxClusterLinks; ++i) turn_count[i] = turns_seen[i] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (p.linked) cluster_sync_all();  // every CTA's hand-off counters are zero before any is raised
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Guard g{abort_flag, p.status, (uint64_t)p.spin_limit_ns};

  const int t_begin = p.cta_off[slot], t_end = p.cta_off[slot + 1];
  const int4 *tasks = p.tasks;

  if (warp < 4) {
    regs_dec();
    if ((warp == 0 || warp == 2) && lane == 0) {
      // ------------------------------------------------------------ producers
      // warp 0: K and V once per KV run, Q and LSE per task; warp 2: dO and
      // delta per task.  Separate rings let Q arrive as soon as its buffer is
      // free, independently of the dO buffer (which also stages half of dQ).
      const bool qside = warp == 0;
      uint64_t *full = qside ? qfullQ : qfullDO;
      uint64_t *empty = qside ? qemptyQ : qemptyDO;
      const CUtensorMap *map = qside ? &tmQ : &tmDO;
      uint8_t *buf0 = smem + (qside ? C::oQ : C::oDO);
      uint8_t *row0p = smem + (qside ? C::oLSE : C::oDELTA);
      const float *rowsrc = qside ? p.lse2 : p.delta;
      uint32_t kv_e_phase = 0;
      PhaseBits e_phase;
      uint32_t f_last[C::kStages] = {};
      bool used[C::kStages] = {};
      bool kv_issued = false;
      uint32_t kv_last = 0, kv_fills = 0;
      int st = 0, runs = 0;
      int4 nxt = t_begin < t_end ? tasks[t_begin] : make_int4(0, 0, 0, 0);
      for (int t = t_begin; t < t_end; ++t) {
        const int4 tk = nxt;
        if (t + 1 < t_end) nxt = tasks[t + 1];
        const int bh = tk.x, kv = tk.y, q = tk.z;
        if (qside && (tk.w & kTaskFirstFlag)) {
          if (runs > 0) {
            mbar_wait(&bars[bKvEmpty], kv_e_phase, g);
            kv_e_phase ^= 1;
          }
          ++runs;
          if (!*g.abort) {
            mbar_arrive_expect_tx(&bars[bKvFull], 2 * C::kKvBytes);
            for (int pn = 0; pn < C::kPanels; ++pn) {
              tma_load_3d(smem + C::oK + pn * C::kKvPanel, &tmK, &bars[bKvFull], pn * 64, kv * T, bh);
              tma_load_3d(smem + C::oV + pn * C::kKvPanel, &tmV, &bars[bKvFull], pn * 64, kv * T, bh);
            }
            kv_issued = true;
            kv_last = kv_fills & 1;
            ++kv_fills;
          }
        }
        if (used[st]) {
          mbar_wait(&empty[st], e_phase[st], g);
          e_phase.flip(st);
        }
        if (!*g.abort) {
          const uint32_t fill = used[st] ? (f_last[st] ^ 1) : 0;
          mbar_arrive_expect_tx(&full[st], C::kQBytes + T * 4);
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(buf0 + st * C::kQBytes + pn * C::kQPanel, map, &full[st], pn * 64, q * T, bh);
          bulk_load(row0p + st * T * 4, rowsrc + ((size_t)bh * p.n + q) * T, T * 4, &full[st]);
          f_last[st] = fill;
          used[st] = true;
        }
        st = (st + 1 == C::kStages) ? 0 : st + 1;
      }
      // let copies still in flight land before the CTA exits
      for (int s = 0; s < C::kStages; ++s)
        if (used[s]) mbar_drain(&full[s], f_last[s], g.limit_ns);
      if (kv_issued) mbar_drain(&bars[bKvFull], kv_last, g.limit_ns);
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idS = idesc_bf16(128, T, 0, 0);    // S^T, dP^T: K-major A and B
      constexpr uint32_t idKV = idesc_bf16(128, D, 0, 1);   // dV, dK: A K-major (TMEM / smem), B MN-major
      constexpr uint32_t idQ = idesc_bf16(128, D, 1, 1);    // dQ: MN-major A and B
      uint32_t kvf_phase = 0, dkve_phase = 0, pf_phase = 0, dsf_phase = 0, tf_phase = 0;
      PhaseBits qfq_phase, qfd_phase;
      int st = 0, runs = 0;
      const uint32_t sK = smem_u32(smem + C::oK), sV = smem_u32(smem + C::oV);
      const uint32_t sDS = smem_u32(smem + C::oDS);
      uint64_t dK_k = sw128_desc(sK, 16, 1024), dV_k = sw128_desc(sV, 16, 1024);  // K-major
      uint64_t dK_m = sw128_desc(sK, C::kKvPanel, 1024);                          // MN-major
      uint64_t dDS_m = sw128_desc(sDS, C::kDsPanel, 1024);                        // dS as A of dQ
      uint64_t dDS_k = sw128_desc(sDS, 16, 1024);                                 // dS^T as A of dK
      bool issued = false, s_early = false, dp_early = false;
      // S^T = K Q^T into the S^T columns (M = 128 KV rows, N = T, K = D).  A
      // descriptor plus (byte offset >> 4) addresses the same tile further on.
      auto issue_s = [&](int stage) {
        const uint64_t dQk = sw128_desc(smem_u32(smem + C::oQ + stage * C::kQBytes), 16, 1024);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kKvPanel + (kk & 3) * 32) >> 4;
          const uint32_t offq = ((kk >> 2) * C::kQPanel + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::cS, dK_k + off, dQk + offq, idS, kk > 0);
        }
        tc_commit(&bars[bSFull]);
        issued = true;
      };
      // dP^T = V dO^T into the dP^T columns (same shape as S^T).
      auto issue_dp = [&](int stage) {
        const uint64_t dDOk = sw128_desc(smem_u32(smem + C::oDO + stage * C::kQBytes), 16, 1024);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kKvPanel + (kk & 3) * 32) >> 4;
          const uint32_t offq = ((kk >> 2) * C::kQPanel + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::cDP, dV_k + off, dDOk + offq, idS, kk > 0);
        }
        tc_commit(&bars[bDpFull]);
      };
      int4 nxt = t_begin < t_end ? tasks[t_begin] : make_int4(0, 0, 0, 0);
      for (int t = t_begin; t < t_end; ++t) {
        const int4 tk = nxt;
        if (t + 1 < t_end) nxt = tasks[t + 1];
        const bool first = tk.w & kTaskFirstFlag, last = tk.w & kTaskLastFlag;
        if (first) {
          mbar_wait(&bars[bKvFull], kvf_phase, g);
          kvf_phase ^= 1;
          if (runs > 0) {
            mbar_wait(&bars[bDkvEmpty], dkve_phase, g);
            dkve_phase ^= 1;
          }
          ++runs;
        }
        const uint32_t sQ = smem_u32(smem + C::oQ + st * C::kQBytes);
        const uint32_t sDO = smem_u32(smem + C::oDO + st * C::kQBytes);
        // keep the per-k-step descriptor sums inside the loop (hoisting all of
        // them out of it would need more registers than this warp has)
        asm volatile("" : "+l"(dK_k), "+l"(dV_k), "+l"(dK_m), "+l"(dDS_m), "+l"(dDS_k));
        if (!s_early) {  // S^T of this task was not issued during the previous one
          mbar_wait(&qfullQ[st], qfq_phase[st], g);
          qfq_phase.flip(st);
          if (!*g.abort) issue_s(st);
        }
        if (!dp_early) {  // dP^T of this task was not issued during the previous one
          mbar_wait(&qfullDO[st], qfd_phase[st], g);
          qfd_phase.flip(st);
          if (C::kDqInDp && t > t_begin) {  // the previous dQ sits in the dP^T columns
            mbar_wait(&bars[bTmemFree], tf_phase, g);
            tf_phase ^= 1;
          }
          trace_put<kTrace>(p, t, kTrMmaDp, clk());
          if (!*g.abort) issue_dp(st);
        }
        mbar_wait(&bars[bPFull], pf_phase, g);
        pf_phase ^= 1;
        trace_put<kTrace>(p, t, kTrMmaDv, clk());
        const uint64_t dQm = sw128_desc(sQ, C::kQPanel, 1024), dDOm = sw128_desc(sDO, C::kQPanel, 1024);
        if (!*g.abort) {
          tc_fence_after();
          // dV += P^T dO: A from TMEM (packed bf16), B MN-major, K = T.  k-step
          // (c, h, j) covers Q rows 32h + 64c + 16j, whose P sits at packed
          // column 32h + 16c + 8j.
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const uint32_t acol = 32 * h + 16 * c + 8 * j, q0 = 32 * h + 64 * c + 16 * j;
                mma_ts(tmem + C::cDV, tmem + C::cS + acol, dDOm + ((q0 * 128) >> 4), idKV,
                       (!first || c + h + j > 0) ? 1u : 0u);
              }
        }
        // The next task's S^T may go now (its columns are free once dV has read
        // P; MMAs run in issue order) if it stays on this KV tile and its Q tile
        // has already landed: the softmax warps then overlap it with dQ and dK.
        s_early = false;
        if (t + 1 < t_end && !(nxt.w & kTaskFirstFlag) && !*g.abort) {
          const int st1 = (st + 1 == C::kStages) ? 0 : st + 1;
          if (mbar_test(&qfullQ[st1], qfq_phase[st1])) {
            qfq_phase.flip(st1);
            issue_s(st1);
            s_early = true;
          }
        }
        trace_put<kTrace>(p, t, kTrMmaDvOut, clk());
        mbar_wait(&bars[bDsFull], dsf_phase, g);
        dsf_phase ^= 1;
        trace_put<kTrace>(p, t, kTrMmaDsSeen, clk());
        // With dQ in columns of its own (D = 64), the next task's dP^T may go
        // ahead of this task's dQ and dK once pass B has read this dP^T, if it
        // stays on this KV tile and its dO tile has landed: the softmax warps
        // then find it done when they finish the next pass A.
        dp_early = false;
        if (!C::kDqInDp && t + 1 < t_end && !(nxt.w & kTaskFirstFlag) && !*g.abort) {
          const int st1 = (st + 1 == C::kStages) ? 0 : st + 1;
          if (mbar_test(&qfullDO[st1], qfd_phase[st1])) {
            qfd_phase.flip(st1);
            trace_put<kTrace>(p, t + 1, kTrMmaDp, clk());
            issue_dp(st1);
            dp_early = true;
          }
        }
        if (!C::kDqInDp && t > t_begin) {
          mbar_wait(&bars[bTmemFree], tf_phase, g);
          tf_phase ^= 1;
        }
        trace_put<kTrace>(p, t, kTrMmaDq, clk());
        if (!*g.abort) {
          tc_fence_after();
          // dQ = dS K first (it is on the critical path: the drain frees the
          // next dP^T's columns), M = 128 Q rows, N = D, K = 128 KV rows
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::cDQ, dDS_m + ((kk * 2048) >> 4), dK_m + ((kk * 2048) >> 4), idQ, kk > 0);
          tc_commit(&bars[bDqFull]);
          // dK += dS^T Q with dS^T read from shared memory as a K-major A operand
          // ([q/64][kv][64 q] is exactly that layout), B = Q MN-major
#pragma unroll
          for (int kk = 0; kk < T / 16; ++kk) {
            const uint32_t offa = ((kk >> 2) * C::kDsPanel + (kk & 3) * 32) >> 4;
            mma_ss(tmem + C::cDK, dDS_k + offa, dQm + ((kk * 16 * 128) >> 4), idKV,
                   (!first || kk > 0) ? 1u : 0u);
          }
          tc_commit(&bars[bKDone]);   // the dS tile is no longer read
          tc_commit(&qemptyQ[st]);    // nor is this task's Q tile
          if (last) {
            tc_commit(&bars[bDkvFull]);
            tc_commit(&bars[bKvEmpty]);
          }
        }
        trace_put<kTrace>(p, t, kTrMmaEnd, clk());
        st = (st + 1 == C::kStages) ? 0 : st + 1;
      }
      if (issued) {  // every MMA has completed before tensor memory is released
        tc_commit(&bars[bFinal]);
        mbar_drain(&bars[bFinal], 0, g.limit_ns);
      }
    }
  } else if (warp < kRedWarp0) {
    // ------------------------------------------------------------ softmax
    regs_softmax();
    const int sub = warp & 3;                 // TMEM sub-partition: KV rows 32*sub ..
    const int half = (warp - kSoftWarp0) >> 2;
    const int L = sub * 32 + lane;            // this thread's KV row (TMEM lane)
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    uint32_t sf_phase = 0, dpf_phase = 0, kd_phase = 0;
    PhaseBits qfq_phase, qfd_phase;
    int st = 0;
    uint8_t *sDS = smem + C::oDS;
    int4 nxt = t_begin < t_end ? tasks[t_begin] : make_int4(0, 0, 0, 0);
    for (int t = t_begin; t < t_end; ++t) {
      const int4 tk = nxt;
      if (t + 1 < t_end) nxt = tasks[t + 1];
      const int kv = tk.y, q = tk.z;
      const float *sL = reinterpret_cast<const float *>(smem + C::oLSE + st * T * 4);
      const float *sDl = reinterpret_cast<const float *>(smem + C::oDELTA + st * T * 4);
      mbar_wait(&qfullQ[st], qfq_phase[st], g);  // LSE
      qfq_phase.flip(st);
      mbar_wait(&bars[bSFull], sf_phase, g);
      sf_phase ^= 1;
      const bool tracer = kTrace && warp == kSoftWarp0 && lane == 0;
      if (tracer) trace_put<kTrace>(p, t, kTrPassA0, clk());
      float pv[C::kChunks][32];  // P of this thread's row and columns, kept for pass B
      if (!warp_aborted(g)) {
        tc_fence_after();
        const int kv_g = kv * T + L;
        const bool row_ok = (L < T) && (kv_g < p.S);
        const int qbase = q * T;
        // Masking is needed only where a row lies past the sequence or, for a
        // causal mask, the tile reaches above the diagonal; the test is made
        // warp-uniform so that the unmasked path does not diverge.
        const bool masked = __any_sync(0xffffffffu, !row_ok || (p.causal && qbase < kv_g));
        // pass A: P = exp(scale * S - LSE) (masked), packed bf16 into the S^T columns
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          const int j0 = 32 * half + 64 * c;         // first Q column of the chunk
          const uint32_t pcol = 32 * half + 16 * c;  // its packed P column
          uint32_t s[32];
          tmem_ld32(tl + C::cS + j0, s);
          uint32_t pk[16];
          if (masked) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int qi = j0 + e;
              float pr = ex2(fmaf(__uint_as_float(s[e]), p.scale_log2, -sL[qi]));
              if (!row_ok || (p.causal && qbase + qi < kv_g)) pr = 0.f;
              pv[c][e] = pr;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              pv[c][e] = ex2(fmaf(__uint_as_float(s[e]), p.scale_log2, -sL[j0 + e]));
          }
#pragma unroll
          for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16(pv[c][e], pv[c][e + 1]);
          tmem_st16(tl + C::cS + pcol, pk);
        }
        tmem_st_wait();
        tc_fence_before();
      }
      __syncwarp();
      if (tracer) trace_put<kTrace>(p, t, kTrPassA1, clk());
      if (kTrace && lane == 0 && (atomicAdd(pass_done, 1u) & 7u) == 7u) trace_put<kTrace>(p, t, kTrPassALast, clk());
      if (lane == 0) {
        mbar_arrive(&bars[bPFull]);
        mbar_arrive(&qemptyQ[st]);  // this warp is done with the stage's LSE
      }
      mbar_wait(&qfullDO[st], qfd_phase[st], g);  // delta
      qfd_phase.flip(st);
      mbar_wait(&bars[bDpFull], dpf_phase, g);
      dpf_phase ^= 1;
      if (t > t_begin) {  // the previous task's dQ and dK MMAs have read the dS tile
        mbar_wait(&bars[bKDone], kd_phase, g);
        kd_phase ^= 1;
      }
      if (tracer) trace_put<kTrace>(p, t, kTrPassB0, clk());
      if (!warp_aborted(g)) {
        tc_fence_after();
        // pass B: dS = P * (dP - delta), into shared memory as [q/64][kv][64 q]:
        // the MN-major A operand of dQ = dS K and the K-major A operand of dK
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          const int j0 = 32 * half + 64 * c;
          uint8_t *rowp = sDS + (j0 >> 6) * C::kDsPanel + L * 128;
#pragma unroll
          for (int sb = 0; sb < 2; ++sb) {  // 16 columns at a time keeps register use down
            uint32_t dp[16];
            tmem_ld16(tl + C::cDP + j0 + 16 * sb, dp);
            uint32_t dk[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const int qi = j0 + 16 * sb + e;
              const float d0 = pv[c][16 * sb + e] * (__uint_as_float(dp[e]) - sDl[qi]);
              const float d1 = pv[c][16 * sb + e + 1] * (__uint_as_float(dp[e + 1]) - sDl[qi + 1]);
              dk[e >> 1] = pack_bf16(d0, d1);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int chunk = ((j0 & 63) >> 3) + 2 * sb + i;
              *reinterpret_cast<uint4 *>(rowp + ((chunk ^ (L & 7)) << 4)) =
                  make_uint4(dk[4 * i], dk[4 * i + 1], dk[4 * i + 2], dk[4 * i + 3]);
            }
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
      }
      __syncwarp();
      if (tracer) trace_put<kTrace>(p, t, kTrPassB1, clk());
      if (kTrace && lane == 0 && (atomicAdd(pass_done + 1, 1u) & 7u) == 7u) trace_put<kTrace>(p, t, kTrPassBLast, clk());
      if (lane == 0) {
        mbar_arrive(&bars[bDsFull]);
        mbar_arrive(&qemptyDO[st]);  // this warp is done with the stage's delta
      }
      st = (st + 1 == C::kStages) ? 0 : st + 1;
    }
  } else {
    // ------------------------------------------------------------ dQ reduction + epilogue
    regs_reduce();
    const int sub = warp & 3;
    const int L = sub * 32 + lane;            // Q row of dQ, KV row of dK/dV
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    const bool ordered = p.ordered != 0;
    const bool leader = threadIdx.x == kRedWarp0 * 32;
    // The turn of a task is awaited by a thread of the next warp: the leader
    // may still be in the previous task's release (its fence), and the wait
    // then overlaps it; the adds start once both are over (the named barrier).
    const bool poller = threadIdx.x == (kRedWarp0 + 1) * 32;
    constexpr int kHalfChunks = D / 8;        // 16-byte chunks per half of a dQ row
    // the atomic schedule's bulk half pays at D = 128 only (measured); at D = 64
    // every schedule adds the whole partial from registers
    constexpr bool kAtomicBulk = (D == 128);
    uint32_t dq_phase = 0, dkvf_phase = 0;
    int st = 0;
    int4 nxt = t_begin < t_end ? tasks[t_begin] : make_int4(0, 0, 0, 0);
    for (int t = t_begin; t < t_end; ++t) {
      const int4 tk = nxt;
      if (t + 1 < t_end) nxt = tasks[t + 1];
      // with cluster hand-offs the task word carries the links above a 16-bit rank
      const int bh = tk.x, kv = tk.y, q = tk.z, rank = tk.w & (p.linked ? kLinkedRankMask : kTaskRankMask);
      const int link = p.linked ? tk.w : 0;
      const bool last = tk.w & kTaskLastFlag;
      // -------- dQ partial: TMEM -> registers; tensor memory is free at once.
      mbar_wait(&bars[bDqFull], dq_phase, g);
      dq_phase ^= 1;
      if (kTrace && leader) {
        trace_put<kTrace>(p, t, kTrRedQ, clk());
        trace_put<kTrace>(p, t, kTrMeta, (long long)smid() * 65536 + slot);
      }
      float acc[D];
      const bool ok = !warp_aborted(g);
      if (ok) {
        tc_fence_after();
        // all D columns in flight at once, one wait: the dQ columns are free
        // (and the next dP^T can go) one load latency after the partial landed
        uint32_t r[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32_nowait(tl + C::cDQ + 32 * c, r[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          reg_order32(r[c]);
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[32 * c + e] = __uint_as_float(r[c][e]);
        }
        tc_fence_before();
      }
      __syncwarp();
      if (kTrace && leader) trace_put<kTrace>(p, t, kTrRedLd, clk());
      if (lane == 0) mbar_arrive(&bars[bTmemFree]);
      // The tile's turn: acquire the semaphore while the partial waits in
      // registers, so that no shared memory is held during the wait.  With
      // two chains, even ranks add into the first accumulator and odd ranks
      // into the second, each in rank order behind its own semaphore.
      const int chain = ordered ? rank % p.chains : 0, pos = ordered ? rank / p.chains : 0;
      const size_t sem_key = ((size_t)bh * p.n + q) * p.chains + chain;
      int *sem = p.sem + (p.sem_idx ? (size_t)p.sem_idx[sem_key] : sem_key * kSemStride);
      float *dst = p.dq_accum + chain * p.chain_stride + ((size_t)bh * p.n + q) * (size_t)(T * D);
      const bool first_rank = ordered && pos == 0;  // first in its chain's order: store
      if (kTrace && poller) {
        trace_put<kTrace>(p, t, kTrClkAtAcq0, clk());
        trace_put<kTrace>(p, t, kTrAcq0, (long long)globaltimer_ns());
      }
      if (poller && ordered && !*g.abort) {
        const uint64_t t0 = globaltimer_ns();
        // the time limit is checked every 64 polls: a timer read per poll
        // would stretch the gap between two polls
        if (link & kLinkTurn) {  // the predecessor runs in this cluster: its counter here
          const int from = (link >> kLinkFromShift) & 0xF;
          const uint32_t want = ++turns_seen[from];
          for (uint32_t it = 1; ld_acquire_cluster_u32(turn_count + from) < want; ++it) {
            if ((it & 63) == 0 && globaltimer_ns() - t0 > (uint64_t)p.spin_limit_ns) {
              guard_fail(g, kStatusSemTimeout);
              break;
            }
          }
        } else {
          for (uint32_t it = 1; ld_acquire_gpu(sem) != pos; ++it) {
            if ((it & 63) == 0 && globaltimer_ns() - t0 > (uint64_t)p.spin_limit_ns) {
              guard_fail(g, kStatusSemTimeout);
              break;
            }
          }
        }
      }
      // The accumulator tile is [D/4][T][4] fp32.  Ordered schedules add the
      // whole partial from registers as vector reductions (stores for the
      // first rank of a chain), so that no shared memory is held while the
      // tile's chain advances and the next tasks' Q and dO tiles load at once.  The atomic schedule,
      // whose adds never wait, stages the second half in this task's dO
      // buffer (dV, its last reader, completed before dQ) for a bulk
      // reduce-add by the TMA engine, which moves data faster than the
      // vector reductions, and adds the first half from registers meanwhile.
      if (kTrace && poller) trace_put<kTrace>(p, t, kTrAcq1, (long long)globaltimer_ns());
      named_bar(kDrainBar, kRedThreads);  // the tile's turn has come
      const bool all_regs = ordered || !kAtomicBulk;
      const int red_vecs = all_regs ? 2 * kHalfChunks : kHalfChunks;
      if (all_regs) {
        if (leader) mbar_arrive(&qemptyDO[st]);  // the dO buffer is not used for dQ
      } else {
        uint8_t *stage = smem + C::oDO + st * C::kQBytes;
        if (ok && L < T) {
#pragma unroll
          for (int c = 0; c < kHalfChunks; ++c) {
            const int a = 4 * (kHalfChunks + c);
            *reinterpret_cast<float4 *>(stage + ((size_t)c * T + L) * 16) =
                make_float4(acc[a], acc[a + 1], acc[a + 2], acc[a + 3]);
          }
        }
        fence_proxy_async_smem();  // the staged half is read next by the TMA engine
        named_bar(kDrainBar, kRedThreads);
        if (leader) {
          if (!*g.abort) {
            fence_proxy_async_global();
            bulk_reduce_add_f32(dst + (size_t)(C::kQBytes / 4), stage, C::kQBytes);
            bulk_commit();
            bulk_wait_read_all();
          }
          mbar_arrive(&qemptyDO[st]);  // the dO buffer may be refilled
        }
      }
      if (ok && L < T && !*g.abort) {
        float *row = dst + (size_t)L * 4;
        if (first_rank) {
#pragma unroll
          for (int c = 0; c < 2 * kHalfChunks; ++c)
            *reinterpret_cast<float4 *>(row + (size_t)c * T * 4) =
                make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
        } else {
          // The reductions are paced to about the rate at which the SM's path
          // to L2 accepts them.  Issued in one burst they fill the load/store
          // queue, and every shared-memory access of the other warps (mbarrier
          // waits, the softmax's loads and stores of LSE, delta and dS) then
          // waits behind them, which stalls the MMA pipeline.
#pragma unroll
          for (int c = 0; c < 2 * kHalfChunks; ++c)
            if (c < red_vecs) {
              red_add_v4(row + (size_t)c * T * 4, acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
              if (c + 1 < red_vecs) {
                if (all_regs)
                  __nanosleep(kRedPauseOrderedNs);
                else if (c % 3 == 2)
                  __nanosleep(kRedPauseAtomicNs);
              }
            }
        }
      }
      if (kTrace && leader) trace_put<kTrace>(p, t, kTrRedIssued, clk());
      if (ordered) {
        named_bar(kDrainBar, kRedThreads);  // every thread's reductions are issued
        if (kTrace && leader) trace_put<kTrace>(p, t, kTrRel0, (long long)globaltimer_ns());
        // The release is cumulative: it covers the other threads' reductions,
        // which the named barrier ordered before it.  Its fence waits until L2
        // has them, so the next rank's adds land after these.
        if (leader && !*g.abort) {
          if (link & kLinkRelease) {
            // the successor runs in this cluster: one fence releases both its
            // counter for this CTA and the semaphore
            fence_acq_rel_gpu();
            red_relaxed_cluster_u32(mapa_rank(turn_count + cluster_rank(), (link >> kLinkToShift) & 0xF), 1u);
            st_relaxed_gpu(sem, pos + 1);
          } else {
            st_release_gpu(sem, pos + 1);
          }
        }
      } else if (kTrace && leader) {
        trace_put<kTrace>(p, t, kTrRel0, (long long)globaltimer_ns());
      }
      if (kTrace && leader) trace_put<kTrace>(p, t, kTrRel1, (long long)globaltimer_ns());
      // -------- end of a KV run: dK, dV out of TMEM
      if (last) {
        mbar_wait(&bars[bDkvFull], dkvf_phase, g);
        dkvf_phase ^= 1;
        if (!warp_aborted(g)) {
          tc_fence_after();
          const int kv_g = kv * T + L;
          const bool row_ok = (L < T) && (kv_g < p.S);
          __nv_bfloat16 *dv_row = p.dv + ((size_t)bh * p.S + kv_g) * D;
          __nv_bfloat16 *dk_row = p.dk + ((size_t)bh * p.S + kv_g) * D;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t a[32], b[32];
            tmem_ld32x2(tl + C::cDV + c0, tl + C::cDK + c0, a, b);
            if (row_ok) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint4 va, vb;
                va.x = pack_bf16(__uint_as_float(a[8 * i + 0]), __uint_as_float(a[8 * i + 1]));
                va.y = pack_bf16(__uint_as_float(a[8 * i + 2]), __uint_as_float(a[8 * i + 3]));
                va.z = pack_bf16(__uint_as_float(a[8 * i + 4]), __uint_as_float(a[8 * i + 5]));
                va.w = pack_bf16(__uint_as_float(a[8 * i + 6]), __uint_as_float(a[8 * i + 7]));
                const float sc = p.scale;
                vb.x = pack_bf16(sc * __uint_as_float(b[8 * i + 0]), sc * __uint_as_float(b[8 * i + 1]));
                vb.y = pack_bf16(sc * __uint_as_float(b[8 * i + 2]), sc * __uint_as_float(b[8 * i + 3]));
                vb.z = pack_bf16(sc * __uint_as_float(b[8 * i + 4]), sc * __uint_as_float(b[8 * i + 5]));
                vb.w = pack_bf16(sc * __uint_as_float(b[8 * i + 6]), sc * __uint_as_float(b[8 * i + 7]));
                *reinterpret_cast<uint4 *>(dv_row + c0 + 8 * i) = va;
                *reinterpret_cast<uint4 *>(dk_row + c0 + 8 * i) = vb;
              }
            }
          }
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[bDkvEmpty]);
      }
      st = (st + 1 == C::kStages) ? 0 : st + 1;
    }
    if (leader && !ordered) bulk_wait_all();  // the atomic schedule's last bulk adds have landed
  }

  tc_fence_before();
  __syncthreads();
  if (p.linked) cluster_sync_all();  // no CTA leaves while a peer may still raise its counters
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// delta, lse2 (padded to n*T rows per head) and zeroing of the workspace.
template <int D>
__global__ void __launch_bounds__(256) dash_bwd_preprocess(const __nv_bfloat16 *__restrict__ o,
                                                          const __nv_bfloat16 *__restrict__ dout,
                                                          const float *__restrict__ lse, float *lse2,
                                                          float *delta, float4 *dq_accum, long long accum_vec4,
                                                          int *sem, int sem_count, int S, int rows_padded,
                                                          long long total_rows) {
  const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  for (long long i = gtid; i < accum_vec4; i += nthreads) dq_accum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = gtid; i < sem_count; i += nthreads) sem[i] = 0;
  // Each lane reads 16 bytes (8 elements) of a row of O and of dO, so a row is
  // D / 8 lanes and one load instruction covers 32 / (D / 8) rows; kU of them
  // per round keep 2 x kU x 16 bytes in flight per lane, which the kernel, bound
  // by the bytes each SM has in flight, needs to approach HBM bandwidth.
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerLoad = 32 / kLanesPerRow;
  constexpr int kU = 4;
  constexpr int kRowsPerRound = kRowsPerLoad * kU;
  const int lane = threadIdx.x & 31, sub = lane / kLanesPerRow, li = lane % kLanesPerRow;
  const long long gwarp = gtid >> 5, nwarps = nthreads >> 5;
  for (long long row0 = gwarp * kRowsPerRound; row0 < total_rows; row0 += nwarps * kRowsPerRound) {
    uint4 a[kU], b[kU];
    float l2[kU];
    bool valid[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const long long row = row0 + u * kRowsPerLoad + sub;
      const long long bh = row / rows_padded;
      const int r = (int)(row - bh * rows_padded);
      valid[u] = row < total_rows && r < S;
      a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
      l2[u] = __int_as_float(0x7f800000);  // +inf: P = 0 for padded rows
      if (valid[u]) {
        const size_t base = ((size_t)bh * S + r) * D + li * 8;
        a[u] = *reinterpret_cast<const uint4 *>(o + base);
        b[u] = *reinterpret_cast<const uint4 *>(dout + base);
        if (li == 0) l2[u] = lse[(size_t)bh * S + r] * 1.4426950408889634f;
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a[u]);
      const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&b[u]);
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fa = __bfloat1622float2(pa[i]), fb = __bfloat1622float2(pb[i]);
        sum = fmaf(fa.x, fb.x, sum);
        sum = fmaf(fa.y, fb.y, sum);
      }
#pragma unroll
      for (int off = kLanesPerRow / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      const long long row = row0 + u * kRowsPerLoad + sub;
      if (li == 0 && row < total_rows) {
        delta[row] = sum;
        lse2[row] = l2[u];
      }
    }
  }
}

// dQ = bf16(scale * accumulator); optionally the unscaled fp32 accumulator in
// [BH][S][D].  With two chains the accumulator is the sum of the two chains'
// copies, chain 0 + chain 1, in that order.
template <int D, int T>
__global__ void __launch_bounds__(256) dash_bwd_convert(const float *__restrict__ acc, int chains,
                                                       long long chain_stride, __nv_bfloat16 *dq,
                                                       float *acc_out, float scale, int S, int n,
                                                       long long total_rows) {
  const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  // Work item i = (group of 4 column chunks, row), rows fastest: a warp reads
  // 32 consecutive rows of a chunk, which are contiguous in the accumulator's
  // [D/4][T][4] tile layout, and each thread writes 32 contiguous bytes of dQ.
  constexpr int kGroups = D / 16;
  const long long total = total_rows * kGroups;
  for (long long i = gtid; i < total; i += nthreads) {
    const int g = (int)(i / total_rows);
    const long long rowg = i - (long long)g * total_rows;  // bh * S + row
    const long long bh = rowg / S;
    const int row = (int)(rowg - bh * S);
    const int qt = row / T, r = row - qt * T;
    const size_t tile = ((size_t)bh * n + qt) * (size_t)(T * D);
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const size_t at = tile + ((size_t)(4 * g + k) * T + r) * 4;
      v[k] = *reinterpret_cast<const float4 *>(acc + at);
      if (chains > 1) {
        const float4 w = *reinterpret_cast<const float4 *>(acc + chain_stride + at);
        v[k] = make_float4(v[k].x + w.x, v[k].y + w.y, v[k].z + w.z, v[k].w + w.w);
      }
    }
    uint4 o0, o1;
    o0.x = pack_bf16(scale * v[0].x, scale * v[0].y);
    o0.y = pack_bf16(scale * v[0].z, scale * v[0].w);
    o0.z = pack_bf16(scale * v[1].x, scale * v[1].y);
    o0.w = pack_bf16(scale * v[1].z, scale * v[1].w);
    o1.x = pack_bf16(scale * v[2].x, scale * v[2].y);
    o1.y = pack_bf16(scale * v[2].z, scale * v[2].w);
    o1.z = pack_bf16(scale * v[3].x, scale * v[3].y);
    o1.w = pack_bf16(scale * v[3].z, scale * v[3].w);
    uint4 *out = reinterpret_cast<uint4 *>(dq + (size_t)rowg * D + 16 * g);
    out[0] = o0;
    out[1] = o1;
    if (acc_out) {
#pragma unroll
      for (int k = 0; k < 4; ++k) *reinterpret_cast<float4 *>(acc_out + (size_t)rowg * D + 16 * g + 4 * k) = v[k];
    }
  }
}

template <int D, int T, bool kTrace>
cudaError_t launch_main_t(const BwdMaps &maps, const BwdMainParams &p, int num_ctas, cudaStream_t stream,
                          int cluster) {
  using C = BwdCfg<D, T>;
  auto kfn = dash_bwd_main<D, T, kTrace>;
  // The setmaxnreg split above assumes the CTA is launched with exactly
  // kRegsLaunch registers per thread; with fewer, an increase could wait forever.
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kfn);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
  const int smem = C::kSmemBytes > (uint32_t)kMinSmemOneCtaPerSm ? (int)C::kSmemBytes : kMinSmemOneCtaPerSm;
  e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: semaphore waits cannot starve
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster > 1) {
    if (num_ctas % cluster != 0 || cluster > kMaxClusterLinks) return cudaErrorInvalidValue;
    if (cluster > 8 && (e = cudaFuncSetAttribute(kfn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) !=
                           cudaSuccess)
      return e;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, kfn, maps.q, maps.k, maps.v, maps.dout, p);
}

template <int D, int T>
int cluster_size_t(int num_ctas) {
  using C = BwdCfg<D, T>;
  auto kfn = dash_bwd_main<D, T, false>;
  const int smem = C::kSmemBytes > (uint32_t)kMinSmemOneCtaPerSm ? (int)C::kSmemBytes : kMinSmemOneCtaPerSm;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 1;
  for (int cl : {16, 8, 4, 2}) {
    if (num_ctas % cl != 0) continue;
    if (cl > 8 && cudaFuncSetAttribute(kfn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      continue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kfn, &cfg) != cudaSuccess) {
      cudaGetLastError();  // clear the error; try a smaller size
      continue;
    }
    if ((long long)active * cl >= num_ctas) return cl;
  }
  return 1;
}

}  // namespace

size_t bwd_main_smem_bytes(int D, int T) {
  if (D == 64 && T == 64) return BwdCfg<64, 64>::kSmemBytes;
  if (D == 64 && T == 128) return BwdCfg<64, 128>::kSmemBytes;
  if (D == 128 && T == 64) return BwdCfg<128, 64>::kSmemBytes;
  if (D == 128 && T == 128) return BwdCfg<128, 128>::kSmemBytes;
  return 0;
}

cudaError_t launch_bwd_preprocess(const BwdPreParams &a, int num_sms, cudaStream_t stream) {
  const int blocks = num_sms * 8;  // 2048 threads per SM
  if (a.D == 64)
    dash_bwd_preprocess<64><<<blocks, 256, 0, stream>>>(
        (const __nv_bfloat16 *)a.o, (const __nv_bfloat16 *)a.dout, a.lse, a.lse2, a.delta, (float4 *)a.dq_accum,
        a.accum_floats / 4, a.sem, a.sem_count, a.S, a.rows_padded, a.total_rows);
  else
    dash_bwd_preprocess<128><<<blocks, 256, 0, stream>>>(
        (const __nv_bfloat16 *)a.o, (const __nv_bfloat16 *)a.dout, a.lse, a.lse2, a.delta, (float4 *)a.dq_accum,
        a.accum_floats / 4, a.sem, a.sem_count, a.S, a.rows_padded, a.total_rows);
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(int D, int T, const BwdMaps &maps, const BwdMainParams &p, int num_ctas,
                            cudaStream_t stream, int cluster) {
  if (p.trace) {  // the traced kernel exists for the 128-row tiles only
    if (D == 64 && T == 128) return launch_main_t<64, 128, true>(maps, p, num_ctas, stream, cluster);
    if (D == 128 && T == 128) return launch_main_t<128, 128, true>(maps, p, num_ctas, stream, cluster);
    return cudaErrorNotSupported;
  }
  if (D == 64 && T == 64) return launch_main_t<64, 64, false>(maps, p, num_ctas, stream, cluster);
  if (D == 64 && T == 128) return launch_main_t<64, 128, false>(maps, p, num_ctas, stream, cluster);
  if (D == 128 && T == 64) return launch_main_t<128, 64, false>(maps, p, num_ctas, stream, cluster);
  if (D == 128 && T == 128) return launch_main_t<128, 128, false>(maps, p, num_ctas, stream, cluster);
  return cudaErrorInvalidValue;
}

int bwd_main_cluster_size(int D, int T, int num_ctas) {
  if (D == 64 && T == 64) return cluster_size_t<64, 64>(num_ctas);
  if (D == 64 && T == 128) return cluster_size_t<64, 128>(num_ctas);
  if (D == 128 && T == 64) return cluster_size_t<128, 64>(num_ctas);
  if (D == 128 && T == 128) return cluster_size_t<128, 128>(num_ctas);
  return 1;
}

cudaError_t launch_bwd_convert(int D, int T, const float *acc, int chains, long long chain_stride, void *dq,
                               float *acc_out, float scale, int BH, int S, int n, int num_sms, cudaStream_t stream) {
  const long long total = (long long)BH * S;  // rows
  const int blocks = num_sms * 8;  // 2048 threads per SM
  auto *out = (__nv_bfloat16 *)dq;
  if (D == 64 && T == 64)
    dash_bwd_convert<64, 64><<<blocks, 256, 0, stream>>>(acc, chains, chain_stride, out, acc_out, scale, S, n, total);
  else if (D == 64 && T == 128)
    dash_bwd_convert<64, 128><<<blocks, 256, 0, stream>>>(acc, chains, chain_stride, out, acc_out, scale, S, n, total);
  else if (D == 128 && T == 64)
    dash_bwd_convert<128, 64><<<blocks, 256, 0, stream>>>(acc, chains, chain_stride, out, acc_out, scale, S, n, total);
  else
    dash_bwd_convert<128, 128><<<blocks, 256, 0, stream>>>(acc, chains, chain_stride, out, acc_out, scale, S, n, total);
  return cudaGetLastError();
}

}  // namespace dash
