// Interface between the host API (api.cpp) and the CUDA kernels (bwd.cu, fwd.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace dash {

// Device status word values (first error wins).
constexpr int kStatusMbarTimeout = 1;     // an mbarrier wait ran out
constexpr int kStatusSemTimeout = 2;      // a dQ semaphore wait ran out
// dQ semaphores sit one 32-byte L2 sector apart: neighbouring tiles' semaphores
// are polled and released by different CTAs at the same time, and sharing a
// sector serialises those accesses at the L2 slice.
constexpr int kSemStride = 8;
constexpr int kStatusSmemMisaligned = 3;  // dynamic shared memory not 1024-byte aligned

// Dynamic shared memory requested by every kernel that allocates all 512
// tensor-memory columns: two such CTAs never fit on one SM, so no CTA can sit
// in tcgen05.alloc behind a CTA that is waiting on it.
constexpr int kMinSmemOneCtaPerSm = 120 * 1024;

constexpr int kTaskFirstFlag = 1 << 28;
constexpr int kTaskLastFlag = 1 << 29;
constexpr int kTaskRankMask = (1 << 24) - 1;

struct BwdMaps {
  CUtensorMap q, k, v, dout;  // 3-D [BH][S][D] bf16, 128-byte swizzle; Q/dO box T rows, K/V box 128 rows
};

struct BwdMainParams {
  const int4 *tasks;     // {bh, kv, q, rank | flags}
  const int *cta_off;    // gridDim.x + 1
  const float *lse2;     // [BH][n*T]  LSE * log2(e), +inf on padded rows
  const float *delta;    // [BH][n*T]  rowsum(dO * O), 0 on padded rows
  float *dq_accum;       // [chains][BH][n][D/4][T][4] fp32
  int *sem;              // [BH][n][chains], kSemStride ints apart
  __nv_bfloat16 *dk;     // [BH][S][D]
  __nv_bfloat16 *dv;     // [BH][S][D]
  int *status;           // device status word
  int S, n;
  float scale;           // softmax scale (applied to dK in the epilogue)
  float scale_log2;      // scale * log2(e)
  int causal;
  int ordered;           // 0: atomic (unordered) reduction
  long long spin_limit_ns;
  int chains;            // ordered schedules: 1, or 2 (ranks split by parity, one accumulator each)
  long long chain_stride;  // floats between the chains' accumulators
  long long *trace = nullptr;  // optional [n_tasks][kTraceSlots] phase stamps (traced kernel), else null
  // Die-aware placement (optional): the CTA on SM s runs slot slot_of_smid[s]
  // (-1: none; the launch then has one CTA per SM), and the semaphore of
  // (head, tile, chain) k sits at sem + sem_idx[k] instead of k * kSemStride.
  const int *slot_of_smid = nullptr;
  int n_smid = 0;
  const int *sem_idx = nullptr;
  // Cluster hand-offs (with a cluster launch): the task words carry the links
  // of cluster_links (schedule.h) above a 16-bit rank; a linked rank takes its
  // turn from a counter in its own shared memory that the predecessor's CTA
  // raises.
  int linked = 0;
};
constexpr int kMaxClusterLinks = 16;  // cluster sizes up to 16: one counter per CTA of the cluster
// Link bits of a task word (host cluster_links and the device table of a linked launch)
constexpr int32_t kLinkedRankMask = 0xFFFF;           // ranks below 2^16 leave room for the links
constexpr int kLinkFromShift = 16;                    // predecessor's rank in the cluster (4 bits)
constexpr int kLinkToShift = 20;                      // successor's rank in the cluster (4 bits)
constexpr int32_t kLinkTurn = 1 << 30;                // the turn comes from the predecessor's counter
constexpr int32_t kLinkRelease = (int32_t)(1u << 31);  // the release also raises the successor's counter

// Phase stamps of the traced main kernel, one row of kTraceSlots int64 per
// task (indexed by the task's position in the table).  "clk" stamps are the
// SM's clock64, "ns" stamps the global timer.
enum TraceSlot {
  kTrMmaDp = 0,      // clk: MMA warp starts dP^T (its waits are over)
  kTrMmaDv = 1,      // clk: MMA warp has P and starts dV
  kTrMmaDq = 2,      // clk: MMA warp has dS and starts dQ
  kTrMmaEnd = 3,     // clk: MMA warp has issued the task's last MMA and commits
  kTrPassA0 = 4,     // clk: softmax warp 4 has S^T (pass A starts)
  kTrPassA1 = 5,     // clk: pass A done
  kTrPassB0 = 6,     // clk: pass B starts (dP^T landed, dS buffer free)
  kTrPassB1 = 7,     // clk: pass B done
  kTrRedQ = 8,       // clk: reduction leader sees the dQ partial in tensor memory
  kTrRedLd = 9,      // clk: the partial is in registers, tensor memory released
  kTrAcq0 = 10,      // ns: the turn's waiter (a lane of the second reduction warp) starts waiting
  kTrAcq1 = 11,      // ns: the tile's turn has come (semaphore acquired; atomic: at once)
  kTrRedIssued = 12, // clk: the leader's own reductions are issued
  kTrRel0 = 13,      // ns: every reduction of the task is issued; the release of rank + 1 starts
  kTrClkAtAcq0 = 14, // clk read next to kTrAcq0, to put both clocks on one axis
  kTrMeta = 15,      // smid * 65536 + the CTA's slot (its task list)
  kTrRel1 = 16,      // ns: the release store has returned (its fence is done)
  kTrPassALast = 17, // clk: the last of the eight softmax warps is done with pass A
  kTrPassBLast = 18, // clk: the last of the eight softmax warps is done with pass B
  kTrMmaDvOut = 19,  // clk: MMA warp has issued dV (and the next S^T, when it goes early)
  kTrMmaDsSeen = 20, // clk: MMA warp's wait for dS has returned
  kTraceSlots = 21
};

struct BwdPreParams {
  const void *o, *dout;  // bf16 [BH][S][D]
  const float *lse;      // [BH][S]
  float *lse2, *delta;   // [BH][n*T]
  float *dq_accum;
  long long accum_floats;
  int *sem;
  int sem_count;
  int S, D, rows_padded;
  long long total_rows;  // BH * n * T
};

struct FwdParams {
  __nv_bfloat16 *o;  // [BH][S][D]
  float *lse;        // [BH][S]
  int *status;
  int S;
  float scale_log2;
  int causal;
  long long spin_limit_ns;
};

size_t bwd_main_smem_bytes(int D, int T);
cudaError_t launch_bwd_preprocess(const BwdPreParams &a, int num_sms, cudaStream_t stream);
// cluster = 1: plain cooperative launch; 2..16: thread-block clusters of that
// size (then p.linked may be set).
cudaError_t launch_bwd_main(int D, int T, const BwdMaps &maps, const BwdMainParams &p, int num_ctas,
                            cudaStream_t stream, int cluster = 1);
// The largest cluster size among 16, 8, 4, 2 that divides num_ctas and lets
// every CTA of the launch be resident at once; 1 if none.
int bwd_main_cluster_size(int D, int T, int num_ctas);
cudaError_t launch_bwd_convert(int D, int T, const float *acc, int chains, long long chain_stride, void *dq,
                               float *acc_out, float scale, int BH,
                               int S, int n, int num_sms, cudaStream_t stream);

// Latency probe of the die-aware placement: lat[cta][line] for one CTA per SM
// over n_lines 128-byte lines of `pool` (which it overwrites), smid_out[cta].
cudaError_t launch_probe_homes(unsigned *pool, int n_lines, unsigned *lat, int *smid_out, int num_sms,
                               cudaStream_t stream);

// CTA-pair forward for D = 128 (tcgen05 cta_group::2): Q and V maps with
// 128-row boxes, K with 64-row boxes (each CTA of a pair loads half a tile).
cudaError_t launch_fwd_pair(const CUtensorMap &q, const CUtensorMap &k_half_rows, const CUtensorMap &v,
                            const FwdParams &p, int BH, cudaStream_t stream);

// Forward: Q/K/V maps with 128-row boxes.
cudaError_t launch_fwd(int D, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                       const FwdParams &p, int BH, cudaStream_t stream);

}  // namespace dash
