// Softmax attention forward for sm_103a (produces O and LSE for the backward).
//
// One CTA per (128-row Q tile, head).  Two passes over the KV tiles: pass 1
// forms S = Q K^T and the exact row statistics (max and sum of exponentials,
// kept in the log2 domain), pass 2 forms S again, P = exp(scale*S - LSE)
// exactly normalised, and accumulates O = P V in tensor memory.  The second
// S costs one extra matmul per tile, which keeps the kernel free of output
// rescaling; the forward sits outside the backward's timed path.
//
// Roles (256 threads): warp 0 TMA, warp 1 tensor memory + MMA issue (one
// lane), warps 4-7 softmax with one thread per Q row (TMEM lane).  Tensor
// memory: S double-buffered at columns 0 and 128 (P overwrites the first 64
// columns of its S buffer as packed bf16), O at column 256.
#include <cuda_runtime.h>

#include "kernels.h"
#include "sm103.cuh"

namespace dash {

using namespace dev;

namespace {

constexpr int kThreads = 256;

template <int D>
struct FwdCfg {
  static constexpr int kPanels = D / 64;
  static constexpr uint32_t kTile = 128 * D * 2;
  static constexpr uint32_t kPanel = 128 * 128;
  static constexpr uint32_t oQ = 0;
  static constexpr uint32_t oK = kTile;
  static constexpr uint32_t oV = oK + 2 * kTile;
  static constexpr uint32_t oBAR = oV + 2 * kTile;
  static constexpr int kNumBars = 13;
  static constexpr uint32_t oMISC = oBAR + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = oMISC + 16;
  static constexpr uint32_t cO = 256;
};

enum { fQFull = 0, fKvFull0 = 1, fKvEmpty0 = 3, fSFull0 = 5, fSEmpty0 = 7, fPFull0 = 9, fOFull = 11, fFinal = 12 };

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dash_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::oBAR);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::oMISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::oMISC + 4);

  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kStatusSmemMisaligned);
    return;
  }
  const int qt = blockIdx.x, bh = blockIdx.y;
  const int nblk = (p.S + 127) / 128;
  const int nkv = p.causal ? min(qt + 1, nblk) : nblk;
  const int iters = 2 * nkv;

  if (threadIdx.x == 0) {
    mbar_init(&bars[fQFull], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[fKvFull0 + i], 1);
      mbar_init(&bars[fKvEmpty0 + i], 1);
      mbar_init(&bars[fSFull0 + i], 1);
      mbar_init(&bars[fSEmpty0 + i], 4);
      mbar_init(&bars[fPFull0 + i], 4);
    }
    mbar_init(&bars[fOFull], 1);
    mbar_init(&bars[fFinal], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Guard g{abort_flag, p.status, (uint64_t)p.spin_limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(&bars[fQFull], C::kTile);
      for (int pn = 0; pn < C::kPanels; ++pn)
        tma_load_3d(smem + C::oQ + pn * C::kPanel, &tmQ, &bars[fQFull], pn * 64, qt * 128, bh);
      uint32_t last_fill[2] = {0, 0};
      bool used[2] = {false, false};
      for (int it = 0; it < iters; ++it) {
        const int st = it & 1, pass = it / nkv, j = it % nkv;
        if (it >= 2) mbar_wait(&bars[fKvEmpty0 + st], ((it >> 1) - 1) & 1, g);
        if (*g.abort) continue;
        const uint32_t bytes = C::kTile * (pass ? 2 : 1);
        mbar_arrive_expect_tx(&bars[fKvFull0 + st], bytes);
        for (int pn = 0; pn < C::kPanels; ++pn) {
          tma_load_3d(smem + C::oK + st * C::kTile + pn * C::kPanel, &tmK, &bars[fKvFull0 + st], pn * 64, j * 128,
                      bh);
          if (pass)
            tma_load_3d(smem + C::oV + st * C::kTile + pn * C::kPanel, &tmV, &bars[fKvFull0 + st], pn * 64,
                        j * 128, bh);
        }
        last_fill[st] = (it >> 1) & 1;
        used[st] = true;
      }
      mbar_drain(&bars[fQFull], 0, g.limit_ns);
      for (int s = 0; s < 2; ++s)
        if (used[s]) mbar_drain(&bars[fKvFull0 + s], last_fill[s], g.limit_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idO = idesc_bf16(128, D, 0, 1);
      const uint32_t sQ = smem_u32(smem + C::oQ);
      bool issued = false;
      uint32_t pf_phase[2] = {0, 0};  // P-ready barriers only see second-pass iterations
      auto do_pv = [&](int i) {
        const int b = i & 1, jj = i % nkv;
        mbar_wait(&bars[fPFull0 + b], pf_phase[b], g);
        pf_phase[b] ^= 1;
        if (*g.abort) return;
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + C::oV + b * C::kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + C::cO, tmem + b * 128 + kk * 8, sw128_desc(sV + kk * 2048, C::kPanel, 1024), idO,
                 (jj > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&bars[fKvEmpty0 + b]);
      };
      mbar_wait(&bars[fQFull], 0, g);
      for (int it = 0; it < iters; ++it) {
        const int st = it & 1, pass = it / nkv;
        mbar_wait(&bars[fKvFull0 + st], (it >> 1) & 1, g);
        if (it >= 2) mbar_wait(&bars[fSEmpty0 + st], ((it >> 1) - 1) & 1, g);
        if (!*g.abort) {
          tc_fence_after();
          const uint32_t sK = smem_u32(smem + C::oK + st * C::kTile);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kPanel + (kk & 3) * 32;
            mma_ss(tmem + st * 128, sw128_desc(sQ + off, 16, 1024), sw128_desc(sK + off, 16, 1024), idS, kk > 0);
          }
          tc_commit(&bars[fSFull0 + st]);
          if (pass == 0) tc_commit(&bars[fKvEmpty0 + st]);
          issued = true;
        }
        if (it >= 1 && (it - 1) / nkv == 1) do_pv(it - 1);
      }
      do_pv(iters - 1);
      if (!*g.abort) tc_commit(&bars[fOFull]);
      if (issued) {  // every MMA has completed before tensor memory is released
        tc_commit(&bars[fFinal]);
        mbar_drain(&bars[fFinal], 0, g.limit_ns);
      }
    }
  } else if (warp >= 4) {
    const int sub = warp & 3;
    const int L = sub * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    const int q_g = qt * 128 + L;
    float m = -INFINITY, l = 0.f;
    for (int it = 0; it < iters; ++it) {
      const int b = it & 1, pass = it / nkv, j = it % nkv;
      mbar_wait(&bars[fSFull0 + b], (it >> 1) & 1, g);
      if (!warp_aborted(g)) {
        tc_fence_after();
        if (pass == 1 && it == nkv) {
          // row statistics are final: LSE in the log2 domain
          m = (l > 0.f) ? m + log2f(l) : INFINITY;
        }
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t s[32];
          tmem_ld32(tl + b * 128 + c0, s);
          float x[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int kv_g = j * 128 + c0 + e;
            const bool masked = (kv_g >= p.S) || (p.causal && kv_g > q_g);
            x[e] = masked ? -INFINITY : __uint_as_float(s[e]) * p.scale_log2;
          }
          if (pass == 0) {
            float mx = m;
#pragma unroll
            for (int e = 0; e < 32; ++e) mx = fmaxf(mx, x[e]);
            if (mx != -INFINITY) {
              float sum = 0.f;
#pragma unroll
              for (int e = 0; e < 32; ++e) sum += ex2(x[e] - mx);
              l = l * ex2(m - mx) + sum;
              m = mx;
            }
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16(ex2(x[e] - m), ex2(x[e + 1] - m));
            tmem_st16(tl + b * 128 + (c0 >> 1), pk);
          }
        }
        if (pass == 1) tmem_st_wait();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) {
        if (pass == 1) mbar_arrive(&bars[fPFull0 + b]);
        mbar_arrive(&bars[fSEmpty0 + b]);
      }
    }
    mbar_wait(&bars[fOFull], 0, g);
    if (!warp_aborted(g)) {
      tc_fence_after();
      const bool row_ok = q_g < p.S;
      __nv_bfloat16 *orow = p.o + ((size_t)bh * p.S + q_g) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tl + C::cO + c0, r);
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(r[8 * i + 0]), __uint_as_float(r[8 * i + 1]));
            v.y = pack_bf16(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3]));
            v.z = pack_bf16(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5]));
            v.w = pack_bf16(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7]));
            *reinterpret_cast<uint4 *>(orow + c0 + 8 * i) = v;
          }
        }
      }
      if (row_ok) p.lse[(size_t)bh * p.S + q_g] = m * 0.6931471805599453f;
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_fwd_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v, const FwdParams &p,
                         int BH, cudaStream_t stream) {
  using C = FwdCfg<D>;
  auto kfn = dash_fwd_kernel<D>;
  const int smem = C::kSmemBytes > (uint32_t)kMinSmemOneCtaPerSm ? (int)C::kSmemBytes : kMinSmemOneCtaPerSm;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.S + 127) / 128, BH);
  kfn<<<grid, kThreads, smem, stream>>>(q, k, v, p);
  return cudaGetLastError();
}

// ------------------------------------------------ CTA-pair forward, D = 128
// A cluster of two CTAs takes two adjacent 128-row Q tiles of a head (CTA r:
// Q tile 2p + r).  The pair's first CTA issues every MMA as an M = 256 pair
// MMA (tcgen05 cta_group::2): S = Q K^T with each CTA's own Q rows as A and
// the KV tile's rows split between the CTAs as B (CTA r loads rows 64r..),
// then O += P V with each CTA's P read from its own tensor memory and V's
// columns split between the CTAs (CTA r loads columns 64r..).  So each CTA
// loads half of every K and V tile, and the MMAs read half of each B operand
// from each CTA's shared memory.  Commits arrive on both CTAs' barriers.  The
// second CTA forwards the landing of its tiles and its softmax warps'
// progress to the first CTA's barriers with remote arrivals.  The softmax is
// that of dash_fwd_kernel, on each CTA's own 128 rows.
namespace pairfwd {
constexpr int kD = 128;
constexpr uint32_t kQTile = 128 * kD * 2;   // two 64-column panels of 128 rows
constexpr uint32_t kQPanel = 128 * 128;
constexpr uint32_t kKHalf = 64 * kD * 2;    // 64 KV rows x D: two panels of 64 rows
constexpr uint32_t kKPanel = 64 * 128;
constexpr uint32_t kVHalf = 128 * 64 * 2;   // 128 KV rows x 64 columns: one panel
constexpr uint32_t oQ = 0;
constexpr uint32_t oK = kQTile;             // two stages
constexpr uint32_t oV = oK + 2 * kKHalf;    // two stages
constexpr uint32_t oBAR = oV + 2 * kVHalf;
enum {
  pQFull = 0, pKvFull0 = 1, pPeerQ = 3, pPeerKv0 = 4, pSFull0 = 6, pSEmpty0 = 8, pPFull0 = 10, pKvEmpty0 = 12,
  pOFull = 14, pFinal = 15, pNumBars = 16
};
constexpr uint32_t oMISC = oBAR + pNumBars * 8;
constexpr uint32_t kSmemBytes = oMISC + 16;
constexpr uint32_t cO = 256;
}  // namespace pairfwd

__global__ void __launch_bounds__(kThreads, 1)
    dash_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKh,
                         const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using namespace pairfwd;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + oBAR);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + oMISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + oMISC + 4);

  if ((smem_u32(smem) & 1023u) != 0) {  // the same in both CTAs of the pair, which both return
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kStatusSmemMisaligned);
    return;
  }
  const uint32_t rank = cluster_rank();  // 0: the CTA that issues the pair's MMAs
  const int pair = blockIdx.x >> 1, bh = blockIdx.y;
  const int qt = 2 * pair + (int)rank;
  const int nblk = (p.S + 127) / 128;
  const int nkv = p.causal ? min(2 * pair + 2, nblk) : nblk;  // KV tiles of the pair's later Q tile
  const int iters = 2 * nkv;

  if (threadIdx.x == 0) {
    mbar_init(&bars[pQFull], 1);
    mbar_init(&bars[pPeerQ], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[pKvFull0 + i], 1);
      mbar_init(&bars[pPeerKv0 + i], 1);
      mbar_init(&bars[pSFull0 + i], 1);
      mbar_init(&bars[pSEmpty0 + i], 8);  // four softmax warps in each CTA
      mbar_init(&bars[pPFull0 + i], 8);
      mbar_init(&bars[pKvEmpty0 + i], 1);
    }
    mbar_init(&bars[pOFull], 1);
    mbar_init(&bars[pFinal], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers and tensor memory are ready
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Guard g{abort_flag, p.status, (uint64_t)p.spin_limit_ns};
  const uint32_t lead_bars = mapa_rank(bars, 0);  // the first CTA's barriers
  auto at_lead = [&](int idx) { return lead_bars + (uint32_t)idx * 8u; };

  if (warp == 0) {
    if (lane == 0) {
      // own Q tile; own half of each K tile (rows 64 * rank) and V tile (columns 64 * rank)
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmKh);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(&bars[pQFull], kQTile);
      for (int pn = 0; pn < 2; ++pn)
        tma_load_3d(smem + oQ + pn * kQPanel, &tmQ, &bars[pQFull], pn * 64, qt * 128, bh);
      uint32_t last_fill[2] = {0, 0};
      bool used[2] = {false, false};
      for (int it = 0; it < iters; ++it) {
        const int st = it & 1, pass = it / nkv, j = it % nkv;
        if (it >= 2) mbar_wait_cluster(&bars[pKvEmpty0 + st], ((it >> 1) - 1) & 1, g);
        if (*g.abort) continue;
        mbar_arrive_expect_tx(&bars[pKvFull0 + st], kKHalf + (pass ? kVHalf : 0u));
        for (int pn = 0; pn < 2; ++pn)
          tma_load_3d(smem + oK + st * kKHalf + pn * kKPanel, &tmKh, &bars[pKvFull0 + st], pn * 64,
                      j * 128 + 64 * (int)rank, bh);
        if (pass) tma_load_3d(smem + oV + st * kVHalf, &tmV, &bars[pKvFull0 + st], 64 * (int)rank, j * 128, bh);
        last_fill[st] = (it >> 1) & 1;
        used[st] = true;
      }
      mbar_drain(&bars[pQFull], 0, g.limit_ns);
      for (int s = 0; s < 2; ++s)
        if (used[s]) mbar_drain(&bars[pKvFull0 + s], last_fill[s], g.limit_ns);
    }
  } else if (warp == 2) {
    if (lane == 0 && rank == 1) {
      // the second CTA tells the first one when its tiles have landed
      if (mbar_wait(&bars[pQFull], 0, g)) mbar_arrive_cluster(at_lead(pPeerQ));
      for (int it = 0; it < iters; ++it) {
        const int st = it & 1;
        if (mbar_wait(&bars[pKvFull0 + st], (it >> 1) & 1, g)) mbar_arrive_cluster(at_lead(pPeerKv0 + st));
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idS = idesc_bf16(256, 128, 0, 0);  // S: Q rows of both CTAs x 128 KV columns
      constexpr uint32_t idO = idesc_bf16(256, kD, 0, 1);   // O: P from tensor memory, V MN-major
      const uint32_t sQ = smem_u32(smem + oQ);
      uint32_t pf_phase[2] = {0, 0};
      auto do_pv = [&](int i) {
        const int b = i & 1, jj = i % nkv;
        mbar_wait_cluster(&bars[pPFull0 + b], pf_phase[b], g);
        pf_phase[b] ^= 1;
        if (*g.abort) return;
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + oV + b * kVHalf);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_pair(tmem + cO, tmem + b * 128 + kk * 8, sw128_desc(sV + kk * 2048, kVHalf, 1024), idO,
                      (jj > 0 || kk > 0) ? 1u : 0u);
        tc_commit_pair(&bars[pKvEmpty0 + b]);
      };
      mbar_wait(&bars[pQFull], 0, g);
      mbar_wait_cluster(&bars[pPeerQ], 0, g);
      for (int it = 0; it < iters; ++it) {
        const int st = it & 1, pass = it / nkv;
        mbar_wait(&bars[pKvFull0 + st], (it >> 1) & 1, g);
        mbar_wait_cluster(&bars[pPeerKv0 + st], (it >> 1) & 1, g);
        if (it >= 2) mbar_wait_cluster(&bars[pSEmpty0 + st], ((it >> 1) - 1) & 1, g);
        if (!*g.abort) {
          tc_fence_after();
          const uint32_t sK = smem_u32(smem + oK + st * kKHalf);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t offq = (kk >> 2) * kQPanel + (kk & 3) * 32;
            const uint32_t offk = (kk >> 2) * kKPanel + (kk & 3) * 32;
            mma_ss_pair(tmem + st * 128, sw128_desc(sQ + offq, 16, 1024), sw128_desc(sK + offk, 16, 1024), idS,
                        kk > 0);
          }
          tc_commit_pair(&bars[pSFull0 + st]);
          if (pass == 0) tc_commit_pair(&bars[pKvEmpty0 + st]);
        }
        if (it >= 1 && (it - 1) / nkv == 1) do_pv(it - 1);
      }
      do_pv(iters - 1);
      if (!*g.abort) tc_commit_pair(&bars[pOFull]);
      tc_commit_pair(&bars[pFinal]);  // arrives once every MMA issued so far has completed (at once if none)
    }
  } else if (warp >= 4) {
    const int sub = warp & 3;
    const int L = sub * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    const int q_g = qt * 128 + L;
    float m = -INFINITY, l = 0.f;
    for (int it = 0; it < iters; ++it) {
      const int b = it & 1, pass = it / nkv, j = it % nkv;
      mbar_wait_cluster(&bars[pSFull0 + b], (it >> 1) & 1, g);
      if (!warp_aborted(g)) {
        tc_fence_after();
        if (pass == 1 && it == nkv) m = (l > 0.f) ? m + log2f(l) : INFINITY;  // LSE in the log2 domain
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t s[32];
          tmem_ld32(tl + b * 128 + c0, s);
          float x[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int kv_g = j * 128 + c0 + e;
            const bool masked = (kv_g >= p.S) || (p.causal && kv_g > q_g);
            x[e] = masked ? -INFINITY : __uint_as_float(s[e]) * p.scale_log2;
          }
          if (pass == 0) {
            float mx = m;
#pragma unroll
            for (int e = 0; e < 32; ++e) mx = fmaxf(mx, x[e]);
            if (mx != -INFINITY) {
              float sum = 0.f;
#pragma unroll
              for (int e = 0; e < 32; ++e) sum += ex2(x[e] - mx);
              l = l * ex2(m - mx) + sum;
              m = mx;
            }
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16(ex2(x[e] - m), ex2(x[e + 1] - m));
            tmem_st16(tl + b * 128 + (c0 >> 1), pk);
          }
        }
        if (pass == 1) tmem_st_wait();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) {
        if (pass == 1) mbar_arrive_cluster(at_lead(pPFull0 + b));
        mbar_arrive_cluster(at_lead(pSEmpty0 + b));
      }
    }
    mbar_wait_cluster(&bars[pOFull], 0, g);
    if (!warp_aborted(g)) {
      tc_fence_after();
      const bool row_ok = q_g < p.S;
      __nv_bfloat16 *orow = p.o + ((size_t)bh * p.S + q_g) * kD;
#pragma unroll 1
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tl + cO + c0, r);
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(r[8 * i + 0]), __uint_as_float(r[8 * i + 1]));
            v.y = pack_bf16(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3]));
            v.z = pack_bf16(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5]));
            v.w = pack_bf16(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7]));
            *reinterpret_cast<uint4 *>(orow + c0 + 8 * i) = v;
          }
        }
      }
      if (row_ok) p.lse[(size_t)bh * p.S + q_g] = m * 0.6931471805599453f;
      tc_fence_before();
    }
  }
  // the pair's MMAs have all completed before either CTA gives tensor memory back
  if (warp == 1 && lane == 0) mbar_drain_cluster(&bars[pFinal], 0, g.limit_ns);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

cudaError_t launch_fwd_pair_t(const CUtensorMap &q, const CUtensorMap &kh, const CUtensorMap &v,
                              const FwdParams &p, int BH, cudaStream_t stream) {
  auto kfn = dash_fwd_pair_kernel;
  const int smem = pairfwd::kSmemBytes > (uint32_t)kMinSmemOneCtaPerSm ? (int)pairfwd::kSmemBytes
                                                                        : kMinSmemOneCtaPerSm;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nblk = (p.S + 127) / 128;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * ((nblk + 1) / 2), BH);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kfn, q, kh, v, p);
}

}  // namespace

cudaError_t launch_fwd_pair(const CUtensorMap &q, const CUtensorMap &k_half_rows, const CUtensorMap &v,
                            const FwdParams &p, int BH, cudaStream_t stream) {
  return launch_fwd_pair_t(q, k_half_rows, v, p, BH, stream);
}

cudaError_t launch_fwd(int D, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                       const FwdParams &p, int BH, cudaStream_t stream) {
  if (D == 64) return launch_fwd_t<64>(q, k, v, p, BH, stream);
  if (D == 128) return launch_fwd_t<128>(q, k, v, p, BH, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dash
