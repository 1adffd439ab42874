// Pieces of the backward main kernel that keeps dQ transposed (fa_bwd_dt.cu):
// tile sizes, warp roles, the persistent schedule over key blocks, the
// visible query range of a key block, and failure reporting.
#pragma once
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_order.cuh"
#include "fa_window.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int BQ = 64;             // queries per step
constexpr int BK = 128;            // keys per work item
constexpr int DH = 128;            // head-dimension columns of dK, dV, dQ per work item
constexpr int KCH = 128 * 128;     // 128 rows x 128 bytes
constexpr int QCH = 64 * 128;      // 64 rows x 128 bytes
constexpr int kRowWarps = 8;       // two per sub-partition, one per 32-query half
constexpr int kDrainWarp0 = 3 + kRowWarps;   // four dQ drain warps
constexpr int kReduceWarp = kDrainWarp0 + 4; // d = 256: issues the dQ bulk reduce-adds
constexpr int kThreads = 32 * (kDrainWarp0 + 4);   // 15 warps (16 with the reduce warp)
// With 15 warps one sub-partition holds four: 128 registers a thread at most
// (the compiler is told 512 threads so that it plans for that).
constexpr int kRegThreads = 512;

enum Site {
  kSiteProdKV = 64, kSiteProdQ, kSiteMmaKV, kSiteMmaQ, kSiteMmaP, kSiteMmaDs, kSiteMmaDq,
  kSiteMmaAcc, kSiteRowS, kSiteRowDp, kSiteRowDsFree, kSiteRowAcc, kSiteDrainDq, kSiteDtDrain,
  kSiteStageFree, kSiteStageFull, kSiteRowV, kSiteMmaV, kSiteProdDo, kSiteMmaDo
};

__device__ __forceinline__ void record_failure(int* status, volatile int* abort, int site) {
  atomicCAS(status, 0, status_code(site));
  *abort = 1;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  bool ok = mbar_wait(bar, parity, abort, kWaitTimeoutNs);
  return __all_sync(0xffffffffu, ok);
}

// Column of the packed bf16 P^T / dS^T for K-step kk (16 queries) within its
// 64-column buffer: queries 32h .. 32h+31 sit in columns 32h .. 32h+15.
__device__ __forceinline__ constexpr uint32_t pcol(int kk) {
  return static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8);
}

// Issuer warps wait as a whole warp (mbar_wait_warp) and report a failure
// from lane 0.
__device__ __forceinline__ void issuer_fail(int* status, volatile int* abort, int lane, int site) {
  if (lane == 0) record_failure(status, abort, site);
}

// Units are (K/V head kvbh, key-block pair or key block, half); a work item
// (one key block) steps over the query heads of kvbh's group and, for each,
// the query blocks its keys are visible to.  Plain causal: key block n meets
// query blocks from its diagonal on, so blocks p and T-1-p are paired,
// longest first.  The halves of one key block are adjacent units so they run
// at the same time and share K, V, Q, dO in L2.
// This CTA's place in the schedule: its round-robin units (and the key
// blocks of a causal pair), then its row of the tail table.
struct DtIter {
  int u, kt, k;
};

// A block mask without a host copy (order != nullptr): the items (K/V head,
// key block; the halves of d adjacent) go in the cost-sorted turning deal of
// fa_order.cuh instead, from the order planned into the workspace.
struct DtSched {
  int T, P, per_bh, units, causal, nsplit;   // units: the round-robin units
  int BH;
  const uint32_t* order;                     // the cost-sorted order, or nullptr
  __device__ DtSched(int BH_, int N, int causal_, int nsplit_, int tail_heads,
                     const uint32_t* order_)
      : causal(causal_), nsplit(nsplit_), BH(BH_), order(order_) {
    T = (N + BK - 1) / BK;
    P = (T + 1) / 2;
    per_bh = causal ? P : T;
    units = (BH - tail_heads) * per_bh * nsplit;
  }
  __device__ void decode(int u, int& bh, int& pp, int& h) const {
    bh = u / (per_bh * nsplit);
    const int rem = u % (per_bh * nsplit);
    pp = rem / nsplit;
    h = rem % nsplit;
  }
  __device__ int nitems(int pp) const {
    if (!causal) return 1;
    return (pp == T - 1 - pp) ? 1 : 2;
  }
  __device__ int block(int pp, int k) const {
    if (!causal) return pp;
    return (k == 0) ? pp : (T - 1 - pp);
  }
  // The next work item of this CTA (K/V head, half of d, key block); false
  // when it has none left.  Every role walks the same sequence.
  __device__ bool next(const TailTable& tail, DtIter& it, int& kvbh, int& h, int& n) const {
    if (order) {   // round it.k of the cost-sorted deal
      const long long k = order_deal(it.k, gridDim.x, blockIdx.x);
      if (k >= static_cast<long long>(BH) * T * nsplit) return false;
      ++it.k;
      h = static_cast<int>(k % nsplit);
      order_item(order, BH, k / nsplit, kvbh, n);
      return true;
    }
    while (it.u < units) {
      int pp;
      decode(it.u, kvbh, pp, h);
      if (it.kt < nitems(pp)) {
        n = block(pp, it.kt);
        ++it.kt;
        return true;
      }
      it.u += gridDim.x;
      it.kt = 0;
    }
    if (tail.heads == 0 || blockIdx.x >= kTailCtas || it.k >= kTailItems) return false;
    const int e = tail.item[blockIdx.x][it.k];
    if (e < 0) return false;
    ++it.k;
    kvbh = tail_head(e);
    h = tail_half(e);
    n = tail_block(e);
    return true;
  }
};

// kv_len of K/V head kvbh's batch entry.
__device__ __forceinline__ int dt_len(const BwdParams& p, int kvbh) {
  int len = p.N;
  if (p.kv_len) {
    len = __ldg(p.kv_len + kvbh / p.H_kv);
    len = len < 0 ? 0 : (len > p.N ? p.N : len);
  }
  return len;
}

// Query-step range [i0, i1) (blocks of 64) that key block n is visible to
// (kv_len, causal and window); empty when no query sees any of its keys.
__device__ __forceinline__ void dt_range(const BwdParams& p, int n, int len, int& i0, int& i1) {
  int q_lo, q_hi;
  visible_queries(n * BK, BK, len, p.N, p.wl, p.wr, q_lo, q_hi);
  if (q_hi <= q_lo) {
    i0 = i1 = 0;
    return;
  }
  i0 = q_lo / BQ;
  i1 = (q_hi + BQ - 1) / BQ;
}

}  // namespace
}  // namespace fa
