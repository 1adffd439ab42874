// Attention backward for sm_103a: three launches on one stream.  The main
// kernel in this file serves head dimension 64; 128 and 256 use the kernel
// in fa_bwd_dt.cu (same pre- and post-kernels).
//
//  1. bwd_pre   D_i = sum_t dO_it * O_it and L2_i = LSE_i * log2(e) per query
//               row (padded to a multiple of 128 rows: D = 0, L2 = +inf past
//               N), and zero the fp32 dQ accumulator.  Memory bound.
//  2. bwd_main  one CTA per (bh, 128-key block), persistent.  K and V of the
//               block stay in shared memory; 128-query blocks of Q and dO
//               stream through a 2-deep ring.  Per query block, on the
//               tensor core with accumulators in tensor memory:
//                 S^T  = K Q_i^T           P^T  = exp2(S^T*c - L2_i)  (recomputed)
//                 dP^T = V dO_i^T          dS^T = P^T o (dP^T - D_i)
//                 dV  += P^T dO_i          dK  += dS^T Q_i
//                 dQ_i = dS K   -> added to the fp32 accumulator in global memory
//               P^T and dS^T go back into tensor memory as bf16 (A operands of
//               the dV / dK products) and dS^T also to shared memory (A operand
//               of dQ).  dK is scaled by `scale` when it is written.
//  3. bwd_post  dQ = bf16(scale * dQ_acc).
//
// The recomputation of P from the saved statistic follows "注意力为什么受限于
// 显存带宽：用算术强度与分块把 FlashAttention 推导清楚" (section 八) and "4.
// FlashAttention 深度剖析" (section 4.3.4, P_ij = exp(S_ij - L_i)).  The pages
// print no gradient formulas; the ones above are the chain rule through the
// row softmax and O = P V.
//
// Warp roles of bwd_main (192 threads): warp 0 loads (TMA), warp 1 issues the
// MMAs and owns tensor memory, warps 2..5 own tensor-memory lanes: as key rows
// for S^T, dP^T, dV, dK and as query rows for dQ.
//
// Tensor memory columns: S^T [0,128) (P^T bf16 written over [0,64)),
// dP^T [128,256) (dS^T bf16 over [128,192)), dV [256,256+D),
// dK [256+D,256+2D), dQ at [384,448) for D=64, and over the S^T columns for
// D=128 (the next S^T waits until dQ has been drained).  Successive
// tcgen05.mma issued by one thread execute in order, so an MMA that writes
// columns an earlier MMA reads as an operand needs no extra wait.
#include <cstring>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_window.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int BM = 128;          // queries per step (MMA N of S^T and dP^T, M of dQ)
constexpr int BN = 128;          // keys per CTA work item (MMA M of S^T, dP^T, dV, dK)
constexpr int CHUNK = 128 * 128; // one 128-row x 128-byte SW128 region
constexpr int kThreads = 192;
constexpr int kStages = 2;

template <int D>
struct BCfg {
  static constexpr int NCH = D / 64;
  static constexpr int TILE_BYTES = NCH * CHUNK;
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_DP = 128;
  static constexpr uint32_t TM_DV = 256;
  static constexpr uint32_t TM_DK = 256 + D;
  static constexpr uint32_t TM_DQ = D == 64 ? 384 : 0;
  static constexpr bool DQ_ALIASES_S = (D != 64);
  static constexpr uint32_t TM_COLS = 512;
  static_assert(256 + 2 * D <= 512, "tensor memory budget");
};

template <int D>
struct BwdSmem {
  alignas(1024) uint8_t k[BCfg<D>::TILE_BYTES];
  alignas(1024) uint8_t v[BCfg<D>::TILE_BYTES];
  alignas(1024) uint8_t q[kStages][BCfg<D>::TILE_BYTES];
  alignas(1024) uint8_t dO[kStages][BCfg<D>::TILE_BYTES];
  alignas(1024) uint8_t ds[2 * CHUNK];           // dS^T bf16: 128 keys x 128 queries
  alignas(16) float lse2[kStages][BM];
  alignas(16) float delta[kStages][BM];
  uint64_t kv_full, kv_empty;
  uint64_t q_full[kStages], q_empty[kStages];
  uint64_t s_full, p_full, dp_full, ds_full, dq_full, dq_free, acc_full, acc_free;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

enum Site {
  kSiteProdKV = 32, kSiteProdQ, kSiteMmaKV, kSiteMmaQ, kSiteMmaDq, kSiteMmaP, kSiteMmaDs,
  kSiteMmaAcc, kSiteSmS, kSiteSmDp, kSiteSmDq, kSiteSmAcc, kSiteBDrain
};

__device__ __forceinline__ void record_failure(int* status, volatile int* abort, int site) {
  atomicCAS(status, 0, status_code(site));
  *abort = 1;
}

__device__ __forceinline__ void issuer_fail(int* status, volatile int* abort, int lane, int site) {
  if (lane == 0) record_failure(status, abort, site);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  bool ok = mbar_wait(bar, parity, abort, kWaitTimeoutNs);
  return __all_sync(0xffffffffu, ok);
}

// Work items (K/V head kvbh, key block n); an item's steps run over the
// query heads of kvbh's group and, for each, the query blocks the key block
// is visible to.  Plain causal: key block n meets query blocks n..T-1, so
// items n and T-1-n are paired (longest first) and every unit costs T+1
// steps per query head; the last tail.heads heads come as single items from
// the tail table.  Otherwise: one item per unit, head-major.
struct BIter {
  int u, kt, k;
};

struct BSched {
  int T, P, units, causal;   // units: the round-robin units
  __device__ BSched(int BH, int N, int causal_, int tail_heads) : causal(causal_) {
    T = (N + BN - 1) / BN;
    P = (T + 1) / 2;
    units = (BH - tail_heads) * (causal ? P : T);
  }
  __device__ int nitems(int u) const {
    if (!causal) return 1;
    const int p = u % P;
    return (p == T - 1 - p) ? 1 : 2;
  }
  __device__ void item(int u, int k, int& bh, int& n) const {
    if (!causal) {
      bh = u / T;
      n = u % T;
    } else {
      bh = u / P;
      const int p = u % P;
      n = (k == 0) ? p : (T - 1 - p);
    }
  }
  // The next item of this CTA; false when it has none left.  Every role walks
  // the same sequence: the round-robin units, then this CTA's tail row.
  __device__ bool next(const TailTable& tail, BIter& it, int& bh, int& n) const {
    while (it.u < units) {
      if (it.kt < nitems(it.u)) {
        item(it.u, it.kt, bh, n);
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
    bh = tail_head(e);
    n = tail_block(e);
    return true;
  }
};

// kv_len of K/V head kvbh's batch entry.
__device__ __forceinline__ int bwd_len(const BwdParams& p, int kvbh) {
  int len = p.N;
  if (p.kv_len) {
    len = __ldg(p.kv_len + kvbh / p.H_kv);
    len = len < 0 ? 0 : (len > p.N ? p.N : len);
  }
  return len;
}

// Query-block range [i0, i1) that key block n is visible to (kv_len, causal
// and window); empty when no query sees any of its keys.
__device__ __forceinline__ void q_range(const BwdParams& p, int n, int len, int& i0, int& i1) {
  int q_lo, q_hi;
  visible_queries(n * BN, BN, len, p.N, p.wl, p.wr, q_lo, q_hi);
  if (q_hi <= q_lo) {
    i0 = i1 = 0;
    return;
  }
  i0 = q_lo / BM;
  i1 = (q_hi + BM - 1) / BM;
}

// BS: the launch carries a block mask (its own instantiation).
template <int D, bool BS>
__global__ void __launch_bounds__(kThreads, 1) bwd_main_kernel(const __grid_constant__ BwdParams p,
                                                                   const __grid_constant__ TailTable tail) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
  const uintptr_t aligned = (raw + 1023) & ~static_cast<uintptr_t>(1023);
  if (aligned - raw + sizeof(BwdSmem<D>) > dynamic_smem_size()) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, status_code(kSiteSmemLayout));
    return;
  }
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(aligned);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  volatile int* abort = &sm.abort;

  if (threadIdx.x == 0) {
    sm.abort = 0;
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.p_full, 4);
    mbar_init(&sm.dp_full, 1);
    mbar_init(&sm.ds_full, 4);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_free, 4);
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_free, 4);
    mbar_init(&sm.mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  const BSched sched(p.B * p.H_kv, p.N, p.causal, tail.heads);
  const int G = p.H / p.H_kv;                     // query heads per K/V head

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tq);
      prefetch_tmap(&p.tk);
      prefetch_tmap(&p.tv);
      prefetch_tmap(&p.tdo);
      uint32_t w_it = 0, g = 0;
      bool ok = true;
      BIter it{static_cast<int>(blockIdx.x), 0, 0};
      for (int kvbh, n; ok && sched.next(tail, it, kvbh, n);) {
        {
          int i0, i1;
          q_range(p, n, bwd_len(p, kvbh), i0, i1);
          const StepMask sk{BS ? p.block_mask + n : nullptr, p.bm_t, 128 / BM};
          const int nst = count_steps(sk, i0, i1);
          if (nst == 0) i1 = i0;
          if (i0 >= i1) continue;
          if (!mbar_wait(&sm.kv_empty, (w_it & 1) ^ 1, abort, kWaitTimeoutNs)) {
            record_failure(p.status, abort, kSiteProdKV);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.kv_full, 2 * C::TILE_BYTES);
#pragma unroll
          for (int c = 0; c < C::NCH; ++c) {
            tma_load_3d(sm.k + c * CHUNK, &p.tk, &sm.kv_full, 64 * c, n * BN, kvbh);
            tma_load_3d(sm.v + c * CHUNK, &p.tv, &sm.kv_full, 64 * c, n * BN, kvbh);
          }
          ++w_it;
          StepWalk wk(i0, i1, q_head_of(kvbh, 0, p.H, p.H_kv), sk);
          for (int s = 0; s < nst * G; ++s, wk.next()) {
            const int i = wk.i;
            const int bh = wk.bh;
            const int st = g % kStages;
            if (!mbar_wait(&sm.q_empty[st], ((g / kStages) & 1) ^ 1, abort, kWaitTimeoutNs)) {
              record_failure(p.status, abort, kSiteProdQ);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sm.q_full[st], 2 * C::TILE_BYTES + 2 * BM * 4);
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
              tma_load_3d(sm.q[st] + c * CHUNK, &p.tq, &sm.q_full[st], 64 * c, i * BM, bh);
              tma_load_3d(sm.dO[st] + c * CHUNK, &p.tdo, &sm.q_full[st], 64 * c, i * BM, bh);
            }
            const size_t roff = static_cast<size_t>(bh) * p.Npad + static_cast<size_t>(i) * BM;
            bulk_load(sm.lse2[st], p.lse2 + roff, BM * 4, &sm.q_full[st]);
            bulk_load(sm.delta[st], p.delta + roff, BM * 4, &sm.q_full[st]);
            ++g;
          }
        }
      }
      // drain: no copy may still be landing when the CTA exits
      if (w_it > 0 && !mbar_wait(&sm.kv_full, (w_it - 1) & 1, nullptr, kWaitTimeoutNs))
        record_failure(p.status, abort, kSiteBDrain);
      for (int s = 0; s < kStages; ++s) {
        if (g > static_cast<uint32_t>(s)) {
          const uint32_t n = (g - 1 - s) / kStages;
          if (!mbar_wait(&sm.q_full[s], n & 1, nullptr, kWaitTimeoutNs))
            record_failure(p.status, abort, kSiteBDrain);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    {
      constexpr uint32_t kIdescS = idesc_bf16_f32(BN, BM, 0, 0);     // S^T, dP^T
      constexpr uint32_t kIdescAcc = idesc_bf16_f32(BN, D, 0, 1);    // dV, dK: B MN-major
      constexpr uint32_t kIdescDq = idesc_bf16_f32(BM, D, 1, 1);     // dQ: A and B MN-major
      const uint64_t dK0 = sdesc_sw128(smem_u32(sm.k), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sm.v), 16, 1024);
      const uint64_t dKmn = sdesc_sw128(smem_u32(sm.k), CHUNK, 1024);
      const uint64_t dDS = sdesc_sw128(smem_u32(sm.ds), CHUNK, 1024);
      uint32_t w_it = 0, g = 0;
      bool ok = true;
      BIter it{static_cast<int>(blockIdx.x), 0, 0};
      for (int kvbh, n; ok && sched.next(tail, it, kvbh, n);) {
        {
          int i0, i1;
          q_range(p, n, bwd_len(p, kvbh), i0, i1);
          const StepMask sk{BS ? p.block_mask + n : nullptr, p.bm_t, 128 / BM};
          const int nst = count_steps(sk, i0, i1);
          if (nst == 0) i1 = i0;
          if (i0 >= i1) continue;
          if (!mbar_wait_warp(&sm.kv_full, w_it & 1, abort, kWaitTimeoutNs)) {
            issuer_fail(p.status, abort, lane, kSiteMmaKV);
            ok = false;
            break;
          }
          const int nsteps = nst * G;
          for (int s = 0; s < nsteps; ++s) {
            const int st = g % kStages;
            const bool first = (s == 0);
            if (!mbar_wait_warp(&sm.q_full[st], (g / kStages) & 1, abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaQ);
              ok = false;
              break;
            }
            // dQ of the previous step must be out of tensor memory before the
            // columns it occupies are written again.
            if (C::DQ_ALIASES_S && g > 0 &&
                !mbar_wait_warp(&sm.dq_free, (g - 1) & 1, abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaDq);
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint64_t dQ0 = sdesc_sw128(smem_u32(sm.q[st]), 16, 1024);
            const uint64_t dO0 = sdesc_sw128(smem_u32(sm.dO[st]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk / 4) * CHUNK + (kk % 4) * 32) >> 4;
              mma_bf16_ss_w(tmem + C::TM_S, dK0 + off, dQ0 + off, kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&sm.s_full);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk / 4) * CHUNK + (kk % 4) * 32) >> 4;
              mma_bf16_ss_w(tmem + C::TM_DP, dV0 + off, dO0 + off, kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&sm.dp_full);
            // dV += P^T dO_i
            if (!mbar_wait_warp(&sm.p_full, g & 1, abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaP);
              ok = false;
              break;
            }
            if (first && !mbar_wait_warp(&sm.acc_free, (w_it & 1) ^ 1, abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaAcc);
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint64_t dOmn = sdesc_sw128(smem_u32(sm.dO[st]), CHUNK, 1024);
            const uint64_t dQmn = sdesc_sw128(smem_u32(sm.q[st]), CHUNK, 1024);
#pragma unroll
            for (int kk = 0; kk < BM / 16; ++kk)
              mma_bf16_ts_w(tmem + C::TM_DV, tmem + C::TM_S + kk * 8, dOmn + ((kk * 2048) >> 4),
                          kIdescAcc, (first && kk == 0) ? 0u : 1u);
            // dK += dS^T Q_i and dQ_i = dS K
            if (!mbar_wait_warp(&sm.ds_full, g & 1, abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaDs);
              ok = false;
              break;
            }
            if (!C::DQ_ALIASES_S && g > 0 &&
                !mbar_wait_warp(&sm.dq_free, (g - 1) & 1, abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaDq);
              ok = false;
              break;
            }
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < BM / 16; ++kk)
              mma_bf16_ts_w(tmem + C::TM_DK, tmem + C::TM_DP + kk * 8, dQmn + ((kk * 2048) >> 4),
                          kIdescAcc, (first && kk == 0) ? 0u : 1u);
            mma_commit_w(&sm.q_empty[st]);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_bf16_ss_w(tmem + C::TM_DQ, dDS + ((kk * 2048) >> 4), dKmn + ((kk * 2048) >> 4),
                          kIdescDq, kk > 0 ? 1u : 0u);
            mma_commit_w(&sm.dq_full);
            if (s == nsteps - 1) {
              mma_commit_w(&sm.acc_full);
              mma_commit_w(&sm.kv_empty);
            }
            ++g;
          }
          ++w_it;
        }
      }
      mma_commit_w(&sm.mma_done);
      if (!mbar_wait_warp(&sm.mma_done, 0, nullptr, kWaitTimeoutNs))
        issuer_fail(p.status, abort, lane, kSiteBDrain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ row warps
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;            // tensor-memory lane owned by this thread
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c2 = p.scale_log2;
    __nv_bfloat16* dk_out = static_cast<__nv_bfloat16*>(p.dk);
    __nv_bfloat16* dv_out = static_cast<__nv_bfloat16*>(p.dv);
    uint32_t w_it = 0, g = 0;
    bool ok = true;
    BIter it{static_cast<int>(blockIdx.x), 0, 0};
    for (int kvbh, n; ok && sched.next(tail, it, kvbh, n);) {
      {
        int i0, i1;
        const int len = bwd_len(p, kvbh);
        q_range(p, n, len, i0, i1);
        const StepMask sk{BS ? p.block_mask + n : nullptr, p.bm_t, 128 / BM};
        const int nst = count_steps(sk, i0, i1);
        if (nst == 0) i1 = i0;
        const int key = n * BN + r;
        const size_t key_off = static_cast<size_t>(kvbh) * p.N + key;
        if (i0 >= i1) {
          // key block entirely past the sequence: zero gradients
          if (key < p.N) {
            uint4* a = reinterpret_cast<uint4*>(dk_out + key_off * D);
            uint4* b = reinterpret_cast<uint4*>(dv_out + key_off * D);
#pragma unroll
            for (int t = 0; t < D / 8; ++t) {
              a[t] = make_uint4(0, 0, 0, 0);
              b[t] = make_uint4(0, 0, 0, 0);
            }
          }
          continue;
        }
        StepWalk wk(i0, i1, q_head_of(kvbh, 0, p.H, p.H_kv), sk);
        for (int s = 0; s < nst * G; ++s, wk.next()) {
          const int i = wk.i;
          const int bh = wk.bh;
          const int st = g % kStages;
          // ---- P^T = exp2(S^T * c - L2), masked
          if (!warp_wait(&sm.s_full, g & 1, abort)) {
            if (lane == 0) record_failure(p.status, abort, kSiteSmS);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const int q0 = i * BM;
          const bool need_mask = (n * BN + BN > len) || (q0 + BM > p.N) ||
                                 (n * BN + BN - 1 > q0 + p.wr) || (n * BN < q0 + BM - 1 - p.wl);
          // visible columns c (query q0 + c) of this key row: [c_lo, c_hi],
          // the queries whose window [q - wl, q + wr] holds the key; none
          // when the key is past len
          const int c_lo = key - p.wr - q0;
          const int c_hi = (key < len) ? key + p.wl - q0 : -1;
          float pr[BM];
#pragma unroll
          for (int c4 = 0; c4 < BM / 32; ++c4) {
            uint32_t sr[32];
            tmem_ld_x32(t_lane + C::TM_S + 32 * c4, sr);
            tmem_wait_ld();
            reg_fence<32>(sr);
            const float4* l2v = reinterpret_cast<const float4*>(sm.lse2[st] + 32 * c4);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float4 l4 = l2v[t];
              const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e)
                pr[32 * c4 + 4 * t + e] = ex2_approx(fmaf(__uint_as_float(sr[4 * t + e]), c2, -lv[e]));
            }
            if (need_mask) {      // diagonal and boundary steps only
#pragma unroll
              for (int c = 32 * c4; c < 32 * c4 + 32; ++c)
                if (c < c_lo || c > c_hi) pr[c] = 0.f;
            }
            uint32_t pk[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) pk[t] = pack_bf16x2(pr[32 * c4 + 2 * t], pr[32 * c4 + 2 * t + 1]);
            tmem_st_x16(t_lane + C::TM_S + 16 * c4, pk);
          }
          tmem_wait_st();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.p_full);
          // ---- dS^T = P^T o (dP^T - D)
          if (!warp_wait(&sm.dp_full, g & 1, abort)) {
            if (lane == 0) record_failure(p.status, abort, kSiteSmDp);
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int c4 = 0; c4 < BM / 32; ++c4) {
            uint32_t dr[32];
            tmem_ld_x32(t_lane + C::TM_DP + 32 * c4, dr);
            tmem_wait_ld();
            reg_fence<32>(dr);
            const float4* dv4 = reinterpret_cast<const float4*>(sm.delta[st] + 32 * c4);
            uint32_t pk[16];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float4 d4 = dv4[t];
              const int c = 32 * c4 + 4 * t;
              const float s0 = pr[c] * (__uint_as_float(dr[4 * t]) - d4.x);
              const float s1 = pr[c + 1] * (__uint_as_float(dr[4 * t + 1]) - d4.y);
              const float s2 = pr[c + 2] * (__uint_as_float(dr[4 * t + 2]) - d4.z);
              const float s3 = pr[c + 3] * (__uint_as_float(dr[4 * t + 3]) - d4.w);
              pk[2 * t] = pack_bf16x2(s0, s1);
              pk[2 * t + 1] = pack_bf16x2(s2, s3);
            }
            tmem_st_x16(t_lane + C::TM_DP + 16 * c4, pk);
            // shared copy, MN-major A of dQ: row = key r, 64-query chunks,
            // 16-byte units XOR-swizzled by (r & 7)
            uint8_t* rowp = sm.ds + (c4 >> 1) * CHUNK + r * 128;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int unit = (c4 & 1) * 4 + t;
              *reinterpret_cast<uint4*>(rowp + ((unit ^ (r & 7)) << 4)) =
                  make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
            }
          }
          fence_proxy_async_smem();
          tmem_wait_st();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.ds_full);
          // ---- dQ_i rows (this thread: query q0 + r) into the fp32 accumulator
          if (!warp_wait(&sm.dq_full, g & 1, abort)) {
            if (lane == 0) record_failure(p.status, abort, kSiteSmDq);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          {
            const int q = q0 + r;
            float* acc = p.dq_acc + (static_cast<size_t>(bh) * p.Npad + q) * D;
#pragma unroll 1
            for (int c4 = 0; c4 < D / 32; ++c4) {
              uint32_t qr[32];
              tmem_ld_x32(t_lane + C::TM_DQ + 32 * c4, qr);
              tmem_wait_ld();
              reg_fence<32>(qr);
              if (q < p.N) {
                float4* dst = reinterpret_cast<float4*>(acc + 32 * c4);
#pragma unroll
                for (int t = 0; t < 8; ++t)
                  atomicAdd(dst + t, make_float4(__uint_as_float(qr[4 * t]), __uint_as_float(qr[4 * t + 1]),
                                                 __uint_as_float(qr[4 * t + 2]),
                                                 __uint_as_float(qr[4 * t + 3])));
              }
            }
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.dq_free);
          ++g;
        }
        if (!ok) break;
        // ---- dK, dV rows of this key block
        if (!warp_wait(&sm.acc_full, w_it & 1, abort)) {
          if (lane == 0) record_failure(p.status, abort, kSiteSmAcc);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        // dV and dK rows leave tensor memory on one wait; the accumulators are
        // then free for the next key block while the rows are converted and
        // stored, 32 bytes a store when both outputs are 32-byte aligned
        static_assert(D == 64, "this kernel serves d = 64");
        uint32_t a[D], b[D];
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          tmem_ld_x32(t_lane + C::TM_DV + 32 * c4, a + 32 * c4);
          tmem_ld_x32(t_lane + C::TM_DK + 32 * c4, b + 32 * c4);
        }
        tmem_wait_ld();
        reg_fence<D>(a);
        reg_fence<D>(b);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_free);
        if (key < p.N) {
          const bool st32 = ((reinterpret_cast<uintptr_t>(dk_out) |
                              reinterpret_cast<uintptr_t>(dv_out)) & 31u) == 0;
#pragma unroll
          for (int c16 = 0; c16 < D / 16; ++c16) {          // 16 columns a step
            uint32_t pv[8], pk[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              pv[t] = pack_bf16x2(__uint_as_float(a[16 * c16 + 2 * t]),
                                  __uint_as_float(a[16 * c16 + 2 * t + 1]));
              pk[t] = pack_bf16x2(__uint_as_float(b[16 * c16 + 2 * t]) * p.scale,
                                  __uint_as_float(b[16 * c16 + 2 * t + 1]) * p.scale);
            }
            __nv_bfloat16* dvp = dv_out + key_off * D + 16 * c16;
            __nv_bfloat16* dkp = dk_out + key_off * D + 16 * c16;
            if (st32) {
              st_global_v8(dvp, pv);
              st_global_v8(dkp, pk);
            } else {
              uint4* v4 = reinterpret_cast<uint4*>(dvp);
              uint4* k4 = reinterpret_cast<uint4*>(dkp);
              v4[0] = make_uint4(pv[0], pv[1], pv[2], pv[3]);
              v4[1] = make_uint4(pv[4], pv[5], pv[6], pv[7]);
              k4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              k4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
          }
        }
        ++w_it;
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, BCfg<D>::TM_COLS);
  }
}

// D, L2 and the dQ accumulator reset.  A group of D/8 lanes handles one row
// (16 bytes of O and dO per lane).
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __grid_constant__ BwdParams p) {
  constexpr int LPR = D / 8;                      // lanes per row
  constexpr int ROWS = 256 / LPR;                 // rows per block
  const int sub = threadIdx.x % LPR;
  const long long row = static_cast<long long>(blockIdx.x) * ROWS + threadIdx.x / LPR;
  const long long total = static_cast<long long>(p.B) * p.H * p.Npad;
  const bool live = row < total;
  const int bh = live ? static_cast<int>(row / p.Npad) : 0;
  const int i = live ? static_cast<int>(row % p.Npad) : 0;
  const bool in_seq = live && i < p.N;
  float acc = 0.f;
  if (in_seq) {
    const size_t off = (static_cast<size_t>(bh) * p.N + i) * D + sub * 8;
    const uint4 ov = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.o) + off);
    const uint4 gv = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.dO) + off);
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 a = __bfloat1622float2(o2[t]);
      const float2 b = __bfloat1622float2(g2[t]);
      acc = fmaf(a.x, b.x, acc);
      acc = fmaf(a.y, b.y, acc);
    }
  }
  if (live) {
    // the accumulator holds Npad * D floats per head in either layout: row
    // `row` of this grid clears its D of them, padding included
    float4* z = reinterpret_cast<float4*>(p.dq_acc + static_cast<size_t>(row) * D + sub * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int m = LPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (live && sub == 0) {
    const size_t o = static_cast<size_t>(bh) * p.Npad + i;
    p.delta[o] = in_seq ? acc : 0.f;
    p.lse2[o] = in_seq ? p.lse[static_cast<size_t>(bh) * p.N + i] * 1.4426950408889634f : INFINITY;
  }
}

// dQ = bf16(scale * dQ_acc) from the [BH, Npad, d] accumulator (d = 64), 8
// elements per thread.
__global__ void __launch_bounds__(256) bwd_post_kernel(const __grid_constant__ BwdParams p,
                                                       long long n8) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n8) return;
  constexpr int D8 = 64 / 8;
  const long long row = t / D8;                       // bh * N + q
  const long long bh = row / p.N;
  const long long src_row = bh * p.Npad + (row - bh * p.N);
  const float4* src = reinterpret_cast<const float4*>(p.dq_acc + src_row * 64) + 2 * (t % D8);
  const float4 a = src[0], b = src[1];
  const float s = p.scale;
  uint4 out;
  out.x = pack_bf16x2(a.x * s, a.y * s);
  out.y = pack_bf16x2(a.z * s, a.w * s);
  out.z = pack_bf16x2(b.x * s, b.y * s);
  out.w = pack_bf16x2(b.z * s, b.w * s);
  reinterpret_cast<uint4*>(p.dq)[t] = out;
}

// dQ = bf16(scale * dQ_acc^T) from the [BH, D, Npad] accumulator.  Thread
// (bh, column group c16, query q): lanes run over q, so each of its 16 column
// reads is a coalesced 128-byte row segment; it writes 16 bf16 of query q in
// one 32-byte store (two 16-byte stores when dQ is only 16-byte aligned).
template <int D>
__global__ void __launch_bounds__(256) bwd_post_t_kernel(const __grid_constant__ BwdParams p,
                                                         long long total) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= total) return;
  const int q = static_cast<int>(t % p.Npad);
  const long long rest = t / p.Npad;
  const int c16 = static_cast<int>(rest % (D / 16));
  const long long bh = rest / (D / 16);
  if (q >= p.N) return;
  const float* src = p.dq_acc + (bh * D + c16 * 16) * p.Npad + q;
  float a[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) a[j] = src[static_cast<size_t>(j) * p.Npad] * p.scale;
  uint32_t pk[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) pk[j] = pack_bf16x2(a[2 * j], a[2 * j + 1]);
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.dq) + (bh * p.N + q) * D + c16 * 16;
  if ((reinterpret_cast<uintptr_t>(p.dq) & 31u) == 0) {
    st_global_v8(dst, pk);
  } else {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  }
}

template <int D>
cudaError_t launch_prep(const BwdParams& p, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.Npad;
  constexpr int ROWS = 256 / (D / 8);
  bwd_pre_kernel<D><<<static_cast<unsigned>((rows + ROWS - 1) / ROWS), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D, bool BS>
cudaError_t launch_main(const BwdParams& p, int num_sms, int max_smem, cudaStream_t stream) {
  const size_t smem = smem_request(sizeof(BwdSmem<D>), max_smem);
  cudaError_t e = cudaFuncSetAttribute(bwd_main_kernel<D, BS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int T = (p.N + BN - 1) / BN;
  const int BH = p.B * p.H_kv;
  long long units = p.causal ? static_cast<long long>(BH) * ((T + 1) / 2)
                             : static_cast<long long>(BH) * T;
  TailTable tail;
  tail.heads = 0;
  if (p.causal || (BS && p.block_mask_host && T == p.bm_t)) {
    // single key blocks in the tail: up to one CTA per block; the tail's
    // K/V heads share their group's Q and dO through L2
    const long long blocks = static_cast<long long>(BH) * T;
    const int g = static_cast<int>(blocks < num_sms ? blocks : num_sms);
    const long long qdo_bytes = 2ll * (p.H / p.H_kv) * p.N * D * 2;
    if (p.causal)
      plan_causal_tail(BH, T, 1, g, false, qdo_bytes, &tail);
    else                       // key blocks cost their computed query steps
      plan_mask_tail(p.block_mask_host, BH, T, 1, g, false, p.N, p.wl, p.wr, qdo_bytes, &tail);
    if (tail.heads > 0) units = g;
  }
  if (tail.heads == 0) std::memset(tail.item, 0xff, sizeof(tail.item));
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  bwd_main_kernel<D, BS><<<grid, kThreads, smem, stream>>>(p, tail);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdParams& p, int d, cudaStream_t stream) {
  switch (d) {
    case 64: return launch_prep<64>(p, stream);
    case 128: return launch_prep<128>(p, stream);
    case 256: return launch_prep<256>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_main(const BwdParams& p, int d, int num_sms, int max_smem,
                            cudaStream_t stream) {
  switch (d) {
    case 64:
      return p.block_mask ? launch_main<64, true>(p, num_sms, max_smem, stream)
                          : launch_main<64, false>(p, num_sms, max_smem, stream);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t launch_bwd_post(const BwdParams& p, int d, cudaStream_t stream) {
  if (d == 64) {
    const long long n8 = static_cast<long long>(p.B) * p.H * p.N * d / 8;
    bwd_post_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, stream>>>(p, n8);
    return cudaGetLastError();
  }
  const long long total = static_cast<long long>(p.B) * p.H * (d / 16) * p.Npad;
  const unsigned grid = static_cast<unsigned>((total + 255) / 256);
  switch (d) {
    case 128: bwd_post_t_kernel<128><<<grid, 256, 0, stream>>>(p, total); break;
    case 256: bwd_post_t_kernel<256><<<grid, 256, 0, stream>>>(p, total); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace fa
