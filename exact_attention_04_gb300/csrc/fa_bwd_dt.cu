// Backward main kernel for head dimensions 128 and 256 ("dQ transposed").
//
// Work item: (K/V head, block of 128 keys, half h of the head dimension).
// The CTA keeps K and V of its key block on chip and streams the query blocks
// of 64 rows (Q_i, dO_i, and the per-row statistics) of every query head that
// shares the K/V head through a ring, so dK and dV sum over the group.
// Per query block, on the tensor core (M = 128 everywhere):
//   S^T   = K Q_i^T            (128 keys x 64 queries, contraction over all of d)
//   dP^T  = V dO_i^T
//   P^T   = exp2(S^T*c - L2_i)  and  dS^T = P^T o (dP^T - D_i)   (row warps)
//   dV_h += P^T dO_i[:, h]      dK_h += dS^T Q_i[:, h]           (A from tensor memory)
//   dQ^T_h = K[:, h]^T dS^T     (128 head-dim rows x 64 queries)
// dQ^T sits in tensor memory with one lane per head-dimension column, and the
// fp32 accumulator in global memory is kept transposed too ([BH, d, Npad]), so
// each drain thread owns one contiguous run of 64 queries.  The four drain
// warps write the tile with 16-byte stores into a swizzled shared staging
// buffer and one thread adds it to the accumulator with two bulk tensor
// reduce-adds (the L2 does the adds).  For d = 128 the staging buffer is a
// buffer of its own.  For d = 256 there is no room for one: the tile (32 KB)
// goes into the step's dO buffer, which no product reads any more once the
// step's dQ^T is complete, and a reduce warp issues the reduce-adds and then
// hands the dO buffer back to the producer.  Q and dO then have barriers of
// their own, so that Q buffers go back to the producer as soon as the
// products have read them.
// With d = 256 the two halves of a key block are separate work items; both
// recompute S^T and dP^T (the price of fitting dK and dV in tensor memory).
//
// Recomputation of P from the saved statistic: "注意力为什么受限于显存带宽：用
// 算术强度与分块把 FlashAttention 推导清楚" section 八; "4. FlashAttention 深度
// 剖析" section 4.3.4.  Gradient formulas: chain rule through the row softmax.
//
// Warps: 0 TMA producer; 1 issuer A (S^T, dP^T; owns tensor memory); 2
// issuer B (dV, dK, dQ^T); 3..10 key-row warps, two per sub-partition, one
// per 32-query half (P^T, dS^T, dK/dV epilogue); 11..14 dQ drain warps; 15
// (d = 256) the reduce warp.  A
// tcgen05.mma instruction holds its issuing warp for about 100 cycles here,
// longer than the tensor core needs for these shapes, so the products of a
// step are split over two issuer warps.  (A third issuer for dP^T measured
// slower: products that run ahead queue in front of issuer B's.)
// Tensor memory columns: NSB S buffers (S^T of a step, then its P^T as bf16),
// NSB dP buffers (dP^T, then dS^T as bf16, then the step's dQ^T), dV_h
// [256,384), dK_h [384,512); NSB = 2 for d = 128, and for d = 256 one of each
// plus V in [128,256), written there by the row warps at each key block,
// which frees the shared memory for a second Q/dO stage.
// Issuer A writes S buffer b again once dV has read P^T out of it (dv_done)
// and dP buffer b once the drain has read dQ^T out of it (dq_free), and
// issues dP^T(g) before S^T(g+1), so that the row warps can compute the next
// P^T while dQ^T(g) is in flight.  Within one issuer the tensor core keeps
// issue order, which orders dQ^T(g) after dK(g)'s reads of dS^T(g) in the
// same columns.
#include <cstring>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_bwd_common.cuh"

namespace fa {
namespace {

using namespace ptx;

template <int D>
struct DtCfg {
  static constexpr int NCH = D / 64;
  static constexpr int NSPLIT = D / DH;
  static constexpr int KV_BYTES = NCH * KCH;
  static constexpr int Q_BYTES = NCH * QCH;
  // d = 256: V lives in tensor memory (the A operand of dP^T), which frees
  // its 64 KB of shared memory for a second Q/dO stage and leaves tensor
  // memory for one S and one dP buffer.
  static constexpr bool V_TMEM = (D == 256);
  static constexpr int STAGES = D == 128 ? 3 : 2;
  static constexpr int NSB = D == 128 ? 2 : 1;       // S and dP buffers
  // dQ^T goes to global memory as bulk reduce-adds of a 64 x 128 fp32 tile
  // staged in shared memory: a buffer of its own at d = 128, the step's dO
  // buffer at d = 256 (STAGE_IN_DO; Q and dO then have separate barriers and
  // a reduce warp returns the dO buffer once the reduce-adds have read it).
  static constexpr bool STAGE_IN_DO = (D == 256);
  static constexpr int THREADS = kThreads + (STAGE_IN_DO ? 32 : 0);
  // NSB S buffers of 64 columns from TM_S: S^T of a step, then P^T (bf16
  // pairs in columns [0,16) and [32,48), see pcol).  NSB dP buffers from
  // TM_DP: dP^T, then dS^T (bf16, same columns), then dQ^T.  d = 256: V
  // rows (bf16 pairs, 128 columns) from TM_V.  dV [256,384), dK [384,512).
  static constexpr uint32_t TM_S = 0, TM_DP = 64 * NSB, TM_V = 128;
  static constexpr uint32_t TM_DV = 256, TM_DK = 384;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int V_SMEM_BYTES = V_TMEM ? 16 : KV_BYTES;
  static_assert(!V_TMEM || (TM_DP + 64 * NSB <= TM_V && TM_V + D / 2 <= TM_DV),
                "tensor-memory columns overlap");
};

template <int D>
struct DtSmem {
  alignas(1024) uint8_t k[DtCfg<D>::KV_BYTES];
  alignas(1024) uint8_t q[DtCfg<D>::STAGES][DtCfg<D>::Q_BYTES];
  alignas(1024) uint8_t dO[DtCfg<D>::STAGES][DtCfg<D>::Q_BYTES];
  alignas(1024) uint8_t ds[2][KCH];              // dS^T bf16, 128 keys x 64 queries, double buffer
  alignas(DtCfg<D>::V_TMEM ? 16 : 1024) uint8_t v[DtCfg<D>::V_SMEM_BYTES];
  alignas(DtCfg<D>::STAGE_IN_DO ? 16 : 1024) float dq_stage[DtCfg<D>::STAGE_IN_DO ? 4 : BQ * DH];   // dQ^T tile, 2 x [d][32 queries]
  alignas(16) float lse2[DtCfg<D>::STAGES][BQ];
  alignas(16) float delta[DtCfg<D>::STAGES][BQ];
  uint64_t kv_full, kv_empty;
  uint64_t q_full[DtCfg<D>::STAGES], q_empty[DtCfg<D>::STAGES];
  // STAGE_IN_DO: dO loaded (do_full), dO buffer free again (do_empty, after the
  // reduce-adds of the dQ^T tile staged in it have read it), tile staged (stg_full)
  uint64_t do_full[DtCfg<D>::STAGES], do_empty[DtCfg<D>::STAGES], stg_full[DtCfg<D>::STAGES];
  // per tensor-memory buffer (g % NSB) or per shared dS buffer (g & 1)
  uint64_t s_full[2], p_full[2], dp_full[2], ds_full[2], ds_free[2];
  uint64_t dq_full[2], dq_free[2], acc_full, acc_free;
  uint64_t dv_done[2];              // cross-issuer: P^T of a step consumed
  uint64_t v_full, v_free;          // d = 256: V rows written to / read from tensor memory
  uint64_t mma_done_b;
  uint64_t stage_full, stage_free;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

// 227 KB of dynamic shared memory per block on sm_103a
static_assert(sizeof(DtSmem<128>) <= 232448 && sizeof(DtSmem<256>) <= 232448,
              "shared-memory layout exceeds the per-block limit");

// BS: the launch carries a block mask (its own instantiation, so that the
// kernel without one keeps the plain step walk).
template <int D, bool BS>
__global__ void __launch_bounds__(kRegThreads, 1) bwd_dt_kernel(const __grid_constant__ BwdParams p,
                                                                 const __grid_constant__ TailTable tail) {
  using C = DtCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
  const uintptr_t aligned = (raw + 1023) & ~static_cast<uintptr_t>(1023);
  if (aligned - raw + sizeof(DtSmem<D>) > dynamic_smem_size()) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, status_code(kSiteSmemLayout));
    return;
  }
  DtSmem<D>& sm = *reinterpret_cast<DtSmem<D>*>(aligned);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  volatile int* abort = &sm.abort;

  if (threadIdx.x == 0) {
    sm.abort = 0;
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 2);             // both MMA issuers read K (and A reads V)
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 2);         // both MMA issuers read the stage
      mbar_init(&sm.do_full[s], 1);
      mbar_init(&sm.do_empty[s], 1);        // the reduce warp
      mbar_init(&sm.stg_full[s], 4);        // the drain warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.p_full[b], kRowWarps);
      mbar_init(&sm.dp_full[b], 1);
      mbar_init(&sm.ds_full[b], kRowWarps);
      mbar_init(&sm.ds_free[b], 1);
      mbar_init(&sm.dv_done[b], 1);
      mbar_init(&sm.dq_full[b], 1);
      mbar_init(&sm.dq_free[b], 4);
    }
    mbar_init(&sm.mma_done_b, 1);
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_free, kRowWarps);
    mbar_init(&sm.v_full, kRowWarps);
    mbar_init(&sm.v_free, 1);
    mbar_init(&sm.stage_full, 4);
    mbar_init(&sm.stage_free, 1);
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
  const DtSched sched(p.B * p.H_kv, p.N, p.causal, C::NSPLIT, tail.heads,
                      BS ? p.cost_order : nullptr);
  const int G = p.H / p.H_kv;                     // query heads per K/V head

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // lane 0: K, V and the Q stages; with STAGE_IN_DO, lane 1 loads the dO
    // stages on their own barriers (lane 0 loads both otherwise)
    const bool dlane = C::STAGE_IN_DO && lane == 1;
    if (lane == 0 || dlane) {
      if (!dlane) {
        prefetch_tmap(&p.tq);
        prefetch_tmap(&p.tk);
        prefetch_tmap(&p.tv);
      }
      prefetch_tmap(&p.tdo);
      uint32_t w_it = 0, g = 0;
      bool ok = true;
      DtIter it{static_cast<int>(blockIdx.x), 0, 0};
      for (int kvbh, h, n; ok && sched.next(tail, it, kvbh, h, n);) {
        {
          int i0, i1;
          dt_range(p, n, dt_len(p, kvbh), i0, i1);
          const StepMask sk{BS ? p.block_mask + n : nullptr, p.bm_t, BK / BQ};
          const int nst = count_steps(sk, i0, i1);
          if (nst == 0) i1 = i0;
          if (i0 >= i1) continue;
          if (!dlane) {
            if (!mbar_wait(&sm.kv_empty, (w_it & 1) ^ 1, abort, kWaitTimeoutNs)) {
              record_failure(p.status, abort, kSiteProdKV);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sm.kv_full, (C::V_TMEM ? 1 : 2) * C::KV_BYTES);
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
              tma_load_3d(sm.k + c * KCH, &p.tk, &sm.kv_full, 64 * c, n * BK, kvbh);
              if constexpr (!C::V_TMEM)
                tma_load_3d(sm.v + c * KCH, &p.tv, &sm.kv_full, 64 * c, n * BK, kvbh);
            }
            ++w_it;
          }
          StepWalk wk(i0, i1, q_head_of(kvbh, 0, p.H, p.H_kv), sk);
          for (int s = 0; s < nst * G; ++s, wk.next()) {
            const int i = wk.i;
            const int bh = wk.bh;
            const int st = g % C::STAGES;
            const size_t roff = static_cast<size_t>(bh) * p.Npad + static_cast<size_t>(i) * BQ;
            if (dlane) {
              // dO and D of the step, once the reduce-adds of the dQ^T tile
              // staged in this buffer STAGES steps ago have read it
              if (!mbar_wait(&sm.do_empty[st], ((g / C::STAGES) & 1) ^ 1, abort, kWaitTimeoutNs)) {
                record_failure(p.status, abort, kSiteProdDo);
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&sm.do_full[st], C::Q_BYTES + BQ * 4);
#pragma unroll
              for (int c = 0; c < C::NCH; ++c)
                tma_load_3d(sm.dO[st] + c * QCH, &p.tdo, &sm.do_full[st], 64 * c, i * BQ, bh);
              bulk_load(sm.delta[st], p.delta + roff, BQ * 4, &sm.do_full[st]);
              ++g;
              continue;
            }
            if (!mbar_wait(&sm.q_empty[st], ((g / C::STAGES) & 1) ^ 1, abort, kWaitTimeoutNs)) {
              record_failure(p.status, abort, kSiteProdQ);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sm.q_full[st], (C::STAGE_IN_DO ? 1 : 2) * (C::Q_BYTES + BQ * 4));
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
              tma_load_3d(sm.q[st] + c * QCH, &p.tq, &sm.q_full[st], 64 * c, i * BQ, bh);
              if constexpr (!C::STAGE_IN_DO)
                tma_load_3d(sm.dO[st] + c * QCH, &p.tdo, &sm.q_full[st], 64 * c, i * BQ, bh);
            }
            bulk_load(sm.lse2[st], p.lse2 + roff, BQ * 4, &sm.q_full[st]);
            if constexpr (!C::STAGE_IN_DO)
              bulk_load(sm.delta[st], p.delta + roff, BQ * 4, &sm.q_full[st]);
            ++g;
          }
        }
      }
      // no copy may still be landing in shared memory when the CTA exits
      if (w_it > 0 && !mbar_wait(&sm.kv_full, (w_it - 1) & 1, nullptr, kWaitTimeoutNs))
        record_failure(p.status, abort, kSiteDtDrain);
      for (int s = 0; s < C::STAGES; ++s) {
        if (g > static_cast<uint32_t>(s)) {
          const uint32_t nph = (g - 1 - s) / C::STAGES;
          if (!mbar_wait(dlane ? &sm.do_full[s] : &sm.q_full[s], nph & 1, nullptr, kWaitTimeoutNs))
            record_failure(p.status, abort, kSiteDtDrain);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ issuer A
    // S^T(g) into S buffer g&1 once the drain has read dQ^T(g-2) out of it;
    // dP^T(g) into dP buffer g&1 once dK(g-2) has read dS^T(g-2).  Runs
    // ahead of the row warps as far as the Q ring and the two buffers allow.
    {
      constexpr uint32_t kIdS = idesc_bf16_f32(BK, BQ, 0, 0);      // S^T, dP^T
      const uint64_t dK0 = sdesc_sw128(smem_u32(sm.k), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sm.v), 16, 1024);
      uint32_t w_it = 0, g = 0;
      bool ok = true;
      DtIter it{static_cast<int>(blockIdx.x), 0, 0};
      for (int kvbh, h, n; ok && sched.next(tail, it, kvbh, h, n);) {
        {
          int i0, i1;
          dt_range(p, n, dt_len(p, kvbh), i0, i1);
          const StepMask sk{BS ? p.block_mask + n : nullptr, p.bm_t, BK / BQ};
          const int nst = count_steps(sk, i0, i1);
          if (nst == 0) i1 = i0;
          if (i0 >= i1) continue;
          const int nsteps = nst * G;
          if (!mbar_wait_warp(&sm.kv_full, w_it & 1, abort, kWaitTimeoutNs)) {
            issuer_fail(p.status, abort, lane, kSiteMmaKV);
            ok = false;
            break;
          }
          // S^T(gg) = K Q^T into S buffer gg%NSB once dV(gg-NSB) has read
          // P^T(gg-NSB) out of it
          auto issue_s = [&](uint32_t gg) -> bool {
            const uint32_t b = gg % C::NSB;
            const uint32_t ph = (gg / C::NSB) & 1;
            const int st = gg % C::STAGES;
            if (gg >= C::NSB && !mbar_wait_warp(&sm.dv_done[b], ph ^ 1, abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaP);
              return false;
            }
            if (!mbar_wait_warp(&sm.q_full[st], (gg / C::STAGES) & 1, abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaQ);
              return false;
            }
            tc_fence_after_sync();
            const uint64_t dq = sdesc_sw128(smem_u32(sm.q[st]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_bf16_ss_w(tmem + C::TM_S + 64 * b, dK0 + (((kk / 4) * KCH + (kk % 4) * 32) >> 4),
                            dq + (((kk / 4) * QCH + (kk % 4) * 32) >> 4), kIdS, kk > 0 ? 1u : 0u);
            mma_commit_w(&sm.s_full[b]);
            if constexpr (C::STAGE_IN_DO) mma_commit_w(&sm.q_empty[st]);   // A's reads of Q(gg)
            return true;
          };
          // dP^T(gg) = V dO^T into dP buffer gg%NSB once the drain has read
          // dQ^T(gg-NSB) out of it (which also means dK(gg-NSB) has read
          // dS^T(gg-NSB)).  d = 256: V (A operand) from tensor memory.
          auto issue_dp = [&](uint32_t gg) -> bool {
            const uint32_t b = gg % C::NSB;
            const uint32_t ph = (gg / C::NSB) & 1;
            const int st = gg % C::STAGES;
            if (gg >= C::NSB && !mbar_wait_warp(&sm.dq_free[b], ph ^ 1, abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaDq);
              return false;
            }
            if (C::STAGE_IN_DO &&
                !mbar_wait_warp(&sm.do_full[st], (gg / C::STAGES) & 1, abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaDo);
              return false;
            }
            tc_fence_after_sync();
            const uint64_t ddo = sdesc_sw128(smem_u32(sm.dO[st]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t bk = ddo + (((kk / 4) * QCH + (kk % 4) * 32) >> 4);
              if constexpr (C::V_TMEM)
                mma_bf16_ts_w(tmem + C::TM_DP + 64 * b, tmem + C::TM_V + 8 * kk, bk, kIdS,
                              kk > 0 ? 1u : 0u);
              else
                mma_bf16_ss_w(tmem + C::TM_DP + 64 * b, dV0 + (((kk / 4) * KCH + (kk % 4) * 32) >> 4),
                              bk, kIdS, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&sm.dp_full[b]);
            if constexpr (!C::STAGE_IN_DO)
              mma_commit_w(&sm.q_empty[st]);        // A's reads of this stage are done
            return true;
          };
          // dP^T(g) goes ahead of S^T(g+1): the row warps need it first
          ok = issue_s(g);
          if (ok && C::V_TMEM && !mbar_wait_warp(&sm.v_full, w_it & 1, abort, kWaitTimeoutNs)) {
            issuer_fail(p.status, abort, lane, kSiteMmaV);
            ok = false;
          }
          for (int s = 0; ok && s < nsteps; ++s, ++g) {
            ok = issue_dp(g) && (s + 1 == nsteps || issue_s(g + 1));
          }
          if (!ok) break;
          mma_commit_w(&sm.kv_empty);               // A's reads of K and V are done
          if constexpr (C::V_TMEM) mma_commit_w(&sm.v_free);   // ... and of V in tensor memory
          ++w_it;
        }
      }
      // every tcgen05 op issued by this thread must finish before exit
      mma_commit_w(&sm.mma_done);
      if (!mbar_wait_warp(&sm.mma_done, 0, nullptr, kWaitTimeoutNs))
        issuer_fail(p.status, abort, lane, kSiteDtDrain);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ issuer B
    {
      constexpr uint32_t kIdAcc = idesc_bf16_f32(BK, DH, 0, 1);    // dV, dK (B MN-major)
      constexpr uint32_t kIdDq = idesc_bf16_f32(DH, BQ, 1, 1);     // dQ^T (A, B MN-major)
      uint32_t w_it = 0, g = 0;
      bool ok = true;
      auto fail = [&](int site) {
        issuer_fail(p.status, abort, lane, site);
        ok = false;
      };
      DtIter it{static_cast<int>(blockIdx.x), 0, 0};
      for (int kvbh, h, n; ok && sched.next(tail, it, kvbh, h, n);) {
        // K[:, h] as the MN-major A operand of dQ^T: 64-column chunks 2h, 2h+1
        const uint64_t dKmn = sdesc_sw128(smem_u32(sm.k) + 2 * h * KCH, KCH, 1024);
        {
          int i0, i1;
          dt_range(p, n, dt_len(p, kvbh), i0, i1);
          const StepMask sk{BS ? p.block_mask + n : nullptr, p.bm_t, BK / BQ};
          const int nst = count_steps(sk, i0, i1);
          if (nst == 0) i1 = i0;
          if (i0 >= i1) continue;
          const int nsteps = nst * G;
          for (int s = 0; s < nsteps; ++s, ++g) {
            const int st = g % C::STAGES;
            const uint32_t b = g % C::NSB;          // tensor-memory S / dP buffer
            const uint32_t ph = (g / C::NSB) & 1;
            const uint32_t bs = g & 1;              // shared dS buffer
            const bool first = (s == 0);
            const bool last = (s + 1 == nsteps);
            // dV_h += P^T dO_i[:, h]
            if (!mbar_wait_warp(&sm.p_full[b], ph, abort, kWaitTimeoutNs)) {
              fail(kSiteMmaP);
              break;
            }
            if (first && !mbar_wait_warp(&sm.acc_free, (w_it & 1) ^ 1, abort, kWaitTimeoutNs)) {
              fail(kSiteMmaAcc);
              break;
            }
            if (C::STAGE_IN_DO &&
                !mbar_wait_warp(&sm.do_full[st], (g / C::STAGES) & 1, abort, kWaitTimeoutNs)) {
              fail(kSiteMmaDo);
              break;
            }
            tc_fence_after_sync();
            const uint64_t dOmn = sdesc_sw128(smem_u32(sm.dO[st]) + 2 * h * QCH, QCH, 1024);
            const uint64_t dQmn = sdesc_sw128(smem_u32(sm.q[st]) + 2 * h * QCH, QCH, 1024);
#pragma unroll
            for (int kk = 0; kk < BQ / 16; ++kk)
              mma_bf16_ts_w(tmem + C::TM_DV, tmem + C::TM_S + 64 * b + pcol(kk),
                          dOmn + ((kk * 2048) >> 4), kIdAcc, (first && kk == 0) ? 0u : 1u);
            mma_commit_w(&sm.dv_done[b]);
            // dK_h += dS^T Q_i[:, h]
            if (!mbar_wait_warp(&sm.ds_full[bs], (g >> 1) & 1, abort, kWaitTimeoutNs)) {
              fail(kSiteMmaDs);
              break;
            }
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < BQ / 16; ++kk)
              mma_bf16_ts_w(tmem + C::TM_DK, tmem + C::TM_DP + 64 * b + pcol(kk),
                          dQmn + ((kk * 2048) >> 4), kIdAcc, (first && kk == 0) ? 0u : 1u);
            mma_commit_w(&sm.q_empty[st]);          // B's reads of this stage are done
            if (last) mma_commit_w(&sm.acc_full);
            // dQ^T_h = K[:, h]^T dS^T into dP buffer b: issued after dK(g) by
            // this thread, so it runs after dK(g) has read dS^T(g) there
            const uint64_t dDS = sdesc_sw128(smem_u32(sm.ds[bs]), KCH, 1024);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_bf16_ss_w(tmem + C::TM_DP + 64 * b, dKmn + ((kk * 2048) >> 4),
                          dDS + ((kk * 2048) >> 4), kIdDq, kk > 0 ? 1u : 0u);
            mma_commit_w(&sm.dq_full[b]);
            mma_commit_w(&sm.ds_free[bs]);
            if (last) mma_commit_w(&sm.kv_empty);   // B's reads of K are done
          }
          if (!ok) break;
          ++w_it;
        }
      }
      mma_commit_w(&sm.mma_done_b);
      if (!mbar_wait_warp(&sm.mma_done_b, 0, nullptr, kWaitTimeoutNs))
        issuer_fail(p.status, abort, lane, kSiteDtDrain);
    }
    __syncwarp();
  } else if (warp < 3 + kRowWarps) {
    // ------------------------------------------------------------ key-row warps
    // Warp w owns key rows 32*(w%4) .. +31 (its tensor-memory lanes) and the
    // query half hh = (w-3)/4: columns 32*hh .. 32*hh+31 of each step, and
    // head-dimension columns 64*hh .. 64*hh+63 of the dK/dV epilogue.
    const int quarter = warp & 3;
    const int hh = (warp - 3) >> 2;
    const int r = quarter * 32 + lane;            // key row of the block = tensor-memory lane
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c2 = p.scale_log2;
    __nv_bfloat16* dk_out = static_cast<__nv_bfloat16*>(p.dk);
    __nv_bfloat16* dv_out = static_cast<__nv_bfloat16*>(p.dv);
    // Each thread stores its own key row; 32-byte stores (when both outputs
    // are 32-byte aligned) halve the lines a warp store touches, which is
    // what the dK/dV epilogue at the end of a key block waits on.
    const bool st32 = ((reinterpret_cast<uintptr_t>(dk_out) | reinterpret_cast<uintptr_t>(dv_out)) &
                       31u) == 0;
    uint32_t w_it = 0, g = 0;
    bool ok = true;
    DtIter it{static_cast<int>(blockIdx.x), 0, 0};
    for (int kvbh, h, n; ok && sched.next(tail, it, kvbh, h, n);) {
      {
        const int len = dt_len(p, kvbh);
        int i0, i1;
        dt_range(p, n, len, i0, i1);
        const StepMask sk{BS ? p.block_mask + n : nullptr, p.bm_t, BK / BQ};
        const int nst = count_steps(sk, i0, i1);
        if (nst == 0) i1 = i0;
        const int key = n * BK + r;
        const size_t out_off = (static_cast<size_t>(kvbh) * p.N + key) * D + h * DH + 64 * hh;
        if (i0 >= i1) {
          // key block entirely past the sequence: zero gradients
          if (key < p.N) {
            uint4* a = reinterpret_cast<uint4*>(dk_out + out_off);
            uint4* bq = reinterpret_cast<uint4*>(dv_out + out_off);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              a[t] = make_uint4(0, 0, 0, 0);
              bq[t] = make_uint4(0, 0, 0, 0);
            }
          }
          continue;
        }
        if constexpr (C::V_TMEM) {
          // V rows of this key block into tensor memory, the A operand of
          // dP^T: row r, head-dimension elements 128*hh .. +127 as bf16 pairs in
          // columns 64*hh .. +63, once the last dP^T of the previous item is done
          if (!warp_wait(&sm.v_free, (w_it & 1) ^ 1, abort)) {
            if (lane == 0) record_failure(p.status, abort, kSiteRowV);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint4* vrow = reinterpret_cast<const uint4*>(
              static_cast<const __nv_bfloat16*>(p.v) + (static_cast<size_t>(kvbh) * p.N + key) * D +
              128 * hh);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t vr[32];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const uint4 x = key < p.N ? __ldg(vrow + 8 * c + t) : make_uint4(0, 0, 0, 0);
              vr[4 * t] = x.x;
              vr[4 * t + 1] = x.y;
              vr[4 * t + 2] = x.z;
              vr[4 * t + 3] = x.w;
            }
            tmem_st_x32(t_lane + C::TM_V + 64 * hh + 32 * c, vr);
          }
          tmem_wait_st();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.v_full);
        }
        StepWalk wk(i0, i1, 0, sk);
        for (int s = 0; s < nst * G; ++s, ++g, wk.next()) {
          const int i = wk.i;
          const int st = g % C::STAGES;
          const int q0 = i * BQ;
          const uint32_t tb = g % C::NSB;                          // tensor-memory S / dP buffer
          const uint32_t tph = (g / C::NSB) & 1;
          // ---- P^T = exp2(S^T * c - L2), masked; bf16 copy back to tensor memory
          const uint32_t t_s = t_lane + C::TM_S + 64 * tb;         // this step's S^T buffer
          if (!warp_wait(&sm.s_full[tb], tph, abort)) {
            if (lane == 0) record_failure(p.status, abort, kSiteRowS);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const bool need_mask = (n * BK + BK > len) || (n * BK + BK - 1 > q0 + p.wr) ||
                                 (n * BK < q0 + BQ - 1 - p.wl);
          // visible columns c (query q = q0 + 32*hh + c) of this key row:
          // [c_lo, c_hi], the queries whose window [q - wl, q + wr] holds the
          // key; none when the key is past len
          const int c_lo = key - p.wr - q0 - 32 * hh;
          const int c_hi = (key < len) ? key + p.wl - q0 - 32 * hh : -1;
          float pr[32];
          const uint64_t c2x2 = f2_make(c2, c2);
          {
            uint32_t sr[32];
            tmem_ld_x32(t_s + 32 * hh, sr);
            tmem_wait_ld();
            reg_fence<32>(sr);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float4 l4 = reinterpret_cast<const float4*>(sm.lse2[st])[8 * hh + t];
              float a[4];
              f2_split(f2_fma(f2_make(__uint_as_float(sr[4 * t]), __uint_as_float(sr[4 * t + 1])),
                              c2x2, f2_make(-l4.x, -l4.y)),
                       a[0], a[1]);
              f2_split(f2_fma(f2_make(__uint_as_float(sr[4 * t + 2]), __uint_as_float(sr[4 * t + 3])),
                              c2x2, f2_make(-l4.z, -l4.w)),
                       a[2], a[3]);
#pragma unroll
              for (int e = 0; e < 4; ++e) pr[4 * t + e] = ex2_approx(a[e]);
            }
            if (need_mask) {      // diagonal and boundary steps only
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (c < c_lo || c > c_hi) pr[c] = 0.f;
            }
            uint32_t pk[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) pk[t] = pack_bf16x2(pr[2 * t], pr[2 * t + 1]);
            // packed over the first 16 of this half's own 32 columns: the other
            // half's warp may still be reading its fp32 columns
            tmem_st_x16(t_s + 32 * hh, pk);
          }
          tmem_wait_st();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.p_full[tb]);
          // ---- dS^T = P^T o (dP^T - D)
          const uint32_t t_dp = t_lane + C::TM_DP + 64 * tb;       // this step's dP^T buffer
          if (!warp_wait(&sm.dp_full[tb], tph, abort)) {
            if (lane == 0) record_failure(p.status, abort, kSiteRowDp);
            ok = false;
            break;
          }
          // the shared copy (B operand of dQ^T) goes to buffer g & 1 once the
          // dQ^T that last read that buffer has finished
          const uint32_t b = g & 1;
          if (!warp_wait(&sm.ds_free[b], ((g >> 1) & 1) ^ 1, abort)) {
            if (lane == 0) record_failure(p.status, abort, kSiteRowDsFree);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          uint8_t* rowp = sm.ds[b] + r * 128;
          {
            uint32_t sr[32];
            tmem_ld_x32(t_dp + 32 * hh, sr);
            tmem_wait_ld();
            reg_fence<32>(sr);
            uint32_t pk[16];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float4 d4 = reinterpret_cast<const float4*>(sm.delta[st])[8 * hh + t];
              const int c = 4 * t;
              float d0, d1, d2, d3;
              f2_split(f2_mul(f2_add(f2_make(__uint_as_float(sr[4 * t]), __uint_as_float(sr[4 * t + 1])),
                                     f2_make(-d4.x, -d4.y)),
                              f2_make(pr[c], pr[c + 1])),
                       d0, d1);
              f2_split(f2_mul(f2_add(f2_make(__uint_as_float(sr[4 * t + 2]), __uint_as_float(sr[4 * t + 3])),
                                     f2_make(-d4.z, -d4.w)),
                              f2_make(pr[c + 2], pr[c + 3])),
                       d2, d3);
              pk[2 * t] = pack_bf16x2(d0, d1);
              pk[2 * t + 1] = pack_bf16x2(d2, d3);
            }
            tmem_st_x16(t_dp + 32 * hh, pk);
            // row = key r, 64 queries = 8 units of 16 bytes, XOR-swizzled by (r & 7)
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int unit = 4 * hh + t;
              *reinterpret_cast<uint4*>(rowp + ((unit ^ (r & 7)) << 4)) =
                  make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
            }
          }
          fence_proxy_async_smem();
          tmem_wait_st();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.ds_full[g & 1]);
        }
        if (!ok) break;
        // ---- dK_h, dV_h rows of this key block, head-dimension columns of half hh
        if (!warp_wait(&sm.acc_full, w_it & 1, abort)) {
          if (lane == 0) record_failure(p.status, abort, kSiteRowAcc);
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll 1
        for (int c4 = 0; c4 < 2; ++c4) {
          uint32_t a[32], bb[32];
          tmem_ld_x32(t_lane + C::TM_DV + 64 * hh + 32 * c4, a);
          tmem_ld_x32(t_lane + C::TM_DK + 64 * hh + 32 * c4, bb);
          tmem_wait_ld();
          reg_fence<32>(a);
          reg_fence<32>(bb);
          if (key < p.N) {
            uint32_t pv[16], pkk[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              pv[t] = pack_bf16x2(__uint_as_float(a[2 * t]), __uint_as_float(a[2 * t + 1]));
              pkk[t] = pack_bf16x2(__uint_as_float(bb[2 * t]) * p.scale,
                                   __uint_as_float(bb[2 * t + 1]) * p.scale);
            }
            if (st32) {
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                st_global_v8(dv_out + out_off + 32 * c4 + 16 * t, pv + 8 * t);
                st_global_v8(dk_out + out_off + 32 * c4 + 16 * t, pkk + 8 * t);
              }
            } else {
              uint4* dvp = reinterpret_cast<uint4*>(dv_out + out_off + 32 * c4);
              uint4* dkp = reinterpret_cast<uint4*>(dk_out + out_off + 32 * c4);
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                dvp[t] = make_uint4(pv[4 * t], pv[4 * t + 1], pv[4 * t + 2], pv[4 * t + 3]);
                dkp[t] = make_uint4(pkk[4 * t], pkk[4 * t + 1], pkk[4 * t + 2], pkk[4 * t + 3]);
              }
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_free);
        ++w_it;
      }
    }
  } else if (warp < kDrainWarp0 + 4) {
    // ------------------------------------------------------------ dQ drain warps
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;            // head-dimension column within the half
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    // issues the bulk reduce-adds (d = 128; at d = 256 the reduce warp does)
    const bool issuer = !C::STAGE_IN_DO && warp == kDrainWarp0 && lane == 0;
    if (issuer) prefetch_tmap(&p.tdq);
    uint32_t g = 0;
    bool ok = true;
    DtIter it{static_cast<int>(blockIdx.x), 0, 0};
    for (int kvbh, h, n; ok && sched.next(tail, it, kvbh, h, n);) {
      {
        int i0, i1;
        dt_range(p, n, dt_len(p, kvbh), i0, i1);
        const StepMask sk{BS ? p.block_mask + n : nullptr, p.bm_t, BK / BQ};
        const int nst = count_steps(sk, i0, i1);
        if (nst == 0) i1 = i0;
        StepWalk wk(i0, i1, q_head_of(kvbh, 0, p.H, p.H_kv), sk);
        for (int s = 0; s < nst * G; ++s, ++g, wk.next()) {
          const int i = wk.i;
          const int bh = wk.bh;
          const uint32_t tb = g % C::NSB;
          if (!warp_wait(&sm.dq_full[tb], (g / C::NSB) & 1, abort)) {
            if (lane == 0) record_failure(p.status, abort, kSiteDrainDq);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const int q0 = i * BQ;
          uint32_t v0[32], v1[32];
          tmem_ld_x32(t_lane + C::TM_DP + 64 * tb, v0);            // dQ^T(g) sits in dP buffer tb
          tmem_ld_x32(t_lane + C::TM_DP + 64 * tb + 32, v1);
          tmem_wait_ld();
          reg_fence<32>(v0);
          reg_fence<32>(v1);
          // the whole tile is in registers: tensor memory is free for the next dQ^T
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.dq_free[tb]);
          if constexpr (C::STAGE_IN_DO) {
            // staging in the step's dO buffer (no product reads it once dQ^T
            // is complete): the same two swizzled boxes, 16 KB apart
            const int st = g % C::STAGES;
            uint4* row0 = reinterpret_cast<uint4*>(sm.dO[st]) + r * 8;
            uint4* row1 = row0 + DH * 8;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              row0[j ^ (r & 7)] = make_uint4(v0[4 * j], v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              row1[j ^ (r & 7)] = make_uint4(v1[4 * j], v1[4 * j + 1], v1[4 * j + 2], v1[4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.stg_full[st]);
          } else {
            // staging: two boxes of [128 columns][32 queries] fp32 in the
            // 128-byte swizzle of the tensor map; this thread owns row r of
            // each and writes it as eight 16-byte chunks, chunk j at j ^ (r & 7)
            // (conflict-free: eight consecutive rows cover all 32 banks)
            if (!warp_wait(&sm.stage_free, (g & 1) ^ 1, abort)) {
              if (lane == 0) record_failure(p.status, abort, kSiteStageFree);
              ok = false;
              break;
            }
            uint4* row0 = reinterpret_cast<uint4*>(sm.dq_stage) + r * 8;
            uint4* row1 = row0 + DH * 8;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              row0[j ^ (r & 7)] = make_uint4(v0[4 * j], v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              row1[j ^ (r & 7)] = make_uint4(v1[4 * j], v1[4 * j + 1], v1[4 * j + 2], v1[4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.stage_full);
            if (issuer) {
              if (!mbar_wait(&sm.stage_full, g & 1, abort, kWaitTimeoutNs)) {
                record_failure(p.status, abort, kSiteStageFull);
                ok = false;
              } else {
                // queries past N land in the padding up to Npad, never read
                tma_reduce_add_3d(&p.tdq, sm.dq_stage, q0, h * DH, bh);
                tma_reduce_add_3d(&p.tdq, sm.dq_stage + 32 * DH, q0 + 32, h * DH, bh);
                bulk_commit_group();
                bulk_wait_group_read<0>();
                mbar_arrive(&sm.stage_free);
              }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
          }
        }
      }
    }
    // every reduce-add must have landed before the CTA exits
    if (issuer) bulk_wait_group<0>();
  } else {
    // ------------------------------------------------------------ reduce warp (d = 256)
    // Adds each step's staged dQ^T tile to the accumulator with two bulk
    // tensor reduce-adds, then returns the dO buffer it was staged in.
    if (C::STAGE_IN_DO && lane == 0) {
      prefetch_tmap(&p.tdq);
      uint32_t g = 0;
      bool ok = true;
      DtIter it{static_cast<int>(blockIdx.x), 0, 0};
      for (int kvbh, h, n; ok && sched.next(tail, it, kvbh, h, n);) {
        int i0, i1;
        dt_range(p, n, dt_len(p, kvbh), i0, i1);
        const StepMask sk{BS ? p.block_mask + n : nullptr, p.bm_t, BK / BQ};
        const int nst = count_steps(sk, i0, i1);
        if (nst == 0) i1 = i0;
        StepWalk wk(i0, i1, q_head_of(kvbh, 0, p.H, p.H_kv), sk);
        for (int s = 0; s < nst * G; ++s, ++g, wk.next()) {
          const int st = g % C::STAGES;
          if (!mbar_wait(&sm.stg_full[st], (g / C::STAGES) & 1, abort, kWaitTimeoutNs)) {
            record_failure(p.status, abort, kSiteStageFull);
            ok = false;
            break;
          }
          // queries past N land in the padding up to Npad, never read
          const float* box = reinterpret_cast<const float*>(sm.dO[st]);
          tma_reduce_add_3d(&p.tdq, box, wk.i * BQ, h * DH, wk.bh);
          tma_reduce_add_3d(&p.tdq, box + 32 * DH, wk.i * BQ + 32, h * DH, wk.bh);
          bulk_commit_group();
          bulk_wait_group_read<0>();
          mbar_arrive(&sm.do_empty[st]);
        }
      }
      // every reduce-add must have landed before the CTA exits
      bulk_wait_group<0>();
    }
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, DtCfg<D>::TM_COLS);
  }
}

template <int D, bool BS>
cudaError_t launch(const BwdParams& p, int num_sms, int max_smem, cudaStream_t stream) {
  const size_t smem = smem_request(sizeof(DtSmem<D>), max_smem);
  cudaError_t e = cudaFuncSetAttribute(bwd_dt_kernel<D, BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int T = (p.N + BK - 1) / BK;
  const int BH = p.B * p.H_kv;
  constexpr int NS = DtCfg<D>::NSPLIT;
  const long long per_bh = p.causal ? (T + 1) / 2 : T;
  long long units = static_cast<long long>(BH) * per_bh * NS;
  TailTable tail;
  tail.heads = 0;
  if (p.causal || (BS && p.block_mask_host && T == p.bm_t)) {
    // single key blocks in the tail: up to one CTA per block
    const long long blocks = static_cast<long long>(BH) * T * NS;
    const int g = static_cast<int>(blocks < num_sms ? blocks : num_sms);
    // the tail's K/V heads share their group's Q and dO through L2
    const long long qdo_bytes = 2ll * (p.H / p.H_kv) * p.N * D * 2;
    if (p.causal)
      plan_causal_tail(BH, T, NS, g, false, qdo_bytes, &tail);
    else                       // key blocks cost their computed query steps
      plan_mask_tail(p.block_mask_host, BH, T, NS, g, false, p.N, p.wl, p.wr, qdo_bytes, &tail);
    if (tail.heads > 0) units = g;
  }
  if (tail.heads == 0) std::memset(tail.item, 0xff, sizeof(tail.item));
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  bwd_dt_kernel<D, BS><<<grid, DtCfg<D>::THREADS, smem, stream>>>(p, tail);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main_dt(const BwdParams& p, int d, int num_sms, int max_smem,
                               cudaStream_t stream) {
  switch (d) {
    case 128:
      return p.block_mask ? launch<128, true>(p, num_sms, max_smem, stream)
                          : launch<128, false>(p, num_sms, max_smem, stream);
    case 256:
      return p.block_mask ? launch<256, true>(p, num_sms, max_smem, stream)
                          : launch<256, false>(p, num_sms, max_smem, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fa
