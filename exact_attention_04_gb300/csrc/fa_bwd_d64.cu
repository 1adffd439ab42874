// Backward main kernel for head dimension 64.
//
// Work item: (K/V head, block of 128 keys).  The CTA keeps K and V of its key
// block in shared memory and streams 128-row query blocks (Q_i, dO_i and the
// per-row statistics) of every query head that shares the K/V head, so dK and
// dV sum over the group.  Per query block, on the tensor core:
//   S^T  = K Q_i^T                   dP^T = V dO_i^T          (M = N = 128, K = 64)
//   P^T  = exp2(S^T*c - L2_i)        dS^T = P^T o (dP^T - D_i)      (row warps)
//   dV  += P^T dO_i                  dK  += dS^T Q_i          (A from tensor memory)
//   dQ_i = dS K                      (128 queries x 64, into columns of its own)
// Recomputation of P from the saved statistic: "注意力为什么受限于显存带宽：用
// 算术强度与分块把 FlashAttention 推导清楚" section 八; "4. FlashAttention 深度
// 剖析" section 4.3.4.  Gradient formulas: chain rule through the row softmax.
//
// Tensor memory (512 columns): S^T [0,128) (then P^T as bf16 pairs),
// dP^T [128,256) (then dS^T as bf16 pairs), dV [256,320), dK [320,384),
// dQ [384,448).  Two issuers keep the tensor core busy across steps: A issues
// S^T(g) once dV(g-1) has read P^T(g-1) and dP^T(g) once dK(g-1) has read
// dS^T(g-1); B issues dV(g), dK(g) and dQ(g).  The products of consecutive
// steps then interleave as dV(g-1) S(g) dK(g-1) dP(g) dQ(g-1) dV(g) ..., each
// waiting on work finished at least one product earlier.
//
// dQ of a step (fp32, 128 x 64 = 32 KB) leaves tensor memory through the row
// warps, which stage it in one of two shared buffers in the 128-byte swizzle
// of the accumulator's tensor map; a reduce warp adds it to the fp32
// accumulator ([BH, Npad, 64]) with two bulk tensor reduce-adds (the L2 does
// the adds) and frees the buffer once they have read it.
//
// Warps (20): 0 TMA producer (lane 0: K, V, Q; lane 1: dO); 1 issuer A (owns
// tensor memory); 2 issuer B; 3 reduce warp; 4..19 row warps, four per
// sub-partition.  Row warp (quarter q, j): tensor-memory lanes 32q .. 32q+31,
// i.e. key rows for S^T, dP^T, dV, dK and query rows for dQ; its share of a
// step is queries 32j .. 32j+31 (P^T, dS^T), dQ columns 16j .. 16j+15, and dK,
// dV columns 16j .. 16j+15.  Per step g a row warp computes P^T(g), then
// dS^T(g) into tensor memory (dK(g) may start), then takes its share of
// dQ(g-1) out of tensor memory into the staging, and only then copies dS(g)
// to shared memory, whose single buffer dQ(g-1) was reading.
// Issuers run converged and one elect.sync lane issues; within one issuer the
// tensor core keeps issue order.  Every wait is bounded: a wait that gives up
// records the site in the status word, raises the CTA's abort flag, and the
// kernel drains its copies and products and returns.
#include <cstring>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_bwd_common.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int SQ = 128;                 // queries per step
constexpr int SD = 64;                  // head dimension
constexpr int SCH = 128 * 128;          // a 128-row x 128-byte SW128 chunk (one 128 x 64 bf16 tile)
constexpr int kSRowWarps = 16;
constexpr int kSRowWarp0 = 4;
constexpr int kSThreads = 32 * (kSRowWarp0 + kSRowWarps);   // 20 warps
constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 320, TM_DQ = 384, TM_COLS = 512;

struct SSmem {
  alignas(1024) uint8_t k[SCH];
  alignas(1024) uint8_t v[SCH];
  alignas(1024) uint8_t q[2][SCH];
  alignas(1024) uint8_t dO[2][SCH];
  alignas(1024) uint8_t ds[2 * SCH];    // dS^T bf16: 128 keys x 128 queries, two 64-query chunks
  alignas(1024) uint8_t stage[2][2 * SCH];   // dQ fp32: two boxes of [128 rows][32 columns]
  alignas(16) float lse2[2][SQ];
  alignas(16) float delta[2][SQ];
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2], do_full[2], do_empty[2];
  // ds_tm: dS^T(g) is in tensor memory (dK(g) may start); ds_full: its copy
  // is in shared memory (dQ(g) may start)
  uint64_t s_full, p_full, dv_done, dp_full, ds_tm, ds_full, dk_done, dq_full, dq_free;
  uint64_t stg_full[2], stg_free[2];
  uint64_t acc_full, acc_free;
  uint64_t mma_done, mma_done_b;
  uint32_t tmem_base;
  int abort;
};

// 227 KB of dynamic shared memory per block on sm_103a
static_assert(sizeof(SSmem) <= 232448, "shared-memory layout exceeds the per-block limit");

// Column of the packed bf16 P^T / dS^T for K-step kk (16 queries) within its
// 128-column buffer: the warp of query quarter j packs queries 32j .. 32j+31
// over the first 16 of its own 32 columns.
__device__ __forceinline__ constexpr uint32_t scol(int kk) {
  return static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8);
}

// Query-block range [i0, i1) (blocks of 128) that key block n is visible to.
__device__ __forceinline__ void s_range(const BwdParams& p, int n, int len, int& i0, int& i1) {
  int q_lo, q_hi;
  visible_queries(n * BK, BK, len, p.N, p.wl, p.wr, q_lo, q_hi);
  if (q_hi <= q_lo) {
    i0 = i1 = 0;
    return;
  }
  i0 = q_lo / SQ;
  i1 = (q_hi + SQ - 1) / SQ;
}

// The steps of the item: (query head, query block) pairs, or none.
struct SItem {
  int i0, i1, nsteps;
  StepMask sk;
};

template <bool BS>
__device__ __forceinline__ SItem s_item(const BwdParams& p, int kvbh, int n, int G) {
  SItem w;
  s_range(p, n, dt_len(p, kvbh), w.i0, w.i1);
  w.sk = StepMask{BS ? p.block_mask + n : nullptr, p.bm_t, 1};
  const int nst = count_steps(w.sk, w.i0, w.i1);
  if (nst == 0) w.i1 = w.i0;
  w.nsteps = nst * G;
  return w;
}

template <bool BS>
__global__ void __launch_bounds__(kSThreads, 1) bwd_d64_kernel(const __grid_constant__ BwdParams p,
                                                               const __grid_constant__ TailTable tail) {
  extern __shared__ uint8_t smem_raw[];
  const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
  const uintptr_t aligned = (raw + 1023) & ~static_cast<uintptr_t>(1023);
  if (aligned - raw + sizeof(SSmem) > dynamic_smem_size()) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, status_code(kSiteSmemLayout));
    return;
  }
  SSmem& sm = *reinterpret_cast<SSmem*>(aligned);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  volatile int* abort = &sm.abort;

  if (threadIdx.x == 0) {
    sm.abort = 0;
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 2);             // issuer A (K, V) and issuer B (K)
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 2);         // A after S^T, B after dK (the row warps are past L2)
      mbar_init(&sm.do_full[s], 1);
      mbar_init(&sm.do_empty[s], 2);        // A after dP^T, B after dK (the row warps are past D)
      mbar_init(&sm.stg_full[s], kSRowWarps);
      mbar_init(&sm.stg_free[s], 1);        // the reduce warp
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.p_full, kSRowWarps);
    mbar_init(&sm.dv_done, 1);
    mbar_init(&sm.dp_full, 1);
    mbar_init(&sm.ds_tm, kSRowWarps);
    mbar_init(&sm.ds_full, kSRowWarps);
    mbar_init(&sm.dk_done, 1);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_free, kSRowWarps);
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_free, kSRowWarps);
    mbar_init(&sm.mma_done, 1);
    mbar_init(&sm.mma_done_b, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  const DtSched sched(p.B * p.H_kv, p.N, p.causal, 1, tail.heads, BS ? p.cost_order : nullptr);
  const int G = p.H / p.H_kv;                     // query heads per K/V head

  // Registers: the launch gives every thread 96.  The first warpgroup
  // (producer, issuers, reduce warp) needs far fewer, and the row warps
  // spill at 96, so the row warpgroups take what the first one gives back:
  // 128 x 64 + 512 x 104 = the launch's 640 x 96 = 61,440.
  static_assert(kSRowWarp0 == 4 && kSRowWarps % 4 == 0, "roles aligned to warpgroups");
  static_assert(128 * 64 + 32 * kSRowWarps * 104 <= kSThreads * 96, "register split");
  if (warp < kSRowWarp0) {
    setmaxnreg_dec<64>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      // lane 0: K, V and the Q stages (with L2); lane 1: the dO stages (with D)
      const bool dlane = lane == 1;
      if (lane < 2) {
        if (!dlane) {
          prefetch_tmap(&p.tq);
          prefetch_tmap(&p.tk);
          prefetch_tmap(&p.tv);
        } else {
          prefetch_tmap(&p.tdo);
        }
        uint32_t w_it = 0, g = 0;
        bool ok = true;
        DtIter it{static_cast<int>(blockIdx.x), 0, 0};
        for (int kvbh, h, n; ok && sched.next(tail, it, kvbh, h, n);) {
          const SItem wi = s_item<BS>(p, kvbh, n, G);
          if (wi.nsteps == 0) continue;
          if (!dlane) {
            if (!mbar_wait(&sm.kv_empty, (w_it & 1) ^ 1, abort, kWaitTimeoutNs)) {
              record_failure(p.status, abort, kSiteProdKV);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sm.kv_full, 2 * SCH);
            tma_load_3d(sm.k, &p.tk, &sm.kv_full, 0, n * BK, kvbh);
            tma_load_3d(sm.v, &p.tv, &sm.kv_full, 0, n * BK, kvbh);
            ++w_it;
          }
          StepWalk wk(wi.i0, wi.i1, q_head_of(kvbh, 0, p.H, p.H_kv), wi.sk);
          for (int s = 0; s < wi.nsteps; ++s, ++g, wk.next()) {
            const int st = g & 1;
            const uint32_t ph = ((g >> 1) & 1) ^ 1;
            const size_t roff = static_cast<size_t>(wk.bh) * p.Npad + static_cast<size_t>(wk.i) * SQ;
            uint64_t* empty = dlane ? &sm.do_empty[st] : &sm.q_empty[st];
            uint64_t* full = dlane ? &sm.do_full[st] : &sm.q_full[st];
            if (!mbar_wait(empty, ph, abort, kWaitTimeoutNs)) {
              record_failure(p.status, abort, dlane ? kSiteProdDo : kSiteProdQ);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full, SCH + SQ * 4);
            tma_load_3d(dlane ? sm.dO[st] : sm.q[st], dlane ? &p.tdo : &p.tq, full, 0, wk.i * SQ,
                        wk.bh);
            bulk_load(dlane ? sm.delta[st] : sm.lse2[st], (dlane ? p.delta : p.lse2) + roff, SQ * 4,
                      full);
          }
        }
        // no copy may still be landing in shared memory when the CTA exits
        if (!dlane && w_it > 0 && !mbar_wait(&sm.kv_full, (w_it - 1) & 1, nullptr, kWaitTimeoutNs))
          record_failure(p.status, abort, kSiteDtDrain);
        for (int s = 0; s < 2; ++s) {
          if (g > static_cast<uint32_t>(s)) {
            const uint32_t nph = (g - 1 - s) / 2;
            if (!mbar_wait(dlane ? &sm.do_full[s] : &sm.q_full[s], nph & 1, nullptr, kWaitTimeoutNs))
              record_failure(p.status, abort, kSiteDtDrain);
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ issuer A
      constexpr uint32_t kId = idesc_bf16_f32(BK, SQ, 0, 0);        // S^T, dP^T
      const uint64_t dK0 = sdesc_sw128(smem_u32(sm.k), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sm.v), 16, 1024);
      uint32_t w_it = 0, g = 0;
      bool ok = true;
      DtIter it{static_cast<int>(blockIdx.x), 0, 0};
      for (int kvbh, h, n; ok && sched.next(tail, it, kvbh, h, n);) {
        const SItem wi = s_item<BS>(p, kvbh, n, G);
        if (wi.nsteps == 0) continue;
        if (!mbar_wait_warp(&sm.kv_full, w_it & 1, abort, kWaitTimeoutNs)) {
          issuer_fail(p.status, abort, lane, kSiteMmaKV);
          ok = false;
          break;
        }
        for (int s = 0; s < wi.nsteps; ++s, ++g) {
          const int st = g & 1;
          // S^T(g) into the S buffer once dV(g-1) has read P^T(g-1) out of it
          if (g > 0 && !mbar_wait_warp(&sm.dv_done, (g - 1) & 1, abort, kWaitTimeoutNs)) {
            issuer_fail(p.status, abort, lane, kSiteMmaP);
            ok = false;
            break;
          }
          if (!mbar_wait_warp(&sm.q_full[st], (g >> 1) & 1, abort, kWaitTimeoutNs)) {
            issuer_fail(p.status, abort, lane, kSiteMmaQ);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t dq = sdesc_sw128(smem_u32(sm.q[st]), 16, 1024);
  #pragma unroll
          for (int kk = 0; kk < SD / 16; ++kk)
            mma_bf16_ss_w(tmem + TM_S, dK0 + ((kk * 32) >> 4), dq + ((kk * 32) >> 4), kId,
                          kk > 0 ? 1u : 0u);
          mma_commit_w(&sm.s_full);
          mma_commit_w(&sm.q_empty[st]);
          // dP^T(g) into the dP buffer once dK(g-1) has read dS^T(g-1) out of it
          if (g > 0 && !mbar_wait_warp(&sm.dk_done, (g - 1) & 1, abort, kWaitTimeoutNs)) {
            issuer_fail(p.status, abort, lane, kSiteMmaDs);
            ok = false;
            break;
          }
          if (!mbar_wait_warp(&sm.do_full[st], (g >> 1) & 1, abort, kWaitTimeoutNs)) {
            issuer_fail(p.status, abort, lane, kSiteMmaDo);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t ddo = sdesc_sw128(smem_u32(sm.dO[st]), 16, 1024);
  #pragma unroll
          for (int kk = 0; kk < SD / 16; ++kk)
            mma_bf16_ss_w(tmem + TM_DP, dV0 + ((kk * 32) >> 4), ddo + ((kk * 32) >> 4), kId,
                          kk > 0 ? 1u : 0u);
          mma_commit_w(&sm.dp_full);
          mma_commit_w(&sm.do_empty[st]);
        }
        if (!ok) break;
        mma_commit_w(&sm.kv_empty);                 // A's reads of K and V are done
        ++w_it;
      }
      // every tcgen05 op issued by this thread must finish before exit
      mma_commit_w(&sm.mma_done);
      if (!mbar_wait_warp(&sm.mma_done, 0, nullptr, kWaitTimeoutNs))
        issuer_fail(p.status, abort, lane, kSiteDtDrain);
      __syncwarp();
    } else if (warp == 2) {
      // ------------------------------------------------------------ issuer B
      constexpr uint32_t kIdAcc = idesc_bf16_f32(BK, SD, 0, 1);     // dV, dK (B MN-major)
      constexpr uint32_t kIdDq = idesc_bf16_f32(SQ, SD, 1, 1);      // dQ (A, B MN-major)
      // dS^T as the MN-major A operand of dQ (64-query chunks SCH apart), K as
      // its MN-major B operand
      const uint64_t dDS = sdesc_sw128(smem_u32(sm.ds), SCH, 1024);
      const uint64_t dKmn = sdesc_sw128(smem_u32(sm.k), SCH, 1024);
      uint32_t w_it = 0, g = 0;
      bool ok = true;
      auto fail = [&](int site) {
        issuer_fail(p.status, abort, lane, site);
        ok = false;
      };
      DtIter it{static_cast<int>(blockIdx.x), 0, 0};
      for (int kvbh, h, n; ok && sched.next(tail, it, kvbh, h, n);) {
        const SItem wi = s_item<BS>(p, kvbh, n, G);
        if (wi.nsteps == 0) continue;
        for (int s = 0; s < wi.nsteps; ++s, ++g) {
          const int st = g & 1;
          const uint32_t ph = g & 1;
          const bool first = (s == 0);
          const bool last = (s + 1 == wi.nsteps);
          // dV += P^T dO_i
          if (!mbar_wait_warp(&sm.p_full, ph, abort, kWaitTimeoutNs)) {
            fail(kSiteMmaP);
            break;
          }
          if (first && !mbar_wait_warp(&sm.acc_free, (w_it & 1) ^ 1, abort, kWaitTimeoutNs)) {
            fail(kSiteMmaAcc);
            break;
          }
          if (!mbar_wait_warp(&sm.do_full[st], (g >> 1) & 1, abort, kWaitTimeoutNs)) {
            fail(kSiteMmaDo);
            break;
          }
          tc_fence_after_sync();
          const uint64_t dOmn = sdesc_sw128(smem_u32(sm.dO[st]), SCH, 1024);
          const uint64_t dQmn = sdesc_sw128(smem_u32(sm.q[st]), SCH, 1024);
  #pragma unroll
          for (int kk = 0; kk < SQ / 16; ++kk)
            mma_bf16_ts_w(tmem + TM_DV, tmem + TM_S + scol(kk), dOmn + ((kk * 2048) >> 4), kIdAcc,
                          (first && kk == 0) ? 0u : 1u);
          mma_commit_w(&sm.dv_done);
          // dK += dS^T Q_i
          if (!mbar_wait_warp(&sm.ds_tm, ph, abort, kWaitTimeoutNs)) {
            fail(kSiteMmaDs);
            break;
          }
          tc_fence_after_sync();
  #pragma unroll
          for (int kk = 0; kk < SQ / 16; ++kk)
            mma_bf16_ts_w(tmem + TM_DK, tmem + TM_DP + scol(kk), dQmn + ((kk * 2048) >> 4), kIdAcc,
                          (first && kk == 0) ? 0u : 1u);
          mma_commit_w(&sm.dk_done);
          mma_commit_w(&sm.q_empty[st]);            // B's reads of Q(g) (and the row warps' of L2)
          mma_commit_w(&sm.do_empty[st]);           // B's reads of dO(g) (and the row warps' of D)
          if (last) mma_commit_w(&sm.acc_full);
          // dQ_i = dS K into its own columns once the row warps have taken
          // dQ(g-1) out of them and written dS(g) to shared memory
          if ((g > 0 && !mbar_wait_warp(&sm.dq_free, (g - 1) & 1, abort, kWaitTimeoutNs)) ||
              !mbar_wait_warp(&sm.ds_full, ph, abort, kWaitTimeoutNs)) {
            fail(kSiteMmaDq);
            break;
          }
          tc_fence_after_sync();
  #pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16_ss_w(tmem + TM_DQ, dDS + ((kk * 2048) >> 4), dKmn + ((kk * 2048) >> 4), kIdDq,
                          kk > 0 ? 1u : 0u);
          mma_commit_w(&sm.dq_full);
          if (last) mma_commit_w(&sm.kv_empty);     // B's reads of K are done
        }
        if (!ok) break;
        ++w_it;
      }
      mma_commit_w(&sm.mma_done_b);
      if (!mbar_wait_warp(&sm.mma_done_b, 0, nullptr, kWaitTimeoutNs))
        issuer_fail(p.status, abort, lane, kSiteDtDrain);
      __syncwarp();
    } else {
      // ------------------------------------------------------------ reduce warp
      // Adds each step's staged dQ to the accumulator with two bulk tensor
      // reduce-adds, and frees the previous step's buffer once its reduce-adds
      // have read it (so two steps' reduce-adds can be in flight).
      if (lane == 0) {
        prefetch_tmap(&p.tdq);
        uint32_t g = 0;
        bool ok = true;
        DtIter it{static_cast<int>(blockIdx.x), 0, 0};
        for (int kvbh, h, n; ok && sched.next(tail, it, kvbh, h, n);) {
          const SItem wi = s_item<BS>(p, kvbh, n, G);
          StepWalk wk(wi.i0, wi.i1, q_head_of(kvbh, 0, p.H, p.H_kv), wi.sk);
          for (int s = 0; s < wi.nsteps; ++s, ++g, wk.next()) {
            const int b = g & 1;
            if (!mbar_wait(&sm.stg_full[b], (g >> 1) & 1, abort, kWaitTimeoutNs)) {
              record_failure(p.status, abort, kSiteStageFull);
              ok = false;
              break;
            }
            // rows (queries) past N land in the padding up to Npad, never read
            tma_reduce_add_3d(&p.tdq, sm.stage[b], 0, wk.i * SQ, wk.bh);
            tma_reduce_add_3d(&p.tdq, sm.stage[b] + SCH, 32, wk.i * SQ, wk.bh);
            bulk_commit_group();
            if (g > 0) {
              bulk_wait_group_read<1>();
              mbar_arrive(&sm.stg_free[b ^ 1]);
            }
          }
        }
        // every reduce-add must have landed before the CTA exits
        bulk_wait_group<0>();
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<104>();
    // ------------------------------------------------------------ row warps
    const int quarter = warp & 3;
    const int j4 = (warp - kSRowWarp0) >> 2;
    const int r = quarter * 32 + lane;            // tensor-memory lane: key row, or query row of dQ
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c2 = p.scale_log2;
    __nv_bfloat16* dk_out = static_cast<__nv_bfloat16*>(p.dk);
    __nv_bfloat16* dv_out = static_cast<__nv_bfloat16*>(p.dv);
    // dQ(gg) leaves tensor memory through this warp's lanes (queries 32q ..
    // 32q+31 of the step) and columns 16j .. 16j+15 into staging buffer gg & 1:
    // box j/2 of [128 rows][32 columns] fp32 in the 128-byte swizzle of the
    // tensor map, row r as 16-byte chunks, chunk c at c ^ (r & 7).
    auto drain = [&](uint32_t gg) -> bool {
      if (!warp_wait(&sm.dq_full, gg & 1, abort)) {
        if (lane == 0) record_failure(p.status, abort, kSiteDrainDq);
        return false;
      }
      tc_fence_after_sync();
      uint32_t v[16];
      tmem_ld_x16(t_lane + TM_DQ + 16 * j4, v);
      tmem_wait_ld();
      reg_fence<16>(v);
      // this warp's part of dQ has left tensor memory
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.dq_free);
      const int b = gg & 1;
      if (gg >= 2 && !warp_wait(&sm.stg_free[b], ((gg >> 1) & 1) ^ 1, abort)) {
        if (lane == 0) record_failure(p.status, abort, kSiteStageFree);
        return false;
      }
      uint4* row = reinterpret_cast<uint4*>(sm.stage[b] + (j4 >> 1) * SCH) + r * 8;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int chunk = 4 * (j4 & 1) + c;
        row[chunk ^ (r & 7)] = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.stg_full[b]);
      return true;
    };
    const bool st32 = ((reinterpret_cast<uintptr_t>(dk_out) | reinterpret_cast<uintptr_t>(dv_out)) &
                       31u) == 0;
    uint32_t w_it = 0, g = 0;
    bool ok = true;
    DtIter it{static_cast<int>(blockIdx.x), 0, 0};
    for (int kvbh, h, n; ok && sched.next(tail, it, kvbh, h, n);) {
      const int len = dt_len(p, kvbh);
      const SItem wi = s_item<BS>(p, kvbh, n, G);
      const int key = n * BK + r;
      const size_t out_off = (static_cast<size_t>(kvbh) * p.N + key) * SD + 16 * j4;
      if (wi.nsteps == 0) {
        // key block seen by no query: zero gradients
        if (key < p.N) {
          uint4* a = reinterpret_cast<uint4*>(dk_out + out_off);
          uint4* bq = reinterpret_cast<uint4*>(dv_out + out_off);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            a[t] = make_uint4(0, 0, 0, 0);
            bq[t] = make_uint4(0, 0, 0, 0);
          }
        }
        continue;
      }
      StepWalk wk(wi.i0, wi.i1, 0, wi.sk);
      for (int s = 0; s < wi.nsteps; ++s, ++g, wk.next()) {
        const int st = g & 1;
        const uint32_t ph = g & 1;
        const int q0 = wk.i * SQ;
        // ---- P^T = exp2(S^T * c - L2), masked; bf16 back to tensor memory
        if (!warp_wait(&sm.s_full, ph, abort)) {
          if (lane == 0) record_failure(p.status, abort, kSiteRowS);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const bool need_mask = (n * BK + BK > len) || (q0 + SQ > p.N) ||
                               (n * BK + BK - 1 > q0 + p.wr) || (n * BK < q0 + SQ - 1 - p.wl);
        // visible columns c (query q = q0 + 32*j4 + c) of this key row:
        // [c_lo, c_hi]; none when the key is past len
        const int c_lo = key - p.wr - q0 - 32 * j4;
        const int c_hi = (key < len) ? key + p.wl - q0 - 32 * j4 : -1;
        const uint32_t t_s = t_lane + TM_S + 32 * j4;
        float pr[32];
        {
          uint32_t sr[32];
          tmem_ld_x32(t_s, sr);
          tmem_wait_ld();
          reg_fence<32>(sr);
          const uint64_t c2x2 = f2_make(c2, c2);
          const float4* l4p = reinterpret_cast<const float4*>(sm.lse2[st]) + 8 * j4;
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float4 l4 = l4p[t];
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
          // packed over the first 16 of this quarter's own 32 columns: the
          // other warps may still be reading their fp32 columns
          tmem_st_x16(t_s, pk);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full);
        // ---- dS^T = P^T o (dP^T - D) into tensor memory (for dK)
        if (!warp_wait(&sm.dp_full, ph, abort)) {
          if (lane == 0) record_failure(p.status, abort, kSiteRowDp);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t t_dp = t_lane + TM_DP + 32 * j4;
        uint32_t dk[16];
        {
          uint32_t sr[32];
          tmem_ld_x32(t_dp, sr);
          tmem_wait_ld();
          reg_fence<32>(sr);
          const float4* d4p = reinterpret_cast<const float4*>(sm.delta[st]) + 8 * j4;
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float4 d4 = d4p[t];
            float d0, d1, d2, d3;
            f2_split(f2_mul(f2_add(f2_make(__uint_as_float(sr[4 * t]), __uint_as_float(sr[4 * t + 1])),
                                   f2_make(-d4.x, -d4.y)),
                            f2_make(pr[4 * t], pr[4 * t + 1])),
                     d0, d1);
            f2_split(f2_mul(f2_add(f2_make(__uint_as_float(sr[4 * t + 2]), __uint_as_float(sr[4 * t + 3])),
                                   f2_make(-d4.z, -d4.w)),
                            f2_make(pr[4 * t + 2], pr[4 * t + 3])),
                     d2, d3);
            dk[2 * t] = pack_bf16x2(d0, d1);
            dk[2 * t + 1] = pack_bf16x2(d2, d3);
          }
          tmem_st_x16(t_dp, dk);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.ds_tm);
        // ---- the previous step's dQ (once it is complete the shared dS
        // buffer it read is free for this step's copy)
        if (g > 0 && !drain(g - 1)) {
          ok = false;
          break;
        }
        // ---- dS for dQ(g): row = key r, this quarter's 32 queries = 4 units
        // of 16 bytes in the 64-query chunk j4 / 2, XOR-swizzled by (r & 7)
        {
          uint8_t* rowp = sm.ds + (j4 >> 1) * SCH + r * 128;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int unit = 4 * (j4 & 1) + u;
            *reinterpret_cast<uint4*>(rowp + ((unit ^ (r & 7)) << 4)) =
                make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.ds_full);
      }
      if (!ok) break;
      // ---- dK, dV rows of this key block, head-dimension columns 16j .. 16j+15
      if (!warp_wait(&sm.acc_full, w_it & 1, abort)) {
        if (lane == 0) record_failure(p.status, abort, kSiteRowAcc);
        ok = false;
        break;
      }
      tc_fence_after_sync();
      {
        uint32_t a[16], bb[16];
        tmem_ld_x16(t_lane + TM_DV + 16 * j4, a);
        tmem_ld_x16(t_lane + TM_DK + 16 * j4, bb);
        tmem_wait_ld();
        reg_fence<16>(a);
        reg_fence<16>(bb);
        // the accumulators are in registers: the next item may start
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_free);
        if (key < p.N) {
          uint32_t pv[8], pkk[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            pv[t] = pack_bf16x2(__uint_as_float(a[2 * t]), __uint_as_float(a[2 * t + 1]));
            pkk[t] = pack_bf16x2(__uint_as_float(bb[2 * t]) * p.scale,
                                 __uint_as_float(bb[2 * t + 1]) * p.scale);
          }
          if (st32) {
            st_global_v8(dv_out + out_off, pv);
            st_global_v8(dk_out + out_off, pkk);
          } else {
            uint4* dvp = reinterpret_cast<uint4*>(dv_out + out_off);
            uint4* dkp = reinterpret_cast<uint4*>(dk_out + out_off);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              dvp[t] = make_uint4(pv[4 * t], pv[4 * t + 1], pv[4 * t + 2], pv[4 * t + 3]);
              dkp[t] = make_uint4(pkk[4 * t], pkk[4 * t + 1], pkk[4 * t + 2], pkk[4 * t + 3]);
            }
          }
        }
      }
      ++w_it;
    }
    // the last step's dQ
    if (ok && g > 0) drain(g - 1);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, TM_COLS);
  }
}

template <bool BS>
cudaError_t launch(const BwdParams& p, int num_sms, int max_smem, cudaStream_t stream) {
  const size_t smem = smem_request(sizeof(SSmem), max_smem);
  cudaError_t e = cudaFuncSetAttribute(bwd_d64_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int T = (p.N + BK - 1) / BK;
  const int BH = p.B * p.H_kv;
  const long long per_bh = p.causal ? (T + 1) / 2 : T;
  long long units = static_cast<long long>(BH) * per_bh;
  TailTable tail;
  tail.heads = 0;
  if (p.causal || (BS && p.block_mask_host && T == p.bm_t)) {
    // single key blocks in the tail: up to one CTA per block; the tail's
    // K/V heads share their group's Q and dO through L2
    const long long blocks = static_cast<long long>(BH) * T;
    const int g = static_cast<int>(blocks < num_sms ? blocks : num_sms);
    const long long qdo_bytes = 2ll * (p.H / p.H_kv) * p.N * SD * 2;
    if (p.causal)
      plan_causal_tail(BH, T, 1, g, false, qdo_bytes, &tail);
    else                       // key blocks cost their computed query steps
      plan_mask_tail(p.block_mask_host, BH, T, 1, g, false, p.N, p.wl, p.wr, qdo_bytes, &tail);
    if (tail.heads > 0) units = g;
  }
  if (tail.heads == 0) std::memset(tail.item, 0xff, sizeof(tail.item));
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  bwd_d64_kernel<BS><<<grid, kSThreads, smem, stream>>>(p, tail);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main_d64(const BwdParams& p, int num_sms, int max_smem,
                                cudaStream_t stream) {
  return p.block_mask ? launch<true>(p, num_sms, max_smem, stream)
                      : launch<false>(p, num_sms, max_smem, stream);
}

}  // namespace fa
