// Attention forward for sm_103a.
//
// One CTA per SM (persistent), 256 threads in five roles:
//   warp 0      TMA producer: Q tile once per tile, then K_j (and, for
//               d <= 128, V_j) into STAGES-deep shared-memory rings
//               (full/empty mbarriers).
//   warp 7      bf16 d = 256: TMA producer of V_j.  There the tensor core is the
//               bound (2048 cycles of products per block), and separate K
//               and V producers keep both rings full; for d <= 128 one
//               producer loading K_j then V_j measured faster (it paces the
//               S products against the P V products on the in-order tensor
//               pipe), and warp 7 idles.
//   warp 1      S issuer: S_j = Q K_j^T into one of NSB S buffers in tensor
//               memory, running ahead of the softmax as far as the buffers
//               allow (a buffer is free again once the softmax has loaded
//               it).  Also allocates and frees the tensor memory.
//   warp 2      P V issuer: O += P_j V_j with P read from tensor memory.
//               A tcgen05.mma holds its issuing thread for about as long as
//               the tensor core needs to run it, so the two products are
//               issued from two warps on different sub-partitions.  Each
//               issuer warp runs converged and one lane chosen by elect.sync
//               issues every MMA and commit.
//   warps 3..6  softmax: thread r owns query row r of the tile (TMEM lane r).
//               Reads its row of S, masks, updates the running max m and sum
//               l, writes P = exp2(S*c - m) as bf16 into one of NPB P
//               buffers in tensor memory,
//               rescales its row of O when m moved, and runs the epilogue
//               O / l, LSE = (m + log2 l) * ln 2 (bf16: after the next
//               tile's first block, so that the wait for the tile's last
//               P V is spent on that block).
// With the key-half split (bf16 d = 64, E4M3 d = 128; 480 threads) warps
// 3..10 are the softmax warps, two a row, each over half of every block's
// keys with a maximum, sum and O part of its own, and warps 11..14 are
// epilogue warps that merge a tile's O parts, divide and store (see Cfg).
//
// The recurrence is the online softmax of "注意力为什么受限于显存带宽：用算术
// 强度与分块把 FlashAttention 推导清楚" (section 六) and "4. FlashAttention 深度
// 剖析" (sections 4.2.3-4.2.4): S is kept in base-2 units (c = scale*log2 e
// folded into one FMA), O~ and l share the reference maximum, and the final
// division by l happens once (section 4.3.2; section 4.4.2 for the point of
// dividing once).  The reference maximum is only raised when the running
// maximum exceeds it by more than kRescaleSlack (log2 units); until then
// P <= 2^kRescaleSlack, which bf16 and fp32 hold exactly as well, and the
// result is the same because O~ and l are always taken against the same
// reference.
//
// Loop order: outer over Q tiles, inner over key blocks (section 4.4.3);
// key blocks entirely above the causal diagonal are never loaded (section
// 4.3.2, last note).  Tensor memory columns: NSB S buffers of 128 (3 for
// bf16 d <= 128, 2 for E4M3), a block's P (packed bf16 pairs, or E4M3
// quads) written over the first columns of its own S buffer (with the
// split: of its half's S columns), then O (with the split: two parts);
// S_{j+NSB} may overwrite S buffer j % NSB only after P_j V_j has completed
// (pv_done).  bf16 d = 256 (O takes 256 columns): one S buffer and two P
// buffers of their own (SEP), so that the S buffer is free as soon as the
// softmax has read S out of it (s_free); the softmax writes P buffer j % NPB
// once P_{j-NPB} V has completed.
#include <cstring>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_order.cuh"
#include "fa_window.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int BM = 128;          // query rows per tile = TMEM lanes = MMA M
constexpr int BN = 128;          // keys per block = MMA N of S
constexpr int CHUNK = 128 * 128; // bytes of one 128-row x 64-column bf16 chunk (SW128 atom rows)
constexpr int kKvlCache = 256;   // batch entries whose kv_len the d = 64 kernels stage
// bf16: the reference maximum moves only when a block exceeds it by more than
// 24 (log2 units), so P <= 2^24, l <= N * 2^24 and O~ stay far inside fp32's
// (and P inside bf16's) range, and most blocks of even large-score rows skip
// the rescale of O (8 measured 8 % slower at scores of standard deviation 9).
constexpr float kRescaleSlack = 24.0f;
// E4M3: the reference maximum moves when a block exceeds it by more than 4
// (log2 units), so P <= 2^4 and the E4M3 operand 16 P <= 256 (largest finite
// E4M3 448); 16 P has the same normal range relative to the row maximum as
// 256 P would with no slack.
constexpr float kFp8Slack = 4.0f;
constexpr float kFp8Shift = 4.0f;   // log2 of the multiplier 16 = 2^(8 - slack)

// FP8 = true: E4M3 Q and K (one byte an element, so a 128-byte swizzle row
// holds 128 of them) and V transposed per K/V head ([d, keys]: a V block is d
// rows of 128 keys, the K-major B operand of P V).
template <int D, bool FP8 = false>
struct Cfg {
  static_assert(!FP8 || D >= 128, "E4M3 rows need at least 128 bytes");
  static constexpr int BOX_COLS = FP8 ? 128 : 64;    // elements in one 128-byte swizzle row
  static constexpr int NCH = D / BOX_COLS;           // 128-byte column chunks per row
  static constexpr int TILE_BYTES = NCH * CHUNK;     // one Q tile or one K block
  static constexpr int V_BYTES = FP8 ? D * 128 : TILE_BYTES;
  static constexpr int STAGES =
      FP8 ? (D == 128 ? 6 : 3) : (D == 64 ? 4 : (D == 128 ? 3 : 1));
  // SEP: P in buffers of its own, with V from a separate producer (bf16
  // d = 256, where the products bound the kernel; E4M3 halves them and
  // measured faster with P over S).
  static constexpr bool SEP = (D == 256 && !FP8);
  // NSB S buffers: block g uses columns [128*(g%NSB), +128).  NPB P buffers
  // (without SEP, P buffer b is the start of S buffer b).
  // (E4M3 at d = 128 takes the key-half split below with two S buffers, so
  // that its two 128-column O parts fit.)
  static constexpr bool F8SPLIT = FP8 && D == 128;
  static constexpr int NSB = SEP ? 1 : (F8SPLIT ? 2 : (D <= 128 ? 3 : 2));
  static constexpr int NPB = SEP ? 2 : NSB;
  static constexpr int PW = FP8 ? BN / 4 : BN / 2;   // columns of one block's P
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_P = SEP ? 128 * NSB : TM_S;
  static constexpr uint32_t P_STRIDE = SEP ? PW : 128;
  static constexpr uint32_t TM_O = SEP ? TM_P + PW * NPB : 128 * NSB;
  static constexpr uint32_t TM_COLS = 512;
  static_assert(TM_O + D <= TM_COLS, "tensor memory budget");
  // NHALF softmax warps per sub-partition, each taking BN / NHALF keys of a
  // block.  At bf16 d = 64 and E4M3 d = 128 the products of a block take a
  // fraction of the time the softmax of one warp does, so two warps share
  // each row, each with a running maximum, row sum and O accumulator of its
  // own over its half of the keys (O in NHALF parts of D columns, merged by
  // the epilogue).  The two warps of a sub-partition never wait for each
  // other, so one computes while the other waits (for tensor memory, on a
  // barrier); elsewhere one warp a row.
  static constexpr int NHALF = ((D == 64 && !FP8) || F8SPLIT) ? 2 : 1;
  static constexpr int OCOLS = D * NHALF;            // columns of O (its key halves)
  // EPI (with the split): four epilogue warps merge each tile's O halves,
  // divide by l, store bf16 O and LSE, off the softmax warps (whose time per
  // tile the epilogue was a large share of at the few key blocks of short
  // sequences).
  static constexpr bool EPI = NHALF == 2;
  static constexpr int NOB = 1;                      // O buffers
  static constexpr int EPI_WARP0 = 3 + 4 * NHALF;    // first epilogue warp
  static constexpr int THREADS = EPI ? 480 : 256;
  static_assert(TM_O + OCOLS * NOB <= TM_COLS, "tensor memory budget (O)");
};

template <int D, bool FP8 = false>
struct FwdSmem {
  using C = Cfg<D, FP8>;
  alignas(1024) uint8_t q[C::TILE_BYTES];
  alignas(1024) uint8_t k[C::STAGES][C::TILE_BYTES];
  alignas(1024) uint8_t v[C::STAGES][C::V_BYTES];
  uint64_t q_full, q_empty;
  uint64_t k_full[C::STAGES], k_empty[C::STAGES];
  uint64_t v_full[C::STAGES], v_empty[C::STAGES];
  uint64_t s_full[C::NSB];   // S of block g is in S buffer g % NSB
  uint64_t s_free[C::NSB];   // SEP: the softmax has loaded S buffer b
  // the softmax wrote (key half h of) P of block g into P buffer g % NPB:
  // p_full[(g % NPB) * NHALF + h]
  uint64_t p_full[C::NPB * C::NHALF];
  uint64_t pv_done[C::NPB];  // O += P V of block g (P buffer g % NPB) has completed
  // O buffer b has been read out of tensor memory
  uint64_t o_free[C::NOB];
  // EPI: the tile's last P V into O buffer b has completed; its rows' row
  // sums and reference maxima are in ostat[b]
  uint64_t o_done[C::NOB], stats_full[C::NOB];
  // EPI: per row, the key halves' row sums [0, NHALF) and reference maxima
  // [NHALF, 2 NHALF)
  float ostat[C::NOB][2 * C::NHALF][C::EPI ? BM : 1];
  // EPI at d = 64: kv_len staged at the start (batches up to kKvlCache)
  int kvl[C::EPI && D == 64 ? kKvlCache : 1];
  uint64_t mma_done, pv_mma_done;
  // a block mask without a host copy: the tiles' costs, then their
  // cost-sorted order (fa_order.cuh)
  uint32_t order[kFwdOrderMaxT];
  uint32_t tmem_base;
  int abort;
};

// Wait sites reported in the status word.
enum Site {
  kSiteProdQ = 1, kSiteProdK, kSiteProdV, kSiteMmaQ, kSiteMmaK, kSiteMmaS, kSiteMmaP, kSiteMmaV,
  kSiteMmaO, kSiteSmS, kSiteSmP, kSiteSmO, kSiteSmEpi, kSiteDrain, kSiteSmPair
};

__device__ __forceinline__ void record_failure(int* status, volatile int* abort, int site) {
  atomicCAS(status, 0, status_code(site));
  *abort = 1;
}

// Static persistent schedule.  Non-causal: one unit per (bh, q-tile), bh-major
// so CTAs running at the same time share K/V in L2 (with a block mask and its
// host copy, the last heads' tiles go in a host-planned tail as below, costed
// by their computed key blocks).  Causal: a unit pairs
// q-tile T-1-p (longest: T-p key blocks) with q-tile p (p+1 key blocks), the
// longest first, so every unit costs T+1 key blocks; the units go
// round-robin, except those of the last tail_heads heads, whose single tiles
// come from the host-planned tail table (longest first on the least-loaded
// CTA), so that the last round of equal units does not leave CTAs idle.
//
// A block mask without a host copy (order != nullptr): the items go in the
// cost-sorted turning deal of fa_order.cuh instead, from this CTA's table.
struct Sched {
  int T, P, units, causal;   // units: the round-robin units (tile pairs when causal)
  int BH;
  const uint32_t* order;     // the cost-sorted order, or nullptr
  const int* kvl;            // kv_len staged in shared memory, or nullptr
  __device__ Sched(int BH_, int N, int causal_, int tail_heads, const uint32_t* order_,
                   const int* kvl_)
      : causal(causal_), BH(BH_), order(order_), kvl(kvl_) {
    T = (N + BM - 1) / BM;
    P = (T + 1) / 2;
    units = (BH - tail_heads) * (causal ? P : T);
  }
  __device__ int ntiles(int u) const {
    if (!causal) return 1;
    const int p = u % P;
    return (p == T - 1 - p) ? 1 : 2;
  }
  __device__ void tile(int u, int k, int& bh, int& m) const {
    if (!causal) {
      bh = u / T;
      m = u % T;
    } else {
      bh = u / P;
      const int p = u % P;
      m = (k == 0) ? (T - 1 - p) : p;
    }
  }
};

// kvl: kv_len staged in shared memory, or nullptr (read from global).
__device__ __forceinline__ int seq_len(const FwdParams& p, int bh, const int* kvl) {
  int len = p.N;
  if (p.kv_len) {
    len = kvl ? kvl[bh / p.H] : __ldg(p.kv_len + bh / p.H);
    len = len < 0 ? 0 : (len > p.N ? p.N : len);
  }
  return len;
}

// Key blocks [jlo, jlo + count) that query tile m can see (causal, window
// and kv_len); blocks outside are never loaded.  Returns the count.
__device__ __forceinline__ int tile_blocks(const FwdParams& p, int m, int len, int& jlo) {
  int k_lo, k_hi;
  visible_keys(m * BM, BM, len, p.wl, p.wr, k_lo, k_hi);
  jlo = k_lo / BN;
  const int jhi = (k_hi + BN - 1) / BN;
  return k_hi > k_lo ? jhi - jlo : 0;
}

__device__ __forceinline__ void issuer_fail(int* status, volatile int* abort, int lane, int site) {
  if (lane == 0) record_failure(status, abort, site);
}

// One tile of the schedule as every role sees it.  Training: query tile m of
// head bh (rows are the positions m*BM ..).  Decode: the H/H_kv query heads
// of one K/V head stacked as rows (Nq rows each, row r at position
// len - Nq + r % Nq) against one chunk of the keys; its outputs are partial
// and merged later.
struct Tile {
  int qy, qz;          // Q tile coordinates in the tensor map (row, head)
  int kvbh;            // K/V head
  int len;             // keys of the batch entry (kv_len)
  int qlo, qhi;        // query positions of the tile's first and last row
  int jlo, nkv;        // key blocks [jlo, jend), nkv of them not masked out
  int jend;
  const uint8_t* bmrow;  // block-mask row of the tile's query block, or nullptr
  long long out0;      // output row of tile row 0
  int rows;            // rows of the tile that are real queries
  int qs;              // index of the tile's Q scale (FP8)
};

// BS: the launch carries a block mask (a separate instantiation, so that the
// kernels without one keep the plain block walk).
template <bool DEC, bool BS = false>
__device__ __forceinline__ void make_tile(const FwdParams& p, int u, int bh, int m, Tile& t,
                                          const int* kvl) {
  if constexpr (!DEC) {
    t.qy = m * BM;
    t.qz = bh;
    t.kvbh = kv_head_of(bh, p.H, p.H_kv);
    t.len = seq_len(p, bh, kvl);
    t.qlo = m * BM;
    t.qhi = m * BM + BM - 1;
    t.nkv = tile_blocks(p, m, t.len, t.jlo);
    t.jend = t.jlo + t.nkv;
    t.bmrow = nullptr;
    if constexpr (BS) {
      t.bmrow = p.block_mask + static_cast<size_t>(m) * p.bm_t;
      int n = 0;
      for (int jb = t.jlo; jb < t.jend; ++jb) n += __ldg(t.bmrow + jb) != 0;
      t.nkv = n;
    }
    t.out0 = static_cast<long long>(bh) * p.N + m * BM;
    t.rows = p.N - m * BM < BM ? p.N - m * BM : BM;
    t.qs = bh * p.nb + m;
  } else {
    const int kvbh = u / p.splits, split = u % p.splits;
    const int row0 = q_head_of(kvbh, 0, p.H, p.H_kv) * p.Nq;
    t.qy = row0;
    t.qz = 0;
    t.kvbh = kvbh;
    t.len = seq_len(p, (kvbh / p.H_kv) * p.H, kvl);
    t.qlo = t.len - p.Nq;
    t.qhi = t.len - 1;
    int k_lo, k_hi;
    visible_keys(t.qlo, p.Nq, t.len, p.wl, p.wr, k_lo, k_hi);
    const int c0 = split * p.chunk_blocks * BN;
    if (k_lo < c0) k_lo = c0;
    if (k_hi > c0 + p.chunk_blocks * BN) k_hi = c0 + p.chunk_blocks * BN;
    t.jlo = k_lo / BN;
    t.nkv = k_hi > k_lo ? (k_hi + BN - 1) / BN - t.jlo : 0;
    t.jend = t.jlo + t.nkv;
    t.bmrow = nullptr;
    t.out0 = static_cast<long long>(split) * p.B * p.H * p.Nq + row0;
    t.rows = (p.H / p.H_kv) * p.Nq;
    t.qs = 0;
  }
}

// The first key block at or after jb that the tile computes: every block of
// [jlo, jend) without a block mask, else those whose mask byte is nonzero
// (every role walks the same sequence).
template <bool BS>
__device__ __forceinline__ int next_block(const Tile& t, int jb) {
  if constexpr (BS)
    while (jb < t.jend && __ldg(t.bmrow + jb) == 0) ++jb;
  return jb;
}

// This CTA's place in the schedule: its round-robin units (and the tiles of
// a causal pair), then its row of the tail table.
struct TileIter {
  int u, kt, k;
};

// The next tile of this CTA into t; false when it has none left.  Every role
// walks the same sequence.
template <bool DEC, bool BS>
__device__ __forceinline__ bool next_tile(const FwdParams& p, const TailTable& tail,
                                          const Sched& sched, int nunits, TileIter& it, Tile& t) {
  if constexpr (DEC) {
    if (it.u >= nunits) return false;
    make_tile<true>(p, it.u, 0, 0, t, sched.kvl);
    it.u += gridDim.x;
    return true;
  } else {
    if (BS && sched.order) {   // round it.k of the cost-sorted deal
      const long long k = order_deal(it.k, gridDim.x, blockIdx.x);
      if (k >= static_cast<long long>(sched.BH) * sched.T) return false;
      ++it.k;
      int bh, m;
      order_item(sched.order, sched.BH, k, bh, m);
      make_tile<false, BS>(p, 0, bh, m, t, sched.kvl);
      return true;
    }
    while (it.u < sched.units) {
      if (it.kt < sched.ntiles(it.u)) {
        int bh, m;
        sched.tile(it.u, it.kt, bh, m);
        ++it.kt;
        make_tile<false, BS>(p, 0, bh, m, t, sched.kvl);
        return true;
      }
      it.u += gridDim.x;
      it.kt = 0;
    }
    if (tail.heads == 0 || blockIdx.x >= kTailCtas || it.k >= kTailItems) return false;
    const int e = tail.item[blockIdx.x][it.k];
    if (e < 0) return false;
    ++it.k;
    make_tile<false, BS>(p, 0, tail_head(e), tail_block(e), t, sched.kvl);
    return true;
  }
}

// All 32 lanes wait; the decision is made uniform across the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  bool ok = mbar_wait(bar, parity, abort, kWaitTimeoutNs);
  return __all_sync(0xffffffffu, ok);
}

template <int D, bool DEC, bool FP8, bool BS>
__global__ void __launch_bounds__(Cfg<D, FP8>::THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ TailTable tail) {
  static_assert(!(DEC && FP8), "decode runs in bf16");
  using C = Cfg<D, FP8>;
  using Smem = FwdSmem<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
  const uintptr_t aligned = (raw + 1023) & ~static_cast<uintptr_t>(1023);
  if (aligned - raw + sizeof(Smem) > dynamic_smem_size()) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, status_code(kSiteSmemLayout));
    return;
  }
  Smem& sm = *reinterpret_cast<Smem*>(aligned);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  volatile int* abort = &sm.abort;
  // The grid is persistent (every CTA resident from the start), so the merge
  // kernel that follows a decode launch may be scheduled beside it now; it
  // waits for this grid's completion before reading the partials.
  if constexpr (DEC) launch_dependents();

  if (threadIdx.x == 0) {
    sm.abort = 0;
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    for (int b = 0; b < C::NSB; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.s_free[b], 4);
    }
    for (int b = 0; b < C::NPB; ++b) {
      for (int h = 0; h < C::NHALF; ++h) mbar_init(&sm.p_full[b * C::NHALF + h], 4);
      mbar_init(&sm.pv_done[b], 1);
    }
    mbar_init(&sm.pv_mma_done, 1);
    for (int b = 0; b < C::NOB; ++b) {
      mbar_init(&sm.o_free[b], 4);
      mbar_init(&sm.o_done[b], 1);
      mbar_init(&sm.stats_full[b], 32 * 4 * C::NHALF);
    }
    mbar_init(&sm.mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, C::TM_COLS);
    tmem_relinquish();
  }
  // (EPI at d = 64, where tiles of short sequences switch often) every tile's setup
  // reads its batch entry's kv_len: stage them once
  if constexpr (C::EPI && D == 64) {
    if (p.kv_len && p.B <= kKvlCache)
      for (int b = threadIdx.x; b < p.B; b += C::THREADS) sm.kvl[b] = __ldg(p.kv_len + b);
  }
  // A block mask without a host copy: every tile's cost (its computed key
  // blocks), then the cost-sorted order, a tile a thread (the launch keeps
  // T <= kFwdOrderMaxT).
  if constexpr (BS && !DEC) {
    static_assert(C::THREADS >= kFwdOrderMaxT, "one tile a thread");
    if (p.cost_sorted) {
      const int T = (p.N + BM - 1) / BM;
      const int t = threadIdx.x;
      if (t < T) {
        int jlo;
        const int n = tile_blocks(p, t, p.N, jlo);
        const uint8_t* row = p.block_mask + static_cast<size_t>(t) * p.bm_t;
        uint32_t c = 0;
        for (int j = jlo; j < jlo + n; ++j) c += __ldg(row + j) != 0;
        sm.order[t] = c;
      }
      __syncthreads();
      uint32_t e = 0;
      const int pos = t < T ? order_rank(sm.order, T, t, e) : 0;
      __syncthreads();
      if (t < T) sm.order[pos] = e;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  const int BH = p.B * p.H;
  const Sched sched(BH, p.N, p.causal, DEC ? 0 : tail.heads,
                    (BS && !DEC && p.cost_sorted) ? sm.order : nullptr,
                    (C::EPI && D == 64 && p.kv_len && p.B <= kKvlCache) ? sm.kvl : nullptr);
  const int nunits = DEC ? p.B * p.H_kv * p.splits : sched.units;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tq);
      prefetch_tmap(&p.tk);
      if constexpr (!C::SEP) prefetch_tmap(&p.tv);
      uint32_t q_it = 0, k_it = 0, v_it = 0;
      bool ok = true;
      TileIter it{static_cast<int>(blockIdx.x), 0, 0};
      for (Tile t; ok && next_tile<DEC, BS>(p, tail, sched, nunits, it, t);) {
        {
          const int jlo = t.jlo, nkv = t.nkv;
          if (nkv == 0) continue;
          const int kvbh = t.kvbh;
          if (!mbar_wait(&sm.q_empty, (q_it & 1) ^ 1, abort, kWaitTimeoutNs)) {
            record_failure(p.status, abort, kSiteProdQ);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.q_full, C::TILE_BYTES);
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(sm.q + c * CHUNK, &p.tq, &sm.q_full, C::BOX_COLS * c, t.qy, t.qz);
          ++q_it;
          for (int j = 0, jbs = next_block<BS>(t, t.jlo); j < nkv;
               ++j, jbs = BS ? next_block<BS>(t, jbs + 1) : jbs) {
            const int jb = BS ? jbs : t.jlo + j;        // key block
            const int st = k_it % C::STAGES;
            const uint32_t ph = (k_it / C::STAGES) & 1;
            if (!mbar_wait(&sm.k_empty[st], ph ^ 1, abort, kWaitTimeoutNs)) {
              record_failure(p.status, abort, kSiteProdK);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sm.k_full[st], C::TILE_BYTES);
#pragma unroll
            for (int c = 0; c < C::NCH; ++c)
              tma_load_3d(sm.k[st] + c * CHUNK, &p.tk, &sm.k_full[st], C::BOX_COLS * c, jb * BN,
                          kvbh);
            ++k_it;
            if constexpr (!C::SEP) {
              if (!mbar_wait(&sm.v_empty[st], ph ^ 1, abort, kWaitTimeoutNs)) {
                record_failure(p.status, abort, kSiteProdV);
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&sm.v_full[st], C::V_BYTES);
              if constexpr (FP8) {
                tma_load_3d(sm.v[st], &p.tv, &sm.v_full[st], jb * BN, 0, kvbh);
              } else {
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                  tma_load_3d(sm.v[st] + c * CHUNK, &p.tv, &sm.v_full[st], 64 * c, jb * BN,
                              kvbh);
              }
              ++v_it;
            }
          }
        }
      }
      // No copy may still be landing in shared memory when the CTA exits:
      // wait (bounded, ignoring the abort flag) for the last phase issued on
      // every full barrier.  In a normal run these phases completed long ago.
      if (q_it > 0 && !mbar_wait(&sm.q_full, (q_it - 1) & 1, nullptr, kWaitTimeoutNs))
        record_failure(p.status, abort, kSiteDrain);
      for (int s = 0; s < C::STAGES; ++s) {
        if (k_it > static_cast<uint32_t>(s)) {
          const uint32_t n = (k_it - 1 - s) / C::STAGES;
          if (!mbar_wait(&sm.k_full[s], n & 1, nullptr, kWaitTimeoutNs))
            record_failure(p.status, abort, kSiteDrain);
        }
        if (v_it > static_cast<uint32_t>(s)) {      // (SEP: v_it stays 0 here)
          const uint32_t n = (v_it - 1 - s) / C::STAGES;
          if (!mbar_wait(&sm.v_full[s], n & 1, nullptr, kWaitTimeoutNs))
            record_failure(p.status, abort, kSiteDrain);
        }
      }
    }
    __syncwarp();
  } else if (C::NHALF == 1 && warp == 7) {
    // ------------------------------------------------------------ V producer (SEP)
    if (C::SEP && lane == 0) {
      prefetch_tmap(&p.tv);
      uint32_t v_it = 0;
      bool ok = true;
      TileIter it{static_cast<int>(blockIdx.x), 0, 0};
      for (Tile t; ok && next_tile<DEC, BS>(p, tail, sched, nunits, it, t);) {
        {
          const int jlo = t.jlo, nkv = t.nkv;
          const int kvbh = t.kvbh;
          for (int j = 0, jbs = next_block<BS>(t, t.jlo); j < nkv;
               ++j, jbs = BS ? next_block<BS>(t, jbs + 1) : jbs) {
            const int jb = BS ? jbs : t.jlo + j;        // key block
            const int st = v_it % C::STAGES;
            const uint32_t ph = (v_it / C::STAGES) & 1;
            if (!mbar_wait(&sm.v_empty[st], ph ^ 1, abort, kWaitTimeoutNs)) {
              record_failure(p.status, abort, kSiteProdV);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sm.v_full[st], C::V_BYTES);
            if constexpr (FP8) {
              // transposed V: one box of D rows x 128 keys
              tma_load_3d(sm.v[st], &p.tv, &sm.v_full[st], jb * BN, 0, kvbh);
            } else {
#pragma unroll
              for (int c = 0; c < C::NCH; ++c)
                tma_load_3d(sm.v[st] + c * CHUNK, &p.tv, &sm.v_full[st], 64 * c, jb * BN, kvbh);
            }
            ++v_it;
          }
        }
      }
      // as for K: no V copy may still be landing when the CTA exits
      for (int s = 0; s < C::STAGES; ++s) {
        if (v_it > static_cast<uint32_t>(s)) {
          const uint32_t n = (v_it - 1 - s) / C::STAGES;
          if (!mbar_wait(&sm.v_full[s], n & 1, nullptr, kWaitTimeoutNs))
            record_failure(p.status, abort, kSiteDrain);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    {
      constexpr uint32_t kIdescS = FP8 ? idesc_e4m3_f32(BM, BN, 0, 0) : idesc_bf16_f32(BM, BN, 0, 0);
      const uint64_t dq0 = sdesc_sw128(smem_u32(sm.q), 16, 1024);
      uint32_t q_it = 0, g = 0;
      bool ok = true;
      TileIter it{static_cast<int>(blockIdx.x), 0, 0};
      for (Tile t; ok && next_tile<DEC, BS>(p, tail, sched, nunits, it, t);) {
        {
          const int nkv = t.nkv;
          if (nkv == 0) continue;
          if (!mbar_wait_warp(&sm.q_full, q_it & 1, abort, kWaitTimeoutNs)) {
            issuer_fail(p.status, abort, lane, kSiteMmaQ);
            ok = false;
            break;
          }
          ++q_it;
          for (int j = 0; j < nkv; ++j, ++g) {
            const uint32_t b = g % C::NSB;
            // buffer b last held block g - NSB: the softmax must have loaded
            // it (SEP), or its P V must be complete (P over S)
            if (g >= static_cast<uint32_t>(C::NSB) &&
                !mbar_wait_warp(C::SEP ? &sm.s_free[b] : &sm.pv_done[b], ((g / C::NSB) & 1) ^ 1,
                                abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaS);
              ok = false;
              break;
            }
            const int st = g % C::STAGES;
            if (!mbar_wait_warp(&sm.k_full[st], (g / C::STAGES) & 1, abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaK);
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint64_t dk0 = sdesc_sw128(smem_u32(sm.k[st]), 16, 1024);
            // one K step is 32 bytes of a row: 16 bf16 or 32 E4M3 values
#pragma unroll
            for (int kk = 0; kk < C::NCH * 4; ++kk) {
              const uint32_t off = (kk / 4) * CHUNK + (kk % 4) * 32;
              if constexpr (FP8)
                mma_e4m3_ss_w(tmem + C::TM_S + 128 * b, dq0 + (off >> 4), dk0 + (off >> 4), kIdescS,
                              kk > 0 ? 1u : 0u);
              else
                mma_bf16_ss_w(tmem + C::TM_S + 128 * b, dq0 + (off >> 4), dk0 + (off >> 4), kIdescS,
                              kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&sm.k_empty[st]);
            mma_commit_w(&sm.s_full[b]);
            if (j == nkv - 1) mma_commit_w(&sm.q_empty);
          }
        }
      }
      // every tcgen05 op issued by this thread must finish before exit
      mma_commit_w(&sm.mma_done);
      if (!mbar_wait_warp(&sm.mma_done, 0, nullptr, kWaitTimeoutNs))
        issuer_fail(p.status, abort, lane, kSiteDrain);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ P V issuer
    {
      constexpr uint32_t kIdescPV = FP8 ? idesc_e4m3_f32(BM, D, 0, 0) : idesc_bf16_f32(BM, D, 0, 1);
      uint32_t g = 0, t_it = 0;
      bool ok = true;
      TileIter it{static_cast<int>(blockIdx.x), 0, 0};
      for (Tile t; ok && next_tile<DEC, BS>(p, tail, sched, nunits, it, t);) {
        {
          const int nkv = t.nkv;
          if (nkv == 0) continue;
          for (int j = 0; j < nkv; ++j, ++g) {
            const uint32_t b = g % C::NPB;
            const int st = g % C::STAGES;
            if (!mbar_wait_warp(&sm.v_full[st], (g / C::STAGES) & 1, abort, kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaV);
              ok = false;
              break;
            }
            // a tile's first P V starts a fresh O: the epilogue of the tile
            // that last used this O buffer must have read it out of tensor memory
            const uint32_t ob = t_it % C::NOB;
            if (j == 0 && !mbar_wait_warp(&sm.o_free[ob], ((t_it / C::NOB) & 1) ^ 1, abort,
                                          kWaitTimeoutNs)) {
              issuer_fail(p.status, abort, lane, kSiteMmaO);
              ok = false;
              break;
            }
            // each key half's product as soon as its P is written, into the
            // half's own part of O (NHALF = 2)
#pragma unroll
            for (int h = 0; h < C::NHALF; ++h) {
              if (!mbar_wait_warp(&sm.p_full[b * C::NHALF + h], (g / C::NPB) & 1, abort,
                                  kWaitTimeoutNs)) {
                issuer_fail(p.status, abort, lane, kSiteMmaP);
                ok = false;
                break;
              }
              tc_fence_after_sync();
              const uint32_t d_o = tmem + C::TM_O + C::OCOLS * ob + D * h;
              if constexpr (FP8) {
                // transposed V block: D rows x 128 keys, the K-major B operand;
                // P as E4M3, four keys a tensor-memory column, 32 keys a step;
                // half h takes the steps [h KH8, (h + 1) KH8), its P at the
                // start of its S columns (BN / NHALF) h
                constexpr int KH8 = BN / 32 / C::NHALF;
                const uint64_t dv0 = sdesc_sw128(smem_u32(sm.v[st]), 16, 1024);
#pragma unroll
                for (int k = 0; k < KH8; ++k) {
                  const int kk = h * KH8 + k;
                  mma_e4m3_ts_w(d_o, tmem + C::TM_P + C::P_STRIDE * b + (BN / C::NHALF) * h + k * 8,
                                dv0 + static_cast<uint64_t>((kk * 32) >> 4), kIdescPV,
                                (j == 0 && k == 0) ? 0u : 1u);
                }
              } else {
                // V block: BN rows (keys) x D columns, MN-major B operand: 64-column
                // chunks BN*128 bytes apart (LBO), 8-key groups 1024 bytes apart
                // (SBO); half h takes the 16-key steps [h KH, (h + 1) KH), its P
                // at the start of its S columns (BN / NHALF) h
                constexpr int KH = BN / 16 / C::NHALF;
                const uint64_t dv0 = sdesc_sw128(smem_u32(sm.v[st]), BN * 128, 1024);
#pragma unroll
                for (int k = 0; k < KH; ++k) {
                  const int kk = h * KH + k;
                  mma_bf16_ts_w(d_o, tmem + C::TM_P + C::P_STRIDE * b + (BN / C::NHALF) * h + k * 8,
                                dv0 + static_cast<uint64_t>((kk * 16 * 128) >> 4), kIdescPV,
                                (j == 0 && k == 0) ? 0u : 1u);
                }
              }
            }
            if (!ok) break;
            mma_commit_w(&sm.v_empty[st]);
            mma_commit_w(&sm.pv_done[b]);
            if (C::EPI && j == nkv - 1) mma_commit_w(&sm.o_done[ob]);
          }
          ++t_it;
        }
      }
      mma_commit_w(&sm.pv_mma_done);
      if (!mbar_wait_warp(&sm.pv_mma_done, 0, nullptr, kWaitTimeoutNs))
        issuer_fail(p.status, abort, lane, kSiteDrain);
    }
    __syncwarp();
  } else if (C::EPI && warp >= C::EPI_WARP0) {
    // ------------------------------------------------------------ epilogue warps
    // One warp per sub-partition (its 32 tensor-memory lanes are 32 query
    // rows); each row's O / l into bf16 O (decode: fp32 partials) and its LSE.
    const int quarter = warp & 3;
    const int row_local = quarter * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o);
    const bool st32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
    uint32_t e_it = 0;
    bool ok = true;
    TileIter it{static_cast<int>(blockIdx.x), 0, 0};
    for (Tile t; ok && next_tile<DEC, BS>(p, tail, sched, nunits, it, t);) {
      const bool row_valid = row_local < t.rows;
      const size_t row_off = static_cast<size_t>(t.out0 + row_local);
      if (t.nkv == 0) {   // no key is visible to the tile's rows: O = 0, LSE = -inf
        if (row_valid) {
          if constexpr (DEC) {
            float4* dst = reinterpret_cast<float4*>(p.o_part + row_off * D);
#pragma unroll
            for (int i = 0; i < D / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            p.lse_part[row_off] = -INFINITY;
          } else {
            uint4* dst = reinterpret_cast<uint4*>(out + row_off * D);
#pragma unroll
            for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
            p.lse[row_off] = -INFINITY;
          }
        }
        continue;
      }
      const uint32_t ob = e_it % C::NOB;
      const uint32_t ph = (e_it / C::NOB) & 1;
      ++e_it;
      if (!warp_wait(&sm.stats_full[ob], ph, abort) || !warp_wait(&sm.o_done[ob], ph, abort)) {
        if (lane == 0) record_failure(p.status, abort, kSiteSmEpi);
        ok = false;
        break;
      }
      tc_fence_after_sync();
      // merge the key halves: each half h holds O_h and l_h relative to its
      // own reference maximum m_h; relative to m = max_h m_h they weigh
      // a_h = 2^(m_h - m), so O = sum_h a_h O_h / l with l = sum_h a_h l_h
      float a[C::NHALF], m = -INFINITY;
#pragma unroll
      for (int h = 0; h < C::NHALF; ++h) m = fmaxf(m, sm.ostat[ob][C::NHALF + h][row_local]);
      float l = 0.f;
#pragma unroll
      for (int h = 0; h < C::NHALF; ++h) {
        const float mh = sm.ostat[ob][C::NHALF + h][row_local];
        a[h] = mh == -INFINITY ? 0.f : ex2_approx(mh - m);
        l += a[h] * sm.ostat[ob][h][row_local];
      }
      // FP8: P entered the product as 16 P (and l sums 16 P), V in units of
      // its head scale
      const float inv_l = l > 0.f ? (FP8 ? __ldg(p.v_scale + t.kvbh) / l : 1.f / l) : 0.f;
      const float lse_row =
          l > 0.f ? (m + (log2f(l) - (FP8 ? kFp8Shift : 0.f))) * 0.69314718055994531f : -INFINITY;
#pragma unroll
      for (int h = 0; h < C::NHALF; ++h) a[h] *= inv_l;
      // 32 columns a round: the halves' columns from tensor memory, merged
      // and stored (O buffer ob, and ostat[ob], are free after the last load)
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orr[C::NHALF][32];
#pragma unroll
        for (int h = 0; h < C::NHALF; ++h)
          tmem_ld_x32(t_lane + C::TM_O + C::OCOLS * ob + D * h + 32 * c, orr[h]);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < C::NHALF; ++h) reg_fence<32>(orr[h]);
        if (c == D / 32 - 1) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.o_free[ob]);
        }
        float o[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          o[e] = __uint_as_float(orr[0][e]) * a[0];
#pragma unroll
          for (int h = 1; h < C::NHALF; ++h) o[e] = fmaf(__uint_as_float(orr[h][e]), a[h], o[e]);
        }
        if (!row_valid) continue;
        if constexpr (DEC) {
          // the workspace is 256-byte aligned and a row is D floats
          float* dst = p.o_part + row_off * D + 32 * c;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t r8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) r8[e] = __float_as_uint(o[8 * i + e]);
            st_global_v8(dst + 8 * i, r8);
          }
        } else {
          __nv_bfloat16* dst = out + row_off * D + 32 * c;
#pragma unroll
          for (int i = 0; i < 2; ++i) {                // 16 columns a step
            uint32_t pk8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) pk8[e] = pack_bf16x2(o[16 * i + 2 * e], o[16 * i + 2 * e + 1]);
            if (st32) {
              st_global_v8(dst + 16 * i, pk8);
            } else {
              uint4* d4 = reinterpret_cast<uint4*>(dst + 16 * i);
              d4[0] = make_uint4(pk8[0], pk8[1], pk8[2], pk8[3]);
              d4[1] = make_uint4(pk8[4], pk8[5], pk8[6], pk8[7]);
            }
          }
        }
      }
      if (row_valid) {
        if constexpr (DEC)
          p.lse_part[row_off] = lse_row;
        else
          p.lse[row_off] = lse_row;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int quarter = warp & 3;                  // TMEM lanes 32*quarter .. +31
    const int hf = (warp - 3) >> 2;                // key half (NHALF = 2)
    constexpr int NC = BN / C::NHALF;              // S columns (keys) of this warp
    constexpr int DO = D;                          // O columns of this warp's O part
    const int row_local = quarter * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t t_o0 = t_lane + C::TM_O + D * hf;    // this warp's O part in O buffer 0
    uint32_t t_o = t_o0;                                 // ... of the current tile's O buffer
    const float c2 = p.scale_log2;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o);
    uint32_t kv_it = 0, e_it = 0;                       // e_it: tiles with key blocks
    // kEarlyS: one warp a row (d = 128, 256) tests for the next block's S
    // while its P store lands, and skips the wait when it is there (1 % on
    // the causal d = 128 forward).  With the key-half split (bf16 d = 64,
    // E4M3 d = 128), where the two warps of a row cover each other's waits,
    // it measured 1-5 % slower.
    constexpr bool kEarlyS = !C::EPI;
    bool ok = true;
    // The epilogue of a tile (O / l into bf16 O, and LSE): run once the next
    // tile's first block of P is written, so that the softmax warps spend the
    // wait for this tile's last P V on that block instead of idling; the next
    // tile's first P V waits for o_free, so O is read before it is replaced.
    auto epilogue = [&](uint32_t last, float l, float m_ref, size_t row_off, bool row_valid,
                        int kvbh) -> bool {
      // wait for the tile's last P V, then O / l and LSE
      if (!warp_wait(&sm.pv_done[last % C::NPB], (last / C::NPB) & 1, abort)) {
        if (lane == 0) record_failure(p.status, abort, kSiteSmEpi);
        return false;
      }
      tc_fence_after_sync();
      // FP8: P entered the product as 16 P (and l sums 16 P), V in units
      // of its head scale
      const float inv_l = l > 0.f ? (FP8 ? __ldg(p.v_scale + kvbh) / l : 1.f / l) : 0.f;
      // O leaves tensor memory up to 128 columns a batch, each batch on one
      // wait; after the last batch the P V issuer may start the next tile
      // while the rows are scaled and stored.  Each thread stores its own
      // row, 32 bytes a store (16 when O is only 16-byte aligned), so a warp
      // store touches half as many lines as with 16-byte stores.
      constexpr int OB = DO < 128 ? DO / 32 : 4;          // 32-column chunks a batch
      const bool st32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
#pragma unroll 1
      for (int c0 = 0; c0 < DO / 32; c0 += OB) {
        uint32_t orr[OB * 32];
#pragma unroll
        for (int c = 0; c < OB; ++c) tmem_ld_x32(t_o + 32 * (c0 + c), orr + 32 * c);
        tmem_wait_ld();
        reg_fence<OB * 32>(orr);
        if (c0 + OB == DO / 32) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.o_free[0]);
        }
        if constexpr (DEC) {
          if (row_valid) {
            // the workspace is 256-byte aligned and a row is D floats
            float* dst = p.o_part + row_off * D + DO * hf + 32 * c0;
#pragma unroll
            for (int i = 0; i < OB * 4; ++i) {
              uint32_t r8[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) r8[e] = __float_as_uint(__uint_as_float(orr[8 * i + e]) * inv_l);
              st_global_v8(dst + 8 * i, r8);
            }
          }
        } else if (row_valid) {
          __nv_bfloat16* dst = out + row_off * D + DO * hf + 32 * c0;
#pragma unroll
          for (int i = 0; i < OB * 2; ++i) {                // 16 columns a step
            uint32_t pk8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              pk8[e] = pack_bf16x2(__uint_as_float(orr[16 * i + 2 * e]) * inv_l,
                                   __uint_as_float(orr[16 * i + 2 * e + 1]) * inv_l);
            if (st32) {
              st_global_v8(dst + 16 * i, pk8);
            } else {
              uint4* d4 = reinterpret_cast<uint4*>(dst + 16 * i);
              d4[0] = make_uint4(pk8[0], pk8[1], pk8[2], pk8[3]);
              d4[1] = make_uint4(pk8[4], pk8[5], pk8[6], pk8[7]);
            }
          }
        }
      }
      if (row_valid && hf == 0) {
        const float lse_row =
            l > 0.f ? (m_ref + (log2f(l) - (FP8 ? kFp8Shift : 0.f))) * 0.69314718055994531f
                    : -INFINITY;
        if constexpr (DEC)
          p.lse_part[row_off] = lse_row;
        else
          p.lse[row_off] = lse_row;
      }
      return true;
    };
    struct Pending {
      bool on;
      uint32_t last;
      float l, m_ref;
      size_t row_off;
      bool row_valid;
      int kvbh;
    } pend{false, 0u, 0.f, 0.f, 0, false, 0};
    auto finish = [&]() -> bool {
      if (!pend.on) return true;
      pend.on = false;
      return epilogue(pend.last, pend.l, pend.m_ref, pend.row_off, pend.row_valid, pend.kvbh);
    };
    TileIter it{static_cast<int>(blockIdx.x), 0, 0};
    for (Tile t; ok && next_tile<DEC, BS>(p, tail, sched, nunits, it, t);) {
      {
        const int len = t.len, jlo = t.jlo, nkv = t.nkv;
        const int row = DEC ? t.qlo + row_local % p.Nq : t.qlo + row_local;   // query position
        // FP8: scores come out of the MMA in units of sq * sk
        const float q_sc = FP8 ? __ldg(p.q_scale + t.qs) : 1.f;
        const bool row_valid = row_local < t.rows;
        const size_t row_off = static_cast<size_t>(t.out0 + row_local);
        if (C::EPI && nkv == 0) continue;   // the epilogue warps write its rows
        if (nkv == 0) {
          if (!finish()) {
            ok = false;
            break;
          }
          if (row_valid) {
            if constexpr (DEC) {
              float4* dst = reinterpret_cast<float4*>(p.o_part + row_off * D + DO * hf);
#pragma unroll
              for (int i = 0; i < DO / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
              if (hf == 0) p.lse_part[row_off] = -INFINITY;
            } else {
              uint4* dst = reinterpret_cast<uint4*>(out + row_off * D + DO * hf);
#pragma unroll
              for (int i = 0; i < DO / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
              if (hf == 0) p.lse[row_off] = -INFINITY;
            }
          }
          continue;
        }
        const uint32_t ob = e_it % C::NOB;   // this tile's O buffer
        t_o = t_o0 + C::OCOLS * ob;
        float m_ref = -INFINITY;    // reference maximum, base-2 units of S*scale
        float l = 0.f;
        bool s_next = false;        // the next block's S was seen complete (kEarlyS)
        for (int j = 0, jbs = next_block<BS>(t, t.jlo); j < nkv;
             ++j, jbs = BS ? next_block<BS>(t, jbs + 1) : jbs) {
          const int jb = BS ? jbs : t.jlo + j;        // key block
          const uint32_t b = kv_it % C::NSB;
          const uint32_t t_s = t_lane + C::TM_S + 128 * b;      // this block's S buffer
          if (!(kEarlyS && __all_sync(0xffffffffu, s_next)) &&
              !warp_wait(&sm.s_full[b], (kv_it / C::NSB) & 1, abort)) {
            if (lane == 0) record_failure(p.status, abort, kSiteSmS);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          uint32_t sr[NC];
#pragma unroll
          for (int c = 0; c < NC / 32; ++c) tmem_ld_x32(t_s + NC * hf + 32 * c, sr + 32 * c);
          tmem_wait_ld();
          reg_fence<NC>(sr);
          if constexpr (C::SEP) {
            // S is in registers: the S issuer may reuse the buffer
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.s_free[b]);
          }
          float s[NC];
#pragma unroll
          for (int c = 0; c < NC; ++c) s[c] = __uint_as_float(sr[c]);
          // masks: keys past the sequence (tail / padding), right of the
          // window (above the diagonal when causal) and left of the window;
          // skipped when every key of the block is visible to every row
          const int key0 = jb * BN + NC * hf;
          if (key0 + NC > len || key0 + NC - 1 > t.qlo + p.wr || key0 < t.qhi - p.wl) {
            // visible columns [c_lo, c_hi]: before the sequence end and
            // inside the window [row - wl, row + wr]
            const int c_hi = min(len - key0 - 1, row + p.wr - key0);
            const int c_lo = row - p.wl - key0;
#pragma unroll
            for (int c = 0; c < NC; ++c)
              if (c > c_hi || c < c_lo) s[c] = -INFINITY;
          }
          // row maximum: four chains of three-input max over s[0 .. NC)
          static_assert(NC % 8 == 0, "the max chains take 8 columns a step");
          float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
          for (int c = 4; c + 8 <= NC; c += 8) {
            mx0 = fmax3(mx0, s[c], s[c + 1]);
            mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
            mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
            mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
          }
          mx0 = fmax3(mx0, s[NC - 4], s[NC - 3]);
          mx1 = fmax3(mx1, s[NC - 2], s[NC - 1]);
          // this block's multiplier from MMA output to base-2 units of S*scale
          const float cb = FP8 ? c2 * q_sc * __ldg(p.k_scale + t.kvbh * p.nb + jb) : c2;
          const float m_blk = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * cb;
          float alpha = 1.f;
          bool rescale = false;
          if (m_ref == -INFINITY) {
            if (m_blk != -INFINITY) {
              alpha = 0.f;
              m_ref = m_blk;
            }
          } else if (m_blk > m_ref + (FP8 ? kFp8Slack : kRescaleSlack)) {
            alpha = ex2_approx(m_ref - m_blk);
            m_ref = m_blk;
            rescale = true;
          }
          // FP8 takes 16 p, the E4M3 operand, straight from the exponent
          // (exp2(x + 4) = 16 exp2(x)); its row sum l is then 16 times the
          // sum of p, and the epilogue divides the 16 back out.
          const float base = ((m_ref == -INFINITY) ? 0.f : m_ref) - (FP8 ? kFp8Shift : 0.f);
          // p = exp2(S*c - m) two lanes at a time: packed FMA for the argument,
          // packed adds for the row sum, one bf16x2 convert per pair
          const uint64_t c2x2 = f2_make(cb, cb);
          const uint64_t nbx2 = f2_make(-base, -base);
          uint64_t rsa = f2_make(0.f, 0.f), rsb = f2_make(0.f, 0.f);
          uint32_t pk[FP8 ? NC / 4 : NC / 2];
#pragma unroll
          for (int c = 0; c < NC / 2; c += 2) {
            float a0, a1, a2, a3;
            f2_split(f2_fma(f2_make(s[2 * c], s[2 * c + 1]), c2x2, nbx2), a0, a1);
            f2_split(f2_fma(f2_make(s[2 * c + 2], s[2 * c + 3]), c2x2, nbx2), a2, a3);
            const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
            const float p2 = ex2_approx(a2), p3 = ex2_approx(a3);
            rsa = f2_add(rsa, f2_make(p0, p1));
            rsb = f2_add(rsb, f2_make(p2, p3));
            if constexpr (FP8) {
              pk[c / 2] = pack_e4m3x4(p0, p1, p2, p3);
            } else {
              pk[c] = pack_bf16x2(p0, p1);
              pk[c + 1] = pack_bf16x2(p2, p3);
            }
          }
          float rs0, rs1, rs2, rs3;
          f2_split(rsa, rs0, rs1);
          f2_split(rsb, rs2, rs3);
          l = l * alpha + ((rs0 + rs1) + (rs2 + rs3));
          // P: 64 columns of bf16 pairs, or 32 of E4M3 quads, over the start of
          // this block's S buffer (S is in registers), or (SEP) into P buffer
          // kv_it % NPB once P_{kv_it-NPB} V has read it
          const uint32_t pb = kv_it % C::NPB;
          if (C::SEP && kv_it >= static_cast<uint32_t>(C::NPB) &&
              !warp_wait(&sm.pv_done[pb], ((kv_it / C::NPB) & 1) ^ 1, abort)) {
            if (lane == 0) record_failure(p.status, abort, kSiteSmP);
            ok = false;
            break;
          }
          if constexpr (C::SEP) tc_fence_after_sync();
          // (NHALF = 2: this warp's keys at the start of its own S columns,
          // NC * hf, which only this warp reads: the other half may still be
          // loading its S)
          constexpr int PCOLS = FP8 ? NC / 4 : NC / 2;
          const uint32_t t_p = t_lane + C::TM_P + C::P_STRIDE * pb + NC * hf;
          tmem_st_x32(t_p, pk);
          if constexpr (PCOLS == 64) tmem_st_x32(t_p + 32, pk + 32);
          // while the store lands: has the next block's S completed?  (That
          // barrier cannot move past the phase: its next one needs this
          // warp's P, or with SEP its load, of that block first.)
          s_next = kEarlyS && j + 1 < nkv &&
                   mbar_test(&sm.s_full[(kv_it + 1) % C::NSB], ((kv_it + 1) / C::NSB) & 1);
          if (__any_sync(0xffffffffu, rescale && j > 0)) {
            // O must hold every earlier P V before it is scaled: wait for the
            // previous block's P V to complete.
            const uint32_t prev = kv_it - 1;
            if (!warp_wait(&sm.pv_done[prev % C::NPB], (prev / C::NPB) & 1, abort)) {
              if (lane == 0) record_failure(p.status, abort, kSiteSmO);
              ok = false;
              break;
            }
            tc_fence_after_sync();
            // this warp's columns of O, up to 128 per round trip (S is no
            // longer live), scaled two at a time
            constexpr int RC = DO < 128 ? DO / 32 : (C::NHALF == 2 ? 1 : 4);
            const uint64_t a2 = f2_make(alpha, alpha);
#pragma unroll 1
            for (int c0 = 0; c0 < DO / 32; c0 += RC) {
              uint32_t orr[RC * 32];
#pragma unroll
              for (int c = 0; c < RC; ++c) tmem_ld_x32(t_o + 32 * (c0 + c), orr + 32 * c);
              tmem_wait_ld();
              reg_fence<RC * 32>(orr);
#pragma unroll
              for (int i = 0; i < RC * 16; ++i) {
                float lo, hi;
                f2_split(f2_mul(f2_make(__uint_as_float(orr[2 * i]), __uint_as_float(orr[2 * i + 1])), a2),
                         lo, hi);
                orr[2 * i] = __float_as_uint(lo);
                orr[2 * i + 1] = __float_as_uint(hi);
              }
#pragma unroll
              for (int c = 0; c < RC; ++c) tmem_st_x32(t_o + 32 * (c0 + c), orr + 32 * c);
            }
          }
          tmem_wait_st();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.p_full[pb * C::NHALF + hf]);
          ++kv_it;
          // the previous tile's epilogue, now that this tile's first P is out
          // (bf16; with E4M3 the call in this loop measured 6 % slower on
          // long tiles, so its epilogue runs at the end of the tile)
          if constexpr (!FP8 && !C::EPI) {
            if (j == 0 && !finish()) {
              ok = false;
              break;
            }
          }
        }
        if (!ok) break;
        if constexpr (C::EPI) {
          // hand the tile to the epilogue warps: this half's row sum and
          // reference maximum into ostat[ob], once the epilogue of the tile
          // that last used O buffer ob has read that slot (it reads the slot
          // before it frees the buffer)
          ++e_it;
          if (!warp_wait(&sm.o_free[ob], (((e_it - 1) / C::NOB) & 1) ^ 1, abort)) {
            if (lane == 0) record_failure(p.status, abort, kSiteSmEpi);
            ok = false;
            break;
          }
          sm.ostat[ob][hf][row_local] = l;
          sm.ostat[ob][C::NHALF + hf][row_local] = m_ref;
          mbar_arrive(&sm.stats_full[ob]);
          continue;
        }
        pend = {true, kv_it - 1, l, m_ref, row_off, row_valid, t.kvbh};
        if constexpr (FP8) {
          if (!finish()) {
            ok = false;
            break;
          }
        }
      }
    }
    if (ok && !finish()) ok = false;
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Cfg<D>::TM_COLS);
  }
}

template <int D, bool DEC, bool FP8 = false, bool BS = false>
cudaError_t launch(const FwdParams& p, int num_sms, int max_smem, cudaStream_t stream) {
  const size_t smem = smem_request(sizeof(FwdSmem<D, FP8>), max_smem);
  cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D, DEC, FP8, BS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  TailTable tail;
  tail.heads = 0;
  long long units;
  if (DEC) {
    units = static_cast<long long>(p.B) * p.H_kv * p.splits;
  } else {
    const int T = (p.N + BM - 1) / BM;
    const int BH = p.B * p.H;
    units = p.causal ? static_cast<long long>(BH) * ((T + 1) / 2) : static_cast<long long>(BH) * T;
    // (the mask planner reads the host copy as [T, T]: tiles and mask blocks
    // are both 128 rows)
    if (p.causal || (BS && p.block_mask_host && T == p.bm_t)) {
      // single tiles in the tail: up to one CTA per tile
      const long long tiles = static_cast<long long>(BH) * T;
      const int g = static_cast<int>(tiles < num_sms ? tiles : num_sms);
      // the tail's heads share their K and V through L2
      const long long kv_bytes = 2ll * p.N * D * (FP8 ? 1 : 2);
      if (p.causal)
        plan_causal_tail(BH, T, 1, g, true, kv_bytes, &tail);
      else                     // tiles cost their computed key blocks
        plan_mask_tail(p.block_mask_host, BH, T, 1, g, true, p.N, p.wl, p.wr, kv_bytes, &tail);
      if (tail.heads > 0) units = g;
    }
  }
  if (tail.heads == 0) std::memset(tail.item, 0xff, sizeof(tail.item));
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  fa_fwd_kernel<D, DEC, FP8, BS><<<grid, Cfg<D, FP8>::THREADS, smem, stream>>>(p, tail);
  return cudaGetLastError();
}

// Merge of the split-KV partials (the associative block merge of "4.
// FlashAttention 深度剖析" 4.2.4, in natural-log units): per row,
// LSE = log sum_s exp(LSE_s) and O = sum_s exp(LSE_s - LSE) O_s, where each O_s
// is already normalised by its own row sum.  One warp per row, D/32 columns a
// lane; a row whose every chunk saw no key gets O = 0, LSE = -inf.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const __grid_constant__ FwdParams p,
                                                             __nv_bfloat16* o, float* lse,
                                                             long long rows) {
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  grid_dependency_wait();                  // the split kernel's partials are complete
  if (row >= rows) return;
  constexpr int PER = D / 32;
  float m = -INFINITY;
  for (int s = 0; s < p.splits; ++s) m = fmaxf(m, p.lse_part[s * rows + row]);
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float sum = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < p.splits; ++s) {
      const float w = expf(p.lse_part[s * rows + row] - m);
      sum += w;
      const float* src = p.o_part + (s * rows + row) * D + lane * PER;
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = fmaf(w, src[i], acc[i]);
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  uint32_t packed[PER / 2];
#pragma unroll
  for (int i = 0; i < PER / 2; ++i) packed[i] = pack_bf16x2(acc[2 * i] * inv, acc[2 * i + 1] * inv);
  uint32_t* dst = reinterpret_cast<uint32_t*>(o + row * D + lane * PER);
#pragma unroll
  for (int i = 0; i < PER / 2; ++i) dst[i] = packed[i];
  if (lane == 0) lse[row] = sum > 0.f ? m + logf(sum) : -INFINITY;
}

}  // namespace

cudaError_t launch_fwd(const FwdParams& p, int d, int num_sms, int max_smem, cudaStream_t stream) {
  switch (d) {
    case 64:
      return p.block_mask ? launch<64, false, false, true>(p, num_sms, max_smem, stream)
                          : launch<64, false>(p, num_sms, max_smem, stream);
    case 128:
      return p.block_mask ? launch<128, false, false, true>(p, num_sms, max_smem, stream)
                          : launch<128, false>(p, num_sms, max_smem, stream);
    case 256:
      return p.block_mask ? launch<256, false, false, true>(p, num_sms, max_smem, stream)
                          : launch<256, false>(p, num_sms, max_smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd_fp8(const FwdParams& p, int d, int num_sms, int max_smem,
                           cudaStream_t stream) {
  switch (d) {
    case 128:
      return p.block_mask ? launch<128, false, true, true>(p, num_sms, max_smem, stream)
                          : launch<128, false, true>(p, num_sms, max_smem, stream);
    case 256:
      return p.block_mask ? launch<256, false, true, true>(p, num_sms, max_smem, stream)
                          : launch<256, false, true>(p, num_sms, max_smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(const FwdParams& p, int d, int num_sms, int max_smem,
                          cudaStream_t stream) {
  switch (d) {
    case 64: return launch<64, true>(p, num_sms, max_smem, stream);
    case 128: return launch<128, true>(p, num_sms, max_smem, stream);
    case 256: return launch<256, true>(p, num_sms, max_smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_combine(const FwdParams& p, int d, void* o, float* lse,
                                  cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.Nq;
  const unsigned grid = static_cast<unsigned>((rows * 32 + 255) / 256);
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
  // Launched as a programmatic dependent of the split kernel, so its launch
  // overlaps that kernel's run instead of following its completion.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (d) {
    case 64: return cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, p, ob, lse, rows);
    case 128: return cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, p, ob, lse, rows);
    case 256: return cudaLaunchKernelEx(&cfg, decode_combine_kernel<256>, p, ob, lse, rows);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
