// Visibility of keys to queries, shared by the forward and backward kernels.
//
// Key j is visible to query i iff j < len (the batch entry's kv_len),
// j >= i - wl and j <= i + wr.  The host folds the causal flag into wr
// (wr = 0) and stores an unbounded side as kUnbounded, so every mask is the
// same three comparisons.  The window is flash-attn's window_size=(left,
// right) ("炉案与百步之外的仓库：Flash Attention 与注意力计算的工艺极限"
// section 六; "4. FlashAttention 深度剖析" 4.8.1); blocks outside it are
// skipped, not masked ("深入浅出 FlashAttention：快如闪电的精确注意力机制与
// IO 感知计算" 第八部分, block-sparse skipping).
#pragma once
#include <cstdint>

namespace fa {

// An unbounded window side.  Query and key indices stay below 2^30, so
// i +- kUnbounded never overflows an int.
constexpr int kUnbounded = 1 << 30;

// Key range [k_lo, k_hi) that query rows [r0, r0 + nrows) can see.
__device__ __forceinline__ void visible_keys(int r0, int nrows, int len, int wl, int wr,
                                             int& k_lo, int& k_hi) {
  k_lo = r0 - wl;
  if (k_lo < 0) k_lo = 0;
  k_hi = r0 + nrows - 1 + wr + 1;
  if (k_hi > len) k_hi = len;
}

// Query range [q_lo, q_hi) that keys [k0, k0 + nkeys) are visible to, among
// N queries (empty when every key is past len).
__device__ __forceinline__ void visible_queries(int k0, int nkeys, int len, int N, int wl,
                                                int wr, int& q_lo, int& q_hi) {
  if (k0 >= len) {
    q_lo = q_hi = 0;
    return;
  }
  const int k_last = (k0 + nkeys < len ? k0 + nkeys : len) - 1;
  q_lo = k0 - wr;
  if (q_lo < 0) q_lo = 0;
  q_hi = k_last + wl + 1;
  if (q_hi > N) q_hi = N;
}

// K/V head of query head (b, h) when H query heads share H_kv K/V heads
// (the same index when they do not share).
__device__ __forceinline__ int kv_head_of(int bh, int H, int H_kv) {
  if (H_kv == H) return bh;
  return (bh / H) * H_kv + (bh % H) / (H / H_kv);
}

// Query head (b, h) of member gi of K/V head kvbh's group.
__device__ __forceinline__ int q_head_of(int kvbh, int gi, int H, int H_kv) {
  if (H_kv == H) return kvbh + gi;
  return (kvbh / H_kv) * H + (kvbh % H_kv) * (H / H_kv) + gi;
}

// The steps of a backward work item in order: query blocks [i0, i1) of the
// group's first query head, then of the next, ...  Kept as counters so that a
// step costs no integer division.
// Block-sparse attention: column n of the row-major [T, T] block mask
// (col = mask + n, stride T), read for query steps that are spb to a 128-row
// query block; a null column computes every step.
struct StepMask {
  const uint8_t* col;
  int stride, spb;
  __device__ __forceinline__ bool on(int s) const {
    return !col || __ldg(col + static_cast<size_t>(s / spb) * stride) != 0;
  }
};

// Steps of [i0, i1) the mask computes.
__device__ __forceinline__ int count_steps(const StepMask& m, int i0, int i1) {
  if (!m.col) return i1 > i0 ? i1 - i0 : 0;
  int c = 0;
  for (int s = i0; s < i1; ++s) c += m.on(s);
  return c;
}

struct StepWalk {
  int i, bh, i0, i1;
  StepMask m;
  __device__ __forceinline__ StepWalk(int i0_, int i1_, int bh0,
                                      const StepMask& m_ = StepMask{nullptr, 0, 1})
      : i(i0_), bh(bh0), i0(i0_), i1(i1_), m(m_) {
    i = skip(i0);
  }
  __device__ __forceinline__ int skip(int s) const {
    while (s < i1 && !m.on(s)) ++s;
    return s;
  }
  __device__ __forceinline__ void next() {
    i = skip(i + 1);
    if (i >= i1) {
      i = skip(i0);
      ++bh;
    }
  }
};

}  // namespace fa
