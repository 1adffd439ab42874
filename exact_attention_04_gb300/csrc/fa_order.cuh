// Cost-sorted deal of a block-sparse schedule, planned on the device (a block
// mask without a host copy; with one, the launch plans a tail on the host).
//
// Every head shares the block mask, so the cost of an item (its computed
// blocks) depends on its tile alone.  The T tiles are sorted by cost, the
// longest first (ties by tile index), and the items (head, tile) follow that
// order; among items of equal cost, head by head, so that the CTAs running at
// the same time share few heads' K and V (forward) or Q and dO (backward)
// through L2.  The items are dealt over the G CTAs in rounds that turn
// direction each round: round r gives item r G + c to CTA c when r is even
// and item r G + G - 1 - c when it is odd, so the CTAs that took the longest
// items of one round take the shortest of the next.  This is the
// longest-first order of LPT scheduling without its search, per item, for
// the least-loaded CTA (which a CTA cannot do for the others at its start).
//
// Position i of the sorted order holds an entry of three 10-bit fields: the
// tile, the first position of the tiles of its cost and their count - 1
// (so T <= kOrderMaxT).
#pragma once
#include <cstdint>

#include "fa_internal.h"

namespace fa {

__host__ __device__ constexpr uint32_t order_entry(int tile, int first, int count) {
  return static_cast<uint32_t>(tile) | (static_cast<uint32_t>(first) << 10) |
         (static_cast<uint32_t>(count - 1) << 20);
}

// The k-th item of the order over BH heads: its head and tile.  The tiles of
// one cost take positions [a, a + n) and so the items [BH a, BH (a + n)).
__device__ __forceinline__ void order_item(const uint32_t* tab, int BH, long long k, int& bh,
                                           int& tile) {
  const uint32_t e = tab[k / BH];
  const int a = static_cast<int>((e >> 10) & 1023u);
  const int n = static_cast<int>((e >> 20) & 1023u) + 1;
  const long long o = k - static_cast<long long>(BH) * a;
  bh = static_cast<int>(o / n);
  tile = static_cast<int>(tab[a + static_cast<int>(o % n)] & 1023u);
}

// Position and entry of tile t in the order, from every tile's cost
// cost[0, T): the tiles before it are the costlier ones and the equally
// costly ones of lower index.
__device__ __forceinline__ int order_rank(const uint32_t* cost, int T, int t, uint32_t& entry) {
  const uint32_t c = cost[t];
  int more = 0, same = 0, same_before = 0;
  for (int u = 0; u < T; ++u) {
    const uint32_t cu = cost[u];
    more += cu > c;
    same += cu == c;
    same_before += (cu == c) & (u < t);
  }
  entry = order_entry(t, more, same);
  return more + same_before;
}

// Item k of CTA `cta`'s round r in the turning deal over G CTAs.
__device__ __forceinline__ long long order_deal(int r, int G, int cta) {
  return static_cast<long long>(r) * G + ((r & 1) ? G - 1 - cta : cta);
}

}  // namespace fa
