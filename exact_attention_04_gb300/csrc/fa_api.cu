// C-ABI front end: argument validation, TMA tensor maps, the per-device
// status word, and dispatch to the kernels.  No allocation, no
// synchronisation (except fa_check), no host copies.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "fa_window.cuh"

// Written by kernels that gave up waiting; read and cleared by fa_check.
__device__ int g_fa_status;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  bool supported = false;
  int num_sms = 0;
  int max_smem = 0;        // opt-in dynamic shared memory per block
  int* status = nullptr;   // device address of g_fa_status on this device
};

DeviceInfo g_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// Per-device facts, looked up once with that device current.
DeviceInfo* device_info(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo& di = g_dev[dev];
  std::call_once(di.once, [&di, dev] {
    int major = 0, minor = 0;
    di.err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (di.err == cudaSuccess)
      di.err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (di.err == cudaSuccess)
      di.err = cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (di.err == cudaSuccess)
      di.err = cudaDeviceGetAttribute(&di.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    di.supported = (major == 10 && minor == 3);
    if (di.err == cudaSuccess && di.supported)
      di.err = cudaGetSymbolAddress(reinterpret_cast<void**>(&di.status), g_fa_status);
  });
  if (dev_out) *dev_out = dev;
  return &di;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status_t check_sizes(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  const long long elems = static_cast<long long>(B) * H * N * d;
  if (elems >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// bf16 [BH, N, d] as a 3-D tensor (d, N, BH): box of 64 columns x box_rows
// rows, 128-byte swizzle, rows past N read as zero.
bool make_map(CUtensorMap* m, const void* base, int d, int N, int BH, int box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(d) * N * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Byte tensor (E4M3) [depth, rows, inner] as 3-D (inner, rows, depth): box of
// box_inner bytes x box_rows rows, 128-byte swizzle, out-of-range reads zero.
bool make_map_u8(CUtensorMap* m, const void* base, int inner, int rows, int depth, int box_inner,
                 int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(depth)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner),
                                 static_cast<cuuint64_t>(inner) * rows};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner),
                             static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Transposed fp32 accumulator [BH, d, Npad] as a 3-D tensor (Npad, d, BH):
// box of 32 queries (128 bytes) x 128 head-dimension rows, 128-byte swizzle
// (the target of bulk reduce-adds).
bool make_acc_map(CUtensorMap* m, void* base, int d, int npad, int BH) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(npad), static_cast<cuuint64_t>(d),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(npad) * 4,
                                 static_cast<cuuint64_t>(npad) * d * 4};
  const cuuint32_t box[3] = {32, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 accumulator [BH, Npad, d] (d = 64) as a 3-D tensor (d, Npad, BH): box
// of 32 columns (128 bytes) x 128 rows, 128-byte swizzle (the target of bulk
// reduce-adds).
bool make_acc_rows_map(CUtensorMap* m, void* base, int d, int npad, int BH) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(npad),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                 static_cast<cuuint64_t>(npad) * d * 4};
  const cuuint32_t box[3] = {32, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t round_up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The variant as the kernels see it: K/V heads, and the window folded with
// causal into the bounds wl, wr (key j visible to query i iff
// i - wl <= j <= i + wr), unbounded sides as fa::kUnbounded.  `pair` is true
// for plain causal attention (no block mask), where the schedule pairs long
// and short tiles.  bm: the block mask or nullptr.
struct Variant {
  int H_kv, wl, wr;
  bool pair;
  const uint8_t* bm;
  const uint8_t* bmh;    // host copy of bm, or nullptr
};

fa_status_t resolve_variant(const fa_variant_t* var, int H, int causal, Variant* out) {
  const int h_kv = var ? var->h_kv : H;
  const int left = var ? var->window_left : -1;
  const int right = var ? var->window_right : -1;
  if (h_kv < 1 || h_kv > H || H % h_kv != 0 || left < -1 || right < -1)
    return FA_ERR_INVALID_ARG;
  out->H_kv = h_kv;
  out->wl = left < 0 ? fa::kUnbounded : left;
  out->wr = right < 0 ? fa::kUnbounded : right;
  if (causal && out->wr > 0) out->wr = 0;
  out->bm = var ? var->block_mask : nullptr;
  out->bmh = out->bm ? var->block_mask_host : nullptr;
  out->pair = causal && left < 0 && !out->bm;
  return FA_OK;
}

}  // namespace

namespace fa {

namespace {

// The plan itself (see plan_causal_tail and plan_mask_tail).  cost[blk]: one
// item of block blk, the same in every head and half; pair: the round-robin
// units pair blocks pp and T - 1 - pp (causal), else each is one item.
void plan_tail_uncached(int BH, int T, int nsplit, int G, bool pair,
                        const std::vector<long long>& cost, long long head_bytes, TailTable* t) {
  std::memset(t->item, 0xff, sizeof(t->item));         // every entry -1
  t->heads = 0;
  if (BH < 1 || T < 1 || T > 2048 || nsplit < 1 || nsplit > 2 || G < 1 || G > kTailCtas) return;
  const int per = pair ? (T + 1) / 2 : T;                // round-robin units of one head
  std::vector<long long> unit_cost(per);
  for (int pp = 0; pp < per; ++pp)
    unit_cost[pp] = !pair || pp == T - 1 - pp ? cost[pp] : cost[pp] + cost[T - 1 - pp];
  // the tail's items longest first (ties in block order)
  std::vector<int> order(T);
  for (int b = 0; b < T; ++b) order[b] = b;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cost[a] > cost[b]; });
  // about six tail items a CTA on average, at most kTailL2Bytes of streamed
  // data; fewer heads if a CTA would overflow its row
  const long long by_l2 = head_bytes > 0 ? std::max(1ll, kTailL2Bytes / head_bytes) : BH;
  const int first = static_cast<int>(
      std::max(1ll, std::min({static_cast<long long>(BH), 6ll * G / (T * nsplit), by_l2})));
  // with this many rounds of units the last one does not matter
  if (static_cast<long long>(BH - first) * per * nsplit > (1ll << 18)) return;
  std::vector<long long> load(G);
  std::vector<int> count(G);
  using Slot = std::pair<long long, int>;                // (work so far, CTA)
  for (int heads = first; heads >= 1; --heads) {
    std::fill(load.begin(), load.end(), 0ll);
    std::fill(count.begin(), count.end(), 0);
    // round-robin: unit u (unit (u / nsplit) % per of its head) on CTA u % G
    const long long units = static_cast<long long>(BH - heads) * per * nsplit;
    int c = 0, half = 0, pp = 0;
    for (long long u = 0; u < units; ++u) {
      load[c] += unit_cost[pp];
      if (++c == G) c = 0;
      if (++half == nsplit) {
        half = 0;
        if (++pp == per) pp = 0;
      }
    }
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> least;
    for (int k = 0; k < G; ++k) least.push({load[k], k});
    bool fits = true;
    for (int r = 0; r < T && fits; ++r) {
      const int blk = order[r];
      for (int h = BH - heads; h < BH && fits; ++h) {
        for (int s = 0; s < nsplit; ++s) {
          const Slot top = least.top();
          least.pop();
          const int k = top.second;
          if (count[k] == kTailItems) {
            fits = false;
            break;
          }
          t->item[k][count[k]++] = tail_code(h, s, blk);
          least.push({top.first + cost[blk], k});
        }
      }
    }
    if (fits) {
      t->heads = heads;
      return;
    }
    std::memset(t->item, 0xff, sizeof(t->item));
  }
}

// The last few plans: a training loop asks for the same few shapes (and
// masks) on every step, and a plan is a pure function of its arguments.  A
// plan is keyed by a hash of its costs: two cost vectors that collide would
// share a plan that balances one of them less well, but any plan for the same
// (BH, T, nsplit, G) runs every item exactly once.
struct TailPlanCache {
  struct Entry {
    bool used;
    int BH, T, nsplit, G;
    bool pair;
    long long head_bytes;
    uint64_t cost_hash;
    TailTable table;
  };
  static constexpr int kEntries = 8;
  std::mutex mu;
  Entry e[kEntries] = {};
  int next = 0;
};

TailPlanCache& tail_plan_cache() {
  static TailPlanCache cache;
  return cache;
}

uint64_t hash_costs(const std::vector<long long>& cost) {
  uint64_t h = 1469598103934665603ull;                  // FNV-1a over the 8-byte values
  for (long long c : cost) {
    uint64_t v = static_cast<uint64_t>(c);
    for (int i = 0; i < 8; ++i, v >>= 8) h = (h ^ (v & 0xff)) * 1099511628211ull;
  }
  return h;
}

void plan_tail(int BH, int T, int nsplit, int G, bool pair, const std::vector<long long>& cost,
               long long head_bytes, TailTable* t) {
  const uint64_t hc = hash_costs(cost);
  TailPlanCache& cache = tail_plan_cache();
  {
    std::lock_guard<std::mutex> lock(cache.mu);
    for (const auto& en : cache.e)
      if (en.used && en.BH == BH && en.T == T && en.nsplit == nsplit && en.G == G &&
          en.pair == pair && en.head_bytes == head_bytes && en.cost_hash == hc) {
        *t = en.table;
        return;
      }
  }
  plan_tail_uncached(BH, T, nsplit, G, pair, cost, head_bytes, t);
  std::lock_guard<std::mutex> lock(cache.mu);
  TailPlanCache::Entry& en = cache.e[cache.next];
  cache.next = (cache.next + 1) % TailPlanCache::kEntries;
  en.used = true;
  en.BH = BH;
  en.T = T;
  en.nsplit = nsplit;
  en.G = G;
  en.pair = pair;
  en.head_bytes = head_bytes;
  en.cost_hash = hc;
  en.table = *t;
}

// Start-up and epilogue of an item, in blocks / steps: a clock64 trace of one
// CTA puts a forward tile boundary near 3 key blocks' time and a backward
// key-block boundary near 4 query steps'.
long long item_fixed_cost(bool fwd) { return fwd ? 3 : 4; }

}  // namespace

void plan_causal_tail(int BH, int T, int nsplit, int G, bool fwd, long long head_bytes,
                      TailTable* t) {
  if (T < 1 || T > 2048) {
    std::memset(t->item, 0xff, sizeof(t->item));
    t->heads = 0;
    return;
  }
  std::vector<long long> cost(T);
  for (int b = 0; b < T; ++b) cost[b] = (fwd ? b + 1 : 2ll * (T - b)) + item_fixed_cost(fwd);
  plan_tail(BH, T, nsplit, G, true, cost, head_bytes, t);
}

void plan_mask_tail(const uint8_t* bm_host, int BH, int T, int nsplit, int G, bool fwd, int N,
                    int wl, int wr, long long head_bytes, TailTable* t) {
  if (!bm_host || T < 1 || T > 2048) {
    std::memset(t->item, 0xff, sizeof(t->item));
    t->heads = 0;
    return;
  }
  // the window in 64-bit: an unbounded side is 2^30
  std::vector<long long> cost(T);
  for (int b = 0; b < T; ++b) {
    const long long lo0 = 128ll * b, hi0 = std::min<long long>(128ll * b + 128, N);   // [lo0, hi0)
    long long lo, hi;                    // the other side's visible positions [lo, hi)
    if (fwd) {                           // keys seen by query rows [lo0, hi0)
      lo = std::max(0ll, lo0 - wl);
      hi = std::min<long long>(N, hi0 - 1 + wr + 1);
    } else {                             // queries that see keys [lo0, hi0)
      lo = std::max(0ll, lo0 - wr);
      hi = std::min<long long>(N, hi0 - 1 + wl + 1);
    }
    long long n = 0;
    if (hi > lo)
      for (long long o = lo / 128; o < (hi + 127) / 128; ++o)
        n += (fwd ? bm_host[static_cast<size_t>(b) * T + o]
                  : bm_host[static_cast<size_t>(o) * T + b]) != 0;
    cost[b] = (fwd ? n : 2 * n) + item_fixed_cost(fwd);
  }
  plan_tail(BH, T, nsplit, G, false, cost, head_bytes, t);
}

}  // namespace fa

extern "C" {

int fa_version(void) { return 1 * 10000 + 2 * 100 + 0; }

const char* fa_status_string(fa_status_t s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
  }
  return "FA_ERR_UNKNOWN";
}

fa_status_t fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int H, int N, int d, float scale, int causal, const int* kv_len,
                   void* stream) {
  return fa_fwd_v(q, k, v, o, lse, B, H, N, d, scale, causal, kv_len, nullptr, stream);
}

fa_status_t fa_fwd_v(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, float scale, int causal, const int* kv_len,
                     const fa_variant_t* variant, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_INVALID_ARG;
  if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return FA_ERR_INVALID_ARG;
  const fa_status_t sz = check_sizes(B, H, N, d, scale);
  if (sz != FA_OK) return sz;
  Variant var;
  const fa_status_t vs = resolve_variant(variant, H, causal, &var);
  if (vs != FA_OK) return vs;
  DeviceInfo* di = device_info(nullptr);
  if (!di || di->err != cudaSuccess) return FA_ERR_CUDA;
  if (!di->supported) return FA_ERR_UNSUPPORTED;
  fa::FwdParams p;
  std::memset(&p, 0, sizeof(p));
  const int BH = B * H;
  if (!make_map(&p.tq, q, d, N, BH) || !make_map(&p.tk, k, d, N, B * var.H_kv) ||
      !make_map(&p.tv, v, d, N, B * var.H_kv))
    return FA_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.kv_len = kv_len;
  p.B = B;
  p.H = H;
  p.N = N;
  p.H_kv = var.H_kv;
  p.wl = var.wl;
  p.wr = var.wr;
  p.causal = var.pair ? 1 : 0;
  p.block_mask = var.bm;
  p.bm_t = (N + 127) / 128;
  p.block_mask_host = var.bmh;
  // a block mask without a host copy: each CTA sorts the tiles by cost
  p.cost_sorted = (var.bm && !var.bmh && !p.causal && p.bm_t <= fa::kFwdOrderMaxT) ? 1 : 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.status = di->status;
  if (fa::launch_fwd(p, d, di->num_sms, di->max_smem, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

// Workspace layout: D [B*H, Npad] fp32, L2 [B*H, Npad] fp32, dQ_acc of
// B*H*Npad*d fp32 ([B*H, Npad, d] for d = 64, [B*H, d, Npad] otherwise), and
// the cost-sorted order of the key blocks (Npad / 128 uint32, used with a
// block mask that has no host copy), each region starting on a 256-byte
// boundary (Npad = N rounded up to 128).
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_sizes(B, H, N, d, 1.f) != FA_OK) return 0;
  const size_t npad = (static_cast<size_t>(N) + 127) / 128 * 128;
  const size_t padded_rows = static_cast<size_t>(B) * H * npad;
  return 2 * round_up256(padded_rows * sizeof(float)) +
         round_up256(padded_rows * d * sizeof(float)) +
         round_up256(npad / 128 * sizeof(uint32_t));
}

}  // extern "C"

namespace {

// Common checks of the backward entry points and the parameter block they
// share.  Pointer arguments are checked by each caller.
fa_status_t bwd_setup(fa::BwdParams* p, DeviceInfo** di, int B, int H, int N, int d, float scale,
                      int causal, const int* kv_len, const fa_variant_t* variant,
                      void* workspace, size_t workspace_bytes) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FA_ERR_INVALID_ARG;
  if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return FA_ERR_INVALID_ARG;
  const fa_status_t sz = check_sizes(B, H, N, d, scale);
  if (sz != FA_OK) return sz;
  Variant var;
  const fa_status_t vs = resolve_variant(variant, H, causal, &var);
  if (vs != FA_OK) return vs;
  if (workspace_bytes < fa_bwd_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID_ARG;
  *di = device_info(nullptr);
  if (!*di || (*di)->err != cudaSuccess) return FA_ERR_CUDA;
  if (!(*di)->supported) return FA_ERR_UNSUPPORTED;
  std::memset(p, 0, sizeof(*p));
  const int BH = B * H;
  const int npad = (N + 127) / 128 * 128;
  const size_t stat_bytes = round_up256(static_cast<size_t>(BH) * npad * sizeof(float));
  p->delta = static_cast<float*>(workspace);
  p->lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + stat_bytes);
  p->dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + 2 * stat_bytes);
  const size_t acc_bytes = round_up256(static_cast<size_t>(BH) * npad * d * sizeof(float));
  p->Npad = npad;
  p->kv_len = kv_len;
  p->B = B;
  p->H = H;
  p->N = N;
  p->H_kv = var.H_kv;
  p->wl = var.wl;
  p->wr = var.wr;
  p->causal = var.pair ? 1 : 0;
  p->block_mask = var.bm;
  p->bm_t = (N + 127) / 128;
  p->block_mask_host = var.bmh;
  // a block mask without a host copy: the key blocks' cost-sorted order,
  // planned on the device into the workspace's last region
  if (var.bm && !var.bmh && !p->causal && p->bm_t <= fa::kOrderMaxT)
    p->cost_order = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + 2 * stat_bytes +
                                                acc_bytes);
  p->scale = scale;
  p->scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p->status = (*di)->status;
  return FA_OK;
}

}  // namespace

namespace fa {

// The checks fa_bwd makes, in fa_bwd's order and with its status codes, for
// a caller that supplies a workspace of exactly workspace_bytes at a valid
// address: pointers, kv_len, sizes, the workspace size, then the device.
fa_status_t bwd_check_args(const void* q, const void* k, const void* v, const void* o,
                           const void* dO, const float* lse, const void* dq, const void* dk,
                           const void* dv, int B, int H, int N, int d, float scale,
                           int causal, const int* kv_len, size_t workspace_bytes) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || !aligned16(dq) || !aligned16(dk) ||
      !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return FA_ERR_INVALID_ARG;
  const fa_status_t sz = check_sizes(B, H, N, d, scale);
  if (sz != FA_OK) return sz;
  Variant var;
  const fa_status_t vs = resolve_variant(nullptr, H, causal, &var);
  if (vs != FA_OK) return vs;
  if (workspace_bytes < fa_bwd_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID_ARG;
  DeviceInfo* di = device_info(nullptr);
  if (!di || di->err != cudaSuccess) return FA_ERR_CUDA;
  if (!di->supported) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

}  // namespace fa

namespace {

fa_status_t bwd_prep_impl(const fa::BwdParams& p, int d, void* stream) {
  return fa::launch_bwd_prep(p, d, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                     : FA_ERR_CUDA;
}

fa_status_t bwd_main_impl(fa::BwdParams& p, const DeviceInfo* di, const void* q, const void* k,
                          const void* v, const void* dO, int d, void* stream) {
  const int BH = p.B * p.H;
  // d = 64: 128-query steps with dQ in query rows (fa_bwd_d64.cu); d = 128,
  // 256: 64-query steps with dQ^T in head-dimension rows (fa_bwd_dt.cu).
  const bool dt = d != 64;
  const int qrows = dt ? 64 : 128;
  const int BHkv = p.B * p.H_kv;
  if (!make_map(&p.tq, q, d, p.N, BH, qrows) || !make_map(&p.tk, k, d, p.N, BHkv) ||
      !make_map(&p.tv, v, d, p.N, BHkv) || !make_map(&p.tdo, dO, d, p.N, BH, qrows))
    return FA_ERR_CUDA;
  if (dt && !make_acc_map(&p.tdq, p.dq_acc, d, p.Npad, BH)) return FA_ERR_CUDA;
  if (!dt && !make_acc_rows_map(&p.tdq, p.dq_acc, d, p.Npad, BH)) return FA_ERR_CUDA;
  p.v = v;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.cost_order && fa::launch_bwd_order(p, s) != cudaSuccess) return FA_ERR_CUDA;
  const cudaError_t e = dt ? fa::launch_bwd_main_dt(p, d, di->num_sms, di->max_smem, s)
                           : fa::launch_bwd_main_d64(p, di->num_sms, di->max_smem, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t bwd_post_impl(const fa::BwdParams& p, int d, void* stream) {
  return fa::launch_bwd_post(p, d, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                     : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

fa_status_t fa_bwd_prep(const void* o, const void* dO, const float* lse, int B, int H, int N,
                        int d, void* workspace, size_t workspace_bytes, void* stream) {
  if (!o || !dO || !lse || !aligned16(o) || !aligned16(dO) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_INVALID_ARG;
  fa::BwdParams p;
  DeviceInfo* di = nullptr;
  const fa_status_t st = bwd_setup(&p, &di, B, H, N, d, 1.f, 0, nullptr, nullptr, workspace,
                                   workspace_bytes);
  if (st != FA_OK) return st;
  p.o = o;
  p.dO = dO;
  p.lse = lse;
  return bwd_prep_impl(p, d, stream);
}

fa_status_t fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk,
                        void* dv, int B, int H, int N, int d, float scale, int causal,
                        const int* kv_len, void* workspace, size_t workspace_bytes,
                        void* stream) {
  return fa_bwd_dkdv_v(q, k, v, dO, dk, dv, B, H, N, d, scale, causal, kv_len, nullptr,
                       workspace, workspace_bytes, stream);
}

fa_status_t fa_bwd_dkdv_v(const void* q, const void* k, const void* v, const void* dO, void* dk,
                          void* dv, int B, int H, int N, int d, float scale, int causal,
                          const int* kv_len, const fa_variant_t* variant, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !dO || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dk) ||
      !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  fa::BwdParams p;
  DeviceInfo* di = nullptr;
  const fa_status_t st = bwd_setup(&p, &di, B, H, N, d, scale, causal, kv_len, variant,
                                   workspace, workspace_bytes);
  if (st != FA_OK) return st;
  p.dk = dk;
  p.dv = dv;
  return bwd_main_impl(p, di, q, k, v, dO, d, stream);
}

fa_status_t fa_bwd_dq(void* dq, int B, int H, int N, int d, float scale, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!dq || !aligned16(dq)) return FA_ERR_INVALID_ARG;
  fa::BwdParams p;
  DeviceInfo* di = nullptr;
  const fa_status_t st = bwd_setup(&p, &di, B, H, N, d, scale, 0, nullptr, nullptr, workspace,
                                   workspace_bytes);
  if (st != FA_OK) return st;
  p.dq = dq;
  return bwd_post_impl(p, d, stream);
}

fa_status_t fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   float scale, int causal, const int* kv_len, void* workspace,
                   size_t workspace_bytes, void* stream) {
  return fa_bwd_v(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, kv_len, nullptr,
                  workspace, workspace_bytes, stream);
}

fa_status_t fa_bwd_v(const void* q, const void* k, const void* v, const void* o,
                     const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                     int H, int N, int d, float scale, int causal, const int* kv_len,
                     const fa_variant_t* variant, void* workspace, size_t workspace_bytes,
                     void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || !aligned16(dq) || !aligned16(dk) ||
      !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  fa::BwdParams p;
  DeviceInfo* di = nullptr;
  const fa_status_t st = bwd_setup(&p, &di, B, H, N, d, scale, causal, kv_len, variant,
                                   workspace, workspace_bytes);
  if (st != FA_OK) return st;
  p.o = o;
  p.dO = dO;
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  fa_status_t r = bwd_prep_impl(p, d, stream);
  if (r == FA_OK) r = bwd_main_impl(p, di, q, k, v, dO, d, stream);
  if (r == FA_OK) r = bwd_post_impl(p, d, stream);
  return r;
}

int fa_decode_splits(int B, int H_kv, int Nk) {
  if (B < 1 || H_kv < 1 || Nk < 1) return 0;
  DeviceInfo* di = device_info(nullptr);
  const int sms = (di && di->err == cudaSuccess && di->num_sms > 0) ? di->num_sms : 148;
  const long long heads = static_cast<long long>(B) * H_kv;
  const int nblk = (Nk + 127) / 128;
  // Fewer K/V heads than SMs: the most chunks that still run in one wave (a
  // unit pays a fixed cost for its Q load, pipeline fill and epilogue, so one
  // wave of long chunks measured faster than four full waves of short ones:
  // 4 x 8 heads, 32K keys: 5.2 TB/s with 4 chunks per head, 4.7 with 19),
  // keeping chunks of at least 8 key blocks.
  if (heads < sms) {
    const long long by_sms = sms / heads;
    const long long by_len = nblk / 8 > 1 ? nblk / 8 : 1;
    return static_cast<int>(by_sms < by_len ? by_sms : by_len);
  }
  // Otherwise chunks of at least 8 key blocks; among those, the count whose
  // units fill the SMs' waves best (ties: fewer chunks, less merging).
  int best = 1;
  double best_eff = -1.0;
  for (int s = 1; s <= nblk; ++s) {
    const int chunk = (nblk + s - 1) / s;
    const int eff_s = (nblk + chunk - 1) / chunk;
    if (eff_s != s || (s > 1 && chunk < 8)) continue;
    const long long units = heads * s;
    const long long waves = (units + sms - 1) / sms;
    const double eff = static_cast<double>(units) / static_cast<double>(waves * sms);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = s;
    }
    if (units >= 4ll * sms) break;
  }
  return best;
}

size_t fa_decode_workspace_bytes(int B, int H, int Nq, int d, int splits) {
  if (B < 1 || H < 1 || Nq < 1 || splits < 1 || (d != 64 && d != 128 && d != 256)) return 0;
  const size_t rows = static_cast<size_t>(B) * H * Nq * splits;
  return round_up256(rows * d * sizeof(float)) + round_up256(rows * sizeof(float));
}

fa_status_t fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Nq, int Nk, int d, float scale, int causal, const int* kv_len,
                      const fa_variant_t* variant, int splits, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FA_ERR_INVALID_ARG;
  if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || splits < 1) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  Variant var;
  const fa_status_t vs = resolve_variant(variant, H, causal, &var);
  if (vs != FA_OK) return vs;
  if (var.bm) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * Nq * d >= (1ll << 31) ||
      static_cast<long long>(B) * var.H_kv * Nk * d >= (1ll << 31))
    return FA_ERR_INVALID_ARG;
  if ((H / var.H_kv) * Nq > 128) return FA_ERR_UNSUPPORTED;   // one 128-row tile per K/V head
  if (workspace_bytes < fa_decode_workspace_bytes(B, H, Nq, d, splits)) return FA_ERR_INVALID_ARG;
  DeviceInfo* di = device_info(nullptr);
  if (!di || di->err != cudaSuccess) return FA_ERR_CUDA;
  if (!di->supported) return FA_ERR_UNSUPPORTED;
  fa::FwdParams p;
  std::memset(&p, 0, sizeof(p));
  const int rows = B * H * Nq;
  if (!make_map(&p.tq, q, d, rows, 1) || !make_map(&p.tk, k, d, Nk, B * var.H_kv) ||
      !make_map(&p.tv, v, d, Nk, B * var.H_kv))
    return FA_ERR_CUDA;
  const int nblk = (Nk + 127) / 128;
  const int chunk = (nblk + splits - 1) / splits;
  p.kv_len = kv_len;
  p.B = B;
  p.H = H;
  p.N = Nk;
  p.H_kv = var.H_kv;
  p.wl = var.wl;
  p.wr = var.wr;
  p.causal = 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.status = di->status;
  p.Nq = Nq;
  p.chunk_blocks = chunk;
  p.splits = (nblk + chunk - 1) / chunk;
  p.o_part = static_cast<float*>(workspace);
  p.lse_part = reinterpret_cast<float*>(
      static_cast<char*>(workspace) +
      round_up256(static_cast<size_t>(rows) * splits * d * sizeof(float)));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fa::launch_decode(p, d, di->num_sms, di->max_smem, s) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::launch_decode_combine(p, d, o, lse, s) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

fa_status_t fa_fp8_quantize(const void* q, const void* k, const void* v, int B, int H, int N,
                            int d, const fa_variant_t* variant, void* q8, float* q_scale,
                            void* k8, float* k_scale, void* v8t, float* v_scale, void* stream) {
  if (!q || !k || !v || !q8 || !q_scale || !k8 || !k_scale || !v8t || !v_scale)
    return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q8) || !aligned16(k8) ||
      !aligned16(v8t) || (reinterpret_cast<uintptr_t>(q_scale) & 3u) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return FA_ERR_INVALID_ARG;
  const fa_status_t sz = check_sizes(B, H, N, d, 1.f);
  if (sz != FA_OK) return sz;
  if (d == 64) return FA_ERR_UNSUPPORTED;
  Variant var;
  const fa_status_t vs = resolve_variant(variant, H, 0, &var);
  if (vs != FA_OK) return vs;
  DeviceInfo* di = device_info(nullptr);
  if (!di || di->err != cudaSuccess) return FA_ERR_CUDA;
  if (!di->supported) return FA_ERR_UNSUPPORTED;
  fa::Fp8QuantArgs a{q, k, v, B, H, var.H_kv, N, q8, q_scale, k8, k_scale, v8t, v_scale};
  return fa::launch_fp8_quantize(a, d, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status_t fa_fwd_fp8(const void* q8, const float* q_scale, const void* k8,
                       const float* k_scale, const void* v8t, const float* v_scale, void* o,
                       float* lse, int B, int H, int N, int d, float scale, int causal,
                       const int* kv_len, const fa_variant_t* variant, void* stream) {
  if (!q8 || !q_scale || !k8 || !k_scale || !v8t || !v_scale || !o || !lse)
    return FA_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8t) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(q_scale) & 3u) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return FA_ERR_INVALID_ARG;
  if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return FA_ERR_INVALID_ARG;
  const fa_status_t sz = check_sizes(B, H, N, d, scale);
  if (sz != FA_OK) return sz;
  if (d == 64) return FA_ERR_UNSUPPORTED;
  Variant var;
  const fa_status_t vs = resolve_variant(variant, H, causal, &var);
  if (vs != FA_OK) return vs;
  DeviceInfo* di = device_info(nullptr);
  if (!di || di->err != cudaSuccess) return FA_ERR_CUDA;
  if (!di->supported) return FA_ERR_UNSUPPORTED;
  fa::FwdParams p;
  std::memset(&p, 0, sizeof(p));
  const int nb = (N + 127) / 128;
  if (!make_map_u8(&p.tq, q8, d, N, B * H, 128, 128) ||
      !make_map_u8(&p.tk, k8, d, N, B * var.H_kv, 128, 128) ||
      !make_map_u8(&p.tv, v8t, nb * 128, d, B * var.H_kv, 128, d))
    return FA_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.kv_len = kv_len;
  p.B = B;
  p.H = H;
  p.N = N;
  p.H_kv = var.H_kv;
  p.wl = var.wl;
  p.wr = var.wr;
  p.causal = var.pair ? 1 : 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.status = di->status;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.nb = nb;
  p.block_mask = var.bm;
  p.bm_t = nb;
  p.block_mask_host = var.bmh;
  p.cost_sorted = (var.bm && !var.bmh && !p.causal && nb <= fa::kFwdOrderMaxT) ? 1 : 0;
  return fa::launch_fwd_fp8(p, d, di->num_sms, di->max_smem, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status_t fa_selftest_wait_timeout(unsigned int timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 1000000u) return FA_ERR_INVALID_ARG;
  DeviceInfo* di = device_info(nullptr);
  if (!di || di->err != cudaSuccess) return FA_ERR_CUDA;
  if (!di->supported) return FA_ERR_UNSUPPORTED;
  return fa::launch_wait_selftest(di->status, 1000ull * timeout_us,
                                  static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status_t fa_check(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  DeviceInfo* di = device_info(nullptr);
  if (!di || di->err != cudaSuccess || !di->supported) return FA_ERR_CUDA;
  int status = 0;
  if (cudaMemcpyFromSymbol(&status, g_fa_status, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (status != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    return (status & 0xff) == fa::kStatusTimeout ? FA_ERR_TIMEOUT : FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // extern "C"
