// Internal interface between the C-ABI front end (fa_api.cu) and the kernel
// translation units.  Not installed; not part of the public header.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa {

// Device status word values written by kernels that gave up waiting:
// low byte FA_ERR_TIMEOUT (4), the rest identifies the wait site.
constexpr int kStatusTimeout = 4;
__host__ __device__ constexpr int status_code(int site) { return kStatusTimeout | (site << 8); }

// Kernels give up on any single wait after this much global time.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

struct FwdParams {
  CUtensorMap tq, tk, tv;      // bf16 [BH, N, d] viewed as 3-D (d, N, BH), box (64, 128, 1), SW128
  void* o;                     // bf16 [B, H, N, d]
  float* lse;                  // fp32 [B, H, N]
  const int* kv_len;           // int32 [B] or nullptr
  int B, H, N;
  int H_kv;                    // K/V heads; query head h reads K/V head h / (H / H_kv)
  int wl, wr;                  // key j visible to query i iff i - wl <= j <= i + wr (and j < len)
  int causal;                  // causal pairing of tiles in the schedule (plain causal only)
  float scale_log2;            // scale * log2(e)
  int* status;                 // device status word
  // decode (split-KV) mode: N is the number of keys; Q is viewed as
  // [B*H*Nq, d] and query t of a head sits at position len - Nq + t
  int Nq;
  int splits, chunk_blocks;    // key chunks per K/V head, key blocks per chunk
  float* o_part;               // fp32 [splits, B*H*Nq, d] partial outputs (normalised)
  float* lse_part;             // fp32 [splits, B*H*Nq] partial log-sum-exp (natural log)
  // FP8 mode: E4M3 Q, K and transposed V with their dequantisation scales
  const float* q_scale;        // [B*H, nb], one per 128-row tile
  const float* k_scale;        // [B*H_kv, nb], one per 128-key block
  const float* v_scale;        // [B*H_kv]
  int nb;                      // ceil(N / 128)
  // block-sparse: [bm_t, bm_t] bytes, nonzero where (query block, key block)
  // is computed (blocks of 128), or nullptr
  const uint8_t* block_mask;
  int bm_t;
  // a host copy of the block mask, or nullptr; read by the launch (never by a
  // kernel) to balance the schedule
  const uint8_t* block_mask_host;
  // nonzero: a block mask without a host copy, whose tiles each CTA sorts
  // by cost at its start (the cost-sorted deal of fa_order.cuh)
  int cost_sorted;
};

struct BwdParams {
  CUtensorMap tq, tk, tv, tdo; // bf16 [BH, N, d] as above
  CUtensorMap tdq;             // fp32 dQ accumulator: d = 128, 256 transposed [BH, d, Npad],
                               // d = 64 [BH, Npad, d]; box (32, 128, 1), SW128
  const void* o;               // bf16 [B, H, N, d]
  const void* dO;              // bf16 [B, H, N, d]
  const void* v;               // bf16 [B, H, N, d] (d = 256 reads V rows directly)
  const float* lse;            // fp32 [B, H, N]
  void* dq;                    // bf16 [B, H, N, d]
  void* dk;                    // bf16
  void* dv;                    // bf16
  float* delta;                // fp32 [B*H, Npad] workspace: D = rowsum(dO o O), 0 past N
  float* lse2;                 // fp32 [B*H, Npad] workspace: LSE * log2(e), +inf past N
  float* dq_acc;               // fp32 workspace: [BH, Npad, d] (d = 64) or [BH, d, Npad]
  const int* kv_len;
  int B, H, N;
  int H_kv;                    // K/V heads; query head h reads K/V head h / (H / H_kv)
  int wl, wr;                  // key j visible to query i iff i - wl <= j <= i + wr (and j < len)
  int Npad;                    // N rounded up to a multiple of 128
  int causal;                  // causal pairing of key blocks in the schedule (plain causal only)
  float scale;
  float scale_log2;
  int* status;
  // block-sparse: [bm_t, bm_t] bytes, nonzero where (query block, key block)
  // is computed (blocks of 128), or nullptr
  const uint8_t* block_mask;
  int bm_t;
  // a host copy of the block mask, or nullptr; read by the launch (never by a
  // kernel) to balance the schedule
  const uint8_t* block_mask_host;
  // a block mask without a host copy: [bm_t] packed entries of the key
  // blocks sorted by cost (fa_order.cuh), written into the workspace by
  // bwd_order_kernel before the main kernel; nullptr otherwise
  uint32_t* cost_order;
};

// Cost-sorted deal of a block-sparse schedule planned on the device (a block
// mask without a host copy): the tiles (forward) or key blocks (backward) are
// sorted by their computed blocks, longest first, and the items dealt over
// the CTAs in that order.  Entries pack 10-bit fields, so T <= kOrderMaxT;
// the forward keeps its table in shared memory, of kFwdOrderMaxT entries.
constexpr int kOrderMaxT = 1024;
constexpr int kFwdOrderMaxT = 256;

// Causal schedules.  A causal work item (a query tile of the forward, a key
// block of the backward) costs in proportion to its distance from one end of
// the sequence, so items are paired (longest with shortest) into units of
// equal cost and the units go round-robin over the CTAs.  Whole rounds of
// equal units leave the last round part-empty; so the units of the last
// `heads` heads are not paired: their single items, longest first, each go to
// the CTA that has the least work so far (planned on the host).  Row c of
// `item` lists CTA c's items in the order it runs them, after its paired units.
constexpr int kTailCtas = 160;               // grids above this take no tail
constexpr int kTailItems = 8;                // items a CTA may take from the tail
struct TailTable {
  int heads;                                 // 0: no tail, every unit round-robin
  int item[kTailCtas][kTailItems];           // tail_code(head, half, block), -1 ends a row
};
__host__ __device__ constexpr int tail_code(int head, int half, int blk) {
  return (head << 12) | (half << 11) | blk;
}
__host__ __device__ constexpr int tail_head(int code) { return code >> 12; }
__host__ __device__ constexpr int tail_half(int code) { return (code >> 11) & 1; }
__host__ __device__ constexpr int tail_block(int code) { return code & 2047; }

// Plans the tail of a causal schedule over BH heads of T blocks (times
// nsplit halves of the head dimension) on G CTAs.  fwd: query tile m costs
// m + 1 key blocks; backward: key block n costs 2 (T - n) query steps; each
// item also costs a fixed start-up and epilogue.  head_bytes: what the items
// of one head stream and share through L2 (K and V for the forward, the
// group's Q and dO for the backward).  The tail runs all its heads at once,
// so it takes at most kTailL2Bytes of them.  Sets t->heads = 0 (no tail)
// when the table cannot describe it (G > kTailCtas, T > 2048, or a CTA would
// take more than kTailItems items).
constexpr long long kTailL2Bytes = 64ll << 20;
void plan_causal_tail(int BH, int T, int nsplit, int G, bool fwd, long long head_bytes,
                      TailTable* t);

// The same tail for a block-sparse schedule, whose items are not paired: the
// units are single items (bh-major) dealt round-robin, and an item costs its
// computed blocks, which the host counts in its copy of the block mask
// (bm_host, [T, T] row-major) within the window (wl, wr) over N positions.
// fwd: query tile m costs its row's computed key blocks; backward: key block
// n costs 2 query steps per computed query block of its column.  Every head
// shares the mask, so the costs are the same for every head.
void plan_mask_tail(const uint8_t* bm_host, int BH, int T, int nsplit, int G, bool fwd, int N,
                    int wl, int wr, long long head_bytes, TailTable* t);

// Wait site recorded when the dynamic shared memory cannot hold the kernel's
// layout at a 1024-byte aligned base.
constexpr int kSiteSmemLayout = 99;

// Dynamic shared memory to request for a layout of `bytes` that must start on
// a 1024-byte boundary: up to 1 KB of slack, never above the per-block limit.
inline size_t smem_request(size_t bytes, int max_optin) {
  const size_t room = static_cast<size_t>(max_optin) > bytes ? max_optin - bytes : 0;
  return bytes + (room < 1024 ? room : 1024);
}

// fa_bwd's argument and device checks, in its order and with its status
// codes, for a workspace of workspace_bytes at a valid address.
fa_status_t bwd_check_args(const void* q, const void* k, const void* v, const void* o,
                           const void* dO, const float* lse, const void* dq, const void* dk,
                           const void* dv, int B, int H, int N, int d, float scale,
                           int causal, const int* kv_len, size_t workspace_bytes);

cudaError_t launch_fwd(const FwdParams& p, int d, int num_sms, int max_smem, cudaStream_t stream);
cudaError_t launch_bwd_prep(const BwdParams& p, int d, cudaStream_t stream);
// Writes p.cost_order (a block mask without a host copy; T <= kOrderMaxT).
cudaError_t launch_bwd_order(const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_post(const BwdParams& p, int d, cudaStream_t stream);
// 64-query-step backward main kernel with dQ^T (head dimensions 128, 256);
// its Q and dO tensor maps have a box of 64 rows.
cudaError_t launch_wait_selftest(int* status, unsigned long long timeout_ns, cudaStream_t s);
struct Fp8QuantArgs {
  const void* q;               // bf16 [B*H, N, d]
  const void* k;               // bf16 [B*H_kv, N, d]
  const void* v;               // bf16 [B*H_kv, N, d]
  int B, H, H_kv, N;
  void* q8;                    // E4M3 [B*H, N, d]
  float* q_scale;              // [B*H, nb]
  void* k8;                    // E4M3 [B*H_kv, N, d]
  float* k_scale;              // [B*H_kv, nb]
  void* v8t;                   // E4M3 [B*H_kv, d, nb*128]
  float* v_scale;              // [B*H_kv]
};

cudaError_t launch_fp8_quantize(const Fp8QuantArgs& a, int d, cudaStream_t stream);
cudaError_t launch_fwd_fp8(const FwdParams& p, int d, int num_sms, int max_smem,
                           cudaStream_t stream);
cudaError_t launch_decode(const FwdParams& p, int d, int num_sms, int max_smem,
                          cudaStream_t stream);
cudaError_t launch_decode_combine(const FwdParams& p, int d, void* o, float* lse,
                                  cudaStream_t stream);
cudaError_t launch_bwd_main_dt(const BwdParams& p, int d, int num_sms, int max_smem,
                               cudaStream_t stream);
// Backward main kernel for head dimension 64 (fa_bwd_d64.cu): 128-query
// steps, dQ staged and added by bulk tensor reduce-adds through tdq, a map of
// the [BH, Npad, 64] accumulator with a box of 32 columns x 128 rows.
cudaError_t launch_bwd_main_d64(const BwdParams& p, int num_sms, int max_smem,
                                cudaStream_t stream);

}  // namespace fa
