// Attention backward for sm_103a: three launches on one stream (four with a
// block mask that has no host copy).  This file holds all but the main
// kernel, which lives in fa_bwd_d64.cu (head dimension 64) and fa_bwd_dt.cu
// (128 and 256).
//
//  1. bwd_pre   D_i = sum_t dO_it * O_it and L2_i = LSE_i * log2(e) per query
//               row (padded to a multiple of 128 rows: D = 0, L2 = +inf past
//               N), and zero the fp32 dQ accumulator.  Memory bound.
//  2. bwd_main  recomputes P from Q, K and L2 per 128-key block, writes dK and
//               dV, and adds dS K into the fp32 dQ accumulator.
//     bwd_order (a block mask without a host copy, before bwd_main) sorts
//               the key blocks by cost for bwd_main's schedule.
//  3. bwd_post  dQ = bf16(scale * dQ_acc) (d = 64: [BH, Npad, d] accumulator;
//               d = 128, 256: transposed [BH, d, Npad]).
//
// The recomputation of P from the saved statistic follows "注意力为什么受限于
// 显存带宽：用算术强度与分块把 FlashAttention 推导清楚" (section 八) and "4.
// FlashAttention 深度剖析" (section 4.3.4, P_ij = exp(S_ij - L_i)).  The pages
// print no gradient formulas; the ones used are the chain rule through the
// row softmax and O = P V.
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

// The key blocks' cost-sorted order (fa_order.cuh) for a block mask without
// a host copy: key block n costs the computed query blocks of its mask
// column among the queries its keys are visible to (the window; kv_len,
// which differs by batch entry, is left out).  One CTA, a key block a
// thread; the mask's column reads are coalesced across the threads.
__global__ void __launch_bounds__(kOrderMaxT) bwd_order_kernel(const __grid_constant__ BwdParams p) {
  __shared__ uint32_t cost[kOrderMaxT];
  const int T = p.bm_t;
  const int n = threadIdx.x;
  if (n < T) {
    int q_lo, q_hi;
    visible_queries(n * 128, 128, p.N, p.N, p.wl, p.wr, q_lo, q_hi);
    uint32_t c = 0;
    if (q_hi > q_lo)
      for (int a = q_lo / 128; a < (q_hi + 127) / 128; ++a)
        c += __ldg(p.block_mask + static_cast<size_t>(a) * p.bm_t + n) != 0;
    cost[n] = c;
  }
  __syncthreads();
  if (n < T) {
    uint32_t e;
    const int pos = order_rank(cost, T, n, e);
    p.cost_order[pos] = e;
  }
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

cudaError_t launch_bwd_order(const BwdParams& p, cudaStream_t stream) {
  if (!p.cost_order || !p.block_mask || p.bm_t < 1 || p.bm_t > kOrderMaxT)
    return cudaErrorInvalidValue;
  const int threads = (p.bm_t + 31) / 32 * 32;
  bwd_order_kernel<<<1, threads, 0, stream>>>(p);
  return cudaGetLastError();
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
