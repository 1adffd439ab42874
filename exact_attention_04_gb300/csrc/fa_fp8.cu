// E4M3 quantisation of Q, K and V for the FP8 forward.
//
// "4. FlashAttention 深度剖析" 4.5.4: FP8 (E4M3) operands for the forward
// pass, a scale per block applied when the block is loaded, FP32
// accumulation.  The scales here: Q per 128-row tile of a head, K per
// 128-key block of a K/V head, V per K/V head (so the P V sum is scaled once
// at the end).  For a block with largest magnitude amax the stored value is
// E4M3(x * (448 / amax)), rounded to nearest even and saturated, and the
// dequantisation scale is amax / 448 (both quotients and the product rounded
// to fp32); an all-zero block has scale 1.  V is written transposed per head,
// [d, keys] with the keys padded to a multiple of 128, so that a V block is
// the K-major B operand of the P V product.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kRowsPerBlock = 128;
constexpr int kThreads = 256;

__device__ __forceinline__ float block_max(float m) {
  __shared__ float red[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < kThreads / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  }
  return m;   // valid in thread 0
}

__device__ __forceinline__ void unpack8(uint4 u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// Largest |x| of each 128-row block of G heads ([G, N, D] bf16), folded into
// out[g] with an integer max on the bit patterns, which orders non-negative
// floats correctly (V: one scale per head).
template <int D>
__global__ void __launch_bounds__(kThreads) head_amax_kernel(const __nv_bfloat16* x, int N, int nb,
                                                             float* out) {
  const int blk = blockIdx.x;
  const int g = blk / nb, b = blk % nb;
  const int r0 = b * kRowsPerBlock;
  const int r1 = r0 + kRowsPerBlock < N ? r0 + kRowsPerBlock : N;
  const uint4* src = reinterpret_cast<const uint4*>(x + (static_cast<size_t>(g) * N + r0) * D);
  const int n8 = (r1 - r0) * (D / 8);
  float m = 0.f;
  for (int i = threadIdx.x; i < n8; i += kThreads) {
    float f[8];
    unpack8(src[i], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(f[e]));
  }
  m = block_max(m);
  if (threadIdx.x == 0) atomicMax(reinterpret_cast<int*>(out + g), __float_as_int(m));
}

__device__ __forceinline__ void scale_of(float amax, float& s, float& mul) {
  s = 1.f;
  mul = 1.f;
  if (amax > 0.f) {
    s = __fdiv_rn(amax, 448.f);
    mul = __fdiv_rn(448.f, amax);
  }
}

// One 128-row block of G heads ([G, N, D] bf16) to E4M3 in one pass: the
// block stays in registers while the CTA reduces its largest |x|, then is
// scaled and converted; scales[g * nb + b] gets the dequantisation scale.
template <int D>
__global__ void __launch_bounds__(kThreads) quant_rows_kernel(const __nv_bfloat16* x, int N,
                                                              int nb, float* scales,
                                                              uint8_t* codes) {
  constexpr int PER = kRowsPerBlock * (D / 8) / kThreads;   // 16-byte loads per thread
  __shared__ float s_amax;
  const int blk = blockIdx.x;
  const int g = blk / nb, b = blk % nb;
  const int r0 = b * kRowsPerBlock;
  const int r1 = r0 + kRowsPerBlock < N ? r0 + kRowsPerBlock : N;
  const size_t off = (static_cast<size_t>(g) * N + r0) * D;
  const uint4* src = reinterpret_cast<const uint4*>(x + off);
  uint2* dst = reinterpret_cast<uint2*>(codes + off);
  const int n8 = (r1 - r0) * (D / 8);
  uint4 v[PER];
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = threadIdx.x + k * kThreads;
    v[k] = i < n8 ? src[i] : make_uint4(0, 0, 0, 0);
    float f[8];
    unpack8(v[k], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(f[e]));
  }
  m = block_max(m);
  if (threadIdx.x == 0) s_amax = m;
  __syncthreads();
  float s, mul;
  scale_of(s_amax, s, mul);
  if (threadIdx.x == 0) scales[blk] = s;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = threadIdx.x + k * kThreads;
    if (i < n8) {
      float f[8];
      unpack8(v[k], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = __fmul_rn(f[e], mul);
      dst[i] = make_uint2(ptx::pack_e4m3x4(f[0], f[1], f[2], f[3]),
                          ptx::pack_e4m3x4(f[4], f[5], f[6], f[7]));
    }
  }
}

// One 128-key block of V to E4M3, transposed: vt[(g*D + c) * npad + key].
// The codes go to shared memory in V's own layout ([key][D] bytes, rows
// padded by one word so that rows 16 apart fall in different banks).  The
// transposed pass gathers 16 keys of a column into one 16-byte store; a warp
// takes 16 adjacent columns and two adjacent 16-key groups, so each column's
// two stores fill one 32-byte sector and the shared-memory reads (16 columns
// = 4 words, two rows 16 apart) hit 8 distinct banks.
template <int D>
__global__ void __launch_bounds__(kThreads) quant_vt_kernel(const __nv_bfloat16* v, int N,
                                                            int npad, int nb,
                                                            const float* head_amax,
                                                            uint8_t* vt) {
  constexpr int kRow = D + 4;                       // padded row, bytes
  __shared__ __align__(16) uint8_t tile[kRowsPerBlock * kRow];
  const int blk = blockIdx.x;
  const int g = blk / nb, b = blk % nb;
  float s, mul;
  scale_of(head_amax[g], s, mul);
  for (int it = threadIdx.x; it < kRowsPerBlock * (D / 8); it += kThreads) {
    const int k = it / (D / 8), c8 = it % (D / 8);
    const int key = b * kRowsPerBlock + k;
    float f[8];
    if (key < N) {
      unpack8(*reinterpret_cast<const uint4*>(v + (static_cast<size_t>(g) * N + key) * D + c8 * 8), f);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = __fmul_rn(f[e], mul);
    uint32_t* row = reinterpret_cast<uint32_t*>(&tile[k * kRow + c8 * 8]);
    row[0] = ptx::pack_e4m3x4(f[0], f[1], f[2], f[3]);
    row[1] = ptx::pack_e4m3x4(f[4], f[5], f[6], f[7]);
  }
  __syncthreads();
  for (int it = threadIdx.x; it < D * (kRowsPerBlock / 16); it += kThreads) {
    const int rest = it / 32;
    const int c = (rest % (D / 16)) * 16 + it % 16;
    const int k16 = (rest / (D / 16)) * 2 + (it / 16) % 2;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t x = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        x |= static_cast<uint32_t>(tile[(16 * k16 + 4 * q + e) * kRow + c]) << (8 * e);
      w[q] = x;
    }
    *reinterpret_cast<uint4*>(vt + (static_cast<size_t>(g) * D + c) * npad + b * kRowsPerBlock +
                              16 * k16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// amax -> dequantisation scale, one value per head.
__global__ void head_scale_kernel(float* io, int G) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= G) return;
  float s, mul;
  scale_of(io[g], s, mul);
  io[g] = s;
}

template <int D>
cudaError_t quantize(const Fp8QuantArgs& a, cudaStream_t st) {
  const int nb = (a.N + kRowsPerBlock - 1) / kRowsPerBlock;
  const int npad = nb * kRowsPerBlock;
  const int gq = a.B * a.H, gk = a.B * a.H_kv;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v);
  cudaError_t e = cudaMemsetAsync(a.v_scale, 0, sizeof(float) * gk, st);
  if (e != cudaSuccess) return e;
  head_amax_kernel<D><<<gk * nb, kThreads, 0, st>>>(v, a.N, nb, a.v_scale);
  quant_rows_kernel<D><<<gq * nb, kThreads, 0, st>>>(q, a.N, nb, a.q_scale,
                                                     static_cast<uint8_t*>(a.q8));
  quant_rows_kernel<D><<<gk * nb, kThreads, 0, st>>>(k, a.N, nb, a.k_scale,
                                                     static_cast<uint8_t*>(a.k8));
  quant_vt_kernel<D><<<gk * nb, kThreads, 0, st>>>(v, a.N, npad, nb, a.v_scale,
                                                   static_cast<uint8_t*>(a.v8t));
  head_scale_kernel<<<(gk + 127) / 128, 128, 0, st>>>(a.v_scale, gk);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8_quantize(const Fp8QuantArgs& a, int d, cudaStream_t stream) {
  switch (d) {
    case 128: return quantize<128>(a, stream);
    case 256: return quantize<256>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
