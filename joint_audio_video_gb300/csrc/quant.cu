// Row-wise E4M3 quantisation (HBM-bound), the operand preparation of the fp8
// projections ("Joint Audio-Video Generation in Production", §5: the active
// block held at FP8; prior art for the fp8 variant of the sub-block).
//
//   s[r] = max_k |x[r][k]| / 448 (448 = largest finite E4M3; 1 for a zero row)
//   q[r][k] = E4M3 round-to-nearest, saturating, of x[r][k] / s[r]
//
// One 256-thread CTA per row: pass 1 reduces the row's absolute maximum,
// pass 2 re-reads the row (from L2) and writes 8 fp8 bytes per 16-byte input
// vector.  Weights use the same kernel on their output-channel rows.
#include <cuda_bf16.h>

#include "kernels.hpp"
#include "ptx.cuh"

namespace h3 {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t q;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q) : "f"(hi), "f"(lo));
  return q;
}

__global__ void __launch_bounds__(kThreads)
    quantize_rows_kernel(const uint4* __restrict__ x, int R, int K, uint2* __restrict__ q,
                         float* __restrict__ scale, int* status) {
  __shared__ float red[kThreads / 32];
  const size_t row = blockIdx.x;
  if (!H3_IN(row < size_t(R), status)) return;   // uniform across the CTA
  const int nvec = K >> 3;
  const uint4* xr = x + row * nvec;
  float am = 0.f;
  for (int c = threadIdx.x; c < nvec; c += kThreads) {
    const uint4 v = xr[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      am = fmaxf(am, fmaxf(fabsf(__uint_as_float(w[i] << 16)),
                           fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  if (lane_id() == 0) red[warp_id()] = am;
  __syncthreads();
  am = red[lane_id() & (kThreads / 32 - 1)];
#pragma unroll
  for (int o = kThreads / 64; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  const float s = am > 0.f ? am / 448.f : 1.f;
  const float inv = am > 0.f ? 448.f / am : 1.f;
  uint2* qr = q + row * nvec;
  for (int c = threadIdx.x; c < nvec; c += kThreads) {
    const uint4 v = xr[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint16_t b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      b[i] = e4m3x2(__uint_as_float(w[i] << 16) * inv, __uint_as_float(w[i] & 0xFFFF0000u) * inv);
    qr[c] = make_uint2(uint32_t(b[0]) | (uint32_t(b[1]) << 16), uint32_t(b[2]) | (uint32_t(b[3]) << 16));
  }
  if (threadIdx.x == 0) scale[row] = s;
}

// Q and K of the packed qkv [L][3d] for the E4M3 score product (the
// "SageAttention"-style quantised attention that "Joint Audio-Video Generation
// in Production", §6 names as prior art, restated): one CTA per (128-token
// block b, head h), 256 threads, 16 threads per token row (8 bf16 each).
//   sq[h][i] = max_c |Q[i][h][c]| / 448,   Q8[i][h][c] = E4M3(Q / sq)
//   sk[h][b] = max over the block's 128 tokens and 128 dims of |K| / 448,
//   K8[i][h][c] = E4M3(K / sk)                      (scale 1 for all-zero data)
// Per-token Q scales fold into the softmax's per-row constant and per-block K
// scales into its per-block constant, so the score product needs no rescaling.
constexpr int kQkRows = 128;

__device__ __forceinline__ float amax8(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
  return m;
}
__device__ __forceinline__ uint2 e4m3x8(const uint4& v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint16_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    b[i] = e4m3x2(__uint_as_float(w[i] << 16) * inv, __uint_as_float(w[i] & 0xFFFF0000u) * inv);
  return make_uint2(uint32_t(b[0]) | (uint32_t(b[1]) << 16), uint32_t(b[2]) | (uint32_t(b[3]) << 16));
}

__global__ void __launch_bounds__(kThreads)
    quantize_qk_kernel(const uint4* __restrict__ qkv, int L, int H, int nkb,
                       uint2* __restrict__ qk8, float* __restrict__ sq, float* __restrict__ sk,
                       int* status) {
  __shared__ float red[kThreads / 32];
  const int b = blockIdx.x % nkb, h = blockIdx.x / nkb;
  if (!H3_IN(h < H, status)) return;   // uniform across the CTA
  const int c = threadIdx.x & 15;                  // 8-element chunk of the head's 128 dims
  const size_t d = size_t(H) * 128;
  const size_t in_row = 3 * d / 8, out_row = 2 * d / 8;   // row pitches in uint4 / uint2
  uint4 qv[8], kv[8];
  float km = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = b * kQkRows + (threadIdx.x >> 4) + 16 * i;
    qv[i] = kv[i] = make_uint4(0u, 0u, 0u, 0u);
    if (r < L) {
      qv[i] = qkv[size_t(r) * in_row + h * 16 + c];
      kv[i] = qkv[size_t(r) * in_row + d / 8 + h * 16 + c];
    }
    km = fmaxf(km, amax8(kv[i]));
  }
  // K: one scale for the whole block
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
  if (lane_id() == 0) red[warp_id()] = km;
  __syncthreads();
  km = red[lane_id() & (kThreads / 32 - 1)];
#pragma unroll
  for (int o = kThreads / 64; o > 0; o >>= 1) km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
  const float k_inv = km > 0.f ? 448.f / km : 1.f;
  if (threadIdx.x == 0) sk[size_t(h) * nkb + b] = km > 0.f ? km / 448.f : 1.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = b * kQkRows + (threadIdx.x >> 4) + 16 * i;
    // Q: one scale per token, reduced over the 16 threads of the row
    float qm = amax8(qv[i]);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, o));
    if (r < L) {
      const float q_inv = qm > 0.f ? 448.f / qm : 1.f;
      qk8[size_t(r) * out_row + h * 16 + c] = e4m3x8(qv[i], q_inv);
      qk8[size_t(r) * out_row + d / 8 + h * 16 + c] = e4m3x8(kv[i], k_inv);
      if (c == 0) sq[size_t(h) * L + r] = qm > 0.f ? qm / 448.f : 1.f;
    }
  }
}

}  // namespace

cudaError_t launch_quantize_qk(const void* qkv, int L, int H, void* qk8, float* sq, float* sk,
                               const DevCtx& ctx, cudaStream_t st) {
  const int nkb = (L + kQkRows - 1) / kQkRows;
  quantize_qk_kernel<<<unsigned(nkb) * unsigned(H), kThreads, 0, st>>>(
      static_cast<const uint4*>(qkv), L, H, nkb, static_cast<uint2*>(qk8), sq, sk, ctx.status);
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const void* x, int R, int K, void* q, float* scale,
                                 const DevCtx& ctx, cudaStream_t st) {
  quantize_rows_kernel<<<R, kThreads, 0, st>>>(static_cast<const uint4*>(x), R, K,
                                               static_cast<uint2*>(q), scale, ctx.status);
  return cudaGetLastError();
}

}  // namespace h3
