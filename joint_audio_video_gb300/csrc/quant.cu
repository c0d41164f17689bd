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
    quantize_rows_kernel(const uint4* __restrict__ x, int K, uint2* __restrict__ q,
                         float* __restrict__ scale) {
  __shared__ float red[kThreads / 32];
  const size_t row = blockIdx.x;
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

}  // namespace

cudaError_t launch_quantize_rows(const void* x, int R, int K, void* q, float* scale,
                                 const DevCtx& ctx, cudaStream_t st) {
  (void)ctx;
  quantize_rows_kernel<<<R, kThreads, 0, st>>>(static_cast<const uint4*>(x), K,
                                               static_cast<uint2*>(q), scale);
  return cudaGetLastError();
}

}  // namespace h3
