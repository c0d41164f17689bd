// One denoising-step update of the packed latent (HBM-bound).
//
// "Joint Audio-Video Generation in Production", §4 Denoising Execution Flow:
// stage 5 turns the predicted velocity into a clean estimate X0 (rectified
// flow), stage 6 advances every modality with a deterministic (eta = 0) Euler
// step on its own noise schedule (sigma_video, sigma_audio), stage 7 writes
// the state back and re-pins the anchor rows.  "多模态强化学习工程解析…", 5.1:
// H3 runs in data-progress time t = 1 - sigma and its velocity is the
// negative of the standard flow-matching one.
//
// With v = -v_h3 (standard sign) and the token's modality m:
//   x0 = z - sigma[m] v,   z' = z + (sigma_next[m] - sigma[m]) v.
// One thread per 4 channels: 16-byte loads/stores of the fp32 state, 8-byte
// loads of the bf16 velocity.  Algorithmic traffic per element: read z (4 B)
// and v (2 B), write z (4 B) and x0 (4 B).
#include <cuda_bf16.h>

#include "kernels.hpp"
#include "ptx.cuh"

namespace h3 {
namespace {

__global__ void __launch_bounds__(256)
    denoise_kernel(float4* __restrict__ z, float4* __restrict__ x0, const uint2* __restrict__ v,
                   const uint8_t* __restrict__ mod, const uint8_t* __restrict__ anchor,
                   const float4* __restrict__ z_anchor, size_t n_vec, int vec_per_row, int n_mod,
                   const __grid_constant__ DenoiseParams dp, int* status) {
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n_vec;
       i += size_t(gridDim.x) * blockDim.x) {
    const size_t r = i / size_t(vec_per_row);
    if (!H3_IN((r + 1) * size_t(vec_per_row) <= n_vec, status)) continue;   // row r of L
    const int m = mod[r];
    if (m >= n_mod) {                       // leave the row as it is and report
      atomicCAS(status, H3_DEV_OK, H3_DEV_BAD_INDEX);
      continue;
    }
    if (anchor != nullptr && anchor[r]) {   // stage 7: re-pin
      const float4 a = z_anchor[i];
      z[i] = a;
      if (x0) x0[i] = a;
      continue;
    }
    const float4 zv = z[i];
    if (!dp.update[m]) {                    // a condition row (text): not a latent
      if (x0) x0[i] = zv;
      continue;
    }
    const uint2 w = __ldcs(v + i);
    // standard-sign velocity: the negated bf16 values
    const float v0 = -__uint_as_float(w.x << 16), v1 = -__uint_as_float(w.x & 0xFFFF0000u);
    const float v2 = -__uint_as_float(w.y << 16), v3 = -__uint_as_float(w.y & 0xFFFF0000u);
    const float s = dp.sigma[m], ds = dp.sigma_next[m] - dp.sigma[m];
    if (x0) x0[i] = make_float4(fmaf(-s, v0, zv.x), fmaf(-s, v1, zv.y), fmaf(-s, v2, zv.z),
                                fmaf(-s, v3, zv.w));
    z[i] = make_float4(fmaf(ds, v0, zv.x), fmaf(ds, v1, zv.y), fmaf(ds, v2, zv.z),
                       fmaf(ds, v3, zv.w));
  }
}

}  // namespace

cudaError_t launch_denoise(float* z, float* x0, const void* v_h3, const uint8_t* mod,
                           const uint8_t* anchor, const float* z_anchor, int L, int C, int n_mod,
                           const DenoiseParams& dp, const DevCtx& ctx, cudaStream_t st) {
  const size_t n_vec = size_t(L) * (C / 4);
  const size_t want = (n_vec + 255) / 256;
  const int grid = int(want < size_t(ctx.num_sms) * 16 ? want : size_t(ctx.num_sms) * 16);
  denoise_kernel<<<grid, 256, 0, st>>>(
      reinterpret_cast<float4*>(z), reinterpret_cast<float4*>(x0),
      static_cast<const uint2*>(v_h3), mod, anchor, reinterpret_cast<const float4*>(z_anchor),
      n_vec, C / 4, n_mod, dp, ctx.status);
  return cudaGetLastError();
}

}  // namespace h3
