// Modality-indexed AdaLN LayerNorm + modulate (HBM-bound).
//
//   y[n] = (x[n] - mean) * rsqrt(biased var + eps) * (1 + scale[m]) + shift[m],
//   m = mod[n]   ("DiffusionNFT on MiniMax H3", section "MiniMax H3 and Why
//   Joint Audio-Video Generation Complicates RL Training": modality-specific
//   AdaLN branches whose outputs are cached per modality).
//
// One 128-thread CTA per token row.  The row (d bf16 = d/8 16-byte vectors)
// is loaded once with streaming 16-byte loads and kept in registers (5 vectors
// per thread at d = 5120; at most 64 registers, so 8 rows, 80 KB, are in flight
// per SM where 256-thread rows managed ~5: the bytes in flight set the HBM
// rate this kernel reaches); mean and
// variance are two exact passes over the registers (fp32 warp shuffles + a
// shared-memory hop across the 8 warps).  The per-modality fp32 vectors are
// tiny (n_mod x d) and served from L1/L2.  Algorithmic traffic: 4*d bytes per
// row (read x, write y).
#include <cuda_bf16.h>

#include "kernels.hpp"
#include "ptx.cuh"

namespace h3 {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane_id() == 0) red[warp_id()] = v;
  __syncthreads();
  // every lane reads the 8 warp partials cyclically, so the xor tree below
  // leaves the full total in all 32 lanes
  float t = red[lane_id() & (kThreads / 32 - 1)];
#pragma unroll
  for (int o = kThreads / 64; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  __syncthreads();
  return t;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <int VPT>
__global__ void __launch_bounds__(kThreads, VPT <= 5 ? 8 : 2)
    adaln_modulate_kernel(const uint4* __restrict__ x, const uint8_t* __restrict__ mod,
                          const float* __restrict__ shift, const float* __restrict__ scale, int d,
                          int n_mod, float eps, uint4* __restrict__ y, int* status) {
  __shared__ float red[kThreads / 32];
  const size_t row = blockIdx.x;
  const int nvec = d >> 3;
  const uint4* xr = x + row * nvec;
  uint4 v[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = threadIdx.x + i * kThreads;
    v[i] = c < nvec ? __ldcs(xr + c) : make_uint4(0, 0, 0, 0);
  }
  const int m = mod[row];

  float s = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    float f[8];
    unpack8(v[i], f);
#pragma unroll
    for (int k = 0; k < 8; ++k) s += f[k];
  }
  const float inv_d = 1.f / float(d);
  const float mean = block_sum(s, red) * inv_d;

  float q = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    if (threadIdx.x + i * kThreads < nvec) {
      float f[8];
      unpack8(v[i], f);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float c = f[k] - mean;
        q = fmaf(c, c, q);
      }
    }
  }
  const float rstd = rsqrtf(block_sum(q, red) * inv_d + eps);

  uint4* yr = y + row * nvec;
  if (m >= n_mod) {  // uniform across the CTA
    if (threadIdx.x == 0) atomicCAS(status, H3_DEV_OK, H3_DEV_BAD_INDEX);
    const uint4 nan4 = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = threadIdx.x + i * kThreads;
      if (c < nvec) yr[c] = nan4;
    }
    return;
  }
  const float4* sc = reinterpret_cast<const float4*>(scale + size_t(m) * d);
  const float4* sh = reinterpret_cast<const float4*>(shift + size_t(m) * d);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = threadIdx.x + i * kThreads;
    if (c < nvec) {
      float f[8];
      unpack8(v[i], f);
      const float4 a0 = __ldg(sc + 2 * c), a1 = __ldg(sc + 2 * c + 1);
      const float4 b0 = __ldg(sh + 2 * c), b1 = __ldg(sh + 2 * c + 1);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float y0 = fmaf((f[2 * k] - mean) * rstd, 1.f + a[2 * k], b[2 * k]);
        const float y1 = fmaf((f[2 * k + 1] - mean) * rstd, 1.f + a[2 * k + 1], b[2 * k + 1]);
        o[k] = pack_bf16x2(y0, y1);
      }
      yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

template <int VPT>
cudaError_t launch_vpt(const void* x, const uint8_t* mod, const float* shift, const float* scale,
                       int L, int d, int n_mod, float eps, void* y, const DevCtx& ctx,
                       cudaStream_t st) {
  adaln_modulate_kernel<VPT><<<L, kThreads, 0, st>>>(
      static_cast<const uint4*>(x), mod, shift, scale, d, n_mod, eps, static_cast<uint4*>(y),
      ctx.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_adaln_modulate(const void* x, const uint8_t* mod, const float* shift,
                                  const float* scale, int L, int d, int n_mod, float eps, void* y,
                                  const DevCtx& ctx, cudaStream_t st) {
  const int vpt = (d / 8 + kThreads - 1) / kThreads;
  switch (vpt) {   // d <= 16384: at most 16 vectors per thread
    case 1: return launch_vpt<1>(x, mod, shift, scale, L, d, n_mod, eps, y, ctx, st);
    case 2: return launch_vpt<2>(x, mod, shift, scale, L, d, n_mod, eps, y, ctx, st);
    case 3: return launch_vpt<3>(x, mod, shift, scale, L, d, n_mod, eps, y, ctx, st);
    case 4: return launch_vpt<4>(x, mod, shift, scale, L, d, n_mod, eps, y, ctx, st);
    case 5: return launch_vpt<5>(x, mod, shift, scale, L, d, n_mod, eps, y, ctx, st);
    case 6: return launch_vpt<6>(x, mod, shift, scale, L, d, n_mod, eps, y, ctx, st);
    case 7: case 8: return launch_vpt<8>(x, mod, shift, scale, L, d, n_mod, eps, y, ctx, st);
    case 9: case 10: case 11: case 12:
      return launch_vpt<12>(x, mod, shift, scale, L, d, n_mod, eps, y, ctx, st);
    case 13: case 14: case 15: case 16:
      return launch_vpt<16>(x, mod, shift, scale, L, d, n_mod, eps, y, ctx, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace h3
