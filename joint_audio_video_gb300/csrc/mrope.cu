// 3D multimodal rotary embedding over (t, h, w), in place on Q and K (HBM-bound).
//
// "DiffusionNFT on MiniMax H3", section "MiniMax H3 and Why Joint Audio-Video
// Generation Complicates RL Training" (rotary position embeddings across time,
// height and width); "Joint Audio-Video Generation in Production", §3 Packed
// Sequences (each token carries its position indices and modality tag into
// the RoPE step).
//
// Pair k of every head covers dims (2k, 2k+1) and turns by
// pos[n][axis(k)] * inv_freq(k).  The 64 angles of a token are shared by all
// H heads of Q and K, so each CTA first tabulates cos/sin for its tokens in
// shared memory (fp32 sincosf of an fp32 angle), then streams the Q|K part of
// each row (2d bf16, contiguous) with 16-byte read-modify-write accesses.
// Algorithmic traffic: 8*d bytes per token (read + write Q and K) + 12 bytes
// of positions.
#include <cuda_bf16.h>

#include <cmath>

#include "kernels.hpp"
#include "ptx.cuh"

namespace h3 {

void make_rope_table(RopeTable* rt, const int32_t sec[3], double base) {
  int k = 0;
  for (int a = 0; a < 3; ++a) {
    const int n_a = sec[a];
    for (int j = 0; j < n_a / 2; ++j, ++k) {
      rt->inv_freq[k] = static_cast<float>(std::pow(base, -2.0 * j / n_a));
      rt->axis[k] = a;
    }
  }
}

namespace {

constexpr int kThreads = 256;
constexpr int kTokens = 4;

__global__ void __launch_bounds__(kThreads)
    mrope_kernel(uint4* __restrict__ qkv, const int32_t* __restrict__ pos, int L, int d,
                 const __grid_constant__ RopeTable rt, int* status) {
  __shared__ float2 cs[kTokens][64];
  const int tok0 = blockIdx.x * kTokens;
  for (int i = threadIdx.x; i < kTokens * 64; i += kThreads) {
    const int t = i >> 6, k = i & 63;
    const int n = tok0 + t;
    float s = 0.f, c = 1.f;
    if (n < L && H3_IN(rt.axis[k] >= 0 && rt.axis[k] < 3, status)) {
      const float ang = float(pos[size_t(n) * 3 + rt.axis[k]]) * rt.inv_freq[k];
      sincosf(ang, &s, &c);
    }
    cs[t][k] = make_float2(c, s);
  }
  __syncthreads();
  const int vec_qk = d >> 2;          // 16-byte vectors in the Q|K part of a row
  const size_t row_vec = size_t(3 * d) >> 3;
  for (int i = threadIdx.x; i < kTokens * vec_qk; i += kThreads) {
    const int t = i / vec_qk, v = i - t * vec_qk;
    const int n = tok0 + t;
    if (n >= L) break;
    // the Q|K part of row n (its first 2d of 3d columns), pairs k0 .. k0 + 3 of the table
    if (!H3_IN(v < vec_qk && ((v * 8) & 127) / 2 + 3 < 64, status)) continue;
    uint4* p = qkv + size_t(n) * row_vec + v;
    uint4 w = *p;
    const int k0 = ((v * 8) & 127) >> 1;   // first pair of this vector inside its head
    uint32_t* u = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = __uint_as_float(u[j] << 16);
      const float b = __uint_as_float(u[j] & 0xFFFF0000u);
      const float2 r = cs[t][k0 + j];
      u[j] = pack_bf16x2(a * r.x - b * r.y, a * r.y + b * r.x);
    }
    *p = w;
  }
}

}  // namespace

cudaError_t launch_mrope(void* qkv, const int32_t* pos, int L, int n_heads, const RopeTable& rt,
                         const DevCtx& ctx, cudaStream_t st) {
  const int grid = (L + kTokens - 1) / kTokens;
  mrope_kernel<<<grid, kThreads, 0, st>>>(static_cast<uint4*>(qkv), pos, L, n_heads * 128, rt,
                                          ctx.status);
  return cudaGetLastError();
}

}  // namespace h3
