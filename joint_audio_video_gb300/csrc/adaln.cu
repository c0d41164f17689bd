// Modality-indexed AdaLN LayerNorm + modulate (HBM-bound).
//
//   y[n] = (x[n] - mean) * rsqrt(biased var + eps) * (1 + scale[m]) + shift[m],
//   m = mod[n]   ("DiffusionNFT on MiniMax H3", section "MiniMax H3 and Why
//   Joint Audio-Video Generation Complicates RL Training": modality-specific
//   AdaLN branches whose outputs are cached per modality).
//
// Persistent CTAs of 128 threads, a few per SM; CTA b handles rows b, b + G,
// b + 2G, ... (G = grid size).  One thread keeps the next kStages rows of the
// CTA in flight as 1-D bulk copies (TMA) into a ring of shared-memory row
// buffers, so HBM reads continue while the warps reduce and write the current
// row: the bytes in flight per SM, not the per-row reduction latency, set the
// rate.  A row (d bf16) is read once from shared memory into registers (5
// 16-byte vectors per thread at d = 5120); mean and variance are two exact
// passes over the registers (fp32 warp shuffles + a shared-memory hop across
// the 4 warps).  For d <= 6144, (1 + scale[m]) and shift[m] of the thread's
// columns stay in registers and are reloaded (from L2: n_mod x d floats in
// all) only when the modality changes from one row to the next; wider rows
// read them per row through L1.  Algorithmic traffic: 4*d bytes
// per row (read x, write y).
#include <cuda_bf16.h>

#include "kernels.hpp"
#include "ptx.cuh"

namespace h3 {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxStages = 4;

// Sum over the CTA.  `red` alternates between two 4-float buffers on
// successive calls, so one barrier suffices: a buffer is rewritten only two
// calls later, after the intervening call's barrier, when every lane has read it.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane_id() == 0) red[warp_id()] = v;
  __syncthreads();
  // every lane reads the 4 warp partials cyclically, so the xor tree below
  // leaves the full total in all 32 lanes
  float t = red[lane_id() & (kThreads / 32 - 1)];
#pragma unroll
  for (int o = kThreads / 64; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
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
__global__ void __launch_bounds__(kThreads)
    adaln_modulate_kernel(const uint4* __restrict__ x, const uint8_t* __restrict__ mod,
                          const float* __restrict__ shift, const float* __restrict__ scale, int L,
                          int d, int n_mod, float eps, int stages, uint4* __restrict__ y,
                          int* status, uint64_t wait_ns) {
  extern __shared__ __align__(128) uint8_t ring[];   // stages x (2d bytes)
  __shared__ uint64_t full[kMaxStages];
  __shared__ float red[2][kThreads / 32];
  __shared__ int abort_flag;
  const int nvec = d >> 3;
  const uint32_t row_bytes = uint32_t(d) * 2u;
  const int G = gridDim.x;
  // rows of this CTA: blockIdx.x + k G, k < nk
  const int nk = blockIdx.x < L ? (L - 1 - int(blockIdx.x)) / G + 1 : 0;
  const WaitCtx wc{&abort_flag, status, wait_ns};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < stages; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int k) {   // row k of this CTA into ring slot k % stages
    const int s = k % stages;
    const uint32_t bar = smem_u32(&full[s]);
    const size_t row = blockIdx.x + size_t(k) * G;
    if (H3_IN(row < size_t(L), status)) {
      mbar_arrive_expect_tx(bar, row_bytes);
      bulk_load_1d(smem_u32(ring + size_t(s) * row_bytes), x + row * nvec, row_bytes, bar);
    } else {
      mbar_arrive(bar);   // checked build: the row is skipped, the slot completes
    }
  };
  int issued = 0;
  if (threadIdx.x == 0)
    for (; issued < stages && issued < nk; ++issued) issue(issued);

  const float inv_d = 1.f / float(d);
  // (1 + scale[m]) and shift[m] of this thread's columns, reloaded only when the
  // modality changes (the strided rows of a CTA cross a segment boundary at most
  // a few times); kept in registers so the streaming rows do not compete with
  // them for L1, which the row ring's shared memory shrinks
  constexpr bool kRegs = VPT <= 6;
  float ga[kRegs ? VPT : 1][8], gb[kRegs ? VPT : 1][8];
  int m_cur = -1;
  int k = 0;
  for (; k < nk; ++k) {
    const int s = k % stages;
    const bool ok = mbar_wait(smem_u32(&full[s]), uint32_t(k / stages) & 1u, wc);
    if (__syncthreads_or(!ok)) break;
    const size_t row = blockIdx.x + size_t(k) * G;
    const uint4* xr = reinterpret_cast<const uint4*>(ring + size_t(s) * row_bytes);
    uint4 v[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = threadIdx.x + i * kThreads;
      v[i] = c < nvec ? xr[c] : make_uint4(0, 0, 0, 0);
    }
    const bool row_ok = H3_IN(row < size_t(L), status);
    const int m = row_ok ? int(mod[row]) : 0;

    // eight independent partial sums per pass: short dependency chains
    float part[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      float f[8];
      unpack8(v[i], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) part[j] += f[j];
    }
    const float sum = ((part[0] + part[1]) + (part[2] + part[3])) +
                      ((part[4] + part[5]) + (part[6] + part[7]));
    // block_sum's barrier also orders every thread's reads of slot s before
    // its refill below
    const float mean = block_sum(sum, red[0]) * inv_d;
    if (threadIdx.x == 0 && issued < nk) issue(issued++);

#pragma unroll
    for (int j = 0; j < 8; ++j) part[j] = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      if (threadIdx.x + i * kThreads < nvec) {
        float f[8];
        unpack8(v[i], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float c = f[j] - mean;
          part[j] = fmaf(c, c, part[j]);
        }
      }
    }
    const float q = ((part[0] + part[1]) + (part[2] + part[3])) +
                    ((part[4] + part[5]) + (part[6] + part[7]));
    const float rstd = rsqrtf(block_sum(q, red[1]) * inv_d + eps);

    uint4* yr = y + row * nvec;
    if (!row_ok) continue;   // checked build only
    if (m >= n_mod) {  // uniform across the CTA
      if (threadIdx.x == 0) atomicCAS(status, H3_DEV_OK, H3_DEV_BAD_INDEX);
      const uint4 nan4 = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * kThreads;
        if (c < nvec) yr[c] = nan4;
      }
      continue;
    }
    const float4* sc = reinterpret_cast<const float4*>(scale + size_t(m) * d);
    const float4* sh = reinterpret_cast<const float4*>(shift + size_t(m) * d);
    if (kRegs && m != m_cur) {
      m_cur = m;
#pragma unroll
      for (int i = 0; i < (kRegs ? VPT : 0); ++i) {
        const int c = threadIdx.x + i * kThreads;
        if (c < nvec) {
          const float4 a0 = __ldg(sc + 2 * c), a1 = __ldg(sc + 2 * c + 1);
          const float4 b0 = __ldg(sh + 2 * c), b1 = __ldg(sh + 2 * c + 1);
          ga[i][0] = 1.f + a0.x; ga[i][1] = 1.f + a0.y; ga[i][2] = 1.f + a0.z; ga[i][3] = 1.f + a0.w;
          ga[i][4] = 1.f + a1.x; ga[i][5] = 1.f + a1.y; ga[i][6] = 1.f + a1.z; ga[i][7] = 1.f + a1.w;
          gb[i][0] = b0.x; gb[i][1] = b0.y; gb[i][2] = b0.z; gb[i][3] = b0.w;
          gb[i][4] = b1.x; gb[i][5] = b1.y; gb[i][6] = b1.z; gb[i][7] = b1.w;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = threadIdx.x + i * kThreads;
      if (c < nvec) {
        float f[8];
        unpack8(v[i], f);
        float a[8], b[8];
        if constexpr (kRegs) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            a[j] = ga[i][j];
            b[j] = gb[i][j];
          }
        } else {
          const float4 a0 = __ldg(sc + 2 * c), a1 = __ldg(sc + 2 * c + 1);
          const float4 b0 = __ldg(sh + 2 * c), b1 = __ldg(sh + 2 * c + 1);
          const float aa[8] = {1.f + a0.x, 1.f + a0.y, 1.f + a0.z, 1.f + a0.w,
                               1.f + a1.x, 1.f + a1.y, 1.f + a1.z, 1.f + a1.w};
          const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            a[j] = aa[j];
            b[j] = bb[j];
          }
        }
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float y0 = fmaf((f[2 * j] - mean) * rstd, a[2 * j], b[2 * j]);
          const float y1 = fmaf((f[2 * j + 1] - mean) * rstd, a[2 * j + 1], b[2 * j + 1]);
          o[j] = pack_bf16x2(y0, y1);
        }
        __stcs(yr + c, make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
  }
  // a wait that gave up: let the copies still in flight land before the CTA
  // (and its shared memory) goes away
  if (k < nk && threadIdx.x == 0) {
    volatile int no_abort = 0;
    WaitCtx drain{&no_abort, status, kDrainWaitNs};
    for (int j = k; j < issued; ++j)
      mbar_wait(smem_u32(&full[j % stages]), uint32_t(j / stages) & 1u, drain);
  }
}

template <int VPT>
cudaError_t launch_vpt(const void* x, const uint8_t* mod, const float* shift, const float* scale,
                       int L, int d, int n_mod, float eps, void* y, const DevCtx& ctx,
                       cudaStream_t st) {
  // ring of row buffers: 4 per CTA while they take at most 64 KB, else 2
  const size_t row_bytes = size_t(d) * 2;
  const int stages = row_bytes * kMaxStages <= 64 * 1024 ? kMaxStages : 2;
  const size_t smem = row_bytes * stages;
  cudaError_t e = cudaFuncSetAttribute(adaln_modulate_kernel<VPT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  // CTAs that fit an SM at once (registers and shared memory), at most 4
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, adaln_modulate_kernel<VPT>, kThreads,
                                                    smem);
  if (e != cudaSuccess) return e;
  per_sm = per_sm < 1 ? 1 : (per_sm > 4 ? 4 : per_sm);
  const long long want = (long long)ctx.num_sms * per_sm;
  const int grid = int(L < want ? L : want);
  adaln_modulate_kernel<VPT><<<grid, kThreads, smem, st>>>(
      static_cast<const uint4*>(x), mod, shift, scale, L, d, n_mod, eps, stages,
      static_cast<uint4*>(y), ctx.status, ctx.wait_ns);
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
