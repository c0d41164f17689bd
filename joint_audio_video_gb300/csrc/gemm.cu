// Persistent tcgen05 GEMM  C[M][N] = A[M][K] * B[N][K]^T  (bf16 or fp8 E4M3 in,
// fp32 accumulate; fp8 results are scaled by a_scale[row] * b_scale[col]) with the
// sub-block's fused epilogues:
//   EPI_PLAIN           C = acc                                     (h3_qkv_proj)
//   EPI_ROPE            Q/K columns rotated by the 3D (t,h,w) RoPE, V as is
//                       (fused QKV projection of the block; "Joint Audio-Video
//                       Generation in Production", §3: tags + RoPE per token)
//   EPI_GATED_RESIDUAL  C = x_res + gate[mod] * acc                 (output projection
//                       + AdaLN gate; "DiffusionNFT on MiniMax H3", modality-specific
//                       AdaLN branches)
//   EPI_GELU            C = gelu(acc), tanh form                    (feed-forward up
//                       projection ff.net.0.proj of the MLP sub-block)
//
// Two forms.  For N % 256 == 0 a CTA pair (tcgen05 cta_group::2, clusters of
// two) computes 256 x 256 tiles; see gemm_pair_kernel below.  Otherwise the
// single-CTA form, laid out as follows (one CTA per SM, 192 threads):
//   warp 0      TMA producer: A tile 128x64 and B tile BNx64 per k-block into a
//               shared-memory ring (128-byte swizzle, 1 KB aligned; 6 stages at
//               BN = 128, the width this form runs at)
//   warp 1      TMEM allocation + tcgen05.mma issue (the warp runs the loop,
//               one elected lane issues)
//               (M=128, N=BN, K=16 per instruction) into one of two TMEM
//               accumulators (2 x BN fp32 columns)
//   warps 2..5  epilogue: tcgen05.ld of one accumulator row per thread, fused
//               epilogue math in fp32, bf16 stores; releases the accumulator
//               so the MMA of the next tile overlaps this epilogue
// Tiles are visited in groups of kGroupM row-tiles (all N tiles of a group
// before the next group), so the working set of A and B stays in L2.
#include <atomic>

#include <cuda_bf16.h>

#include "kernels.hpp"
#include "ptx.cuh"
#include "tmap.hpp"

namespace h3 {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;          // bf16 elements per k-block (128 bytes; fp8: 128 elements)
constexpr int kThreads = 192;
constexpr int kGroupM = 16;

template <int BN>
struct GemmCfg {
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr uint32_t kABytes = BM * BK * 2;
  static constexpr uint32_t kBBytes = BN * BK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
  static constexpr size_t kSmem = size_t(kStages) * kStageBytes + 2 * BM * 64 + 1024;
};

struct GemmDev {
  __nv_bfloat16* C;
  int M, N, K;
  int num_m, num_n;
  const int32_t* pos;
  int d;
  const __nv_bfloat16* x_res;
  const uint8_t* mod;
  const float* gate;
  int n_mod;
  int* status;
  uint64_t wait_ns;
  const float* a_scale;
  const float* b_scale;
};

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int& mb, int& nb,
                                            int group_m = kGroupM) {
  const int per_group = group_m * num_n;
  const int g = t / per_group;
  const int first_m = g * group_m;
  const int gsz = min(num_m - first_m, group_m);
  const int r = t - g * per_group;
  mb = first_m + r % gsz;
  nb = r / gsz;
}

// Epilogue of one 32-column chunk held in r[] (fp32 bits) for row `grow`,
// global columns gc .. gc+31.
template <int EPI, bool FP8>
__device__ __forceinline__ void epilogue_chunk(const GemmDev& p, const RopeTable& rt,
                                               uint32_t (&r)[32], int grow, int gc,
                                               const int32_t (&pr)[3], int m, float sa,
                                               uint32_t (&pk)[16]) {
  // columns gc .. gc + 31 of C, x_res, gate and b_scale
  if (!H3_IN(gc >= 0 && gc + 32 <= p.N, p.status)) return;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
  if constexpr (FP8) {   // dequantise: row scale of A times column scale of B
    const float4* sb = reinterpret_cast<const float4*>(p.b_scale + gc);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 b = __ldg(sb + i);
      v[4 * i + 0] *= sa * b.x;
      v[4 * i + 1] *= sa * b.y;
      v[4 * i + 2] *= sa * b.z;
      v[4 * i + 3] *= sa * b.w;
    }
  }
  if constexpr (EPI == EPI_ROPE) {
    if (gc < 2 * p.d) {   // Q or K block: rotate pairs (2k, 2k+1) of the head
      const int k0 = (gc & 127) >> 1;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int k = k0 + j;
        const int ax = rt.axis[k];
        const int pa = ax == 0 ? pr[0] : (ax == 1 ? pr[1] : pr[2]);
        const float ang = float(pa) * rt.inv_freq[k];
        float s, c;
        sincosf(ang, &s, &c);
        const float a = v[2 * j], b = v[2 * j + 1];
        v[2 * j] = a * c - b * s;
        v[2 * j + 1] = a * s + b * c;
      }
    }
  }
  if constexpr (EPI == EPI_GELU) {
    // 0.5 u (1 + tanh(sqrt(2/pi) (u + 0.044715 u^3))), tanh by the MUFU
    // instruction (relative error ~2^-11, below the bf16 rounding of the result)
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float u = v[i];
      float t;
      asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.7978845608028654f * fmaf(0.044715f * u, u * u, u)));
      v[i] = 0.5f * u * (1.f + t);
    }
  }
  if constexpr (EPI == EPI_GATED_RESIDUAL) {
    const uint4* xr = reinterpret_cast<const uint4*>(p.x_res + size_t(grow) * p.N + gc);
    const float4* gr = reinterpret_cast<const float4*>(p.gate + size_t(m) * p.N + gc);
    uint4 xv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) xv[i] = xr[i];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 g = __ldg(gr + i);
      const uint32_t w0 = (&xv[i >> 1].x)[(i & 1) * 2];
      const uint32_t w1 = (&xv[i >> 1].x)[(i & 1) * 2 + 1];
      v[4 * i + 0] = fmaf(g.x, v[4 * i + 0], __uint_as_float(w0 << 16));
      v[4 * i + 1] = fmaf(g.y, v[4 * i + 1], __uint_as_float(w0 & 0xFFFF0000u));
      v[4 * i + 2] = fmaf(g.z, v[4 * i + 2], __uint_as_float(w1 << 16));
      v[4 * i + 3] = fmaf(g.w, v[4 * i + 3], __uint_as_float(w1 & 0xFFFF0000u));
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
}

// The epilogue hands C to the TMA in 128-row x 32-column chunks staged in shared
// memory (64-byte rows with the 64-byte swizzle: 16-byte chunk c of row r at
// c ^ ((r / 2) % 4)), two staging buffers; each chunk is one bulk tensor store,
// so C leaves the SM as whole lines instead of one 16-byte piece per row.
constexpr uint32_t kStageC = BM * 64;   // bytes of one staging buffer
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// At most one committed store group may still be reading shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void epi_bar() {   // the 128 epilogue threads
  asm volatile("bar.sync 1, 128;" ::: "memory");
}
__device__ __forceinline__ bool epi_bar_and(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q, a;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred a, 1, 128, q;\n\tselp.u32 %0, 1, 0, a;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(pred))
      : "memory");
  return r != 0;
}

// Epilogue of one finished accumulator: 128 rows (this thread's row is
// row_in_tile) x BN columns at tensor-memory address tacc, written as C rows
// row0 .. row0 + 127, columns col0 .. col0 + BN - 1.  Returns true if the
// row's modality id was out of range (the row is written as NaN).
template <int BN, int EPI, bool FP8>
__device__ __forceinline__ bool epilogue_tile(const GemmDev& p, const RopeTable& rt,
                                              const CUtensorMap* tmC, uint32_t tacc, int row0,
                                              int col0, int row_in_tile, bool leader, uint32_t sC,
                                              int& chunk) {
  const uint32_t srow = uint32_t(row_in_tile) * 64;
  const uint32_t ssw = uint32_t(row_in_tile >> 1) & 3u;
  const int grow = row0 + row_in_tile;
  const bool live = grow < p.M;
  int32_t pr[3] = {0, 0, 0};
  int m = 0;
  if constexpr (EPI == EPI_ROPE) {
    if (live) {
      pr[0] = p.pos[size_t(grow) * 3 + 0];
      pr[1] = p.pos[size_t(grow) * 3 + 1];
      pr[2] = p.pos[size_t(grow) * 3 + 2];
    }
  }
  float sa = 1.f;
  if constexpr (FP8) {
    if (live) sa = __ldg(p.a_scale + grow);
  }
  bool bad = false;
  if constexpr (EPI == EPI_GATED_RESIDUAL) {
    if (live) {
      m = p.mod[grow];
      if (m >= p.n_mod) { bad = true; m = 0; }
    }
  }
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(tacc + c * 32, r);
    tmem_ld_wait(r);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = 0u;   // rows past M: clipped by the store
    if (live) {
      if (bad) {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0x7FC00000u;   // NaN row
      }
      epilogue_chunk<EPI, FP8>(p, rt, r, grow, col0 + c * 32, pr, m, sa, pk);
    }
    // the store that last read this buffer (two chunks ago) has read it
    const uint32_t sb = sC + uint32_t(chunk & 1) * kStageC;
    if (leader) bulk_wait_read_1();
    epi_bar();
#pragma unroll
    for (int i = 0; i < 4; ++i)
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sb + srow + ((uint32_t(i) ^ ssw) << 4)),
                   "r"(pk[4 * i]), "r"(pk[4 * i + 1]), "r"(pk[4 * i + 2]), "r"(pk[4 * i + 3])
                   : "memory");
    fence_async_shared();
    epi_bar();
    if (leader) {
      tma_store_2d(tmC, sb, col0 + c * 32, row0);
      bulk_commit();
    }
    ++chunk;
  }
  return bad;
}

template <int BN, int EPI, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ GemmDev p,
                const __grid_constant__ RopeTable rt) {
  using Cfg = GemmCfg<BN>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[S], bar_empty[S], bar_acc_full[2], bar_acc_empty[2], bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = warp_id();
  const WaitCtx wc{&abort_flag, p.status, p.wait_ns};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&bar_acc_full[a]), 1);
      mbar_init(smem_u32(&bar_acc_empty[a]), 128);
    }
    mbar_init(smem_u32(&bar_drain), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), Cfg::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  const int num_tiles = p.num_m * p.num_n;
  const int kblocks = FP8 ? p.K / (2 * BK) : p.K / BK;   // 128-byte k-blocks

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane_id() == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, p.num_m, p.num_n, mb, nb);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(smem_u32(&bar_empty[stage]), phase ^ 1u, wc)) { ok = false; break; }
          const uint32_t fb = smem_u32(&bar_full[stage]);
          const uint32_t sa = base + stage * Cfg::kStageBytes;
          mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
          const int kx = FP8 ? kb * 2 * BK : kb * BK;   // element coordinate of the k-block
          tma_load_2d(sa, &tmA, fb, kx, mb * BM);
          tma_load_2d(sa + Cfg::kABytes, &tmB, fb, kx, nb * BN);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // unwind: let copies already in flight land before the CTA exits
        WaitCtx drain{&abort_flag, p.status, kDrainWaitNs};
        volatile int no_abort = 0;
        drain.abort = &no_abort;
        for (int s = 0; s < S; ++s) {
          // a stage is in flight iff its full barrier is one phase behind the ring
          const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
          mbar_wait(smem_u32(&bar_full[s]), par, drain);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop (waits and descriptor arithmetic stay
    // warp-uniform); one elected lane issues the products and commits.
    const bool leader = elect_one();
    constexpr uint32_t idesc = FP8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN, 0, 0);
    // stages are kStageBytes apart: precomputed descriptors plus one add per MMA
    const SDesc dA0 = sdesc_split(sdesc_sw128(base, 16, 1024));
    const SDesc dB0 = sdesc_split(sdesc_sw128(base + Cfg::kABytes, 16, 1024));
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_acc_empty[acc]), acc_phase ^ 1u, wc));
      if (!ok) break;
      tc_fence_after();
      const uint32_t dtm = tmem + acc * BN;
      for (int kb = 0; kb < kblocks; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_full[stage]), phase, wc));
        if (!ok) break;
        tc_fence_after();
        const uint32_t soff = stage * (Cfg::kStageBytes >> 4);
        const SDesc dA{dA0.lo + soff, dA0.hi}, dB{dB0.lo + soff, dB0.hi};
        if (leader) {
          // 4 steps of 32 bytes along K: K=16 for bf16, K=32 for fp8
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if constexpr (FP8)
              mma_f8_ss(dtm, sdesc_at(dA, k * 32), sdesc_at(dB, k * 32), idesc, (kb | k) != 0);
            else
              mma_bf16_ss(dtm, sdesc_at(dA, k * 32), sdesc_at(dB, k * 32), idesc, (kb | k) != 0);
          }
          tc_commit(smem_u32(&bar_empty[stage]));
        }
        __syncwarp();
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (leader) tc_commit(smem_u32(&bar_acc_full[acc]));
      __syncwarp();
    }
    // drain: every MMA issued so far has finished before TMEM is released
    if (leader) tc_commit(smem_u32(&bar_drain));
    __syncwarp();
    WaitCtx drain{&abort_flag, p.status, kDrainWaitNs};
    volatile int no_abort = 0;
    drain.abort = &no_abort;
    mbar_wait(smem_u32(&bar_drain), 0, drain);
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int row_in_tile = q * 32 + lane_id();
    const bool leader = threadIdx.x == 64;   // issues the C stores
    const uint32_t sC = base + S * Cfg::kStageBytes;
    int chunk = 0;                           // C chunks staged so far (buffer parity)
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      int mb, nb;
      tile_coords(t, p.num_m, p.num_n, mb, nb);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      // all four epilogue warps leave together (they share the staging barrier)
      const bool ok = epi_bar_and(mbar_wait(smem_u32(&bar_acc_full[acc]), acc_phase, wc));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tacc = tmem + acc * BN + (uint32_t(q * 32) << 16);
      const bool bad = epilogue_tile<BN, EPI, FP8>(p, rt, &tmC, tacc, mb * BM, nb * BN,
                                                   row_in_tile, leader, sC, chunk);
      if (bad) atomicCAS(p.status, H3_DEV_OK, H3_DEV_BAD_INDEX);
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_acc_empty[acc]));
    }
    // every C store has finished before the CTA (and its shared memory) goes away
    if (leader) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, Cfg::kTmemCols);
}

// ---------------------------------------------------------------------------
// CTA-pair form (tcgen05 cta_group::2), used when N % 256 == 0.  A cluster of
// two CTAs computes one 256 x 256 tile: per k-block each CTA loads 128 rows of
// A and 128 rows of B into its own shared memory (32 KB per stage, 6 stages),
// the MMA thread of the even CTA issues M = 256, N = 256 products that read
// the operands of both CTAs and write 128 accumulator rows into the tensor
// memory of each, and each CTA's epilogue writes its own 128 rows of C.
// Against the single-CTA form a stage holds half of the B tile, so the ring is
// deeper for the same shared memory and each SM streams 2/3 of the bytes.
constexpr int kPairStages = 6;
constexpr int kPairGroupM = 16;                       // 256-row tiles per group
constexpr uint32_t kPairABytes = BM * 128;            // 128 rows x 128 bytes
constexpr uint32_t kPairBBytes = 128 * 128;           // 128 rows of B x 128 bytes
constexpr uint32_t kPairStageBytes = kPairABytes + kPairBBytes;
constexpr size_t kPairSmem = size_t(kPairStages) * kPairStageBytes + 2 * kStageC + 1024;

template <int EPI, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ GemmDev p,
                     const __grid_constant__ RopeTable rt) {
  constexpr int BN = 256;
  constexpr int S = kPairStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[S], bar_empty[S], bar_acc_full[2], bar_acc_empty[2], bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = warp_id();
  const uint32_t rank = cluster_ctarank();   // 0: issues the pair's products
  const bool lead = rank == 0;
  const WaitCtx wc{&abort_flag, p.status, p.wait_ns};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);    // the even CTA's: both CTAs' bytes
      mbar_init(smem_u32(&bar_empty[s]), 1);   // one multicast commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&bar_acc_full[a]), 1);
      mbar_init(smem_u32(&bar_acc_empty[a]), 2);   // the even CTA's: one per CTA
    }
    mbar_init(smem_u32(&bar_drain), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&tmem_base_sh), 2 * BN);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before any signal crosses
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const int num_tiles = p.num_m * p.num_n;
  const int kblocks = FP8 ? p.K / (2 * BK) : p.K / BK;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane_id() == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = cid; t < num_tiles && ok; t += ncl) {
        int mb, nb;
        tile_coords(t, p.num_m, p.num_n, mb, nb, kPairGroupM);
        const int ya = mb * 256 + int(rank) * 128, yb = nb * BN + int(rank) * 128;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(smem_u32(&bar_empty[stage]), phase ^ 1u, wc)) { ok = false; break; }
          const uint32_t fb = smem_u32(&bar_full[stage]);
          if (lead) mbar_arrive_expect_tx(fb, 2 * kPairStageBytes);
          const uint32_t cfb = cluster_addr(fb, 0);
          const uint32_t sa = base + stage * kPairStageBytes;
          const int kx = FP8 ? kb * 2 * BK : kb * BK;
          tma_load_2d_pair(sa, &tmA, cfb, kx, ya);
          tma_load_2d_pair(sa + kPairABytes, &tmB, cfb, kx, yb);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) abort_grace();
      if (!ok && lead) {
        // unwind: let the stages armed here land before the CTA exits (the
        // odd CTA's copies of a stage count on the same barrier)
        WaitCtx drain{&abort_flag, p.status, kDrainWaitNs};
        volatile int no_abort = 0;
        drain.abort = &no_abort;
        for (int s = 0; s < S; ++s) {
          const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
          mbar_wait(smem_u32(&bar_full[s]), par, drain);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lead) {
      const bool leader = elect_one();
      constexpr uint32_t idesc = FP8 ? idesc_e4m3_f32(256, BN) : idesc_bf16_f32(256, BN, 0, 0);
      const SDesc dA0 = sdesc_split(sdesc_sw128(base, 16, 1024));
      const SDesc dB0 = sdesc_split(sdesc_sw128(base + kPairABytes, 16, 1024));
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = cid; t < num_tiles && ok; t += ncl, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        ok = __all_sync(0xffffffffu,
                        mbar_wait_cluster(smem_u32(&bar_acc_empty[acc]), acc_phase ^ 1u, wc));
        if (!ok) break;
        tc_fence_after();
        const uint32_t dtm = tmem + acc * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_full[stage]), phase, wc));
          if (!ok) break;
          tc_fence_after();
          const uint32_t soff = stage * (kPairStageBytes >> 4);
          const SDesc dA{dA0.lo + soff, dA0.hi}, dB{dB0.lo + soff, dB0.hi};
          if (leader) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if constexpr (FP8)
                mma_f8_ss_pair(dtm, sdesc_at(dA, k * 32), sdesc_at(dB, k * 32), idesc, (kb | k) != 0);
              else
                mma_bf16_ss_pair(dtm, sdesc_at(dA, k * 32), sdesc_at(dB, k * 32), idesc,
                                 (kb | k) != 0);
            }
            tc_commit_pair(smem_u32(&bar_empty[stage]), 0x3);
          }
          __syncwarp();
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (leader) tc_commit_pair(smem_u32(&bar_acc_full[acc]), 0x3);
        __syncwarp();
      }
      if (leader) tc_commit_pair(smem_u32(&bar_drain), 0x3);
      __syncwarp();
    }
    // every product that writes this CTA's tensor memory has finished
    WaitCtx drain{&abort_flag, p.status, kDrainWaitNs};
    volatile int no_abort = 0;
    drain.abort = &no_abort;
    mbar_wait(smem_u32(&bar_drain), 0, drain);
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane_id();
    const bool leader = threadIdx.x == 64;
    const uint32_t sC = base + S * kPairStageBytes;
    const uint32_t acc_empty_c[2] = {cluster_addr(smem_u32(&bar_acc_empty[0]), 0),
                                     cluster_addr(smem_u32(&bar_acc_empty[1]), 0)};
    int chunk = 0;
    int it = 0;
    for (int t = cid; t < num_tiles; t += ncl, ++it) {
      int mb, nb;
      tile_coords(t, p.num_m, p.num_n, mb, nb, kPairGroupM);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const bool ok = epi_bar_and(mbar_wait(smem_u32(&bar_acc_full[acc]), acc_phase, wc));
      if (!ok) break;
      tc_fence_after();
      const int row0 = mb * 256 + int(rank) * 128;
      bool bad = false;
      if (row0 < p.M) {   // a CTA whose rows all lie past M has nothing to write
        const uint32_t tacc = tmem + acc * BN + (uint32_t(q * 32) << 16);
        bad = epilogue_tile<BN, EPI, FP8>(p, rt, &tmC, tacc, row0, nb * BN, row_in_tile, leader,
                                          sC, chunk);
      }
      if (bad) atomicCAS(p.status, H3_DEV_OK, H3_DEV_BAD_INDEX);
      tc_fence_before();
      epi_bar();
      if (leader) mbar_arrive_cluster(acc_empty_c[acc]);
    }
    if (leader) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // neither CTA leaves while the other may still signal it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, 2 * BN);
}

template <int EPI, bool FP8>
cudaError_t launch_pair(const GemmArgs& a, const DevCtx& ctx, cudaStream_t st) {
  CUtensorMap tmA, tmB, tmC;
  if constexpr (FP8) {
    if (!make_tmap_u8_2d(&tmA, a.A, a.M, a.K, a.K, BM)) return cudaErrorInvalidValue;
    if (!make_tmap_u8_2d(&tmB, a.B, a.N, a.K, a.K, 128)) return cudaErrorInvalidValue;
  } else {
    if (!make_tmap_bf16_2d(&tmA, a.A, a.M, a.K, a.K, BM, BK)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16_2d(&tmB, a.B, a.N, a.K, a.K, 128, BK)) return cudaErrorInvalidValue;
  }
  if (!make_tmap_bf16_2d_sw64(&tmC, a.C, a.M, a.N, a.N, BM)) return cudaErrorInvalidValue;
  GemmDev p{};
  p.C = static_cast<__nv_bfloat16*>(a.C);
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.num_m = (a.M + 255) / 256;
  p.num_n = a.N / 256;
  p.pos = a.pos;
  p.d = a.d;
  p.x_res = static_cast<const __nv_bfloat16*>(a.x_res);
  p.mod = a.mod;
  p.gate = a.gate;
  p.n_mod = a.n_mod;
  p.status = ctx.status;
  p.wait_ns = ctx.wait_ns;
  p.a_scale = a.a_scale;
  p.b_scale = a.b_scale;
  RopeTable rt{};
  if (a.rope) rt = *a.rope;
  auto kern = gemm_pair_kernel<EPI, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(kPairSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(ctx.num_sms & ~1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // how many pairs can be resident at once (SM pairs of the GPU), asked once per
  // device; callers on several host threads may race to fill the entry with the
  // same value
  static std::atomic<int> resident[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int nres = resident[dev].load(std::memory_order_relaxed);
  if (nres <= 0) {
    e = cudaOccupancyMaxActiveClusters(&nres, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (nres <= 0) return cudaErrorInvalidConfiguration;
    resident[dev].store(nres, std::memory_order_relaxed);
  }
  const int tiles = p.num_m * p.num_n;
  const int ncl = tiles < nres ? tiles : nres;
  cfg.gridDim = dim3(unsigned(2 * ncl));
  e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, p, rt);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool FP8>
cudaError_t launch_pair_epi(const GemmArgs& a, const DevCtx& ctx, cudaStream_t st) {
  switch (a.epilogue) {
    case EPI_PLAIN: return launch_pair<EPI_PLAIN, FP8>(a, ctx, st);
    case EPI_ROPE: return launch_pair<EPI_ROPE, FP8>(a, ctx, st);
    case EPI_GATED_RESIDUAL: return launch_pair<EPI_GATED_RESIDUAL, FP8>(a, ctx, st);
    case EPI_GELU: return launch_pair<EPI_GELU, FP8>(a, ctx, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int BN, int EPI, bool FP8>
cudaError_t launch_typed(const GemmArgs& a, const DevCtx& ctx, cudaStream_t st) {
  using Cfg = GemmCfg<BN>;
  CUtensorMap tmA, tmB;
  if constexpr (FP8) {
    if (!make_tmap_u8_2d(&tmA, a.A, a.M, a.K, a.K, BM)) return cudaErrorInvalidValue;
    if (!make_tmap_u8_2d(&tmB, a.B, a.N, a.K, a.K, BN)) return cudaErrorInvalidValue;
  } else {
    if (!make_tmap_bf16_2d(&tmA, a.A, a.M, a.K, a.K, BM, BK)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16_2d(&tmB, a.B, a.N, a.K, a.K, BN, BK)) return cudaErrorInvalidValue;
  }
  CUtensorMap tmC;
  if (!make_tmap_bf16_2d_sw64(&tmC, a.C, a.M, a.N, a.N, BM)) return cudaErrorInvalidValue;
  GemmDev p{};
  p.C = static_cast<__nv_bfloat16*>(a.C);
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.num_m = (a.M + BM - 1) / BM;
  p.num_n = a.N / BN;
  p.pos = a.pos;
  p.d = a.d;
  p.x_res = static_cast<const __nv_bfloat16*>(a.x_res);
  p.mod = a.mod;
  p.gate = a.gate;
  p.n_mod = a.n_mod;
  p.status = ctx.status;
  p.wait_ns = ctx.wait_ns;
  p.a_scale = a.a_scale;
  p.b_scale = a.b_scale;
  RopeTable rt{};
  if (a.rope) rt = *a.rope;
  auto kern = gemm_kernel<BN, EPI, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(Cfg::kSmem));
  if (e != cudaSuccess) return e;
  const int tiles = p.num_m * p.num_n;
  const int grid = tiles < ctx.num_sms ? tiles : ctx.num_sms;
  kern<<<grid, kThreads, Cfg::kSmem, st>>>(tmA, tmB, tmC, p, rt);
  return cudaGetLastError();
}

template <int BN, bool FP8>
cudaError_t launch_bn(const GemmArgs& a, const DevCtx& ctx, cudaStream_t st) {
  switch (a.epilogue) {
    case EPI_PLAIN: return launch_typed<BN, EPI_PLAIN, FP8>(a, ctx, st);
    case EPI_ROPE: return launch_typed<BN, EPI_ROPE, FP8>(a, ctx, st);
    case EPI_GATED_RESIDUAL: return launch_typed<BN, EPI_GATED_RESIDUAL, FP8>(a, ctx, st);
    case EPI_GELU: return launch_typed<BN, EPI_GELU, FP8>(a, ctx, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, const DevCtx& ctx, cudaStream_t st) {
  if (a.fp8) {
    if (a.N % 256 == 0) return launch_pair_epi<true>(a, ctx, st);
    return launch_bn<128, true>(a, ctx, st);
  }
  if (a.N % 256 == 0) return launch_pair_epi<false>(a, ctx, st);
  return launch_bn<128, false>(a, ctx, st);
}

}  // namespace h3
