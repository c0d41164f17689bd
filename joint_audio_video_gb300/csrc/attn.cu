// Joint attention over the whole packed sequence on tcgen05 / TMEM.
//
//   O[n, h] = softmax_j(q_n . k_j * sm_scale [j <= n if causal]) v_j,  j in [0, L)
//
// "Joint Audio-Video Generation in Production", §1 Unified Architecture (all
// modalities share one attention context at every step) and §6 Boundary
// Trimming for Packed Attention (only the L effective tokens may take part:
// keys >= L are masked here, nothing is padded); "多模态强化学习工程解析…",
// 三 目标模型 (causal attention over the packed sequence, kept as an option).
//
// One cluster of two CTAs (a CTA pair, tcgen05 cta_group::2) = one head x 512
// query rows; each CTA holds 256 of them as two 128-row tiles Q0, Q1.  The
// products of tile g are issued once for the pair (M = 256: the g-th tiles of
// both CTAs) by the even CTA's MMA warp: S_g = Q_g K^T reads each CTA's Q_g
// and the 64 keys of K that each CTA holds, P_g V reads each CTA's P_g from its
// tensor memory and the 64 head dims of V that each CTA holds, and every
// product writes 128 rows into the tensor memory of each CTA.  So each SM
// loads half of every K/V block and issues half the products of a single-CTA
// kernel.  320 threads per CTA:
//   warp 0      TMA producer: Q0|Q1 once, then per key block j the pair
//               (K_j, V_{j-1}) that block's products read -- this CTA's 64 keys
//               of K_j (two 64 x 64 boxes, 128-byte swizzle) and its 64 dims of
//               V_{j-1} (one 128 x 64 box) -- into a ring of pair slots; the
//               copies of both CTAs count on the even CTA's barrier
//   warp 1      TMEM owner (both CTAs allocate together); in the even CTA the
//               tcgen05.mma issuer (the warp runs the loop, one elected lane
//               issues and commits to the barriers of both CTAs)
//   warps 2..5  softmax warpgroup of tile 0 (one query row per thread)
//   warps 6..9  softmax warpgroup of tile 1
// Tensor memory (512 columns per CTA): S0 | S1 | O0 | O1, 128 fp32 columns
// each.  The softmax writes P (bf16 pairs) over the last 64 columns of its S
// buffer and the P.V product reads it from TMEM as the A operand; V is the
// MN-major B operand straight from the TMA tile.
// MMA order per key block j:  P0V(j-1), S0(j), P1V(j-1), S1(j), so the tensor
// cores compute one tile's products while the other tile's softmax runs.
// Softmax works in the log2 domain with a per-row running maximum that is
// only moved (and O, l rescaled in TMEM) when the block maximum exceeds it by
// more than 8 (factor 256): the final O / l is exact for any such maximum.
// The exponentials are computed against the running maximum in the same pass
// that takes the block maximum; a block that moves it is redone.
//
// FP8 scores (the quantised-attention prior art that §6 of "Joint Audio-Video
// Generation in Production" names, in the form that keeps P.V in bf16): Q and
// K arrive as E4M3 (128 bytes per head row: one 16 KB box per Q tile, one 8 KB
// box of 64 keys per CTA and K block) with a per-token Q scale and a
// per-128-key-block K scale; S = Q8 K8^T runs as four
// kind::f8f6f4 products of K = 32, and the two scales fold into the softmax's
// per-row, per-block constant: s = sq[i] sk[b] (q8 . k8).
#include <cuda_bf16.h>

#include "kernels.hpp"
#include "ptx.cuh"
#include "tmap.hpp"

namespace h3 {
namespace {

constexpr int kThreads = 320;
constexpr int kSlots = 4;                     // pair slots (K_j half | V_{j-1} half)
constexpr uint32_t kTile = 128 * 128 * 2;     // one 128x128 bf16 tile (two 16 KB boxes)
constexpr uint32_t kBox = 128 * 64 * 2;       // 128 rows x 64 bf16
constexpr uint32_t kHalfBox = 64 * 64 * 2;    // 64 rows x 64 bf16
constexpr uint32_t kTile8 = 128 * 128;        // one 128x128 E4M3 tile (one 16 KB box)
constexpr uint32_t kSlotBytes = 2 * kBox;     // this CTA's K half (16 KB) | V half (16 KB)
constexpr size_t kSmem = 2 * kTile + kSlots * kSlotBytes + 1024;
constexpr float kRescaleThreshold = 8.0f;     // log2 units

struct AttnDev {
  __nv_bfloat16* O;
  float* lse;
  int L, H, d;
  int causal;
  float scale_log2;   // sm_scale * log2(e)
  int num_quads;                  // clusters per head: 512 query rows each
  int* status;
  uint64_t wait_ns;
  int n_seg;                      // 0: one segment [0, L)
  int32_t cu[kMaxSegments + 1];   // segment starts, cu[n_seg] = L
  const float* sq;                // fp8 scores: [H][L] Q scales
  const float* sk;                // fp8 scores: [H][nkb] K block scales
  int nkb;
};

// Segment of token i: the last s with cu[s] <= i (skips empty segments).
__device__ __forceinline__ int segment_of(const AttnDev& p, int i) {
  int lo = 0, hi = p.n_seg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu[mid] <= i) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Packed pairs of fp32 in one 64-bit register (low word = first value).
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// p = 2^(s*c - m) for 32 raw scores: 16 bf16 pairs into pk, row sum into acc.
__device__ __forceinline__ void exp32(const uint32_t (&r)[32], uint64_t cc, uint64_t nm,
                                      uint32_t* pk, uint64_t (&acc)[2]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float a, b;
    unf2(ffma2(f2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), cc, nm), a, b);
    a = ex2(a);
    b = ex2(b);
    acc[i & 1] = fadd2(acc[i & 1], f2(a, b));
    pk[i] = pack_bf16x2(a, b);
  }
}

// exp32, plus the maximum of the 32 raw scores folded into two running chains
// (for the pass that computes the exponentials before the block maximum is known).
__device__ __forceinline__ void exp32_max(const uint32_t (&r)[32], uint64_t cc, uint64_t nm,
                                          uint32_t* pk, uint64_t (&acc)[2], float (&mc)[2]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float s0 = __uint_as_float(r[2 * i]), s1 = __uint_as_float(r[2 * i + 1]);
    mc[i & 1] = max3(mc[i & 1], s0, s1);
    float a, b;
    unf2(ffma2(f2(s0, s1), cc, nm), a, b);
    a = ex2(a);
    b = ex2(b);
    acc[i & 1] = fadd2(acc[i & 1], f2(a, b));
    pk[i] = pack_bf16x2(a, b);
  }
}

// O (this thread's row, 128 fp32 columns in TMEM) times f.
__device__ __forceinline__ void rescale_o(uint32_t tO, float f) {
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t o[32];
    tmem_ld32(tO + c * 32, o);
    tmem_ld_wait(o);
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
    tmem_st32(tO + c * 32, o);
  }
  tmem_st_wait();
}

// Keys of block column c visible to the row iff lo_rel <= c < hi_rel.
__device__ __forceinline__ void mask32(uint32_t (&r)[32], int base, int lo_rel, int hi_rel) {
  constexpr uint32_t kNegInf = 0xFF800000u;
#pragma unroll
  for (int c = 0; c < 32; ++c)
    if (c + base < lo_rel || c + base >= hi_rel) r[c] = kNegInf;
}

// The MMA issuer keeps every operand descriptor precomputed: issuing one
// 256x128x16 pair product (64 tensor-core cycles on each SM) must cost far
// less than 64 cycles of the issuing thread, or the tensor cores wait on it.
// S = Q K^T: both K-major, 8 steps of K=16 over the two 64-column boxes (each
// CTA: Q boxes of 128 rows, K boxes of its 64 keys).
template <bool FP8>
__device__ __forceinline__ void s_product(uint32_t d_tmem, SDesc q, SDesc k) {
  if constexpr (FP8) {
    // E4M3: one 128-byte row holds the head's 128 dims; 4 steps of K = 32
    constexpr uint32_t idesc = idesc_e4m3_f32(256, 128);
#pragma unroll
    for (int s = 0; s < 4; ++s)
      mma_f8_ss_pair(d_tmem, sdesc_at(q, s * 32), sdesc_at(k, s * 32), idesc, s > 0);
  } else {
    constexpr uint32_t idesc = idesc_bf16_f32(256, 128, 0, 0);
#pragma unroll
    for (int s = 0; s < 8; ++s)
      mma_bf16_ss_pair(d_tmem, sdesc_at(q, (s >> 2) * kBox + (s & 3) * 32),
                       sdesc_at(k, (s >> 2) * kHalfBox + (s & 3) * 32), idesc, s > 0);
  }
}

// O += P V: P (bf16 pairs) from TMEM, V as the MN-major operand (each CTA: its
// 64 head dims), 8 steps of 16 keys.
__device__ __forceinline__ void pv_product(uint32_t o_tmem, uint32_t p_tmem, SDesc v,
                                           bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(256, 128, 0, 1);
#pragma unroll
  for (int s = 0; s < 8; ++s)
    mma_bf16_ts_pair(o_tmem, p_tmem + s * 8, sdesc_at(v, s * 2048), idesc, accumulate || s > 0);
}

// Registers are split over the SM's four sub-partitions (16K each) and warp w
// runs on sub-partition w % 4, so with 10 warps three share one sub-partition:
// at most 168 registers per thread.
template <bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tm8, const __grid_constant__ CUtensorMap tm8k,
                    const __grid_constant__ AttnDev p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_kv_full[kSlots], bar_kv_empty[kSlots], bar_s[2], bar_p[2],
      bar_o, bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;                 // Q0 at sQ, Q1 at sQ + kTile
  const uint32_t sRing = base + 2 * kTile;
  const int warp = warp_id();
  const uint32_t rank = cluster_ctarank();  // 0: issues the pair's products
  const bool lead = rank == 0;
  const WaitCtx wc{&abort_flag, p.status, p.wait_ns};

  const int cl = blockIdx.x >> 1;
  int quad = cl % p.num_quads;
  const int h = cl / p.num_quads;
  if (p.causal) quad = p.num_quads - 1 - quad;   // longest rows first
  const int c0 = quad * 512;                     // the pair's rows: c0 .. c0 + 511
  const int c_last = min(c0 + 511, p.L - 1);
  const int q0 = c0 + int(rank) * 256;           // this CTA's rows: q0 .. q0 + 255
  // keys the pair visits: the union of its rows' segments, cut at the diagonal
  int kv_lo = 0, kv_hi = p.L;
  if (p.n_seg > 0) {
    kv_lo = p.cu[segment_of(p, c0)];
    kv_hi = p.cu[segment_of(p, c_last) + 1];
  }
  if (p.causal) kv_hi = min(kv_hi, c_last + 1);
  const int nblk = (kv_hi - kv_lo + 127) / 128;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_u32(&bar_kv_full[s]), 1);    // the even CTA's: both CTAs' bytes
      mbar_init(smem_u32(&bar_kv_empty[s]), 1);   // one multicast commit
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bar_s[t]), 1);
      mbar_init(smem_u32(&bar_p[t]), 8);          // the even CTA's: 4 softmax warps per CTA
    }
    mbar_init(smem_u32(&bar_o), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(FP8 ? &tm8 : &tm);
    tma_prefetch_desc(FP8 ? &tm8k : &tmk);
    if (FP8) tma_prefetch_desc(&tm);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before any signal crosses
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane_id() == 0) {
      const int xq = h * 128, xk = p.d + h * 128, xv = 2 * p.d + h * 128;
      const uint32_t qb = smem_u32(&bar_q);
      const uint32_t cqb = cluster_addr(qb, 0);
      if (FP8) {   // E4M3 Q | K rows: Q at byte column h*128, K at d + h*128
        if (lead) mbar_arrive_expect_tx(qb, 2 * 2 * kTile8);
        tma_load_2d_pair(sQ, &tm8, cqb, xq, q0);
        tma_load_2d_pair(sQ + kTile, &tm8, cqb, xq, q0 + 128);
      } else {
        if (lead) mbar_arrive_expect_tx(qb, 2 * 2 * kTile);
        tma_load_2d_pair(sQ, &tm, cqb, xq, q0);
        tma_load_2d_pair(sQ + kBox, &tm, cqb, xq + 64, q0);
        tma_load_2d_pair(sQ + kTile, &tm, cqb, xq, q0 + 128);
        tma_load_2d_pair(sQ + kTile + kBox, &tm, cqb, xq + 64, q0 + 128);
      }
      // pair j = this CTA's halves of K_j (j < nblk) and V_{j-1} (j >= 1), the
      // tiles block j's products read, into slot j % kSlots (K half at the
      // slot's start, V half one box further)
      bool ok = true;
      int issued = 0;
      for (int j = 0; j <= nblk && ok; ++j) {
        const int slot = j % kSlots;
        if (!mbar_wait(smem_u32(&bar_kv_empty[slot]), ((j / kSlots) & 1) ^ 1u, wc)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&bar_kv_full[slot]);
        const uint32_t cfb = cluster_addr(fb, 0);
        const uint32_t dst = sRing + slot * kSlotBytes;
        const uint32_t kbytes = j < nblk ? (FP8 ? kTile8 / 2 : kBox) : 0u;
        if (lead) mbar_arrive_expect_tx(fb, 2 * (kbytes + (j >= 1 ? kBox : 0u)));
        if (j < nblk) {
          const int key0 = kv_lo + j * 128 + int(rank) * 64;
          if (FP8) {
            tma_load_2d_pair(dst, &tm8k, cfb, xk, key0);
          } else {
            tma_load_2d_pair(dst, &tmk, cfb, xk, key0);
            tma_load_2d_pair(dst + kHalfBox, &tmk, cfb, xk + 64, key0);
          }
        }
        if (j >= 1) tma_load_2d_pair(dst + kBox, &tm, cfb, xv + int(rank) * 64, kv_lo + (j - 1) * 128);
        issued = j + 1;
      }
      // the even CTA lets every copy it armed land before the CTA can exit
      // (earlier pairs were consumed before their slot was refilled); the odd
      // CTA's copies count on the even CTA's barriers
      if (!ok) abort_grace();
      if (lead) {
        WaitCtx drain{&abort_flag, p.status, kDrainWaitNs};
        volatile int no_abort = 0;
        drain.abort = &no_abort;
        if (!ok)
          for (int k = max(0, issued - kSlots); k < issued; ++k)
            mbar_wait(smem_u32(&bar_kv_full[k % kSlots]), (k / kSlots) & 1, drain);
        mbar_wait(qb, 0, drain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lead) {
      // The whole warp runs the loop (waits and descriptor arithmetic stay
      // warp-uniform); one elected lane issues the products and commits to
      // the barriers of both CTAs.
      const bool leader = elect_one();
      auto wait_all = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc));
      };
      auto wait_p = [&](int g, uint32_t parity) {   // arrivals from both CTAs
        return __all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(&bar_p[g]), parity, wc));
      };
      bool ok = wait_all(smem_u32(&bar_q), 0);
      // descriptors of Q0, Q1 and of every slot read as K (K-major) or V (MN-major)
      const SDesc dQ0 = sdesc_split(sdesc_sw128(sQ, 16, 1024));
      const SDesc dQ1 = sdesc_split(sdesc_sw128(sQ + kTile, 16, 1024));
      // slots are kSlotBytes apart, V one box after K: a descriptor is the
      // first slot's plus the byte offset / 16
      const SDesc dK0 = sdesc_split(sdesc_sw128(sRing, 16, 1024));
      const SDesc dV0 = sdesc_split(sdesc_sw128(sRing + kBox, kBox, 1024));
      auto dK = [&](int j) {
        return SDesc{dK0.lo + uint32_t(j % kSlots) * (kSlotBytes >> 4), dK0.hi};
      };
      auto dV = [&](int j) {
        return SDesc{dV0.lo + uint32_t(j % kSlots) * (kSlotBytes >> 4), dV0.hi};
      };
      auto pair_full = [&](int j) {
        return wait_all(smem_u32(&bar_kv_full[j % kSlots]), (j / kSlots) & 1);
      };
      auto pair_empty = [&](int j) { return smem_u32(&bar_kv_empty[j % kSlots]); };
      const uint32_t tS0 = tmem, tS1 = tmem + 128, tO0 = tmem + 256, tO1 = tmem + 384;
      if (ok) ok = pair_full(0);
      if (ok) {
        tc_fence_after();
        if (leader) {
          s_product<FP8>(tS0, dQ0, dK(0));
          tc_commit_pair(smem_u32(&bar_s[0]), 0x3);
          s_product<FP8>(tS1, dQ1, dK(0));
          tc_commit_pair(smem_u32(&bar_s[1]), 0x3);
          tc_commit_pair(pair_empty(0), 0x3);
        }
        __syncwarp();
      }
      // block j: P(j-1).V_{j-1} and S(j) for each tile, both tiles from pair j
      for (int j = 1; j < nblk && ok; ++j) {
        const uint32_t pph = (j - 1) & 1;
        ok = pair_full(j) && wait_p(0, pph);
        if (!ok) break;
        tc_fence_after();
        if (leader) {
          pv_product(tO0, tS0 + 64, dV(j), j > 1);
          s_product<FP8>(tS0, dQ0, dK(j));
          tc_commit_pair(smem_u32(&bar_s[0]), 0x3);
        }
        __syncwarp();
        ok = wait_p(1, pph);
        if (!ok) break;
        tc_fence_after();
        if (leader) {
          pv_product(tO1, tS1 + 64, dV(j), j > 1);
          s_product<FP8>(tS1, dQ1, dK(j));
          tc_commit_pair(smem_u32(&bar_s[1]), 0x3);
          tc_commit_pair(pair_empty(j), 0x3);
        }
        __syncwarp();
      }
      if (ok) {
        const int j = nblk;
        const uint32_t pph = (j - 1) & 1;
        ok = pair_full(j) && wait_p(0, pph);
        if (ok) {
          tc_fence_after();
          if (leader) pv_product(tO0, tS0 + 64, dV(j), j > 1);
          __syncwarp();
          ok = wait_p(1, pph);
        }
        if (ok) {
          tc_fence_after();
          if (leader) {
            pv_product(tO1, tS1 + 64, dV(j), j > 1);
            tc_commit_pair(pair_empty(j), 0x3);
            tc_commit_pair(smem_u32(&bar_o), 0x3);
          }
          __syncwarp();
        }
      }
      // let every product issued so far finish before either CTA frees tensor memory
      if (leader) tc_commit_pair(smem_u32(&bar_drain), 0x3);
      __syncwarp();
    }
    WaitCtx drain{&abort_flag, p.status, kDrainWaitNs};
    volatile int no_abort = 0;
    drain.abort = &no_abort;
    mbar_wait(smem_u32(&bar_drain), 0, drain);
  } else {
    // ------------------------------------------------------------ softmax
    const int g = (warp - 2) >> 2;          // tile 0 or 1
    const int q = warp & 3;                 // TMEM lane quarter
    const int row = q * 32 + lane_id();
    const int tile_q0 = q0 + g * 128;
    const int qi = tile_q0 + row;
    const uint32_t lane_off = uint32_t(q * 32) << 16;
    const uint32_t tS = tmem + g * 128 + lane_off;
    const uint32_t tO = tmem + 256 + g * 128 + lane_off;
    const uint32_t bs = smem_u32(&bar_s[g]);
    const uint32_t bp = cluster_addr(smem_u32(&bar_p[g]), 0);   // the even CTA's
    // keys visible to this row: its segment, up to itself when causal
    int row_lo = 0, row_hi = p.L;
    if (p.n_seg > 0) {
      const int sg = segment_of(p, min(qi, p.L - 1));
      if (H3_IN(sg >= 0 && sg < p.n_seg, p.status)) {
        row_lo = p.cu[sg];
        row_hi = p.cu[sg + 1];
      }
    }
    if (p.causal) row_hi = min(row_hi, qi + 1);
    float m_used = -INFINITY, l = 0.f;
    // exponent constant: sm_scale log2(e), times the row's Q scale for fp8 scores
    float c_row = p.scale_log2;
    const bool head_ok = H3_IN(h < p.H, p.status);   // column h*128 of O, rows h of lse, sq, sk
    if (FP8 && head_ok) c_row *= p.sq[size_t(h) * p.L + min(qi, p.L - 1)];
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      // ... and the key block's K scale (fp8 scores have kv_lo = 0)
      const float c =
          FP8 && head_ok && H3_IN(j < p.nkb, p.status) ? c_row * p.sk[size_t(h) * p.nkb + j] : c_row;
      ok = __all_sync(0xffffffffu, mbar_wait(bs, j & 1, wc));
      if (!ok) break;
      tc_fence_after();
      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_ld32(tS, r0);
      tmem_ld32(tS + 32, r1);
      tmem_ld32(tS + 64, r2);
      tmem_ld32(tS + 96, r3);
      tmem_ld_wait(r0);
      tmem_ld_wait(r1);
      tmem_ld_wait(r2);
      tmem_ld_wait(r3);
      // block columns c are keys kv_lo + 128 j + c; visible iff lo_rel <= c < hi_rel
      const int kv0 = kv_lo + j * 128;
      const int lo_rel = row_lo - kv0, hi_rel = row_hi - kv0;
      const bool masked = __any_sync(0xffffffffu, lo_rel > 0 || hi_rel < 128);
      if (masked) {
        mask32(r0, 0, lo_rel, hi_rel);
        mask32(r1, 32, lo_rel, hi_rel);
        mask32(r2, 64, lo_rel, hi_rel);
        mask32(r3, 96, lo_rel, hi_rel);
      }
      // P (bf16 pairs) goes over the second half of S (columns 64..127): the
      // first half keeps the raw scores of keys 0..63 for an exact redo, and
      // the scores of keys 64..127 are still in r2, r3 when P overwrites them
      // p = 2^(s * c - m_used) straight away, with the block maximum taken in
      // the same pass.  Only when that maximum exceeds the running one by more
      // than the threshold is the block redone against the new maximum: rare
      // once a row has seen a few blocks, and always for a row's first visible
      // block (no running maximum yet: the pass runs against 0 and is discarded).
      uint64_t acc[2] = {0ull, 0ull};
      uint32_t pk0[32], pk1[32];
      const uint64_t cc = f2(c, c);
      float neg_m = m_used == -INFINITY ? 0.f : -m_used;
      uint64_t nm = f2(neg_m, neg_m);
      float mc[2] = {-INFINITY, -INFINITY};
      exp32_max(r0, cc, nm, pk0, acc, mc);
      exp32_max(r1, cc, nm, pk0 + 16, acc, mc);
      tmem_st32(tS + 64, pk0);
      exp32_max(r2, cc, nm, pk1, acc, mc);
      exp32_max(r3, cc, nm, pk1 + 16, acc, mc);
      tmem_st32(tS + 96, pk1);
      // raw maximum times c (> 0); -inf while no key of the row is visible
      const float mx = fmaxf(mc[0], mc[1]) * c;
      const bool need = mx > m_used + kRescaleThreshold;   // -inf + 8 = -inf: a first key
      if (__any_sync(0xffffffffu, need)) {
        // O and l hold the blocks before this one against m_used; nothing yet
        // for a row without a running maximum (f = 0 keeps them at zero)
        const float m_new = need ? mx : m_used;
        const float f = need ? (m_used == -INFINITY ? 0.f : ex2(m_used - m_new)) : 1.f;
        rescale_o(tO, f);
        l *= f;
        m_used = m_new;
        // the speculative P stores land before their replacements; keys 0..63
        // come back from the first half of S, keys 64..127 are still in r2, r3
        tmem_st_wait();
        tmem_ld32(tS, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld_wait(r0);
        tmem_ld_wait(r1);
        if (masked) {
          mask32(r0, 0, lo_rel, hi_rel);
          mask32(r1, 32, lo_rel, hi_rel);
        }
        neg_m = m_used == -INFINITY ? 0.f : -m_used;
        nm = f2(neg_m, neg_m);
        acc[0] = acc[1] = 0ull;
        exp32(r0, cc, nm, pk0, acc);
        exp32(r1, cc, nm, pk0 + 16, acc);
        tmem_st32(tS + 64, pk0);
        exp32(r2, cc, nm, pk1, acc);
        exp32(r3, cc, nm, pk1 + 16, acc);
        tmem_st32(tS + 96, pk1);
      }
      float a0, a1, b0, b1;
      unf2(acc[0], a0, a1);
      unf2(acc[1], b0, b1);
      l += (a0 + a1) + (b0 + b1);
      // P (and a rescaled O) are in tensor memory: one arrival per warp
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane_id() == 0) mbar_arrive_cluster(bp);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_o), 0, wc));
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      __nv_bfloat16* orow = p.O + size_t(qi) * p.d + h * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait(o);
        if (qi < p.L && head_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float* f = reinterpret_cast<const float*>(o + 8 * i);
            dst[i] = make_uint4(pack_bf16x2(f[0] * inv_l, f[1] * inv_l),
                                pack_bf16x2(f[2] * inv_l, f[3] * inv_l),
                                pack_bf16x2(f[4] * inv_l, f[5] * inv_l),
                                pack_bf16x2(f[6] * inv_l, f[7] * inv_l));
          }
        }
      }
      if (p.lse != nullptr && qi < p.L && head_ok)
        p.lse[size_t(h) * p.L + qi] = (m_used + __log2f(l)) * 0.69314718055994531f;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // neither CTA leaves while the other may still signal it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& a, const DevCtx& ctx, cudaStream_t st) {
  const int d = a.H * 128;
  // Q and V in 128-row boxes, K in 64-row boxes (each CTA of a pair holds 64 keys)
  CUtensorMap tm, tmk, tm8, tm8k;
  if (!make_tmap_bf16_2d(&tm, a.qkv, a.L, 3 * d, 3 * d, 128, 64)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16_2d(&tmk, a.qkv, a.L, 3 * d, 3 * d, 64, 64)) return cudaErrorInvalidValue;
  if (a.fp8) {
    if (a.n_seg != 0 || a.qk8 == nullptr || a.sq == nullptr || a.sk == nullptr)
      return cudaErrorInvalidValue;
    if (!make_tmap_u8_2d(&tm8, a.qk8, a.L, 2 * d, 2 * d, 128)) return cudaErrorInvalidValue;
    if (!make_tmap_u8_2d(&tm8k, a.qk8, a.L, 2 * d, 2 * d, 64)) return cudaErrorInvalidValue;
  } else {
    tm8 = tm;   // unused
    tm8k = tmk;
  }
  AttnDev p{};
  p.O = static_cast<__nv_bfloat16*>(a.O);
  p.lse = a.lse;
  p.L = a.L;
  p.H = a.H;
  p.d = d;
  p.causal = a.causal;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.num_quads = (a.L + 511) / 512;
  p.status = ctx.status;
  p.wait_ns = ctx.wait_ns;
  p.n_seg = a.n_seg;
  for (int i = 0; i <= a.n_seg && a.cu_seqlens; ++i) p.cu[i] = a.cu_seqlens[i];
  p.sq = a.sq;
  p.sk = a.sk;
  p.nkb = (a.L + 127) / 128;
  auto kernel = a.fp8 ? attn_fwd_kernel<true> : attn_fwd_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(2LL * p.num_quads * a.H));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, tm, tmk, tm8, tm8k, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace h3
