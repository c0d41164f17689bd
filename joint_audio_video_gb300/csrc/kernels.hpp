// Internal launch interface between the C ABI (h3attn_api.cu) and the kernels.
// Every launcher returns the launch's cudaError_t; arguments are validated by
// the caller before any launcher runs.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace h3 {

struct DevCtx {
  int* status;          // device status word
  uint64_t wait_ns;     // bound on every in-kernel wait
  int num_sms;
};

// Per-pair rotary table: pair k of a head covers dims (2k, 2k+1).
struct RopeTable {
  float inv_freq[64];   // base^(-2j/n_a), computed in double, rounded once
  int32_t axis[64];     // 0 = t, 1 = h, 2 = w
};

// Fills `rt` for sections sec[0..2] (even, summing to 128) and `base`.
void make_rope_table(RopeTable* rt, const int32_t sec[3], double base);

cudaError_t launch_adaln_modulate(const void* x, const uint8_t* mod, const float* shift,
                                  const float* scale, int L, int d, int n_mod, float eps, void* y,
                                  const DevCtx& ctx, cudaStream_t st);

cudaError_t launch_mrope(void* qkv, const int32_t* pos, int L, int n_heads, const RopeTable& rt,
                         const DevCtx& ctx, cudaStream_t st);

enum GemmEpilogue : int { EPI_PLAIN = 0, EPI_ROPE = 1, EPI_GATED_RESIDUAL = 2, EPI_GELU = 3 };

struct GemmArgs {
  const void* A;        // [M][K] bf16, row-major
  const void* B;        // [N][K] bf16, row-major (nn.Linear weight)
  void* C;              // [M][N] bf16
  int M, N, K;
  int epilogue;         // GemmEpilogue
  // EPI_ROPE: Q block = columns [0, d), K block = [d, 2d); V untouched
  const int32_t* pos;   // [M][3]
  int d;
  const RopeTable* rope;
  // EPI_GATED_RESIDUAL: C = x_res + gate[mod] * (A B^T)
  const void* x_res;    // [M][N] bf16
  const uint8_t* mod;   // [M]
  const float* gate;    // [n_mod][N]
  int n_mod;
  // fp8 operands: A and B are E4M3 bytes; acc is scaled by a_scale[row] * b_scale[col]
  int fp8;
  const float* a_scale; // [M]
  const float* b_scale; // [N]
};

cudaError_t launch_gemm(const GemmArgs& a, const DevCtx& ctx, cudaStream_t st);

constexpr int kMaxSegments = 64;

struct AttnArgs {
  const void* qkv;      // [L][3*H*128] bf16
  void* O;              // [L][H*128] bf16
  float* lse;           // [H][L] or nullptr
  int L, H;
  int causal;
  float sm_scale;
  int n_seg;                  // 0: one segment [0, L)
  const int32_t* cu_seqlens;  // host array [n_seg + 1], validated, n_seg <= kMaxSegments
  // E4M3 scores (n_seg == 0 only): Q and K from qk8 [L][2*H*128] bytes (Q | K),
  // sq [H][L] per-token Q scales, sk [H][ceil(L/128)] per-key-block K scales;
  // V is still read as bf16 from qkv.
  int fp8 = 0;
  const void* qk8 = nullptr;
  const float* sq = nullptr;
  const float* sk = nullptr;
};

cudaError_t launch_attention(const AttnArgs& a, const DevCtx& ctx, cudaStream_t st);

// Row-wise E4M3 quantisation: q[r] = RN(x[r] / s[r]) with s[r] = max|x[r]| / 448.
// E4M3 Q and K for the fp8 scores: per-token Q scale, per-128-key-block K scale.
cudaError_t launch_quantize_qk(const void* qkv, int L, int H, void* qk8, float* sq, float* sk,
                               const DevCtx& ctx, cudaStream_t st);
cudaError_t launch_quantize_rows(const void* x, int R, int K, void* q, float* scale,
                                 const DevCtx& ctx, cudaStream_t st);

// Per-modality noise levels of one denoising step (host-validated).
struct DenoiseParams {
  float sigma[256];
  float sigma_next[256];
  uint8_t update[256];   // 1: the modality is a denoised latent; 0: a condition
};

cudaError_t launch_denoise(float* z, float* x0, const void* v_h3, const uint8_t* mod,
                           const uint8_t* anchor, const float* z_anchor, int L, int C, int n_mod,
                           const DenoiseParams& dp, const DevCtx& ctx, cudaStream_t st);

cudaError_t launch_wait_selftest(const DevCtx& ctx, cudaStream_t st);

}  // namespace h3
