// C ABI of the joint audio-video attention sub-block (include/h3attn.h).
//
// Every entry point validates its arguments on the host and returns an
// h3_status before anything is launched; launches go to the caller's stream.
// Kernels report asynchronous problems (bounded wait ran out, modality id out
// of range) through one status word per device, read by h3_sync_status().
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "../../include/h3attn.h"
#include "kernels.hpp"
#include "ptx.cuh"

namespace h3 {

__device__ int g_status_word;

namespace {

constexpr uint64_t kDefaultWaitNs = 2000000000ull;
constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

// Per device: the status word's device address and the SM count, looked up
// once and kept (a cudaDeviceReset() while the library is loaded is not
// supported: the address would point into the destroyed context).
struct DevInfo {
  std::atomic<int> ready{0};
  int* status = nullptr;
  int num_sms = 0;
};
DevInfo g_dev[kMaxDevices];

h3_status dev_ctx(DevCtx* ctx) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return H3_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return H3_ERR_UNSUPPORTED;
  DevInfo& di = g_dev[dev];
  if (!di.ready.load(std::memory_order_acquire)) {
    void* p = nullptr;
    int sms = 0;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return H3_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return H3_ERR_CUDA;
    di.status = static_cast<int*>(p);
    di.num_sms = sms;
    di.ready.store(1, std::memory_order_release);
  }
  ctx->status = di.status;
  ctx->num_sms = di.num_sms;
  ctx->wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  return H3_OK;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

bool valid_d(int32_t d) { return d >= 128 && d <= 16384 && d % 128 == 0; }
// head counts of 128-wide heads that give a valid d (checked before any
// multiplication, so a huge count cannot wrap around to a valid width)
bool valid_heads(int32_t n_heads) { return n_heads >= 1 && n_heads <= 16384 / 128; }

h3_status launched(cudaError_t e) { return e == cudaSuccess ? H3_OK : H3_ERR_CUDA; }

// An NVTX range named after the entry point around its host-side work, so a
// timeline tool shows which call enqueued which kernels.
struct Trace {
  explicit Trace(const char* name) { nvtxRangePushA(name); }
  ~Trace() { nvtxRangePop(); }
  Trace(const Trace&) = delete;
  Trace& operator=(const Trace&) = delete;
};

// H3_DEBUG_SYNC=1 (read once per process): every entry point that launches
// work waits for its stream before returning and returns the device status,
// so an asynchronous fault or a kernel-reported error (timeout, bad modality
// id) surfaces at the call that caused it.  A stream that is being captured
// is not waited on.
bool debug_sync() {
  static const bool on = [] {
    const char* e = std::getenv("H3_DEBUG_SYNC");
    return e != nullptr && e[0] == '1' && e[1] == '\0';
  }();
  return on;
}

}  // namespace
}  // namespace h3

extern "C" h3_status h3_sync_status(h3_stream_t stream);

namespace h3 {
namespace {

h3_status finish(h3_status s, h3_stream_t stream) {
  if (s != H3_OK || !debug_sync()) return s;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cap) != cudaSuccess)
    return H3_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return s;
  return h3_sync_status(stream);
}

h3_status check_rope(const int32_t sec[3], int32_t head_dim, float base) {
  if (sec == nullptr) return H3_ERR_INVALID_ARG;
  int sum = 0;
  for (int a = 0; a < 3; ++a) {
    if (sec[a] < 0 || sec[a] % 2 != 0) return H3_ERR_INVALID_ARG;
    sum += sec[a];
  }
  if (sum != head_dim) return H3_ERR_INVALID_ARG;
  if (!(base > 0.f) || !std::isfinite(base)) return H3_ERR_INVALID_ARG;
  return H3_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// cu_seqlens: host array, 0 = c_0 <= c_1 <= ... <= c_n = L, 1 <= n <= kMaxSegments.
h3_status check_segments(const int32_t* cu, int32_t n_seg, int32_t L) {
  if (n_seg < 1 || n_seg > kMaxSegments || cu == nullptr) return H3_ERR_INVALID_ARG;
  if (cu[0] != 0 || cu[n_seg] != L) return H3_ERR_INVALID_ARG;
  for (int s = 0; s < n_seg; ++s)
    if (cu[s + 1] < cu[s]) return H3_ERR_INVALID_ARG;
  return H3_OK;
}

// ------------------------------------------------------------------ self-test kernel
__global__ void wait_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  const WaitCtx wc{&abort_flag, status, limit_ns};
  // nothing ever arrives on `bar`: the wait must run out and record a timeout
  mbar_wait(smem_u32(&bar), 0, wc);
}

}  // namespace

// One-element target of the bounds self-test.
__device__ int g_selftest_cell;

// One thread addresses element `i` of the one-element g_selftest_cell through
// the checked path: with i >= 1 the access is skipped and the status word
// records H3_DEV_OUT_OF_BOUNDS (checked build only; the normal build never
// launches it).
__global__ void bounds_selftest_kernel(int i, int* status) {
  int* cell = &g_selftest_cell;
  if (H3_IN(i >= 0 && i < 1, status)) cell[i] = 1;
}

cudaError_t launch_wait_selftest(const DevCtx& ctx, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(ctx.status, ctx.wait_ns);
  return cudaGetLastError();
}

}  // namespace h3

using namespace h3;

extern "C" {

const char* h3_status_string(h3_status s) {
  switch (s) {
    case H3_OK: return "ok";
    case H3_ERR_INVALID_ARG: return "invalid argument (nothing launched)";
    case H3_ERR_UNSUPPORTED: return "unsupported shape or option (nothing launched)";
    case H3_ERR_CUDA: return "CUDA runtime error";
    case H3_ERR_TIMEOUT: return "a kernel gave up on a bounded wait";
    case H3_ERR_BAD_INDEX: return "modality id out of range";
    case H3_ERR_WORKSPACE: return "workspace too small";
    case H3_ERR_OUT_OF_BOUNDS: return "a kernel index fell outside its buffer (checked build)";
    default: return "unknown status";
  }
}

const char* h3_version(void) { return "h3attn 0.1.0 sm_103a"; }

void h3_set_wait_limit_ns(uint64_t limit_ns) {
  g_wait_ns.store(limit_ns == 0 ? kDefaultWaitNs : limit_ns, std::memory_order_relaxed);
}

h3_status h3_adaln_modulate(const uint16_t* x, const uint8_t* mod, const float* shift,
                            const float* scale, int32_t L, int32_t d, int32_t n_mod, float eps,
                            uint16_t* y, h3_stream_t stream) {
  const Trace trace_("h3_adaln_modulate");
  if (L < 1 || !valid_d(d) || n_mod < 1 || n_mod > 255) return H3_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return H3_ERR_INVALID_ARG;
  if (!aligned16(x) || mod == nullptr || !aligned16(shift) || !aligned16(scale) || !aligned16(y))
    return H3_ERR_INVALID_ARG;
  const size_t bytes = size_t(L) * d * 2;
  if (x != y && overlap(x, bytes, y, bytes)) return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  return finish(launched(launch_adaln_modulate(x, mod, shift, scale, L, d, n_mod, eps, y, ctx,
                                        reinterpret_cast<cudaStream_t>(stream))), stream);
}

h3_status h3_qkv_proj(const uint16_t* y, const uint16_t* Wqkv, int32_t L, int32_t d, uint16_t* qkv,
                      h3_stream_t stream) {
  const Trace trace_("h3_qkv_proj");
  if (L < 1 || !valid_d(d)) return H3_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(Wqkv) || !aligned16(qkv)) return H3_ERR_INVALID_ARG;
  if (overlap(y, size_t(L) * d * 2, qkv, size_t(L) * 3 * d * 2)) return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  GemmArgs a{};
  a.A = y;
  a.B = Wqkv;
  a.C = qkv;
  a.M = L;
  a.N = 3 * d;
  a.K = d;
  a.epilogue = EPI_PLAIN;
  return finish(launched(launch_gemm(a, ctx, reinterpret_cast<cudaStream_t>(stream))),
                stream);
}

h3_status h3_mrope_apply(uint16_t* qkv, const int32_t* pos, int32_t L, int32_t n_heads,
                         int32_t head_dim, const int32_t sec[3], float base, h3_stream_t stream) {
  const Trace trace_("h3_mrope_apply");
  if (L < 1 || n_heads < 1) return H3_ERR_INVALID_ARG;
  if (head_dim != 128) return H3_ERR_UNSUPPORTED;
  if (!valid_heads(n_heads)) return H3_ERR_INVALID_ARG;
  if (h3_status s = check_rope(sec, head_dim, base)) return s;
  if (!aligned16(qkv) || pos == nullptr || (reinterpret_cast<uintptr_t>(pos) & 3u))
    return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  RopeTable rt;
  make_rope_table(&rt, sec, base);
  return finish(launched(launch_mrope(qkv, pos, L, n_heads, rt, ctx,
                                      reinterpret_cast<cudaStream_t>(stream))),
                stream);
}

h3_status h3_joint_attn_fwd(const uint16_t* qkv, int32_t L, int32_t n_heads, int32_t head_dim,
                            int32_t causal, float sm_scale, uint16_t* O, float* lse,
                            h3_stream_t stream) {
  const Trace trace_("h3_joint_attn_fwd");
  if (L < 1 || n_heads < 1) return H3_ERR_INVALID_ARG;
  if (head_dim != 128) return H3_ERR_UNSUPPORTED;
  if (!valid_heads(n_heads)) return H3_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return H3_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return H3_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(O)) return H3_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return H3_ERR_INVALID_ARG;
  const size_t d = size_t(n_heads) * 128;
  if (overlap(qkv, size_t(L) * 3 * d * 2, O, size_t(L) * d * 2)) return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  AttnArgs a{};
  a.qkv = qkv;
  a.O = O;
  a.lse = lse;
  a.L = L;
  a.H = n_heads;
  a.causal = causal;
  a.sm_scale = sm_scale;
  return finish(launched(launch_attention(a, ctx, reinterpret_cast<cudaStream_t>(stream))),
                stream);
}

h3_status h3_joint_attn_varlen_fwd(const uint16_t* qkv, const int32_t* cu_seqlens,
                                   int32_t n_seg, int32_t L, int32_t n_heads, int32_t head_dim,
                                   int32_t causal, float sm_scale, uint16_t* O, float* lse,
                                   h3_stream_t stream) {
  const Trace trace_("h3_joint_attn_varlen_fwd");
  if (L < 1 || n_heads < 1) return H3_ERR_INVALID_ARG;
  if (head_dim != 128) return H3_ERR_UNSUPPORTED;
  if (!valid_heads(n_heads)) return H3_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return H3_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return H3_ERR_INVALID_ARG;
  if (h3_status s = check_segments(cu_seqlens, n_seg, L)) return s;
  if (!aligned16(qkv) || !aligned16(O)) return H3_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return H3_ERR_INVALID_ARG;
  const size_t d = size_t(n_heads) * 128;
  if (overlap(qkv, size_t(L) * 3 * d * 2, O, size_t(L) * d * 2)) return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  AttnArgs a{};
  a.qkv = qkv;
  a.O = O;
  a.lse = lse;
  a.L = L;
  a.H = n_heads;
  a.causal = causal;
  a.sm_scale = sm_scale;
  a.n_seg = n_seg;
  a.cu_seqlens = cu_seqlens;
  return finish(launched(launch_attention(a, ctx, reinterpret_cast<cudaStream_t>(stream))),
                stream);
}

// Workspace of the fp8-score attention: qk8 [L][2d] bytes | sq [H][L] | sk [H][nkb].
static size_t attn_fp8_bytes(size_t L, size_t H) {
  const size_t d = H * 128, nkb = (L + 127) / 128;
  return round256(L * 2 * d) + round256(H * L * 4) + round256(H * nkb * 4);
}

h3_status h3_attn_workspace_size_fp8(int32_t L, int32_t n_heads, int32_t head_dim,
                                     size_t* bytes) {
  if (bytes == nullptr || L < 1 || n_heads < 1) return H3_ERR_INVALID_ARG;
  if (head_dim != 128) return H3_ERR_UNSUPPORTED;
  if (!valid_heads(n_heads)) return H3_ERR_INVALID_ARG;
  *bytes = attn_fp8_bytes(size_t(L), size_t(n_heads));
  return H3_OK;
}

h3_status h3_quantize_qk_fp8(const uint16_t* qkv, int32_t L, int32_t n_heads, int32_t head_dim,
                             uint8_t* qk8, float* sq, float* sk, h3_stream_t stream) {
  const Trace trace_("h3_quantize_qk_fp8");
  if (L < 1 || n_heads < 1) return H3_ERR_INVALID_ARG;
  if (head_dim != 128) return H3_ERR_UNSUPPORTED;
  if (!valid_heads(n_heads)) return H3_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(qk8) || sq == nullptr || sk == nullptr ||
      (reinterpret_cast<uintptr_t>(sq) & 3u) || (reinterpret_cast<uintptr_t>(sk) & 3u))
    return H3_ERR_INVALID_ARG;
  const size_t d = size_t(n_heads) * 128, nkb = (size_t(L) + 127) / 128;
  const size_t qkv_b = size_t(L) * 3 * d * 2;
  if (overlap(qkv, qkv_b, qk8, size_t(L) * 2 * d) ||
      overlap(qkv, qkv_b, sq, size_t(n_heads) * L * 4) ||
      overlap(qkv, qkv_b, sk, size_t(n_heads) * nkb * 4))
    return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  return finish(launched(launch_quantize_qk(qkv, L, n_heads, qk8, sq, sk, ctx,
                                     reinterpret_cast<cudaStream_t>(stream))), stream);
}

h3_status h3_joint_attn_fwd_fp8(const uint16_t* qkv, int32_t L, int32_t n_heads,
                                int32_t head_dim, int32_t causal, float sm_scale,
                                void* workspace, size_t workspace_bytes, uint16_t* O, float* lse,
                                h3_stream_t stream) {
  const Trace trace_("h3_joint_attn_fwd_fp8");
  if (L < 1 || n_heads < 1) return H3_ERR_INVALID_ARG;
  if (head_dim != 128) return H3_ERR_UNSUPPORTED;
  if (!valid_heads(n_heads)) return H3_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return H3_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return H3_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(O) || workspace == nullptr ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return H3_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return H3_ERR_INVALID_ARG;
  const size_t need = attn_fp8_bytes(size_t(L), size_t(n_heads));
  if (workspace_bytes < need) return H3_ERR_WORKSPACE;
  const size_t d = size_t(n_heads) * 128;
  const size_t qkv_b = size_t(L) * 3 * d * 2, o_b = size_t(L) * d * 2;
  if (overlap(qkv, qkv_b, O, o_b) || overlap(workspace, need, qkv, qkv_b) ||
      overlap(workspace, need, O, o_b) ||
      (lse != nullptr && overlap(workspace, need, lse, size_t(n_heads) * L * 4)))
    return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* qk8 = ws;
  float* sq = reinterpret_cast<float*>(ws + round256(size_t(L) * 2 * d));
  float* sk = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sq) + round256(size_t(n_heads) * L * 4));
  if (launch_quantize_qk(qkv, L, n_heads, qk8, sq, sk, ctx, st) != cudaSuccess) return H3_ERR_CUDA;
  AttnArgs a{};
  a.qkv = qkv;
  a.O = O;
  a.lse = lse;
  a.L = L;
  a.H = n_heads;
  a.causal = causal;
  a.sm_scale = sm_scale;
  a.fp8 = 1;
  a.qk8 = qk8;
  a.sq = sq;
  a.sk = sk;
  return finish(launched(launch_attention(a, ctx, st)), stream);
}

h3_status h3_out_proj_gated_residual(const uint16_t* O, const uint16_t* Wo,
                                     const uint16_t* x_res, const uint8_t* mod,
                                     const float* gate, int32_t L, int32_t d, int32_t n_mod,
                                     uint16_t* out, h3_stream_t stream) {
  const Trace trace_("h3_out_proj_gated_residual");
  if (L < 1 || !valid_d(d) || n_mod < 1 || n_mod > 255) return H3_ERR_INVALID_ARG;
  if (!aligned16(O) || !aligned16(Wo) || !aligned16(x_res) || mod == nullptr ||
      !aligned16(gate) || !aligned16(out))
    return H3_ERR_INVALID_ARG;
  const size_t bytes = size_t(L) * d * 2;
  if (overlap(O, bytes, out, bytes)) return H3_ERR_INVALID_ARG;
  if (x_res != out && overlap(x_res, bytes, out, bytes)) return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  GemmArgs a{};
  a.A = O;
  a.B = Wo;
  a.C = out;
  a.M = L;
  a.N = d;
  a.K = d;
  a.epilogue = EPI_GATED_RESIDUAL;
  a.x_res = x_res;
  a.mod = mod;
  a.gate = gate;
  a.n_mod = n_mod;
  return finish(launched(launch_gemm(a, ctx, reinterpret_cast<cudaStream_t>(stream))),
                stream);
}

h3_status h3_denoise_step(float* z, float* x0, const uint16_t* v_h3, const uint8_t* mod,
                          const uint8_t* anchor, const float* z_anchor, int32_t L, int32_t C,
                          int32_t n_mod, const float* sigma, const float* sigma_next,
                          const uint8_t* update, h3_stream_t stream) {
  const Trace trace_("h3_denoise_step");
  if (L < 1 || C < 4 || C % 4 != 0 || n_mod < 1 || n_mod > 255) return H3_ERR_INVALID_ARG;
  if (!aligned16(z) || !aligned16(v_h3) || mod == nullptr) return H3_ERR_INVALID_ARG;
  if (x0 != nullptr && !aligned16(x0)) return H3_ERR_INVALID_ARG;
  if (anchor != nullptr && !aligned16(z_anchor)) return H3_ERR_INVALID_ARG;
  if (sigma == nullptr || sigma_next == nullptr || update == nullptr) return H3_ERR_INVALID_ARG;
  const size_t n = size_t(L) * C;
  if (x0 != nullptr && overlap(z, n * 4, x0, n * 4)) return H3_ERR_INVALID_ARG;
  DenoiseParams dp{};
  for (int m = 0; m < n_mod; ++m) {
    if (!(sigma[m] >= 0.f && sigma[m] <= 1.f) || !(sigma_next[m] >= 0.f && sigma_next[m] <= 1.f))
      return H3_ERR_INVALID_ARG;
    dp.sigma[m] = sigma[m];
    dp.sigma_next[m] = sigma_next[m];
    dp.update[m] = update[m] ? 1 : 0;
  }
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  return finish(launched(launch_denoise(z, x0, v_h3, mod, anchor, z_anchor, L, C, n_mod, dp, ctx,
                                 reinterpret_cast<cudaStream_t>(stream))), stream);
}

static h3_status check_mlp(const h3_mlp_desc* desc) {
  if (desc == nullptr) return H3_ERR_INVALID_ARG;
  if (desc->L < 1 || !valid_d(desc->d) || desc->n_mod < 1 || desc->n_mod > 255)
    return H3_ERR_INVALID_ARG;
  if (desc->hidden < 128 || desc->hidden % 128 != 0 || desc->hidden > 65536)
    return H3_ERR_INVALID_ARG;
  if (!(desc->ln_eps >= 0.f) || !std::isfinite(desc->ln_eps)) return H3_ERR_INVALID_ARG;
  return H3_OK;
}

h3_status h3_mlp_workspace_size(const h3_mlp_desc* desc, size_t* bytes) {
  if (bytes == nullptr) return H3_ERR_INVALID_ARG;
  if (h3_status s = check_mlp(desc)) return s;
  const size_t L = size_t(desc->L);
  *bytes = round256(L * desc->d * 2) + round256(L * size_t(desc->hidden) * 2);
  return H3_OK;
}

h3_status h3_mlp_block_fwd(const h3_mlp_desc* desc, const uint16_t* x, const uint8_t* mod,
                           const float* shift, const float* scale, const float* gate,
                           const uint16_t* W1, const uint16_t* W2, void* workspace,
                           size_t workspace_bytes, uint16_t* out, h3_stream_t stream) {
  const Trace trace_("h3_mlp_block_fwd");
  size_t need = 0;
  if (h3_status s = h3_mlp_workspace_size(desc, &need)) return s;
  if (!aligned16(x) || mod == nullptr || !aligned16(shift) || !aligned16(scale) ||
      !aligned16(gate) || !aligned16(W1) || !aligned16(W2) || !aligned16(out) ||
      workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return H3_ERR_INVALID_ARG;
  if (workspace_bytes < need) return H3_ERR_WORKSPACE;
  const size_t L = size_t(desc->L), d = size_t(desc->d);
  if (x != out && overlap(x, L * d * 2, out, L * d * 2)) return H3_ERR_INVALID_ARG;
  if (overlap(workspace, need, x, L * d * 2) || overlap(workspace, need, out, L * d * 2))
    return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* y = ws;
  void* hbuf = ws + round256(L * d * 2);
  if (launch_adaln_modulate(x, mod, shift, scale, desc->L, desc->d, desc->n_mod, desc->ln_eps, y,
                            ctx, st) != cudaSuccess)
    return H3_ERR_CUDA;
  GemmArgs up{};
  up.A = y;
  up.B = W1;
  up.C = hbuf;
  up.M = desc->L;
  up.N = desc->hidden;
  up.K = desc->d;
  up.epilogue = EPI_GELU;
  if (launch_gemm(up, ctx, st) != cudaSuccess) return H3_ERR_CUDA;
  GemmArgs down{};
  down.A = hbuf;
  down.B = W2;
  down.C = out;
  down.M = desc->L;
  down.N = desc->d;
  down.K = desc->hidden;
  down.epilogue = EPI_GATED_RESIDUAL;
  down.x_res = x;
  down.mod = mod;
  down.gate = gate;
  down.n_mod = desc->n_mod;
  if (launch_gemm(down, ctx, st) != cudaSuccess) return H3_ERR_CUDA;
  return finish(H3_OK, stream);
}

h3_status h3_quantize_rows_fp8(const uint16_t* x, int32_t R, int32_t K, uint8_t* q, float* scale,
                               h3_stream_t stream) {
  const Trace trace_("h3_quantize_rows_fp8");
  if (R < 1 || K < 16 || K % 16 != 0) return H3_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || scale == nullptr ||
      (reinterpret_cast<uintptr_t>(scale) & 3u))
    return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  return finish(launched(launch_quantize_rows(x, R, K, q, scale, ctx,
                                       reinterpret_cast<cudaStream_t>(stream))), stream);
}

h3_status h3_gemm_fp8(const uint8_t* A, const float* a_scale, const uint8_t* B,
                      const float* b_scale, int32_t M, int32_t N, int32_t K, uint16_t* C,
                      h3_stream_t stream) {
  const Trace trace_("h3_gemm_fp8");
  if (M < 1 || N < 128 || N % 128 != 0 || K < 128 || K % 128 != 0) return H3_ERR_INVALID_ARG;
  // the kernels count output tiles (at least 128 x 128) in 32-bit integers
  if ((int64_t(M) + 127) / 128 * (int64_t(N) / 128) > INT32_MAX) return H3_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || !aligned16(a_scale) ||
      !aligned16(b_scale))
    return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  GemmArgs g{};
  g.A = A;
  g.B = B;
  g.C = C;
  g.M = M;
  g.N = N;
  g.K = K;
  g.epilogue = EPI_PLAIN;
  g.fp8 = 1;
  g.a_scale = a_scale;
  g.b_scale = b_scale;
  return finish(launched(launch_gemm(g, ctx, reinterpret_cast<cudaStream_t>(stream))),
                stream);
}

static h3_status check_desc(const h3_block_desc* desc);

h3_status h3_workspace_size_fp8(const h3_block_desc* desc, size_t* bytes) {
  if (bytes == nullptr) return H3_ERR_INVALID_ARG;
  if (h3_status s = check_desc(desc)) return s;
  const size_t L = size_t(desc->L), d = size_t(desc->d);
  *bytes = round256(L * d * 2) + round256(L * 3 * d * 2) + round256(L * d) + round256(L * 4);
  if (desc->n_seg == 0) *bytes += attn_fp8_bytes(L, size_t(desc->n_heads));
  return H3_OK;
}

h3_status h3_attn_block_fwd_fp8(const h3_block_desc* desc, const uint16_t* x, const uint8_t* mod,
                                const int32_t* pos, const float* shift, const float* scale,
                                const float* gate, const uint8_t* Wqkv_q, const float* Wqkv_s,
                                const uint8_t* Wo_q, const float* Wo_s, void* workspace,
                                size_t workspace_bytes, uint16_t* out, h3_stream_t stream) {
  const Trace trace_("h3_attn_block_fwd_fp8");
  size_t need = 0;
  if (h3_status s = h3_workspace_size_fp8(desc, &need)) return s;
  if (!aligned16(x) || mod == nullptr || pos == nullptr || (reinterpret_cast<uintptr_t>(pos) & 3u) ||
      !aligned16(shift) || !aligned16(scale) || !aligned16(gate) || !aligned16(Wqkv_q) ||
      !aligned16(Wqkv_s) || !aligned16(Wo_q) || !aligned16(Wo_s) || !aligned16(out) ||
      workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return H3_ERR_INVALID_ARG;
  if (workspace_bytes < need) return H3_ERR_WORKSPACE;
  const size_t L = size_t(desc->L), d = size_t(desc->d);
  if (x != out && overlap(x, L * d * 2, out, L * d * 2)) return H3_ERR_INVALID_ARG;
  if (overlap(workspace, need, x, L * d * 2) || overlap(workspace, need, out, L * d * 2))
    return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* y = ws;                                        // y, then O
  void* qkv = ws + round256(L * d * 2);
  void* q8 = ws + round256(L * d * 2) + round256(L * 3 * d * 2);
  float* s8 = reinterpret_cast<float*>(static_cast<uint8_t*>(q8) + round256(L * d));
  const int Li = desc->L, di = desc->d;
  if (launch_adaln_modulate(x, mod, shift, scale, Li, di, desc->n_mod, desc->ln_eps, y, ctx, st) !=
          cudaSuccess ||
      launch_quantize_rows(y, Li, di, q8, s8, ctx, st) != cudaSuccess)
    return H3_ERR_CUDA;
  RopeTable rt;
  make_rope_table(&rt, desc->rope_sec, desc->rope_base);
  GemmArgs g{};
  g.A = q8;
  g.B = Wqkv_q;
  g.C = qkv;
  g.M = Li;
  g.N = 3 * di;
  g.K = di;
  g.epilogue = EPI_ROPE;
  g.pos = pos;
  g.d = di;
  g.rope = &rt;
  g.fp8 = 1;
  g.a_scale = s8;
  g.b_scale = Wqkv_s;
  if (launch_gemm(g, ctx, st) != cudaSuccess) return H3_ERR_CUDA;
  AttnArgs a{};
  a.qkv = qkv;
  a.O = y;
  a.L = Li;
  a.H = desc->n_heads;
  a.causal = desc->causal;
  a.sm_scale = 1.0f / std::sqrt(float(desc->head_dim));
  a.n_seg = desc->n_seg;
  a.cu_seqlens = desc->cu_seqlens;
  if (desc->n_seg == 0) {   // E4M3 scores; per-segment attention stays bf16
    uint8_t* qk8 = static_cast<uint8_t*>(q8) + round256(L * d) + round256(L * 4);
    float* sq = reinterpret_cast<float*>(qk8 + round256(L * 2 * d));
    float* sk = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sq) +
                                         round256(size_t(desc->n_heads) * L * 4));
    if (launch_quantize_qk(qkv, Li, desc->n_heads, qk8, sq, sk, ctx, st) != cudaSuccess)
      return H3_ERR_CUDA;
    a.fp8 = 1;
    a.qk8 = qk8;
    a.sq = sq;
    a.sk = sk;
  }
  if (launch_attention(a, ctx, st) != cudaSuccess ||
      launch_quantize_rows(y, Li, di, q8, s8, ctx, st) != cudaSuccess)
    return H3_ERR_CUDA;
  GemmArgs o{};
  o.A = q8;
  o.B = Wo_q;
  o.C = out;
  o.M = Li;
  o.N = di;
  o.K = di;
  o.epilogue = EPI_GATED_RESIDUAL;
  o.x_res = x;
  o.mod = mod;
  o.gate = gate;
  o.n_mod = desc->n_mod;
  o.fp8 = 1;
  o.a_scale = s8;
  o.b_scale = Wo_s;
  return finish(launched(launch_gemm(o, ctx, st)), stream);
}

static h3_status check_mlp(const h3_mlp_desc* desc);

h3_status h3_mlp_workspace_size_fp8(const h3_mlp_desc* desc, size_t* bytes) {
  if (bytes == nullptr) return H3_ERR_INVALID_ARG;
  if (h3_status s = check_mlp(desc)) return s;
  const size_t L = size_t(desc->L), d = size_t(desc->d), hid = size_t(desc->hidden);
  *bytes = round256(L * d * 2) + round256(L * hid * 2) + round256(L * hid) + round256(L * 4);
  return H3_OK;
}

h3_status h3_mlp_block_fwd_fp8(const h3_mlp_desc* desc, const uint16_t* x, const uint8_t* mod,
                               const float* shift, const float* scale, const float* gate,
                               const uint8_t* W1_q, const float* W1_s, const uint8_t* W2_q,
                               const float* W2_s, void* workspace, size_t workspace_bytes,
                               uint16_t* out, h3_stream_t stream) {
  const Trace trace_("h3_mlp_block_fwd_fp8");
  size_t need = 0;
  if (h3_status s = h3_mlp_workspace_size_fp8(desc, &need)) return s;
  if (!aligned16(x) || mod == nullptr || !aligned16(shift) || !aligned16(scale) ||
      !aligned16(gate) || !aligned16(W1_q) || !aligned16(W1_s) || !aligned16(W2_q) ||
      !aligned16(W2_s) || !aligned16(out) || workspace == nullptr ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return H3_ERR_INVALID_ARG;
  if (workspace_bytes < need) return H3_ERR_WORKSPACE;
  const size_t L = size_t(desc->L), d = size_t(desc->d), hid = size_t(desc->hidden);
  if (x != out && overlap(x, L * d * 2, out, L * d * 2)) return H3_ERR_INVALID_ARG;
  if (overlap(workspace, need, x, L * d * 2) || overlap(workspace, need, out, L * d * 2))
    return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* y = ws;
  void* hbuf = ws + round256(L * d * 2);
  void* q8 = static_cast<uint8_t*>(hbuf) + round256(L * hid * 2);   // y_q, later h_q
  float* s8 = reinterpret_cast<float*>(static_cast<uint8_t*>(q8) + round256(L * hid));
  if (launch_adaln_modulate(x, mod, shift, scale, desc->L, desc->d, desc->n_mod, desc->ln_eps, y,
                            ctx, st) != cudaSuccess ||
      launch_quantize_rows(y, desc->L, desc->d, q8, s8, ctx, st) != cudaSuccess)
    return H3_ERR_CUDA;
  GemmArgs up{};
  up.A = q8;
  up.B = W1_q;
  up.C = hbuf;
  up.M = desc->L;
  up.N = desc->hidden;
  up.K = desc->d;
  up.epilogue = EPI_GELU;
  up.fp8 = 1;
  up.a_scale = s8;
  up.b_scale = W1_s;
  if (launch_gemm(up, ctx, st) != cudaSuccess ||
      launch_quantize_rows(hbuf, desc->L, desc->hidden, q8, s8, ctx, st) != cudaSuccess)
    return H3_ERR_CUDA;
  GemmArgs down{};
  down.A = q8;
  down.B = W2_q;
  down.C = out;
  down.M = desc->L;
  down.N = desc->d;
  down.K = desc->hidden;
  down.epilogue = EPI_GATED_RESIDUAL;
  down.x_res = x;
  down.mod = mod;
  down.gate = gate;
  down.n_mod = desc->n_mod;
  down.fp8 = 1;
  down.a_scale = s8;
  down.b_scale = W2_s;
  return finish(launched(launch_gemm(down, ctx, st)), stream);
}

static h3_status check_desc(const h3_block_desc* desc) {
  if (desc == nullptr) return H3_ERR_INVALID_ARG;
  if (desc->L < 1 || desc->n_heads < 1 || desc->n_mod < 1 || desc->n_mod > 255)
    return H3_ERR_INVALID_ARG;
  if (desc->head_dim != 128) return H3_ERR_UNSUPPORTED;
  if (!valid_heads(desc->n_heads) || desc->d != desc->n_heads * desc->head_dim ||
      !valid_d(desc->d))
    return H3_ERR_INVALID_ARG;
  if (desc->causal != 0 && desc->causal != 1) return H3_ERR_INVALID_ARG;
  if (!(desc->ln_eps >= 0.f) || !std::isfinite(desc->ln_eps)) return H3_ERR_INVALID_ARG;
  if (desc->n_seg != 0) {
    if (h3_status s = check_segments(desc->cu_seqlens, desc->n_seg, desc->L)) return s;
  }
  return check_rope(desc->rope_sec, desc->head_dim, desc->rope_base);
}

h3_status h3_workspace_size(const h3_block_desc* desc, size_t* bytes) {
  if (bytes == nullptr) return H3_ERR_INVALID_ARG;
  if (h3_status s = check_desc(desc)) return s;
  const size_t L = size_t(desc->L), d = size_t(desc->d);
  *bytes = round256(L * d * 2) + round256(L * 3 * d * 2);
  return H3_OK;
}

h3_status h3_attn_block_fwd(const h3_block_desc* desc, const uint16_t* x, const uint8_t* mod,
                            const int32_t* pos, const float* shift, const float* scale,
                            const float* gate, const uint16_t* Wqkv, const uint16_t* Wo,
                            void* workspace, size_t workspace_bytes, uint16_t* out,
                            h3_stream_t stream) {
  const Trace trace_("h3_attn_block_fwd");
  return h3_attn_block_fwd_profiled(desc, x, mod, pos, shift, scale, gate, Wqkv, Wo, workspace,
                                    workspace_bytes, out, stream, nullptr);
}

h3_status h3_attn_block_fwd_profiled(const h3_block_desc* desc, const uint16_t* x,
                                     const uint8_t* mod, const int32_t* pos, const float* shift,
                                     const float* scale, const float* gate, const uint16_t* Wqkv,
                                     const uint16_t* Wo, void* workspace, size_t workspace_bytes,
                                     uint16_t* out, h3_stream_t stream, void* const* events) {
  const Trace trace_("h3_attn_block_fwd_profiled");
  size_t need = 0;
  if (h3_status s = h3_workspace_size(desc, &need)) return s;
  if (!aligned16(x) || mod == nullptr || pos == nullptr || (reinterpret_cast<uintptr_t>(pos) & 3u) ||
      !aligned16(shift) || !aligned16(scale) || !aligned16(gate) || !aligned16(Wqkv) ||
      !aligned16(Wo) || !aligned16(out) || workspace == nullptr ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return H3_ERR_INVALID_ARG;
  if (workspace_bytes < need) return H3_ERR_WORKSPACE;
  const size_t L = size_t(desc->L), d = size_t(desc->d);
  const size_t xbytes = L * d * 2;
  if (x != out && overlap(x, xbytes, out, xbytes)) return H3_ERR_INVALID_ARG;
  if (overlap(workspace, need, x, xbytes) || overlap(workspace, need, out, xbytes))
    return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* y = ws;                              // y, later reused for O
  void* qkv = ws + round256(L * d * 2);
  const int Li = desc->L, di = desc->d;
  auto mark = [&](int i) -> bool {
    return events == nullptr ||
           cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) == cudaSuccess;
  };
  if (!mark(0)) return H3_ERR_CUDA;

  cudaError_t e = launch_adaln_modulate(x, mod, shift, scale, Li, di, desc->n_mod, desc->ln_eps, y,
                                        ctx, st);
  if (e != cudaSuccess || !mark(1)) return H3_ERR_CUDA;

  RopeTable rt;
  make_rope_table(&rt, desc->rope_sec, desc->rope_base);
  GemmArgs g{};
  g.A = y;
  g.B = Wqkv;
  g.C = qkv;
  g.M = Li;
  g.N = 3 * di;
  g.K = di;
  g.epilogue = EPI_ROPE;
  g.pos = pos;
  g.d = di;
  g.rope = &rt;
  if (launch_gemm(g, ctx, st) != cudaSuccess || !mark(2)) return H3_ERR_CUDA;

  AttnArgs a{};
  a.qkv = qkv;
  a.O = y;
  a.lse = nullptr;
  a.L = Li;
  a.H = desc->n_heads;
  a.causal = desc->causal;
  a.sm_scale = 1.0f / std::sqrt(float(desc->head_dim));
  a.n_seg = desc->n_seg;
  a.cu_seqlens = desc->cu_seqlens;
  if (launch_attention(a, ctx, st) != cudaSuccess || !mark(3)) return H3_ERR_CUDA;

  GemmArgs o{};
  o.A = y;
  o.B = Wo;
  o.C = out;
  o.M = Li;
  o.N = di;
  o.K = di;
  o.epilogue = EPI_GATED_RESIDUAL;
  o.x_res = x;
  o.mod = mod;
  o.gate = gate;
  o.n_mod = desc->n_mod;
  if (launch_gemm(o, ctx, st) != cudaSuccess || !mark(4)) return H3_ERR_CUDA;
  return finish(H3_OK, stream);
}

h3_status h3_sync_status(h3_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return H3_ERR_CUDA;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  int v = 0;
  if (cudaMemcpy(&v, ctx.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return H3_ERR_CUDA;
  if (v != H3_DEV_OK && cudaMemset(ctx.status, 0, sizeof(int)) != cudaSuccess) return H3_ERR_CUDA;
  switch (v) {
    case H3_DEV_OK: return H3_OK;
    case H3_DEV_TIMEOUT: return H3_ERR_TIMEOUT;
    case H3_DEV_BAD_INDEX: return H3_ERR_BAD_INDEX;
    case H3_DEV_OUT_OF_BOUNDS: return H3_ERR_OUT_OF_BOUNDS;
    default: return H3_ERR_CUDA;
  }
}

h3_status h3_selftest_wait_timeout(uint64_t limit_ns, h3_stream_t stream) {
  const Trace trace_("h3_selftest_wait_timeout");
  if (limit_ns == 0 || limit_ns > 10000000000ull) return H3_ERR_INVALID_ARG;
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  ctx.wait_ns = limit_ns;
  return finish(launched(launch_wait_selftest(ctx, reinterpret_cast<cudaStream_t>(stream))),
                stream);
}

int32_t h3_checked_build(void) {
#ifdef H3_CHECKED
  return 1;
#else
  return 0;
#endif
}

h3_status h3_selftest_bounds_check(h3_stream_t stream) {
  const Trace trace_("h3_selftest_bounds_check");
#ifdef H3_CHECKED
  DevCtx ctx;
  if (h3_status s = dev_ctx(&ctx)) return s;
  bounds_selftest_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(1, ctx.status);
  return finish(launched(cudaGetLastError()), stream);
#else
  (void)stream;
  return H3_ERR_UNSUPPORTED;
#endif
}

}  // extern "C"
