/*
 * h3attn — C ABI of the GB300 (sm_103a) joint audio-video attention sub-block.
 *
 * One attention sub-block of a single-stream joint audio-video Diffusion
 * Transformer of the MiniMax-H3 kind, run over one packed sequence of text,
 * video and audio tokens:
 *
 *   y   = LN(x) * (1 + scale[mod]) + shift[mod]          h3_adaln_modulate
 *   qkv = y Wqkv^T                                        h3_qkv_proj
 *   Q,K <- 3D (t,h,w) rotary embedding                    h3_mrope_apply
 *   O   = softmax(Q K^T / sqrt(dh) [+ causal]) V          h3_joint_attn_fwd
 *   out = x + gate[mod] * (O Wo^T)                        h3_out_proj_gated_residual
 *   all of the above in one call                          h3_attn_block_fwd
 *
 * Sources (web pages):
 *   [H3-RL] "DiffusionNFT on MiniMax H3: Open-Source RL Training for Joint
 *           Audio-Video Generation", section "MiniMax H3 and Why Joint
 *           Audio-Video Generation Complicates RL Training" (3D multimodal RoPE
 *           over time/height/width; modality-specific AdaLN branches whose
 *           outputs are cacheable) and section "How VeRL-Omni's Adapter
 *           Architecture Keeps H3-Specific Logic Contained" (to_q, to_k, to_v,
 *           to_out.0 projections, fused in the rollout network).
 *   [VeRL]  "多模态强化学习工程解析：VeRL-Omni 架构与 MiniMax-H3 训练实录",
 *           三 目标模型 (shared attention weights and AdaLN modulation across
 *           modalities; causal attention mentioned) and 5.2 LoRA 权重切分不一致
 *           (Q, K, V packed into one matrix for inference).
 *   [vLLM]  "Joint Audio-Video Generation in Production: Architecture Deep Dive
 *           into MiniMax-H3 and vLLM-Omni", §1 Unified Architecture (one shared
 *           attention context over 58,758 tokens, 50 denoising steps), §3 Packed
 *           Sequences and Modality Identity Preservation (tags, positions),
 *           §6 Boundary Trimming for Packed Attention (only the effective
 *           tokens may enter the kernel).
 *
 * Conventions common to every call
 *   - bf16 tensors are passed as uint16_t bit patterns; fp32 as float.
 *   - Matrices are row-major; a row is one token.  Weights use the
 *     nn.Linear layout W[out_features][in_features].
 *   - Every device pointer must be 16-byte aligned and non-NULL (except an
 *     optional output documented as such).  The caller owns every buffer;
 *     no call allocates device memory.
 *   - Every device call is asynchronous on the caller's stream.  Argument
 *     errors are detected on the host before anything is launched.
 *   - L is the exact token count (>= 1); nothing is padded and no token past
 *     L is read as a key (the pages' boundary-trim requirement).
 *   - d % 128 == 0, 128 <= d <= 16384; head_dim must be 128; 1 <= n_mod <= 255.
 *   - A kernel that finds an out-of-range modality id or gives up on a
 *     bounded wait records it in a per-device status word; h3_sync_status()
 *     reports and clears it.  No C++ exception crosses this boundary.
 *   - With H3_DEBUG_SYNC=1 in the environment (read once per process), every
 *     call that launches work waits for its stream before returning and
 *     returns what h3_sync_status() would, so an error surfaces at the call
 *     that caused it; a stream that is being captured is not waited on.
 *   - Every call that launches work opens an NVTX range named after itself
 *     around its host-side work (visible to a timeline profiler).
 *   - The library looks up the device addresses of its own device variables
 *     once per device and keeps them: cudaDeviceReset() on a device while the
 *     library is loaded is not supported (the kept addresses would point
 *     into the destroyed context); restart the process instead.
 */
#ifndef H3ATTN_H_
#define H3ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int h3_status;
#define H3_OK 0
#define H3_ERR_INVALID_ARG 1   /* bad pointer, size or alignment; nothing launched */
#define H3_ERR_UNSUPPORTED 2   /* valid but not implemented (e.g. head_dim != 128) */
#define H3_ERR_CUDA 3          /* a CUDA runtime call or launch failed */
#define H3_ERR_TIMEOUT 4       /* a kernel gave up on a bounded wait (device status) */
#define H3_ERR_BAD_INDEX 5     /* a modality id >= n_mod was met (device status) */
#define H3_ERR_WORKSPACE 6     /* workspace smaller than h3_workspace_size() */
#define H3_ERR_OUT_OF_BOUNDS 7 /* checked build only: a kernel index fell outside its
                                  buffer; the access was skipped (device status) */

/* Same handle as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* h3_stream_t;

/* Shape and options of one sub-block. */
typedef struct {
  int32_t L;            /* tokens in the packed sequence, >= 1 */
  int32_t d;            /* hidden size = n_heads * head_dim */
  int32_t n_heads;
  int32_t head_dim;     /* must be 128 */
  int32_t rope_sec[3];  /* rotary dims of the t, h, w axes; even, summing to head_dim */
  float rope_base;      /* frequency base (> 1), e.g. 10000 */
  float ln_eps;         /* LayerNorm epsilon (>= 0), e.g. 1e-6 */
  int32_t causal;       /* 0: full bidirectional attention; 1: key index <= query index */
  int32_t n_mod;        /* number of modalities (rows of shift/scale/gate) */
  int32_t n_seg;        /* 0: attention over the whole sequence; else number of segments */
  const int32_t* cu_seqlens; /* host [n_seg + 1] when n_seg > 0 (see h3_joint_attn_varlen_fwd) */
} h3_block_desc;

/* Shape of one MLP sub-block (the feed-forward half of a DiT layer). */
typedef struct {
  int32_t L;            /* tokens, >= 1 */
  int32_t d;            /* hidden size, d % 128 == 0 */
  int32_t hidden;       /* feed-forward width (e.g. 4d), hidden % 128 == 0, <= 65536 */
  float ln_eps;         /* LayerNorm epsilon (>= 0) */
  int32_t n_mod;        /* rows of shift/scale/gate */
} h3_mlp_desc;

/* Largest number of segments a cu_seqlens array may describe. */
#define H3_MAX_SEGMENTS 64

/* Text for a status code (static storage). */
const char* h3_status_string(h3_status s);

/* Library version, e.g. "h3attn 0.1.0 sm_103a". */
const char* h3_version(void);

/*
 * Packed layout metadata (host, integer; [vLLM] §3 data-flow table: row type,
 * position indices, modality tags).  Token order: text [0, T), video
 * row-major over (t, h, w), audio channel-major (token T + V + c*S + s).
 * mod: 0 text, 1 video, 2 audio.  pos[n] = (t, h, w): text (i, i, i), video
 * (t, h, w), audio (step, 0, channel), zero-based per modality.
 *   mod [capacity] uint8, pos [capacity][3] int32: host buffers owned by the caller.
 * Writes L = T + t*h*w + channels*steps tokens; returns H3_ERR_INVALID_ARG if a
 * count is negative, L == 0, L > capacity or L > INT32_MAX.
 */
h3_status h3_build_packed_layout(int32_t n_text, int32_t video_t, int32_t video_h,
                                 int32_t video_w, int32_t audio_channels, int32_t audio_steps,
                                 uint8_t* mod, int32_t* pos, int64_t capacity);

/*
 * Modality-indexed AdaLN LayerNorm + modulate ([H3-RL] AdaLN branches;
 * [VeRL] 三):  y[n] = (x[n] - mean) / sqrt(biased var + eps) * (1 + scale[m])
 * + shift[m], m = mod[n]; statistics in fp32.
 *   x [L][d] bf16, mod [L] uint8, shift/scale [n_mod][d] fp32 -> y [L][d] bf16.
 * A row whose modality id is >= n_mod is written as NaN and flags H3_ERR_BAD_INDEX.
 */
h3_status h3_adaln_modulate(const uint16_t* x, const uint8_t* mod, const float* shift,
                            const float* scale, int32_t L, int32_t d, int32_t n_mod, float eps,
                            uint16_t* y, h3_stream_t stream);

/*
 * Fused QKV projection ([VeRL] 5.2: Q, K, V packed in one matrix):
 *   qkv[n] = y[n] Wqkv^T, no bias; fp32 accumulation on the tensor cores.
 *   y [L][d] bf16, Wqkv [3d][d] bf16 -> qkv [L][3d] bf16, columns [Q | K | V],
 *   head h at columns h*128 .. h*128+127 inside each block.  Q and K are NOT
 *   rotated (see h3_mrope_apply).  qkv must not alias y.
 */
h3_status h3_qkv_proj(const uint16_t* y, const uint16_t* Wqkv, int32_t L, int32_t d,
                      uint16_t* qkv, h3_stream_t stream);

/*
 * 3D multimodal rotary embedding over (t, h, w) ([H3-RL]; [vLLM] §3), in place
 * on the Q and K blocks of qkv [L][3*H*dh]; V is untouched.  Head dims
 * [0, s0) follow t, [s0, s0+s1) follow h, the rest w.  Inside a section of
 * n_a dims, pair (2j, 2j+1) turns by pos[n][a] * base^(-2j/n_a):
 *   (u, v) -> (u cos - v sin, u sin + v cos); fp32 math, bf16 storage.
 *   pos [L][3] int32 (t, h, w).
 */
h3_status h3_mrope_apply(uint16_t* qkv, const int32_t* pos, int32_t L, int32_t n_heads,
                         int32_t head_dim, const int32_t sec[3], float base, h3_stream_t stream);

/*
 * Joint attention over the whole packed sequence ([vLLM] §1 shared attention
 * context; §6 only the L effective tokens take part; [VeRL] 三 causal option):
 *   O[n, h] = sum_j softmax_j(q_n . k_j * sm_scale) v_j over keys j in [0, L)
 *   (j <= n when causal).  bf16 tensor-core products, fp32 softmax/accumulation.
 *   qkv [L][3*H*dh] bf16 (Q, K rotated) -> O [L][H*dh] bf16.
 *   lse: optional [H][L] fp32 natural-log sum of exp(scores*sm_scale), or NULL.
 *   sm_scale > 0 (1/sqrt(head_dim) for the block).  O must not alias qkv.
 */
h3_status h3_joint_attn_fwd(const uint16_t* qkv, int32_t L, int32_t n_heads, int32_t head_dim,
                            int32_t causal, float sm_scale, uint16_t* O, float* lse,
                            h3_stream_t stream);

/*
 * Joint attention restricted to sub-sequences ([vLLM] §3 Packed Sequences and
 * Modality Identity Preservation: cu_seqlens is a 1-D array of segment offsets
 * and a token takes softmax only over the keys of its own segment; worked
 * example [0, 10, 30]: token 15 sees keys 10..29).
 *   cu_seqlens: HOST array [n_seg + 1], cu_seqlens[0] = 0, non-decreasing,
 *   cu_seqlens[n_seg] = L, 1 <= n_seg <= H3_MAX_SEGMENTS (empty segments
 *   allowed).  causal: additionally key index <= query index.  Other arguments
 *   and layouts as h3_joint_attn_fwd.  Key blocks outside a CTA's segments are
 *   not visited.
 */
h3_status h3_joint_attn_varlen_fwd(const uint16_t* qkv, const int32_t* cu_seqlens,
                                   int32_t n_seg, int32_t L, int32_t n_heads, int32_t head_dim,
                                   int32_t causal, float sm_scale, uint16_t* O, float* lse,
                                   h3_stream_t stream);

/*
 * Output projection + per-modality gated residual ([H3-RL] to_out.0 and the
 * AdaLN gate):  out[n] = x_res[n] + gate[mod[n]] * (O[n] Wo^T); fp32 epilogue.
 *   O [L][d] bf16, Wo [d][d] bf16, x_res [L][d] bf16, mod [L] uint8,
 *   gate [n_mod][d] fp32 -> out [L][d] bf16.  out may alias x_res (each element
 *   is read before it is written by the same thread); it must not alias O.
 */
h3_status h3_out_proj_gated_residual(const uint16_t* O, const uint16_t* Wo,
                                     const uint16_t* x_res, const uint8_t* mod,
                                     const float* gate, int32_t L, int32_t d, int32_t n_mod,
                                     uint16_t* out, h3_stream_t stream);

/*
 * One denoising-step update of the packed latent ([vLLM] §4 Denoising
 * Execution Flow, stages 5-7; [VeRL] 5.1: H3 time t = 1 - sigma, H3 velocity
 * = minus the standard flow-matching velocity).  For each token n with
 * modality m = mod[n] and update[m] != 0, with v = -v_h3[n]:
 *   x0[n] = z[n] - sigma[m] v            (rectified-flow clean estimate)
 *   z[n]  = z[n] + (sigma_next[m] - sigma[m]) v   (deterministic Euler step)
 * Rows with update[m] == 0 (conditions such as text) keep z (x0 = z).  Rows
 * with anchor[n] != 0 are re-pinned: z[n] = x0[n] = z_anchor[n].
 *   z [L][C] fp32 device, in place; x0 [L][C] fp32 device or NULL;
 *   v_h3 [L][C] bf16 device; mod [L] uint8 device; anchor [L] uint8 device or
 *   NULL (then z_anchor is ignored), z_anchor [L][C] fp32 device.
 *   sigma, sigma_next [n_mod] fp32 and update [n_mod] uint8: HOST arrays,
 *   0 <= sigma <= 1.  C % 4 == 0.  A modality id >= n_mod leaves its row
 *   unchanged and flags H3_ERR_BAD_INDEX.
 */
h3_status h3_denoise_step(float* z, float* x0, const uint16_t* v_h3, const uint8_t* mod,
                          const uint8_t* anchor, const float* z_anchor, int32_t L, int32_t C,
                          int32_t n_mod, const float* sigma, const float* sigma_next,
                          const uint8_t* update, h3_stream_t stream);

/*
 * The MLP sub-block that completes a DiT layer ([H3-RL]: feed-forward
 * projections ff.net.0.proj and ff.net.2 next to the attention's to_q/k/v and
 * to_out.0; modality-specific AdaLN branches; the pages give neither the
 * width nor the activation: GELU, tanh form):
 *   y   = LN(x) * (1 + scale[mod]) + shift[mod]
 *   h   = gelu(y W1^T)                       W1 [hidden][d] bf16
 *   out = x + gate[mod] * (h W2^T)           W2 [d][hidden] bf16
 * Three launches on `stream`: modulate, up projection with the GELU in its
 * epilogue, down projection with the gated residual in its epilogue.
 * workspace >= h3_mlp_workspace_size() bytes, 256-byte aligned.  out may alias x.
 */
h3_status h3_mlp_workspace_size(const h3_mlp_desc* desc, size_t* bytes);
h3_status h3_mlp_block_fwd(const h3_mlp_desc* desc, const uint16_t* x, const uint8_t* mod,
                           const float* shift, const float* scale, const float* gate,
                           const uint16_t* W1, const uint16_t* W2, void* workspace,
                           size_t workspace_bytes, uint16_t* out, h3_stream_t stream);

/*
 * FP8 (E4M3) variant of the projections ([vLLM] §5 Distributed Layerwise
 * Offload: the active block held at FP8 -- prior art; the oracle is the same
 * fp64 block, the tolerance follows from the E4M3 unit roundoff 2^-4).
 *
 * Row-wise quantisation: scale[r] = max|x[r]| / 448 (1 for an all-zero row),
 * q[r][k] = E4M3(x[r][k] / scale[r]), round-to-nearest, saturating.
 *   x [R][K] bf16 -> q [R][K] bytes, scale [R] fp32; K % 16 == 0.
 * Used on activations (one scale per token) and on weights (one scale per
 * output channel: the rows of W[out][in]).
 */
h3_status h3_quantize_rows_fp8(const uint16_t* x, int32_t R, int32_t K, uint8_t* q, float* scale,
                               h3_stream_t stream);

/*
 * C[m][n] = a_scale[m] * b_scale[n] * sum_k A[m][k] B[n][k] with E4M3 A [M][K]
 * and B [N][K] (tcgen05 kind::f8f6f4, fp32 accumulation) -> C [M][N] bf16.
 * N % 128 == 0, K % 128 == 0.
 */
h3_status h3_gemm_fp8(const uint8_t* A, const float* a_scale, const uint8_t* B,
                      const float* b_scale, int32_t M, int32_t N, int32_t K, uint16_t* C,
                      h3_stream_t stream);

/*
 * Joint attention with E4M3 scores ([vLLM] §6 Boundary Trimming for Packed
 * Attention names quantised attention kernels as prior art; this is the form
 * that quantises Q and K and keeps P V in bf16).  Same result as
 * h3_joint_attn_fwd up to the E4M3 rounding of Q and K:
 *   sq[h][i] = max_c |Q[i][h][c]| / 448          (one scale per token and head)
 *   sk[h][b] = max over tokens 128b..128b+127 and c of |K[i][h][c]| / 448
 *   Q8 = E4M3(Q / sq), K8 = E4M3(K / sk)          (round-to-nearest, saturating;
 *                                                   scale 1 for all-zero data)
 *   s_ij = sm_scale * sq[h][i] * sk[h][j/128] * (Q8_i . K8_j),  O = softmax(s) V
 * with V, P and O in bf16 and fp32 accumulation as in h3_joint_attn_fwd.
 *   qkv [L][3 * n_heads * 128] bf16 (Q, K after the rotary embedding) ->
 *   O [L][n_heads * 128] bf16, lse [n_heads][L] fp32 or NULL; causal 0 or 1.
 *   workspace: >= h3_attn_workspace_size_fp8(L, n_heads, 128) bytes, 256-byte
 *   aligned, caller-owned, holding qk8 [L][2 * n_heads * 128] bytes (Q8 | K8),
 *   then sq [n_heads][L] and sk [n_heads][ceil(L / 128)] fp32, each region at a
 *   256-byte boundary.  No cu_seqlens form.
 * h3_quantize_qk_fp8 is the first of the two launches on its own: it writes
 * qk8, sq and sk as above (qk8 8-byte aligned; sq, sk 4-byte aligned).
 */
h3_status h3_attn_workspace_size_fp8(int32_t L, int32_t n_heads, int32_t head_dim,
                                     size_t* bytes);
h3_status h3_quantize_qk_fp8(const uint16_t* qkv, int32_t L, int32_t n_heads, int32_t head_dim,
                             uint8_t* qk8, float* sq, float* sk, h3_stream_t stream);
h3_status h3_joint_attn_fwd_fp8(const uint16_t* qkv, int32_t L, int32_t n_heads,
                                int32_t head_dim, int32_t causal, float sm_scale,
                                void* workspace, size_t workspace_bytes, uint16_t* O, float* lse,
                                h3_stream_t stream);

/*
 * h3_attn_block_fwd with the two projections in FP8: y and O are quantised
 * per token before the QKV projection (RoPE in its epilogue) and the output
 * projection (gated residual in its epilogue).  Without segments
 * (desc->n_seg == 0) the attention takes E4M3 scores as in
 * h3_joint_attn_fwd_fp8; with segments it stays bf16.
 *   Wqkv_q [3d][d], Wo_q [d][d]: E4M3 weights from h3_quantize_rows_fp8, with
 *   their per-output-channel scales Wqkv_s [3d], Wo_s [d].
 * workspace >= h3_workspace_size_fp8(desc) bytes, 256-byte aligned.
 */
h3_status h3_workspace_size_fp8(const h3_block_desc* desc, size_t* bytes);
h3_status h3_attn_block_fwd_fp8(const h3_block_desc* desc, const uint16_t* x, const uint8_t* mod,
                                const int32_t* pos, const float* shift, const float* scale,
                                const float* gate, const uint8_t* Wqkv_q, const float* Wqkv_s,
                                const uint8_t* Wo_q, const float* Wo_s, void* workspace,
                                size_t workspace_bytes, uint16_t* out, h3_stream_t stream);

/* h3_mlp_block_fwd with both feed-forward projections in FP8 (y and h
 * quantised per token; W1_q [hidden][d], W2_q [d][hidden] with per-output-
 * channel scales W1_s [hidden], W2_s [d]). */
h3_status h3_mlp_workspace_size_fp8(const h3_mlp_desc* desc, size_t* bytes);
h3_status h3_mlp_block_fwd_fp8(const h3_mlp_desc* desc, const uint16_t* x, const uint8_t* mod,
                               const float* shift, const float* scale, const float* gate,
                               const uint8_t* W1_q, const float* W1_s, const uint8_t* W2_q,
                               const float* W2_s, void* workspace, size_t workspace_bytes,
                               uint16_t* out, h3_stream_t stream);

/* Bytes of device workspace h3_attn_block_fwd needs for `desc`. */
h3_status h3_workspace_size(const h3_block_desc* desc, size_t* bytes);

/*
 * The whole sub-block ([vLLM] §1: the step run 50 times over 58,758 tokens):
 * modulate -> QKV projection with the rotary embedding applied in its
 * epilogue -> joint attention (over the whole sequence, or per segment when
 * desc->n_seg > 0) -> output projection with gated residual, four launches on
 * `stream`.  workspace: >= h3_workspace_size() bytes of device
 * memory, 256-byte aligned, owned by the caller, not read before written.
 *   x [L][d] bf16, mod [L] uint8, pos [L][3] int32, shift/scale/gate
 *   [n_mod][d] fp32, Wqkv [3d][d] bf16, Wo [d][d] bf16 -> out [L][d] bf16.
 *   out may alias x.
 */
h3_status h3_attn_block_fwd(const h3_block_desc* desc, const uint16_t* x, const uint8_t* mod,
                            const int32_t* pos, const float* shift, const float* scale,
                            const float* gate, const uint16_t* Wqkv, const uint16_t* Wo,
                            void* workspace, size_t workspace_bytes, uint16_t* out,
                            h3_stream_t stream);

/*
 * h3_attn_block_fwd that also records five caller-created CUDA events
 * (cudaEvent_t[5], created on the current device) on `stream`: before the
 * first launch and after each of the four launches (modulate, QKV projection
 * + RoPE, attention, output projection), so the caller can time each kernel
 * inside a running step.  events == NULL behaves exactly like
 * h3_attn_block_fwd.
 */
h3_status h3_attn_block_fwd_profiled(const h3_block_desc* desc, const uint16_t* x,
                                     const uint8_t* mod, const int32_t* pos, const float* shift,
                                     const float* scale, const float* gate, const uint16_t* Wqkv,
                                     const uint16_t* Wo, void* workspace, size_t workspace_bytes,
                                     uint16_t* out, h3_stream_t stream, void* const* events);

/* Size of the workspace that h3_attn_block_fwd_noalloc keeps on every GPU: 64 MiB. */
#define H3_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * h3_attn_block_fwd for callers that cannot allocate device memory (the pages
 * have no counterpart: this is an interface convenience, not part of the
 * method).  An engine that plans every device buffer before it runs and hands
 * its plugins only their inputs and outputs, or a process whose caching
 * allocator already holds the GPU's memory, cannot get a workspace from
 * cudaMalloc at call time.  This call uses instead a workspace the library
 * keeps in device global memory: H3_NOALLOC_SCRATCH_BYTES per GPU that loads
 * the library, held until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *   - Arguments as in h3_attn_block_fwd, without workspace and size.
 *   - Returns H3_ERR_WORKSPACE, launching nothing, when h3_workspace_size(desc)
 *     exceeds H3_NOALLOC_SCRATCH_BYTES (e.g. 4,096 tokens at d = 2048 fit
 *     exactly; 58,758 tokens at d = 5120 do not).
 *   - The first call on a device looks up the workspace's device address
 *     (cudaGetSymbolAddress) with that device current.  With CUDA's lazy
 *     module loading that lookup is also when the 64 MiB are reserved on the
 *     device, so make the first call during set-up: before the caller's
 *     allocator or engine takes the device's memory, and before any stream
 *     capture begins.
 *   - All calls on a device share the one workspace and it keeps the last
 *     call's contents (nothing in it needs to start at zero).  Calls that
 *     overlap on the GPU race on it: order them on one stream or with events.
 */
h3_status h3_attn_block_fwd_noalloc(const h3_block_desc* desc, const uint16_t* x,
                                    const uint8_t* mod, const int32_t* pos, const float* shift,
                                    const float* scale, const float* gate, const uint16_t* Wqkv,
                                    const uint16_t* Wo, uint16_t* out, h3_stream_t stream);

/*
 * Synchronise `stream`, then report and clear the current device's status
 * word: H3_OK, H3_ERR_TIMEOUT, H3_ERR_BAD_INDEX, H3_ERR_OUT_OF_BOUNDS (checked
 * build) or H3_ERR_CUDA.
 */
h3_status h3_sync_status(h3_stream_t stream);

/*
 * Upper bound, in nanoseconds of GPU global-timer time, on every wait inside
 * the kernels (default 2e9).  A wait that exceeds it makes the kernel unwind
 * and record H3_ERR_TIMEOUT.  0 restores the default.
 */
void h3_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Self-test of the bounded-wait path: launches one CTA that waits on a
 * shared-memory barrier nothing arrives on, with the given limit.  The wait
 * must run out and the following h3_sync_status() must return H3_ERR_TIMEOUT.
 */
h3_status h3_selftest_wait_timeout(uint64_t limit_ns, h3_stream_t stream);

/*
 * The checked build.  The library can be compiled with H3_CHECKED defined
 * (libh3attn_checked.so, joint_audio_video_gb300/build.py, build(checked=True)):
 * then every global-memory load or store that a kernel addresses itself (all
 * but the TMA copies, which the hardware bounds) first tests its row and
 * column against the extents of its buffer; a test that fails records
 * H3_ERR_OUT_OF_BOUNDS in the device status word, skips the access, and the
 * kernel goes on.  Results are bit-identical to the normal build's.  This is a
 * debugging aid with no counterpart on the pages (the pages' lesson is that
 * kernel failures at this sequence length are silent: "Joint Audio-Video
 * Generation in Production", §6 Boundary Trimming for Packed Attention).
 *
 * h3_checked_build(): 1 in the checked build, 0 otherwise.
 * h3_selftest_bounds_check(): in the checked build, launches one thread that
 * addresses element 1 of a one-element buffer through the checked path, so the
 * following h3_sync_status() must return H3_ERR_OUT_OF_BOUNDS (nothing is
 * written); in the normal build it returns H3_ERR_UNSUPPORTED and launches
 * nothing.
 */
int32_t h3_checked_build(void);
h3_status h3_selftest_bounds_check(h3_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* H3ATTN_H_ */
