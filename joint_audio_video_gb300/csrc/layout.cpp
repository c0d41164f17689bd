// Host-side packed layout of one request ("Joint Audio-Video Generation in
// Production", §3 Packed Sequences and Modality Identity Preservation: every
// row carries its modality tag and its position indices into the DiT).
//
// Token order: text [0, T), video row-major over (t, h, w), audio
// channel-major (token T + V + c*S + s).  Positions (t, h, w): text (i, i, i),
// video (t, h, w), audio (step, 0, channel), all zero-based per modality.
#include <cstdint>

#include "../../include/h3attn.h"

extern "C" h3_status h3_build_packed_layout(int32_t n_text, int32_t video_t, int32_t video_h,
                                            int32_t video_w, int32_t audio_channels,
                                            int32_t audio_steps, uint8_t* mod, int32_t* pos,
                                            int64_t capacity) {
  if (n_text < 0 || video_t < 0 || video_h < 0 || video_w < 0 || audio_channels < 0 ||
      audio_steps < 0 || mod == nullptr || pos == nullptr)
    return H3_ERR_INVALID_ARG;
  // h * w first (< 2^62); a frame larger than any valid L is rejected before
  // the product with t could leave 64 bits
  const int64_t n_frame = int64_t(video_h) * video_w;
  if (video_t > 0 && n_frame > INT32_MAX) return H3_ERR_INVALID_ARG;
  const int64_t n_video = int64_t(video_t) * n_frame;
  const int64_t n_audio = int64_t(audio_channels) * audio_steps;
  const int64_t L = int64_t(n_text) + n_video + n_audio;
  if (L < 1 || L > capacity || L > INT32_MAX) return H3_ERR_INVALID_ARG;
  int64_t n = 0;
  for (int32_t i = 0; i < n_text; ++i, ++n) {
    mod[n] = 0;
    pos[3 * n + 0] = i;
    pos[3 * n + 1] = i;
    pos[3 * n + 2] = i;
  }
  for (int32_t t = 0; t < video_t; ++t)
    for (int32_t h = 0; h < video_h; ++h)
      for (int32_t w = 0; w < video_w; ++w, ++n) {
        mod[n] = 1;
        pos[3 * n + 0] = t;
        pos[3 * n + 1] = h;
        pos[3 * n + 2] = w;
      }
  for (int32_t c = 0; c < audio_channels; ++c)
    for (int32_t s = 0; s < audio_steps; ++s, ++n) {
      mod[n] = 2;
      pos[3 * n + 0] = s;
      pos[3 * n + 1] = 0;
      pos[3 * n + 2] = c;
    }
  return H3_OK;
}
