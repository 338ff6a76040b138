// Launch parameters of stochastic (rejection-sampling) verify
// (stochastic_accept.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace specv {

struct StochasticParams {
  const float* logits;       // [B * q_len, vocab]
  const int32_t* draft_ids;  // [B, q_len]
  const float* draft_probs;  // optional [B, q_len - 1, vocab]
  const int32_t* q_lens;     // optional [B]
  const float* temperature;  // [B]
  const float* u_accept;     // [B, q_len - 1] (unused when q_len == 1)
  const float* u_sample;     // [B]
  const int32_t* seq_lens;   // optional [B], with new_seq_lens
  int32_t* new_seq_lens;
  int32_t* accept_len;       // [B]
  int32_t* next_token;       // [B]
  int32_t* out_tokens;       // optional [B, q_len]
  float* part_max;           // [rows, chunks] chunk maxima of the logits
  float* part_sum;           // [rows, chunks] sum exp2((x - max) k)
  float* chunk_w;            // [B, chunks] draw weight per chunk
  int batch, q_len, vocab, chunks;
  int vec4;                  // logits rows 16-byte aligned, vocab % 4 == 0
};

constexpr int kSampleChunk = 8192;   // logits per CTA of the streaming pass
constexpr int kSampleThreads = 256;
constexpr int kMaxSampleChunks = 128;  // vocab <= 128 * 8192

cudaError_t launch_stochastic_accept(const StochasticParams& p,
                                     cudaStream_t s);

}  // namespace specv
