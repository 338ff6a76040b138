// Greedy acceptance: launch parameters shared by the kernel and the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace specv {

struct AcceptParams {
  const float* logits;
  const int32_t* draft_ids;
  const int32_t* q_lens;     // optional [B]: rows of each block (<= q_len)
  const int32_t* seq_lens;   // optional [B], with new_seq_lens
  int32_t* new_seq_lens;     // optional [B]: seq_len - q_b + a + 1
  int32_t* accept_len;
  int32_t* next_token;
  int32_t* out_tokens;
  float* part_val;   // [rows, chunks]
  int32_t* part_idx; // [rows, chunks]
  int32_t* counters; // [batch]: finished CTAs per request (zeroed per call)
  int batch, q_len, vocab, rows, chunks;
  int vec4;          // logits rows are 16-byte aligned and vocab % 4 == 0
};
constexpr int kAcceptChunk = 8192;   // logits per argmax-partial CTA
constexpr int kAcceptThreads = 256;

cudaError_t launch_greedy_accept(const AcceptParams& p, cudaStream_t s);

}  // namespace specv
