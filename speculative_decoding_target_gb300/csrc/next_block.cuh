// Launch parameters of the next-block preparation kernel (next_block.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace specv {

struct NextBlockParams {
  const int32_t* q_lens;        // optional [B]: rows verified this step
  const int32_t* accept_len;    // [B]
  const int32_t* next_token;    // [B]
  const int32_t* new_seq_lens;  // [B]
  float* state;                 // [B] EWMA value or K (unused when fixed)
  const int32_t* page_table;    // [B, max_pages]
  int32_t* next_q_lens;         // [B]
  int32_t* next_seq_lens;       // [B]
  int32_t* block_ids;           // optional [B, q_max]
  int32_t* positions;           // optional [B, q_max]
  int64_t* cache_loc;           // optional [B, q_max]
  uint32_t* status;             // optional: SPEC_STATUS_NO_SLOT is OR-ed in
  int batch, policy, q_max, min_width, mask_id;
  int max_pages, page_size, num_pages;
  float alpha, offset;
};

cudaError_t launch_prepare_next_block(const NextBlockParams& p, cudaStream_t s);

}  // namespace specv
