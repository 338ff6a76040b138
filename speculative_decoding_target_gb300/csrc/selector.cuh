// Launch parameters of the DFlash2 candidate selector (dflash2_select.cu).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace specv {

struct SelectParams {
  const float* cand_logits;     // [B, P-1, V]
  const int32_t* boundary;      // [B]
  const __nv_bfloat16* hidden;  // [B, P-1, D]
  const __nv_bfloat16* w_h;     // [R, D]
  const __nv_bfloat16* code_a;  // [V, R]
  const __nv_bfloat16* code_b;  // [V, R]
  int32_t* cand_ids;            // [B, P-1, K]
  float* cand_logit;            // [B, P-1, K]
  float* trans;                 // [B, P-1, K, K]
  int32_t* draft_ids;           // [B, P]
  float* part_val;              // [rows, chunks, K] chunk top-K values
  int32_t* part_idx;            // [rows, chunks, K] and token ids
  float* proj;                  // [D / 128, rows, R] slices of W_H h
  int* counters;                // [B] finished table CTAs (zeroed per call)
  int batch, positions, vocab, top, rank, dim, mode, chunks;
  int vec4;                     // logits rows 16-byte aligned, vocab % 4 == 0
};

constexpr int kSelChunk = 8192;     // logits per CTA of the top-K pass
constexpr int kSelThreads = 256;
constexpr int kSelMaxChunks = 32;   // vocab <= 32 * 8192 = 262,144
constexpr int kSelMaxRank = 256;

cudaError_t launch_dflash2_select(const SelectParams& p, cudaStream_t s);

}  // namespace specv
