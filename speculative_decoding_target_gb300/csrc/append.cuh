// Launch parameters of the block KV append kernel (kv_append.cu).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace specv {

struct AppendParams {
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  void* k_pages;
  void* v_pages;
  __half* k_scales;
  __half* v_scales;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* q_lens;  // optional [B]: rows of each block (<= q_len)
  int32_t* positions;   // optional
  int64_t* cache_loc;   // optional
  uint32_t* status;     // checked mode only
  int batch, q_len, hkv, page_size, log2_ps, num_pages, max_pages;
  long long max_tokens;
  int fp8;
};

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t s);

}  // namespace specv
