// Verify attention for callers that cannot allocate device memory.
//
// spec_verify_attention needs a caller-provided workspace for its split
// partials.  Some callers cannot provide one: code that runs where no
// allocator is reachable (a plugin or callback handed only the input and
// output buffers of an engine that owns all device memory, or a runtime
// whose memory pool is fixed before this library is loaded) can neither
// call cudaMalloc nor hold a pool of its own.  For them this file keeps the
// split partials in a fixed, file-scope device array that the CUDA runtime
// reserves when the library's module is loaded on a device, and runs the
// same split and merge kernels on it.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "spec_verify.h"

namespace {

// Scratch for split partials.  Every GPU that loads this library holds it
// until the process exits.
static __device__ __align__(256) unsigned char
    g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch

// Device address of the scratch array on the current device, looked up once
// per device.  In host code g_noalloc_scratch names a host-side stand-in,
// never the device array, so it is never passed to a kernel directly.
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return specv::set_error(SPEC_ERR_CUDA, "cudaGetDevice: %s",
                            cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return specv::set_error(SPEC_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return specv::set_error(SPEC_ERR_CUDA,
                              "cudaGetSymbolAddress of the scratch: %s",
                              cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" int spec_verify_attention_noalloc(
    const spec_attn_desc* desc, const void* q, const void* k_pages,
    const void* v_pages, const void* k_scales, const void* v_scales,
    const int32_t* page_table, const int32_t* seq_lens, float scale,
    void* out, void* stream) {
  if (!desc) return specv::set_error(SPEC_ERR_ARG, "desc is NULL");
  if (desc->flags & SPEC_FLAG_CHECKED)
    return specv::set_error(SPEC_ERR_UNSUPPORTED,
                            "SPEC_FLAG_CHECKED needs a caller workspace to "
                            "report through; use spec_verify_attention");
  const size_t need = spec_verify_workspace_size(desc);
  if (need == 0) return SPEC_ERR_ARG;  // message set by the size query
  if (need > SPEC_NOALLOC_SCRATCH_BYTES)
    return specv::set_error(
        SPEC_ERR_WORKSPACE,
        "this shape needs %zu bytes of split scratch; the no-alloc entry "
        "point holds %zu (use spec_verify_attention with a workspace)",
        need, (size_t)SPEC_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc) return rc;
  // The split kernel writes every partial the merge kernel reads within
  // this call, so no part of the scratch has to start at zero.
  return spec_verify_attention(desc, q, k_pages, v_pages, k_scales, v_scales,
                               page_table, seq_lens, scale, out, scratch,
                               SPEC_NOALLOC_SCRATCH_BYTES, stream);
}
