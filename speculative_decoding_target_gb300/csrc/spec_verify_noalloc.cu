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

// The array's device address belongs to the CUDA context that loaded this
// module, not to the device: a caller may run in a context of its own (an
// engine that creates and owns its driver context), and a device reset
// replaces the primary context.  So the address is cached per context,
// keyed by the context's process-unique id (cuCtxGetId; a handle value can
// be reused by a later context, an id is never reused).
using PFN_ctx_get_current = CUresult (*)(CUcontext*);
using PFN_ctx_get_id = CUresult (*)(CUcontext, unsigned long long*);

constexpr int kMaxContexts = 64;
std::mutex g_mu;
PFN_ctx_get_current g_get_current = nullptr;
PFN_ctx_get_id g_get_id = nullptr;
struct Entry {
  unsigned long long ctx_id;
  void* addr;
};
Entry g_cache[kMaxContexts];
int g_cached = 0, g_next = 0;

int driver_entry(const char* name, int version, void** fn) {
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion(name, fn, version,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !*fn)
    return specv::set_error(SPEC_ERR_CUDA, "%s unavailable: %s", name,
                            cudaGetErrorString(e));
  return SPEC_OK;
}

// Id of the calling thread's current context, or 0 when none is current.
int current_context_id(unsigned long long* id) {
  *id = 0;
  CUcontext ctx = nullptr;
  CUresult r = g_get_current(&ctx);
  if (r != CUDA_SUCCESS)
    return specv::set_error(SPEC_ERR_CUDA, "cuCtxGetCurrent failed (%d)",
                            (int)r);
  if (!ctx) return SPEC_OK;
  r = g_get_id(ctx, id);
  if (r != CUDA_SUCCESS)
    return specv::set_error(SPEC_ERR_CUDA, "cuCtxGetId failed (%d)", (int)r);
  return SPEC_OK;
}

int symbol_address(void** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p)
    return specv::set_error(SPEC_ERR_CUDA,
                            "cudaGetSymbolAddress of the scratch: %s",
                            cudaGetErrorString(e));
  *out = p;
  return SPEC_OK;
}

// Device address of the scratch array in the current context, looked up
// once per context.  In host code g_noalloc_scratch names a host-side
// stand-in, never the device array, so it is never passed to a kernel.
int scratch_address(void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  int rc;
  if (!g_get_current || !g_get_id) {
    void *f1 = nullptr, *f2 = nullptr;
    if ((rc = driver_entry("cuCtxGetCurrent", 4000, &f1))) return rc;
    if ((rc = driver_entry("cuCtxGetId", 12000, &f2))) return rc;
    g_get_current = reinterpret_cast<PFN_ctx_get_current>(f1);
    g_get_id = reinterpret_cast<PFN_ctx_get_id>(f2);
  }
  unsigned long long id = 0;
  if ((rc = current_context_id(&id))) return rc;
  void* addr = nullptr;
  if (id == 0) {
    // no context is current yet: the runtime makes the current device's
    // primary context current while it looks the symbol up
    if ((rc = symbol_address(&addr))) return rc;
    if ((rc = current_context_id(&id))) return rc;
  }
  for (int i = 0; i < g_cached; ++i)
    if (id != 0 && g_cache[i].ctx_id == id) {
      *out = g_cache[i].addr;
      return SPEC_OK;
    }
  if (!addr && (rc = symbol_address(&addr))) return rc;
  if (id != 0) {  // remember it (the oldest entry makes room)
    const int slot = g_cached < kMaxContexts ? g_cached++ : g_next;
    if (g_cached == kMaxContexts) g_next = (slot + 1) % kMaxContexts;
    g_cache[slot] = {id, addr};
  }
  *out = addr;
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
