// C ABI of the verify library: host-side validation, workspace layout and
// kernel launches.  Every error is detected here, before anything is
// enqueued, except a failed launch (SPEC_ERR_CUDA).
#include <cstdarg>
#include <cstdio>
#include <atomic>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "append.cuh"
#include "next_block.cuh"
#include "selector.cuh"
#include "stochastic.cuh"
#include "accept.cuh"
#include "common.cuh"
#include "spec_verify.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];
int g_occ[kMaxDevices][12];  // split-kernel CTAs per SM: [w] mma.sync with w
                             // compute warps, [9] tcgen05 bf16, [10] tcgen05
                             // FP8, [11] tcgen05 FP8 with TMEM KV operands
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
// main-loop wait bound of the split kernels for SPEC_FLAG_CHECKED calls
// (spec_verify_set_wait_limit); 0 = the default bound
std::atomic<long long> g_checked_wait_cycles{0};

bool use_tc(const spec_attn_desc* d) {
  return d->page_size >= specv::kTcMinPageSize;
}

// FP8 KV blocks of at most kFp8tMaxRows rows take the kernel whose K and V^T
// tiles are tensor-memory operands.
bool use_fp8t(const spec_attn_desc* d) {
  return d->kv_dtype == SPEC_KV_FP8_E4M3 && use_tc(d) &&
         (long long)d->q_len * (d->num_q_heads / d->num_kv_heads) <=
             specv::kFp8tMaxRows;
}

int tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion(
        "cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f)
      return fail(SPEC_ERR_CUDA, "cuTensorMapEncodeTiled unavailable: %s",
                  cudaGetErrorString(e));
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  *fn = g_encode;
  return SPEC_OK;
}

// 2-D view of a bf16 page pool: rows = num_pages * Hkv * page_size, 256
// elements (512 bytes) per row; boxes of 64 elements x box_rows rows with
// the 128-byte swizzle.
int make_pool_map(CUtensorMap* map, const void* base, long long rows,
                  int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int rc = tensor_map_encoder(&enc);
  if (rc) return rc;
  cuuint64_t dims[2] = {(cuuint64_t)specv::kHeadDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)specv::kHeadDim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t elem[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, elem,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(SPEC_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return SPEC_OK;
}

// 2-D view of an FP8 page pool: rows = num_pages * Hkv * page_size, 256
// bytes per row; boxes of 128 bytes x box_rows rows with the 128-byte
// swizzle.
int make_pool_map_u8(CUtensorMap* map, const void* base, long long rows,
                     int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int rc = tensor_map_encoder(&enc);
  if (rc) return rc;
  cuuint64_t dims[2] = {(cuuint64_t)specv::kHeadDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)specv::kHeadDim};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t elem[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                   const_cast<void*>(base), dims, strides, box, elem,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(SPEC_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return SPEC_OK;
}

int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess)
    return fail(SPEC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (*dev < 0 || *dev >= kMaxDevices)
    return fail(SPEC_ERR_UNSUPPORTED, "device ordinal %d too large", *dev);
  return SPEC_OK;
}

// Split-kernel grid for `rows` query rows per KV head on the current device:
// every SM filled with as many CTAs as fit.
int split_grid(int rows, bool tc, bool fp8, int* grid) {
  int dev;
  int rc = current_device(&dev);
  if (rc) return rc;
  const bool fp8t = tc && fp8 && rows <= specv::kFp8tMaxRows;
  const int w = fp8t ? 11 : (tc ? (fp8 ? 10 : 9) : (rows + 15) / 16);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    cudaError_t e =
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || n <= 0)
      return fail(SPEC_ERR_CUDA, "SM count: %s", cudaGetErrorString(e));
    g_sms[dev] = n;
  }
  if (!g_occ[dev][w]) {
    int occ = fp8t ? specv::verify_split_fp8t_ctas_per_sm()
              : tc  ? specv::verify_split_tc_ctas_per_sm(fp8)
                    : specv::verify_split_bf16_ctas_per_sm(rows);
    if (occ <= 0)
      return fail(SPEC_ERR_CUDA, "split kernel does not fit on an SM");
    g_occ[dev][w] = occ;
  }
  *grid = g_sms[dev] * g_occ[dev][w];
  return SPEC_OK;
}

int check_desc(const spec_attn_desc* d) {
  if (!d) return fail(SPEC_ERR_ARG, "desc is NULL");
  if (d->batch < 0 || d->batch > specv::kMaxBatch)
    return fail(SPEC_ERR_ARG, "batch %d outside [0, %d]", d->batch,
                specv::kMaxBatch);
  if (d->q_len < 1 || d->q_len > 16)
    return fail(SPEC_ERR_ARG, "q_len %d outside [1, 16]", d->q_len);
  if (d->num_q_heads < 1 || d->num_kv_heads < 1 ||
      d->num_q_heads % d->num_kv_heads)
    return fail(SPEC_ERR_ARG, "num_q_heads %d not a multiple of num_kv_heads %d",
                d->num_q_heads, d->num_kv_heads);
  if (d->head_dim != specv::kHeadDim)
    return fail(SPEC_ERR_UNSUPPORTED, "head_dim %d (only 256)", d->head_dim);
  const long long rows =
      (long long)d->q_len * (d->num_q_heads / d->num_kv_heads);
  if (rows > specv::kMaxRows)
    return fail(SPEC_ERR_UNSUPPORTED, "q_len * group = %lld > %d", rows,
                specv::kMaxRows);
  if (d->page_size < 1 || d->page_size > 4096 ||
      (d->page_size & (d->page_size - 1)))
    return fail(SPEC_ERR_ARG, "page_size %d is not a power of two in [1, 4096]",
                d->page_size);
  if (d->num_pages < 1 || d->max_pages_per_seq < 1)
    return fail(SPEC_ERR_ARG, "num_pages %d / max_pages_per_seq %d must be >= 1",
                d->num_pages, d->max_pages_per_seq);
  const long long max_tokens = (long long)d->max_pages_per_seq * d->page_size;
  if (max_tokens > (1LL << 30))
    return fail(SPEC_ERR_ARG, "max_pages_per_seq * page_size exceeds 2^30");
  const long long units = (long long)d->batch * d->num_kv_heads *
                          ((max_tokens + specv::kUnit - 1) / specv::kUnit +
                           specv::kMaxPieceCost);
  if (units > (1LL << 30))
    return fail(SPEC_ERR_ARG, "batch * kv heads * units exceeds 2^30");
  if (d->batch * (long long)d->num_kv_heads > 65535)
    return fail(SPEC_ERR_ARG, "batch * num_kv_heads exceeds 65535");
  if (d->kv_dtype != SPEC_KV_BF16 && d->kv_dtype != SPEC_KV_FP8_E4M3)
    return fail(SPEC_ERR_ARG, "kv_dtype %d", d->kv_dtype);
  if (d->flags & ~SPEC_FLAG_CHECKED)
    return fail(SPEC_ERR_ARG, "unknown flags 0x%x", d->flags);
  if (d->q_lens && !aligned(d->q_lens, 4))
    return fail(SPEC_ERR_ALIGN, "q_lens must be 4-byte aligned");
  if ((long long)d->num_pages * d->num_kv_heads * d->page_size >= (1LL << 31))
    return fail(SPEC_ERR_UNSUPPORTED,
                "num_pages * num_kv_heads * page_size must be < 2^31");
  if (d->kv_dtype == SPEC_KV_FP8_E4M3 && d->page_size < specv::kTcMinPageSize)
    return fail(SPEC_ERR_UNSUPPORTED, "FP8 KV needs page_size >= %d",
                specv::kTcMinPageSize);
  return SPEC_OK;
}

struct Layout {
  int rows, grid, nslots;
  size_t o_off, lse_off, bytes;
};

int layout(const spec_attn_desc* d, Layout* L) {
  L->rows = d->q_len * (d->num_q_heads / d->num_kv_heads);
  int rc = split_grid(L->rows, use_tc(d), d->kv_dtype == SPEC_KV_FP8_E4M3,
                      &L->grid);
  if (rc) return rc;
  // partial slots: chunk + segment index, below chunks + segments
  L->nslots = L->grid + d->batch * d->num_kv_heads;
  const size_t o_bytes =
      (size_t)L->nslots * L->rows * specv::kHeadDim * sizeof(float);
  const size_t lse_bytes = (size_t)L->nslots * L->rows * sizeof(float);
  L->o_off = specv::kWsHeader;
  L->lse_off = L->o_off + round_up(o_bytes, 256);
  L->bytes = L->lse_off + round_up(lse_bytes, 256);
  return SPEC_OK;
}

}  // namespace

namespace specv {
int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}
}  // namespace specv

extern "C" {

const char* spec_last_error(void) { return g_err; }

const char* spec_version(void) { return "spec_verify 0.2 (sm_103a)"; }

size_t spec_verify_workspace_size(const spec_attn_desc* desc) {
  if (check_desc(desc)) return 0;
  Layout L;
  if (layout(desc, &L)) return 0;
  return L.bytes;
}

int spec_verify_attention(const spec_attn_desc* desc, const void* q,
                          const void* k_pages, const void* v_pages,
                          const void* k_scales, const void* v_scales,
                          const int32_t* page_table, const int32_t* seq_lens,
                          float scale, void* out, void* workspace,
                          size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  int rc = check_desc(desc);
  if (rc) return rc;
  if (desc->batch == 0) return SPEC_OK;
  if (!q || !k_pages || !v_pages || !page_table || !seq_lens || !out)
    return fail(SPEC_ERR_ARG, "NULL tensor pointer");
  if (!(scale > 0.f) || scale > 3.0e38f)
    return fail(SPEC_ERR_ARG, "scale must be finite and > 0");
  if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) ||
      !aligned(out, 16))
    return fail(SPEC_ERR_ALIGN, "q, k_pages, v_pages and out must be 16-byte aligned");
  if (!aligned(page_table, 4) || !aligned(seq_lens, 4))
    return fail(SPEC_ERR_ALIGN, "page_table and seq_lens must be 4-byte aligned");
  const bool fp8 = desc->kv_dtype == SPEC_KV_FP8_E4M3;
  if (fp8) {
    if (!k_scales || !v_scales)
      return fail(SPEC_ERR_ARG, "FP8 KV needs k_scales and v_scales");
    if (!aligned(k_scales, 16) || !aligned(v_scales, 16))
      return fail(SPEC_ERR_ALIGN, "scales must be 16-byte aligned");
  }
  Layout L;
  rc = layout(desc, &L);
  if (rc) return rc;
  if (!workspace) return fail(SPEC_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 256))
    return fail(SPEC_ERR_ALIGN, "workspace must be 256-byte aligned");
  if (workspace_bytes < L.bytes)
    return fail(SPEC_ERR_WORKSPACE, "workspace %zu bytes < %zu needed",
                workspace_bytes, L.bytes);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  specv::AttnParams p;
  std::memset(&p, 0, sizeof p);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_pages = k_pages;
  p.v_pages = v_pages;
  p.k_scales = fp8 ? static_cast<const __half*>(k_scales) : nullptr;
  p.v_scales = fp8 ? static_cast<const __half*>(v_scales) : nullptr;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.q_lens = desc->q_lens;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.part_o = reinterpret_cast<float*>(ws + L.o_off);
  p.part_lse = reinterpret_cast<float*>(ws + L.lse_off);
  p.status = nullptr;
  p.batch = desc->batch;
  p.q_len = desc->q_len;
  p.hq = desc->num_q_heads;
  p.hkv = desc->num_kv_heads;
  p.group = desc->num_q_heads / desc->num_kv_heads;
  p.rows = L.rows;
  p.page_size = desc->page_size;
  p.log2_ps = 0;
  while ((1 << p.log2_ps) < desc->page_size) ++p.log2_ps;
  p.num_pages = desc->num_pages;
  p.max_pages = desc->max_pages_per_seq;
  p.max_tokens = desc->max_pages_per_seq * desc->page_size;
  p.grid = L.grid;
  p.piece_cost = use_fp8t(desc) ? specv::kFp8tPieceCost
                 : use_tc(desc) ? specv::kTcPieceCost
                                : specv::kMmaPieceCost;
  p.box_rows = specv::verify_split_tc_box_rows(desc->page_size);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_cycles = specv::kDrainWaitCycles;
  if (desc->flags & SPEC_FLAG_CHECKED) {
    const long long w = g_checked_wait_cycles.load(std::memory_order_relaxed);
    if (w > 0) p.wait_cycles = w;
  }
  const bool tc = use_tc(desc);
  const bool fp8t = use_fp8t(desc);
  CUtensorMap tm_k, tm_v;
  std::memset(&tm_k, 0, sizeof tm_k);  // unused by the bulk-copy FP8 kernel
  std::memset(&tm_v, 0, sizeof tm_v);
  const long long pool_rows =
      (long long)desc->num_pages * desc->num_kv_heads * desc->page_size;
  if (tc && !fp8) {
    rc = make_pool_map(&tm_k, k_pages, pool_rows, p.box_rows);
    if (!rc) rc = make_pool_map(&tm_v, v_pages, pool_rows, p.box_rows);
    if (rc) return rc;
  } else if (fp8t) {
    rc = make_pool_map_u8(&tm_k, k_pages, pool_rows, p.box_rows);
    if (!rc) rc = make_pool_map_u8(&tm_v, v_pages, pool_rows, p.box_rows);
    if (rc) return rc;
  }

  cudaError_t e;
  if (desc->flags & SPEC_FLAG_CHECKED) {
    p.status = reinterpret_cast<uint32_t*>(ws);
    e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess)
      return fail(SPEC_ERR_CUDA, "status reset: %s", cudaGetErrorString(e));
  }
  e = fp8t ? specv::launch_verify_split_fp8t(p, tm_k, tm_v, s)
       : tc  ? specv::launch_verify_split_tc(p, tm_k, tm_v, s)
             : specv::launch_verify_split_bf16(p, s);
  if (e != cudaSuccess)
    return fail(SPEC_ERR_CUDA, "split kernel launch: %s", cudaGetErrorString(e));
  e = specv::launch_verify_merge(p, s);
  if (e != cudaSuccess)
    return fail(SPEC_ERR_CUDA, "merge kernel launch: %s", cudaGetErrorString(e));
  return SPEC_OK;
}

int spec_verify_set_wait_limit(int64_t cycles) {
  g_err[0] = 0;
  if (cycles < 0 || cycles > specv::kDrainWaitCycles)
    return fail(SPEC_ERR_ARG, "wait limit %lld outside [0, %lld]",
                (long long)cycles, specv::kDrainWaitCycles);
  g_checked_wait_cycles.store(cycles, std::memory_order_relaxed);
  return SPEC_OK;
}

int spec_verify_status(const void* workspace, uint32_t* status_out,
                       int32_t clear, void* stream) {
  g_err[0] = 0;
  if (!workspace || !status_out)
    return fail(SPEC_ERR_ARG, "NULL workspace or status_out");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(status_out, workspace, sizeof(uint32_t),
                                  cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear)
    e = cudaMemsetAsync(const_cast<void*>(workspace), 0, sizeof(uint32_t), s);
  if (e != cudaSuccess)
    return fail(SPEC_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  return SPEC_OK;
}

int spec_kv_append(const spec_attn_desc* desc, const void* k_new,
                   const void* v_new, void* k_pages, void* v_pages,
                   void* k_scales, void* v_scales, const int32_t* page_table,
                   const int32_t* seq_lens, int32_t* positions,
                   int64_t* cache_loc, void* workspace, void* stream) {
  g_err[0] = 0;
  int rc = check_desc(desc);
  if (rc) return rc;
  if (desc->batch == 0) return SPEC_OK;
  if (!k_new || !v_new || !k_pages || !v_pages || !page_table || !seq_lens)
    return fail(SPEC_ERR_ARG, "NULL tensor pointer");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pages, 16) ||
      !aligned(v_pages, 16))
    return fail(SPEC_ERR_ALIGN, "k_new, v_new and the pools must be 16-byte aligned");
  if (!aligned(page_table, 4) || !aligned(seq_lens, 4) ||
      (positions && !aligned(positions, 4)) ||
      (cache_loc && !aligned(cache_loc, 8)))
    return fail(SPEC_ERR_ALIGN, "index arrays are misaligned");
  const bool fp8 = desc->kv_dtype == SPEC_KV_FP8_E4M3;
  if (fp8 && (!k_scales || !v_scales))
    return fail(SPEC_ERR_ARG, "FP8 KV needs k_scales and v_scales");
  if (fp8 && (!aligned(k_scales, 16) || !aligned(v_scales, 16)))
    return fail(SPEC_ERR_ALIGN, "scales must be 16-byte aligned");
  const bool checked = desc->flags & SPEC_FLAG_CHECKED;
  if (checked && !workspace)
    return fail(SPEC_ERR_WORKSPACE, "SPEC_FLAG_CHECKED needs a workspace");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  specv::AppendParams p;
  std::memset(&p, 0, sizeof p);
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.k_pages = k_pages;
  p.v_pages = v_pages;
  p.k_scales = fp8 ? static_cast<__half*>(k_scales) : nullptr;
  p.v_scales = fp8 ? static_cast<__half*>(v_scales) : nullptr;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.q_lens = desc->q_lens;
  p.positions = positions;
  p.cache_loc = cache_loc;
  p.batch = desc->batch;
  p.q_len = desc->q_len;
  p.hkv = desc->num_kv_heads;
  p.page_size = desc->page_size;
  p.log2_ps = 0;
  while ((1 << p.log2_ps) < desc->page_size) ++p.log2_ps;
  p.num_pages = desc->num_pages;
  p.max_pages = desc->max_pages_per_seq;
  p.max_tokens = (long long)desc->max_pages_per_seq * desc->page_size;
  p.fp8 = fp8;
  cudaError_t e;
  if (checked) {
    p.status = static_cast<uint32_t*>(workspace);
    e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess)
      return fail(SPEC_ERR_CUDA, "status reset: %s", cudaGetErrorString(e));
  }
  e = specv::launch_kv_append(p, s);
  if (e != cudaSuccess)
    return fail(SPEC_ERR_CUDA, "append kernel launch: %s", cudaGetErrorString(e));
  return SPEC_OK;
}

int spec_prepare_next_block(const spec_width_policy* pol, int32_t batch,
                            const int32_t* q_lens, const int32_t* accept_len,
                            const int32_t* next_token,
                            const int32_t* new_seq_lens, float* state,
                            const int32_t* page_table,
                            int32_t max_pages_per_seq, int32_t page_size,
                            int32_t num_pages, int32_t* next_q_lens,
                            int32_t* next_seq_lens, int32_t* block_ids,
                            int32_t* positions, int64_t* cache_loc,
                            uint32_t* status, void* stream) {
  g_err[0] = 0;
  if (!pol) return fail(SPEC_ERR_ARG, "policy is NULL");
  if (pol->policy < SPEC_WIDTH_FIXED || pol->policy > SPEC_WIDTH_DOUBLING)
    return fail(SPEC_ERR_ARG, "unknown width policy %d", pol->policy);
  if (pol->q_max < 1 || pol->q_max > 16)
    return fail(SPEC_ERR_ARG, "q_max %d outside [1, 16]", pol->q_max);
  if (pol->min_width < 1 || pol->min_width > pol->q_max)
    return fail(SPEC_ERR_ARG, "min_width %d outside [1, q_max]", pol->min_width);
  if (!(pol->alpha >= 0.f && pol->alpha <= 1.f) ||
      !(pol->offset > -1e6f && pol->offset < 1e6f))
    return fail(SPEC_ERR_ARG, "alpha must lie in [0, 1] and offset be finite");
  if (batch < 0 || batch > (1 << 24))
    return fail(SPEC_ERR_ARG, "batch %d outside [0, 2^24]", batch);
  if (page_size < 1 || max_pages_per_seq < 1 || num_pages < 1)
    return fail(SPEC_ERR_ARG, "page_size, max_pages_per_seq and num_pages must be >= 1");
  if (batch == 0) return SPEC_OK;
  if (!accept_len || !next_token || !new_seq_lens || !page_table ||
      !next_q_lens || !next_seq_lens)
    return fail(SPEC_ERR_ARG, "NULL tensor pointer");
  if (pol->policy != SPEC_WIDTH_FIXED && !state)
    return fail(SPEC_ERR_ARG, "this width policy needs its state array");
  const void* a4[] = {q_lens, accept_len, next_token, new_seq_lens, state,
                      page_table, next_q_lens, next_seq_lens, block_ids,
                      positions, status};
  for (const void* q : a4)
    if (q && !aligned(q, 4))
      return fail(SPEC_ERR_ALIGN, "int32 / float buffers must be 4-byte aligned");
  if (cache_loc && !aligned(cache_loc, 8))
    return fail(SPEC_ERR_ALIGN, "cache_loc must be 8-byte aligned");
  specv::NextBlockParams p;
  std::memset(&p, 0, sizeof p);
  p.q_lens = q_lens;
  p.accept_len = accept_len;
  p.next_token = next_token;
  p.new_seq_lens = new_seq_lens;
  p.state = state;
  p.page_table = page_table;
  p.next_q_lens = next_q_lens;
  p.next_seq_lens = next_seq_lens;
  p.block_ids = block_ids;
  p.positions = positions;
  p.cache_loc = cache_loc;
  p.status = status;
  p.batch = batch;
  p.policy = pol->policy;
  p.q_max = pol->q_max;
  p.min_width = pol->min_width;
  p.mask_id = pol->mask_id;
  p.max_pages = max_pages_per_seq;
  p.page_size = page_size;
  p.num_pages = num_pages;
  p.alpha = pol->alpha;
  p.offset = pol->offset;
  cudaError_t e =
      specv::launch_prepare_next_block(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(SPEC_ERR_CUDA, "prepare kernel launch: %s", cudaGetErrorString(e));
  return SPEC_OK;
}

size_t spec_stochastic_workspace_size(int32_t batch, int32_t q_len,
                                      int32_t vocab) {
  if (batch < 0 || q_len < 1 || q_len > 16 || vocab < 1) {
    fail(SPEC_ERR_ARG, "batch %d / q_len %d / vocab %d", batch, q_len, vocab);
    return 0;
  }
  const size_t chunks = (vocab + specv::kSampleChunk - 1) / specv::kSampleChunk;
  const size_t rows = (size_t)batch * q_len;
  return 2 * round_up(rows * chunks * sizeof(float), 256) +
         round_up((size_t)batch * chunks * sizeof(float), 256);
}

int spec_stochastic_accept(const float* logits, const int32_t* draft_ids,
                           const float* draft_probs, const int32_t* q_lens,
                           int32_t batch, int32_t q_len, int32_t vocab,
                           const float* temperature, const float* u_accept,
                           const float* u_sample, const int32_t* seq_lens,
                           int32_t* new_seq_lens, int32_t* accept_len,
                           int32_t* next_token, int32_t* out_tokens,
                           void* workspace, size_t workspace_bytes,
                           void* stream) {
  g_err[0] = 0;
  if (batch < 0) return fail(SPEC_ERR_ARG, "batch %d < 0", batch);
  if (q_len < 1 || q_len > 16)
    return fail(SPEC_ERR_ARG, "q_len %d outside [1, 16]", q_len);
  if (vocab < 1 || vocab > specv::kMaxSampleChunks * specv::kSampleChunk)
    return fail(SPEC_ERR_ARG, "vocab %d outside [1, %d]", vocab,
                specv::kMaxSampleChunks * specv::kSampleChunk);
  if ((long long)batch * q_len > 65535)
    return fail(SPEC_ERR_ARG, "batch * q_len exceeds 65535");
  if (batch == 0) return SPEC_OK;
  if (!logits || !draft_ids || !temperature || !u_sample || !accept_len ||
      !next_token || (q_len > 1 && !u_accept))
    return fail(SPEC_ERR_ARG, "NULL tensor pointer");
  if (!seq_lens != !new_seq_lens)
    return fail(SPEC_ERR_ARG, "seq_lens and new_seq_lens go together");
  const void* a4[] = {logits, draft_ids, draft_probs, q_lens, temperature,
                      u_accept, u_sample, seq_lens, new_seq_lens, accept_len,
                      next_token, out_tokens};
  for (const void* q : a4)
    if (q && !aligned(q, 4))
      return fail(SPEC_ERR_ALIGN, "tensors must be 4-byte aligned");
  if (!workspace) return fail(SPEC_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 16))
    return fail(SPEC_ERR_ALIGN, "workspace must be 16-byte aligned");
  const size_t need = spec_stochastic_workspace_size(batch, q_len, vocab);
  if (workspace_bytes < need)
    return fail(SPEC_ERR_WORKSPACE, "workspace %zu bytes < %zu needed",
                workspace_bytes, need);
  specv::StochasticParams p;
  std::memset(&p, 0, sizeof p);
  p.logits = logits;
  p.draft_ids = draft_ids;
  p.draft_probs = draft_probs;
  p.q_lens = q_lens;
  p.temperature = temperature;
  p.u_accept = u_accept;
  p.u_sample = u_sample;
  p.seq_lens = seq_lens;
  p.new_seq_lens = new_seq_lens;
  p.accept_len = accept_len;
  p.next_token = next_token;
  p.out_tokens = out_tokens;
  p.batch = batch;
  p.q_len = q_len;
  p.vocab = vocab;
  p.chunks = (vocab + specv::kSampleChunk - 1) / specv::kSampleChunk;
  p.vec4 = (vocab % 4 == 0) && aligned(logits, 16);
  const size_t rows = (size_t)batch * q_len;
  const size_t part = round_up(rows * p.chunks * sizeof(float), 256);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.part_max = reinterpret_cast<float*>(ws);
  p.part_sum = reinterpret_cast<float*>(ws + part);
  p.chunk_w = reinterpret_cast<float*>(ws + 2 * part);
  cudaError_t e =
      specv::launch_stochastic_accept(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(SPEC_ERR_CUDA, "stochastic accept launch: %s",
                cudaGetErrorString(e));
  return SPEC_OK;
}

namespace {
int check_select(const spec_select_desc* d) {
  if (!d) return fail(SPEC_ERR_ARG, "desc is NULL");
  if (d->batch < 0 || d->positions < 2 || d->positions > 16)
    return fail(SPEC_ERR_ARG, "batch %d / positions %d (2..16)", d->batch,
                d->positions);
  if (d->top < 1 || d->top > 16)
    return fail(SPEC_ERR_ARG, "top %d outside [1, 16]", d->top);
  if (d->vocab < d->top || d->vocab > specv::kSelMaxChunks * specv::kSelChunk)
    return fail(SPEC_ERR_ARG, "vocab %d outside [top, %d]", d->vocab,
                specv::kSelMaxChunks * specv::kSelChunk);
  if (d->rank < 8 || d->rank > specv::kSelMaxRank || d->rank % 8)
    return fail(SPEC_ERR_ARG, "rank %d: a multiple of 8 in [8, %d]", d->rank,
                specv::kSelMaxRank);
  if (d->dim < 16 || d->dim % 16)
    return fail(SPEC_ERR_ARG, "dim %d: a multiple of 16", d->dim);
  if (d->mode != SPEC_SELECT_GREEDY && d->mode != SPEC_SELECT_MAP)
    return fail(SPEC_ERR_ARG, "mode %d", d->mode);
  if ((long long)d->batch * (d->positions - 1) > 65535)
    return fail(SPEC_ERR_ARG, "batch * (positions - 1) exceeds 65535");
  return SPEC_OK;
}

struct SelectLayout {
  size_t part_val, part_idx, proj, trans, cand_ids, cand_logit, counters,
      bytes;
};

SelectLayout select_layout(const spec_select_desc* d) {
  const size_t rows = (size_t)d->batch * (d->positions - 1);
  const size_t chunks = (d->vocab + specv::kSelChunk - 1) / specv::kSelChunk;
  SelectLayout L;
  size_t o = 0;
  auto take = [&](size_t n) {
    const size_t at = o;
    o += round_up(n, 256);
    return at;
  };
  L.part_val = take(rows * chunks * d->top * sizeof(float));
  L.part_idx = take(rows * chunks * d->top * sizeof(int32_t));
  L.proj = take((size_t)((d->dim + 127) / 128) * rows * d->rank * sizeof(float));
  L.trans = take(rows * d->top * d->top * sizeof(float));
  L.cand_ids = take(rows * d->top * sizeof(int32_t));
  L.cand_logit = take(rows * d->top * sizeof(float));
  L.counters = take((size_t)d->batch * sizeof(int));
  L.bytes = o;
  return L;
}
}  // namespace

size_t spec_select_workspace_size(const spec_select_desc* desc) {
  if (check_select(desc)) return 0;
  return select_layout(desc).bytes;
}

int spec_dflash2_select(const spec_select_desc* desc, const float* cand_logits,
                        const int32_t* boundary, const void* hidden,
                        const void* w_h, const void* code_a, const void* code_b,
                        int32_t* draft_ids, int32_t* cand_ids,
                        float* cand_logit, float* trans, void* workspace,
                        size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  int rc = check_select(desc);
  if (rc) return rc;
  if (desc->batch == 0) return SPEC_OK;
  if (!cand_logits || !boundary || !hidden || !w_h || !code_a || !code_b ||
      !draft_ids)
    return fail(SPEC_ERR_ARG, "NULL tensor pointer");
  const void* a4[] = {cand_logits, boundary, hidden, w_h, draft_ids,
                      cand_ids, cand_logit, trans};
  for (const void* q : a4)
    if (q && !aligned(q, 4))
      return fail(SPEC_ERR_ALIGN, "tensors must be 4-byte aligned");
  if (!aligned(code_a, 2) || !aligned(code_b, 2))
    return fail(SPEC_ERR_ALIGN, "codebooks must be 2-byte aligned");
  if (!workspace) return fail(SPEC_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 256))
    return fail(SPEC_ERR_ALIGN, "workspace must be 256-byte aligned");
  const SelectLayout L = select_layout(desc);
  if (workspace_bytes < L.bytes)
    return fail(SPEC_ERR_WORKSPACE, "workspace %zu bytes < %zu needed",
                workspace_bytes, L.bytes);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  specv::SelectParams p;
  std::memset(&p, 0, sizeof p);
  p.cand_logits = cand_logits;
  p.boundary = boundary;
  p.hidden = static_cast<const __nv_bfloat16*>(hidden);
  p.w_h = static_cast<const __nv_bfloat16*>(w_h);
  p.code_a = static_cast<const __nv_bfloat16*>(code_a);
  p.code_b = static_cast<const __nv_bfloat16*>(code_b);
  p.cand_ids = cand_ids ? cand_ids : reinterpret_cast<int32_t*>(ws + L.cand_ids);
  p.cand_logit = cand_logit ? cand_logit
                            : reinterpret_cast<float*>(ws + L.cand_logit);
  p.trans = trans ? trans : reinterpret_cast<float*>(ws + L.trans);
  p.draft_ids = draft_ids;
  p.part_val = reinterpret_cast<float*>(ws + L.part_val);
  p.part_idx = reinterpret_cast<int32_t*>(ws + L.part_idx);
  p.proj = reinterpret_cast<float*>(ws + L.proj);
  p.counters = reinterpret_cast<int*>(ws + L.counters);
  p.batch = desc->batch;
  p.positions = desc->positions;
  p.vocab = desc->vocab;
  p.top = desc->top;
  p.rank = desc->rank;
  p.dim = desc->dim;
  p.mode = desc->mode;
  p.chunks = (desc->vocab + specv::kSelChunk - 1) / specv::kSelChunk;
  p.vec4 = (desc->vocab % 4 == 0) && aligned(cand_logits, 16);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(p.counters, 0, desc->batch * sizeof(int), s);
  if (e != cudaSuccess)
    return fail(SPEC_ERR_CUDA, "counter reset: %s", cudaGetErrorString(e));
  e = specv::launch_dflash2_select(p, s);
  if (e != cudaSuccess)
    return fail(SPEC_ERR_CUDA, "selector launch: %s", cudaGetErrorString(e));
  return SPEC_OK;
}

size_t spec_accept_workspace_size(int32_t rows, int32_t vocab) {
  if (rows < 0 || vocab < 1) {
    fail(SPEC_ERR_ARG, "rows %d / vocab %d", rows, vocab);
    return 0;
  }
  const size_t chunks = ((size_t)vocab + specv::kAcceptChunk - 1) /
                        specv::kAcceptChunk;
  return round_up((size_t)rows * chunks * sizeof(float), 256) +
         round_up((size_t)rows * chunks * sizeof(int32_t), 256) +
         round_up((size_t)rows * sizeof(int32_t), 256) + 256;
}

int spec_greedy_accept(const float* logits, const int32_t* draft_ids,
                       int32_t batch, int32_t q_len, int32_t vocab,
                       int32_t* accept_len, int32_t* next_token,
                       int32_t* out_tokens, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return spec_greedy_accept_commit(logits, draft_ids, nullptr, batch, q_len,
                                   vocab, nullptr, nullptr, accept_len,
                                   next_token, out_tokens, workspace,
                                   workspace_bytes, stream);
}

int spec_greedy_accept_commit(const float* logits, const int32_t* draft_ids,
                              const int32_t* q_lens, int32_t batch,
                              int32_t q_len, int32_t vocab,
                              const int32_t* seq_lens, int32_t* new_seq_lens,
                              int32_t* accept_len, int32_t* next_token,
                              int32_t* out_tokens, void* workspace,
                              size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  if (batch < 0) return fail(SPEC_ERR_ARG, "batch %d < 0", batch);
  if (q_len < 1 || q_len > 16)
    return fail(SPEC_ERR_ARG, "q_len %d outside [1, 16]", q_len);
  if (vocab < 1) return fail(SPEC_ERR_ARG, "vocab %d < 1", vocab);
  if ((long long)batch * q_len > 65535)
    return fail(SPEC_ERR_ARG, "batch * q_len exceeds 65535");
  if (batch == 0) return SPEC_OK;
  if (!logits || !draft_ids || !accept_len || !next_token)
    return fail(SPEC_ERR_ARG, "NULL tensor pointer");
  if (!aligned(logits, 4) || !aligned(draft_ids, 4) || !aligned(accept_len, 4) ||
      !aligned(next_token, 4) || (out_tokens && !aligned(out_tokens, 4)) ||
      (q_lens && !aligned(q_lens, 4)) || (seq_lens && !aligned(seq_lens, 4)) ||
      (new_seq_lens && !aligned(new_seq_lens, 4)))
    return fail(SPEC_ERR_ALIGN, "logits and int32 buffers must be 4-byte aligned");
  if (!seq_lens != !new_seq_lens)
    return fail(SPEC_ERR_ARG, "seq_lens and new_seq_lens go together");
  if (!workspace) return fail(SPEC_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 16))
    return fail(SPEC_ERR_ALIGN, "workspace must be 16-byte aligned");
  const int rows = batch * q_len;
  const size_t need = spec_accept_workspace_size(rows, vocab);
  if (workspace_bytes < need)
    return fail(SPEC_ERR_WORKSPACE, "workspace %zu bytes < %zu needed",
                workspace_bytes, need);
  specv::AcceptParams p;
  p.logits = logits;
  p.draft_ids = draft_ids;
  p.q_lens = q_lens;
  p.seq_lens = seq_lens;
  p.new_seq_lens = new_seq_lens;
  p.accept_len = accept_len;
  p.next_token = next_token;
  p.out_tokens = out_tokens;
  p.batch = batch;
  p.q_len = q_len;
  p.vocab = vocab;
  p.rows = rows;
  p.chunks = (vocab + specv::kAcceptChunk - 1) / specv::kAcceptChunk;
  p.vec4 = (vocab % 4 == 0) && aligned(logits, 16);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.part_val = reinterpret_cast<float*>(ws);
  const size_t idx_off = round_up((size_t)rows * p.chunks * sizeof(float), 256);
  p.part_idx = reinterpret_cast<int32_t*>(ws + idx_off);
  p.counters = reinterpret_cast<int32_t*>(
      ws + idx_off + round_up((size_t)rows * p.chunks * sizeof(int32_t), 256));
  cudaError_t e = specv::launch_greedy_accept(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(SPEC_ERR_CUDA, "accept kernel launch: %s", cudaGetErrorString(e));
  return SPEC_OK;
}

}  // extern "C"
